"""Host-side checks of the C ABI (no GPU work): the library builds and loads,
exports every function include/escha.h declares, and rejects bad arguments
with the documented status codes before touching the device."""
import ctypes
import os
import re
import subprocess

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "escha.h")


def _lib():
    from bit_trellis_quantized_gb300 import native

    if not os.path.exists(native.LIB_PATH):
        from bit_trellis_quantized_gb300 import build

        build.build()
    return native, native.lib()


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w]*\s*\**\s*([a-z][a-z0-9_]+)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "sizeof")))


def test_header_declarations_are_exported():
    native, _ = _lib()
    declared = _declared_functions()
    assert "escha_trellis_gemv" in declared and "escha_moe_block" in declared and "int8_w8a16_matvec" in declared
    out = subprocess.run(["nm", "-D", "--defined-only", native.LIB_PATH], capture_output=True, text=True, check=True)
    exported = set(line.split()[-1] for line in out.stdout.splitlines() if line.strip())
    missing = [n for n in declared if n not in exported]
    assert not missing, f"declared but not exported: {missing}"
    assert sorted(native.EXPORTS) == declared


def test_struct_layout_matches_header():
    native, _ = _lib()
    # 4 ints, 1 pointer, (pointer, int, pointer, pointer) x 2, int + 5 pointers, natural alignment
    assert ctypes.sizeof(native.EschaMoeLayer) == 136
    # char[256] + 10 ints; char[8], int, (pad 4), long long[8], size_t
    assert ctypes.sizeof(native.EschaProjInfo) == 296
    assert ctypes.sizeof(native.EschaTensorInfo) == 88


def test_version():
    _, L = _lib()
    assert L.escha_version() >= 100


def _fake_ptr(v):
    return ctypes.c_void_p(v)


def test_gemv_argument_validation_before_launch():
    native, L = _lib()
    good = 0x10000
    args = dict(codes=good, inn=256, out=256, K=2, x=good, xd=native.ESCHA_F16, batch=1, rin=good, rout=good, y=good)

    def call(**kw):
        a = dict(args)
        a.update(kw)
        return L.escha_trellis_gemv(a["codes"], a["inn"], a["out"], a["K"], a["x"], a["xd"], a["batch"], a["rin"],
                                    a["rout"], a["y"], None, 0, None)

    assert call(K=4) == native.ESCHA_E_K
    assert call(K=1) == native.ESCHA_E_K
    assert call(inn=200) == native.ESCHA_E_SHAPE
    assert call(out=16) == native.ESCHA_E_SHAPE
    assert call(inn=0) == native.ESCHA_E_SHAPE
    assert call(codes=None) == native.ESCHA_E_ARG
    assert call(y=None) == native.ESCHA_E_ARG
    assert call(xd=7) == native.ESCHA_E_ARG
    assert call(batch=0) == native.ESCHA_E_ARG
    assert call(codes=good + 8) == native.ESCHA_E_ALIGN
    assert call(x=good + 2) == native.ESCHA_E_ALIGN
    assert b"K=4" in L.escha_last_error() or True
    call(K=4)
    assert b"K=4" in L.escha_last_error()


def test_dense_linear_validation_before_launch():
    native, L = _lib()
    g = 0x10000
    ws_bytes = L.escha_dense_linear_workspace(256, 256, 2, 4)
    assert ws_bytes >= 16
    # the GEMM route needs its B image: more workspace for more tokens
    assert L.escha_dense_linear_workspace(5120, 17408, 2, 2048) > L.escha_dense_linear_workspace(5120, 17408, 2, 64)
    args = dict(codes=g, inn=256, out=256, K=2, nt=1, x=g, xd=native.ESCHA_F16, M=4, rin=g, rout=g, bias=None, y=g,
                ws=g, wsb=ws_bytes)

    def call(**kw):
        a = dict(args)
        a.update(kw)
        return L.escha_dense_linear(a["codes"], a["inn"], a["out"], a["K"], a["nt"], a["x"], a["xd"], a["M"],
                                    a["rin"], a["rout"], a["bias"], a["y"], a["ws"], a["wsb"], None)

    assert call(K=4) == native.ESCHA_E_K
    assert call(inn=200) == native.ESCHA_E_SHAPE
    assert call(out=64) == native.ESCHA_E_SHAPE
    assert call(inn=65536 + 128) == native.ESCHA_E_SHAPE
    assert call(nt=2) == native.ESCHA_E_ARG
    assert call(xd=native.ESCHA_BF16) == native.ESCHA_E_ARG
    assert call(M=0) == native.ESCHA_E_ARG
    assert call(M=65537) == native.ESCHA_E_ARG
    assert call(ws=None) == native.ESCHA_E_ARG
    assert call(wsb=0) == native.ESCHA_E_WORKSPACE
    assert call(bias=g + 4) == native.ESCHA_E_ALIGN
    assert call(y=g + 8) == native.ESCHA_E_ALIGN
    assert L.escha_codes_to_nt_major(g, 32, 32, 2, g + 16, None) == native.ESCHA_E_ARG  # overlapping buffers
    assert L.escha_codes_to_nt_major(g, 32, 32, 7, g + 65536, None) == native.ESCHA_E_K
    assert L.escha_codes_to_nt_major(g, 32, 32, 2, None, None) == native.ESCHA_E_ARG


def test_checkpoint_entry_points_reject_null_handles():
    native, L = _lib()
    info = native.EschaProjInfo()
    assert L.escha_ckpt_num_projections(None) == 0
    assert L.escha_ckpt_projection(None, 0, ctypes.byref(info)) == native.ESCHA_E_ARG
    assert L.escha_ckpt_read(None, b"x", None, 0, 0, None) == native.ESCHA_E_ARG
    h = ctypes.c_void_p()
    assert L.escha_ckpt_open(None, 0, ctypes.byref(h)) == native.ESCHA_E_ARG
    L.escha_ckpt_close(None)  # a null handle is ignored


def test_decode_validation():
    native, L = _lib()
    g = 0x10000
    assert L.escha_trellis_decode(g, 32, 32, 5, g, None) == native.ESCHA_E_K
    assert L.escha_trellis_decode(g, 24, 32, 2, g, None) == native.ESCHA_E_SHAPE
    assert L.escha_trellis_decode(None, 32, 32, 2, g, None) == native.ESCHA_E_ARG
    assert L.escha_trellis_decode(g, 32, 32, 2, None, None) == native.ESCHA_E_ARG


def test_int8_validation():
    native, L = _lib()
    g = 0x10000
    f = L.int8_w8a16_matvec
    assert f(None, g, 16, 32, g, native.ESCHA_BF16, 1, g, None, 0, None) == native.ESCHA_E_ARG
    assert f(g, g, 16, 30, g, native.ESCHA_BF16, 1, g, None, 0, None) == native.ESCHA_E_SHAPE
    assert f(g, g, 0, 32, g, native.ESCHA_BF16, 1, g, None, 0, None) == native.ESCHA_E_ARG
    assert f(g, g, 16, 32, g, 9, 1, g, None, 0, None) == native.ESCHA_E_ARG
    assert f(g + 4, g, 16, 32, g, native.ESCHA_BF16, 1, g, None, 0, None) == native.ESCHA_E_ALIGN


def test_moe_validation_and_workspace():
    native, L = _lib()
    g = 0x10000
    lay = native.EschaMoeLayer()
    lay.hidden, lay.inter, lay.n_experts, lay.topk = 2048, 512, 256, 8
    for f in ("router_w", "gu_codes", "gu_rin", "gu_rout", "dn_codes", "dn_rin", "dn_rout"):
        setattr(lay, f, g)
    lay.gu_K, lay.dn_K = 3, 2
    lay.sh_inter = 0
    need = L.escha_moe_block_workspace(ctypes.byref(lay), 1)
    assert need > 0
    assert L.escha_moe_block_workspace(ctypes.byref(lay), 64) > need
    call = lambda ws_bytes, **kw: L.escha_moe_block(ctypes.byref(lay), g, 1, g, None, None, g, ws_bytes, None)
    assert call(need - 1) == native.ESCHA_E_WORKSPACE
    lay.gu_K = 4
    assert call(need) == native.ESCHA_E_K
    lay.gu_K = 3
    lay.topk = 9
    assert call(need) == native.ESCHA_E_SHAPE
    lay.topk = 8
    lay.hidden = 2000
    assert call(need) == native.ESCHA_E_SHAPE
    lay.hidden = 2048
    lay.router_w = None
    assert call(need) == native.ESCHA_E_ARG
    lay.router_w = g
    lay.sh_inter = 512
    assert call(need) == native.ESCHA_E_ARG  # shared-expert pointers missing
    assert L.escha_moe_block(None, g, 1, g, None, None, g, need, None) == native.ESCHA_E_ARG
    # the residual call: its own arguments are checked before the block's
    lay.sh_inter = 0
    h, x, out = 0x100000, 0x200000, 0x300000  # [1][2048] f32 / fp16 / f32, apart
    resid = lambda h_, add_, eps_, x_, out_: L.escha_moe_block_resid(ctypes.byref(lay), h_, add_, eps_, x_, 1, out_,
                                                                        None, None, g, need, None)
    assert resid(None, None, 1e-6, x, out) == native.ESCHA_E_ARG
    assert resid(h, None, 1e-6, None, out) == native.ESCHA_E_ARG
    assert resid(h, None, -1.0, x, out) == native.ESCHA_E_ARG
    assert resid(h + 4, None, 1e-6, x, out) == native.ESCHA_E_ALIGN
    assert resid(h, h + 8192 + 4, 1e-6, x, out) == native.ESCHA_E_ALIGN  # add not 16-byte aligned
    assert resid(h, None, 1e-6, h + 4096, out) == native.ESCHA_E_ARG  # x inside h
    assert resid(h, None, 1e-6, x, x - 4096) == native.ESCHA_E_ARG  # out overlaps x
    assert resid(h, x - 8192 + 16, 1e-6, x, out) == native.ESCHA_E_ARG  # add's tail overlaps x
    assert L.escha_moe_block_resid(None, h, None, 1e-6, x, 1, out, None, None, g, need, None) == native.ESCHA_E_ARG
    # empty and oversized batches are rejected before anything is enqueued
    assert L.escha_moe_block(ctypes.byref(lay), g, 0, g, None, None, g, need, None) == native.ESCHA_E_ARG
    assert L.escha_moe_block(ctypes.byref(lay), g, 8193, g, None, None, g, 1 << 40, None) == native.ESCHA_E_SHAPE
    assert L.escha_moe_block_resid(ctypes.byref(lay), h, None, 1e-6, x, 0, out, None, None, g, need,
                                   None) == native.ESCHA_E_ARG
    assert L.escha_moe_block_noalloc(ctypes.byref(lay), g, 0, g, None, None, None) == native.ESCHA_E_ARG
    assert L.escha_moe_block_workspace(ctypes.byref(lay), 0) == 0
    assert L.escha_residual_rmsnorm(h, None, 0, 2048, 1e-6, x, None) == native.ESCHA_E_SHAPE
    assert L.escha_residual_rmsnorm(h, None, 1, 8193, 1e-6, x, None) == native.ESCHA_E_SHAPE


def test_product_path_has_no_oracle_import():
    pkg = os.path.join(ROOT, "bit_trellis_quantized_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in src.replace("the oracle", ""), f"{f} mentions the oracle"


def test_sequence_validation_before_launch():
    """escha_moe_blocks / escha_moe_stack reject their arguments on the host:
    block counts outside 1..48, null arrays, layers of different shapes,
    shapes the sequence kernel does not cover, a short workspace, aliasing
    stack buffers; the workspace query returns 0 for what it cannot size."""
    native, L = _lib()
    g = 0x10000

    def layer(hidden=2048, inter=512, sh_inter=0):
        lay = native.EschaMoeLayer()
        lay.hidden, lay.inter, lay.n_experts, lay.topk = hidden, inter, 256, 8
        for f in ("router_w", "gu_codes", "gu_rin", "gu_rout", "dn_codes", "dn_rin", "dn_rout"):
            setattr(lay, f, g)
        lay.gu_K, lay.dn_K = 3, 2
        lay.sh_inter = sh_inter
        return lay

    def arr(layers):
        return (ctypes.POINTER(native.EschaMoeLayer) * len(layers))(*[ctypes.pointer(x) for x in layers])

    vp = ctypes.c_void_p
    ptrs = lambda n, base: (vp * n)(*[base + 0x10000 * i for i in range(n)])
    two = [layer(), layer()]
    need = L.escha_moe_seq_workspace(arr(two), 2)
    assert need > 0
    assert L.escha_moe_seq_workspace(arr(two), 0) == 0
    assert L.escha_moe_seq_workspace(arr([layer()] * 49), 49) == 0
    assert L.escha_moe_seq_workspace(None, 2) == 0
    blocks = lambda layers, n, x, out, ws_bytes: L.escha_moe_blocks(
        arr(layers) if layers is not None else None, n, x, out, None, None, g, ws_bytes, None)
    x2, o2 = ptrs(2, 0x1000000), ptrs(2, 0x2000000)
    assert blocks(two, 0, x2, o2, need) == native.ESCHA_E_ARG
    assert blocks([layer()] * 49, 49, ptrs(49, 0x1000000), ptrs(49, 0x4000000), 1 << 40) == native.ESCHA_E_ARG
    assert blocks(None, 2, x2, o2, need) == native.ESCHA_E_ARG
    assert blocks(two, 2, None, o2, need) == native.ESCHA_E_ARG
    assert blocks(two, 2, x2, None, need) == native.ESCHA_E_ARG
    assert blocks([layer(), layer(inter=256)], 2, x2, o2, need) == native.ESCHA_E_SHAPE
    assert blocks([layer(hidden=4096), layer(hidden=4096)], 2, x2, o2, 1 << 40) == native.ESCHA_E_SHAPE
    assert blocks(two, 2, x2, o2, need - 1) == native.ESCHA_E_WORKSPACE
    stack = lambda layers, n, h, xb, ob, ws_bytes: L.escha_moe_stack(arr(layers), n, h, 1e-6, xb, ob, None, None, g,
                                                                   ws_bytes, None)
    h, xb, ob = 0x100000, 0x200000, 0x300000
    assert stack(two, 2, None, xb, ob, need) == native.ESCHA_E_ARG
    assert stack(two, 2, h, xb, h + 4096, need) == native.ESCHA_E_ARG  # out_buf inside h
    assert stack(two, 2, h + 4, xb, ob, need) == native.ESCHA_E_ALIGN
    assert stack(two, 0, h, xb, ob, need) == native.ESCHA_E_ARG
    assert L.escha_moe_stack(arr(two), 2, h, -1.0, xb, ob, None, None, g, need, None) == native.ESCHA_E_ARG
