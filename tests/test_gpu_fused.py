"""The one-token fused path (the router kernel, then one cooperative grid for
top-k, gate_up, down, the shared expert's down rows and the combine) against
the three per-slot kernels (bit for bit) and against the oracle, through the
C ABI; and its bounded waits, made to run out on purpose through the
diagnostic hook that keeps the gate_up outputs unpublished (no fault, no
hang: the kernel ends and reports it)."""
import time

import numpy as np
import pytest

from escha_synth import gen
from gpu_common import TOL, dev, rel_err_rows
from oracle import escha_oracle as o

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def native():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_trellis_quantized_gb300 import native as n

    n.lib()
    yield n
    n.set_moe_route(0)
    n.set_fused_wait()


# (seed, hidden, inter, experts, topk, K gate_up, K down, shared inter)
LAYERS = [
    (1002, 2048, 512, 256, 8, 3, 2, 512),  # the Qwen3.6-35B-A3B-shaped layer
    (31, 256, 128, 8, 2, 2, 2, 0),  # no shared expert
    (32, 768, 384, 24, 8, 2, 3, 384),  # the pages' K pairing, 6 hidden blocks, odd inter blocks
    (33, 512, 256, 16, 4, 3, 3, 256),
    (34, 1024, 128, 64, 1, 2, 2, 16),  # top-1, a 16-wide shared expert
    (35, 256, 256, 8, 8, 3, 2, 128),  # top-k = every expert
]


def _layer(seed, hidden, inter, E, topk, kg, kd, sh):
    d = gen.moe_layer(seed, hidden=hidden, inter=inter, n_experts=E, k_gu=kg, k_dn=kd, sh_inter=max(sh, 16))
    if sh == 0:
        d["sh_inter"] = 0
    return d


def _run(native, block, x, mode):
    native.set_moe_route(mode)
    try:
        out, ids, w = block(x)
        torch.cuda.synchronize()
        status = int(block.workspace(1)[:4].view(torch.int32).item())
    finally:
        native.set_moe_route(0)
    return out.clone(), ids.clone(), w.clone(), status


@pytest.mark.parametrize("cfg", LAYERS, ids=[f"h{c[1]}_i{c[2]}_e{c[3]}_k{c[4]}_K{c[5]}{c[6]}_sh{c[7]}" for c in LAYERS])
def test_fused_bit_identical_to_per_slot_kernels(native, cfg):
    seed, hidden, inter, E, topk, kg, kd, sh = cfg
    d = _layer(*cfg)
    block = native.MoeBlock(d, topk=topk)
    x = gen.fp16_normal(gen.rng(seed + 100), (1, hidden))
    xd = dev(x)
    o1, i1, w1, s1 = _run(native, block, xd, 1)
    o2, i2, w2, s2 = _run(native, block, xd, 2)
    assert s1 == 0 and s2 == 0, (s1, s2)
    assert torch.equal(i1, i2)
    assert torch.equal(w1, w2)
    assert torch.equal(o1, o2), float((o1 - o2).abs().max())
    # and against the oracle (the routed sum alone when there is no shared expert)
    layer = o.MoeLayer(**d)
    ref, ref_ids, ref_w, _ = o.moe_block(layer, x, k=topk)
    if sh == 0:
        xv = o.f16_to_f64(x.view(np.uint16))[0]
        ref = sum(ref_w[0, j] * o.moe_expert(layer, ref_ids[0, j], xv) for j in range(topk))[None]
    assert np.array_equal(i2.cpu().numpy(), ref_ids)
    assert np.allclose(w2.cpu().numpy(), ref_w, rtol=1e-5, atol=1e-6)
    assert rel_err_rows(o2.cpu().numpy(), ref).max() <= TOL


def test_fused_repeatable_and_default_route(native):
    """The default route at one token (the per-slot kernels) agrees with the
    fused one bit for bit, and repeated fused calls on one workspace give the
    same bits (the counters are re-zeroed by every call)."""
    d = gen.moe_layer(1002)
    block = native.MoeBlock(d, topk=8)
    xs = dev(gen.fp16_normal(gen.rng(777), (3, 2048)))
    first = [_run(native, block, xs[t:t + 1], 2)[0] for t in range(3)]
    assert block.path(1) == native.ESCHA_PATH_SLOT
    for t in range(3):
        out, _, _ = block(xs[t:t + 1])
        assert torch.equal(out, first[t])
    for t in (2, 0, 1):
        assert torch.equal(_run(native, block, xs[t:t + 1], 2)[0], first[t])


@pytest.mark.parametrize("with_add", [False, True])
def test_fused_residual_block_bit_identical(native, with_add):
    """escha_moe_block_resid at one token: h, x, the output and the routing
    are the same bits on both routes, with and without the previous block's
    output added (the output written over that same buffer)."""
    d = gen.moe_layer(1003)
    block = native.MoeBlock(d, topk=8)
    g = torch.Generator(device="cuda").manual_seed(5)
    h0 = torch.randn((1, 2048), device="cuda", generator=g) * 3
    add0 = torch.randn((1, 2048), device="cuda", generator=g) * 50
    res = []
    for mode in (1, 2):
        h = h0.clone()
        add = add0.clone()
        x = torch.empty((1, 2048), dtype=torch.float16, device="cuda")
        native.set_moe_route(mode)
        try:
            out, ids, w = block.resid(h, add if with_add else None, x, out=add if with_add else None)
            torch.cuda.synchronize()
        finally:
            native.set_moe_route(0)
        assert int(block.workspace(1)[:4].view(torch.int32).item()) == 0
        res.append([h, x, out.clone(), ids.clone(), w.clone()])
    for a, b in zip(res[0], res[1]):
        assert torch.equal(a, b)
    # h really took the add, and x is the oracle's norm of it
    want_h = (h0 + add0) if with_add else h0
    assert torch.equal(res[1][0], want_h)
    _, xref = o.residual_rmsnorm(want_h.cpu().numpy(), eps=1e-6)
    assert np.array_equal(res[1][1].cpu().numpy().view(np.uint16), xref)


def test_fused_stack_bit_identical(native):
    """Three residual blocks at one token: the h after the stack is the same
    on both routes."""
    blocks = []
    for l in range(3):
        kg, kd = gen.stack_k(l)
        blocks.append(native.MoeBlock(gen.moe_layer(5000 + l, k_gu=kg, k_dn=kd), topk=8))
    stack = native.MoeStack(blocks)
    h0 = torch.randn((1, 2048), device="cuda", generator=torch.Generator(device="cuda").manual_seed(9))
    hs = []
    for mode in (1, 2):
        native.set_moe_route(mode)
        try:
            h = h0.clone()
            stack(h)
            torch.cuda.synchronize()
        finally:
            native.set_moe_route(0)
        hs.append(h)
    assert torch.equal(hs[0], hs[1])


def test_fused_bounded_wait_runs_out(native):
    """With the gate_up outputs kept unpublished and a 2 ms bound, every down
    unit gives up waiting for them: the kernel ends, the status word reports
    it (5 = the wait for an expert's gate_up outputs), and the context stays
    usable: the next call with the default settings is correct."""
    d = gen.moe_layer(1002)
    block = native.MoeBlock(d, topk=8)
    x = dev(gen.fp16_normal(gen.rng(2002), (1, 2048)))
    ref, _, _, s = _run(native, block, x, 1)
    assert s == 0
    native.set_moe_route(2)
    native.set_fused_wait(2_000_000, skip_publish=True)
    try:
        t0 = time.time()
        block(x)
        torch.cuda.synchronize()
        dt = time.time() - t0
        status = int(block.workspace(1)[:4].view(torch.int32).item())
    finally:
        native.set_fused_wait()
        native.set_moe_route(0)
    assert status == 5, status
    assert dt < 5.0
    out, _, _, s = _run(native, block, x, 2)
    assert s == 0
    assert torch.equal(out, ref)


def test_fused_route_rejects_uncovered_layers(native):
    """Forcing the fused kernel on a layer it does not cover (hidden 4096) is
    an ESCHA_E_SHAPE error before anything is enqueued; the default route
    then takes the per-slot kernels."""
    d = gen.moe_layer(36, hidden=4096, inter=128, n_experts=8, sh_inter=64)
    block = native.MoeBlock(d, topk=2)
    x = dev(gen.fp16_normal(gen.rng(37), (1, 4096)))
    native.set_moe_route(2)
    try:
        with pytest.raises(native.EschaError) as ei:
            block(x)
        assert ei.value.code == native.ESCHA_E_SHAPE
    finally:
        native.set_moe_route(0)
    out, ids, w = block(x)
    ref, ref_ids, _, _ = o.moe_block(o.MoeLayer(**d), gen.fp16_normal(gen.rng(37), (1, 4096)), k=2)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    assert rel_err_rows(out.cpu().numpy(), ref).max() <= TOL
