"""GPU check of escha_moe_block_noalloc, the MoE-block entry point that takes
no workspace.

Some callers cannot allocate device memory while they run the block: an
operator plugin inside a framework that owns every device allocation, code
that issues work while a stream is captured into a CUDA graph in a mode that
forbids cudaMalloc, or a process whose memory is fixed at start-up. For them
the library keeps the block's scratch in a device buffer compiled into the
library. Its results must match escha_moe_block (the entry point with a
caller workspace) and stay right on the next call, which reuses the buffer.
"""
import ctypes

import numpy as np
import pytest

from escha_synth import gen
from gpu_common import TOL, dev, rel_err_rows

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_trellis_quantized_gb300 import native

    L = native.lib()
    d = gen.moe_layer(31, hidden=2048, inter=512, n_experts=64, k_gu=3, k_dn=2)
    block = native.MoeBlock(d, topk=8)
    T = 3
    for seed in (41, 42):  # two calls in a row through the built-in buffer
        x = dev(gen.fp16_normal(gen.rng(seed), (T, 2048)))
        ref_out, ref_ids, ref_w = block(x)  # escha_moe_block with a caller workspace
        out = torch.full_like(ref_out, float("nan"))
        ids = torch.full_like(ref_ids, -1)
        w = torch.full_like(ref_w, float("nan"))
        rc = L.escha_moe_block_noalloc(ctypes.byref(block.layer), native.ptr(x), T, native.ptr(out), native.ptr(ids),
                                       native.ptr(w), native.stream_handle())
        assert rc == native.ESCHA_OK, L.escha_last_error()
        torch.cuda.synchronize()
        assert torch.equal(ids, ref_ids)
        assert np.allclose(w.cpu().numpy(), ref_w.cpu().numpy(), rtol=1e-6, atol=0)
        err = rel_err_rows(out.cpu().numpy(), ref_out.cpu().numpy().astype(np.float64))
        assert err.max() <= TOL, err


def test_noalloc_rejects_work_beyond_the_buffer():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_trellis_quantized_gb300 import native

    L = native.lib()
    d = gen.moe_layer(32, hidden=2048, inter=512, n_experts=16)
    block = native.MoeBlock(d, topk=8)
    x = dev(gen.fp16_normal(gen.rng(1), (1, 2048)))
    out = torch.empty((1, 2048), dtype=torch.float32, device="cuda")
    need = L.escha_moe_block_workspace(ctypes.byref(block.layer), 4096)
    assert need > (2 << 20)
    # T = 4096 would need more scratch than the buffer holds: refused before
    # anything is enqueued (so the too-short x and out are never touched)
    rc = L.escha_moe_block_noalloc(ctypes.byref(block.layer), native.ptr(x), 4096, native.ptr(out), None, None,
                                   native.stream_handle())
    assert rc == native.ESCHA_E_WORKSPACE
    assert b"built-in buffer" in L.escha_last_error()
    torch.cuda.synchronize()
