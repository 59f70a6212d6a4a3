"""GPU parity of the residual stream between MoE blocks (f32 residual, fp16
input from a weightless RMSNorm) and of a stack of blocks, against the CPU
oracle, through the C ABI."""
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
    return n


@pytest.mark.parametrize("H", [2048, 768, 100, 8192])
def test_residual_rmsnorm_bit_exact(native, H):
    g = gen.rng(H)
    h = (g.standard_normal((37, H)) * g.uniform(0.01, 1e4, (37, 1))).astype(np.float32)
    add = (g.standard_normal((37, H)) * 30).astype(np.float32)
    hd = dev(h)
    x = native.residual_rmsnorm(hd, dev(add), eps=1e-6)
    ref_h, ref_x = o.residual_rmsnorm(h, add, eps=1e-6)
    assert np.array_equal(hd.cpu().numpy().view(np.uint32), ref_h.view(np.uint32))
    assert np.array_equal(x.cpu().numpy().view(np.uint16), ref_x)
    # without the add, and the add alone
    hd2 = dev(h)
    x2 = native.residual_rmsnorm(hd2, None, eps=1e-6)
    assert np.array_equal(x2.cpu().numpy().view(np.uint16), o.residual_rmsnorm(h, None, eps=1e-6)[1])
    native.residual_add(hd2, dev(add))
    assert np.array_equal(hd2.cpu().numpy().view(np.uint32), ref_h.view(np.uint32))


@pytest.mark.parametrize("T", [1, 2, 6])
def test_stack_small_each_block_against_oracle(native, T):
    """Three small blocks with mixed K: at every block, x is the oracle's norm
    of the GPU's h bit for bit, and the block output matches the oracle's
    block on that x (1 token: the norm inside the router grid; 2 and 6: the
    norm kernel)."""
    layers = [gen.moe_layer(80 + i, hidden=512, inter=256, n_experts=16, k_gu=k[0], k_dn=k[1])
              for i, k in enumerate([(3, 2), (2, 3), (2, 2)])]
    stack = native.MoeStack([native.MoeBlock(d, topk=4) for d in layers])
    x0 = gen.fp16_normal(gen.rng(90 + T), (T, 512))
    h = dev(x0.astype(np.float32))
    trace = []
    stack(h, trace=trace)
    for d, (h_before, x, out) in zip(layers, trace):
        _, ref_x = o.residual_rmsnorm(h_before.numpy(), None, eps=1e-6)
        assert np.array_equal(x.numpy().view(np.uint16), ref_x)
        ref, _, _, _ = o.moe_block(o.MoeLayer(**d), x.numpy(), k=4)
        assert rel_err_rows(out.numpy(), ref).max() <= TOL
    final = (trace[-1][0].numpy() + trace[-1][2].numpy()).astype(np.float32)
    assert np.array_equal(h.cpu().numpy().view(np.uint32), final.view(np.uint32))


@pytest.mark.parametrize("T", [1, 8, 128])
def test_stack_40_blocks_full_size(native, T):
    """The 40-block stack of full-size blocks (K per projection from seed
    5000 + layer) at decode batches 1, 8 and 128: finite, no bounded wait gave
    up, and block 17 (generated on the host) matches the oracle on the x it
    received (every token's norm; the outputs of sampled tokens)."""
    from escha_synth.gen_torch import moe_layer_device

    d17 = None
    blocks = []
    for l in range(40):
        kg, kd = gen.stack_k(l)
        if l == 17:
            d17 = gen.moe_layer(5000 + l, k_gu=kg, k_dn=kd)
            blocks.append(native.MoeBlock(d17))
        else:
            blocks.append(native.MoeBlock(moe_layer_device(5000 + l, torch.device("cuda"), k_gu=kg, k_dn=kd)))
    stack = native.MoeStack(blocks)
    x0 = gen.fp16_normal(gen.rng(91 + T), (T, 2048))
    h = dev(x0.astype(np.float32))
    x_buf = torch.empty((T, 2048), dtype=torch.float16, device="cuda")
    out_buf = torch.empty((T, 2048), dtype=torch.float32, device="cuda")
    trace = []
    stack(h, x_buf, out_buf, trace=trace)
    assert torch.isfinite(h).all()
    assert int(stack.workspace(T)[:4].view(torch.int32).item()) == 0
    h_before, x, out = trace[17]
    _, ref_x = o.residual_rmsnorm(h_before.numpy(), None, eps=1e-6)
    assert np.array_equal(x.numpy().view(np.uint16), ref_x)
    rows = list(range(T)) if T <= 8 else [0, 37, 64, 127]
    ref, _, _, _ = o.moe_block(o.MoeLayer(**d17), x.numpy()[rows], k=8)
    assert rel_err_rows(out.numpy()[rows], ref).max() <= TOL
    del blocks, stack
    torch.cuda.empty_cache()


def test_stack_prefill_chunk_2048_one_block(native):
    """A 2048-token prefill chunk through one full-size residual block (norm
    kernel, then the grouped tensor-core path): every token's x is the
    oracle's norm bit for bit, the outputs of sampled tokens match the
    oracle's block, and h ends as h + output."""
    kg, kd = gen.stack_k(0)
    d = gen.moe_layer(5000, k_gu=kg, k_dn=kd)
    stack = native.MoeStack([native.MoeBlock(d)])
    x0 = gen.fp16_normal(gen.rng(93), (2048, 2048)).astype(np.float32)
    h = dev(x0)
    trace = []
    stack(h, trace=trace)
    assert int(stack.workspace(2048)[:4].view(torch.int32).item()) == 0
    h_before, x, out = trace[0]
    _, ref_x = o.residual_rmsnorm(h_before.numpy(), None, eps=1e-6)
    assert np.array_equal(x.numpy().view(np.uint16), ref_x)
    rows = [0, 777, 1500, 2047]
    ref, _, _, _ = o.moe_block(o.MoeLayer(**d), x.numpy()[rows], k=8)
    assert rel_err_rows(out.numpy()[rows], ref).max() <= TOL
    final = (h_before.numpy() + out.numpy()).astype(np.float32)
    assert np.array_equal(h.cpu().numpy().view(np.uint32), final.view(np.uint32))


@pytest.mark.parametrize("T,H", [(1, 2048), (1, 768), (2, 2048), (2, 768), (1, 256), (3, 2048), (1, 4096), (20, 512)])
@pytest.mark.parametrize("with_add", [True, False])
def test_moe_block_resid_equals_norm_then_block(native, T, H, with_add):
    """escha_moe_block_resid against escha_residual_rmsnorm followed by
    escha_moe_block: h, x, outputs, ids and weights bit for bit, whether the
    norm runs inside the router grid (1 token, hidden <= 2048) or as its own
    kernel; the output written over the add buffer."""
    d = gen.moe_layer(300 + T + H, hidden=H, inter=128, n_experts=8, sh_inter=128)
    block = native.MoeBlock(d, topk=2)
    g = gen.rng(301 + T * H)
    h0 = (g.standard_normal((T, H)) * g.uniform(0.1, 10.0, (T, 1))).astype(np.float32)
    add0 = (g.standard_normal((T, H)) * 3).astype(np.float32)
    # reference: the two calls
    h_ref = dev(h0)
    x_ref = native.residual_rmsnorm(h_ref, dev(add0) if with_add else None, eps=1e-5)
    out_ref, ids_ref, w_ref = block(x_ref)
    # fused call, out over the add buffer
    h = dev(h0)
    add = dev(add0)
    x = torch.empty((T, H), dtype=torch.float16, device="cuda")
    out, ids, w = block.resid(h, add if with_add else None, x, eps=1e-5, out=add)
    torch.cuda.synchronize()
    assert torch.equal(h.view(torch.int32), h_ref.view(torch.int32))
    assert torch.equal(x.view(torch.int16), x_ref.view(torch.int16))
    assert torch.equal(ids, ids_ref)
    assert torch.equal(w.view(torch.int32), w_ref.view(torch.int32))
    assert torch.equal(out.view(torch.int32), out_ref.view(torch.int32))
    assert int(block.workspace(T)[:4].view(torch.int32).item()) == 0
