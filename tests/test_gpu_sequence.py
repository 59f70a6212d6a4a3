"""A sequence of one-token MoE blocks in one cooperative launch (independent
blocks, and the residual stack of a decode step) against the same blocks run
one call at a time (bit for bit) and against the oracle, through the C ABI;
the sequence kernel's bounded waits made to run out on purpose; and its
argument checks."""
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
    """These tests run the sequence kernel: escha_moe_blocks is held on it
    (independent blocks of up to 16 would otherwise take the per-slot
    kernels, tested in test_gpu_blocks.py)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_trellis_quantized_gb300 import native as n

    n.lib()
    n.set_blocks_route(2)
    yield n
    n.set_blocks_route(0)
    n.set_fused_wait()


def _status(ws):
    return int(ws[:4].view(torch.int32).item())


def _per_block(blocks, xs):
    outs, ids, ws = [], [], []
    for b, x in zip(blocks, xs):
        o_, i_, w_ = b(x.view(1, -1))
        outs.append(o_.clone())
        ids.append(i_.clone())
        ws.append(w_.clone())
    torch.cuda.synchronize()
    return outs, ids, ws


def _sequence(native, blocks, xs):
    n = len(blocks)
    topk = blocks[0].topk
    outs = [torch.empty(blocks[0].hidden, dtype=torch.float32, device="cuda") for _ in range(n)]
    ids = [torch.empty(topk, dtype=torch.int32, device="cuda") for _ in range(n)]
    w = [torch.empty(topk, dtype=torch.float32, device="cuda") for _ in range(n)]
    ws = torch.empty(native.seq_workspace_bytes(blocks), dtype=torch.uint8, device="cuda")
    native.moe_blocks(blocks, xs, outs, ids=ids, w=w, ws=ws)
    torch.cuda.synchronize()
    return outs, ids, w, _status(ws)


# (hidden, inter, experts, topk, shared inter, [(K gate_up, K down) per block])
SMALL = [
    (512, 256, 16, 4, 256, [(3, 2), (2, 3), (2, 2), (3, 3), (3, 2)]),
    (256, 128, 8, 2, 0, [(2, 2), (3, 3), (2, 3)]),
    (768, 384, 24, 8, 384, [(2, 3), (3, 2)]),
    (1024, 128, 64, 1, 16, [(2, 2)]),
]


@pytest.mark.parametrize("cfg", SMALL, ids=[f"h{c[0]}_i{c[1]}_e{c[2]}_k{c[3]}_sh{c[4]}_n{len(c[5])}" for c in SMALL])
def test_blocks_bit_identical_to_per_block_calls(native, cfg):
    hidden, inter, E, topk, sh, ks = cfg
    layers = []
    for i, (kg, kd) in enumerate(ks):
        d = gen.moe_layer(400 + 10 * i + hidden, hidden=hidden, inter=inter, n_experts=E, k_gu=kg, k_dn=kd,
                          sh_inter=max(sh, 16))
        if sh == 0:
            d["sh_inter"] = 0
        layers.append(d)
    blocks = [native.MoeBlock(d, topk=topk) for d in layers]
    xs_np = [gen.fp16_normal(gen.rng(500 + i), (hidden,)) for i in range(len(blocks))]
    xs = [dev(x) for x in xs_np]
    ref_out, ref_ids, ref_w = _per_block(blocks, xs)
    out, ids, w, status = _sequence(native, blocks, xs)
    assert status == 0
    for i in range(len(blocks)):
        assert torch.equal(ids[i], ref_ids[i][0])
        assert torch.equal(w[i], ref_w[i][0])
        assert torch.equal(out[i], ref_out[i][0]), (i, float((out[i] - ref_out[i][0]).abs().max()))
    # the last block against the oracle
    d = layers[-1]
    layer = o.MoeLayer(**d)
    x1 = xs_np[-1][None]
    ref, r_ids, r_w, _ = o.moe_block(layer, x1, k=topk)
    if sh == 0:
        xv = o.f16_to_f64(x1.view(np.uint16))[0]
        ref = sum(r_w[0, j] * o.moe_expert(layer, r_ids[0, j], xv) for j in range(topk))[None]
    assert np.array_equal(ids[-1].cpu().numpy(), r_ids[0])
    assert rel_err_rows(out[-1].cpu().numpy()[None], ref).max() <= TOL


def test_blocks_full_size_bit_identical(native):
    """Eight Qwen3.6-35B-A3B-shaped blocks (hidden 2048, 256 experts, top-8,
    gate_up K=3, down K=2, int8 shared expert), each on its own token."""
    from escha_synth.gen_torch import moe_layer_device

    blocks = [native.MoeBlock(moe_layer_device(1002 + l, torch.device("cuda")), topk=8) for l in range(8)]
    xs = [dev(gen.fp16_normal(gen.rng(2002 + l), (2048,))) for l in range(8)]
    ref_out, ref_ids, ref_w = _per_block(blocks, xs)
    for rep in range(2):  # the counters are re-zeroed by every launch
        out, ids, w, status = _sequence(native, blocks, xs)
        assert status == 0
        for i in range(8):
            assert torch.equal(ids[i], ref_ids[i][0])
            assert torch.equal(out[i], ref_out[i][0])
    del blocks
    torch.cuda.empty_cache()


def _stack_layers(n, hidden=512, inter=256, E=16, sh=128):
    return [gen.moe_layer(600 + l, hidden=hidden, inter=inter, n_experts=E, k_gu=2 + l % 2, k_dn=2 + (l // 2) % 2,
                          sh_inter=sh) for l in range(n)]


@pytest.mark.parametrize("n", [1, 2, 5])
def test_stack_bit_identical_to_block_by_block(native, n):
    """A residual stack in one launch gives the h, x and output of the blocks
    run one call at a time (escha_moe_block_resid, then the final add)."""
    blocks = [native.MoeBlock(d, topk=4) for d in _stack_layers(n)]
    stack = native.MoeStack(blocks)
    h0 = torch.randn((1, 512), device="cuda", generator=torch.Generator(device="cuda").manual_seed(n)) * 4
    res = []
    for seq in (False, True):
        h = h0.clone()
        x = torch.empty((1, 512), dtype=torch.float16, device="cuda")
        out = torch.empty((1, 512), dtype=torch.float32, device="cuda")
        stack(h, x, out, sequence=seq)
        torch.cuda.synchronize()
        res.append((h, x, out))
    assert _status(stack._seq_ws) == 0
    for a, b in zip(res[0], res[1]):
        assert torch.equal(a, b)


def test_stack_one_block_against_oracle(native):
    """One residual block in one launch: x is the oracle's norm of h (bit for
    bit), the output matches the oracle's block on that x, and h ends as h +
    output (one f32 add)."""
    layers = _stack_layers(1)
    blocks = [native.MoeBlock(d, topk=4) for d in layers]
    h0 = gen.fp16_normal(gen.rng(77), (1, 512)).astype(np.float32) * 3
    h = dev(h0)
    x = torch.empty((1, 512), dtype=torch.float16, device="cuda")
    out = torch.empty((1, 512), dtype=torch.float32, device="cuda")
    native.MoeStack(blocks)(h, x, out, sequence=True)
    torch.cuda.synchronize()
    _, ref_x = o.residual_rmsnorm(h0, None, eps=1e-6)
    assert np.array_equal(x.cpu().numpy().view(np.uint16), ref_x)
    ref, _, _, _ = o.moe_block(o.MoeLayer(**layers[0]), x.cpu().numpy(), k=4)
    assert rel_err_rows(out.cpu().numpy(), ref).max() <= TOL
    want = (h0 + out.cpu().numpy()).astype(np.float32)
    assert np.array_equal(h.cpu().numpy().view(np.uint32), want.view(np.uint32))


def test_stack_40_blocks_full_size_bit_identical(native):
    """The 40-block stack of full-size blocks (K per projection from seed 5000
    + layer) in one launch against block by block: the same h bits."""
    from escha_synth.gen_torch import moe_layer_device

    blocks = []
    for l in range(40):
        kg, kd = gen.stack_k(l)
        blocks.append(native.MoeBlock(moe_layer_device(5000 + l, torch.device("cuda"), k_gu=kg, k_dn=kd)))
    stack = native.MoeStack(blocks)
    assert stack.sequence_ok()
    h0 = dev(gen.fp16_normal(gen.rng(92), (1, 2048)).astype(np.float32))
    hs = []
    for seq in (False, True):
        h = h0.clone()
        stack(h, sequence=seq)
        torch.cuda.synchronize()
        hs.append(h)
    assert _status(stack._seq_ws) == 0
    assert torch.isfinite(hs[1]).all()
    assert torch.equal(hs[0], hs[1])
    del blocks, stack
    torch.cuda.empty_cache()


def test_sequence_bounded_wait_runs_out(native):
    """With every expert's gate_up outputs kept unpublished and a 2 ms bound,
    the down units give up, and so do the combine units that wait for them:
    the launch ends and the status word names the first wait that ran out
    (10 = a down unit's wait for its expert's gate_up outputs, 14 = a combine
    unit's wait for the down partial sums; which comes first depends on when
    each unit was taken); the next launch with the default settings is
    correct again."""
    blocks = [native.MoeBlock(d, topk=4) for d in _stack_layers(2)]
    xs = [dev(gen.fp16_normal(gen.rng(700 + i), (512,))) for i in range(2)]
    ref_out, _, _ = _per_block(blocks, xs)
    native.set_fused_wait(2_000_000, skip_publish=True)
    try:
        t0 = time.time()
        _, _, _, status = _sequence(native, blocks, xs)
        dt = time.time() - t0
    finally:
        native.set_fused_wait()
    assert status in (10, 14), status
    assert dt < 10.0
    out, _, _, status = _sequence(native, blocks, xs)
    assert status == 0
    for i in range(2):
        assert torch.equal(out[i], ref_out[i][0])


def test_sequence_argument_checks(native):
    small = [native.MoeBlock(d, topk=4) for d in _stack_layers(2)]
    other = native.MoeBlock(gen.moe_layer(801, hidden=512, inter=128, n_experts=16, sh_inter=128), topk=4)
    xs = [torch.zeros(512, dtype=torch.float16, device="cuda") for _ in range(2)]
    outs = [torch.empty(512, device="cuda") for _ in range(2)]
    ws = torch.empty(1 << 24, dtype=torch.uint8, device="cuda")
    with pytest.raises(native.EschaError) as ei:  # different inter
        native.moe_blocks([small[0], other], xs, outs, ws=ws)
    assert ei.value.code == native.ESCHA_E_SHAPE
    with pytest.raises(native.EschaError) as ei:  # too many blocks
        native.moe_blocks([small[0]] * 49, (xs * 25)[:49], (outs * 25)[:49], ws=ws)
    assert ei.value.code == native.ESCHA_E_ARG
    big = native.MoeBlock(gen.moe_layer(802, hidden=4096, inter=128, n_experts=8, sh_inter=64), topk=2)
    with pytest.raises(native.EschaError) as ei:  # hidden above the sequence kernel's 2048
        native.moe_blocks([big], [torch.zeros(4096, dtype=torch.float16, device="cuda")],
                          [torch.empty(4096, device="cuda")], ws=ws)
    assert ei.value.code == native.ESCHA_E_SHAPE
    with pytest.raises(native.EschaError) as ei:  # workspace too small
        native.moe_blocks(small, xs, outs, ws=ws[:1024])
    assert ei.value.code == native.ESCHA_E_WORKSPACE
