"""Independent one-token blocks on the per-slot kernels (escha_moe_blocks,
ESCHA_PATH_SLOT): one launch each of the router, gate_up and down/combine
kernels over every block's slots, token t with layer t. Checked bit for bit
against escha_moe_block over n tokens of one layer (n copies of that layer),
against one-token calls for a single block, against the sequence kernel and
the oracle within the block's tolerance for distinct layers, and for the
route's choice and argument checks."""
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
    n.set_blocks_route(0)
    yield n
    n.set_blocks_route(0)


def _run(native, blocks, xs, route=0):
    n = len(blocks)
    topk = blocks[0].topk
    outs = [torch.full((blocks[0].hidden,), float("nan"), device="cuda") for _ in range(n)]
    ids = [torch.full((topk,), -1, dtype=torch.int32, device="cuda") for _ in range(n)]
    w = [torch.empty(topk, device="cuda") for _ in range(n)]
    ws = torch.empty(native.seq_workspace_bytes(blocks), dtype=torch.uint8, device="cuda")
    native.set_blocks_route(route)
    try:
        native.moe_blocks(blocks, xs, outs, ids=ids, w=w, ws=ws)
        torch.cuda.synchronize()
    finally:
        native.set_blocks_route(0)
    assert int(ws[:4].view(torch.int32).item()) == 0
    return outs, ids, w


@pytest.mark.parametrize("n", [2, 5, 8, 16])
def test_copies_of_one_layer_equal_a_multi_token_call(native, n):
    """n copies of one layer on n tokens give escha_moe_block's n-token
    outputs, ids and weights bit for bit (same kernels, same splits)."""
    d = gen.moe_layer(1002)
    block = native.MoeBlock(d, topk=8)
    xs = dev(gen.fp16_normal(gen.rng(3100 + n), (n, 2048)))
    ref_out, ref_ids, ref_w = block(xs)
    torch.cuda.synchronize()
    blocks = [block] * n
    assert native.blocks_path(blocks) == native.ESCHA_PATH_SLOT
    out, ids, w = _run(native, blocks, [xs[i] for i in range(n)])
    for i in range(n):
        assert torch.equal(ids[i], ref_ids[i])
        assert torch.equal(w[i], ref_w[i])
        assert torch.equal(out[i], ref_out[i]), (i, float((out[i] - ref_out[i]).abs().max()))


def test_one_block_equals_a_one_token_call(native):
    d = gen.moe_layer(1003)
    block = native.MoeBlock(d, topk=8)
    x = dev(gen.fp16_normal(gen.rng(3200), (1, 2048)))
    ref, ref_ids, ref_w = block(x)
    out, ids, w = _run(native, [block], [x[0]], route=1)
    assert torch.equal(out[0], ref[0]) and torch.equal(ids[0], ref_ids[0]) and torch.equal(w[0], ref_w[0])


def test_distinct_full_size_layers_match_the_sequence_kernel(native):
    """Eight distinct Qwen3.6-35B-A3B-shaped layers: the routing equals the
    sequence kernel's bit for bit (the logits do not depend on the splits)
    and the outputs agree within the block's tolerance."""
    from escha_synth.gen_torch import moe_layer_device

    blocks = [native.MoeBlock(moe_layer_device(1002 + l, torch.device("cuda")), topk=8) for l in range(8)]
    xs = [dev(gen.fp16_normal(gen.rng(2002 + l), (2048,))) for l in range(8)]
    assert native.blocks_path(blocks) == native.ESCHA_PATH_SLOT
    o1, i1, w1 = _run(native, blocks, xs, route=1)
    o2, i2, w2 = _run(native, blocks, xs, route=2)
    for i in range(8):
        assert torch.equal(i1[i], i2[i])
        assert torch.equal(w1[i], w2[i])
        err = rel_err_rows(o1[i].cpu().numpy()[None], o2[i].cpu().numpy()[None]).max()
        assert err <= 1e-5, (i, err)
    del blocks
    torch.cuda.empty_cache()


def test_distinct_small_layers_against_the_oracle(native):
    """Distinct small layers (K per block, top-4, a shared expert) against the
    oracle's block on each token."""
    layers = [gen.moe_layer(3300 + i, hidden=512, inter=256, n_experts=16, k_gu=3, k_dn=2, sh_inter=256)
              for i in range(6)]
    blocks = [native.MoeBlock(d, topk=4) for d in layers]
    xs_np = [gen.fp16_normal(gen.rng(3400 + i), (512,)) for i in range(6)]
    out, ids, w = _run(native, blocks, [dev(x) for x in xs_np], route=1)
    for i, d in enumerate(layers):
        ref, r_ids, r_w, _ = o.moe_block(o.MoeLayer(**d), xs_np[i][None], k=4)
        assert np.array_equal(ids[i].cpu().numpy(), r_ids[0])
        assert np.allclose(w[i].cpu().numpy(), r_w[0], rtol=1e-5, atol=1e-6)
        assert rel_err_rows(out[i].cpu().numpy()[None], ref).max() <= TOL


# (hidden, inter, experts, topk, shared inter (0: none), K gate_up, K down, blocks)
SHAPES = [
    (256, 128, 8, 2, 0, 2, 2, 3),
    (768, 384, 24, 8, 384, 2, 3, 2),
    (1024, 128, 64, 1, 16, 3, 3, 4),
    (512, 256, 16, 4, 256, 3, 2, 16),
]


@pytest.mark.parametrize("cfg", SHAPES, ids=[f"h{c[0]}_i{c[1]}_e{c[2]}_k{c[3]}_sh{c[4]}_K{c[5]}{c[6]}_n{c[7]}"
                                             for c in SHAPES])
def test_distinct_layer_shapes(native, cfg):
    """Distinct layers of other shapes (no shared expert, top-1 / 2 / 8, K = 2
    or 3 on either projection, 16 blocks): routing bit-exact against the
    oracle and the sequence kernel, outputs within the tolerance of the
    oracle and within 1e-5 of the sequence kernel (whose input splits
    differ)."""
    hidden, inter, E, topk, sh, kg, kd, n = cfg
    layers = []
    for i in range(n):
        d = gen.moe_layer(3600 + 10 * i + hidden, hidden=hidden, inter=inter, n_experts=E, k_gu=kg, k_dn=kd,
                          sh_inter=max(sh, 16))
        if sh == 0:
            d["sh_inter"] = 0
        layers.append(d)
    blocks = [native.MoeBlock(d, topk=topk) for d in layers]
    assert native.blocks_path(blocks) == native.ESCHA_PATH_SLOT
    xs_np = [gen.fp16_normal(gen.rng(3700 + i), (hidden,)) for i in range(n)]
    xs = [dev(x) for x in xs_np]
    out, ids, w = _run(native, blocks, xs, route=1)
    s_out, s_ids, s_w = _run(native, blocks, xs, route=2)
    for i, d in enumerate(layers):
        assert torch.equal(ids[i], s_ids[i])
        assert torch.equal(w[i], s_w[i])
        err = float((out[i] - s_out[i]).abs().max() / s_out[i].abs().max())
        assert err <= 1e-5, (i, err)
        layer = o.MoeLayer(**d)
        x1 = xs_np[i][None]
        ref, r_ids, r_w, _ = o.moe_block(layer, x1, k=topk)
        if sh == 0:
            xv = o.f16_to_f64(x1.view(np.uint16))[0]
            ref = sum(r_w[0, j] * o.moe_expert(layer, r_ids[0, j], xv) for j in range(topk))[None]
        assert np.array_equal(ids[i].cpu().numpy(), r_ids[0])
        assert np.allclose(w[i].cpu().numpy(), r_w[0], rtol=1e-5, atol=1e-6)
        assert rel_err_rows(out[i].cpu().numpy()[None], ref).max() <= TOL


def test_route_choice(native):
    """Mixed K pairs, or more than 16 blocks, take the sequence kernel; forcing
    the per-slot route on them is an error before anything is enqueued."""
    a = native.MoeBlock(gen.moe_layer(3500, hidden=512, inter=256, n_experts=16, k_gu=3, k_dn=2, sh_inter=128), topk=4)
    b = native.MoeBlock(gen.moe_layer(3501, hidden=512, inter=256, n_experts=16, k_gu=2, k_dn=2, sh_inter=128), topk=4)
    assert native.blocks_path([a, a]) == native.ESCHA_PATH_SLOT
    assert native.blocks_path([a, b]) == native.ESCHA_PATH_SEQUENCE
    assert native.blocks_path([a] * 17) == native.ESCHA_PATH_SEQUENCE
    native.set_blocks_route(1)
    try:
        with pytest.raises(native.EschaError) as ei:
            native.blocks_path([a, b])
        assert ei.value.code == native.ESCHA_E_SHAPE
        xs = [torch.zeros(512, dtype=torch.float16, device="cuda")] * 2
        outs = [torch.empty(512, device="cuda") for _ in range(2)]
        with pytest.raises(native.EschaError) as ei:
            native.moe_blocks([a, b], xs, outs)
        assert ei.value.code == native.ESCHA_E_SHAPE
    finally:
        native.set_blocks_route(0)
    native.set_blocks_route(2)
    try:
        assert native.blocks_path([a, a]) == native.ESCHA_PATH_SEQUENCE
    finally:
        native.set_blocks_route(0)
    with pytest.raises(native.EschaError):
        native.set_blocks_route(3)
