"""GPU parity of the router and the whole MoE block against the CPU oracle,
called through the C ABI."""
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


def _check_block(native, d, x, topk, tokens=None):
    block = native.MoeBlock(d, topk=topk)
    out, ids, w = block(dev(x))
    out = out.cpu().numpy()
    ids = ids.cpu().numpy()
    w = w.cpu().numpy()
    layer = o.MoeLayer(**d)
    ref, ref_ids, ref_w, _ = o.moe_block(layer, x, k=topk, tokens=tokens)
    assert np.array_equal(ids, ref_ids), "routing ids must match bit for bit"
    assert np.allclose(w, ref_w, rtol=1e-5, atol=1e-6)
    rows = slice(None) if tokens is None else list(tokens)
    err = rel_err_rows(out[rows], ref)
    status = int(block.workspace(x.shape[0])[:4].view(torch.int32).item())
    assert status == 0, "a bounded wait gave up"
    assert err.max() <= TOL, err
    return out, ids, w


def test_moe_block_small(native):
    d = gen.moe_layer(11, hidden=512, inter=256, n_experts=16, k_gu=3, k_dn=2)
    x = gen.fp16_normal(gen.rng(12), (3, 512))
    _check_block(native, d, x, topk=4)


def test_moe_block_pages_k_pairing_and_ragged(native):
    """gate_up K=2 / down K=3 (the pairing the checkpoint's layer_meta
    records), hidden 768 (6 blocks), inter 384, 5 tokens."""
    d = gen.moe_layer(13, hidden=768, inter=384, n_experts=24, k_gu=2, k_dn=3)
    x = gen.fp16_normal(gen.rng(14), (5, 768))
    _check_block(native, d, x, topk=8)


@pytest.mark.parametrize("T", [2, 40])
def test_moe_block_no_shared_expert(native, T):
    """No shared expert (sh_inter = 0): the per-slot path (2 tokens) and the
    grouped path (40 tokens) give the routed sum alone."""
    d = gen.moe_layer(15, hidden=256, inter=128, n_experts=8, sh_inter=0)
    d["sh_inter"] = 0
    x = gen.fp16_normal(gen.rng(16), (T, 256))
    block = native.MoeBlock(d, topk=2)
    out, ids, w = block(dev(x))
    layer = o.MoeLayer(**d)
    xv = o.f16_to_f64(x.view(np.uint16))
    ref_ids, ref_w, _ = o.route(x, d["Wg"], 2)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    for b in range(0, T, max(1, T // 8)):
        want = sum(ref_w[b, j] * o.moe_expert(layer, ref_ids[b, j], xv[b]) for j in range(2))
        assert rel_err_rows(out.cpu().numpy()[b:b + 1], want[None]).max() <= TOL


def test_moe_block_full_size_batch1(native):
    """One full Qwen3.6-35B-A3B-shaped block at decode batch 1: hidden 2048,
    256 experts, top-8, gate_up K=3, down K=2, int8 shared expert."""
    d = gen.moe_layer(1002)
    x = gen.fp16_normal(gen.rng(2002), (1, 2048))
    out, ids, w = _check_block(native, d, x, topk=8)
    assert len(set(ids[0])) == 8


@pytest.mark.parametrize("T", [4, 12, 16])
def test_moe_block_per_slot_path_full_size(native, T):
    """Full-size block on the per-slot path: 4 tokens (gate_up inputs split
    over two CTAs in 1.3 waves), 12, and 16 tokens, the largest batch of the
    path (128 slots, the fused shared expert in four passes of 4 tokens)."""
    d = gen.moe_layer(1005)
    x = gen.fp16_normal(gen.rng(2006 + T), (T, 2048))
    _check_block(native, d, x, topk=8, tokens=[0, T // 2, T - 1])


def test_router_ids_bit_exact_many_tokens(native):
    d = gen.moe_layer(1003, hidden=2048, inter=128, n_experts=256)
    x = gen.fp16_normal(gen.rng(2003), (64, 2048))
    block = native.MoeBlock(d, topk=8)
    _, ids, w = block(dev(x))
    ref_ids, ref_w, _ = o.route(x, d["Wg"], 8)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    assert np.allclose(w.cpu().numpy(), ref_w, rtol=1e-5, atol=1e-6)


def test_router_ties_at_the_boundary(native):
    """Integer-valued inputs make exact logit ties; the lower id must win."""
    E, H = 16, 256
    Wg = np.zeros((E, H), dtype=np.float16)
    x = np.zeros((1, H), dtype=np.float16)
    x[0, :4] = 1.0
    # experts 3, 5, 9, 12 tie at logit 2; expert 7 has 3; topk 3 -> 7, 3, 5
    for e, v in ((3, 2.0), (5, 2.0), (9, 2.0), (12, 2.0), (7, 3.0)):
        Wg[e, 0] = v
    d = gen.moe_layer(17, hidden=H, inter=128, n_experts=E)
    d["Wg"] = Wg
    block = native.MoeBlock(d, topk=3)
    _, ids, w = block(dev(x))
    assert list(ids.cpu().numpy()[0]) == [7, 3, 5]
    ref_ids, _, _ = o.route(x, Wg, 3)
    assert list(ref_ids[0]) == [7, 3, 5]


def test_moe_block_deterministic(native):
    d = gen.moe_layer(19, hidden=512, inter=256, n_experts=16)
    x = dev(gen.fp16_normal(gen.rng(20), (4, 512)))
    block = native.MoeBlock(d, topk=4)
    a = block(x)[0].cpu().numpy()
    b = block(x)[0].cpu().numpy()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_moe_pruned_gate_up_channels_stay_zero(native):
    """Through the whole block: with down's input pinned to the pruned
    channels only, nothing leaks. Checked on gate_up's own output via the
    single-projection call with an expert's rout."""
    d = gen.moe_layer(21, hidden=512, inter=256, n_experts=4)
    e = 2
    x = gen.fp16_normal(gen.rng(22), (1, 512))
    y = native.trellis_gemv(dev(d["gu_codes"][e]), dev(x), dev(d["gu_rin"][e]), dev(d["gu_rout"][e])).cpu().numpy()
    pruned = d["gu_rout"][e] == 0
    assert pruned[:256].sum() == pruned[256:].sum() > 0
    assert np.array_equal(pruned[:256], pruned[256:])
    assert np.all(y[0, pruned] == 0)


# --------------------------------------------------------------- grouped path
# More than 16 tokens per call run the grouped path: tokens sorted by expert,
# each expert decoded once per work item of up to 128 tokens into tcgen05
# MMAs.


def test_moe_grouped_small_groups(native):
    d = gen.moe_layer(23, hidden=512, inter=256, n_experts=16, k_gu=3, k_dn=2)
    x = gen.fp16_normal(gen.rng(24), (40, 512))
    _check_block(native, d, x, topk=4)


def test_moe_grouped_multiple_items_per_expert(native):
    """300 tokens over 8 experts, top-2: about 75 slots per expert, so each
    expert spans two 64-token work items."""
    d = gen.moe_layer(25, hidden=256, inter=128, n_experts=8, k_gu=2, k_dn=3)
    x = gen.fp16_normal(gen.rng(26), (300, 256))
    _check_block(native, d, x, topk=2, tokens=range(0, 300, 7))


def test_moe_grouped_full_size_batch64_sampled(native):
    """The full Qwen3.6-35B-A3B-shaped block at batch 64; the oracle checks a
    sample of tokens one by one (routing for all 64)."""
    d = gen.moe_layer(1003)
    x = gen.fp16_normal(gen.rng(2004), (64, 2048))
    _check_block(native, d, x, topk=8, tokens=[0, 17, 38, 63])


def test_moe_grouped_full_size_batch256_sampled(native):
    """The full Qwen3.6-35B-A3B-shaped block at batch 256 (the batched-decode
    workload): routing checked for every token (the oracle routes 64 tokens
    at a time), outputs for a sample of tokens."""
    d = gen.moe_layer(1003)
    x = gen.fp16_normal(gen.rng(2006), (256, 2048))
    block = native.MoeBlock(d, topk=8)
    out, ids, w = block(dev(x))
    out, ids, w = out.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy()
    assert int(block.workspace(256)[:4].view(torch.int32).item()) == 0
    for c in range(0, 256, 64):
        ref_ids, ref_w, _ = o.route(x[c:c + 64], d["Wg"], 8)
        assert np.array_equal(ids[c:c + 64], ref_ids), c
        assert np.allclose(w[c:c + 64], ref_w, rtol=1e-5, atol=1e-6)
    sample = [0, 101, 170, 255]
    ref, _, _, _ = o.moe_block(o.MoeLayer(**d), x[sample], k=8)
    assert rel_err_rows(out[sample], ref).max() <= TOL


@pytest.mark.parametrize("T,E,topk,tokens", [
    (17, 64, 8, None),                    # item capacity 16, runs of 1-4 tokens
    (96, 32, 4, range(0, 96, 5)),         # capacity 32
    (700, 4, 1, range(0, 700, 23)),       # capacity 128, two and more items per expert
    (130, 16, 8, range(0, 130, 9)),       # capacity 128, ragged runs
])
def test_moe_grouped_capacities(native, T, E, topk, tokens):
    d = gen.moe_layer(40 + T, hidden=512, inter=256, n_experts=E, k_gu=3, k_dn=2)
    x = gen.fp16_normal(gen.rng(41 + T), (T, 512))
    _check_block(native, d, x, topk=topk, tokens=tokens)


def test_moe_grouped_prefill_2048_sampled(native):
    """2048-token prefill chunk through the full-size block (capacity 128):
    routing checked for every token (the oracle routes 64 tokens at a time),
    outputs for a sample of tokens."""
    d = gen.moe_layer(1004)
    x = gen.fp16_normal(gen.rng(2005), (2048, 2048))
    block = native.MoeBlock(d, topk=8)
    out, ids, w = block(dev(x))
    out, ids, w = out.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy()
    assert int(block.workspace(2048)[:4].view(torch.int32).item()) == 0
    for c in range(0, 2048, 64):
        ref_ids, ref_w, _ = o.route(x[c:c + 64], d["Wg"], 8)
        assert np.array_equal(ids[c:c + 64], ref_ids), c
        assert np.allclose(w[c:c + 64], ref_w, rtol=1e-5, atol=1e-6)
    sample = [0, 511, 1024, 2047]
    ref, _, _, _ = o.moe_block(o.MoeLayer(**d), x[sample], k=8)
    assert rel_err_rows(out[sample], ref).max() <= TOL


def test_moe_grouped_deterministic(native):
    d = gen.moe_layer(27, hidden=512, inter=256, n_experts=16)
    x = dev(gen.fp16_normal(gen.rng(28), (33, 512)))
    block = native.MoeBlock(d, topk=4)
    a = block(x)[0].cpu().numpy()
    b = block(x)[0].cpu().numpy()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_moe_grouped_status_word_clear(native):
    d = gen.moe_layer(29, hidden=512, inter=256, n_experts=16)
    x = dev(gen.fp16_normal(gen.rng(30), (20, 512)))
    block = native.MoeBlock(d, topk=4)
    block(x)
    torch.cuda.synchronize()
    assert int(block.workspace(20)[:4].view(torch.int32).item()) == 0


# ---------------------------------------------------------- routing diagnostic
# escha_moe_route copies out the router logits and the grouping, so the router
# sum order, the top-k selection and the stable counting sort are checked bit
# for bit against the oracle.


def _check_route(native, d, x, topk):
    block = native.MoeBlock(d, topk=topk)
    r = {k: v.cpu().numpy() for k, v in block.route(dev(x)).items()}
    ref_ids, ref_w, ref_logits = o.route(x, d["Wg"], topk)
    assert np.array_equal(r["logits"].view(np.uint16), ref_logits), "router logits must match bit for bit"
    assert np.array_equal(r["ids"], ref_ids)
    assert np.allclose(r["w"], ref_w, rtol=1e-5, atol=1e-6)
    counts, offsets, perm = o.group_by_expert(ref_ids, d["Wg"].shape[0])
    assert np.array_equal(r["counts"], counts)
    assert np.array_equal(r["offsets"], offsets)
    assert np.array_equal(r["perm"], perm)


@pytest.mark.parametrize("T", [1, 3, 16, 64, 257])
def test_route_bit_exact(native, T):
    """Both router kernels (T < 16 one expert per warp, T >= 16 tiled) and the
    grouping; 257 tokens span several 256-slot rounds and a ragged tail."""
    d = gen.moe_layer(50 + T, hidden=2048, inter=128, n_experts=256)
    x = gen.fp16_normal(gen.rng(60 + T), (T, 2048))
    _check_route(native, d, x, topk=8)


def test_route_hidden_not_multiple_of_1024(native):
    """hidden 768: the tiled router's last column chunk is partial."""
    d = gen.moe_layer(70, hidden=768, inter=128, n_experts=40)
    x = gen.fp16_normal(gen.rng(71), (37, 768))
    _check_route(native, d, x, topk=6)


def test_route_skewed_load(native):
    """Most tokens prefer the same few experts (inputs along one direction):
    long runs per expert, several grouping rounds per warp segment."""
    d = gen.moe_layer(72, hidden=512, inter=128, n_experts=16)
    g = gen.rng(73)
    base = g.standard_normal(512)
    x = (base[None, :] + 0.1 * g.standard_normal((600, 512))).astype(np.float16)
    _check_route(native, d, x, topk=2)


# ------------------------------------------------------------- edge cases


@pytest.mark.parametrize("T", [3, 20])
def test_moe_single_expert_top1(native, T):
    """One expert, top-1: every slot goes to expert 0 with weight exactly 1
    (per-slot path at T = 3, one grouped item at T = 20)."""
    d = gen.moe_layer(95 + T, hidden=256, inter=128, n_experts=1)
    x = gen.fp16_normal(gen.rng(96 + T), (T, 256))
    out, ids, w = _check_block(native, d, x, topk=1)
    assert np.all(ids == 0) and np.all(w == 1.0)


def test_moe_max_tokens_per_call(native):
    """T = 8192, the largest batch of one call, on a small layer: 16,384 slots
    over 8 experts (items of 128 tokens, ~16 per expert); routing of every
    token is checked, outputs on a sample."""
    d = gen.moe_layer(97, hidden=256, inter=128, n_experts=8)
    x = gen.fp16_normal(gen.rng(98), (8192, 256))
    block = native.MoeBlock(d, topk=2)
    out, ids, w = block(dev(x))
    ref_ids, ref_w, _ = o.route(x, d["Wg"], 2)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    assert int(block.workspace(8192)[:4].view(torch.int32).item()) == 0
    sample = [0, 1, 4095, 4096, 8190, 8191]
    ref, _, _, _ = o.moe_block(o.MoeLayer(**d), x[sample], k=2)
    assert rel_err_rows(out.cpu().numpy()[sample], ref).max() <= TOL


@pytest.mark.parametrize("T", [1, 2, 3])
@pytest.mark.parametrize("hidden", [256, 768, 2048, 8192])
def test_moe_block_few_token_shared_rows(native, hidden, T):
    """The router grid's shared-expert CTAs: for 1-2 tokens and hidden <= 2048
    int8 rows and x in registers (768: a lane's last 512-column chunk is
    partial), for 3 tokens rows in registers and x staged in shared memory,
    above 2048 (8192) rows read from L2 and x staged."""
    d = gen.moe_layer(120 + hidden // 256, hidden=hidden, inter=128, n_experts=8, sh_inter=256)
    x = gen.fp16_normal(gen.rng(121 + hidden + T), (T, hidden))
    _check_block(native, d, x, topk=2)


@pytest.mark.parametrize("T", [2, 24])
def test_moe_max_hidden(native, T):
    """hidden = 8192, the largest the boundary accepts: the router's column
    chunks, 64 input blocks of gate_up, an 8192-row down projection and an
    int8 shared expert with 8192 inputs."""
    d = gen.moe_layer(99, hidden=8192, inter=128, n_experts=4, sh_inter=64)
    x = gen.fp16_normal(gen.rng(100), (T, 8192))
    _check_block(native, d, x, topk=2, tokens=[0, T - 1])


def test_moe_grouped_in_cuda_graph_matches_eager(native):
    """The grouped path captured in a CUDA graph (the shared expert forks onto
    the library's second stream and joins back inside the capture) replays to
    the eager outputs bit for bit."""
    d = gen.moe_layer(81, hidden=512, inter=256, n_experts=16, k_gu=3, k_dn=2)
    block = native.MoeBlock(d, topk=4)
    x = dev(gen.fp16_normal(gen.rng(82), (40, 512)))
    eager, ids_e, w_e = block(x)  # also creates the second stream outside any capture
    eager = eager.clone()
    s = torch.cuda.Stream()
    out = torch.empty_like(eager)
    ws = block.workspace(40)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            block(x, out=out, ws=ws)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)


@pytest.mark.parametrize("T", [1, 4])
def test_cluster_reduction_wait_runs_out(native, T):
    """Ranks != 0 of the per-slot cluster reductions kept from storing into
    rank 0 and from arriving (a test hook), with a 2^10-poll bound: rank 0's
    mbarrier waits run out, the status word reports it (1: gate_up, 2: down),
    the call returns without hanging, and the next call with the default
    settings is correct bit for bit."""
    import time

    block = native.MoeBlock(gen.moe_layer(1002), topk=8)
    x = dev(gen.fp16_normal(gen.rng(2100 + T), (T, 2048)))
    ref, ref_ids, _ = block(x)
    torch.cuda.synchronize()
    assert int(block.workspace(T)[:4].view(torch.int32).item()) == 0
    native.set_cluster_wait(10, skip_arrive=True)
    try:
        t0 = time.time()
        block(x)
        torch.cuda.synchronize()
        dt = time.time() - t0
        status = int(block.workspace(T)[:4].view(torch.int32).item())
    finally:
        native.set_cluster_wait()
    assert status in (1, 2), status
    assert dt < 5.0
    out, ids, _ = block(x)
    torch.cuda.synchronize()
    assert int(block.workspace(T)[:4].view(torch.int32).item()) == 0
    assert torch.equal(ids, ref_ids)
    assert torch.equal(out, ref)


def test_cluster_wait_setting_rejects_bad_values(native):
    with pytest.raises(native.EschaError) as ei:
        native.set_cluster_wait(7)
    assert ei.value.code == native.ESCHA_E_ARG
    assert native.lib().escha_debug_set_cluster_wait(31, 0) == native.ESCHA_E_ARG
    assert native.lib().escha_debug_set_cluster_wait(24, 2) == native.ESCHA_E_ARG
    native.set_cluster_wait()
