"""Pins for the CPU oracle: each test checks the oracle against something other
than itself (values the pages print, closed forms, invariants, independent
algorithms, library routines, brute force on tiny inputs)."""
import math
import struct

import numpy as np
import pytest

from conftest import golden_path
from escha_synth import gen
from oracle import escha_oracle as o


def _golden():
    rne, trunc, differs, distinct = {}, {}, None, None
    with open(golden_path("cba_pins.txt")) as f:
        for line in f:
            line = line.split("#")[0].split()
            if not line:
                continue
            if line[0] == "rne":
                rne[int(line[1], 16)] = int(line[2], 16)
            elif line[0] == "trunc":
                trunc[int(line[1], 16)] = int(line[2], 16)
            elif line[0] == "trunc_differs_in_0_7":
                differs = sorted(int(v, 16) for v in line[1:])
            elif line[0] == "distinct":
                distinct = int(line[1])
    return rne, trunc, differs, distinct


# ---------------------------------------------------------------- binary16 ---


def test_f16_decode_matches_numpy_for_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = o.f16_to_f64(bits)
    ref = bits.view(np.float16).astype(np.float64)
    finite = np.isfinite(ref)
    assert np.array_equal(ours[finite], ref[finite])
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    assert np.array_equal(ours[np.isinf(ref)], ref[np.isinf(ref)])


def test_f16_rne_matches_struct_half_packing():
    g = gen.rng(7)
    v = g.standard_normal(20000) * np.exp(g.uniform(-22, 12, 20000))
    # exact ties between neighbouring halves, in normal and subnormal ranges
    a = np.arange(1, 2000, dtype=np.float64)
    ties = np.concatenate([(a + 0.5) * 2.0 ** -24, (1024 + a + 0.5) * 2.0 ** -10, (1024 + a + 0.5) * 2.0 ** -20])
    v = np.concatenate([v, ties, -ties, [0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, 2.0 ** -25, 2.0 ** -26]])
    ours = o.f64_to_f16(v)
    ref = []
    for x in v:
        try:
            ref.append(struct.unpack("<H", struct.pack("<e", x))[0])
        except OverflowError:
            ref.append(0xFC00 if x < 0 else 0x7C00)
    assert np.array_equal(ours, np.array(ref, dtype=np.uint16))


# ---------------------------------------------------------------- codebook ---


def test_codebook_pins_printed_on_the_pages():
    rne, trunc, differs, distinct = _golden()
    for s, want in rne.items():
        assert int(o.codebook_f16(np.array([s]))[0]) == want
    alphabet = o.codebook_f16(np.arange(65536))
    assert len(np.unique(alphabet)) == distinct


def _trunc_f16(v):
    """Planted mistake: round the exact sum toward zero instead of to nearest."""
    v = float(v)
    a = abs(v)
    e = math.floor(math.log2(a))
    q = 2.0 ** (max(e, -14) - 10)
    n = math.floor(a / q)
    bits = ((max(e, -14) + 15) << 10) + n - 1024
    return bits | (0x8000 if v < 0 else 0)


def test_truncating_sum_fails_the_pins():
    rne, trunc, differs, _ = _golden()
    r = o.codebook_r(np.arange(8))
    exact = o.f16_to_f64(r & 0xFFFF) + o.f16_to_f64(r >> 16)
    t = [_trunc_f16(v) for v in exact]
    for s, want in trunc.items():
        assert t[s] == want
    good = o.codebook_f16(np.arange(8))
    assert sorted(s for s in range(8) if t[s] != good[s]) == differs


def test_codebook_closed_form_properties():
    alphabet = o.f16_to_f64(o.codebook_f16(np.arange(65536)))
    # both halves have exponent fields 12..15 after the mask and xor
    r = o.codebook_r(np.arange(65536))
    for half in (r & 0xFFFF, r >> 16):
        ex = (half >> 10) & 0x1F
        assert ex.min() >= 12 and ex.max() <= 15
    assert alphabet.max() == -alphabet.min() == 3.94921875
    assert np.all(np.isfinite(alphabet))
    nz = np.abs(alphabet[alphabet != 0])
    assert nz.min() >= 2.0 ** -13  # never subnormal in fp16


def test_codebook_hash_against_python_integers():
    for s in (0, 1, 3, 255, 4096, 0x7FFF, 0x8000, 0xFFFF):
        u = (s * 0xCBAC1FED) % (1 << 32)
        r = (u & 0x8FFF8FFF) ^ 0x3B603B60
        lo = struct.unpack("<e", struct.pack("<H", r & 0xFFFF))[0]
        hi = struct.unpack("<e", struct.pack("<H", r >> 16))[0]
        want = struct.unpack("<H", struct.pack("<e", lo + hi))[0]
        assert int(o.codebook_r(np.array([s]))[0]) == r
        assert int(o.codebook_f16(np.array([s]))[0]) == want


# ------------------------------------------------------------- bit stream ---


def _states_bit_by_bit(words, K):
    """Independent reader: the tile as one Python big integer, MSB first."""
    nbits = 16 * len(words)
    stream = 0
    for w in words:
        stream = (stream << 16) | int(w)
    bits = [(stream >> (nbits - 1 - p)) & 1 for p in range(nbits)]
    out = []
    for t in range(256):
        s = 0
        for b in range(16):
            s = (s << 1) | bits[(t * K + b) % nbits]
        out.append(s)
    return out


@pytest.mark.parametrize("K", [2, 3])
def test_tile_states_match_bit_by_bit_reader(K):
    g = gen.rng(11 + K)
    for _ in range(6):
        words = g.integers(0, 65536, size=16 * K, dtype=np.uint16)
        assert list(o.tile_states(words, K)) == _states_bit_by_bit(words, K)


@pytest.mark.parametrize("K", [2, 3])
def test_constant_streams(K):
    zeros = np.zeros(16 * K, dtype=np.uint16)
    ones = np.full(16 * K, 0xFFFF, dtype=np.uint16)
    assert np.all(o.tile_states(zeros, K) == 0)
    assert np.all(o.tile_states(ones, K) == 0xFFFF)


def test_k_from_code_shape():
    assert o.k_from_codes(np.zeros((2, 3, 32), np.uint16)) == 2
    assert o.k_from_codes(np.zeros((2, 3, 48), np.uint16)) == 3
    for bad in (16, 64, 40):
        with pytest.raises(ValueError):
            o.k_from_codes(np.zeros((1, 1, bad), np.uint16))


@pytest.mark.parametrize("K", [2, 3])
def test_tile_grid_layout(K):
    """Tile codes[kt][nt] fills rows 16kt.. and columns 16nt.. of W[in][out]."""
    codes = np.zeros((3, 4, 16 * K), dtype=np.uint16)
    codes[1, 2, :] = 0xFFFF
    W = o.decode_weights_f16(codes)
    assert W.shape == (48, 64)
    v0 = int(o.codebook_f16(np.array([0]))[0])
    v1 = int(o.codebook_f16(np.array([0xFFFF]))[0])
    expect = np.full((48, 64), v0, dtype=np.uint16)
    expect[16:32, 32:48] = v1
    assert np.array_equal(W, expect)


@pytest.mark.parametrize("K", [2, 3])
def test_within_tile_order_row_major_input_rows(K):
    """Weight t = 16 r + q of a tile sits at input row r, output column q."""
    g = gen.rng(5)
    words = g.integers(0, 65536, size=16 * K, dtype=np.uint16)
    states = _states_bit_by_bit(words, K)
    W = o.decode_weights_f16(words.reshape(1, 1, -1))
    for r in range(16):
        for q in range(16):
            assert W[r, q] == o.codebook_f16(np.array([states[16 * r + q]]))[0]


# ---------------------------------------------------------------- Hadamard ---


def _fwht(v):
    """Fast Walsh-Hadamard butterfly (independent of the explicit matrix)."""
    v = np.array(v, dtype=np.float64)
    h = 1
    while h < v.shape[-1]:
        for i in range(0, v.shape[-1], 2 * h):
            a = v[..., i:i + h].copy()
            b = v[..., i + h:i + 2 * h].copy()
            v[..., i:i + h] = a + b
            v[..., i + h:i + 2 * h] = a - b
        h *= 2
    return v


def test_h128_properties():
    H = o.hadamard(128)
    assert np.array_equal(H @ H.T, 128 * np.eye(128))
    assert np.all(H[0] == 1) and np.all(H[:, 0] == 1)
    g = gen.rng(3)
    v = g.standard_normal((3, 384))
    assert np.allclose(o.h128_blocks(o.h128_blocks(v)), v, atol=1e-12, rtol=0)
    ref = _fwht(v.reshape(3, 3, 128)).reshape(3, 384) / math.sqrt(128)
    assert np.allclose(o.h128_blocks(v), ref, atol=1e-12, rtol=0)


def test_input_order_rin_before_hadamard():
    """H(rin * e0) is -1/sqrt(128) everywhere when rin[0] = -1; the other
    order, rin * H(e0), would give rin / sqrt(128)."""
    x = np.zeros(128)
    x[0] = 1.0
    rin = np.ones(128)
    rin[0] = -1.0
    rin[5] = -1.0
    got = o.input_transform(x, rin)
    assert np.allclose(got, -1.0 / math.sqrt(128), atol=1e-15)


def test_output_order_rout_last_keeps_pruned_exactly_zero():
    g = gen.rng(9)
    z = g.standard_normal(256) * 50
    rout = g.uniform(0.5, 1.5, 256)
    rout[[3, 77, 200]] = 0.0
    y = o.output_transform(z, rout)
    assert np.all(y[[3, 77, 200]] == 0.0)
    assert np.all(y[rout != 0] != 0.0)


# ------------------------------------------------------------------- GEMV ---


@pytest.mark.parametrize("K,state,word", [(2, 0, 0x0000), (3, 0xFFFF, 0xFFFF)])
def test_gemv_closed_form_constant_weights(K, state, word):
    """All states equal -> W is the constant c; then z_o = c * sum_i x~_i,
    sum_i x~_i = sqrt(128) * sum_blocks v[128 b] with v = rin * x, and y has
    rout_o * sqrt(128) * z at the first channel of each output block, 0 at
    the others."""
    n_in, n_out = 256, 384
    codes = np.full((n_in // 16, n_out // 16, 16 * K), word, dtype=np.uint16)
    c = float(o.f16_to_f64(o.codebook_f16(np.array([state])))[0])
    g = gen.rng(21)
    x = g.standard_normal(n_in)
    rin = np.where(g.integers(0, 2, n_in) == 1, 1.0, -1.0)
    rout = g.uniform(0.5, 1.5, n_out)
    v = rin * x
    z = c * math.sqrt(128) * v[::128].sum()
    want = np.zeros(n_out)
    want[::128] = rout[::128] * math.sqrt(128) * z
    got = o.trellis_gemv(codes, x, rin, rout)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-9)


def test_gemv_brute_force_small():
    """Tiny case against dense arithmetic written out with Python loops."""
    K = 3
    g = gen.rng(31)
    codes = g.integers(0, 65536, size=(8, 8, 16 * K), dtype=np.uint16)
    x = g.standard_normal(128)
    rin = np.where(g.integers(0, 2, 128) == 1, 1.0, -1.0)
    rout = g.uniform(0.5, 1.5, 128)
    H = [[(-1) ** bin(i & j).count("1") for j in range(128)] for i in range(128)]
    s = 1 / math.sqrt(128)
    xt = [s * sum(H[i][j] * rin[j] * x[j] for j in range(128)) for i in range(128)]
    W = np.zeros((128, 128))
    for kt in range(8):
        for nt in range(8):
            st = _states_bit_by_bit(codes[kt, nt], K)
            for r in range(16):
                for q in range(16):
                    W[16 * kt + r, 16 * nt + q] = o.f16_to_f64(o.codebook_f16(np.array([st[16 * r + q]])))[0]
    z = [sum(W[i, j] * xt[i] for i in range(128)) for j in range(128)]
    y = [rout[i] * s * sum(H[i][j] * z[j] for j in range(128)) for i in range(128)]
    assert np.allclose(o.trellis_gemv(codes, x, rin, rout), y, rtol=1e-11, atol=1e-9)


def test_nan_weight_behind_zero_activation_propagates():
    W = np.ones((128, 128))
    W[5, 9] = np.nan
    y = o.trellis_gemv(None, np.zeros(128), np.ones(128), np.ones(128), W=W)
    assert np.all(np.isnan(y))


# ------------------------------------------------------------ dense linear ---


@pytest.mark.parametrize("K", [2, 3])
def test_nt_major_makes_consecutive_kt_adjacent(K):
    """In the nt-major grid the tiles of one output tile column are stored
    one after another: flat tile index nt * KT + kt holds tile (kt, nt)."""
    KT, NT = 5, 3
    codes = np.zeros((KT, NT, 16 * K), dtype=np.uint16)
    for kt in range(KT):
        for nt in range(NT):
            codes[kt, nt, :] = 1000 * kt + 10 * nt + np.arange(16 * K)
    t = o.codes_to_nt_major(codes)
    flat = t.reshape(-1, 16 * K)
    for kt in range(KT):
        for nt in range(NT):
            assert np.array_equal(flat[nt * KT + kt], codes[kt, nt])
    assert np.array_equal(o.codes_from_nt_major(t), codes)


@pytest.mark.parametrize("K", [2, 3])
def test_nt_major_decodes_to_identical_weights(K):
    """Whole tiles move, so the decoded weights of both grids are identical."""
    codes = gen.trellis_codes(gen.rng(40 + K), 128, 256, K)
    nt = o.codes_to_nt_major(codes)
    x = gen.rng(41).standard_normal((2, 128))
    rin = np.ones(128)
    rout = np.ones(256)
    assert np.array_equal(o.dense_linear(nt, x, rin, rout, nt_major=True), o.dense_linear(codes, x, rin, rout))


def test_dense_bias_lands_after_the_output_transform():
    """x = 0 gives exactly the bias, and a pruned channel (rout = 0) gives
    exactly its bias for any x; a bias added before the output Hadamard or
    before the rout multiply would spread over or vanish from those channels."""
    g = gen.rng(42)
    codes = gen.trellis_codes(g, 256, 384, 2)
    rin = np.where(g.integers(0, 2, 256) == 1, 1.0, -1.0)
    rout = g.uniform(0.5, 1.5, 384)
    rout[[0, 17, 300]] = 0.0
    bias = g.standard_normal(384) * 8
    y0 = o.dense_linear(codes, np.zeros((1, 256)), rin, rout, bias=bias)
    assert np.array_equal(y0[0], bias)
    x = g.standard_normal((3, 256))
    y = o.dense_linear(codes, x, rin, rout, bias=bias)
    assert np.all(y[:, [0, 17, 300]] == bias[[0, 17, 300]])
    live = rout != 0
    assert np.all(np.abs(y[:, live] - bias[live]) > 0)


def test_dense_closed_form_constant_weights_with_bias():
    """Constant weights c: y = rout * sqrt(128) * c * sqrt(128) * sum_b v[128 b]
    at the first channel of each output block, 0 elsewhere, plus the bias."""
    K, n_in, n_out = 3, 256, 256
    codes = np.full((n_in // 16, n_out // 16, 16 * K), 0xFFFF, dtype=np.uint16)
    c = float(o.f16_to_f64(o.codebook_f16(np.array([0xFFFF])))[0])
    g = gen.rng(43)
    x = g.standard_normal(n_in)
    rin = np.where(g.integers(0, 2, n_in) == 1, 1.0, -1.0)
    rout = g.uniform(0.5, 1.5, n_out)
    bias = g.standard_normal(n_out)
    v = rin * x
    want = bias.copy()
    want[::128] += rout[::128] * 128.0 * c * v[::128].sum()
    got = o.dense_linear(o.codes_to_nt_major(codes), x, rin, rout, bias=bias, nt_major=True)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-9)


def test_swiglu_gate_is_first_half():
    y = np.array([2.0, 3.0])
    assert o.swiglu(y)[0] == pytest.approx(2.0 / (1 + math.exp(-2.0)) * 3.0)
    assert o.swiglu(y)[0] != pytest.approx(3.0 / (1 + math.exp(-3.0)) * 2.0)
    assert o.silu(np.array([-1000.0]))[0] == 0.0


# ----------------------------------------------------------------- router ---


def test_router_exact_for_integer_inputs():
    """Small integers: every partial sum is exact, so the logits must equal
    the f16 rounding of the exact dot product, whatever the order."""
    g = gen.rng(41)
    x = g.integers(-4, 5, size=(3, 512)).astype(np.float16)
    Wg = g.integers(-3, 4, size=(16, 512)).astype(np.float16)
    exact = x.astype(np.float64) @ Wg.astype(np.float64).T
    want = exact.astype(np.float16).view(np.uint16)
    assert np.array_equal(o.router_logits(x, Wg), want)


def test_router_logits_close_to_exact_dot():
    d = gen.moe_layer(1002, hidden=512, inter=128, n_experts=32)
    x = gen.fp16_normal(gen.rng(5), (4, 512))
    got = o.f16_to_f64(o.router_logits(x, d["Wg"]))
    exact = x.astype(np.float64) @ d["Wg"].astype(np.float64).T
    assert np.max(np.abs(got - exact) / np.maximum(np.abs(exact), 1e-3)) < 2e-3


def test_topk_ties_go_to_lower_id_and_weights_renormalise():
    logits = np.zeros((1, 12))
    logits[0, [2, 5, 7, 9]] = [3.0, 1.0, 1.0, 1.0]
    bits = o.f64_to_f16(logits)
    ids, w = o.topk_from_logits(bits, 3)
    assert list(ids[0]) == [2, 5, 7]
    e = np.exp([3.0, 1.0, 1.0])
    assert np.allclose(w[0], e / e.sum())
    assert w[0].sum() == pytest.approx(1.0)


def test_group_by_expert_is_a_stable_counting_sort():
    g = gen.rng(51)
    ids = g.integers(0, 16, size=(13, 4)).astype(np.int32)
    counts, offsets, perm = o.group_by_expert(ids, 16)
    flat = ids.reshape(-1)
    assert np.array_equal(counts, np.bincount(flat, minlength=16))
    assert offsets[-1] == flat.size and np.all(np.diff(offsets) == counts)
    assert np.array_equal(np.sort(perm), np.arange(flat.size))
    ref = np.argsort(flat, kind="stable")
    assert np.array_equal(perm, ref)


# ------------------------------------------------------------------- int8 ---


def test_int8_dequant_is_one_f32_multiply():
    g = gen.rng(61)
    w = np.arange(-128, 128, dtype=np.int8)
    W = np.tile(w, (64, 1))
    s = g.uniform(1e-3, 1e-2, 64).astype(np.float32)
    deq = o.int8_dequant(W, s)
    exact = s.astype(np.float64)[:, None] * W.astype(np.float64)  # exact in float64
    assert np.array_equal(deq, exact.astype(np.float32))
    assert deq.dtype == np.float32


def test_int8_matvec_against_loops():
    W, s = gen.int8_matrix(3, 8, 16)
    x = np.arange(16) * 0.25 - 2
    y = o.int8_matvec(W, s, x[None, :])[0]
    for n in range(8):
        acc = 0.0
        for i in range(16):
            acc += float(np.float32(s[n]) * np.float32(W[n, i])) * x[i]
        assert y[n] == pytest.approx(acc, rel=1e-14, abs=1e-14)


# -------------------------------------------------------------------- MoE ---


def _small_layer(seed=77, E=8, hidden=256, inter=128, same=False):
    d = gen.moe_layer(seed, hidden=hidden, inter=inter, n_experts=E)
    if same:
        for k in ("gu_codes", "dn_codes", "gu_rin", "gu_rout", "dn_rin", "dn_rout"):
            d[k] = np.broadcast_to(d[k][:1], d[k].shape).copy()
    return o.MoeLayer(**d)


def test_moe_identical_experts_reduce_to_one_expert():
    layer = _small_layer(same=True)
    x = gen.fp16_normal(gen.rng(8), (3, 256))
    out, ids, w, _ = o.moe_block(layer, x, k=4)
    sh = o.shared_expert(layer, x)
    for b in range(3):
        one = o.moe_expert(layer, 0, o.f16_to_f64(x[b].view(np.uint16)))
        assert np.allclose(out[b] - sh[b], one, rtol=1e-12, atol=1e-9)


def test_moe_routes_selected_experts_only():
    layer = _small_layer()
    x = gen.fp16_normal(gen.rng(9), (2, 256))
    out, ids, w, _ = o.moe_block(layer, x, k=2)
    xv = o.f16_to_f64(x.view(np.uint16))
    sh = o.shared_expert(layer, x)
    for b in range(2):
        want = sum(w[b, j] * o.moe_expert(layer, ids[b, j], xv[b]) for j in range(2)) + sh[b]
        assert np.allclose(out[b], want, rtol=1e-12)
        assert len(set(ids[b])) == 2


# ------------------------------------------------------------ R-NORM (stack)


def test_rmsnorm_constant_row_closed_form():
    """h = c everywhere: sum = H c^2 exactly, mean = c^2, x = c / |c| = +-1."""
    for H in (512, 768, 100):
        for c in (2.0, -0.5, 8.0):
            h = np.full((3, H), c, dtype=np.float32)
            h2, x = o.residual_rmsnorm(h, eps=0.0)
            assert np.array_equal(h2, h)
            assert np.all(x == (0x3C00 if c > 0 else 0xBC00))


def test_rmsnorm_within_one_ulp_of_float64():
    """Against an float64 RMSNorm computed directly (numpy's own sum):
    the fixed-order f32 version lands on the same or an adjacent fp16."""
    g = np.random.default_rng(5)
    for H in (2048, 256, 300):
        h = (g.standard_normal((16, H)) * g.uniform(0.1, 1e3, (16, 1))).astype(np.float32)
        _, x = o.residual_rmsnorm(h, eps=1e-6)
        hv = h.astype(np.float64)
        ref = hv / np.sqrt(np.mean(hv * hv, axis=1, keepdims=True) + 1e-6)
        xv = o.f16_to_f64(x)
        ulp = np.abs(ref) * 2.0 ** -10 + 2.0 ** -24
        assert np.all(np.abs(xv - ref) <= ulp)
        # normalised rows have mean square 1 up to the fp16 rounding
        assert np.allclose(np.mean(xv * xv, axis=1), 1.0, atol=2e-3)


def test_rmsnorm_residual_add_and_scale_invariance():
    g = np.random.default_rng(6)
    h = g.standard_normal((4, 512)).astype(np.float32)
    add = g.standard_normal((4, 512)).astype(np.float32)
    h2, x = o.residual_rmsnorm(h, add, eps=0.0)
    assert np.array_equal(h2, (h + add).astype(np.float32))
    # multiplying a row by a power of two changes nothing (exact in f32)
    _, x4 = o.residual_rmsnorm(h2 * np.float32(4.0), eps=0.0)
    assert np.array_equal(x, x4)
