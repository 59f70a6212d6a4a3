"""Pins for the oracle's composed steps: one routed expert (gate_up -> SwiGLU
-> down), the int8 shared expert with its sigmoid gate, the router's fixed
f32 summation order, and the top-k weighted combine of a whole block.

Each expected value here is computed without the oracle: closed forms of
constant-weight experts, Python loops over tiny int8 matrices, the router
order written out from its statement with numpy float32 scalars, and f16
rounding by numpy's own float32 -> float16 cast. A plausible slip in the
oracle (a dropped sigmoid, a lost sign of a rout vector, gate and up
swapped, a different summation order, the wrong expert or weight in the
combine) fails at least one of these tests.

Sources: hipfire PR #694 "Escha-W2 port: 2-bit trellis decoded in the GEMV",
commit "Executed the moeblk golden against real shipped layer-0 weights"
(the block: routed experts gate_up -> SwiGLU -> down, weighted combine, the
sigmoid-gated shared expert; logits rounded to f16 before top-k); the MLX
model card "dogfoodai/Qwen3.6-35B-A3B-Escha-W2-trellis-mlx", table
"Exactness of every tensor" (int8 dequant is one f32 multiply).
"""
import math
import struct

import numpy as np
import pytest

from oracle import escha_oracle as o

SQ128 = math.sqrt(128.0)


def _half(bits: int) -> float:
    return struct.unpack("<e", struct.pack("<H", bits))[0]


def _codebook_value(s: int) -> float:
    """Decoded weight of state s, from the hash written with Python integers
    and struct's binary16 packing (independent of the oracle's codebook)."""
    u = (s * 0xCBAC1FED) % (1 << 32)
    r = (u & 0x8FFF8FFF) ^ 0x3B603B60
    return _half(struct.unpack("<H", struct.pack("<e", _half(r & 0xFFFF) + _half(r >> 16)))[0])


def _constant_tile_words(pattern_bits: str, K: int) -> np.ndarray:
    """Words of a tile whose cyclic stream repeats ``pattern_bits`` (length K):
    every window starts at a multiple of K, so all 256 states are equal to the
    first 16 bits of the repeated pattern."""
    stream = (pattern_bits * (16 * 16 * K // len(pattern_bits)))[: 16 * 16 * K]
    words = [int(stream[16 * j:16 * j + 16], 2) for j in range(16 * K)]
    return np.array(words, dtype=np.uint16)


def _constant_state(pattern_bits: str) -> int:
    return int((pattern_bits * 16)[:16], 2)


def _silu(g: float) -> float:
    return g / (1.0 + math.exp(-g))


def _sig(v: float) -> float:
    return 1.0 / (1.0 + math.exp(-v))


# Constant-state patterns: gate_up at K = 3, down at K = 2.
GU_PATTERNS = ["000", "111", "001", "011"]
DN_PATTERNS = ["00", "11", "01", "10"]


def _expert_constants(e: int):
    return _constant_state(GU_PATTERNS[e % 4]), _constant_state(DN_PATTERNS[(e + 1) % 4])


def _constant_expert_layer(E: int, hidden: int = 256, inter: int = 128, sh_inter: int = 4, seed: int = 0):
    """A layer whose experts have constant decoded weights (a different
    constant per expert and projection), fp16 sign/scale vectors with mixed
    signs and distinct magnitudes, and a small random int8 shared expert."""
    g = np.random.default_rng(seed)
    gu_codes = np.zeros((E, hidden // 16, 2 * inter // 16, 48), dtype=np.uint16)
    dn_codes = np.zeros((E, inter // 16, hidden // 16, 32), dtype=np.uint16)
    for e in range(E):
        gu_codes[e, :, :] = _constant_tile_words(GU_PATTERNS[e % 4], 3)
        dn_codes[e, :, :] = _constant_tile_words(DN_PATTERNS[(e + 1) % 4], 2)
    sgn = lambda shape: np.where(g.integers(0, 2, size=shape) == 1, 1.0, -1.0)
    d = {
        "Wg": np.zeros((E, hidden), dtype=np.float16),
        "gu_codes": gu_codes,
        "dn_codes": dn_codes,
        "gu_rin": sgn((E, hidden)).astype(np.float16),
        "dn_rin": sgn((E, inter)).astype(np.float16),
        # small gate/up scales keep the SiLU out of its saturated range
        "gu_rout": (sgn((E, 2 * inter)) * g.uniform(0.004, 0.03, (E, 2 * inter))).astype(np.float16),
        "dn_rout": (sgn((E, hidden)) * g.uniform(0.5, 1.5, (E, hidden))).astype(np.float16),
        "sh_gu_w8": g.integers(-127, 128, size=(2 * sh_inter, hidden), dtype=np.int8),
        "sh_gu_s": g.uniform(1e-3, 1e-2, size=2 * sh_inter).astype(np.float32),
        "sh_dn_w8": g.integers(-127, 128, size=(hidden, sh_inter), dtype=np.int8),
        "sh_dn_s": g.uniform(1e-3, 1e-2, size=hidden).astype(np.float32),
        "sh_gate": (g.standard_normal(hidden) * 0.05).astype(np.float16),
    }
    return d


def _expert_closed_form(d, e: int, x: np.ndarray) -> np.ndarray:
    """Output of expert e with constant weights cg (gate_up) and cd (down).

    gate_up: v = rin * x; the input transform sums to sqrt(128) * v[128 b]
    over each block b (column 0 of H is all ones, every other column sums to
    zero), so z_o = cg * sqrt(128) * S with S = sum_b v[128 b], the same for
    every output; the output transform of a constant block is sqrt(128) z at
    its first channel and 0 elsewhere, so y[128 b] = rout[128 b] * 128 cg S.
    With inter = 128: gate = y[0], up = y[128], h[0] = silu(gate) * up and
    h[j] = 0 otherwise. down: the same steps with v' = dn_rin[0] h[0] at
    index 0 give d[128 b] = dn_rout[128 b] * 128 * cd * dn_rin[0] * h[0]."""
    hidden = x.shape[0]
    sg, sd = _expert_constants(e)
    cg, cd = _codebook_value(sg), _codebook_value(sd)
    rin = d["gu_rin"][e].astype(np.float64)
    S = sum(rin[128 * b] * float(x[128 * b]) for b in range(hidden // 128))
    gu_rout = d["gu_rout"][e].astype(np.float64)
    gate = gu_rout[0] * 128.0 * cg * S
    up = gu_rout[128] * 128.0 * cg * S
    h0 = _silu(gate) * up
    out = np.zeros(hidden)
    dn_rout = d["dn_rout"][e].astype(np.float64)
    for b in range(hidden // 128):
        out[128 * b] = dn_rout[128 * b] * 128.0 * cd * float(d["dn_rin"][e][0]) * h0
    return out


def _shared_by_loops(d, x: np.ndarray) -> np.ndarray:
    """sigmoid(g . x) * down(SwiGLU(gate_up(x))) with int8 weights dequantised
    as one f32 multiply each, every sum a Python loop in float64."""
    w1, s1, w2, s2, gv = d["sh_gu_w8"], d["sh_gu_s"], d["sh_dn_w8"], d["sh_dn_s"], d["sh_gate"]
    n1, hidden = w1.shape
    inter = n1 // 2
    xs = [float(v) for v in x]
    gu = []
    for o_ in range(n1):
        acc = 0.0
        for i in range(hidden):
            acc += float(np.float32(s1[o_]) * np.float32(w1[o_, i])) * xs[i]
        gu.append(acc)
    h = [_silu(gu[j]) * gu[inter + j] for j in range(inter)]
    gate = 0.0
    for i in range(hidden):
        gate += float(gv[i]) * xs[i]
    out = np.zeros(hidden)
    for o_ in range(hidden):
        acc = 0.0
        for j in range(inter):
            acc += float(np.float32(s2[o_]) * np.float32(w2[o_, j])) * h[j]
        out[o_] = _sig(gate) * acc
    return out


# ---------------------------------------------------------- routed expert ---


def test_constant_tile_patterns_give_constant_states():
    for p in GU_PATTERNS:
        assert np.all(o.tile_states(_constant_tile_words(p, 3), 3) == _constant_state(p))
    for p in DN_PATTERNS:
        assert np.all(o.tile_states(_constant_tile_words(p, 2), 2) == _constant_state(p))


@pytest.mark.parametrize("e", [0, 1, 2, 3])
def test_moe_expert_closed_form(e):
    """gate_up -> SwiGLU (gate = first half) -> down of one expert equals its
    closed form; the signs of both rout vectors and of dn_rin reach the
    output, and the expert index selects that expert's weights."""
    d = _constant_expert_layer(4, seed=3)
    layer = o.MoeLayer(**d)
    g = np.random.default_rng(11)
    x = (g.standard_normal(256)).astype(np.float16).astype(np.float64)
    got = o.moe_expert(layer, e, x)
    want = _expert_closed_form(d, e, x)
    assert np.all(want[[0, 128]] != 0)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12 * np.abs(want).max())


def test_moe_expert_closed_form_has_teeth():
    """The closed form separates the slips it is meant to catch: with the
    down rout's sign dropped, or gate and up swapped, it changes."""
    d = _constant_expert_layer(4, seed=3)
    x = np.random.default_rng(11).standard_normal(256).astype(np.float16).astype(np.float64)
    e = next(e for e in range(4) if d["dn_rout"][e][0] < 0 or d["dn_rout"][e][128] < 0)
    want = _expert_closed_form(d, e, x)
    d2 = dict(d, dn_rout=np.abs(d["dn_rout"]))
    assert not np.allclose(_expert_closed_form(d2, e, x), want, rtol=1e-6)
    d3 = dict(d, gu_rout=np.concatenate([d["gu_rout"][:, 128:], d["gu_rout"][:, :128]], axis=1))
    assert not np.allclose(_expert_closed_form(d3, e, x), want, rtol=1e-6)


# ---------------------------------------------------------- shared expert ---


def test_shared_expert_against_loops():
    """int8 gate_up -> SwiGLU -> int8 down, times sigmoid(g . x) (an
    unrounded dot product), for two tokens, against Python loops."""
    g = np.random.default_rng(5)
    hidden, inter = 12, 3
    d = {
        "sh_gu_w8": g.integers(-127, 128, size=(2 * inter, hidden), dtype=np.int8),
        "sh_gu_s": g.uniform(1e-3, 1e-2, size=2 * inter).astype(np.float32),
        "sh_dn_w8": g.integers(-127, 128, size=(hidden, inter), dtype=np.int8),
        "sh_dn_s": g.uniform(1e-3, 1e-2, size=hidden).astype(np.float32),
        # a gate vector whose dot with x is well away from 0, where sigmoid(v) and v differ
        "sh_gate": np.full(hidden, 0.0625, dtype=np.float16),
    }
    layer = o.MoeLayer(**d)
    x = (np.abs(g.standard_normal((2, hidden))) + 1.0).astype(np.float16)
    got = o.shared_expert(layer, x)
    for b in range(2):
        want = _shared_by_loops(d, x[b].astype(np.float64))
        gate = sum(float(v) for v in x[b]) * 0.0625
        assert abs(gate) > 0.5 and abs(_sig(gate) - gate) > 0.1
        assert np.allclose(got[b], want, rtol=1e-12, atol=1e-12 * np.abs(want).max())


# ----------------------------------------------------------------- router ---


def _router_by_loops(x16: np.ndarray, w16: np.ndarray, lane_of) -> np.ndarray:
    """Router logits in a given lane assignment: lane l accumulates, one at a
    time in ascending index order, the f32 products x_i * w_i of the indices
    with lane_of(i) == l; the 32 lane sums combine by the xor butterfly
    (every lane l adds lane l ^ m, for m = 16, 8, 4, 2, 1) and lane 0's sum is
    rounded to f16 by numpy's float32 -> float16 cast."""
    B, H = x16.shape
    E = w16.shape[0]
    out = np.zeros((B, E), dtype=np.float16)
    for b in range(B):
        for e in range(E):
            acc = [np.float32(0.0)] * 32
            for i in range(H):
                lane = lane_of(i)
                acc[lane] = np.float32(acc[lane] + np.float32(x16[b, i]) * np.float32(w16[e, i]))
            for m in (16, 8, 4, 2, 1):
                acc = [np.float32(acc[lane] + acc[lane ^ m]) for lane in range(32)]
            out[b, e] = np.float16(acc[0])
    return out


def _cancelling_router_case(seed: int, E: int = 32, H: int = 512):
    """Products with large pairs that cancel exactly, plus small terms: the
    f32 rounding of every partial sum depends on which terms meet in which
    lane, so the f16 logits depend on the summation order."""
    g = np.random.default_rng(seed)
    x = g.choice([-1.0, 1.0], size=(2, H)).astype(np.float16)
    x[1] = (x[1] * 0.5).astype(np.float16)
    w = (g.standard_normal((E, H)) * 0.25).astype(np.float16)
    for e in range(E):
        pos = g.permutation(H)[:32]
        big = g.choice([-1.0, 1.0], 16) * 2.0 ** g.integers(10, 14, 16)
        w[e, pos[:16]] = (big * x[0, pos[:16]]).astype(np.float16)
        w[e, pos[16:]] = (-big * x[0, pos[16:]]).astype(np.float16)
    return x, w


def test_router_order_written_out_from_its_statement():
    """Lane l takes the products with floor(i / 8) mod 32 == l (eight
    consecutive inputs per lane per pass), then the xor butterfly; on inputs
    where the order decides the rounding, the oracle's f16 logits equal this
    order bit for bit."""
    x, w = _cancelling_router_case(17)
    want = _router_by_loops(x, w, lambda i: (i // 8) % 32).view(np.uint16)
    got = o.router_logits(x, w)
    assert np.array_equal(got, want)


def test_router_order_case_has_teeth():
    """The case above separates the stated order from its near neighbours:
    strided lanes (i mod 32), sixteen consecutive inputs per lane, one
    running sum, and the exact dot product rounded once."""
    x, w = _cancelling_router_case(17)
    want = _router_by_loops(x, w, lambda i: (i // 8) % 32)
    for other in (lambda i: i % 32, lambda i: (i // 16) % 32, lambda i: 0):
        assert np.mean(_router_by_loops(x, w, other) != want) > 0.25
    exact = (x.astype(np.float64) @ w.astype(np.float64).T).astype(np.float16)
    assert np.mean(exact != want) > 0.25


# ---------------------------------------------------------------- combine ---


def test_moe_block_combine_with_hand_built_logits():
    """x is nonzero at inputs 0 and 128 only and the router weights at those
    columns are chosen so each logit is exact: the top-4 (ties to the lower
    id), their softmax weights and the combine sum_j w_j d_j + sigmoid(g . x)
    * shared(x) follow by hand from the expert closed forms and the shared
    expert's loops."""
    E, k = 8, 4
    d = _constant_expert_layer(E, seed=9)
    # logits = Wg[e,0] * 0.5 + Wg[e,128] * (-0.25), all exact in fp16
    col0 = [0.5, 2.0, -1.0, 1.5, 1.0, 0.25, 3.0, -2.0]
    col128 = [0.0, 0.0, 2.0, -1.0, -4.0, 1.0, 0.0, 0.0]
    for e in range(E):
        d["Wg"][e, 0] = col0[e]
        d["Wg"][e, 128] = col128[e]
    logits = [0.5 * a - 0.25 * b for a, b in zip(col0, col128)]
    # logits: [0.25, 1.0, -1.0, 1.0, 1.5, -0.125, 1.5, -1.0]
    order = sorted(range(E), key=lambda e: (-logits[e], e))[:k]
    assert order == [4, 6, 1, 3]  # 1.5 ties -> 4 before 6; 1.0 ties -> 1 before 3
    ex = [math.exp(logits[e] - logits[order[0]]) for e in order]
    wts = [v / sum(ex) for v in ex]

    x = np.zeros((1, 256), dtype=np.float16)
    x[0, 0], x[0, 128] = 0.5, -0.25
    layer = o.MoeLayer(**d)
    out, ids, w, lg = o.moe_block(layer, x, k=k)
    assert list(ids[0]) == order
    assert np.allclose(w[0], wts, rtol=1e-13)
    assert np.array_equal(o.f16_to_f64(lg[0]), np.array(logits))

    xv = x[0].astype(np.float64)
    want = sum(wts[j] * _expert_closed_form(d, order[j], xv) for j in range(k)) + _shared_by_loops(d, xv)
    assert np.allclose(out[0], want, rtol=1e-12, atol=1e-12 * np.abs(want).max())
