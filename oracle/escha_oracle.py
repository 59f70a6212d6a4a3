"""CPU oracle for the Escha-W2 ("eschamoe") trellis MoE expert path.

TEST INFRASTRUCTURE. Only the test suite, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module. The product path (the CUDA library in ``bit_trellis_quantized_gb300``
and its Python binding) never imports, calls or links it, and the two share no
code: no kernels, headers, helpers, tables or constants.

It is deliberately plain and slow: numpy arrays, float64 wherever the method
does not fix a narrower precision, no blocking, fusion or reordering beyond
what the definitions below state. Each function cites the passage it follows.
Sources, by page:

* hipfire PR #694 "Escha-W2 port: 2-bit trellis decoded in the GEMV"
  (the summary section "What it is" and the commit messages of the PR);
* the model card "dogfoodai/Qwen3.6-35B-A3B-Escha-W2-trellis-mlx", table
  "Exactness of every tensor" and the Hadamard note under it;
* the model card "EschaLabs/Qwen3.6-35B-A3B-Escha-W2", section "Format notes".

Readings taken where the pages are silent (each one is listed, with its
reason, in the design notes of the repository):

* R-BITS  the 16*K words of a tile form one cyclic bit stream of 256*K bits,
  most significant bit of each word first, word 0 first. Weight t
  (t = 0..255) takes the 16 bits that start at bit t*K (wrapping around the
  end of the stream: tail-biting), first bit most significant. Inside a tile,
  t = 16*r + q with r the input row and q the output column, so weight
  W[16*kt + r][16*nt + q] comes from tile codes[kt][nt]. Parity unpinned
  against real checkpoints (their golden tensors are not available).
* R-H     the blockwise Hadamard-128 is scaled by 1/sqrt(128) on both sides.
* R-ORD   input side: H(rin * x); output side: rout * H(z), rout last.
* R-ROUTER logits are f32 sums of exact fp16*fp16 products in a fixed order
  (see ``router_logits``), then rounded to f16; top-k ties go to the lower
  expert id.
* R-GATE  the shared-expert gate logit is an unrounded dot product.
* R-NORM  a stack of blocks keeps an f32 residual h and feeds each block
  fp16(h / sqrt(mean(h^2) + eps)), a weightless RMSNorm, with the sum of
  squares in a fixed f32 order (see ``residual_rmsnorm``).
"""
from __future__ import annotations

import math

import numpy as np

# ----------------------------------------------------------------------------
# IEEE-754 binary16, written from the format's definition (1 sign bit, 5
# exponent bits with bias 15, 10 fraction bits), so no compiler or library
# half type decides any rounding here.
# ----------------------------------------------------------------------------


def f16_to_f64(bits) -> np.ndarray:
    """Value of binary16 bit patterns, as float64 (exact)."""
    b = np.asarray(bits).astype(np.uint32)
    sign = np.where((b >> 15) & 1, -1.0, 1.0)
    e = ((b >> 10) & 0x1F).astype(np.int64)
    f = (b & 0x3FF).astype(np.float64)
    sub = np.ldexp(f, -24)  # e == 0: f * 2^-24
    nrm = np.ldexp(f + 1024.0, (e - 25).astype(np.int64))  # (1024+f) * 2^(e-25)
    val = np.where(e == 0, sub, nrm)
    val = np.where(e == 31, np.where(f == 0, np.inf, np.nan), val)
    return sign * val


def _round_half_even(v: np.ndarray) -> np.ndarray:
    """Nearest integer, ties to the even integer (v >= 0, exact float64)."""
    fl = np.floor(v)
    d = v - fl
    odd = np.mod(fl, 2.0) == 1.0
    up = (d > 0.5) | ((d == 0.5) & odd)
    return fl + up


def f64_to_f16(v) -> np.ndarray:
    """Round float64 values to binary16 bit patterns, round-to-nearest-even.

    Every ``f16(...)`` of the Escha contract is round-to-nearest-even (hipfire
    PR #694, commits "Ports EschaLabs escha-mlx's cbA trellis codec" and
    "Task 1 found by TDD that crate::float16::f32_to_f16 truncates").
    """
    v = np.asarray(v, dtype=np.float64)
    sign = np.signbit(v).astype(np.uint32) << 15
    a = np.abs(v)
    finite = np.isfinite(a) & (a > 0)
    a_safe = np.where(finite, a, 1.0)
    _, E = np.frexp(a_safe)  # a = m * 2^E, m in [0.5, 1)
    e = E.astype(np.int64) - 1  # a in [2^e, 2^(e+1))
    qexp = np.maximum(e, -14) - 10  # quantum of the binade (subnormals: 2^-24)
    n = _round_half_even(np.ldexp(a_safe, -qexp))
    # normal: ((e+15) << 10) + (n - 1024); subnormal (e < -14): n. One formula
    # covers both, and n == 2048 (or 1024 below the normal range) carries into
    # the next exponent by itself.
    mag = ((np.maximum(e, -14) + 15) << 10) + n.astype(np.int64) - 1024
    mag = np.where(mag >= 0x7C00, 0x7C00, mag)
    mag = np.where(finite, mag, 0)
    mag = np.where(np.isinf(a), 0x7C00, mag)
    mag = np.where(np.isnan(a), 0x7E00, mag)
    return (sign | mag.astype(np.uint32)).astype(np.uint16)


def f32_round(v) -> np.ndarray:
    """IEEE single rounding of float64 values (numpy's float32 cast is RNE)."""
    return np.asarray(v, dtype=np.float64).astype(np.float32)


# ----------------------------------------------------------------------------
# The trellis codebook ("cbA"): hipfire PR #694 summary, "What it is";
# MLX model card, table "Exactness of every tensor".
#   r = ((s * 0xCBAC1FED) & 0x8FFF8FFF) ^ 0x3B603B60
#   value = f16_lo(r) + f16_hi(r), summed with round-to-nearest-even to fp16.
# ----------------------------------------------------------------------------

CB_MUL = 0xCBAC1FED
CB_MASK = 0x8FFF8FFF
CB_XOR = 0x3B603B60


def codebook_r(states) -> np.ndarray:
    """The 32-bit hash word r of each 16-bit trellis state."""
    s = np.asarray(states).astype(np.uint64)
    u = (s * np.uint64(CB_MUL)) & np.uint64(0xFFFFFFFF)
    return ((u & np.uint64(CB_MASK)) ^ np.uint64(CB_XOR)).astype(np.uint32)


def codebook_f16(states) -> np.ndarray:
    """fp16 bit pattern of the weight each 16-bit state decodes to."""
    r = codebook_r(states)
    lo = r & 0xFFFF  # low half: bits 0..15
    hi = r >> 16  # high half: bits 16..31
    exact = f16_to_f64(lo) + f16_to_f64(hi)  # exact in float64
    return f64_to_f16(exact)


# ----------------------------------------------------------------------------
# Trellis code layout (R-BITS, see module docstring). The code tensor is
# int16 [in/16][out/16][16*K]; K is the last dimension / 16 (hipfire PR #694,
# commit "Read Escha's test suite rather than only their reference
# implementation"; Escha model card, "Format notes").
# ----------------------------------------------------------------------------


def k_from_codes(codes) -> int:
    last = codes.shape[-1]
    if last % 16 != 0 or last // 16 not in (2, 3):
        raise ValueError(f"code last dimension {last} is not 16*K with K in (2, 3)")
    return last // 16


def tile_states(words, K: int) -> np.ndarray:
    """States of the 256 weights of each tile.

    ``words``: [..., 16*K] uint16 tile words. Returns [..., 256] int64, where
    entry t is the 16-bit window starting at bit t*K of the tile's cyclic
    stream (most significant bit first).
    """
    w = np.asarray(words).astype(np.int64)
    nwords = 16 * K
    assert w.shape[-1] == nwords
    t = np.arange(256)
    start = t * K
    j = start // 16  # word holding the window's first bit
    o = start % 16  # offset of that bit inside the word (from the MSB)
    first = w[..., j]
    second = w[..., (j + 1) % nwords]  # tail-biting: wraps to word 0
    window = (first << 16) | second  # 32 consecutive stream bits
    return (window >> (16 - o)) & 0xFFFF


def decode_weights_f16(codes) -> np.ndarray:
    """Dense fp16 bit patterns W[in][out] of a code tensor [in/16][out/16][16K].

    The oracle may materialise the weights; the GPU path never does.
    """
    K = k_from_codes(codes)
    KT, NT = codes.shape[0], codes.shape[1]
    st = tile_states(codes, K)  # [KT][NT][256]
    val = codebook_f16(st).reshape(KT, NT, 16, 16)  # [kt][nt][r][q]
    return val.transpose(0, 2, 1, 3).reshape(KT * 16, NT * 16)


def decode_weights(codes) -> np.ndarray:
    """Dense float64 weights W[in][out] (exact values of the fp16 weights)."""
    return f16_to_f64(decode_weights_f16(codes))


# ----------------------------------------------------------------------------
# Hadamard-128 and the two transforms around each trellis GEMV.
# Rotation: hipfire PR #694 summary ("H128 (Sylvester) on both sides");
# scale 1/sqrt(128): MLX model card, note on mx.hadamard_transform.
# Order: input H(rin * x) (R-ORD); output rout * H(z) with rout the final
# multiply, so pruned channels come out exactly zero (hipfire PR #694, commits
# "Second review pass" and "Naive one-thread-per-block butterfly").
# ----------------------------------------------------------------------------


def hadamard(n: int = 128) -> np.ndarray:
    """Sylvester Hadamard matrix, H[i][j] = (-1)^popcount(i & j), unscaled."""
    i = np.arange(n)
    parity = np.zeros((n, n), dtype=np.int64)
    anded = i[:, None] & i[None, :]
    for b in range(int(math.log2(n)) + 1):
        parity ^= (anded >> b) & 1
    return np.where(parity == 1, -1.0, 1.0)


_H128 = hadamard(128)
_INV_SQRT128 = 1.0 / math.sqrt(128.0)


def h128_blocks(v) -> np.ndarray:
    """(1/sqrt(128)) * H128 applied to each consecutive block of 128 values of
    the last axis, as an explicit matrix product."""
    v = np.asarray(v, dtype=np.float64)
    n = v.shape[-1]
    assert n % 128 == 0
    blk = v.reshape(v.shape[:-1] + (n // 128, 128))
    out = np.einsum("...bj,ij->...bi", blk, _H128) * _INV_SQRT128
    return out.reshape(v.shape)


def input_transform(x, rin) -> np.ndarray:
    """x~ = (1/sqrt(128)) H128_blockwise(rin * x)."""
    return h128_blocks(np.asarray(x, dtype=np.float64) * np.asarray(rin, dtype=np.float64))


def output_transform(z, rout) -> np.ndarray:
    """y = rout * ((1/sqrt(128)) H128_blockwise(z)); rout multiplies last."""
    return np.asarray(rout, dtype=np.float64) * h128_blocks(z)


def trellis_gemv(codes, x, rin, rout, W=None) -> np.ndarray:
    """One trellis-coded projection: y = rout * H(W^T H(rin * x)).

    ``codes`` [in/16][out/16][16K] uint16; ``x`` [..., in] float values;
    ``rin`` [in], ``rout`` [out] float values. The matvec is unconditional:
    no activation is skipped, so a non-finite weight always reaches the
    output (hipfire PR #694, commit "The accumulation loop treated a zero
    activation as a no-op shortcut").
    """
    if W is None:
        W = decode_weights(codes)
    xt = input_transform(x, rin)
    z = xt @ W  # float64 accumulate
    return output_transform(z, rout)


# ----------------------------------------------------------------------------
# Dense linear. hipfire PR #694: a dense projection is the one-expert case of
# the expert GEMV (commit "EschaProj holds what a trellis weight needs"); the
# dense export adds a per-projection output bias at the point where each
# projection's result is complete, before SwiGLU for gate/up (commit adding
# the escha dense export's biases in decode and prefill); the checkpoint's
# kt-major tile grid may be moved at load to nt-major, whole tiles, contents
# untouched (commit on the nt-major tile grid).
# ----------------------------------------------------------------------------


def codes_to_nt_major(codes) -> np.ndarray:
    """[in/16][out/16][16K] -> [out/16][in/16][16K]: tile (kt, nt) moves to
    position (nt, kt); its words are not changed."""
    c = np.asarray(codes)
    KT, NT, L = c.shape
    out = np.empty((NT, KT, L), dtype=c.dtype)
    for kt in range(KT):
        for nt in range(NT):
            out[nt, kt] = c[kt, nt]
    return out


def codes_from_nt_major(codes_nt) -> np.ndarray:
    """Inverse of ``codes_to_nt_major``."""
    c = np.asarray(codes_nt)
    NT, KT, L = c.shape
    out = np.empty((KT, NT, L), dtype=c.dtype)
    for nt in range(NT):
        for kt in range(KT):
            out[kt, nt] = c[nt, kt]
    return out


def dense_linear(codes, x, rin, rout, bias=None, nt_major: bool = False, W=None) -> np.ndarray:
    """y[m] = rout * H(W^T H(rin * x[m])) + bias for each token m.

    ``codes`` is kt-major, or nt-major with ``nt_major`` (then the grid is
    moved back before decoding). ``bias`` (length out) is added after the
    output transform, i.e. after rout, so a pruned channel (rout = 0) yields
    exactly its bias."""
    if W is None:
        W = decode_weights(codes_from_nt_major(codes) if nt_major else codes)
    y = trellis_gemv(None, x, rin, rout, W=W)
    if bias is not None:
        y = y + np.asarray(bias, dtype=np.float64)
    return y


# ----------------------------------------------------------------------------
# Router. Logits are rounded to f16 before top-k (hipfire PR #694, commit
# "Executed the moeblk golden against real shipped layer-0 weights"), which is
# what makes exact ties possible. Softmax over all experts renormalised over
# the selected k equals a softmax over the k selected logits.
#
# R-ROUTER summation order, fixed so that the rounding to f16 is reproducible:
# each fp16*fp16 product is exact in f32. Partial sum l (l = 0..31) adds, one
# at a time in ascending index order, the products whose index i satisfies
# floor(i / 8) mod 32 == l. The 32 partials are then combined by the xor
# butterfly p[l] <- p[l] + p[l ^ m] for m = 16, 8, 4, 2, 1 (f32 adds) and
# partial 0 is rounded to f16.
# ----------------------------------------------------------------------------


def router_logits(x, Wg) -> np.ndarray:
    """f16 bit patterns of the router logits, [B][E]."""
    xf = f16_to_f64(np.asarray(x).view(np.uint16)).astype(np.float32)
    wf = f16_to_f64(np.asarray(Wg).view(np.uint16)).astype(np.float32)
    B, H = xf.shape
    E = wf.shape[0]
    assert H % 256 == 0
    prod = xf[:, None, :] * wf[None, :, :]  # exact f32 products, [B][E][H]
    chunks = prod.reshape(B, E, H // 256, 32, 8)  # [.., pass, lane, 8 consecutive]
    acc = np.zeros((B, E, 32), dtype=np.float32)
    for p in range(H // 256):
        for k in range(8):
            acc = (acc + chunks[:, :, p, :, k]).astype(np.float32)
    lanes = np.arange(32)
    for m in (16, 8, 4, 2, 1):
        acc = (acc + acc[:, :, lanes ^ m]).astype(np.float32)
    return f64_to_f16(acc[:, :, 0].astype(np.float64))


def topk_from_logits(logits_f16, k: int):
    """Top-k expert ids ordered by (logit descending, id ascending) and their
    softmax weights renormalised over the k selected logits (float64)."""
    lv = f16_to_f64(logits_f16)
    B, E = lv.shape
    ids = np.zeros((B, k), dtype=np.int32)
    w = np.zeros((B, k), dtype=np.float64)
    for b in range(B):
        order = sorted(range(E), key=lambda e: (-lv[b, e], e))[:k]
        ids[b] = order
        sel = lv[b, order]
        ex = np.exp(sel - sel.max())
        w[b] = ex / ex.sum()
    return ids, w


def route(x, Wg, k: int = 8):
    logits = router_logits(x, Wg)
    ids, w = topk_from_logits(logits, k)
    return ids, w, logits


def group_by_expert(ids, E: int):
    """Counting sort of the (token, slot) pairs by expert, stable in
    (token, slot) order: counts [E], offsets [E+1], perm [B*k] where perm
    holds flat slot indices b*k + j."""
    flat = np.asarray(ids).reshape(-1)
    counts = np.bincount(flat, minlength=E).astype(np.int32)
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    perm = np.zeros(flat.size, dtype=np.int32)
    fill = offsets[:-1].copy()
    for s, e in enumerate(flat):
        perm[fill[e]] = s
        fill[e] += 1
    return counts, offsets, perm


# ----------------------------------------------------------------------------
# SwiGLU (gate = first half of gate_up: hipfire PR #694, commit "The
# accumulation loop treated a zero activation as a no-op shortcut", test
# swiglu_uses_gate_first_half) and the sigmoid.
# ----------------------------------------------------------------------------


def silu(g) -> np.ndarray:
    g = np.asarray(g, dtype=np.float64)
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def swiglu(y) -> np.ndarray:
    y = np.asarray(y, dtype=np.float64)
    half = y.shape[-1] // 2
    return silu(y[..., :half]) * y[..., half:]


def sigmoid(v) -> np.ndarray:
    v = np.asarray(v, dtype=np.float64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-v))


# ----------------------------------------------------------------------------
# int8 w8a16: dequant is one IEEE f32 multiply, scale * w8, with a per-row
# f32 scale (MLX model card, table "Exactness of every tensor": "dequant =
# f32 scale*w8").
# ----------------------------------------------------------------------------


def int8_dequant(W8, scales) -> np.ndarray:
    """f32 dequantised weights [N][Kin]: fl32(scale[o] * w8[o][i])."""
    s = np.asarray(scales, dtype=np.float32)
    w = np.asarray(W8).astype(np.float32)
    return (s[:, None] * w).astype(np.float32)


def int8_matvec(W8, scales, x) -> np.ndarray:
    """y[m][o] = sum_i deq[o][i] * x[m][i], float64 accumulate."""
    deq = int8_dequant(W8, scales).astype(np.float64)
    return np.asarray(x, dtype=np.float64) @ deq.T


# ----------------------------------------------------------------------------
# The MoE block.
# ----------------------------------------------------------------------------


class MoeLayer:
    """Weights of one MoE block (numpy arrays, fp16 tensors as np.float16).

    Shapes: Wg [E][hidden]; gu_codes [E][hidden/16][2*inter/16][16*Kgu];
    gu_rin [E][hidden]; gu_rout [E][2*inter]; dn_codes
    [E][inter/16][hidden/16][16*Kdn]; dn_rin [E][inter]; dn_rout [E][hidden];
    sh_gu_w8 [2*inter_sh][hidden] int8, sh_gu_s [2*inter_sh] f32;
    sh_dn_w8 [hidden][inter_sh] int8, sh_dn_s [hidden] f32; sh_gate [hidden].
    """

    def __init__(self, **arrays):
        self.__dict__.update(arrays)
        self._cache = {}

    def expert_weights(self, proj: str, e: int) -> np.ndarray:
        """Decoded dense weights of one expert projection, memoised: decoding
        per (token, slot) is needlessly slow (hipfire PR #694, commit
        "Executed the moeblk golden")."""
        key = (proj, int(e))
        if key not in self._cache:
            codes = self.gu_codes[e] if proj == "gu" else self.dn_codes[e]
            self._cache[key] = decode_weights(codes)
        return self._cache[key]


def _f16v(a) -> np.ndarray:
    return f16_to_f64(np.asarray(a).view(np.uint16))


def moe_expert(layer: MoeLayer, e: int, x_row) -> np.ndarray:
    """Routed expert e on one token: gate_up -> SwiGLU -> down."""
    y = trellis_gemv(None, x_row, _f16v(layer.gu_rin[e]), _f16v(layer.gu_rout[e]),
                     W=layer.expert_weights("gu", e))
    h = swiglu(y)
    return trellis_gemv(None, h, _f16v(layer.dn_rin[e]), _f16v(layer.dn_rout[e]),
                        W=layer.expert_weights("dn", e))


def shared_expert(layer: MoeLayer, x) -> np.ndarray:
    """int8 shared expert times its sigmoid gate, [B][hidden] (R-GATE)."""
    xv = _f16v(x)
    gu = int8_matvec(layer.sh_gu_w8, layer.sh_gu_s, xv)
    h = swiglu(gu)
    dn = int8_matvec(layer.sh_dn_w8, layer.sh_dn_s, h)
    gate = sigmoid(xv @ _f16v(layer.sh_gate))
    return gate[:, None] * dn


def moe_block(layer: MoeLayer, x, k: int = 8, tokens=None):
    """out[b] = sum_j w[b,j] * expert(ids[b,j], x[b]) + sigmoid(g.x) * shared(x).

    ``x`` [B][hidden] fp16. ``tokens`` optionally restricts the expert work to
    a subset of rows (the router still runs for all of them). Returns
    (out [len(tokens)][hidden] float64, ids, w, logits).
    """
    ids, w, logits = route(x, layer.Wg, k)
    rows = range(x.shape[0]) if tokens is None else tokens
    xv = _f16v(x)
    sh = shared_expert(layer, np.asarray(x)[list(rows)])
    out = np.zeros((len(list(rows)), xv.shape[1]), dtype=np.float64)
    for n, b in enumerate(rows):
        acc = np.zeros(xv.shape[1], dtype=np.float64)
        for j in range(k):
            acc += w[b, j] * moe_expert(layer, ids[b, j], xv[b])
        out[n] = acc + sh[n]
    return out, ids, w, logits


# ----------------------------------------------------------------------------
# Residual stream of a stack of blocks (reading R-NORM). Every escha
# projection of the pages' model takes a plain RMS-normed input (hipfire PR
# #694, commit on escha_run_proj / escha_run_resid). With random weights the
# block outputs grow by ~1e4 per block without a norm, so a synthetic stack
# normalises the f32 residual (no learned weight) and rounds to fp16. Since
# that rounding feeds the router, the arithmetic is fixed: f32 multiply then
# f32 add of h^2 per partial sum p = 0..255 over i = p, p+256, ... ascending;
# the partials of each group of 32 combined by the xor butterfly (offsets 16,
# 8, 4, 2, 1), the 8 group sums added in order; mean = sum / hidden; IEEE f32
# sqrt and division; x = f16_rne(h * (1 / sqrt(mean + eps))).
# ----------------------------------------------------------------------------


def residual_rmsnorm(h, add=None, eps: float = 1e-6):
    """Returns (h + add as f32 [T][H], x fp16 bit patterns [T][H])."""
    h = np.array(h, dtype=np.float32, ndmin=2)
    if add is not None:
        h = (h + np.asarray(add, dtype=np.float32)).astype(np.float32)
    T, H = h.shape
    n = -(-H // 256)
    hp = np.zeros((T, n * 256), dtype=np.float32)
    hp[:, :H] = h
    hp = hp.reshape(T, n, 256)
    s = np.zeros((T, 256), dtype=np.float32)
    for j in range(n):
        present = (j * 256 + np.arange(256)) < H
        sq = (hp[:, j, :] * hp[:, j, :]).astype(np.float32)
        s = np.where(present, (sq + s).astype(np.float32), s)
    s = s.reshape(T, 8, 32)
    lanes = np.arange(32)
    for m in (16, 8, 4, 2, 1):
        s = (s + s[:, :, lanes ^ m]).astype(np.float32)
    tot = s[:, 0, 0].copy()
    for w in range(1, 8):
        tot = (tot + s[:, w, 0]).astype(np.float32)
    mean = (tot / np.float32(H)).astype(np.float32)
    inv = (np.float32(1.0) / np.sqrt((mean + np.float32(eps)).astype(np.float32))).astype(np.float32)
    x = f64_to_f16((h * inv[:, None]).astype(np.float32).astype(np.float64))
    return h, x
