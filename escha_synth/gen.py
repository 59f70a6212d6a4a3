"""Seeded synthetic inputs with the shapes and value distributions of the
Escha-W2 Qwen3.6-35B-A3B MoE layer (hidden 2048, 256 experts, top-8,
moe_inter 512).

Every generator takes an explicit seed and uses numpy's PCG64, so the oracle
and the CUDA path always see identical bytes. Half-precision tensors are
returned as ``np.float16`` arrays; trellis codes as ``np.uint16`` arrays of
shape [in/16][out/16][16*K] (the code tensor's own layout).

Recipes:

* trellis codes: uniform random 16-bit words;
* activations x: N(0, 1) rounded to fp16;
* rin: random +-1; rout: U(0.5, 1.5) * (+-1) rounded to fp16; gate_up rout
  carries a prune mask that zeroes the same intermediate channels in the
  gate half and the up half;
* router weights: N(0, 0.02) in fp16; shared-expert gate: N(0, 0.02) fp16;
* int8 weights: uniform integers in [-127, 127]; per-row f32 scales
  U(1e-3, 1e-2); bf16 activations N(0, 1);
* dense projections: the trellis recipe above for one weight, plus an f32
  output bias N(0, 8^2) (large enough to be seen next to outputs of
  magnitude ~sqrt(in)).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "rng",
    "trellis_codes",
    "signs",
    "rout_vector",
    "fp16_normal",
    "projection",
    "dense_projection",
    "moe_layer",
    "int8_matrix",
    "bf16_normal_bits",
    "prune_count",
]


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def trellis_codes(g: np.random.Generator, n_in: int, n_out: int, K: int, lead=()) -> np.ndarray:
    """Uniform random code words, shape lead + [n_in/16][n_out/16][16*K]."""
    shape = tuple(lead) + (n_in // 16, n_out // 16, 16 * K)
    return g.integers(0, 65536, size=shape, dtype=np.uint16)


def signs(g: np.random.Generator, shape) -> np.ndarray:
    return np.where(g.integers(0, 2, size=shape) == 1, 1.0, -1.0).astype(np.float16)


def fp16_normal(g: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    return (g.standard_normal(size=shape) * std).astype(np.float16)


def prune_count(rate: float, channels: int) -> int:
    return int(round(rate * channels))


def rout_vector(g: np.random.Generator, n_out: int, prune: int = 0, glu: bool = False) -> np.ndarray:
    """rout = U(0.5, 1.5) * (+-1) in fp16. With ``glu`` the vector covers a
    gate half and an up half of n_out/2 channels each, and ``prune`` channels
    chosen at random are zeroed in both halves alike."""
    mag = g.uniform(0.5, 1.5, size=n_out)
    sg = np.where(g.integers(0, 2, size=n_out) == 1, 1.0, -1.0)
    r = (mag * sg).astype(np.float16)
    if prune:
        half = n_out // 2 if glu else n_out
        ch = g.choice(half, size=prune, replace=False)
        r[ch] = 0
        if glu:
            r[half + ch] = 0
    return r


def projection(seed: int, n_in: int, n_out: int, K: int, prune_rate: float = 0.55, glu: bool = True,
               batch: int = 1):
    """One expert projection at batch ``batch``: codes, x [batch][n_in],
    rin [n_in], rout [n_out] (gate/up prune mask of round(rate * n_out/2)
    channels when ``glu``)."""
    g = rng(seed)
    codes = trellis_codes(g, n_in, n_out, K)
    x = fp16_normal(g, (batch, n_in))
    rin = signs(g, n_in)
    prune = prune_count(prune_rate, n_out // 2 if glu else n_out) if prune_rate else 0
    rout = rout_vector(g, n_out, prune=prune, glu=glu)
    return {"codes": codes, "x": x, "rin": rin, "rout": rout, "K": K}


def dense_projection(seed: int, n_in: int, n_out: int, K: int, M: int, prune_rate: float = 0.0,
                     bias: bool = True):
    """One dense projection for M tokens: codes (kt-major), x [M][n_in] fp16,
    rin, rout (``prune_rate`` of the output channels zeroed), and an f32
    output bias [n_out] (None without ``bias``)."""
    g = rng(seed)
    codes = trellis_codes(g, n_in, n_out, K)
    x = fp16_normal(g, (M, n_in))
    rin = signs(g, n_in)
    rout = rout_vector(g, n_out, prune=prune_count(prune_rate, n_out), glu=False)
    b = (g.standard_normal(size=n_out) * 8.0).astype(np.float32) if bias else None
    return {"codes": codes, "x": x, "rin": rin, "rout": rout, "bias": b, "K": K}


def moe_layer(seed: int, hidden: int = 2048, inter: int = 512, n_experts: int = 256, k_gu: int = 3,
              k_dn: int = 2, prune_lo: float = 0.14, prune_hi: float = 0.58, sh_inter: int | None = None):
    """All weights of one MoE block. Returns a dict of numpy arrays whose keys
    match the fields of the oracle's MoeLayer and of the C-ABI layer struct."""
    if sh_inter is None:
        sh_inter = inter
    g = rng(seed)
    E = n_experts
    d = {}
    d["Wg"] = fp16_normal(g, (E, hidden), 0.02)
    d["gu_codes"] = trellis_codes(g, hidden, 2 * inter, k_gu, lead=(E,))
    d["dn_codes"] = trellis_codes(g, inter, hidden, k_dn, lead=(E,))
    d["gu_rin"] = signs(g, (E, hidden))
    d["dn_rin"] = signs(g, (E, inter))
    rates = g.uniform(prune_lo, prune_hi, size=E)
    d["prune_rates"] = rates
    d["gu_rout"] = np.stack([rout_vector(g, 2 * inter, prune=prune_count(rates[e], inter), glu=True)
                             for e in range(E)])
    d["dn_rout"] = np.stack([rout_vector(g, hidden) for _ in range(E)])
    d["sh_gu_w8"] = g.integers(-127, 128, size=(2 * sh_inter, hidden), dtype=np.int8)
    d["sh_gu_s"] = g.uniform(1e-3, 1e-2, size=2 * sh_inter).astype(np.float32)
    d["sh_dn_w8"] = g.integers(-127, 128, size=(hidden, sh_inter), dtype=np.int8)
    d["sh_dn_s"] = g.uniform(1e-3, 1e-2, size=hidden).astype(np.float32)
    d["sh_gate"] = fp16_normal(g, hidden, 0.02)
    d["hidden"], d["inter"], d["n_experts"], d["sh_inter"] = hidden, inter, E, sh_inter
    d["k_gu"], d["k_dn"] = k_gu, k_dn
    return d


def int8_matrix(seed: int, N: int, Kin: int):
    g = rng(seed)
    W = g.integers(-127, 128, size=(N, Kin), dtype=np.int8)
    s = g.uniform(1e-3, 1e-2, size=N).astype(np.float32)
    return W, s


def bf16_normal_bits(g: np.random.Generator, shape) -> np.ndarray:
    """N(0, 1) samples rounded to bfloat16 (round to nearest even), returned as
    uint16 bit patterns."""
    f = g.standard_normal(size=shape).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounding = ((u >> 16) & 1) + 0x7FFF
    return ((u + rounding) >> 16).astype(np.uint16)


def stack_k(layer: int):
    """Bits per weight (2 or 3) of gate_up and down in block `layer` of the
    synthetic 40-block stack, drawn from seed 5000 + layer."""
    k = rng(5000 + layer).integers(2, 4, size=2)
    return int(k[0]), int(k[1])
