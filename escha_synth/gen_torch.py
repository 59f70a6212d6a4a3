"""Seeded synthetic MoE-layer weights drawn directly on a CUDA device.

Same shapes and value distributions as ``gen.moe_layer`` (see its recipe),
drawn with torch's seeded device generator instead of numpy's PCG64, for
workloads too large to draw on the host in reasonable time (many distinct
layers). Random draws only: none of the method's arithmetic lives here.
"""
from __future__ import annotations

import torch


def moe_layer_device(seed: int, device, hidden: int = 2048, inter: int = 512, n_experts: int = 256, k_gu: int = 3,
                     k_dn: int = 2, prune_lo: float = 0.14, prune_hi: float = 0.58, sh_inter: int | None = None):
    if sh_inter is None:
        sh_inter = inter
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    E = n_experts
    kw = dict(device=device, generator=g)

    def codes(n_in, n_out, K):
        return torch.randint(-32768, 32768, (E, n_in // 16, n_out // 16, 16 * K), dtype=torch.int16, **kw)

    def signs(*shape):
        return (torch.randint(0, 2, shape, **kw) * 2 - 1).to(torch.float16)

    def rout(n_out, prune_counts=None):
        r = torch.rand((E, n_out), **kw) + 0.5
        r = (r * (torch.randint(0, 2, (E, n_out), **kw) * 2 - 1)).to(torch.float16)
        if prune_counts is not None:
            half = n_out // 2
            order = torch.rand((E, half), **kw).argsort(dim=1)
            rank = torch.empty_like(order)
            rank.scatter_(1, order, torch.arange(half, device=device).expand(E, half))
            mask = rank < prune_counts[:, None]
            r[:, :half][mask] = 0
            r[:, half:][mask] = 0
        return r

    d = {}
    d["Wg"] = (torch.randn((E, hidden), **kw) * 0.02).to(torch.float16)
    d["gu_codes"] = codes(hidden, 2 * inter, k_gu)
    d["dn_codes"] = codes(inter, hidden, k_dn)
    d["gu_rin"] = signs(E, hidden)
    d["dn_rin"] = signs(E, inter)
    rates = torch.rand(E, **kw) * (prune_hi - prune_lo) + prune_lo
    d["gu_rout"] = rout(2 * inter, torch.round(rates * inter).to(torch.int64))
    d["dn_rout"] = rout(hidden)
    d["sh_gu_w8"] = torch.randint(-127, 128, (2 * sh_inter, hidden), dtype=torch.int8, **kw)
    d["sh_gu_s"] = torch.rand(2 * sh_inter, **kw) * 9e-3 + 1e-3
    d["sh_dn_w8"] = torch.randint(-127, 128, (hidden, sh_inter), dtype=torch.int8, **kw)
    d["sh_dn_s"] = torch.rand(hidden, **kw) * 9e-3 + 1e-3
    d["sh_gate"] = (torch.randn(hidden, **kw) * 0.02).to(torch.float16)
    d["hidden"], d["inter"], d["n_experts"], d["sh_inter"] = hidden, inter, E, sh_inter
    d["k_gu"], d["k_dn"] = k_gu, k_dn
    return d


def projections_device(seed: int, device, P: int, n_in: int = 2048, n_out: int = 1024, K: int = 2,
                       prune_rate: float = 0.55):
    """P independent single projections (the gate_up shape by default):
    codes [P][n_in/16][n_out/16][16K], rin +-1 [P][n_in], rout = U(0.5,1.5)*+-1
    [P][n_out] with round(rate * n_out/2) channels zeroed by a mask shared by
    the gate half and the up half, x ~ N(0,1) fp16 [P][n_in]."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    kw = dict(device=device, generator=g)
    d = {"codes": torch.randint(-32768, 32768, (P, n_in // 16, n_out // 16, 16 * K), dtype=torch.int16, **kw),
         "rin": ((torch.randint(0, 2, (P, n_in), **kw) * 2 - 1).to(torch.float16))}
    r = torch.rand((P, n_out), **kw) + 0.5
    r = r * (torch.randint(0, 2, (P, n_out), **kw) * 2 - 1)
    half = n_out // 2
    prune = int(round(prune_rate * half))
    order = torch.rand((P, half), **kw).argsort(dim=1)
    mask = torch.zeros((P, half), dtype=torch.bool, device=device)
    mask.scatter_(1, order[:, :prune], True)
    r[:, :half][mask] = 0
    r[:, half:][mask] = 0
    d["rout"] = r.to(torch.float16)
    d["x"] = torch.randn((P, n_in), **kw).to(torch.float16)
    return d
