"""Seeded synthetic safetensors shards in the layout of an Escha-W2 export.

A shard is written from its definition: an 8-byte little-endian header
length, a JSON header {name: {"dtype", "shape", "data_offsets"}} (offsets
relative to the data, tensors laid out back to back in the order given),
padded with spaces to a multiple of 8 bytes, then the data. Nothing here
does any of the method's arithmetic; the tensors come from ``gen``.

Tensor names follow the pages' module names (``mlp.experts``, ``mlp.gate``,
``mlp.{gate,up,down}_proj``, ``self_attn.{q,k,v,o}_proj``) with the escha
leaves ``escha_code``, ``escha_rin``, ``escha_rout`` (plus the optional
``escha_s_in``, ``escha_s_out``, ``escha_config``) and ``bias``.
"""
from __future__ import annotations

import json
import struct

import numpy as np

from . import gen

_DT = {np.dtype(np.float16): "F16", np.dtype(np.float32): "F32", np.dtype(np.float64): "F64",
       np.dtype(np.int8): "I8", np.dtype(np.uint8): "U8", np.dtype(np.int16): "I16", np.dtype(np.uint16): "U16",
       np.dtype(np.int32): "I32", np.dtype(np.int64): "I64"}


def write_safetensors(path, tensors: dict, metadata: dict | None = None, dtypes: dict | None = None,
                      header_override: dict | None = None) -> None:
    """Write ``tensors`` (name -> numpy array) as one shard. ``dtypes`` maps
    a name to a dtype string other than the array's own (e.g. "BF16" for
    uint16 bit patterns); ``header_override`` replaces header entries as
    given (used to write deliberately broken files)."""
    dtypes = dtypes or {}
    header, blobs, off = {}, [], 0
    for name, a in tensors.items():
        a = np.ascontiguousarray(a)
        b = a.tobytes()
        header[name] = {"dtype": dtypes.get(name, _DT[a.dtype]), "shape": list(a.shape),
                        "data_offsets": [off, off + len(b)]}
        blobs.append(b)
        off += len(b)
    if metadata is not None:
        header["__metadata__"] = metadata
    if header_override:
        header.update(header_override)
    h = json.dumps(header).encode()
    h += b" " * ((-len(h)) % 8)
    with open(path, "wb") as f:
        f.write(struct.pack("<Q", len(h)))
        f.write(h)
        for b in blobs:
            f.write(b)


def coded_projection(g: np.random.Generator, prefix: str, n_in: int, n_out: int, K: int, experts: int = 0,
                     bias: bool = False, optional: bool = False) -> dict:
    """The leaves of one coded projection (stacked experts when ``experts``)."""
    lead = (experts,) if experts else ()
    t = {
        f"{prefix}.escha_code": gen.trellis_codes(g, n_in, n_out, K, lead=lead).view(np.int16),
        f"{prefix}.escha_rin": gen.signs(g, lead + (n_in,)),
        f"{prefix}.escha_rout": (g.uniform(0.5, 1.5, size=lead + (n_out,)) * gen.signs(g, lead + (n_out,))).astype(
            np.float16),
    }
    if optional:
        t[f"{prefix}.escha_s_in"] = np.ones(lead + (n_in,), dtype=np.float16)
        t[f"{prefix}.escha_s_out"] = np.ones(lead + (n_out,), dtype=np.float16)
        cfg = np.zeros(lead + (9,), dtype=np.int32)
        cfg[..., 1] = K
        t[f"{prefix}.escha_config"] = cfg
    if bias:
        t[f"{prefix}.bias"] = (g.standard_normal(n_out) * 8.0).astype(np.float32)
    return t


def small_export(seed: int, hidden: int = 256, inter: int = 128, n_experts: int = 8, dense_inter: int = 384) -> dict:
    """A two-layer export: layer 0 a MoE block (stacked gate_up K=3 and down
    K=2 experts, fp16 router, int8 shared expert), layer 1 dense coded
    attention and MLP projections with biases. name -> array."""
    g = gen.rng(seed)
    t = {}
    t.update(coded_projection(g, "model.layers.0.mlp.experts.gate_up_proj", hidden, 2 * inter, 3, experts=n_experts,
                              optional=True))
    t.update(coded_projection(g, "model.layers.0.mlp.experts.down_proj", inter, hidden, 2, experts=n_experts))
    t["model.layers.0.mlp.gate.weight"] = gen.fp16_normal(g, (n_experts, hidden), std=0.02)
    W8, s = gen.int8_matrix(seed + 1, 2 * inter, hidden)
    t["model.layers.0.mlp.shared_expert.gate_up_proj.weight_int8"] = W8
    t["model.layers.0.mlp.shared_expert.gate_up_proj.weight_scale"] = s
    for name, (i, o, K) in {"self_attn.q_proj": (hidden, hidden, 2), "self_attn.o_proj": (hidden, hidden, 2),
                            "mlp.gate_proj": (hidden, dense_inter, 2), "mlp.up_proj": (hidden, dense_inter, 3),
                            "mlp.down_proj": (dense_inter, hidden, 3)}.items():
        t.update(coded_projection(g, f"model.layers.1.{name}", i, o, K, bias=True))
    return t


def moe_layer_export(d: dict, prefix: str = "model.layers.0.mlp") -> dict:
    """The tensors of one MoE block (a ``gen.moe_layer`` dict) under export
    names: stacked expert projections as coded leaves, the fp16 router
    ``gate.weight``, the int8 shared expert (``weight_int8`` with an f32
    ``weight_scale`` per row) and its fp16 sigmoid gate."""
    t = {
        f"{prefix}.experts.gate_up_proj.escha_code": d["gu_codes"].view(np.int16),
        f"{prefix}.experts.gate_up_proj.escha_rin": d["gu_rin"],
        f"{prefix}.experts.gate_up_proj.escha_rout": d["gu_rout"],
        f"{prefix}.experts.down_proj.escha_code": d["dn_codes"].view(np.int16),
        f"{prefix}.experts.down_proj.escha_rin": d["dn_rin"],
        f"{prefix}.experts.down_proj.escha_rout": d["dn_rout"],
        f"{prefix}.gate.weight": d["Wg"],
    }
    if d.get("sh_inter"):
        t[f"{prefix}.shared_expert.gate_up_proj.weight_int8"] = d["sh_gu_w8"]
        t[f"{prefix}.shared_expert.gate_up_proj.weight_scale"] = d["sh_gu_s"]
        t[f"{prefix}.shared_expert.down_proj.weight_int8"] = d["sh_dn_w8"]
        t[f"{prefix}.shared_expert.down_proj.weight_scale"] = d["sh_dn_s"]
        t[f"{prefix}.shared_expert_gate.weight"] = d["sh_gate"]
    return t
