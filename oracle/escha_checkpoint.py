"""CPU oracle for the Escha-W2 checkpoint leaf contract.

TEST INFRASTRUCTURE. Only the test suite may import this module; the native
loader in ``bit_trellis_quantized_gb300`` shares no code with it.

It reads safetensors shards with Python's ``json`` and ``struct`` and states
the contract as the pages give it, one rule per check, in the order below.
Sources:

* hipfire PR #694, commit that read Escha's test suite: the required leaves
  are exactly escha_code / escha_rin / escha_rout and a missing one fails
  at load; escha_config (with s_in / s_out / bias) is optional; K comes from
  the code tensor's shape (last dimension 16 K); unknown escha_* leaves are
  rejected by name, the example being escha_rotation_theta;
* model card "EschaLabs/Qwen3.6-35B-A3B-Escha-W2", section "Format notes":
  escha_s_in / escha_s_out ship as all ones and must not be applied on top
  of rin / rout; escha_config (int32[9]) is informational;
* hipfire PR #694, commit on the dense export's biases: a layer ships its
  biases together or not at all; a half-biased layer is corrupt.

Readings where the pages are silent: a bias leaf is named ``<prefix>.bias``;
stacked experts carry a leading expert dimension on every leaf and no bias;
escha_config[1] is reported as K but never trusted (the pages call it
unreliable), so a disagreement is not an error.
"""
from __future__ import annotations

import json
import re
import struct

import numpy as np

REQUIRED = ("escha_code", "escha_rin", "escha_rout")
OPTIONAL = ("escha_s_in", "escha_s_out", "escha_config")
_SIZES = {"F64": 8, "I64": 8, "U64": 8, "F32": 4, "I32": 4, "U32": 4, "F16": 2, "BF16": 2, "I16": 2, "U16": 2,
          "I8": 1, "U8": 1, "BOOL": 1, "F8_E4M3": 1, "F8_E5M2": 1}


class ContractError(Exception):
    """kind: "io" (not a readable safetensors shard) or "contract"."""

    def __init__(self, kind: str, msg: str):
        super().__init__(msg)
        self.kind = kind


def read_header(path):
    """(tensors, data_start, file_bytes) of one shard; tensors maps a name to
    (dtype, shape, begin, end) with absolute byte offsets."""
    with open(path, "rb") as f:
        raw = f.read()
    if len(raw) < 8:
        raise ContractError("io", f"{path}: too short")
    (n,) = struct.unpack("<Q", raw[:8])
    if n == 0 or 8 + n > len(raw):
        raise ContractError("io", f"{path}: bad header length")
    try:
        hdr = json.loads(raw[8:8 + n].decode("utf-8"))
    except (UnicodeDecodeError, json.JSONDecodeError) as e:
        raise ContractError("io", f"{path}: header is not JSON ({e})")
    if not isinstance(hdr, dict):
        raise ContractError("io", f"{path}: header is not an object")
    data0 = 8 + n
    out = {}
    for name, t in hdr.items():
        if name == "__metadata__":
            continue
        try:
            dt, shape, (b, e) = t["dtype"], list(t["shape"]), t["data_offsets"]
        except (TypeError, KeyError, ValueError):
            raise ContractError("io", f"malformed entry for {name}")
        if dt not in _SIZES:
            raise ContractError("io", f"unknown dtype {dt} of {name}")
        if any((not isinstance(d, int)) or isinstance(d, bool) or d < 0 for d in shape):
            raise ContractError("io", f"bad shape of {name}")
        count = 1
        for d in shape:
            count *= d
        if not (isinstance(b, int) and isinstance(e, int)) or b < 0 or e < b or data0 + e > len(raw) or \
                e - b != count * _SIZES[dt]:
            raise ContractError("io", f"data_offsets of {name} do not match its shape")
        out[name] = (dt, tuple(shape), data0 + b, data0 + e)
    return out, raw


def _array(raw, entry):
    dt, shape, b, e = entry
    np_dt = {"F16": np.float16, "F32": np.float32, "I32": np.int32, "BF16": np.uint16}[dt]
    return np.frombuffer(raw[b:e], dtype=np_dt).reshape(shape)


def _layer_key(prefix: str) -> str:
    m = None
    for m in re.finditer(r"layers\.(\d+)\.", prefix):
        break
    return prefix[:m.end()] if m else prefix


def validate(paths):
    """The coded projections of the shards, sorted by prefix, as dicts
    (prefix, K, n_experts, in, out, has_bias, has_s_in, has_s_out,
    has_config, scales_all_ones, config_k); raises ContractError."""
    tensors, raws = {}, {}
    for i, p in enumerate(paths):
        t, raw = read_header(p)
        raws[i] = raw
        for name, entry in t.items():
            if name in tensors:
                raise ContractError("contract", f"{name} appears twice")
            tensors[name] = (i, entry)
    groups = {}
    for name in sorted(tensors):
        prefix, dot, leaf = name.rpartition(".")
        if not dot:
            prefix, leaf = "", name
        if not leaf.startswith("escha_"):
            continue
        if leaf not in REQUIRED + OPTIONAL:
            raise ContractError("contract", f"unsupported escha leaf '{leaf}' ({name})")
        if not prefix:
            raise ContractError("contract", f"escha leaf without a prefix: {name}")
        groups.setdefault(prefix, {})[leaf] = tensors[name]
    projs = []
    for prefix in sorted(groups):
        leaves = groups[prefix]
        for req in REQUIRED:
            if req not in leaves:
                raise ContractError("contract", f"{prefix} lacks the required leaf {req}")
        _, (cdt, cshape, _, _) = leaves["escha_code"]
        if cdt not in ("I16", "U16"):
            raise ContractError("contract", f"{prefix}.escha_code dtype {cdt}")
        if len(cshape) not in (3, 4):
            raise ContractError("contract", f"{prefix}.escha_code rank {len(cshape)}")
        if cshape[-1] not in (32, 48):
            raise ContractError("contract", f"{prefix}.escha_code last dimension {cshape[-1]} is not 16 K, K in 2, 3")
        K = cshape[-1] // 16
        E = cshape[0] if len(cshape) == 4 else 0
        n_in, n_out = 16 * cshape[-3], 16 * cshape[-2]
        if n_in == 0 or n_out == 0 or (len(cshape) == 4 and E == 0):
            raise ContractError("contract", f"{prefix}.escha_code has an empty grid")
        lead = (E,) if E else ()
        for leaf, n in (("escha_rin", n_in), ("escha_rout", n_out)):
            _, (dt, shape, _, _) = leaves[leaf]
            if dt != "F16" or tuple(shape) != lead + (n,):
                raise ContractError("contract", f"{prefix}.{leaf} must be F16 {lead + (n,)}")
        ones = True
        for leaf in ("escha_s_in", "escha_s_out"):
            if leaf in leaves:
                si, entry = leaves[leaf]
                if entry[0] not in ("F16", "F32", "BF16"):
                    ones = False
                    continue
                a = _array(raws[si], entry)
                if entry[0] == "BF16":
                    ones = ones and bool(np.all(a == 0x3F80))
                else:
                    ones = ones and bool(np.all(a == 1.0))
        config_k = -1
        if "escha_config" in leaves:
            si, entry = leaves["escha_config"]
            if entry[0] == "I32" and len(entry[1]) >= 1 and entry[1][-1] == 9:
                cfg = _array(raws[si], entry).reshape(-1)
                config_k = int(cfg[1]) if cfg.size >= 2 else -1  # an empty config has no K to report
        has_bias = False
        if f"{prefix}.bias" in tensors:
            _, (bdt, bshape, _, _) = tensors[f"{prefix}.bias"]
            if E or bdt not in ("F32", "F16", "BF16") or tuple(bshape) != (n_out,):
                raise ContractError("contract", f"{prefix}.bias must be a vector of {n_out} on a dense projection")
            has_bias = True
        projs.append({"prefix": prefix, "K": K, "n_experts": E, "in": n_in, "out": n_out, "has_bias": has_bias,
                      "has_s_in": "escha_s_in" in leaves, "has_s_out": "escha_s_out" in leaves,
                      "has_config": "escha_config" in leaves, "scales_all_ones": ones, "config_k": config_k})
    per_layer = {}
    for p in projs:
        if p["n_experts"]:
            continue
        per_layer.setdefault(_layer_key(p["prefix"]), []).append(p["has_bias"])
    for key, flags in per_layer.items():
        if any(flags) and not all(flags):
            raise ContractError("contract", f"layer {key} biases {sum(flags)} of its {len(flags)} coded projections")
    return projs
