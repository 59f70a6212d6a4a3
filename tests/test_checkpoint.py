"""The checkpoint leaf contract: the oracle against the pages' rules, and the
native loader (opened and read on the host, no GPU) against the oracle."""
import json
import struct

import numpy as np
import pytest

from escha_synth import ckpt, gen
from oracle import escha_checkpoint as oc


@pytest.fixture(scope="module")
def native():
    torch = pytest.importorskip("torch")  # noqa: F841 - the binding imports torch
    from bit_trellis_quantized_gb300 import native as n

    n.lib()
    return n


def _write(tmp_path, tensors, name="model.safetensors", **kw):
    p = tmp_path / name
    ckpt.write_safetensors(p, tensors, **kw)
    return str(p)


def _native_verdict(native, paths):
    try:
        c = native.Checkpoint(paths)
    except native.EschaError as e:
        return ("io" if e.code == native.ESCHA_E_IO else "contract" if e.code == native.ESCHA_E_CKPT else "other",
                str(e))
    try:
        return "ok", c.projections()
    finally:
        c.close()


def _oracle_verdict(paths):
    try:
        return "ok", oc.validate(paths)
    except oc.ContractError as e:
        return e.kind, str(e)


# ----------------------------------------------------------- oracle pins ---


def test_format_pin_hand_assembled_shard(tmp_path):
    """A shard assembled byte by byte from the format's definition: u64 LE
    header length, JSON, data."""
    hdr = json.dumps({"p.escha_code": {"dtype": "I16", "shape": [1, 1, 32], "data_offsets": [0, 64]},
                      "p.escha_rin": {"dtype": "F16", "shape": [16], "data_offsets": [64, 96]},
                      "p.escha_rout": {"dtype": "F16", "shape": [16], "data_offsets": [96, 128]},
                      "__metadata__": {"format": "pt"}}).encode()
    data = bytes(range(64)) + np.ones(16, np.float16).tobytes() + np.full(16, -1, np.float16).tobytes()
    p = tmp_path / "hand.safetensors"
    p.write_bytes(struct.pack("<Q", len(hdr)) + hdr + data)
    (proj,) = oc.validate([str(p)])
    assert (proj["prefix"], proj["K"], proj["n_experts"], proj["in"], proj["out"]) == ("p", 2, 0, 16, 16)
    t, raw = oc.read_header(str(p))
    b, e = t["p.escha_code"][2:]
    assert raw[b:e] == bytes(range(64))


def test_pages_rules_on_the_oracle(tmp_path):
    """Each rule the pages state, on a minimal projection: K from the last
    dimension; a missing required leaf fails naming it; the rotation leaf
    is rejected by name; a half-biased layer is corrupt."""
    g = gen.rng(1)
    base = ckpt.coded_projection(g, "model.layers.3.mlp.up_proj", 128, 256, 3)
    (p,) = oc.validate([_write(tmp_path, base)])
    assert p["K"] == 3 and p["in"] == 128 and p["out"] == 256
    for leaf in oc.REQUIRED:
        t = {k: v for k, v in base.items() if not k.endswith(leaf)}
        with pytest.raises(oc.ContractError, match=leaf) as ei:
            oc.validate([_write(tmp_path, t, name=f"miss_{leaf}.safetensors")])
        assert ei.value.kind == "contract"
    t = dict(base)
    t["model.layers.3.mlp.up_proj.escha_rotation_theta"] = np.zeros(4, np.float32)
    with pytest.raises(oc.ContractError, match="escha_rotation_theta"):
        oc.validate([_write(tmp_path, t, name="rot.safetensors")])
    t = dict(base)
    t.update(ckpt.coded_projection(g, "model.layers.3.mlp.gate_proj", 128, 256, 2, bias=True))
    with pytest.raises(oc.ContractError, match="biases 1 of its 2"):
        oc.validate([_write(tmp_path, t, name="half.safetensors")])


def test_scales_are_reported_not_applied(tmp_path):
    g = gen.rng(2)
    t = ckpt.coded_projection(g, "a.proj", 128, 128, 2, optional=True)
    (p,) = oc.validate([_write(tmp_path, t)])
    assert p["has_s_in"] and p["has_s_out"] and p["has_config"] and p["scales_all_ones"] and p["config_k"] == 2
    t["a.proj.escha_s_out"] = t["a.proj.escha_s_out"] * np.float16(2)
    t["a.proj.escha_config"][1] = 3  # informational: reported, not trusted
    (p,) = oc.validate([_write(tmp_path, t, name="b.safetensors")])
    assert not p["scales_all_ones"] and p["config_k"] == 3 and p["K"] == 2
