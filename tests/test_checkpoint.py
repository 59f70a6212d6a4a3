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


def _native_outcome(native, paths):
    try:
        c = native.Checkpoint(paths)
    except native.EschaError as e:
        return ("io" if e.code == native.ESCHA_E_IO else "contract" if e.code == native.ESCHA_E_CKPT else "other",
                str(e))
    try:
        return "ok", c.projections()
    finally:
        c.close()


def _oracle_outcome(paths):
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


# ------------------------------------------------- native loader vs oracle ---


def _cases(tmp_path):
    """(name, list of shard paths): valid exports and one file per way of
    breaking the contract or the format."""
    out = []
    exp = ckpt.small_export(7)
    names = sorted(exp)
    half = len(names) // 2
    out.append(("export_one_shard", [_write(tmp_path, exp, name="one.safetensors")]))
    out.append(("export_two_shards", [_write(tmp_path, {k: exp[k] for k in names[:half]}, name="s1.safetensors"),
                                      _write(tmp_path, {k: exp[k] for k in names[half:]}, name="s2.safetensors")]))
    out.append(("duplicate_across_shards", [_write(tmp_path, exp, name="d1.safetensors"),
                                            _write(tmp_path, {names[0]: exp[names[0]]}, name="d2.safetensors")]))
    g = gen.rng(3)
    base = ckpt.coded_projection(g, "model.layers.0.mlp.down_proj", 256, 128, 2, bias=True)

    def variant(tag, edit=None, **kw):
        t = dict(base)
        if edit:
            edit(t)
        out.append((tag, [_write(tmp_path, t, name=f"{tag}.safetensors", **kw)]))

    variant("dense_biased")
    for leaf in oc.REQUIRED:
        variant(f"missing_{leaf}", lambda t, leaf=leaf: t.pop(f"model.layers.0.mlp.down_proj.{leaf}"))
    variant("rotation_theta", lambda t: t.update({"model.layers.0.mlp.down_proj.escha_rotation_theta":
                                                  np.zeros(8, np.float32)}))
    variant("unknown_escha_leaf", lambda t: t.update({"x.escha_zeta": np.zeros(2, np.float16)}))
    variant("k4_code", lambda t: t.update({"model.layers.0.mlp.down_proj.escha_code":
                                           np.zeros((16, 8, 64), np.int16)}))
    variant("f32_code", lambda t: t.update({"model.layers.0.mlp.down_proj.escha_code":
                                            np.zeros((16, 8, 32), np.float32)}))
    variant("short_rin", lambda t: t.update({"model.layers.0.mlp.down_proj.escha_rin": np.ones(128, np.float16)}))
    variant("f32_rout", lambda t: t.update({"model.layers.0.mlp.down_proj.escha_rout": np.ones(128, np.float32)}))
    variant("bad_bias_len", lambda t: t.update({"model.layers.0.mlp.down_proj.bias": np.ones(64, np.float32)}))
    variant("half_biased", lambda t: t.update(ckpt.coded_projection(gen.rng(4), "model.layers.0.mlp.up_proj",
                                                                    128, 256, 3)))
    variant("other_layer_unbiased", lambda t: t.update(ckpt.coded_projection(gen.rng(4), "model.layers.1.mlp.up_proj",
                                                                             128, 256, 3)))
    variant("bf16_bias", lambda t: t.update({"model.layers.0.mlp.down_proj.bias": np.zeros(128, np.uint16)}),
            dtypes={"model.layers.0.mlp.down_proj.bias": "BF16"})
    variant("expert_bias", lambda t: t.update(
        {**ckpt.coded_projection(gen.rng(5), "model.layers.2.mlp.experts.gate_up_proj", 128, 256, 3, experts=4),
         "model.layers.2.mlp.experts.gate_up_proj.bias": np.zeros(256, np.float32)}))
    variant("bad_offsets", header_override={"model.layers.0.mlp.down_proj.bias":
                                            {"dtype": "F32", "shape": [128], "data_offsets": [0, 100]}})
    variant("unknown_dtype", header_override={"model.layers.0.mlp.down_proj.bias":
                                              {"dtype": "Q4", "shape": [128], "data_offsets": [0, 512]}})
    # a shape whose element count wraps around 64 bits (2^33 * 2^31 * 4 bytes)
    # over an empty byte range must not pass as an empty tensor
    variant("wrapping_shape", header_override={"model.layers.0.mlp.down_proj.bias":
                                               {"dtype": "F32", "shape": [2 ** 33, 2 ** 31], "data_offsets": [0, 0]}})
    # an empty escha_config: reported as absent K, nothing read past it
    variant("empty_config", lambda t: t.update({"model.layers.0.mlp.down_proj.escha_config":
                                                np.zeros((0, 9), np.int32)}))
    bad = tmp_path / "not_json.safetensors"
    bad.write_bytes(struct.pack("<Q", 8) + b"{not js}")
    out.append(("not_json", [str(bad)]))
    out.append(("missing_file", [str(tmp_path / "absent.safetensors")]))
    return out


def test_loader_matches_oracle_on_every_case(native, tmp_path):
    expect = {"export_one_shard": "ok", "export_two_shards": "ok", "dense_biased": "ok",
              "other_layer_unbiased": "ok", "bf16_bias": "ok", "empty_config": "ok", "wrapping_shape": "io"}
    for tag, paths in _cases(tmp_path):
        if tag == "missing_file":
            ov = ("io", "")
        else:
            ov = _oracle_outcome(paths)
        nv = _native_outcome(native, paths)
        assert nv[0] == ov[0], (tag, nv, ov)
        assert ov[0] == expect.get(tag, ov[0] if ov[0] != "ok" else "error"), (tag, ov)
        if ov[0] == "ok":
            assert nv[1] == ov[1], tag
        elif tag.startswith("missing_escha") or tag in ("rotation_theta",):
            leaf = "escha_rotation_theta" if tag == "rotation_theta" else tag[len("missing_"):]
            assert leaf in nv[1] and leaf in ov[1], (tag, nv, ov)


def test_export_projections_and_raw_reads(native, tmp_path):
    exp = ckpt.small_export(11)
    path = _write(tmp_path, exp)
    c = native.Checkpoint(path)
    projs = {p["prefix"]: p for p in c.projections()}
    gu = projs["model.layers.0.mlp.experts.gate_up_proj"]
    assert (gu["K"], gu["n_experts"], gu["in"], gu["out"]) == (3, 8, 256, 256)
    assert gu["has_config"] and gu["config_k"] == 3 and gu["scales_all_ones"]
    assert projs["model.layers.0.mlp.experts.down_proj"]["K"] == 2
    dense = [p for k, p in projs.items() if k.startswith("model.layers.1.")]
    assert len(dense) == 5 and all(p["has_bias"] for p in dense)
    for name in ("model.layers.0.mlp.gate.weight", "model.layers.0.mlp.shared_expert.gate_up_proj.weight_int8",
                 "model.layers.1.mlp.up_proj.escha_code", "model.layers.1.mlp.down_proj.bias"):
        got = c.read(name)
        assert got.shape == exp[name].shape and got.tobytes() == np.ascontiguousarray(exp[name]).tobytes(), name
    with pytest.raises(native.EschaError):
        c.tensor_info("no.such.tensor")
    c.close()


def test_loader_matches_oracle_on_generated_exports(native, tmp_path):
    """Random exports (seeded draws of projection shapes, K, expert counts,
    optional leaves, biases, missing or unknown leaves, shard splits): the
    native loader and the oracle agree on every outcome and, for valid
    exports, on every projection's description."""
    rng = np.random.default_rng(20261202)
    for case in range(60):
        g = gen.rng(1000 + case)
        t = {}
        n_proj = int(rng.integers(1, 5))
        for i in range(n_proj):
            layer = int(rng.integers(0, 3))
            prefix = f"model.layers.{layer}.p{i}"
            experts = int(rng.integers(0, 3)) if rng.random() < 0.5 else 0
            n_in, n_out = 16 * int(rng.integers(1, 5)), 16 * int(rng.integers(1, 5))
            K = int(rng.integers(2, 4))
            t.update(ckpt.coded_projection(g, prefix, n_in, n_out, K, experts=experts,
                                           bias=(not experts) and rng.random() < 0.5,
                                           optional=rng.random() < 0.3))
        names = sorted(t)
        fault = rng.random()
        if fault < 0.15:
            victim = names[int(rng.integers(0, len(names)))]
            if ".escha_" in victim or victim.endswith(".bias"):
                del t[victim]
        elif fault < 0.25:
            t[names[0].rsplit(".", 1)[0] + ".escha_rotation_theta"] = np.zeros(3, np.float32)
        elif fault < 0.35:
            code = [n for n in names if n.endswith(".escha_code")][0]
            sh = list(t[code].shape)
            sh[-1] = int(rng.choice([16, 40, 64]))
            t[code] = np.zeros(sh, np.int16)
        t["model.embed_tokens.weight_int8"] = np.ones((4, 16), np.int8)
        names = sorted(t)
        if rng.random() < 0.5:
            cut = int(rng.integers(1, len(names)))
            paths = [_write(tmp_path, {k: t[k] for k in names[:cut]}, name=f"g{case}a.safetensors"),
                     _write(tmp_path, {k: t[k] for k in names[cut:]}, name=f"g{case}b.safetensors")]
        else:
            paths = [_write(tmp_path, t, name=f"g{case}.safetensors")]
        ov, nv = _oracle_outcome(paths), _native_outcome(native, paths)
        assert nv[0] == ov[0], (case, nv, ov)
        if ov[0] == "ok":
            assert nv[1] == ov[1], case
