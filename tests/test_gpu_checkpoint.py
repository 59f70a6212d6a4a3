"""GPU side of the checkpoint loader: a projection's leaves copied into device
memory (kt-major, or moved to the nt-major grid at load), biases widened to
f32, and a dense linear run on the loaded tensors against the oracle."""
import numpy as np
import pytest

from escha_synth import ckpt, gen
from gpu_common import TOL, rel_err_rows
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


def _u16(t):
    return t.cpu().numpy().view(np.uint16)


def test_load_projections_kt_and_nt_major(native, tmp_path):
    exp = ckpt.small_export(21)
    path = tmp_path / "x.safetensors"
    ckpt.write_safetensors(path, exp)
    c = native.Checkpoint(str(path))
    for i, p in enumerate(c.projections()):
        pre = p["prefix"]
        code = exp[pre + ".escha_code"].view(np.uint16)
        got = c.load_projection(i)
        assert np.array_equal(_u16(got["codes"]), code), pre
        assert np.array_equal(got["rin"].cpu().numpy(), exp[pre + ".escha_rin"])
        assert np.array_equal(got["rout"].cpu().numpy(), exp[pre + ".escha_rout"])
        if p["has_bias"]:
            assert np.array_equal(got["bias"].cpu().numpy(), exp[pre + ".bias"].astype(np.float32))
        if p["n_experts"]:
            with pytest.raises(native.EschaError):
                c.load_projection(i, nt_major=True)
        else:
            nt = c.load_projection(i, nt_major=True)
            assert np.array_equal(_u16(nt["codes"]), o.codes_to_nt_major(code)), pre
    c.close()


@pytest.mark.parametrize("bias_dtype", ["F32", "F16", "BF16"])
def test_bias_widened_to_f32(native, tmp_path, bias_dtype):
    g = gen.rng(22)
    t = ckpt.coded_projection(g, "m.layers.0.o_proj", 128, 256, 2, bias=True)
    b32 = t["m.layers.0.o_proj.bias"]
    dtypes = {}
    if bias_dtype == "F16":
        t["m.layers.0.o_proj.bias"] = b32.astype(np.float16)
        want = b32.astype(np.float16).astype(np.float32)
    elif bias_dtype == "BF16":
        bits = (b32.view(np.uint32) >> 16).astype(np.uint16)  # truncated to bf16, stored as bit patterns
        t["m.layers.0.o_proj.bias"] = bits
        dtypes = {"m.layers.0.o_proj.bias": "BF16"}
        want = (bits.astype(np.uint32) << 16).view(np.float32)
    else:
        want = b32
    path = tmp_path / "b.safetensors"
    ckpt.write_safetensors(path, t, dtypes=dtypes)
    c = native.Checkpoint(str(path))
    got = c.load_projection(0)["bias"].cpu().numpy()
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    c.close()


@pytest.mark.parametrize("M", [1, 40])
def test_dense_linear_on_loaded_tensors(native, tmp_path, M):
    exp = ckpt.small_export(23)
    path = tmp_path / "e.safetensors"
    ckpt.write_safetensors(path, exp)
    c = native.Checkpoint(str(path))
    i = [p["prefix"] for p in c.projections()].index("model.layers.1.mlp.down_proj")
    lin = native.DenseLinear.from_checkpoint(c, i, nt_major=True)
    p = c.projections()[i]
    x = gen.fp16_normal(gen.rng(24), (M, p["in"]))
    y = lin(torch.from_numpy(x).cuda()).cpu().numpy()
    pre = p["prefix"]
    ref = o.dense_linear(exp[pre + ".escha_code"].view(np.uint16), x.astype(np.float64),
                         exp[pre + ".escha_rin"].astype(np.float64), exp[pre + ".escha_rout"].astype(np.float64),
                         bias=exp[pre + ".bias"].astype(np.float64))
    assert rel_err_rows(y, ref).max() <= TOL
    c.close()


@pytest.mark.parametrize("T", [3, 20])
def test_moe_block_from_checkpoint_matches_arrays(native, tmp_path, T):
    """A MoE block built from an export (stacked coded experts, fp16 router,
    int8 shared expert) gives bit for bit the outputs of the same block built
    from the arrays, on the per-slot (3 tokens) and grouped (20) paths."""
    d = gen.moe_layer(31, hidden=512, inter=256, n_experts=16, k_gu=3, k_dn=2)
    path = tmp_path / "moe.safetensors"
    ckpt.write_safetensors(path, ckpt.moe_layer_export(d))
    c = native.Checkpoint(str(path))
    blk_c = native.MoeBlock.from_checkpoint(c, "model.layers.0.mlp", topk=4)
    blk_a = native.MoeBlock(d, topk=4)
    assert (blk_c.gu_K, blk_c.dn_K, blk_c.sh_inter) == (3, 2, 256)
    x = torch.from_numpy(gen.fp16_normal(gen.rng(32), (T, 512))).cuda()
    out_c, ids_c, w_c = blk_c(x)
    out_a, ids_a, w_a = blk_a(x)
    assert torch.equal(ids_c, ids_a) and torch.equal(w_c, w_a)
    assert torch.equal(out_c, out_a)
    c.close()
