"""GPU parity of the int8 w8a16 path against the CPU oracle (C ABI)."""
import numpy as np
import pytest

from escha_synth import gen
from gpu_common import TOL, dev, rel_err_rows
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


def _bf16_tensor(bits):
    return dev(bits.view(np.int16)).view(torch.bfloat16)


def _bf16_values(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_dequant_bit_exact(native):
    W = np.tile(np.arange(-128, 128, dtype=np.int8), (64, 4))
    s = gen.rng(1).uniform(1e-3, 1e-2, 64).astype(np.float32)
    got = native.int8_w8a16_dequant(dev(W), dev(s)).cpu().numpy()
    assert np.array_equal(got.view(np.uint32), o.int8_dequant(W, s).view(np.uint32))


@pytest.mark.parametrize("N,Kin,M", [(4096, 2048, 1), (2048, 4096, 1), (1000, 528, 3), (256, 2048, 8), (300, 1024, 11)])
def test_matvec_bf16(native, N, Kin, M):
    W, s = gen.int8_matrix(N + Kin, N, Kin)
    xb = gen.bf16_normal_bits(gen.rng(M), (M, Kin))
    y = native.int8_w8a16_matvec(dev(W), dev(s), _bf16_tensor(xb)).cpu().numpy()
    ref = o.int8_matvec(W, s, _bf16_values(xb))
    assert rel_err_rows(y, ref).max() <= TOL


def test_matvec_f16_and_f32(native):
    W, s = gen.int8_matrix(9, 512, 1024)
    x16 = gen.fp16_normal(gen.rng(2), (2, 1024))
    ref = o.int8_matvec(W, s, x16.astype(np.float64))
    assert rel_err_rows(native.int8_w8a16_matvec(dev(W), dev(s), dev(x16)).cpu().numpy(), ref).max() <= TOL
    x32 = x16.astype(np.float32)
    assert rel_err_rows(native.int8_w8a16_matvec(dev(W), dev(s), dev(x32)).cpu().numpy(), ref).max() <= TOL


def test_matvec_lm_head_shape_sampled_rows(native):
    """152064 x 2048 output-head shape at batch 1; the oracle checks a sample
    of 512 rows one by one."""
    N, Kin = 152064, 2048
    W, s = gen.int8_matrix(4003, N, Kin)
    xb = gen.bf16_normal_bits(gen.rng(4), (1, Kin))
    y = native.int8_w8a16_matvec(dev(W), dev(s), _bf16_tensor(xb)).cpu().numpy()[0]
    rows = gen.rng(5).choice(N, size=512, replace=False)
    ref = o.int8_matvec(W[rows], s[rows], _bf16_values(xb))[0]
    full_scale = np.abs(y).max()
    assert np.max(np.abs(y[rows] - ref)) / full_scale <= TOL


# ------------------------------------------------------- tensor-core GEMM route
# From 16 tokens on (Kin a multiple of 128) the product runs as a tcgen05 GEMM:
# int8 rows converted exactly to the activation's 16-bit type, f32 activations
# split into bf16 hi + lo.


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("N,Kin,M", [(1000, 1024, 16), (256, 2048, 300), (4096, 2048, 64), (384, 512, 517)])
def test_gemm_route(native, dtype, N, Kin, M):
    W, s = gen.int8_matrix(N * 7 + M, N, Kin)
    if dtype == "bf16":
        xb = gen.bf16_normal_bits(gen.rng(M + 1), (M, Kin))
        x, xv = _bf16_tensor(xb), _bf16_values(xb)
    else:
        x16 = gen.fp16_normal(gen.rng(M + 2), (M, Kin))
        xv = x16.astype(np.float64)
        x = dev(x16) if dtype == "f16" else dev(x16.astype(np.float32))
        if dtype == "f32":  # values that need more than 16 bits
            x32 = (x16.astype(np.float32) * np.float32(1.0009765625)).astype(np.float32)
            xv = x32.astype(np.float64)
            x = dev(x32)
    y = native.int8_w8a16_matvec(dev(W), dev(s), x).cpu().numpy()
    ref = o.int8_matvec(W, s, xv)
    assert np.all(np.isfinite(y))
    assert rel_err_rows(y, ref).max() <= TOL


def test_gemm_route_matches_gemv_route(native):
    """The same rows through the GEMM (M = 16) and the GEMV (M = 8, twice)."""
    W, s = gen.int8_matrix(77, 640, 1024)
    x16 = gen.fp16_normal(gen.rng(78), (16, 1024))
    y_gemm = native.int8_w8a16_matvec(dev(W), dev(s), dev(x16)).cpu().numpy()
    y_a = native.int8_w8a16_matvec(dev(W), dev(s), dev(x16[:8])).cpu().numpy()
    y_b = native.int8_w8a16_matvec(dev(W), dev(s), dev(x16[8:])).cpu().numpy()
    ref = o.int8_matvec(W, s, x16.astype(np.float64))
    assert rel_err_rows(y_gemm, ref).max() <= 1e-5
    assert rel_err_rows(np.concatenate([y_a, y_b]), ref).max() <= 1e-5


def test_gemm_route_lm_head_prefill_sampled(native):
    """152064 x 2048 output head at 2048 tokens (bf16): sampled rows and tokens."""
    N, Kin, M = 152064, 2048, 2048
    W, s = gen.int8_matrix(4005, N, Kin)
    xb = gen.bf16_normal_bits(gen.rng(6), (M, Kin))
    y = native.int8_w8a16_matvec(dev(W), dev(s), _bf16_tensor(xb))
    rows = gen.rng(7).choice(N, size=256, replace=False)
    toks = gen.rng(8).choice(M, size=16, replace=False)
    got = y[torch.as_tensor(toks, device=y.device)][:, torch.as_tensor(rows, device=y.device)].cpu().numpy()
    ref = o.int8_matvec(W[rows], s[rows], _bf16_values(xb[toks]))
    assert rel_err_rows(got, ref).max() <= TOL


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("N,Kin", [(777, 528), (130, 8192), (64, 12288), (1000, 1536), (33, 16)])
def test_matvec_m1_chunk_layouts(native, dtype, N, Kin):
    """Batch 1: row groups x 512-column chunks per CTA (1, 2, 3->4 chunks per
    warp), ragged last chunk, rows not a multiple of the tile."""
    W, s = gen.int8_matrix(N + 3 * Kin, N, Kin)
    g = gen.rng(Kin)
    if dtype == "bf16":
        xb = gen.bf16_normal_bits(g, (1, Kin))
        x, xv = _bf16_tensor(xb), _bf16_values(xb)
    else:
        x16 = gen.fp16_normal(g, (1, Kin))
        xv = x16.astype(np.float64)
        x = dev(x16) if dtype == "f16" else dev(x16.astype(np.float32))
    y = native.int8_w8a16_matvec(dev(W), dev(s), x).cpu().numpy()
    assert rel_err_rows(y, o.int8_matvec(W, s, xv)).max() <= TOL
