"""GPU parity of the trellis decode and the fused trellis GEMV against the CPU
oracle, called through the C ABI."""
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


@pytest.mark.parametrize("K", [2, 3])
def test_decode_all_65536_states_bit_exact(native, K):
    """Every state appears: with K=2 the weights t = 0, 8, 16, .. of a tile
    start on a word boundary, so their state is that word; with K=3 the
    weights t = 0, 16, 32, .. do. Words run through all 65536 values."""
    per_tile = 32 if K == 2 else 16
    n_tiles = 65536 // per_tile
    words = np.zeros((n_tiles, 16 * K), dtype=np.uint16)
    g = gen.rng(100 + K)
    words[:] = g.integers(0, 65536, size=words.shape, dtype=np.uint16)
    step = 1 if K == 2 else 3  # word index of weight t: t*K/16
    idx = np.arange(per_tile) * step
    words[:, idx] = np.arange(65536, dtype=np.uint32).reshape(n_tiles, per_tile).astype(np.uint16)
    codes = words.reshape(n_tiles // 64, 64, 16 * K)
    W = native.trellis_decode(dev(codes)).cpu().numpy().view(np.uint16)
    ref = o.decode_weights_f16(codes)
    assert np.array_equal(W, ref)
    # the controlled weights carry the whole codebook
    tiles = W.reshape(n_tiles // 64, 16, 64, 16).transpose(0, 2, 1, 3).reshape(n_tiles, 256)
    t_idx = np.arange(per_tile) * (8 if K == 2 else 16)
    got = tiles[:, t_idx].reshape(-1)
    assert np.array_equal(got, o.codebook_f16(np.arange(65536)))


@pytest.mark.parametrize("K,shape", [(2, (2048, 1024)), (3, (512, 2048)), (2, (48, 80))])
def test_decode_random_bit_exact(native, K, shape):
    n_in, n_out = shape
    codes = gen.trellis_codes(gen.rng(7 * K), n_in, n_out, K)
    W = native.trellis_decode(dev(codes)).cpu().numpy().view(np.uint16)
    assert np.array_equal(W, o.decode_weights_f16(codes))


def _gemv_case(native, n_in, n_out, K, batch, x_f32=False, seed=0):
    p = gen.projection(seed, n_in, n_out, K, batch=batch)
    x = p["x"].astype(np.float32) if x_f32 else p["x"]
    y = native.trellis_gemv(dev(p["codes"]), dev(x), dev(p["rin"]), dev(p["rout"])).cpu().numpy()
    ref = o.trellis_gemv(p["codes"], x.astype(np.float64), p["rin"].astype(np.float64),
                         p["rout"].astype(np.float64))
    return y, ref, p


def test_gemv_single_projection_gate_up_shape(native):
    """1024 x 2048 gate_up-shaped projection, K=2, batch 1 (55% prune mask)."""
    y, ref, p = _gemv_case(native, 2048, 1024, 2, 1, seed=1001)
    err = rel_err_rows(y, ref)
    assert err.max() <= TOL, err
    pruned = p["rout"] == 0
    assert pruned.sum() == 2 * 282
    assert np.all(y[0, pruned] == 0.0)
    assert np.all(y[0, ~pruned] != 0.0)


@pytest.mark.parametrize("n_in,n_out,K,batch", [
    (128, 128, 2, 1), (384, 640, 3, 1), (640, 384, 2, 3), (2048, 2048, 3, 2), (512, 2048, 2, 5),
    (1152, 256, 3, 4), (5120, 128, 2, 1), (2048, 1024, 3, 7),
])
def test_gemv_shapes(native, n_in, n_out, K, batch):
    y, ref, _ = _gemv_case(native, n_in, n_out, K, batch, seed=n_in + n_out + K + batch)
    assert rel_err_rows(y, ref).max() <= TOL


def test_gemv_f32_input(native):
    y, ref, _ = _gemv_case(native, 1024, 512, 3, 2, x_f32=True, seed=5)
    assert rel_err_rows(y, ref).max() <= TOL


def test_gemv_deterministic(native):
    p = gen.projection(77, 2048, 1024, 3, batch=1)
    args = [dev(p["codes"]), dev(p["x"]), dev(p["rin"]), dev(p["rout"])]
    a = native.trellis_gemv(*args).cpu().numpy()
    b = native.trellis_gemv(*args).cpu().numpy()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_gemv_constant_state_closed_form(native):
    """All code words zero: every weight is the state-0 value c, so y has
    rout * sqrt(128) * c * sqrt(128) * sum_blocks v[128 b] at the first channel
    of each output block and exactly 0 elsewhere."""
    n_in, n_out = 512, 256
    codes = np.zeros((n_in // 16, n_out // 16, 32), dtype=np.uint16)
    g = gen.rng(3)
    x = gen.fp16_normal(g, (1, n_in))
    rin = gen.signs(g, n_in)
    rout = gen.rout_vector(g, n_out)
    y = native.trellis_gemv(dev(codes), dev(x), dev(rin), dev(rout)).cpu().numpy()[0]
    c = o.f16_to_f64(o.codebook_f16(np.array([0])))[0]
    v = rin.astype(np.float64) * x[0].astype(np.float64)
    z = c * np.sqrt(128) * v[::128].sum()
    want = np.zeros(n_out)
    want[::128] = rout[::128].astype(np.float64) * np.sqrt(128) * z
    assert np.allclose(y, want, rtol=1e-5, atol=1e-3 * abs(want).max())
    mask = np.ones(n_out, bool)
    mask[::128] = False
    assert np.all(np.abs(y[mask]) <= 1e-4 * abs(want).max())
