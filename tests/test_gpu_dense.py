"""GPU parity of the dense trellis linear (the one-expert case of the expert
kernels, with an additive output bias) and of the load-time nt-major tile
transpose, against the CPU oracle, through the C ABI."""
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


def _to_numpy_u16(t):
    return t.cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("K,n_in,n_out", [(2, 2048, 1024), (3, 128, 640), (2, 48, 80), (3, 5120, 256)])
def test_nt_major_transpose_bit_exact(native, K, n_in, n_out):
    codes = gen.trellis_codes(gen.rng(900 + K), n_in, n_out, K)
    got = _to_numpy_u16(native.codes_to_nt_major(dev(codes)))
    assert np.array_equal(got, o.codes_to_nt_major(codes))


def _dense(native, p, x, nt_major, use_bias):
    bias = dev(p["bias"]) if use_bias else None
    lin = native.DenseLinear(dev(p["codes"]), dev(p["rin"]), dev(p["rout"]), bias=bias, nt_major=nt_major)
    y = lin(dev(x)).cpu().numpy()
    torch.cuda.synchronize()
    assert lin.status() == 0
    return y


def _ref(p, x, use_bias, cols=None):
    codes, rout, bias = p["codes"], p["rout"], p["bias"]
    if cols is not None:  # whole 128-output blocks: the output transform is blockwise
        codes = codes[:, cols.start // 16:cols.stop // 16]
        rout, bias = rout[cols], bias[cols]
    return o.dense_linear(codes, x.astype(np.float64), p["rin"].astype(np.float64), rout.astype(np.float64),
                          bias=bias.astype(np.float64) if use_bias else None)


# For this 1024 x 768 weight M = 1..12 run the fused GEMV, M >= 13 the
# grouped tensor-core GEMM (items of 16, 32, 64 or 128 tokens, inputs split
# over 4 CTAs); 300 tokens leave a ragged last item of 44.
@pytest.mark.parametrize("M", [1, 3, 12, 13, 64, 300])
@pytest.mark.parametrize("nt_major", [False, True])
def test_dense_linear_matches_oracle(native, M, nt_major):
    K = 3 if M % 2 else 2
    p = gen.dense_projection(1000 + M, 1024, 768, K, M, prune_rate=0.1)
    y = _dense(native, p, p["x"], nt_major, True)
    ref = _ref(p, p["x"], True)
    assert rel_err_rows(y, ref).max() <= TOL
    pruned = p["rout"] == 0
    assert pruned.sum() == 77
    assert np.array_equal(y[:, pruned], np.broadcast_to(p["bias"][pruned], (M, pruned.sum())))


# M = 1: one tile row per warp, weights decoded before the wait on the
# preceding kernel; M = 2: the two-token GEMV; M = 40: the GEMM route
@pytest.mark.parametrize("M", [1, 2, 40])
def test_dense_linear_no_bias_f32_input(native, M):
    p = gen.dense_projection(2000 + M, 640, 384, 2, M)
    x = p["x"].astype(np.float32) * np.float32(1.37)  # not representable in fp16
    y = _dense(native, p, x, True, False)
    assert rel_err_rows(y, _ref(p, x, False)).max() <= TOL


def test_dense_linear_layouts_agree_bit_for_bit(native):
    """Both grids hold the same tiles, and the per-column accumulation order
    does not depend on where a tile sits, so the outputs are identical."""
    for M in (1, 5, 70):
        p = gen.dense_projection(3000 + M, 1024, 512, 3, M)
        a = _dense(native, p, p["x"], False, True)
        b = _dense(native, p, p["x"], True, True)
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), M


def test_dense_linear_zero_input_gives_bias(native):
    for M in (1, 20):
        p = gen.dense_projection(4000 + M, 512, 256, 2, M)
        y = _dense(native, p, np.zeros_like(p["x"]), True, True)
        assert np.array_equal(y, np.broadcast_to(p["bias"], y.shape))


def test_dense_linear_rows_independent_of_batch(native):
    """A token's output on the GEMM route does not depend on the other tokens
    of its item beyond rounding: rows of a 100-token call match the same rows
    computed in a 20-token call to the tolerance."""
    p = gen.dense_projection(5000, 1024, 512, 2, 100)
    y100 = _dense(native, p, p["x"], True, True)
    y20 = _dense(native, p, p["x"][:20].copy(), True, True)
    assert rel_err_rows(y100[:20], y20).max() <= 1e-5


@pytest.mark.parametrize("n_in,n_out,K,M", [(5120, 17408, 2, 1), (5120, 17408, 2, 3), (5120, 17408, 2, 2048),
                                             (17408, 5120, 3, 13), (17408, 5120, 3, 200)])
def test_dense_linear_full_size_sampled(native, n_in, n_out, K, M):
    """The 27B-class dense MLP shapes (gate/up 5120 -> 17408, down 17408 ->
    5120), nt-major with bias: two 128-output blocks (the first and the last)
    checked against the oracle on every token up to 32 tokens, else on 24
    sampled tokens. From 3 tokens on these shapes run the GEMM; at 3, 13
    and 200 tokens its inputs are split over several CTAs (partial sums
    reduced in order)."""
    g = gen.rng(6000 + M)
    codes = gen.trellis_codes(g, n_in, n_out, K)
    x = gen.fp16_normal(g, (M, n_in))
    rin = gen.signs(g, n_in)
    rout = gen.rout_vector(g, n_out)
    bias = (g.standard_normal(n_out) * 8.0).astype(np.float32)
    p = {"codes": codes, "rin": rin, "rout": rout, "bias": bias}
    y = _dense(native, p, x, True, True)
    rows = np.arange(M) if M <= 32 else np.sort(gen.rng(7).choice(M, 24, replace=False))
    for cols in (slice(0, 128), slice(n_out - 128, n_out)):
        ref = _ref(p, x[rows], True, cols=cols)
        assert rel_err_rows(y[rows][:, cols], ref).max() <= TOL


def test_dense_linear_rejects_bad_arguments(native):
    lib = native.lib()
    p = gen.dense_projection(7000, 256, 256, 2, 4)
    c, rin, rout = dev(p["codes"]), dev(p["rin"]), dev(p["rout"])
    x = dev(p["x"])
    y = torch.empty((4, 256), dtype=torch.float32, device="cuda")
    ws = torch.empty(lib.escha_dense_linear_workspace(256, 256, 2, 4), dtype=torch.uint8, device="cuda")
    ok = lib.escha_dense_linear(c.data_ptr(), 256, 256, 2, 1, x.data_ptr(), 1, 4, rin.data_ptr(), rout.data_ptr(),
                                None, y.data_ptr(), ws.data_ptr(), ws.numel(), None)
    assert ok == 0
    bad = [
        dict(nt_major=2),
        dict(M=0),
        dict(x_dtype=2),
        dict(ws_bytes=0),
        dict(n_in=200),
        dict(K=4),
    ]
    for b in bad:
        a = dict(n_in=256, K=2, nt_major=1, x_dtype=1, M=4, ws_bytes=ws.numel())
        a.update(b)
        r = lib.escha_dense_linear(c.data_ptr(), a["n_in"], 256, a["K"], a["nt_major"], x.data_ptr(), a["x_dtype"],
                                   a["M"], rin.data_ptr(), rout.data_ptr(), None, y.data_ptr(), ws.data_ptr(),
                                   a["ws_bytes"], None)
        assert r < 0, b
    torch.cuda.synchronize()
