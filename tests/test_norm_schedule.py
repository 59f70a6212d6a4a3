"""CPU check of the summation schedule the router grid uses for the residual
norm at one token: 128 threads, thread r holding the two partial sums of the
256-partial order (partials 2r and 2r + 1, one float2 per step), a half-warp
xor butterfly over lane offsets 8, 4, 2, 1 followed by the add of the
thread's two sums. The schedule must give, bit for bit, the sums of the
oracle's 256-partial definition (xor butterfly 16, 8, 4, 2, 1 within groups of
32 partials, group sums added in order); here it is replayed in float32 with
numpy and compared with the oracle on inputs of several magnitudes."""
import numpy as np
import pytest

from escha_synth import gen
from oracle import escha_oracle as o


def _schedule_x(v: np.ndarray, eps: float) -> np.ndarray:
    """x of one row v (f32, length H <= 2048, H % 256 == 0) by the 128-thread
    schedule; returns fp16 bit patterns."""
    H = v.shape[0]
    f32 = np.float32
    s = np.zeros((128, 2), dtype=f32)  # thread r: partials 2r (0) and 2r + 1 (1)
    for j in range(H // 256):
        for c in range(2):
            vv = v[2 * np.arange(128) + c + 256 * j].astype(f32)
            s[:, c] = (vv * vv).astype(f32) + s[:, c]
    s = s.reshape(4, 32, 2)  # warp, lane, component
    lanes = np.arange(32)
    for m in (8, 4, 2, 1):
        s = (s + s[:, lanes ^ m, :]).astype(f32)
    s0 = (s[:, :, 0] + s[:, :, 1]).astype(f32)  # [warp][lane]
    wsum = np.empty(8, dtype=f32)
    for w in range(4):
        wsum[2 * w] = s0[w, 0]
        wsum[2 * w + 1] = s0[w, 16]
    tot = wsum[0]
    for w in range(1, 8):
        tot = f32(tot + wsum[w])
    mean = f32(tot / f32(H))
    inv = f32(f32(1.0) / np.sqrt(f32(mean + f32(eps))))
    return o.f64_to_f16((v.astype(f32) * inv).astype(f32).astype(np.float64))


@pytest.mark.parametrize("H", [256, 768, 2048])
@pytest.mark.parametrize("scale", [1e-3, 1.0, 3e3])
def test_half_warp_schedule_equals_oracle_order(H, scale):
    g = gen.rng(H + int(scale * 10))
    for _ in range(4):
        h = (g.standard_normal(H) * scale * g.uniform(0.5, 2.0, H)).astype(np.float32)
        add = (g.standard_normal(H) * scale).astype(np.float32)
        v, ref_x = o.residual_rmsnorm(h[None], add[None], eps=1e-6)
        x = _schedule_x(v[0], 1e-6)
        assert np.array_equal(x, ref_x[0])


def test_schedule_detects_a_swapped_group_order():
    """The comparison is sensitive: adding the 8 group sums in another order
    changes some outputs of the same inputs."""
    g = gen.rng(7)
    diffs = 0
    for _ in range(64):
        v = (g.standard_normal(2048) * g.uniform(1e-3, 1e3, 2048)).astype(np.float32)
        _, ref_x = o.residual_rmsnorm(v[None], None, eps=1e-6)
        s = (v.reshape(8, 256) * v.reshape(8, 256)).astype(np.float32)
        # the per-partial sums in the right order, then the group totals reversed
        part = np.zeros(256, dtype=np.float32)
        for j in range(8):
            part = (s[j] + part).astype(np.float32)
        grp = part.reshape(8, 32)
        for m in (16, 8, 4, 2, 1):
            grp = (grp + grp[:, np.arange(32) ^ m]).astype(np.float32)
        tot = grp[7, 0]
        for w in range(6, -1, -1):
            tot = np.float32(tot + grp[w, 0])
        inv = np.float32(np.float32(1.0) / np.sqrt(np.float32(np.float32(tot / np.float32(2048)) + np.float32(1e-6))))
        x = o.f64_to_f16((v * inv).astype(np.float32).astype(np.float64))
        diffs += int(not np.array_equal(x, ref_x[0]))
    assert diffs > 0
