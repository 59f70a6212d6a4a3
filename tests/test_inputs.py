"""The seeded synthetic inputs: the same seed gives the same arrays, another
seed different ones, and the drawn values have the stated shapes, ranges and
structure (prune masks shared by the gate and up halves, +-1 input signs,
int8 range, bf16 rounding)."""
import numpy as np

from escha_synth import gen


def test_moe_layer_is_reproducible_and_seed_dependent():
    a = gen.moe_layer(77, hidden=256, inter=128, n_experts=4)
    b = gen.moe_layer(77, hidden=256, inter=128, n_experts=4)
    c = gen.moe_layer(78, hidden=256, inter=128, n_experts=4)
    for k, v in a.items():
        if isinstance(v, np.ndarray):
            assert np.array_equal(v, b[k]), k
    assert not np.array_equal(a["gu_codes"], c["gu_codes"])
    assert not np.array_equal(a["Wg"], c["Wg"])


def test_moe_layer_structure():
    d = gen.moe_layer(5, hidden=256, inter=128, n_experts=6, k_gu=3, k_dn=2)
    E, H, I = 6, 256, 128
    assert d["gu_codes"].shape == (E, H // 16, 2 * I // 16, 48) and d["gu_codes"].dtype == np.uint16
    assert d["dn_codes"].shape == (E, I // 16, H // 16, 32)
    assert set(np.unique(d["gu_rin"].astype(np.float32))) <= {-1.0, 1.0}
    for e in range(E):
        r = d["gu_rout"][e].astype(np.float32)
        gate, up = r[:I], r[I:]
        assert np.array_equal(gate == 0, up == 0)  # one prune mask for both halves
        assert (gate == 0).sum() == gen.prune_count(d["prune_rates"][e], I)
        nz = np.abs(r[r != 0])
        assert nz.min() >= 0.5 - 1e-3 and nz.max() <= 1.5 + 1e-3
    assert d["sh_gu_w8"].min() >= -127 and d["sh_gu_w8"].max() <= 127
    assert d["sh_gu_s"].min() >= 1e-3 and d["sh_gu_s"].max() <= 1e-2


def test_bf16_bits_round_to_nearest_even():
    g = gen.rng(3)
    bits = gen.bf16_normal_bits(g, (4096,))
    f = gen.rng(3).standard_normal(size=(4096,)).astype(np.float32)
    back = (bits.astype(np.uint32) << 16).view(np.float32)
    # within half a bf16 ulp of the f32 sample, and exact ties go to an even mantissa
    away = np.where(back < 0, np.float32(-np.inf), np.float32(np.inf)).astype(np.float32)
    ulp = np.abs(np.nextafter(back, away) - back).astype(np.float64) * 65536  # bf16 ulp above |back|
    assert np.all(np.abs(back.astype(np.float64) - f) <= ulp / 2 + 1e-30)
    tie = np.array([0x3F808000], dtype=np.uint32).view(np.float32)  # 1 + 2^-8: halfway, rounds to even (1.0)
    u = tie.view(np.uint32).astype(np.uint64)
    assert int(((u + ((u >> 16) & 1) + 0x7FFF) >> 16)[0]) == 0x3F80


def test_stack_k_draws_two_or_three():
    ks = [gen.stack_k(l) for l in range(40)]
    assert all(k in (2, 3) for pair in ks for k in pair)
    assert len(set(ks)) > 1
    assert ks == [gen.stack_k(l) for l in range(40)]
