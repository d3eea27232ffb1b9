"""The test-side comparison helpers are themselves checked (no GPU)."""
import numpy as np

from vit_vision_encoder_fusedinputnorm_gb300 import synth
import vitfe_testutil as U


def test_f64_to_bf16_matches_f32_rounding_on_f32_values():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(20000) * 10.0 ** rng.integers(-6, 4, 20000)).astype(np.float32)
    assert np.array_equal(U.f64_to_bf16_bits(x.astype(np.float64)), synth.f32_to_bf16_bits(x))


def test_f64_to_bf16_ties_and_near_ties():
    one = 1.0
    ulp = 2.0 ** -7                     # bf16 spacing in [1, 2)
    # exact tie between 1 and 1+ulp rounds to even (1.0); just above the tie rounds up
    assert U.f64_to_bf16_bits(np.array([one + ulp / 2]))[0] == 0x3F80
    assert U.f64_to_bf16_bits(np.array([one + ulp / 2 + 2 ** -40]))[0] == 0x3F81
    assert U.f64_to_bf16_bits(np.array([one + 1.5 * ulp]))[0] == 0x3F82       # tie -> even
    assert U.f64_to_bf16_bits(np.array([-(one + ulp / 2 + 2 ** -40)]))[0] == 0xBF81


def test_ulp_distance_across_zero():
    a = np.array([0x0001, 0x8001, 0x3F80], np.uint16)
    b = np.array([0x8001, 0x0000, 0x3F81], np.uint16)
    assert U.ulp_distance(a, b).tolist() == [2, 1, 1]


def test_embed_errors_per_item():
    ref = np.ones((6, 4))
    g = ref.copy()
    g[4:] += 0.01
    rel, mx = U.embed_errors(g, ref, [0, 4, 6])
    # half a bf16 ulp at 1.0 is 2^-8
    assert abs(rel - 0.01) < 1e-12 and abs(mx - (0.01 - 2 ** -8)) < 1e-12


def test_half_ulp():
    assert U.bf16_half_ulp(np.array([1.0, 1.5, 4.0, 7.9, 8.0, -5.0])).tolist() == \
        [2 ** -8, 2 ** -8, 2 ** -6, 2 ** -6, 2 ** -5, 2 ** -6]
