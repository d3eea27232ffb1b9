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


def test_rne_bf16_values_agrees_with_the_candidate_rounding():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(50000) * 10.0 ** rng.integers(-4, 2, 50000)
    ties = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(2 + 2 ** -7), 0.0])
    x = np.concatenate([x, ties])
    assert np.array_equal(U.rne_bf16_values(x), U.bits_to_f64(U.f64_to_bf16_bits(x)))


def test_beyond_rounding():
    ulp = 2.0 ** -7                                # bf16 spacing in [1, 2); 2^-8 in [0.5, 1)
    g = np.array([1.0, 1.0, 1.0, 1.0 + ulp, -1.0, 0.0, 1.0])
    y = np.array([1.0 + ulp / 2, 1.0 + ulp, 1.0 - 2 ** -9, 1.0 + 0.5 * ulp, -(1.0 + 0.75 * ulp), 3e-3,
                  1.0 - 2 ** -8])
    got = U.beyond_rounding(g, y).tolist()
    # rounds to g (tie, inside): 0; above by ulp: ulp - ulp/2; below 1.0 the spacing is
    # 2^-8, so 1 - 2^-9 still rounds to 1 (tie to even) and 1 - 2^-8 lies 2^-9 beyond
    assert got == [0.0, ulp / 2, 0.0, 0.0, 0.75 * ulp - ulp / 2, 3e-3, 2 ** -9]


def test_embed_report_per_item_and_split():
    ref = np.ones((6, 4))
    ref_m = ref + 2 ** -10                         # the model-dtype cast moved the exact sum
    g = np.ones((6, 4))
    g[4:, 0] = 1.0 + 2 ** -7                       # one output a whole bf16 step up
    rep = U.embed_report(g, ref, ref_m, [0, 4, 6])
    assert rep["rows"] == 6 and rep["flips"] == 2
    assert abs(rep["rel"] - np.sqrt(2 * 2 ** -14 / 8)) < 1e-12
    assert rep["max_abs"] == 2 ** -7 - 2 ** -10 and rep["raw_max_abs"] == 2 ** -7
    assert rep["cast"] == 2 ** -10 and rep["out_round"] == 2 ** -10 and rep["max_y"] == 1.0
    assert rep["acc"] == 2 ** -7 - 2 ** -10 - 2 ** -8
    U.check_embed(rep)
    g[0, 0] = 1.0 + 2 ** -4 * 3                    # 0.1875 off
    try:
        U.check_embed(U.embed_report(g, ref, ref_m, [0, 4, 6]))
    except AssertionError:
        pass
    else:
        raise AssertionError("check_embed accepted an error of 0.19")


def test_half_ulp():
    assert U.bf16_half_ulp(np.array([1.0, 1.5, 4.0, 7.9, 8.0, -5.0])).tolist() == \
        [2 ** -8, 2 ** -8, 2 ** -6, 2 ** -6, 2 ** -5, 2 ** -6]
