"""The parity bar itself (tests/util.py), on the CPU: what it accepts and
what it rejects, so that a loosened or broken bar fails here."""
import numpy as np

import moe_synth as S
from oracle import moe_oracle as OM
from tests.util import MAX_ERR_OVER_RMS, bf16_half_ulp, err_stats


def _case():
    rng = np.random.default_rng(0)
    ref = rng.standard_normal(100000) * 2.9
    ref[0] = 19.37  # beyond 6 rms: half a bf16 ulp there (2^-4) exceeds 2e-2 rms
    rb = OM.bf16_bits_to_f64(S.f32_to_bf16_bits(ref.astype(np.float32)))
    return ref, rb


def test_correctly_rounded_output_passes():
    ref, rb = _case()
    s = err_stats(rb, ref)
    assert s["worst_err_over_bar"] < 1.0 and s["n_over_literal"] == 0


def test_other_bf16_neighbour_passes_only_where_bf16_cannot_meet_the_literal_bar():
    ref, rb = _case()
    rms = np.sqrt(np.mean(ref ** 2))
    assert bf16_half_ulp(ref[0]) > MAX_ERR_OVER_RMS * rms
    g = rb.copy()
    ulp = 2 * bf16_half_ulp(ref[0])
    g[0] = rb[0] + ulp if rb[0] < ref[0] else rb[0] - ulp  # the other bracketing bf16 value
    s = err_stats(g, ref)
    assert s["worst_err_over_bar"] < 1.0 and s["n_over_literal"] == 1
    # the same one-ulp step on an ordinary element (half ulp < 2e-2 rms) is
    # still within 2e-2 rms there, so pick an error just above the literal bar
    g2 = rb.copy()
    g2[7] = ref[7] + 1.05 * MAX_ERR_OVER_RMS * rms
    assert err_stats(g2, ref)["worst_err_over_bar"] > 1.0


def test_two_ulps_at_an_extreme_element_fail():
    ref, rb = _case()
    g = rb.copy()
    g[0] = ref[0] + 4 * bf16_half_ulp(ref[0])
    assert err_stats(g, ref)["worst_err_over_bar"] > 1.0
