"""Plants plausible mistakes in copies of the oracle source (on the CPU) and
checks that the pins catch every one of them."""
import os

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "swa_oracle.c")

MUTANTS = {
    "window_off_by_one": ("if (j >= t - w + 1) return 1;", "if (j >= t - w) return 1;"),
    "window_short_by_one": ("if (j >= t - w + 1) return 1;", "if (j >= t - w + 2) return 1;"),
    "sinks_dropped": ("if (j < s) return 1;", "if (0) return 1;"),
    "diagonal_dropped": ("for (int64_t j = 0; j <= t; ++j) {", "for (int64_t j = 0; j < t; ++j) {"),
    "gqa_interleaved": ("int64_t kvh = hq / group;\n", "int64_t kvh = hq % Hkv;\n"),
    "scale_dropped": ("x[i] = scale * dot;", "x[i] = dot;"),
    "no_max_shift": ("x[i] = exp(x[i] - m);", "x[i] = exp(x[i]);"),
    "not_normalised": ("out[c] = acc / z;", "out[c] = acc / (z + 1e-3);"),
    "ring_wraps_wrong": ("if (ptr == w) ptr = 0;", "if (ptr == w) ptr = 1 % w;"),
    "ring_sinks_evicted": ("if (p < s) {", "if (p < 0) {"),
    "bwd_delta_dropped": ("delta += p[i] * dp[i];", "delta += 0.0 * dp[i];"),
    "bwd_dk_sign": ("dkrow[c] += scale * ds", "dkrow[c] -= scale * ds"),
    "bwd_dq_scale_dropped": ("dqrow[c] += scale * ds", "dqrow[c] += ds"),
    "bwd_dv_unweighted": ("dvrow[c] += p[i] * gout[c];", "dvrow[c] += gout[c] / n;"),
    "weights_scale_dropped": ("weights[i] = scale * dot;", "weights[i] = dot;"),
    "weights_gqa_interleaved": ("int64_t group = Hq / Hkv, kvh = hq / group;",
                                "int64_t group = Hq / Hkv, kvh = hq % Hkv;"),
    "bwd_group_first_head_only": ("hq < (kvh + 1) * group; ++hq)", "hq < kvh * group + 1; ++hq)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(before) >= 1, f"mutation anchor for {name} not found"
    mut_src = tmp_path / "mutant.c"
    mut_src.write_text(src.replace(before, after))
    so = tmp_path / "mutant.so"
    oracle.build(str(mut_src), str(so))
    lib = oracle.load(str(so))
    failures = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(lib)
        except AssertionError:
            failures.append(check.__name__)
        except (ValueError, OverflowError, FloatingPointError):
            failures.append(check.__name__)
    assert failures, f"no pin caught mutant {name}"
