"""Plant plausible mistakes in copies of the oracle (CPU only) and check that
the pins catch every one of them.

Each mutant is the oracle's C source with one textual change: a dropped term,
a wrong index, a wrong sign, a wrong order inside an expert group, a wrong
group boundary, a wrong exponent bias.  A mutant that passes every pin would
mean the pins cannot tell that mistake from the real definition.
"""

import os
import subprocess
import sys

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "a2av_ref.c")

MUTANTS = {
    "sources_descending_inside_expert": (
        "for (int32_t w = 0; w < W; ++w) {\n            dst_off[w * e + j] = at;",
        "for (int32_t w = W - 1; w >= 0; --w) {\n            dst_off[w * e + j] = at;"),
    "dropped_last_k_term": (
        "for (int64_t k = 0; k < K; ++k) {",
        "for (int64_t k = 0; k + 1 < K; ++k) {"),
    "wrong_weight_column": (
        "o[n] += a * dec[wk[n]];",
        "o[n] += a * dec[wk[N - 1 - n]];"),
    "row_assigned_to_previous_group": (
        "while (i >= start + group_rows[j]) {\n            start += group_rows[j];\n            ++j;\n"
        "        }\n        expert[r] = j;",
        "while (i > start + group_rows[j] && j + 1 < e) {\n            start += group_rows[j];\n            ++j;\n"
        "        }\n        expert[r] = j;"),
    "mx_row_assigned_to_previous_group": (
        "while (i >= start + group_rows[j]) {\n            start += group_rows[j];\n            ++j;\n"
        "        }\n        double *x",
        "while (i > start + group_rows[j] && j + 1 < e) {\n            start += group_rows[j];\n            ++j;\n"
        "        }\n        double *x"),
    "fp16_exponent_bias_off_by_one": (
        "ldexp((double)(1024 + frac), expo - 25)",
        "ldexp((double)(1024 + frac), expo - 24)"),
    "fp16_sign_dropped": (
        "expo - 25);  /* (1 + frac/2^10) * 2^(expo-15) */\n    return sign ? -v : v;",
        "expo - 25);  /* (1 + frac/2^10) * 2^(expo-15) */\n    return v;"),
    "accumulator_not_cleared": ("o[n] = 0.0;", "o[n] = (n == 0);"),
    "counts_read_expert_major": (
        "int32_t c = recvCounts[w * e + j];",
        "int32_t c = recvCounts[j * W + w];"),
    "sum_rule_not_checked": ("if (total != A)\n        return REF_BAD_COUNTS;", ""),
    "first_group_weight_for_all": (
        "(row_weight_index ? row_weight_index[r] : 0)", "0"),
    "amp_tracker_kept_on_overflow": (
        "            *scale = grown;\n        *growth_tracker = 0;",
        "            *scale = grown;\n        else\n            *growth_tracker = *growth_tracker + 1;"),
    "amp_growth_one_step_late": (
        "} else if (*growth_tracker + 1 == growth_interval) {",
        "} else if (*growth_tracker == growth_interval) {"),
    "e4m3_exponent_bias_off_by_one": (
        "ldexp((double)(8 + frac), expo - 10)", "ldexp((double)(8 + frac), expo - 9)"),
    "e8m0_bias_off_by_one": ("ldexp(1.0, (int)e - 127)", "ldexp(1.0, (int)e - 128)"),
    "scale_group_index_wrong": ("[row * ng + h / group]);", "[row * ng + (h / group) / 2]);"),
    "quant_reduce_drops_last_rank": (
        "            for (int32_t w = 0; w < W; ++w) {\n                const int64_t row",
        "            for (int32_t w = 0; w + 1 < W; ++w) {\n                const int64_t row"),
    "mx_weight_scale_ignores_column": ("e8m0_value(sj[n * nb + k / 32])", "e8m0_value(sj[k / 32])"),
    "mx_weight_read_transposed": ("q_value(qw, wj[n * K + k])", "q_value(qw, wj[k * N + n])"),
    "mx_activation_scale_block_64": ("e8m0_value(sa[i * nb + k / 32])", "e8m0_value(sa[i * nb + k / 64])"),
    "mx_first_expert_weight_for_all": ("const uint8_t *wj = w + (int64_t)j * N * K;", "const uint8_t *wj = w;"),
    "amp_backoff_keeps_tracker": (
        "        *scale = *scale * backoff_factor;\n        *growth_tracker = 0;",
        "        *scale = *scale * backoff_factor;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(old, new))
    so = oracle.build(str(mut), str(tmp_path / "libmutant.so"))
    # A child process runs the pins, so that a mutant that crashes (a wrong
    # offset can read out of bounds) counts as caught without ending pytest.
    tests_dir = os.path.dirname(os.path.abspath(__file__))
    code = (
        "import sys, oracle\n"
        "from oracle_pins import ALL_PINS\n"
        f"orc = oracle.Oracle(oracle.load_from({str(so)!r}))\n"
        "caught = []\n"
        "for pin in ALL_PINS:\n"
        "    try:\n"
        "        pin(orc)\n"
        "    except (AssertionError, oracle.OracleError):\n"
        "        caught.append(pin.__name__)\n"
        "print('CAUGHT', len(caught), ' '.join(caught))\n"
        "sys.exit(0 if caught else 3)\n")
    env = dict(os.environ, PYTHONPATH=os.pathsep.join([os.path.dirname(tests_dir), tests_dir]))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=600)
    if r.returncode == 3:
        pytest.fail(f"no pin caught mutant {name}")
    # returncode 0: some pins failed; negative: the mutant crashed.
    assert r.returncode == 0 or r.returncode < 0, r.stderr[-2000:]
