"""The pins are strong enough to catch a plausible mistake anywhere in the oracle.

Each case plants one mistake in a scratch copy of the oracle's C source (on the
CPU), builds it, and runs the oracle pin files against that build in a fresh
pytest process: at least one pin must fail. A control build of the unmodified
source must pass them all.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "kvevict_oracle.c")
HDR = os.path.join(ROOT, "oracle", "kvevict_oracle.h")
PIN_FILES = [os.path.join(ROOT, "tests", f) for f in (
    "test_oracle_schedule.py", "test_oracle_hash.py", "test_oracle_fp16_rope.py",
    "test_oracle_step.py", "test_oracle_values.py")]

# name: (text in the source, planted replacement, count of replacements or 0 = all)
MUTATIONS = {
    "rotation_sign": ("float x = ac - bs;", "float x = ac + bs;"),
    "shift_direction": (", D, -1, c, s)", ", D, 1, c, s)"),
    "rope_frequency": ("-(2.0 * (double)i) / (double)D", "-(1.0 * (double)i) / (double)D"),
    "new_row_left_out_of_normaliser": ("for (int32_t j = 0; j < n1; ++j) l += exp(logit[j] - m);",
                                       "for (int32_t j = 0; j < n1 - 1; ++j) l += exp(logit[j] - m);"),
    "attention_unnormalised": ("double attn = exp(logit[j] - m) / l;",
                               "double attn = exp(logit[j] - m);"),
    "tova_accumulates": ("if (mode == ORC_SCORE_CURRENT) score[j] = attn;",
                         "if (mode == ORC_SCORE_CURRENT) score[j] += attn;"),
    "ties_to_highest_slot": ("r[j] < r[best]", "r[j] <= r[best]"),
    "sinks_unprotected": ("for (int32_t j = n_sink; j < n - recent; ++j)",
                          "for (int32_t j = 0; j < n - recent; ++j)"),
    "recent_window_ignored": ("for (int32_t j = n_sink; j < n - recent; ++j)",
                              "for (int32_t j = n_sink; j < n; ++j)"),
    "tau_slope_reversed": ("(double)t * (tau_end - tau_init)", "(double)t * (tau_init - tau_end)"),
    "gumbel_sign": ("double g = -log(-log(u));", "double g = log(-log(u));"),
    "positions_reassigned": ("pos[j - 1] = pos[j];", "pos[j - 1] = j - 1;"),
    "prompt_diagonal_dropped": ("for (int32_t j = 0; j <= i; ++j) colsum[j] += exp(row[j] - lse);",
                                "for (int32_t j = 0; j < i; ++j) colsum[j] += exp(row[j] - lse);"),
    "fp16_ties_away_from_zero": ("rest > 0x1000u || (rest == 0x1000u && (h & 1u))",
                                 "rest >= 0x1000u"),
    "taper_slope": ("1.0 - 2.0 * (double)l", "1.0 - 1.0 * (double)l"),
    "prompt_select_takes_highest": ("while (b >= 0 && r[idx[b]] > r[v])", "while (b >= 0 && r[idx[b]] < r[v])"),
    "gumbel_u_from_53_bits": ("uint64_t k = h >> 12;", "uint64_t k = h >> 11;"),
    "gumbel_u_offset_dropped": ("double u = (double)(2 * k + 1) * 0x1p-53;",
                                "double u = (double)(2 * k) * 0x1p-53;"),
    "values_shift_up": ("memcpy(V + (size_t)(j - 1) * D, V + (size_t)j * D,",
                        "memcpy(V + (size_t)j * D, V + (size_t)(j - 1) * D,"),
    "values_not_moved": ("for (int32_t j = e + 1; j < n; ++j)\n    memcpy(V",
                         "for (int32_t j = n; j < n; ++j)\n    memcpy(V"),
    "prompt_values_from_kept_slot": ("memcpy(V + (size_t)n * D, values + (size_t)j * D,",
                                     "memcpy(V + (size_t)n * D, values + (size_t)n * D,"),
}


def _build(tmp_path, source):
    (tmp_path / "kvevict_oracle.c").write_text(source)
    shutil.copy(HDR, tmp_path / "kvevict_oracle.h")
    so = tmp_path / "liboracle_variant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                           "-ffp-contract=off", "-o", str(so), str(tmp_path / "kvevict_oracle.c"),
                           "-lm"])
    return str(so)


def _run_pins(so):
    env = dict(os.environ, KVEVICT_ORACLE_LIB=so)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        *PIN_FILES], env=env, capture_output=True, text=True, cwd=ROOT)
    return r.returncode, r.stdout[-2000:]


def test_control_build_passes_the_pins(tmp_path):
    rc, out = _run_pins(_build(tmp_path, open(SRC).read()))
    assert rc == 0, out


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(tmp_path, name):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert old in src, f"mutation site for {name} not found"
    rc, out = _run_pins(_build(tmp_path, src.replace(old, new)))
    assert rc != 0, f"no pin caught the planted mistake {name!r}"
