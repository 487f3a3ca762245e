"""The oracle's pins are not vacuous: plant a plausible mistake in a copy of
the oracle's C source, rebuild it, rerun the pins, and expect failures.

Each mutant is a one-line edit of ``oracle/gdn_oracle.c`` in a temporary
copy of the repository; the real oracle is never touched.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    "drop_beta": ("((double)vt[i] - sk[i]) * beta", "((double)vt[i] - sk[i])"),
    "update_sign": ("S[i * dk + j] + delta * (double)kt[j]", "S[i * dk + j] - delta * (double)kt[j]"),
    "swap_decay_order": ("if (!decay_after) {", "if (decay_after) {"),
    "transposed_state": ("const size_t src = state_base + j + dk * i;",
                         "const size_t src = state_base + i + dv * j;"),
    "swap_khead_mapping": ("vh / (nv / nk) : vh % nk", "vh % nk : vh / (nv / nk)"),
    "readout_with_key": ("acc += S[i * dk + j] * (double)qt[j];",
                         "acc += S[i * dk + j] * (double)kt[j];"),
    "drop_q_scale": ("const double y = p->q_scale * acc;", "const double y = acc;"),
    "qk_token_seq_swapped": ("const float *qt = job->q + dk * (kh + nk * (t + nt * s));",
                             "const float *qt = job->q + dk * (kh + nk * (s + nt * t));"),
    "gate_index_swapped": ("const size_t sc = vh + nv * (t + nt * s);",
                           "const size_t sc = vh + nv * (s + nt * t);"),
    "decay_after_drops_alpha": ("S[i * dk + j] = alpha * S[i * dk + j] + beta * delta",
                                "S[i * dk + j] = S[i * dk + j] + beta * delta"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(tmp_path, name):
    old, new = MUTANTS[name]
    dst = tmp_path / "repo"
    dst.mkdir()
    for d in ("oracle", "serving_gdn_decode_gb300"):
        shutil.copytree(os.path.join(ROOT, d), dst / d,
                        ignore=shutil.ignore_patterns("*.so", "__pycache__", "csrc", "*.o"))
    (dst / "tests").mkdir()
    for f in ("conftest.py", "test_oracle_pins.py"):
        shutil.copy(os.path.join(ROOT, "tests", f), dst / "tests" / f)
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), dst / "tests" / "golden")
    src = dst / "oracle" / "gdn_oracle.c"
    text = src.read_text()
    assert text.count(old) == 1, f"mutation site for {name} not found exactly once"
    src.write_text(text.replace(old, new))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_oracle_pins.py"], cwd=dst, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
