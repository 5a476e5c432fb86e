"""The pins bite: plant a plausible mistake in a copy of the oracle and check a pin fails.

Each mutation edits a private copy of ``oracle/m3_oracle.c`` (on the CPU, in a
temporary directory), rebuilds it there and runs ``test_oracle_pins.py``
against the copy in a subprocess.  A mutation that every pin lets through
would mean the oracle is not pinned against that mistake.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

ADVANCE = "    for (int k = 0; k < K; ++k) phi[k] += dt[t] * theta[(size_t)t * K + k];\n"

MUTATIONS = {
    # trapezoid's previous-token term dropped (back to a two-term rule)
    "drop_beta": [("+ beta * prev_term + gamma * cur_term;", "+ gamma * cur_term;")],
    # beta without the decay factor alpha
    "beta_without_alpha": [("(1.0 - lam[t]) * dt[t] * alpha;", "(1.0 - lam[t]) * dt[t];")],
    # lambda and 1 - lambda exchanged
    "lambda_swapped": [("const double gamma = lam[t] * dt[t];",
                        "const double gamma = (1.0 - lam[t]) * dt[t];")],
    # rotation by +phi instead of -phi
    "rotation_sign": [("*ou = c * u + s * v;\n  *ov = -s * u + c * v;",
                       "*ou = c * u - s * v;\n  *ov = s * u + c * v;")],
    # previous token rotated by the current angle instead of its own
    "prev_token_current_angle": [(ADVANCE, ""),
                                 ("    /* 2. previous token", ADVANCE + "    /* 2. previous token")],
    # angle exclusive of the current token
    "angle_exclusive": [("    /* 4. rotate the current B_t",
                         "    for (int k = 0; k < K; ++k) phi[k] -= dt[t] * theta[(size_t)t * K + k];\n"
                         "    /* 4. rotate the current B_t")],
    # MIMO: rank columns of B and X mismatched
    "mimo_columns_mismatched": [("cur_term += Bt[r * N + n] * xcur[r * P + p];",
                                 "cur_term += Bt[((r + 1) % R) * N + n] * xcur[r * P + p];")],
    # MIMO output summed over the rank columns of C
    "mimo_output_summed": [("for (int n = 0; n < N; ++n) acc += h[(size_t)n * P + p] * Ct[r * N + n];",
                            "for (int n = 0; n < N; ++n) for (int q = 0; q < R; ++q) "
                            "acc += h[(size_t)n * P + p] * Ct[q * N + n];")],
    # previous token never remembered
    "prev_not_kept": [("memcpy(prevB, Bcur, sizeof(double) * (size_t)R * N);", "")],
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    shutil.copytree(os.path.join(ROOT, "oracle"), tmp_path / "oracle",
                    ignore=shutil.ignore_patterns("*.so", "__pycache__"))
    os.makedirs(tmp_path / "tests")
    for f in ("conftest.py", "test_oracle_pins.py"):
        shutil.copy(os.path.join(ROOT, "tests", f), tmp_path / "tests" / f)
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), tmp_path / "tests" / "golden")
    src_path = tmp_path / "oracle" / "m3_oracle.c"
    src = src_path.read_text()
    for a, b in MUTATIONS[name]:
        assert a in src, f"mutation anchor not found: {a!r}"
        src = src.replace(a, b, 1)
    src_path.write_text(src)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                        "tests/test_oracle_pins.py"], cwd=tmp_path, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode != 0 and "failed" in r.stdout, r.stdout[-2000:]
