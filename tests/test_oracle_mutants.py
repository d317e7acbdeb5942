"""The oracle's pins catch planted mistakes (CPU only).

Each case copies the oracle's C source to a temporary directory, plants one
plausible mistake (an off-by-one distance, a wrong mask boundary, a dropped or
mis-signed term, a swapped operand, a wrong sinusoid phase, a perturbed
normaliser), builds it, and runs the pin tests against that build in a
subprocess.  The real oracle is never modified.
"""

import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "txl_oracle.c")

MUTANTS = {
    "distance_off_by_one": ("const int delta = M + i - j;", "const int delta = M + i - j + 1;"),
    "mask_excludes_own_position": ("if (delta < 0) { A[j] = -INFINITY; continue; }",
                                   "if (delta <= 0 && j > 0) { A[j] = -INFINITY; continue; }"),
    "term_b_uses_key": ("const double b = dotd(qi, rd, dh);", "const double b = dotd(qi, kj, dh);"),
    "term_d_sign": ("const double d = dotd(vb, rd, dh);", "const double d = -dotd(vb, rd, dh);"),
    "term_d_dropped": ("A[j] = scale * (a + b + c + d);", "A[j] = scale * (a + b + c);"),
    "term_c_wrong_bias": ("const double c = dotd(u, kj, dh);", "const double c = dotd(vb, kj, dh);"),
    "sinusoid_phase": ("R[(size_t)p * d + 2 * k] = (double)sinl(a);",
                       "R[(size_t)p * d + 2 * k] = (double)cosl(a);"),
    "normaliser": ("oi[t] = acc / sum;", "oi[t] = acc / (sum + 1e-9);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site not found: {old}"
    mut_c = tmp_path / "mutant.c"
    mut_c.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11", "-o", str(so),
                    str(mut_c), "-lm"], check=True)
    env = dict(os.environ, TXL_ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        os.path.join(ROOT, "tests", "test_oracle_recurrence.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"


# Planted mistakes in the backward, run against its own pins.
BWD_MUTANTS = {
    "bwd_row_mean_dropped": ("G[j] = scale * P[j] * (G[j] - mean);", "G[j] = scale * P[j] * G[j];"),
    "bwd_scale_dropped": ("G[j] = scale * P[j] * (G[j] - mean);", "G[j] = P[j] * (G[j] - mean);"),
    "bwd_dq_no_position": ("dqi[t] += G[j] * (kj[t] + rd[t]);", "dqi[t] += G[j] * kj[t];"),
    "bwd_dk_no_u": ("dkj[t] += G[j] * (qi[t] + u[t]);", "dkj[t] += G[j] * qi[t];"),
    "bwd_dv_uses_score_grad": ("dvj[t] += P[j] * doi[t];", "dvj[t] += G[j] * doi[t];"),
    "bwd_dvb_uses_key": ("dvb[t] += G[j] * rd[t];", "dvb[t] += G[j] * kj[t];"),
    "bwd_drel_uses_u": ("drd[t] += G[j] * (qi[t] + vb[t]);", "drd[t] += G[j] * (qi[t] + u[t]);"),
}


@pytest.mark.parametrize("name", sorted(BWD_MUTANTS))
def test_backward_pins_reject_mutant(name, tmp_path):
    old, new = BWD_MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site not found once: {old}"
    mut_c = tmp_path / "mutant.c"
    mut_c.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11", "-o", str(so),
                    str(mut_c), "-lm"], check=True)
    env = dict(os.environ, TXL_ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_bwd.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the backward pins:\n{r.stdout[-2000:]}"
