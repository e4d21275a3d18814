"""The oracle's pins catch plausible mistakes.

Each case copies oracle/oracle.cpp, plants one plausible mistake (a dropped
term, a wrong sign, a wrong index, a transposed operand, an off-by-one in the
cached key range, ...), builds the copy on the CPU and runs
tests/test_oracle_pins.py against it in a subprocess.  The pins must fail for
every mutant.  Nothing here touches a GPU or the CUDA library.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.cpp")

MUTANTS = {
    "rope_sign": ("v[i] = a * c - b * s;", "v[i] = a * c + b * s;"),
    "rope_frequency": ("-2.0 * (double)i / (double)d", "-1.0 * (double)i / (double)d"),
    "rope_pairing": ("const double a = v[i], b = v[i + half];", "const double a = v[i], b = v[(i + 1) % d];"),
    "linear_transposed": ("acc[i] += xr[k] * w[i][k];", "acc[i] += xr[k] * W[k * nout + gi * 8 + i];"),
    "linear_group_offset": ("const int64_t n = gi * 8 + i < nout ? gi * 8 + i : nout - 1;",
                            "const int64_t n = gi * 8 + i + 1 < nout ? gi * 8 + i + 1 : nout - 1;"),
    "rms_mean_divisor": ("ss / (double)D + eps", "ss / (double)(D - 1) + eps"),
    "rms_no_eps": ("ss / (double)D + eps", "ss / (double)D"),
    "attention_no_scale": ("S[j] = scale * dot;", "S[j] = dot;"),
    "attention_no_max_shift": ("l += exp(S[j] - m);", "l += exp(S[j]);"),
    "online_l_without_alpha": ("*l = alpha * (*l) + rs;", "*l = (*l) + rs;"),
    "online_O_without_alpha": ("Ot[c] *= alpha;", "Ot[c] *= 1.0;"),
    "build_includes_block_keys": ("if (j < c_lo || j >= c_hi) keys.push_back(j);", "keys.push_back(j);"),
    "merge_block_off_by_one": ("for (int64_t j = t0; j < c_hi && j < t0 + bc; ++j)",
                               "for (int64_t j = t0 + 1; j < c_hi && j < t0 + bc; ++j)"),
    "alg1_fresh_rows_from_cache": ("if (genstep || row_fresh[r]) {  // attention over every key",
                                   "if (genstep) {  // attention over every key"),
    "bf16_ties_away": ("(frac == 0.5 && fmod(r, 2.0) != 0.0)", "(frac == 0.5)"),
    "softmax_argmax_last_of_ties": ("      if (zr[v] > m) {\n        m = zr[v];\n        am = v;",
                                    "      if (zr[v] >= m) {\n        m = zr[v];\n        am = v;"),
    "softmax_lse_without_max": ("lse[r] = m + log(s);", "lse[r] = log(s);"),
    "e4m3_ties_away": ("double r = nearbyint(a / step) * step;", "double r = round(a / step) * step;"),
    "quant_scale_without_qmax": ("const float sc = amax / 448.f;", "const float sc = amax;"),
    "rms_f32_no_eps": ("const float inv = (float)(1.0 / sqrt(ms + eps));",
                       "const float inv = (float)(1.0 / sqrt(ms));"),
    "e4m3_subnormal_exponent": ("ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mut = tmp_path / "oracle_mut.cpp"
    mut.write_text(src.replace(old, new))
    lib = tmp_path / "liboracle_mut.so"
    subprocess.run(["g++", "-O1", "-std=c++17", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", str(mut), "-o",
                    str(lib)], check=True)
    env = dict(os.environ, DLLM_ORACLE_LIB=str(lib), OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
