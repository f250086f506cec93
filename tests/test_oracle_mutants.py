"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a temporary copy of ``oracle/oracle.c``
(never in the real file), builds it, and runs the oracle pin suites against
the broken library: at least one pin must fail.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "tap direction flipped": ("const int s = t - padding + k * dilation;",
                              "const int s = t + padding - k * dilation;"),
    "padding applied to x, not z": (
        "if (s < 0 || s >= L) continue;              /* zero-padded z */",
        "if (s < 0 || s >= L) { row[t] += wk * bn_eval_relu(0.0, rm[c], rv[c], gamma[c], "
        "beta[c], eps); continue; }"),
    "conv weight transposed": ("const double wk = w[((size_t)o * C + c) * K + k];",
                               "const double wk = w[((size_t)c * C + o) * K + k];"),
    "residual dropped": ("row[t] += xo[t];", "row[t] += 0.0 * xo[t];"),
    "bn mean sign": ("double y = (xv - rm)", "double y = (xv + rm)"),
    "relu dropped": ("return y > 0.0 ? y : 0.0;", "return y;"),
    "gn unbiased variance": ("const double var = ss / (double)cnt;",
                             "const double var = ss / (double)(cnt - 1);"),
    "gn strided group map": ("const int o = g * cpg + j;\n        double *yrow = yg + (size_t)j * To;\n        for (int t = 0; t < To; ++t) yrow[t] = bias",
                             "const int o = j * G + g;\n        double *yrow = yg + (size_t)j * To;\n        for (int t = 0; t < To; ++t) yrow[t] = bias"),
    "running var biased": ("momentum * var * (double)B / (double)(B - 1);",
                           "momentum * var;"),
    "divide dropped": ("double u = (v + add_bias) / divide_value;", "double u = (v + add_bias);"),
    "sigmoid sign": ("return 1.0 / (1.0 + exp(-u));", "return 1.0 / (1.0 + exp(u));"),
    "bn train uses running stats": ("mu = s / B;", "mu = running_mean ? running_mean[j] : s / B;"),
    "gn stride ignored in the taps": ("const int s = t * stride - padding + k * dilation;",
                                     "const int s = t - padding + k * dilation;"),
    "gn dilation ignored in the taps": ("const int s = t * stride - padding + k * dilation;",
                                       "const int s = t * stride - padding + k;"),
    "gn conv bias dropped": ("for (int t = 0; t < To; ++t) yrow[t] = bias ? bias[o] : 0.0;",
                             "for (int t = 0; t < To; ++t) yrow[t] = 0.0;"),
    "block train: running var biased": ("momentum * var * cnt / (cnt - 1.0);", "momentum * var;"),
    "block train: unbiased var normalizes": ("const double var = ss / cnt;",
                                             "const double var = ss / (cnt - 1.0);"),
    "block train: first sample only": ("for (int t = 0; t < L; ++t) s += xc[t];",
                                       "for (int t = 0; t < L; ++t) s += n == 0 ? N * xc[t] : 0.0;"),
    "block train: momentum swapped": (
        "running_mean[c] = (1.0 - momentum) * running_mean[c] + momentum * mu;",
        "running_mean[c] = momentum * running_mean[c] + (1.0 - momentum) * mu;"),
}


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    mutant_c = tmp_path / "oracle_mutant.c"
    mutant_c.write_text(src.replace(old, new, 1))
    so = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", str(so),
                    str(mutant_c), "-lm"], check=True)
    env = dict(os.environ, ORACLE_LIB_OVERRIDE=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "tests/test_oracle_block.py", "tests/test_oracle_block_train.py",
                        "tests/test_oracle_gn.py", "tests/test_oracle_properties.py",
                        "tests/test_oracle_linear.py"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 1, f"mutant '{name}' survived the pins:\n{r.stdout[-2000:]}"
