"""The oracle's pins catch plausible mistakes in it.

Each case plants one mistake (a dropped term, a wrong sign, index or
divisor, a swapped operand, a bound too tight for the device's documented
error) in a copy of oracle.c, compiles the copy to a
library of its own in a temporary directory, and runs the CPU pins with the
oracle loading that library (ORACLE_LIB).  At least one pin must fail; the
committed oracle.c is never touched.
"""
import os
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(ROOT, "oracle", "oracle.c")
PINS = ["test_oracle_fixed_ops.py", "test_oracle_layernorm.py", "test_oracle_rmsnorm_linear.py",
        "test_oracle_chain.py", "test_oracle_rounding.py"]

MUTATIONS = [
    ("rmsnorm mean over K-1", "    ms /= (double)hidden;\n",
     "    ms /= (double)(hidden > 1 ? hidden - 1 : 1);\n"),
    ("rmsnorm eps outside the root", "    double rstd = 1.0 / sqrt(ms + (double)eps);\n",
     "    double rstd = 1.0 / sqrt(ms) + (double)eps;\n"),
    ("rmsnorm weight dropped",
     "      y[r * hidden + k] = res_out[r * hidden + k] * rstd * load_elem(w, dt, k);\n",
     "      y[r * hidden + k] = res_out[r * hidden + k] * rstd;\n"),
    ("rope rotation sign", "          dst[out + i] = x1 * c - x2 * s;\n",
     "          dst[out + i] = x1 * c + x2 * s;\n"),
    ("rope frequency exponent", "pow(base, -2.0 * i / D)", "pow(base, -1.0 * i / D)"),
    ("rope adjacent pairs", "src + i + half);", "src + 2 * i + 1);"),
    ("layernorm unbiased variance", "    double var = s2 / (double)hidden - mean * mean;\n",
     "    double var = (s2 - (double)hidden * mean * mean) / (double)(hidden > 1 ? hidden - 1 : 1);\n"),
    ("layernorm eps outside the root", "    double s = 1.0 / sqrt(var + (double)eps);\n",
     "    double s = 1.0 / sqrt(var) + (double)eps;\n"),
    ("detect x offset sign", "              o = (2.0 * p - 0.5 + x) * strides[s];\n",
     "              o = (2.0 * p + 0.5 + x) * strides[s];\n"),
    ("detect grid axes swapped", "              o = (2.0 * p - 0.5 + y) * strides[s];\n",
     "              o = (2.0 * p - 0.5 + x) * strides[s];\n"),
    ("detect width without its square",
     "              o = (2.0 * p) * (2.0 * p) * anchors[(s * na + a) * 2 + 0];\n",
     "              o = (2.0 * p) * anchors[(s * na + a) * 2 + 0];\n"),
    ("chain sigmoid sign", "return 1.0 / (1.0 + exp(-x));", "return 1.0 / (1.0 + exp(x));"),
    ("chain check sigmoid sign", "      vn = 1.0 / (1.0 + exp(-v));", "      vn = 1.0 / (1.0 + exp(v));"),
    ("chain relu keeps -0", "case OP_RELU: return x > 0.0 ? x : 0.0;",
     "case OP_RELU: return x >= 0.0 ? x : 0.0;"),
    ("chain scale ignored", "case OP_SCALE: return x * c;", "case OP_SCALE: return x;"),
    ("shuffle direction", "int64_t co = j * groups + i, ci = i * cpg + j;",
     "int64_t co = i * cpg + j, ci = j * groups + i;"),
    ("rmsnorm residual out is x", "      res_out[r * hidden + k] = hk;\n",
     "      res_out[r * hidden + k] = load_elem(x, dt, r * hidden + k);\n"),
    ("layernorm beta dropped", "      double b = beta ? load_elem(beta, dt, k) : 0.0;",
     "      double b = 0.0;"),
    ("rope v from the k block", "        int64_t src = ((t * 3 + which) * heads + h) * (int64_t)D;",
     "        int64_t src = ((t * 3 + (which == 2 ? 1 : which)) * heads + h) * (int64_t)D;"),
    ("detect anchor w and h swapped",
     "              o = (2.0 * p) * (2.0 * p) * anchors[(s * na + a) * 2 + 0];",
     "              o = (2.0 * p) * (2.0 * p) * anchors[(s * na + a) * 2 + 1];"),
    ("detect channels anchor-minor", "            int64_t src = ((int64_t)(a * no + k) * H + y) * W + x;",
     "            int64_t src = ((int64_t)(k * na + a) * H + y) * W + x;"),
    ("rmsnorm-linear bias dropped", "      out[i * N + n] = (double)scale * (acc + b);",
     "      out[i * N + n] = (double)scale * acc;"),
    ("chain check without the exp's own error",
     "      En = vn * expm1(E) + 4 * U32 * exp(v + E) + ETA;", "      En = vn * expm1(E) + ETA;"),
    ("chain check with 3u for the sigmoid",
     "const double c = op == OP_SIGMOID ? 10.0 :", "const double c = op == OP_SIGMOID ? 3.0 :"),
    ("chain check with 1u for the exp",
     "      En = vn * expm1(E) + 4 * U32 * exp(v + E) + ETA;",
     "      En = vn * expm1(E) + 1 * U32 * exp(v + E) + ETA;"),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_a_planted_mistake_fails_a_pin(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"{name}: the line to mutate is not in oracle.c"
    mutated = tmp_path / "oracle.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "liboracle.so"
    subprocess.check_call(["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-std=c11",
                           "-shared", "-fPIC", str(mutated), "-o", str(lib), "-lm"])
    env = dict(os.environ, ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "-m", "not gpu"] + [os.path.join(HERE, f) for f in PINS],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 1, f"{name}: no pin failed\n{r.stdout[-2000:]}"
