"""The oracle's pins catch plausible mistakes (CPU only).

Each mutant is a copy of oracle/coat_oracle.c with one mistake planted by a
text substitution, compiled with gcc into a temporary directory; the pin
suite is then run against it in a subprocess and must fail.  Nothing here
touches the product path or a GPU.
"""
import concurrent.futures as cf
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "coat_oracle.c")
PINS = ["tests/test_oracle_e4m3.py", "tests/test_oracle_dre.py", "tests/test_oracle_adamw.py"]

MUTANTS = {
    "un-expand with k instead of 1/k": ("pow(a, 1.0 / (double)k)", "pow(a, (double)k)"),
    "first-moment EMA coefficient halved": ("(1.0 - s->b1) * gi);", "(1.0 - s->b1) * gi * 0.5);"),
    "eps inside the square root": ("mhat / (sqrt(vhat) + s->eps)", "mhat / sqrt(vhat + s->eps)"),
    "beta1 in the second-moment EMA": ("(1.0 - s->b2) * gi * gi", "(1.0 - s->b1) * gi * gi"),
    "no bias correction of m": ("(double)m / s->bc1;", "(double)m;"),
    "no bias correction of v": ("(double)v / s->bc2;", "(double)v;"),
    "min over zeros too": ("if (a != 0.0 && a < mn)", "if (a < mn)"),
    "k formula off by 1%": ("p.k_formula = log(R) / log(mx / mn);",
                            "p.k_formula = log(R) / log(mx / mn) * 1.01;"),
    "weight decay dropped": ("+ s->wd * w));", "+ 0.0 * w));"),
    "weight decay coupled into the gradient": ("double gi = bf16_to_double(s->g[i]);",
                                               "double gi = bf16_to_double(s->g[i]) + s->wd * (double)s->w[i];"),
    "ties away from even": ("(d == best_d && (c & 1) == 0)", "(d == best_d && (c & 1) == 1)"),
    "sign dropped on dequantize": ("return (float)(d < 0.0 ? -r : r);", "return (float)r;"),
    "scale without the exponent": ("p.S32 = (float)(pow(mx, (double)p.k32) / ORACLE_DELTA_MAX);",
                                   "p.S32 = (float)(mx / ORACLE_DELTA_MAX);"),
    "cap at 16": ("#define ORACLE_K_CAP 8.0", "#define ORACLE_K_CAP 16.0"),
    "subnormal decode off by one exponent": ("mag = ldexp((double)mant / 8.0, -6);",
                                             "mag = ldexp((double)mant / 8.0, -7);"),
    "S guard dropped": ("if (bound < k)\n            k = bound;\n    } else if", "if (0)\n            k = bound;\n    } else if"),
}


def _run_mutant(name, old, new, tmp):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {name}"
    d = os.path.join(tmp, "m%d" % abs(hash(name)))
    os.makedirs(d, exist_ok=True)
    c = os.path.join(d, "coat_oracle.c")
    with open(c, "w") as fh:
        fh.write(src.replace(old, new, 1))
    so = os.path.join(d, "lib.so")
    subprocess.run(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
                    "-D_GNU_SOURCE", "-o", so, c, "-lm"], check=True)
    env = dict(os.environ, COAT_ORACLE_LIB=so)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        *PINS], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return name, r.returncode


def test_pins_reject_every_mutant(tmp_path):
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
        futs = [ex.submit(_run_mutant, n, o, w, str(tmp_path)) for n, (o, w) in MUTANTS.items()]
        results = dict(f.result() for f in futs)
    survived = [n for n, rc in results.items() if rc == 0]
    assert not survived, f"mutants not caught by the pins: {survived}"
