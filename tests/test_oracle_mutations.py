"""The pins catch plausible mistakes in the oracle.  Each case copies the
oracle, the input generator and the pin tests into tests/_build, plants one
mistake in the copy of ptq_oracle.c, and runs test_oracle_pins.py there: at
least one pin must fail (a failure, not a build or collection error).  The
oracle in the repository is never touched."""
import os
import shutil
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

# (name, text in oracle/ptq_oracle.c, the planted replacement)
MUTATIONS = [
    ("fp16 exponent bias off by one", "v = ldexp((double)(m + 1024), e - 25);",
     "v = ldexp((double)(m + 1024), e - 24);"),
    ("fp16 subnormals scaled by 2^-23", "v = ldexp((double)m, -24);", "v = ldexp((double)m, -23);"),
    ("bf16 exponent bias off by one", "v = ldexp((double)(m + 128), e - 134);",
     "v = ldexp((double)(m + 128), e - 133);"),
    ("encode rounds down", "(256 * v + 242) / 243", "(256 * v) / 243"),
    ("padding digit 0 past the block", "int d = pos < ORC_WEIGHTS_PER_BLOCK ? t[pos] + 1 : 1;",
     "int d = pos < ORC_WEIGHTS_PER_BLOCK ? t[pos] + 1 : 0;"),
    ("definition rotation without the signs", "acc += h * (double)sb[i] * xb[i];",
     "acc += h * (double)(sb[i] * 0 + 1) * xb[i];"),
    ("digits of a byte reversed", "int pos = ORC_TRITS_PER_BYTE * j + i;",
     "int pos = ORC_TRITS_PER_BYTE * j + (ORC_TRITS_PER_BYTE - 1 - i);"),
    ("trit decoded as the digit", "t[pos] = (int8_t)(orc_peel_digit(in[j], i) - 1);",
     "t[pos] = (int8_t)(orc_peel_digit(in[j], i));"),
    ("butterfly difference reversed", "v[j + h] = a - c;", "v[j + h] = c - a;"),
    ("sign index shifted", "for (int i = 0; i < ORC_ROT; ++i) v[i] = (double)sb[i] * xb[i];",
     "for (int i = 0; i < ORC_ROT; ++i) v[i] = (double)sb[(i + 1) % ORC_ROT] * xb[i];"),
    ("rotation not normalised", "for (int i = 0; i < ORC_ROT; ++i) yb[i] = v[i] / 32.0;",
     "for (int i = 0; i < ORC_ROT; ++i) yb[i] = v[i] / 16.0;"),
    ("inverse rotation drops the sign", "xb[i] = (double)sb[i] * acc / 32.0;",
     "xb[i] = (double)(sb[i] * 0 + 1) * acc / 32.0;"),
    ("scale index shifted", "double s = orc_half_to_double(scales[n * nb + b]);",
     "double s = orc_half_to_double(scales[n * nb + (b + 1) % nb]);"),
    ("second rotation skipped", "orc_fwht_fast(h, signs_mid, h, M, I);", "(void)signs_mid;"),
    ("first rotation with the second's signs", "orc_fwht_fast(x, signs_in, xr, M, H);",
     "orc_fwht_fast(x, signs_mid, xr, M, H); (void)signs_in;"),
    ("silu with the wrong sign", "g[i] / (1.0 + exp(-g[i])) * u[i]", "g[i] / (1.0 + exp(g[i])) * u[i]"),
    ("gate and up swapped", "orc_swiglu(gu + m * 2 * I, gu + m * 2 * I + I, h + m * I, I);",
     "orc_swiglu(gu + m * 2 * I + I, gu + m * 2 * I, h + m * I, I);"),
    ("norm gain dropped", "xn[m * H + k] = xm[k] * inv * norm_w[l][k];",
     "xn[m * H + k] = xm[k] * inv * (norm_w[l][k] * 0.0 + 1.0);"),
    ("norm gain index shifted", "xn[m * H + k] = xm[k] * inv * norm_w[l][k];",
     "xn[m * H + k] = xm[k] * inv * norm_w[l][(k + 1) % H];"),
    ("layer 0's gains everywhere", "xn[m * H + k] = xm[k] * inv * norm_w[l][k];",
     "xn[m * H + k] = xm[k] * inv * norm_w[0][k];"),
    ("eps outside the root", "const double inv = 1.0 / sqrt(ss / (double)H + eps);",
     "const double inv = 1.0 / (sqrt(ss / (double)H) + eps);"),
    ("sum of squares for the mean", "const double inv = 1.0 / sqrt(ss / (double)H + eps);",
     "const double inv = 1.0 / sqrt(ss + eps);"),
    ("no residual add", "x[i] += y[i];", "x[i] = y[i];"),
    ("activations of the next token", "const double* xm = x + m * K;",
     "const double* xm = x + ((m + 1) % M) * K;"),
    ("norm of the next token's row", "const double* xm = x + m * H;",
     "const double* xm = x + ((m + 1) % M) * H;"),
    ("PQ2_0 code taken as the trit", "(2 * (i % ORC_PQ2_PER_BYTE))) & 3) - 1);",
     "(2 * (i % ORC_PQ2_PER_BYTE))) & 3));"),
    ("embedding row of the next id", "orc_unrotate_def(table + (int64_t)ids[m] * H, signs, om, 1, H);",
     "orc_unrotate_def(table + (int64_t)((ids[m] + 1) % V) * H, signs, om, 1, H);"),
    ("PTQ1_0 embedding scale of the next block",
     "orc_half_to_double(scales[v * nb + k / ORC_WEIGHTS_PER_BLOCK]);",
     "orc_half_to_double(scales[v * nb + (k / ORC_WEIGHTS_PER_BLOCK + 1) % nb]);"),
]


def _copy_tree(dst):
    os.makedirs(os.path.join(dst, "tests"))
    for pkg in ("oracle", "synth"):
        shutil.copytree(os.path.join(ROOT, pkg), os.path.join(dst, pkg),
                        ignore=shutil.ignore_patterns("*.so", "__pycache__"))
    for f in ("conftest.py", "parity.py", "test_oracle_pins.py"):
        shutil.copy(os.path.join(HERE, f), os.path.join(dst, "tests", f))
    shutil.copytree(os.path.join(HERE, "golden"), os.path.join(dst, "tests", "golden"))


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_a_planted_mistake_fails_a_pin(name, old, new):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not found")
    dst = os.path.join(HERE, "_build", f"mutant_{os.getpid()}_{MUTATIONS.index((name, old, new))}")
    if os.path.exists(dst):
        shutil.rmtree(dst)
    try:
        _copy_tree(dst)
        src = os.path.join(dst, "oracle", "ptq_oracle.c")
        text = open(src).read()
        assert text.count(old) == 1, f"the text to mutate for '{name}' is not unique"
        open(src, "w").write(text.replace(old, new))
        r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_oracle_pins.py", "-q",
                            "-p", "no:cacheprovider"], cwd=dst, capture_output=True, text=True,
                           timeout=600)
        tail = (r.stdout + r.stderr).strip().splitlines()[-1] if (r.stdout + r.stderr).strip() else ""
        assert r.returncode != 0, f"'{name}': every pin still passes ({tail})"
        assert " failed" in tail and " error" not in tail, f"'{name}': {tail}"
    finally:
        shutil.rmtree(dst, ignore_errors=True)
