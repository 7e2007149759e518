"""The pins must catch plausible mistakes: each case plants one mistake in a
temporary copy of the oracle's C source (on the CPU), builds it, and runs the
pin suite against it in a subprocess; the suite has to fail."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "mha_oracle.c")

MUTATIONS = [
    ("scale dropped", "s[j] = scale * dot;", "s[j] = dot;"),
    ("causal mask off by one", "if ((mask_kind & MASK_CAUSAL_BIT) && j > i)",
     "if ((mask_kind & MASK_CAUSAL_BIT) && j >= i)"),
    ("padding mask off by one", "key_lens && j >= key_lens[b]", "key_lens && j > key_lens[b]"),
    ("weights not normalised", "double w = s[j] / denom;", "double w = s[j];"),
    ("wrong exponent sign", "s[j] = exp(s[j] - m);", "s[j] = exp(m - s[j]);"),
    ("key feature index reversed", "qi[c] * kb[(size_t)j * dk + c]",
     "qi[c] * kb[(size_t)j * dk + (dk - 1 - c)]"),
    ("value row index reversed", "oi[c] += w * vb[(size_t)j * dv + c];",
     "oi[c] += w * vb[(size_t)(Tk - 1 - j) * dv + c];"),
    ("heads concatenated in reverse", "+ (size_t)hh * d, sizeof(double) * d);",
     "+ (size_t)(H - 1 - hh) * d, sizeof(double) * d);"),
    ("W^K used for the value projection", "matmul(x_kv, Wv, vp, Mk, D, H * dv);",
     "matmul(x_kv, Wk, vp, Mk, D, H * dv);"),
    ("W^O transposed", "const double *wr = W + (size_t)kk * N;\n            for (int n = 0; n < N; ++n)\n                yr[n] += a * wr[n];",
     "for (int n = 0; n < N; ++n)\n                yr[n] += a * W[(size_t)(K == N ? n * K + kk : kk * N + n)];"),
    ("layer norm with the unbiased variance", "var /= D;", "var /= (D - 1);"),
    ("layer norm without the variance's square root", "const double sigma = sqrt(var + eps);",
     "const double sigma = var + eps;"),
    ("layer norm eps outside the square root", "const double sigma = sqrt(var + eps);",
     "const double sigma = sqrt(var) + eps;"),
    ("layer norm gain and shift swapped", "* gamma[c] + beta[c];", "* beta[c] + gamma[c];"),
    ("residual left out of the normalised value", "yr[c] = (xr[c] + sr[c] - mu)",
     "yr[c] = (sr[c] - mu)"),
    ("log-sum-exp without its maximum", "lse[r] = m + log(sum);", "lse[r] = log(sum);"),
    ("log-sum-exp sum without the scale", "sum += exp(scale * dot - m);", "sum += exp(dot - m);"),
    ("backward without the softmax row term", "const double ds = p[j] * (dp[j] - pdp);",
     "const double ds = p[j] * dp[j];"),
    ("backward dQ without the scale", "dqb[(size_t)i * d + c] += scale * ds *",
     "dqb[(size_t)i * d + c] += ds *"),
    ("backward dV from dP instead of P", "dvb[(size_t)j * d + c] += p[j] * gi[c];",
     "dvb[(size_t)j * d + c] += dp[j] * gi[c];"),
    ("positional encoding sin and cos swapped", "(c % 2 == 0) ? sin(angle) : cos(angle)",
     "(c % 2 == 0) ? cos(angle) : sin(angle)"),
    ("positional encoding exponent i instead of 2i", "const int i2 = c - (c % 2); /* 2i */",
     "const int i2 = c / 2; /* 2i */"),
    ("feed-forward network without the ReLU", "hid[(size_t)r * F + f] = a > 0.0 ? a : 0.0;",
     "hid[(size_t)r * F + f] = a;"),
    ("feed-forward network output bias dropped", "y[(size_t)r * D + c] += b2[c];",
     "y[(size_t)r * D + c] += 0.0;"),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, name
    bad = tmp_path / "planted.c"
    bad.write_text(src.replace(old, new))
    lib = tmp_path / "libplanted.so"
    subprocess.check_call(["gcc", "-std=c99", "-O1", "-fopenmp", "-shared", "-fPIC", str(bad),
                           "-o", str(lib), "-lm"])
    env = dict(os.environ, MHA_ORACLE_LIB=str(lib), OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, "pins did not catch: " + name
