"""The oracle's pins catch plausible mistakes (CPU only).

Each case copies the oracle's C source, plants one plausible mistake (a wrong index,
an off-by-one, a dropped term, a wrong tie rule), builds it into a temporary library
and runs the relevant pin tests against it in a subprocess: at least one must fail.
The planted mistakes live only in the temporary copy.
"""

import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "kvd_oracle.c")

ATT = "tests/test_oracle_attention.py"
ACC = "tests/test_oracle_accept_beam.py"
APP = "tests/test_oracle_formats_append.py"
TINY = "tests/test_oracle_tiny_model.py"
ROPE = "tests/test_oracle_rope.py"
SEL = "tests/test_oracle_beam_select.py"
SMP = "tests/test_oracle_sample.py"

MUTANTS = [
    ("causal limit off by one", "int limit = causal ? len - nq + 1 + i : len;",
     "int limit = causal ? len - nq + i : len;", [ATT]),
    ("query head mapped to the wrong KV head", "int h = hq / group;",
     "int h = hq % n_kv_heads;", [ATT]),
    ("score scale dropped", "                    s *= scale;\n                    double w",
     "                    double w", [ATT]),
    ("beam rows mapped to the wrong window buffer", "int bk = r / rows_per_kv;",
     "int bk = r % (batch / rows_per_kv);", [ATT]),
    ("softmax normaliser dropped", "for (int d = 0; d < head_dim; ++d) o[d] /= l;",
     "for (int d = 0; d < head_dim; ++d) o[d] /= 1.0;", [ATT]),
    ("K and V swapped in the weighted sum",
     "o[d] += w * load(dtype, V, bk", "o[d] += w * load(dtype, K, bk", [ATT]),
    ("accept count one too far", "                n = i;\n                break;",
     "                n = i + 1;\n                break;", [ACC]),
    ("ties take the highest index", "return cand > best;", "return cand >= best;", [ACC]),
    ("NaN not ranked first", "if (isnan(cand)) return 1;", "if (isnan(cand)) return 0;",
     [ACC]),
    ("corrected token taken from the wrong row", "next_token[b] = amax[n];",
     "next_token[b] = amax[n > 0 ? n - 1 : 0];", [ACC]),
    ("append one slot late", "(int64_t)(len + j) * st + d;",
     "(int64_t)(len + j + 1) * st + d;", [APP]),
    ("length not advanced", "if (lens_out) lens_out[b] = len + q;",
     "if (lens_out) lens_out[b] = len;", [APP, TINY]),
    ("reorder copies one position too many", "int from = t < len ? p : r;",
     "int from = t <= len ? p : r;", [ACC]),
    ("reorder ignores the window check", "if (p < w * beam || p >= (w + 1) * beam) {",
     "if (p < 0 || p >= rows) {", [ACC]),
    ("binary16 exponent bias off by one", "mag = ldexp((double)(1024 + frac), expo - 25);",
     "mag = ldexp((double)(1024 + frac), expo - 24);", [APP]),
    ("bfloat16 subnormal scale wrong", "mag = ldexp((double)frac, -133);",
     "mag = ldexp((double)frac, -134);", [APP]),
    ("rotary pairs taken as adjacent dims", "double x1 = load(dtype, x, row + i + half);",
     "double x1 = load(dtype, x, row + (i ^ 1));", [ROPE]),
    ("rotary frequency exponent halved", "double theta = pow(base, -2.0 * i / head_dim);",
     "double theta = pow(base, -1.0 * i / head_dim);", [ROPE]),
    ("rotary sine sign flipped", "y[row + i] = x0 * cos(a) - x1 * sin(a);",
     "y[row + i] = x0 * cos(a) + x1 * sin(a);", [ROPE]),
    ("rotary position not offset by the start", "double pos = (double)((pos0 ? pos0[b] : 0) + j);",
     "double pos = (double)j;", [ROPE]),
    ("blank ids masked at every step", "            if (first_step) {\n                for (int i = 0; i < n_blank;",
     "            if (1) {\n                for (int i = 0; i < n_blank;", [SEL]),
    ("EOT not masked at the first step", "                x[eot] = -INFINITY;\n", "", [SEL]),
    ("cumulative score dropped", "score[j * kk + k] = c + lp;", "score[j * kk + k] = lp;",
     [SEL]),
    ("EOT continuations kept as live beams", "if (tok[best] == eot) {", "if (0) {", [SEL]),
    ("row tokens tie to the higher id", "(best < 0 || x[v] > x[best])) best = v;",
     "(best < 0 || x[v] >= x[best])) best = v;", [SEL]),
    ("log-softmax normaliser dropped", "lse = mx + log(sum);", "lse = mx;", [SEL]),
    ("equal scores tie to the later beam", "score[cnd] > score[best])) best = cnd;",
     "score[cnd] >= score[best])) best = cnd;", [SEL]),
    ("suppression list ignored", "else x[suppress[i]] = -INFINITY;",
     "else x[suppress[i]] = x[suppress[i]];", [SEL]),
    ("residual not clamped at zero", "w[v] = p[v] - q[v] > 0.0 ? p[v] - q[v] : 0.0;",
     "w[v] = p[v];", [SMP]),
    ("acceptance ratio inverted", "(double)r[b * k + i] * q[x] < p[x]",
     "(double)r[b * k + i] * p[x] < q[x]", [SMP]),
    ("inverse CDF boundary not strict", "if (run > u * total) return v;",
     "if (run >= u * total) return v;", [SMP]),
    ("temperature ignored", "p[v] = y / temperature;", "p[v] = y;", [SMP]),
    ("bonus token drawn from the last drafted row", "target + ((int64_t)b * (k + 1) + k) * vocab",
     "target + ((int64_t)b * (k + 1) + (k > 0 ? k - 1 : 0)) * vocab", [SMP]),
]


@pytest.mark.parametrize("name,old,new,files", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new, files):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique for {name!r}"
    mutant_c = tmp_path / "mutant.c"
    mutant_c.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared",
                    "-o", str(lib), str(mutant_c), "-lm"], check=True)
    env = dict(os.environ, KVD_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        *files], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 1, f"pins did not catch: {name}\n{r.stdout[-2000:]}"
