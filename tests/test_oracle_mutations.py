"""Planted mistakes in the C++ oracle must fail its pins.

Each case copies oracle/echo_oracle.cpp with one plausible mistake planted (a
dropped term, a flipped comparison, a wrong index ...), builds it with the oracle's
own flags into a temporary library, and runs the pin suite (test_oracle_pins.py and
the prefill-bucket property pins) against it in a child process.  The pins must
fail for every planted mistake, and pass for the unmodified source.  CPU only."""

import os
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "echo_oracle.cpp")
PINS = ["tests/test_oracle_pins.py", "tests/test_oracle_cross.py::test_bucket_monotone_in_d",
        "tests/test_oracle_cross.py::test_bucket_zero_splits_the_range",
        "tests/test_oracle_cross.py::test_bucket_width_grows_with_distance_from_zero"]

# (name, text in the source, replacement)
MUTATIONS = [
    ("relu dropped", "const double relu = dot > 0.0 ? dot : 0.0;", "const double relu = dot;"),
    ("head weight dropped", "score += w[h] * relu;", "score += relu;"),
    ("ties to the higher index", "    return a < b;\n  });\n  const int64_t n = std::min(k, L);",
     "    return a > b;\n  });\n  const int64_t n = std::min(k, L);"),
    ("k-th is the best score", "*kth = n > 0 ? s[order[n - 1]] : -kInf;", "*kth = n > 0 ? s[order[0]] : -kInf;"),
    ("EMA operands swapped", "const float x = a * kth;\n  const float y = b * theta;",
     "const float x = a * theta;\n  const float y = b * kth;"),
    ("EMA ignores the first observation", "if (std::isinf(theta) && theta > 0.0f) return kth;", ""),
    ("threshold not strict", "if (scores[t] > (double)theta && !resident[t])",
     "if (scores[t] >= (double)theta && !resident[t])"),
    ("prefetch ignores residency", "if (scores[t] > (double)theta && !resident[t])", "if (scores[t] > (double)theta)"),
    ("cap keeps the last tokens", "for (int64_t t = 0; t < L && n < cap; ++t)",
     "for (int64_t t = L - 1; t >= 0 && n < cap; --t)"),
    ("cap rounds down", "const int64_t c = L >= 0 ? (L + cap_div - 1) / cap_div : -((-L) / cap_div);",
     "const int64_t c = L / cap_div;"),
    ("LRU tie to the higher host index", "return c->gpu2host[a] < c->gpu2host[b];",
     "return c->gpu2host[a] > c->gpu2host[b];"),
    ("touched-this-step slots evictable", "if (c->gpu2host[g] >= 0 && c->priority[g] < c->step) elig.push_back(g);",
     "if (c->gpu2host[g] >= 0 && c->priority[g] <= c->step) elig.push_back(g);"),
    ("selection not protected", "c->priority[g] = c->step;            /* protect: touched in this step */", ""),
    ("staged rows not bound", "for (int64_t t : staged_sorted[b]) to_bind.push_back(host_base[b] + t);", ""),
    ("no step increment", "c->step += 1;\n  for (int64_t b = 0; b < B; ++b) {\n    const int64_t h = host_base[b] + seq_len[b];\n    new_h[b] = h;",
     "for (int64_t b = 0; b < B; ++b) {\n    const int64_t h = host_base[b] + seq_len[b];\n    new_h[b] = h;"),
    ("no step increment in block mode", "c->step += 1;\n  std::vector<char> ok(B, 0);", "std::vector<char> ok(B, 0);"),
    ("12 bytes per slot", "return 4 * n_host + 13 * n_gpu;", "return 4 * n_host + 12 * n_gpu;"),
    ("value width off by one", "out[h * v_width + v] += p * c[j * D + v];", "out[h * v_width + v] += p * c[j * D + v + 1];"),
    ("no softmax scale", "logit[j] = scale * dot;\n      if (logit[j] > m) m = logit[j];",
     "logit[j] = dot;\n      if (logit[j] > m) m = logit[j];"),
    ("lse without the max", "lse[h] = m + std::log(l);", "lse[h] = std::log(l);"),
    ("negative keys not inverted", "out[i] = (u >> 31) ? ~u : (u | 0x80000000u);", "out[i] = (u >> 31) ? u : (u | 0x80000000u);"),
    ("bucket from the score, not score - prediction", "const float d = s[i] - kth_pred;", "const float d = s[i];"),
    ("threshold bucket included", "if (bk[t] > thr) cand[n++] = t;", "if (bk[t] >= thr) cand[n++] = t;"),
    ("prefill causal range short by one", "const int64_t L = pos0 + j + 1;", "const int64_t L = pos0 + j;"),
    ("adaptive cap ignores the error", "const float grow = 1.0f + pred_err;", "const float grow = 1.0f;"),
    ("adaptive cap without slack", "const int64_t c = (int64_t)std::ceil(want) + slack;",
     "const int64_t c = (int64_t)std::ceil(want);"),
    ("adaptive cap above the context rule", "return std::min(base, std::max<int64_t>(c, 0));",
     "return std::max<int64_t>(c, 0);"),
    ("prediction error relative to theta", "return d / std::fabs(kth);", "return d / std::fabs(theta);"),
    ("transfer counts the hits", "fresh += cat[b * k + j] != 0 ? 1 : 0;", "fresh += 1;"),
    ("block score from the first token", "for (int64_t t = j * T; t < std::min(L, j * T + T); ++t) m = std::max(m, scores[t]);",
     "m = scores[j * T];"),
    ("block slot taken in the middle of a block", "if (h % T != 0 || c->host2gpu[hb] >= 0) continue;",
     "if (c->host2gpu[hb] >= 0) continue;"),
    ("receiving block not touched", "if (ok[b] && c->host2gpu[new_blk[b]] >= 0) c->priority[c->host2gpu[new_blk[b]]] = c->step;",
     ";"),
    ("GQA value read from the key half", "out[g * d + e] += p * rows[j * w + d + e];",
     "out[g * d + e] += p * rows[j * w + e];"),
    ("GQA logits from the value half", "dot += q[g * d + e] * rows[j * w + e];",
     "dot += q[g * d + e] * rows[j * w + d + e];"),
    ("GQA scale dropped", "rows[j * w + e];\n      logit[j] = scale * dot;", "rows[j * w + e];\n      logit[j] = dot;"),
]


def _build(src_text: str, out_dir: str, tag: str) -> str:
    sys.path.insert(0, ROOT)
    from oracle import build as B
    src = os.path.join(out_dir, f"oracle_{tag}.cpp")
    lib = os.path.join(out_dir, f"liboracle_{tag}.so")
    with open(src, "w") as f:
        f.write(src_text)
    r = subprocess.run([B.compiler(), *B.FLAGS, src, "-o", lib], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return lib


def _run_pins(lib: str) -> subprocess.CompletedProcess:
    env = dict(os.environ, ECHO_ORACLE_LIB=lib, OMP_NUM_THREADS="2")
    return subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", "-m", "not gpu",
                           *PINS], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_every_planted_mistake_fails_a_pin():
    src = open(SRC).read()
    for name, old, new in MUTATIONS:
        assert src.count(old) == 1, f"mutation '{name}': its text must occur exactly once in the oracle"
    with tempfile.TemporaryDirectory() as d:
        jobs = [("orig", src)] + [(str(i), src.replace(old, new)) for i, (_, old, new) in enumerate(MUTATIONS)]
        with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
            libs = dict(zip([t for t, _ in jobs], ex.map(lambda j: _build(j[1], d, j[0]), jobs)))
            results = dict(zip(libs, ex.map(lambda t: _run_pins(libs[t]), libs)))
        base = results.pop("orig")
        assert base.returncode == 0, "the unmodified oracle must pass its pins:\n" + base.stdout[-2000:]
        survived = [MUTATIONS[int(t)][0] for t, r in results.items() if r.returncode == 0]
        assert not survived, f"planted mistakes that no pin caught: {survived}"
