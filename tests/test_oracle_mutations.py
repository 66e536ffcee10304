"""The oracle's pins must catch plausible mistakes: each case below plants one
mistake in a temporary copy of the oracle's C source (never in the repository),
builds it, and runs the pin suites against it; at least one pin has to fail."""

import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

FWD = "attention_oracle.c"
BWD = "attention_bwd_oracle.c"

# (file, exact original text, planted mistake, what it breaks)
MUTATIONS = [
    (FWD, "if (mask == ORACLE_MASK_CAUSAL) return j <= pos;",
     "if (mask == ORACLE_MASK_CAUSAL) return j < pos;", "causal mask off by one"),
    (FWD, "return j >= pos - wl && j <= pos + wr;", "return j >= pos - wr && j <= pos + wl;",
     "window bounds swapped"),
    (FWD, "        LSE[i - r0] = m + log(l);\n        if (P)", "        LSE[i - r0] = log(l);\n        if (P)",
     "LSE without the row max"),
    (FWD, "                s = jb->scale * dot;\n            }\n            srow[j] = s;",
     "                s = dot;\n            }\n            srow[j] = s;", "scale not applied"),
    (FWD, "orow[c] += p * v[j * d + c];", "orow[c] += p * v[j * d + (d - 1 - c)];",
     "value columns reversed"),
    (FWD, "const int64_t bkv = b * jb->Hk + h / (jb->H / jb->Hk);",
     "const int64_t bkv = b * jb->Hk + h % jb->Hk;", "grouped heads mapped round-robin"),
    (FWD, "            if (is_visible(i + jb->N - jb->Nq, j, jb->mask, jb->wl, jb->wr)) {\n                double dot = 0.0;\n                for (int64_t c = 0; c < d; ++c) dot += q[i * d + c] * k[j * d + c];\n                s = jb->scale * dot;\n            }\n            srow[j] = s;",
     "            if (is_visible(i, j, jb->mask, jb->wl, jb->wr)) {\n                double dot = 0.0;\n                for (int64_t c = 0; c < d; ++c) dot += q[i * d + c] * k[j * d + c];\n                s = jb->scale * dot;\n            }\n            srow[j] = s;",
     "queries not placed at the last key positions"),
    (FWD, "v = ldexp((double)(f | 0x400), e - 25);", "v = ldexp((double)(f | 0x400), e - 24);",
     "fp16 exponent bias"),
    (BWD, "const double ds = p[j] * (dp[j] - rs);", "const double ds = p[j] * dp[j];",
     "softmax Jacobian row term dropped"),
    (BWD, "dqi[c] += jb->scale * ds * k[j * d + c];", "dqi[c] += ds * k[j * d + c];",
     "dQ without the scale"),
    (BWD, "dv[j * d + c] += p[j] * dO[i * d + c];", "dv[j * d + c] += p[j] * dO[i * d + (d - 1 - c)];",
     "dO columns reversed in dV"),
    (BWD, "const int64_t bh = b * jb->H + hk * group + g;", "const int64_t bh = b * jb->H + hk + g * jb->Hk;",
     "query heads of a group interleaved"),
    (BWD, "    if (mask == 1) return j <= pos;", "    if (mask == 1) return j < pos;",
     "backward causal mask off by one"),
    (BWD, "        const int64_t pos = i + N - Nq;", "        const int64_t pos = i;",
     "backward queries not placed at the last key positions"),
    (BWD, "dk[j * d + c] += jb->scale * ds * q[i * d + c];", "dk[j * d + c] += ds * q[i * d + c];",
     "dK without the scale"),
    (BWD, "for (int64_t j = 0; j < N; ++j) p[j] /= l;", "for (int64_t j = 0; j < N; ++j) p[j] /= (l + 1.0);",
     "backward P not normalised"),
    (BWD, "    if (mask == 2) return j >= pos - wl && j <= pos + wr;",
     "    if (mask == 2) return j >= pos - wl && j < pos + wr;", "backward window right bound exclusive"),
    (FWD, "v = ldexp((double)(f | 0x80), e - 134);", "v = ldexp((double)(f | 0x80), e - 133);",
     "bf16 exponent bias"),
    (FWD, "v = ldexp((double)f, -24); /* subnormal", "v = ldexp((double)f, -23); /* subnormal",
     "fp16 subnormal scale"),
]


@pytest.mark.parametrize("mutation", MUTATIONS, ids=[m[3] for m in MUTATIONS])
def test_pins_catch_planted_mistake(mutation, tmp_path):
    fname, original, planted, _ = mutation
    pkg = tmp_path / "oracle"
    shutil.copytree(os.path.join(ROOT, "oracle"), pkg,
                    ignore=shutil.ignore_patterns("*.so", "*.so.tmp*", "__pycache__"))
    src = pkg / fname
    text = src.read_text()
    assert text.count(original) == 1, "mutation site not found exactly once"
    src.write_text(text.replace(original, planted))
    env = dict(os.environ, PYTHONPATH=f"{tmp_path}{os.pathsep}{ROOT}")
    tests = [os.path.join(ROOT, "tests", t) for t in ("test_oracle.py", "test_oracle_bwd.py")]
    r = subprocess.run([sys.executable, "-m", "pytest", *tests, "-x", "-q", "-p", "no:cacheprovider",
                        "--rootdir", str(tmp_path)], env=env, cwd=str(tmp_path),
                       capture_output=True, text=True, timeout=600)
    # the copy must have been the one under test, and a pin must have failed
    assert "failed" in r.stdout.splitlines()[-1], r.stdout[-2000:]
    assert r.returncode == 1, r.stdout[-2000:]
