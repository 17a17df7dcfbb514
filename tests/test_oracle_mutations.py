"""The oracle's pins must fail when a plausible mistake is planted in it.

Each case copies the oracle package to a temporary directory, applies one
textual mistake to oracle.c (or to the package's Python half), and runs
tests/test_oracle.py against the mutated copy in a child process: the run has
to fail.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = {
    "top-left corner": ("j > i + nk - nq", "j > i"),
    "no max shift in the weights": ("double w = exp(s[j] - m);", "double w = exp(s[j]);"),
    "alternating head map": ("h / group, i, nq", "h % jb->Hkv, i, nq"),
    "lse off by a little": ("*lse = m + log(l);", "*lse = m + log(l) + 1e-9;"),
    "varlen key offset": ("return ks->first_token + j;", "return ks->first_token + j + (ks->first_token > 0);"),
    "page slot off by one": ("return page * ks->page_size + j % ks->page_size;",
                             "return page * ks->page_size + (j + 1) % ks->page_size;"),
    "normaliser perturbed": ("out[c] /= l;", "out[c] /= (l + 1e-13);"),
    "scale dropped": ("s[j] = scale * dot;", "s[j] = dot;"),
    "empty row lse zero": ("*lse = -INFINITY;\n        return;", "*lse = 0.0;\n        return;"),
    "window left side off by one": ("j < i + nk - nq - left)", "j <= i + nk - nq - left)"),
    "window right side mirrored": ("j > i + nk - nq + right)", "j > i + nk - nq - right)"),
    "window measured from the top-left": ("j < i + nk - nq - left)", "j < i - left)"),
    "multi-query decode reads query 0 for every row": ("(((long)b * jb->Nq + i) * jb->Hq + h)",
                                                        "(((long)b * jb->Nq) * jb->Hq + h)"),
    "multi-query decode ignores causal": ("attend_row(jb->q, q_row, &ks, h / group, i, jb->Nq, len, jb->causal,",
                                          "attend_row(jb->q, q_row, &ks, h / group, i, jb->Nq, len, 0,"),
    "backward drops the row term D": ("const double ds = p[j] * (dp[j] - D);", "const double ds = p[j] * dp[j];"),
    "backward dK without the scale": ("dk_row[c] += jb->scale * ds * bf16_value(q_row[c]);",
                                      "dk_row[c] += ds * bf16_value(q_row[c]);"),
    "backward dV from dP": ("dv_row[c] += p[j] * bf16_value(g_row[c]);", "dv_row[c] += dp[j] * bf16_value(g_row[c]);"),
    "backward dQ from values": ("dq_row[c] += jb->scale * ds * bf16_value(k_row[c]);",
                                "dq_row[c] += jb->scale * ds * bf16_value(jb->v[((k_first + j) * jb->Hkv + g) * (long)d + c]);"),
    "E4M3 rounding truncates": ("const double v = rint(a / ulp) * ulp;", "const double v = floor(a / ulp) * ulp;"),
    "E4M3 subnormal spacing": ("if (ue < -6)\n        ue = -6;", "if (ue < -7)\n        ue = -7;"),
    "E4M3 exponent bias off by one": ("ldexp((double)(8 + m), e - 10)", "ldexp((double)(8 + m), e - 11)"),
    "fp8 scale for another largest code": ("amax / 448.0f", "amax / 240.0f"),
    "fp8 tiles ignore the sequence start": ("const long idx = first / 128 + b + t;", "const long idx = b + t;"),
    # the in-place append lives in the Python half of the oracle
    "append position off by one": ("pos = lens[b] - Nq + i\n", "pos = lens[b] - Nq + i + 1\n", "__init__.py"),
    "append reads seq_lens as the length before the append": ("pos = lens[b] - Nq + i\n", "pos = lens[b] + i\n",
                                                              "__init__.py"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new, *where = MUTATIONS[name]
    fname = where[0] if where else "oracle.c"
    dst = tmp_path / "oracle"
    shutil.copytree(os.path.join(ROOT, "oracle"), dst,
                    ignore=shutil.ignore_patterns("*.so", "__pycache__", "*.tmp*"))
    src = (dst / fname).read_text()
    assert old in src, f"mutation anchor not found: {old!r}"
    (dst / fname).write_text(src.replace(old, new, 1))
    env = dict(os.environ)
    env["PYTHONPATH"] = os.pathsep.join([str(tmp_path), ROOT])
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle.py")],
                       cwd=str(tmp_path), env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch: {name}\n{r.stdout[-2000:]}"
    # make sure the mutated copy (not the tree's oracle) was the one under test
    assert (dst / "liboracle.so").exists()
