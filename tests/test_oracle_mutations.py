"""The oracle's pins catch plausible mistakes (no GPU).

Each case plants one mistake in a private copy of the C oracle (a dropped term, a wrong
sign, index or order, a missing mask or reset), rebuilds that copy and runs the pin suite
(tests/test_oracle_pins.py) against it in a subprocess: the suite must fail.  An unchanged
copy must pass, so that the failures come from the planted mistakes and nothing else.
Test infrastructure only: the copies live in pytest's temporary directory.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, text in oracle/quest_oracle.c, replacement)
MUTATIONS = [
    ("box min and max swapped",
     "mn[i] = lo;\n                    mx[i] = hi;", "mn[i] = hi;\n                    mx[i] = lo;"),
    ("box over every slot of a partial page",
     "if (n_valid > P) n_valid = P;", "n_valid = P;"),
    ("bound takes the smaller corner",
     "        u += (a > c) ? a : c;\n                    }\n                    if (u > best)",
     "        u += (a < c) ? a : c;\n                    }\n                    if (u > best)"),
    ("group reads the wrong query heads",
     "for (int h = g * G; h < (g + 1) * G; ++h) {\n                    const float* qh",
     "for (int h = g; h < g + G; ++h) {\n                    const float* qh"),
    ("group maximum lost", "if (u > best) best = u;", "best = u;"),
    ("ties to the higher page",
     "return (a->page < b->page) ? -1 : (a->page > b->page) ? 1 : 0;",
     "return (a->page > b->page) ? -1 : (a->page < b->page) ? 1 : 0;"),
    ("attention reads one slot past the length",
     "if (p * P + t >= L) break;", "if (p * P + t > L) break;"),
    ("attention without 1/sqrt(d)", "z[n_tok] = dot * inv_sqrt_d;", "z[n_tok] = dot;"),
    ("page-opening append keeps the stale box",
     "                if (slot == 0) {\n                    mn[i] = kn[i];",
     "                if (0) {\n                    mn[i] = kn[i];"),
    ("selection count off by one",
     "            for (int r = n_out; r < K; ++r) out[r] = -1;\n            count[(size_t)b * s->num_kv_heads + g] = n_out;",
     "            for (int r = n_out; r < K; ++r) out[r] = -1;\n            count[(size_t)b * s->num_kv_heads + g] = n_out > 0 ? n_out - 1 : 0;"),
    ("log-sum-exp without its maximum",
     "lse[(size_t)b * s->num_q_heads + h] = m + log(denom);",
     "lse[(size_t)b * s->num_q_heads + h] = log(denom);"),
]


def _copy(tmp_path):
    dst = tmp_path / "repo"
    ignore = shutil.ignore_patterns("_build", "__pycache__", "*.so", "*.o")
    shutil.copytree(os.path.join(ROOT, "oracle"), dst / "oracle", ignore=ignore)
    shutil.copytree(os.path.join(ROOT, "query_aware_kv_gb300"), dst / "query_aware_kv_gb300",
                    ignore=shutil.ignore_patterns("_build", "__pycache__", "csrc"))
    (dst / "tests").mkdir()
    for name in ("conftest.py", "test_oracle_pins.py"):
        shutil.copy(os.path.join(ROOT, "tests", name), dst / "tests" / name)
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), dst / "tests" / "golden")
    return dst


def _run_pins(repo):
    env = dict(os.environ, PYTHONDONTWRITEBYTECODE="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_oracle_pins.py", "-x", "-q",
                        "-p", "no:cacheprovider"], cwd=repo, env=env, capture_output=True,
                       text=True, timeout=600)
    return r.returncode, r.stdout[-2000:]


def test_unchanged_copy_passes(tmp_path):
    rc, out = _run_pins(_copy(tmp_path))
    assert rc == 0, out


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_fails_a_pin(tmp_path, name, old, new):
    repo = _copy(tmp_path)
    src = repo / "oracle" / "quest_oracle.c"
    text = src.read_text()
    assert text.count(old) == 1, f"{name}: the text to change is not unique in the oracle"
    src.write_text(text.replace(old, new))
    rc, out = _run_pins(repo)
    assert rc != 0, f"{name}: every pin still passes\n{out}"
