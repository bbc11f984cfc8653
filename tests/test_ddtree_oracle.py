"""The DDTree construction / acceptance oracle against its pins, and planted
mistakes in copies of it that some pin must catch (no GPU needed).

A mutant is a text edit of oracle/ddtree.py loaded from a temporary file in a
child process (a mutant may loop or fail in any way without taking the test
runner down).  The committed oracle is never modified.
"""
import os
import subprocess
import sys

import pytest

from oracle import ddtree
from tests import ddtree_pins as pins

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(ddtree)


MUTANTS = {
    "child_logp_wrong_depth": [("score[i] + lp[d, k]", "score[i] + lp[d - 1, k]")],
    "score_not_accumulated": [("np.float32(score[i] + lp[d, k])", "np.float32(lp[d, k])")],
    "best_is_lowest_score": [("key=lambda c: (-c[0], c[1])", "key=lambda c: (c[0], c[1])")],
    "ties_to_larger_ranks": [("key=lambda c: (-c[0], c[1])",
                              "key=lambda c: (-c[0], tuple(-x for x in c[1]))")],
    "parent_always_root": [("ranks[i] + (k,), i)", "ranks[i] + (k,), 0)")],
    "token_from_first_depth": [("cand_token[len(r) - 1, r[-1]]", "cand_token[0, r[-1]]")],
    "siblings_dropped": [("for k in range(K)]", "for k in range(1)]")],
    "accept_target_of_child": [("tt[j] == tg[cur]", "tt[j] == tg[j]")],
    "accept_one_level": [("if nxt is None:\n            break", "if nxt is None or len(path) > 1:\n            break")],
    "bonus_from_root": [("return path, int(tg[cur]), slots", "return path, int(tg[0]), slots")],
    "accept_any_parent": [("if tp[j] == cur and tt[j] == tg[cur]:", "if tp[j] >= 0 and tt[j] == tg[cur]:")],
}

RUNNER = r"""
import importlib.util, sys
sys.path.insert(0, {root!r})
spec = importlib.util.spec_from_file_location("ddtree_mutant", {path!r})
mod = importlib.util.module_from_spec(spec)
spec.loader.exec_module(mod)
from tests import ddtree_pins as pins
failed = []
for pin in pins.ALL_PINS:
    try:
        pin(mod)
    except Exception:
        failed.append(pin.__name__)
print("FAILED:" + ",".join(failed))
"""


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    src = open(ddtree.__file__).read()
    for old, new in MUTANTS[name]:
        assert old in src, f"mutation anchor missing: {old!r}"
        src = src.replace(old, new)
    path = tmp_path / "ddtree_mutant.py"
    path.write_text(src)
    try:
        r = subprocess.run([sys.executable, "-c", RUNNER.format(root=ROOT, path=str(path))],
                           capture_output=True, text=True, timeout=120)
    except subprocess.TimeoutExpired:
        return  # a mutant that never finishes is caught too
    failed = [l for l in r.stdout.splitlines() if l.startswith("FAILED:")]
    assert r.returncode != 0 or (failed and failed[0] != "FAILED:"), r.stdout + r.stderr


def test_oracle_equals_brute_force_on_random_tiny_drafts():
    hyp = pytest.importorskip("hypothesis")
    st = hyp.strategies
    import numpy as np

    values = [0.0, -0.25, -0.5, -1.0, -3.0, float("-inf")]

    @hyp.settings(max_examples=300, deadline=None)
    @hyp.given(L=st.integers(1, 4), K=st.integers(1, 3), data=st.data())
    def check(L, K, data):
        lp = np.array([sorted(data.draw(st.lists(st.sampled_from(values), min_size=K, max_size=K)), reverse=True)
                       for _ in range(L)], dtype=np.float32)
        tok = np.arange(L * K, dtype=np.int32).reshape(L, K) + 100
        budget = data.draw(st.integers(1, ddtree.node_count(L, K)))
        got = ddtree.build_tree_one(7, tok, lp, budget)
        want = pins._brute(7, tok, lp, budget)
        assert got[0].tolist() == want[0] and got[1].tolist() == want[1] and got[2].tolist() == want[2]

    check()
