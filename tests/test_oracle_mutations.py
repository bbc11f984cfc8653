"""Plant plausible mistakes in copies of the oracle; some pin must catch each.

Every mutant is a text edit of oracle/mla_oracle.c compiled into a temporary
directory and exercised in a child process (a mutant may read out of bounds,
which must not take the test runner down).  The committed oracle is never
modified.
"""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    "drop_rope_term": [("s[j] = pr->scale * (dot_lat + dot_pe);", "s[j] = pr->scale * dot_lat;")],
    "scale_latent_only": [("s[j] = pr->scale * (dot_lat + dot_pe);",
                           "s[j] = pr->scale * dot_lat + dot_pe;")],
    "lse_base2": [("m + log(Z)", "m + log2(Z)")],
    "mask_parent_only": [("(anc[(int64_t)b * Q + p] | self)", "(((uint64_t)1 << p) | self)")],
    "mask_self_excluded": [("anc[(int64_t)b * Q + i] = (p < 0) ? self : (anc[(int64_t)b * Q + p] | self);",
                            "anc[(int64_t)b * Q + i] = (p < 0) ? 0 : (anc[(int64_t)b * Q + p] | ((uint64_t)1 << p));")],
    "prefix_short_by_one": [("int64_t nv = P;", "int64_t nv = P > 0 ? P - 1 : 0;"),
                            ("for (int64_t p = 0; p < P; ++p)", "for (int64_t p = 0; p + 1 < P; ++p)")],
    "tail_shifted": [("pos[k++] = P + t;", "pos[k++] = P + (t + 1) % Q;")],
    "no_max_in_normaliser": [("Z += exp(s[j] - m);", "Z += exp(s[j]);")],
    "value_includes_rope": [("o[d] += w * elem(pr->kv_c, pr->dtype, slot * pr->kv_c_stride + d);",
                             "o[d] += w * elem(pr->kv_c, pr->dtype, slot * pr->kv_c_stride + d + 64);")],
    "paged_offset_swapped": [("s = page * pr->page_size + p % pr->page_size;",
                              "s = page + (p % pr->page_size) * pr->page_size;")],
    "bf16_shift": [("<< 16;", "<< 15;")],
    "anc_wrong_sequence": [("anc[(int64_t)b * Q + i];\n", "anc[i];\n")],
}

RUNNER = r"""
import sys, traceback
sys.path.insert(0, {root!r})
import oracle
from tests import oracle_pins as pins
orc = oracle.Oracle({lib!r})
failed = []
for pin in pins.ALL_PINS:
    try:
        pin(orc)
    except Exception:
        failed.append(pin.__name__)
print("FAILED:" + ",".join(failed))
"""


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    src = open(oracle.SRC).read()
    for old, new in MUTANTS[name]:
        assert old in src, f"mutation anchor missing: {old!r}"
        src = src.replace(old, new)
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src)
    lib = oracle.build(str(mpath), str(tmp_path / "libmutant.so"))
    code = RUNNER.format(root=ROOT, lib=lib)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                       timeout=300, env={**os.environ, "OMP_NUM_THREADS": "2"})
    line = [l for l in r.stdout.splitlines() if l.startswith("FAILED:")]
    # a crash of the child (e.g. an out-of-bounds read) also counts as caught
    caught = (r.returncode != 0) or (line and line[0] != "FAILED:")
    assert caught, f"no pin caught mutant {name}: {r.stdout[-400:]} {r.stderr[-400:]}"
