"""Negative controls for the oracle pins: plant one plausible mistake at a time
in a copy of the oracle's C source, build it, and check that the pin suite
goes red.  A pin suite that stays green on a broken oracle proves nothing.
All of this runs on the CPU.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "pgqa_oracle.c")

MUTATIONS = {
    "no_max_subtraction": ("s[i] = exp(s[i] - m);", "s[i] = exp(s[i]);"),
    "kv_head_modulo": ("int kh = h / (j->nh / j->nkv);", "int kh = h % j->nkv;"),
    "window_off_by_one": ("lo = qp + 1 - j->window;", "lo = qp - j->window;"),
    "slot_page_swapped": ("return ((phys * j->nkv + kh) * 16 + p % 16) * (int64_t)j->hd;",
                          "return ((phys * j->nkv + kh) * 16 + p / 16) * (int64_t)j->hd;"),
    "page_map_ignored": ("phys = j->page_map[phys];", "phys = phys;"),
    "output_rounded_to_nearest": ("return (uint16_t)(u >> 16);",
                                  "return (uint16_t)((u + 0x7fffu + ((u >> 16) & 1u)) >> 16);"),
    "no_normalisation": ("double w = s[i] / z;", "double w = s[i];"),
    "score_sign": ("acc += bf16_value(qv[d]) * bf16_value(kv[d]);",
                   "acc -= bf16_value(qv[d]) * bf16_value(kv[d]);"),
    "offset_ignored": ("j->block_table[(int64_t)j->off[t] + p / 16]", "j->block_table[p / 16]"),
    "kvpos_ignored": ("if (j->kvpos && j->kvpos[t] < hi)", "if (0)"),
    "kvpos_clamp_dropped": ("if (j->kvpos && j->kvpos[t] < hi)", "if (j->kvpos)"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_fail_on_planted_mistake(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    bad = tmp_path / "bad.c"
    bad.write_text(src.replace(old, new))
    lib = tmp_path / "libbad.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                           "-fno-fast-math", "-ffp-contract=off", "-o", str(lib), str(bad), "-lm"])
    env = dict(os.environ, PGQA_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins stayed green with mutation {name}:\n{r.stdout[-2000:]}"
