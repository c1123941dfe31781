"""Negative controls for the prep-oracle pins: plant one plausible mistake at a
time in a copy of pgqa_prep_oracle.c, build it, and check that the pins go red.
CPU only."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "pgqa_prep_oracle.c")

MUTATIONS = {
    "rotation_sign": ("y[i] = lo * c - hi * s;", "y[i] = lo * c + hi * s;"),
    "adjacent_pairs": ("double lo = y[i], hi = y[i + half];", "double lo = y[2 * i], hi = y[2 * i + 1];"),
    "frequency_exponent": ("pow(theta, -2.0 * i / rotary_dim)", "pow(theta, -1.0 * i / rotary_dim)"),
    "sum_not_mean": ("sqrt(ss / hd + eps)", "sqrt(ss + eps)"),
    "weight_ignored": ("* (w ? bf16_value(w[d]) : 1.0)", "* 1.0"),
    "tail_rotated": ("int half = rotary_dim / 2;", "int half = rotary_dim / 2 + 1;"),
    "slot_is_page_index": ("pos[t] % 16) * (int64_t)hd;", "pos[t] / 16) * (int64_t)hd;"),
    "page_map_ignored": ("page = page_map[page];", "page = page;"),
    "v_rotated": ("rms_norm(xv, NULL, hd, eps, yv);", "{ rms_norm(xv, NULL, hd, eps, yv); rope(yv, rotary_dim, theta, pos[t]); }"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_prep_pins_fail_on_planted_mistake(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    bad = tmp_path / "bad.c"
    bad.write_text(src.replace(old, new))
    lib = tmp_path / "libbad.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off",
                           "-o", str(lib), str(bad), "-lm"])
    env = dict(os.environ, PGQA_PREP_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_prep_oracle_pins.py")],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins stayed green with mutation {name}:\n{r.stdout[-2000:]}"
