"""The oracle against its committed regression snapshots (tests/golden/).

The snapshots were written by ``tests/golden/make_golden.py`` from the oracle
alone.  They are not pins (the pins are in test_oracle_pins.py and
test_prep_oracle_pins.py); they make any change to the oracle's arithmetic or
to the seeded inputs fail here until it is explained and the snapshot is
rewritten.  bf16 outputs and slots must match exactly; f64 values within a
relative 1e-12, which allows the last-ulp differences of another libm's exp,
pow, sin and cos.
"""
import importlib.util
import os

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden")


def _maker():
    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(GOLDEN, "make_golden.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _close(a: str, b: str) -> bool:
    x, y = float.fromhex(a), float.fromhex(b)
    return abs(x - y) <= 1e-12 * max(abs(x), abs(y)) + 1e-300


def _compare(name, fresh, stored):
    body_f = [ln for ln in fresh if not ln.startswith("#")]
    body_s = [ln for ln in stored if not ln.startswith("#")]
    assert len(body_f) == len(body_s), f"{name}: {len(body_f)} lines now, {len(body_s)} stored"
    for lf, ls in zip(body_f, body_s):
        if "|" in lf:          # decode: row head | bf16 hex | f64 hex
            kf, bits_f, f64_f = (p.strip() for p in lf.split("|"))
            ks, bits_s, f64_s = (p.strip() for p in ls.split("|"))
            assert (kf, bits_f) == (ks, bits_s), f"{name}: bf16 output differs at ({kf})"
        else:                  # prep: slot lines exact, value lines by tag
            tf, ts = lf.split(), ls.split()
            if tf[0] == "slot":
                assert tf == ts, f"{name}: {lf!r} != {ls!r}"
                continue
            nkey = 3
            assert tf[:nkey] == ts[:nkey], f"{name}: {lf!r} vs {ls!r}"
            f64_f, f64_s = " ".join(tf[nkey:]), " ".join(ts[nkey:])
            kf = " ".join(tf[:nkey])
        vf, vs = f64_f.split(), f64_s.split()
        assert len(vf) == len(vs)
        for a, b in zip(vf, vs):
            assert _close(a, b), f"{name}: f64 value at ({kf}) moved: {float.fromhex(a)!r} vs {float.fromhex(b)!r}"


@pytest.mark.parametrize("name", ["decode_nh8_nkv2_hd64_w40_ctx100_r3.txt", "prep_nh4_nkv2_hd64_rd32_r5.txt"])
def test_oracle_matches_snapshot(name):
    mod = _maker()
    fresh = mod.FILES[name]()
    with open(os.path.join(GOLDEN, name)) as f:
        stored = f.read().splitlines()
    _compare(name, fresh, stored)


def test_snapshot_catches_a_moved_value():
    """The comparison is load-bearing: one changed bf16 digit or one f64 ulp-scale shift beyond 1e-12 fails."""
    mod = _maker()
    fresh = mod.FILES["decode_nh8_nkv2_hd64_w40_ctx100_r3.txt"]()
    body = [i for i, ln in enumerate(fresh) if not ln.startswith("#")]
    bad = list(fresh)
    k, bits, f64 = bad[body[5]].split("|")
    bits = bits.strip()
    bad[body[5]] = f"{k}| {bits[:-1]}{'0' if bits[-1] != '0' else '1'} |{f64}"
    with pytest.raises(AssertionError):
        _compare("planted", fresh, bad)
    bad = list(fresh)
    k, bits, f64 = bad[body[7]].split("|")
    vals = f64.split()
    vals[0] = (float.fromhex(vals[0]) * (1 + 1e-9)).hex()
    bad[body[7]] = f"{k}|{bits}| {' '.join(vals)}"
    with pytest.raises(AssertionError):
        _compare("planted", fresh, bad)
