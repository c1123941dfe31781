"""Writes the regression snapshots in this folder from the f64 CPU oracle alone.

    python tests/golden/make_golden.py

The pages print no worked numeric example for paged decode attention or for
the QK-RMSNorm / RoPE write (their gates print only rel-RMS results, and the
fixture values behind the negative controls they quote are not given), so
every stored number here comes from ``oracle/`` on inputs drawn by
``paged_gqa_decode_attn_gb300.workloads``.  These files are regression
snapshots, not pins: the oracle's pins are the closed forms, brute force and
negative controls in ``tests/test_oracle_pins.py`` and
``tests/test_prep_oracle_pins.py``.  A snapshot turns any later change to the
oracle's arithmetic, or to the seeded inputs, into a failing CPU test that
has to be explained.
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from oracle import prep as oprep  # noqa: E402
from paged_gqa_decode_attn_gb300 import workloads as wl  # noqa: E402

F64_DIMS = 4          # f64 values kept per (row, head): the first dims


def decode_snapshot_case():
    """Sliding window of 40 over a ragged 100-token context, 3 rows, the page's LCG draw."""
    return wl.page_case(8, 2, 64, 40, 100, 3, dist="page", name="decode_nh8_nkv2_hd64_w40_ctx100_r3")


def prep_snapshot_case():
    """Half rotation, scattered positions, V normed."""
    return wl.prep_case(4, 2, 64, 32, 5, 40, positions="scattered", seed=5, name="prep_nh4_nkv2_hd64_rd32_r5")


def decode_lines():
    c = decode_snapshot_case()
    o64, o16 = oracle.decode_case(c)
    out = [f"# {c.name}: f64 CPU oracle of paged GQA decode attention",
           "# Definition: the `reference` function of the page's decode gate (span-02, "
           "engine/crates/kernels/tests/gpu.rs): scale 1.0, causal window, softmax in f64, bf16 output.",
           "# Inputs: paged_gqa_decode_attn_gb300.workloads.page_case(8, 2, 64, 40, 100, 3, dist='page').",
           "# Written by tests/golden/make_golden.py (calls only oracle/). A regression snapshot, not a pin.",
           "# Line: row head | bf16 bits of o[row][head][0..hd) as hex | f64 o[row][head][0..4) as float.hex"]
    for r in range(c.rows):
        for h in range(c.nh):
            bits = "".join(f"{int(x):04x}" for x in o16[r, h])
            f = " ".join(float(v).hex() for v in o64[r, h, :F64_DIMS])
            out.append(f"{r} {h} | {bits} | {f}")
    return out


def prep_lines():
    c = prep_snapshot_case()
    q, k, v, slot = oprep.prep_case(c)
    out = [f"# {c.name}: f64 CPU oracle of per-head RMSNorm + rotary embedding and the paged K/V write",
           "# Definition: the QK-RMSNorm / RoPE pool write whose device gates pegainfer PR #1002 describes: "
           "RMSNorm with weight, rotation of dims i and i + rotary_dim/2 for i < rotary_dim/2 (the rope-lo and "
           "rope-hi halves), the tail passed through, K and V landing at the paged slot of each position.",
           "# Inputs: paged_gqa_decode_attn_gb300.workloads.prep_case(4, 2, 64, 32, 5, 40, "
           "positions='scattered', seed=5).",
           "# Written by tests/golden/make_golden.py (calls only oracle/). A regression snapshot, not a pin.",
           "# Lines: 'slot row slot' (pool element offset of the row's K/V, head 0); "
           "'q|k|v row head f64[0..4) as float.hex'"]
    for r in range(slot.size):
        out.append(f"slot {r} {int(slot[r])}")
    for tag, a in (("q", q), ("k", k), ("v", v)):
        for r in range(a.shape[0]):
            for h in range(a.shape[1]):
                out.append(f"{tag} {r} {h} " + " ".join(float(x).hex() for x in a[r, h, :F64_DIMS]))
    return out


FILES = {"decode_nh8_nkv2_hd64_w40_ctx100_r3.txt": decode_lines,
         "prep_nh4_nkv2_hd64_rd32_r5.txt": prep_lines}


def main():
    for name, fn in FILES.items():
        with open(os.path.join(HERE, name), "w") as f:
            f.write("\n".join(fn()) + "\n")
        print("wrote", name)


if __name__ == "__main__":
    main()
