"""Negative controls of the three GPU gates: each gate must go red, naming the first
differing element, when the library is fed a wrong but in-bounds input.

The gates are those of `run` in span-02 ``engine/crates/kernels/tests/gpu.rs`` (rel-RMS
against the reference, counters merge == combine kernel bit for bit, identity pool ==
page-map pool bit for bit).  pegainfer PR #1002 asks for such controls: perturb the
metadata a kernel reads (an origin, an address) and see the gate fail, because a gate
that stays green on a wrong input proves nothing.  Every input here stays in bounds:
nothing faults, traps or hangs; only the answer is wrong.
"""
import dataclasses
import os
import sys

import numpy as np
import pytest

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from paged_gqa_decode_attn_gb300 import workloads as wl  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch  # noqa: F401
    import paged_gqa_decode_attn_gb300 as pgqa
    pgqa.build()
    pgqa.load()
    yield


def spans_case(seed=61, nh=16, nkv=4, hd=128):
    """Four rows, each with its own span of one permuted table (distinct non-zero off)."""
    rng = wl.Lcg(seed)
    npages = 4 * 20
    n = npages * nkv * 16 * hd
    k = wl.draw_bf16(rng, n, "sym")
    v = wl.draw_bf16(rng, n, "sym")
    q = wl.draw_bf16(rng, 4 * nh * hd, "sym")
    bt = wl.lcg_permutation(npages, seed + 1)
    off = np.array([0, 20, 40, 60], dtype=np.int32)
    qpos = np.array([300, 299, 310, 257], dtype=np.int32)
    return wl.Case("spans", nh, nkv, hd, 0, 4, q, k, v, bt, off, qpos, ctx=320, npg=npages)


@pytest.mark.parametrize("splits", [1, 4])
def test_rel_rms_gate_fails_when_a_row_reads_another_rows_span(splits):
    from gpu_util import DevCase, parity_verdict
    good = spans_case()
    d = DevCase(good, splits)
    ok, msg, _ = parity_verdict(good, d.result(), "control: correct off")
    assert ok, msg
    wrong_off = good.off.copy()
    wrong_off[2] = good.off[1]                 # row 2 reads row 1's span (in bounds: same length)
    dw = DevCase(dataclasses.replace(good, off=wrong_off), splits)
    ok, msg, _ = parity_verdict(good, dw.result(), "row 2 off -> row 1's span", oracle_case=good)
    assert not ok, "the parity gate stayed green with a row reading another row's span"
    assert "first (row, head, dim) (2," in msg, msg


def test_page_map_gate_fails_when_two_live_pages_swap():
    from gpu_util import DevCase, first_difference
    c = wl.page_case(16, 8, 256, 1024, 1500, 5)
    d = DevCase(c)
    ref = d.result()
    m = wl.with_mapped_pool(c)
    assert np.array_equal(DevCase(m, d.splits).result(), ref)      # the gate itself holds
    pm = m.page_map.copy()
    live = np.nonzero(pm)[0]
    a, b = int(live[len(live) // 2]), int(live[len(live) // 2 + 1])
    pm[a], pm[b] = pm[b], pm[a]                # two live pages trade places
    got = DevCase(dataclasses.replace(m, page_map=pm), d.splits).result()
    assert not np.array_equal(got, ref), "the page-map gate stayed green with two live pages swapped"
    assert first_difference(got, ref).startswith(tuple("123456789")), first_difference(got, ref)


@pytest.mark.parametrize("window", [16, 1024])
def test_rel_rms_gate_fails_on_a_window_one_position_too_wide(window):
    from gpu_util import DevCase, parity_verdict
    c = wl.page_case(16, 8, 256, window, 1500, 5)
    ok, msg, _ = parity_verdict(c, DevCase(c, 4).result(), "control")
    assert ok, msg
    wide = dataclasses.replace(c, window=window + 1)
    ok, msg, _ = parity_verdict(wide, DevCase(wide, 4).result(), f"window {window + 1} for {window}",
                                oracle_case=c)
    assert not ok, f"the parity gate stayed green with window {window + 1} in place of {window}"
    assert "first (row, head, dim)" in msg


def test_merge_gate_fails_when_the_partition_differs():
    """The merge gate compares bits: the same attention cut into a different number of splits
    (a different summation order) must show up, so the gate does test the low bits."""
    from gpu_util import DevCase, first_difference
    c = wl.page_case(16, 8, 256, 1024, 1500, 5)
    d = DevCase(c, 8)
    a = d.result(counters=True)
    assert np.array_equal(d.result(counters=False), a)
    b = d.result(counters=False, splits=7)
    assert not np.array_equal(b, a), "8 and 7 splits gave the same bits: the gate could not see the order"
    assert "differ; first at" in first_difference(b, a)
