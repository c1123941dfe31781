"""Negative controls of the GPU tests' element bound (``parity.py``), on the CPU.

A bound that passes the kernels' output must still reject the mistakes a kernel
could make: an element off by a few percent, or a mask one token off on a long
context.  These tests build such wrong outputs from the oracle alone (its f64
result rounded to bf16, then perturbed, or the oracle run with the mistake) and
check that the bound names them, while the correctly rounded oracle output passes.
"""
import dataclasses
import os
import sys

import numpy as np
import pytest

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import oracle  # noqa: E402
import parity  # noqa: E402
from paged_gqa_decode_attn_gb300 import workloads as wl  # noqa: E402


def rne_bf16(x):
    """f64 -> f32 -> bf16 bits, round to nearest even: what the kernels store."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


CASES = [lambda: wl.page_case(16, 8, 256, 1024, 1500, 5), lambda: wl.page_case(16, 2, 512, 0, 700, 1),
         lambda: wl.sliding(), lambda: wl.sweep(128, 4096, 4, 1024, mapped=False)]


@pytest.mark.parametrize("make", CASES, ids=["page_hd256", "page_hd512", "sliding", "sweep_hd128"])
def test_correctly_rounded_output_passes(make):
    c = make()
    o64, _ = oracle.decode_case(c)
    for coef in (parity.COEF_DECODE, parity.COEF_TILED):
        assert not parity.beyond_bound(rne_bf16(o64), o64, coef).any()


@pytest.mark.parametrize("make", CASES, ids=["page_hd256", "page_hd512", "sliding", "sweep_hd128"])
def test_one_element_five_percent_off_is_rejected(make):
    """Any single element moved by 5% of max(|o|, its (row, head)'s RMS) is beyond the bound, at both
    coefficients: 5% exceeds 2^-8 + 2^-6 of that size."""
    c = make()
    o64, _ = oracle.decode_case(c)
    rms = np.sqrt(np.mean(o64 * o64, axis=-1, keepdims=True))
    size = np.maximum(np.abs(o64), rms)
    rng = np.random.default_rng(5)
    flat = np.arange(o64.size)
    picks = rng.choice(flat, size=min(200, o64.size), replace=False)
    picks = np.concatenate([picks, [int(np.argmax(np.abs(o64))), int(np.argmin(np.abs(o64)))]])
    for i in picks:
        idx = np.unravel_index(int(i), o64.shape)
        for sign in (1.0, -1.0):
            bad = o64.copy()
            bad[idx] += sign * 0.05 * size[idx]
            got = rne_bf16(bad)
            out = parity.beyond_bound(got, o64, parity.COEF_TILED)
            assert out[idx], f"{c.name}: element {idx} moved 5% passed the bound"
            assert out.sum() == 1


def test_one_token_mask_error_at_32k_is_rejected():
    """The 32K-context shape (nh32 nkv4 hd512) with Q = 0, so every visible position weighs the same
    and the output is the mean of V over 32768 positions: a mask that drops the last position moves
    each element by (o - v)/32768, about 1% of the output's RMS where |v| is near 1.  The bound rejects
    that output (hundreds of elements), and the rel-RMS against the f64 values shows it too."""
    c = wl.long_ctx()
    c0 = dataclasses.replace(c, q=np.zeros_like(c.q))
    good, _ = oracle.decode_case(c0)
    wrong, _ = oracle.decode_case(dataclasses.replace(c0, kvpos=c0.qpos - 1))
    assert not parity.beyond_bound(rne_bf16(good), good, parity.COEF_DECODE).any()
    out = parity.beyond_bound(rne_bf16(wrong), good, parity.COEF_DECODE)
    assert out.sum() > 100, int(out.sum())
    assert parity.rel_rms_f64(rne_bf16(wrong), good) > parity.REL_RMS_F64_GATE
    assert parity.rel_rms_f64(rne_bf16(good), good) < parity.REL_RMS_F64_GATE / 2


def test_window_one_token_off_is_rejected():
    """A sliding window one position too wide (the page's first decode case, window 1024 read as 1025)."""
    c = wl.page_case(16, 8, 256, 1024, 1500, 5)
    good, _ = oracle.decode_case(c)
    wrong, _ = oracle.decode_case(dataclasses.replace(c, window=1025))
    assert parity.beyond_bound(rne_bf16(wrong), good, parity.COEF_TILED).any()


def test_empty_row_must_be_exactly_zero():
    o64 = np.zeros((1, 2, 64))
    assert not parity.beyond_bound(np.zeros((1, 2, 64), np.uint16), o64).any()
    got = np.zeros((1, 2, 64), np.uint16)
    got[0, 1, 3] = 0x0001                     # the smallest subnormal
    assert parity.beyond_bound(got, o64).sum() == 1
