"""Pins of the f64 QK-RMSNorm / RoPE / paged-write oracle (oracle/pgqa_prep_oracle.c)
to facts it cannot get from itself: closed forms, invariants of a rotation, and
the K/V address as the (separately pinned) decode oracle reads it back.
CPU only."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from oracle import prep as op  # noqa: E402
from paged_gqa_decode_attn_gb300 import workloads as wl  # noqa: E402

ONE = np.uint16(0x3F80)           # bf16 1.0


def bf(x):
    return wl.bf16_trunc(np.asarray(x, dtype=np.float32).reshape(-1)).reshape(np.shape(x))


def run(x, pos, hd, rotary_dim, theta=10000.0, eps=0.0, w=None, norm_v=True, nh=1, nkv=1):
    """One head vector x (f32 values exactly representable in bf16) as Q, K and V of every row."""
    rows = len(pos)
    xb = np.tile(bf(x), rows * max(nh, nkv)).astype(np.uint16)
    wq = np.full(hd, ONE, np.uint16) if w is None else bf(w)
    ctx = int(max(pos)) + 1
    npages = (ctx + 15) // 16
    return op.prep(xb[:rows * nh * hd], xb[:rows * nkv * hd], xb[:rows * nkv * hd], wq, wq,
                   np.asarray(pos, np.int32), np.arange(npages, dtype=np.int32), np.zeros(rows, np.int32), None,
                   nh, nkv, hd, rotary_dim, theta, eps, norm_v)


def test_constant_vector_normalises_to_sign_times_weight():
    hd = 64
    w = 1.0 + np.arange(hd) / 64.0
    q, k, v, _ = run(np.full(hd, -0.5, np.float32), [0], hd, 0, w=w)
    np.testing.assert_array_equal(q[0, 0], -wl.bf16_to_f32(bf(w)).astype(np.float64))
    np.testing.assert_array_equal(v[0, 0], -np.ones(hd))        # weightless norm of V


@pytest.mark.parametrize("i,upper", [(0, False), (1, False), (5, False), (3, True)])
def test_one_hot_rotates_by_position_times_frequency(i, upper):
    """x = c e_j: the norm gives sqrt(hd) sign(c) e_j, then the pair (i, i + rd/2)
    turns by pos * theta^(-2i/rd): cos on j, +sin (j low) or -sin (j high) on the partner."""
    hd, rd, theta = 64, 32, 500.0
    half = rd // 2
    j = i + half if upper else i
    x = np.zeros(hd, np.float32)
    x[j] = 0.25
    pos = [0, 1, 7, 33, 1000]
    q, _, _, _ = run(x, pos, hd, rd, theta=theta)
    y = np.sqrt(hd)
    for t, p in enumerate(pos):
        a = p * theta ** (-2.0 * i / rd)
        want = np.zeros(hd)
        if upper:
            want[i + half] = y * np.cos(a)
            want[i] = -y * np.sin(a)
        else:
            want[i] = y * np.cos(a)
            want[i + half] = y * np.sin(a)
        np.testing.assert_allclose(q[t, 0], want, rtol=0, atol=1e-12)


def test_tail_beyond_rotary_dim_passes_through():
    hd, rd = 128, 48
    x = np.linspace(-1, 1, hd).astype(np.float32)
    q0, _, _, _ = run(x, [0], hd, 0)            # normed, no rotation
    q, _, _, _ = run(x, [777], hd, rd)
    np.testing.assert_array_equal(q[0, 0, rd:], q0[0, 0, rd:])
    assert not np.allclose(q[0, 0, :rd], q0[0, 0, :rd])


def test_position_zero_is_the_identity_rotation():
    hd = 256
    x = np.cos(np.arange(hd) * 0.37).astype(np.float32)
    q0, _, _, _ = run(x, [0], hd, 0)
    q, _, _, _ = run(x, [0], hd, hd)
    np.testing.assert_allclose(q, q0, rtol=0, atol=1e-15)


def test_rotation_keeps_each_pair_norm():
    hd, rd = 128, 128
    x = np.sin(np.arange(hd) * 1.7 + 0.3).astype(np.float32)
    q0, _, _, _ = run(x, [0], hd, 0)
    q, _, _, _ = run(x, [12345], hd, rd, theta=1e6)
    half = rd // 2
    n0 = q0[0, 0, :half] ** 2 + q0[0, 0, half:rd] ** 2
    n1 = q[0, 0, :half] ** 2 + q[0, 0, half:rd] ** 2
    np.testing.assert_allclose(n1, n0, rtol=1e-12)


def test_v_is_never_rotated_and_copied_without_norm_v():
    hd = 64
    x = np.full(hd, 0.75, np.float32)
    _, _, v, _ = run(x, [999], hd, hd)
    np.testing.assert_allclose(v[0, 0], np.ones(hd), rtol=1e-15)
    _, _, v2, _ = run(x, [999], hd, hd, norm_v=False)
    np.testing.assert_array_equal(v2[0, 0], np.full(hd, 0.75))


def test_eps_keeps_a_zero_vector_zero():
    q, k, v, _ = run(np.zeros(64, np.float32), [3], 64, 64, eps=1e-6)
    assert np.all(q == 0) and np.all(k == 0) and np.all(v == 0)


def test_kv_slots_are_where_the_decode_oracle_reads():
    """Place the oracle's V rows at its slots in a pool, then ask the (separately
    pinned) decode oracle with window 1 -- which returns V[qpos] exactly -- for every
    position: it must return each row's V, through a permuted table and page map."""
    c = wl.prep_case(2, 2, 64, 64, 40, 96, positions="scattered", mapped=True, seed=5)
    npg = c.npg + 3
    pmap = wl.lcg_permutation(npg, 9)[:c.npg].astype(np.int32)
    c.page_map = pmap
    _, _, v, slot = op.prep_case(c)
    pool_v = np.zeros(npg * c.nkv * 16 * c.hd, np.uint16)
    vb = wl.bf16_trunc(v.astype(np.float32))
    for t in range(c.rows):
        for kh in range(c.nkv):
            s0 = slot[t] + kh * 16 * c.hd
            pool_v[s0:s0 + c.hd] = vb[t, kh]
    q = np.zeros(c.rows * c.nkv * c.hd, np.uint16)
    _, got = oracle.decode(q, np.zeros_like(pool_v), pool_v, c.block_table, c.off, c.pos, c.nkv, c.nkv, c.hd, 1,
                           page_map=pmap)
    np.testing.assert_array_equal(got.reshape(c.rows, c.nkv, c.hd), vb)
