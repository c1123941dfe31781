"""GPU parity of libpgqa's QK-RMSNorm / RoPE / paged K-V write against its f64 oracle.

What pegainfer PR #1002's gates check, carried over: the normed, rotated Q and
K, and V, against the operator's definition; K and V landing at the paged
layout address with every other pool element untouched; and the same bits
through a permuted block table behind a page map.  The element bound follows
from the arithmetic: bf16 rounding of the output (2^-9 relative) plus f32
norm and angle rounding, held as |o - o_f64| <= 2^-8 |o_f64| + 2^-8 rms(vector).
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

SENTINEL = 0x5555


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch  # noqa: F401
    import paged_gqa_decode_attn_gb300 as pgqa
    pgqa.build()
    pgqa.load()
    yield


def compact(c):
    """Point the used logical pages at distinct small physical pages (the others at 0),
    so far positions need no pool of ctx tokens."""
    used = sorted({int(o) + int(q) // 16 for o, q in zip(c.off, c.pos)})
    bt = np.zeros_like(c.block_table)
    for i, e in enumerate(used):
        bt[e] = i + 1
    return dataclasses.replace(c, block_table=bt, npg=len(used) + 1)


def run_device(c):
    """q_out [rows][nh][hd], k_pool, v_pool [npg][nkv][16][hd] as bf16 bits."""
    import torch
    import paged_gqa_decode_attn_gb300 as pgqa
    from gpu_util import dev_i16, dev_i32
    npool = max(int(c.block_table.max()) + 1, c.npg)
    if c.page_map is not None:
        npool = max(npool, int(c.page_map.max()) + 1)
    k_pool = torch.full((npool * c.nkv * 16 * c.hd,), SENTINEL, dtype=torch.int16, device="cuda")
    v_pool = torch.full_like(k_pool, SENTINEL)
    q_out = torch.full((c.rows * c.nh * c.hd,), SENTINEL, dtype=torch.int16, device="cuda")
    pgqa.qk_norm_rope_write(q_out, k_pool, v_pool, dev_i16(c.q_in), dev_i16(c.k_in), dev_i16(c.v_in),
                            dev_i16(c.q_weight), dev_i16(c.k_weight), dev_i32(c.pos), dev_i32(c.block_table),
                            dev_i32(c.off), dev_i32(c.page_map), c.rows, c.nh, c.nkv, c.hd, c.rotary_dim, c.theta,
                            c.eps, c.norm_v)
    torch.cuda.synchronize()

    def host(t, shape):
        return t.cpu().numpy().view(np.uint16).reshape(shape)
    return (host(q_out, (c.rows, c.nh, c.hd)), host(k_pool, (npool, c.nkv, 16, c.hd)),
            host(v_pool, (npool, c.nkv, 16, c.hd)))


def within_bound(got_bits, ref, label):
    got = wl.bf16_to_f32(got_bits).astype(np.float64)
    rms = np.sqrt(np.mean(ref ** 2, axis=-1, keepdims=True))
    bad = np.abs(got - ref) > 2.0 ** -8 * np.abs(ref) + 2.0 ** -8 * rms
    assert not bad.any(), f"{label}: {int(bad.sum())} elements beyond the bound, first {np.argwhere(bad)[0]}"
    assert np.all(np.isfinite(got))


def check(c):
    from oracle import prep as op
    q_ref, k_ref, v_ref, slot = op.prep_case(c)
    q, kp, vp = run_device(c)
    within_bound(q, q_ref, f"{c.name} q")
    written = np.zeros(kp.size, dtype=bool)
    kf, vf = kp.reshape(-1), vp.reshape(-1)
    for kh in range(c.nkv):
        idx = slot[:, None] + kh * 16 * c.hd + np.arange(c.hd)[None, :]
        within_bound(kf[idx], k_ref[:, kh], f"{c.name} k head {kh}")
        within_bound(vf[idx], v_ref[:, kh], f"{c.name} v head {kh}")
        written[idx.reshape(-1)] = True
    assert np.all(kf[~written] == SENTINEL) and np.all(vf[~written] == SENTINEL), "pool written outside the slots"
    return q, kp, vp


@pytest.mark.parametrize("hd", [64, 128, 256, 512])
@pytest.mark.parametrize("rd_frac", [1.0, 0.5, 0.0])
def test_head_dims_and_rotary_widths(hd, rd_frac):
    rd = int(hd * rd_frac)
    check(compact(wl.prep_case(8, 2, hd, rd, 33, 200, positions="scattered", seed=hd + rd)))


@pytest.mark.parametrize("positions,ctx", [("prefill", 300), ("decode", 100000), ("scattered", 70000)])
@pytest.mark.parametrize("norm_v", [True, False])
def test_positions_far_and_near_and_v_modes(positions, ctx, norm_v):
    check(compact(wl.prep_case(16, 8, 256, 256, 40, ctx, positions=positions, norm_v=norm_v, theta=500000.0,
                               seed=ctx)))


@pytest.mark.parametrize("nh,nkv", [(4, 4), (32, 2), (24, 8)])
def test_group_sizes(nh, nkv):
    check(compact(wl.prep_case(nh, nkv, 128, 64, 25, 500, positions="decode", dist="gauss", seed=nh)))


def test_page_map_gives_the_same_bits():
    """A permuted table behind a page map: Q bit-identical, K/V rows bit-identical at their mapped slots."""
    c = wl.prep_case(8, 4, 256, 128, 48, 600, positions="scattered", seed=3)
    q0, k0, v0 = check(c)
    m = wl.prep_case(8, 4, 256, 128, 48, 600, positions="scattered", seed=3, mapped=True)
    pmap = wl.lcg_permutation(m.npg + 5, 11)[:m.npg].astype(np.int32)
    m = dataclasses.replace(m, page_map=pmap)
    q1, k1, v1 = check(m)
    np.testing.assert_array_equal(q1, q0)
    for t in range(c.rows):
        p, s = int(c.pos[t]) // 16, int(c.pos[t]) % 16
        np.testing.assert_array_equal(k1[pmap[m.block_table[p]], :, s], k0[c.block_table[p], :, s])
        np.testing.assert_array_equal(v1[pmap[m.block_table[p]], :, s], v0[c.block_table[p], :, s])


def test_several_sequences_by_offset():
    """Rows of two sequences, each through its own span of one block table."""
    c = wl.prep_case(8, 2, 128, 128, 30, 320, positions="scattered", seed=21)
    bt = np.concatenate([c.block_table, wl.lcg_permutation(c.npg, 4).astype(np.int32) + c.npg])
    off = np.where(np.arange(c.rows) % 2 == 0, 0, c.npg).astype(np.int32)
    check(dataclasses.replace(c, block_table=bt, off=off, npg=2 * c.npg))


def test_prep_long_full_size():
    """The benchmark's workload in its launch configuration: 8192 rows, nh16 nkv8 hd256,
    full rotation (many items per persistent CTA), every element and every pool slot."""
    check(wl.prep_long())


def test_zero_rows_is_a_no_op():
    import torch
    import paged_gqa_decode_attn_gb300 as pgqa
    x = torch.zeros(16, dtype=torch.int16, device="cuda")
    pgqa.qk_norm_rope_write(x, x, x, x, x, x, x, x, x, x, x, None, 0, 8, 2, 128, 128, 10000.0, 1e-6)
    torch.cuda.synchronize()
    assert int(x.abs().sum().item()) == 0
