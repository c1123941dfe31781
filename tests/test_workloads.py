"""Seeded input generators: the LCG of span-02 ``engine/crates/kernels/tests/gpu.rs``
(``Rng``, ``bf``, ``mapped_pool``, ``run``) and the workload recipes built on it."""
import os
import sys

import dataclasses

import numpy as np
import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from paged_gqa_decode_attn_gb300 import workloads as wl  # noqa: E402

M64 = (1 << 64) - 1


def scalar_lcg(seed, n):
    s = seed
    out = []
    for _ in range(n):
        s = (s * 6364136223846793005 + 1442695040888963407) & M64
        out.append(s)
    return out


def test_vectorised_lcg_equals_scalar_recurrence_across_blocks():
    n = (1 << 16) + 1000                      # crosses one jump-ahead block boundary
    rng = wl.Lcg(12345 + 128)
    a = rng.states(n)
    b = np.array(scalar_lcg(12345 + 128, n), dtype=np.uint64)
    assert np.array_equal(a, b)
    # continuing the stream after a partial block
    c = rng.states(70000)
    d = np.array(scalar_lcg(int(b[-1]), 70000), dtype=np.uint64)
    assert np.array_equal(c, d)


def test_page_uniform_matches_rust_f32_semantics():
    """u32(s>>33) as f32 (round to nearest) / 2^31 - 1, all in f32."""
    st = wl.Lcg(777).states(5000)
    got = wl.uniform_page(st)
    for i in range(0, 5000, 37):
        v = np.float32(np.uint32(int(st[i]) >> 33)) / np.float32(2147483648.0) - np.float32(1.0)
        assert got[i] == v
    assert got.min() >= -1.0 and got.max() <= 0.0     # the page's generator is one-sided


def test_symmetric_uniform_range_and_exactness():
    st = wl.Lcg(99).states(200000)
    x = wl.uniform_sym(st)
    assert x.min() >= -1.0 and x.max() < 1.0
    assert x.min() < -0.99 and x.max() > 0.99
    ref = (st >> np.uint64(40)).astype(np.float64) * 2.0 ** -23 - 1.0
    assert np.array_equal(x.astype(np.float64), ref)


def test_bf16_truncation_values():
    v = np.array([1.0, -1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 0.0], dtype=np.float32)
    assert wl.bf16_trunc(v).tolist() == [0x3F80, 0xBF80, 0x3F80, 0x3F81, 0xC020, 0x0000]
    assert np.array_equal(wl.bf16_to_f32(wl.bf16_trunc(v))[[0, 1, 4, 5]], v[[0, 1, 4, 5]])


def test_mapped_pool_layout():
    npg, nkv, hd = 6, 2, 4
    pe = nkv * 16 * hd
    k = np.arange(npg * pe, dtype=np.uint16)
    v = k + 1
    mk, mv, pm = wl.mapped_pool(k, v, npg, nkv, hd, first_live=2)
    assert mk.size == (npg + 1) * pe
    assert pm.tolist() == [0, 0, 4, 3, 2, 1]
    for p in range(2, npg):
        s = npg - p
        assert np.array_equal(mk[s * pe:(s + 1) * pe], k[p * pe:(p + 1) * pe])
        assert np.array_equal(mv[s * pe:(s + 1) * pe], v[p * pe:(p + 1) * pe])
    assert np.all(mk[0:pe] == wl.BF16_NAN) and np.all(mk[5 * pe:6 * pe] == wl.BF16_NAN)


def test_lcg_permutation_is_a_permutation():
    p = wl.lcg_permutation(5000, 3)
    assert sorted(p.tolist()) == list(range(5000))
    assert not np.array_equal(p, np.arange(5000))


def test_page_case_draw_order_and_metadata():
    c = wl.page_case(16, 8, 256, 1024, 1500, 5)
    npg = (1500 + 15) // 16 + 1
    n = npg * 8 * 16 * 256
    rng = wl.Lcg(12345 + 256)
    assert np.array_equal(c.k_pool, wl.bf16_trunc(wl.uniform_page(rng.states(n))))
    assert np.array_equal(c.v_pool, wl.bf16_trunc(wl.uniform_page(rng.states(n))))
    assert np.array_equal(c.q, wl.bf16_trunc(wl.uniform_page(rng.states(5 * 16 * 256))))
    assert c.qpos.tolist() == [1495, 1496, 1497, 1498, 1499]
    assert c.block_table.tolist() == list(range(94))
    assert c.npg == npg


def test_algorithmic_bytes_of_the_named_workloads():
    assert wl.algorithmic_bytes(8, 2, 128, 0, [255], [0]) == 266_240
    assert wl.algorithmic_bytes(16, 8, 256, 1024, list(range(8188, 8192)), [0] * 4) == 8_478_720
    assert wl.algorithmic_bytes(32, 4, 512, 0, [32767], [0]) == 268_500_992
    assert wl.algorithmic_bytes(32, 8, 128, 0, [4095] * 64, [256 * r for r in range(64)]) == 1_074_790_400


def test_sweep_has_108_points_and_gaussian_peaky_keys():
    pts = wl.sweep_points()
    assert len(pts) == 108 and len(set(pts)) == 108
    c = wl.sweep(128, 1024, 1, 0, mapped=False)
    kf = wl.bf16_to_f32(c.k_pool).reshape(-1, 128).astype(np.float64)
    norms = np.sqrt((kf ** 2).mean(axis=1))
    frac_big = float((norms > 4.0).mean())          # x8 keys have RMS ~8, others ~1
    assert 0.03 < frac_big < 0.07
    vf = wl.bf16_to_f32(c.v_pool).astype(np.float64)
    assert abs(vf.mean()) < 0.01 and 0.97 < vf.std() < 1.03


@pytest.mark.parametrize("fold", [False, True])
def test_with_mapped_pool_variants(fold):
    c = wl.page_case(16, 8, 64, 100, 300, 3, dist="sym", seed=5)
    m = wl.with_mapped_pool(c, fold_into_table=fold)
    first_live = wl.window_lo(int(c.qpos[0]), 100) // 16
    if fold:
        assert m.page_map is None
        assert m.block_table.tolist() == [0 if j < first_live else c.npg - j
                                          for j in range(len(c.block_table))]
    else:
        assert m.page_map is not None and m.block_table is c.block_table


def test_live_pages_follow_the_rows_windows_through_the_table():
    """The page's sliding case (identity table): live pages are lo(row 0)/16 .. the last row's page.
    Behind a permuted table the same logical pages are live, at their permuted physical ids; a row
    with no visible position adds nothing."""
    c = wl.page_case(8, 2, 64, 100, 300, 3, dist="sym", seed=5)
    live = wl.live_pages(c)
    first = wl.window_lo(int(c.qpos[0]), 100) // 16
    last = int(c.qpos[-1]) // 16
    assert np.flatnonzero(live).tolist() == list(range(first, last + 1))
    perm = wl.lcg_permutation(c.npg, 3).astype(np.int32)
    pc = dataclasses.replace(c, block_table=perm[:len(c.block_table)])
    assert sorted(np.flatnonzero(wl.live_pages(pc)).tolist()) == sorted(perm[first:last + 1].tolist())
    kv = c.qpos.copy()
    kv[:] = c.qpos - 200                      # below every row's window: nothing visible
    assert not wl.live_pages(dataclasses.replace(c, kvpos=kv)).any()

