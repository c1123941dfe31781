"""GPU parity of libpgqa's split-KV paged decode attention against the f64 oracle.

The three gates follow the `run` function of span-02
``engine/crates/kernels/tests/gpu.rs``:
  1. rel-RMS of the bf16 output against the oracle's bf16 output < 1e-2;
  2. merge counters (the split kernel merges, up to 8 splits) == separate combine
     kernel, bit for bit;
  3. identity pool == permuted pool behind a page map with the NaN null page 0
     for pages outside every row's window, bit for bit (also with the map
     folded into the block table).
On top of the page's gate every element is held to a bound derived from the
arithmetic (bf16 P and output rounding; ``parity.py``):
|o - o_f64| <= 2^-8 |o_f64| + 2^-7 rms_h(o_f64), per (row, head).
"""
import os
import sys

import numpy as np
import pytest

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import oracle  # noqa: E402
from paged_gqa_decode_attn_gb300 import workloads as wl  # noqa: E402

pytestmark = pytest.mark.gpu

from gpu_util import REL_RMS_GATE, bits_to_f64, check_parity  # noqa: E402,F401


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch  # noqa: F401
    import paged_gqa_decode_attn_gb300 as pgqa
    pgqa.build()
    pgqa.load()
    yield


def full_gates(case, splits=None, mapped=True):
    """Gates 1-3 on one case; returns the identity-pool output."""
    from gpu_util import DevCase, first_difference
    d = DevCase(case, splits)
    a = d.result(counters=True)
    check_parity(case, a, case.name)
    b = d.result(counters=False)
    assert np.array_equal(a, b), "merge modes differ: " + first_difference(b, a)
    assert int(d.cnt.abs().sum().item()) == 0, "merge counters not left at zero"
    if mapped:
        for fold in (False, True):
            m = wl.with_mapped_pool(case, fold_into_table=fold)
            dm = DevCase(m, d.splits)
            am = dm.result(counters=True)
            assert np.array_equal(am, a), f"page map (fold={fold}) differs: " + first_difference(am, a)
            bm = dm.result(counters=False)
            assert np.array_equal(bm, a), f"page map (fold={fold}) combine differs: " + first_difference(bm, a)
    return a, d


@pytest.mark.parametrize("args", [(16, 8, 256, 1024, 1500, 5), (16, 2, 512, 0, 700, 1)],
                         ids=["hd256_w1024_ctx1500_r5", "hd512_w0_ctx700_r1"])
def test_page_decode_cases(args):
    full_gates(wl.page_case(*args))


def test_tiny_full_attention():
    full_gates(wl.tiny())


def test_sliding_window_multirow():
    full_gates(wl.sliding())


def test_long_context_32k_both_merge_modes():
    full_gates(wl.long_ctx(), mapped=True)


def test_batched_64_rows_shared_permuted_table():
    full_gates(wl.batched(), mapped=False)


SWEEP_SAMPLE = [
    (128, 1024, 1, 0), (128, 4096, 16, 1024), (128, 65536, 4, 4096), (128, 65536, 1, 0),
    (256, 1024, 16, 4096), (256, 4096, 4, 0), (256, 16384, 1, 1024),
    (512, 1024, 4, 1024), (512, 4096, 1, 4096), (512, 16384, 16, 0),
]


@pytest.mark.parametrize("pt", SWEEP_SAMPLE, ids=lambda p: "hd%d_ctx%d_r%d_w%d" % p)
def test_sweep_points_gaussian_peaky_permuted(pt):
    """Gaussian Q/K/V with 5% of keys x8, served from the permuted pool with the NaN null page."""
    c = wl.sweep(*pt, mapped=False)
    a, d = full_gates(c, mapped=True)


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 64, 256])
def test_any_split_count_matches_oracle(splits):
    """More splits than pages leaves empty splits; all counts must pass the gates."""
    c = wl.page_case(8, 2, 128, 0, 300, 3, dist="sym", seed=11)
    full_gates(c, splits=splits)


@pytest.mark.parametrize("hd", [64, 128, 256, 512])
@pytest.mark.parametrize("nh,nkv", [(4, 4), (8, 1), (32, 2), (24, 2)])
def test_head_dims_and_group_sizes(hd, nh, nkv):
    """g = 1, 8, 16 (two head subgroups per kv head) and 12 (a partial subgroup)."""
    c = wl.page_case(nh, nkv, hd, 0, 200, 2, dist="sym", seed=hd + nh)
    full_gates(c, splits=3, mapped=False)


@pytest.mark.parametrize("hd", [64, 128, 256, 512])
@pytest.mark.parametrize("splits", [9, 13, 70])
def test_two_level_combine_every_head_dim(hd, splits):
    """Above 8 splits the combine kernel merges in two levels, with or without counters (which it leaves
    untouched): ragged last groups (9 = 8 + 1, 13 = 8 + 5, 70 = 8 * 8 + 6), every count of 128-dim slices
    (hd 64 uses half the lanes), g = 8 so every CTA serves 8 query rows."""
    import paged_gqa_decode_attn_gb300 as pgqa
    assert pgqa.decode_kernel_count(splits, True) == 2
    c = wl.page_case(16, 2, hd, 0, 90 * 16 + 7, 2, dist="sym", seed=hd + splits)
    full_gates(c, splits=splits, mapped=False)


@pytest.mark.parametrize("hd", [64, 128, 256, 512])
@pytest.mark.parametrize("splits", [2, 4, 8])
def test_on_chip_cluster_merge_every_head_dim(hd, splits):
    """2, 4 and 8 splits merge inside a thread-block cluster when counters are given."""
    c = wl.page_case(16, 2, hd, 0, 40 * 16 + 5, 2, dist="sym", seed=hd * splits)
    full_gates(c, splits=splits, mapped=False)


@pytest.mark.parametrize("window,ctx,rows", [(1, 50, 3), (5000, 700, 2), (17, 33, 4), (0, 1, 1), (16, 16, 1)])
def test_window_and_tiny_context_edges(window, ctx, rows):
    c = wl.page_case(16, 4, 128, window, ctx, rows, dist="sym", seed=window + ctx)
    full_gates(c, splits=4)


def ragged_case(seed=21, nh=16, nkv=4, hd=128, window=40):
    """Rows with distinct non-zero offsets, positions mid-page, and one empty row (kvpos < lo)."""
    rng = wl.Lcg(seed)
    npages = 64
    n = npages * nkv * 16 * hd
    k = wl.draw_bf16(rng, n, "sym")
    v = wl.draw_bf16(rng, n, "sym")
    rows = 5
    q = wl.draw_bf16(rng, rows * nh * hd, "sym")
    perm = wl.lcg_permutation(npages, seed + 1)
    bt = np.concatenate([perm[:20], perm[20:44], perm[44:64]]).astype(np.int32)
    off = np.array([0, 20, 44, 20, 5], dtype=np.int32)
    qpos = np.array([300, 383, 250, 17, 100], dtype=np.int32)
    # row 3's kvpos lies past its qpos (causal: that changes nothing); row 4 is empty
    kvpos = np.array([300, 383, 250, 19, 30], dtype=np.int32)
    return wl.Case("ragged", nh, nkv, hd, window, rows, q, k, v, bt, off, qpos, kvpos=kvpos,
                   ctx=384, npg=npages)


@pytest.mark.parametrize("window", [0, 40])
def test_ragged_rows_offsets_kvpos_and_empty_row(window):
    from gpu_util import DevCase
    c = ragged_case(window=window)
    for splits in (1, 5):
        d = DevCase(c, splits)
        a = d.result(counters=True)
        check_parity(c, a, f"ragged w{window} s{splits}")
        assert np.array_equal(a, d.result(counters=False))
        if window:
            assert np.all(a[4] == 0), "row with no visible position must be zero"


@pytest.mark.parametrize("splits", [1, 4, 13])
def test_kvpos_past_qpos_changes_nothing(splits):
    """The attention is causal: a second position array past qpos gives the bits of kvpos = qpos,
    even with NaN in every slot past the rows' query positions (they are never read into o)."""
    import dataclasses
    from gpu_util import DevCase, first_difference
    c = wl.page_case(16, 4, 128, 0, 700, 4, dist="sym", seed=19)
    c = dataclasses.replace(c, qpos=np.array([650, 651, 652, 653], np.int32))
    ref = DevCase(c, splits).result()
    pk = c.k_pool.copy().reshape(c.npg, c.nkv, 16, c.hd)
    pv = c.v_pool.copy().reshape(c.npg, c.nkv, 16, c.hd)
    for pos in range(654, c.npg * 16):
        pk[pos // 16, :, pos % 16, :] = wl.BF16_NAN
        pv[pos // 16, :, pos % 16, :] = wl.BF16_NAN
    ahead = dataclasses.replace(c, k_pool=pk.reshape(-1), v_pool=pv.reshape(-1),
                                kvpos=c.qpos + np.array([1, 5, 16, 40], np.int32))
    d = DevCase(ahead, splits)
    for counters in (True, False):
        got = d.result(counters=counters)
        assert np.array_equal(got, ref), first_difference(got, ref)


def packing_case(kind, seed=31, nh=16, nkv=8, hd=256, window=300):
    """Four rows of one table (g = 2: groups of four rows pack when their windows overlap)."""
    rng = wl.Lcg(seed)
    npages = 40
    n = npages * nkv * 16 * hd
    k = wl.draw_bf16(rng, n, "sym")
    v = wl.draw_bf16(rng, n, "sym")
    rows = 4
    q = wl.draw_bf16(rng, rows * nh * hd, "sym")
    bt = wl.lcg_permutation(npages, seed + 1)
    off = np.zeros(rows, dtype=np.int32)
    if kind == "overlap":        # packed: windows [301..600] .. [330..629] overlap
        qpos = np.array([600, 610, 620, 629], dtype=np.int32)
    elif kind == "disjoint":     # refused: row 0's window ends before the others start
        qpos = np.array([100, 610, 620, 629], dtype=np.int32)
    else:                        # refused: one row has its own span
        qpos = np.array([300, 301, 302, 303], dtype=np.int32)
        off = np.array([0, 0, 5, 0], dtype=np.int32)
    return wl.Case(f"pack_{kind}", nh, nkv, hd, window, rows, q, k, v, bt, off, qpos, ctx=640, npg=npages)


@pytest.mark.parametrize("kind", ["overlap", "disjoint", "mixed_off"])
@pytest.mark.parametrize("splits", [1, 3, 19])
def test_row_packing_groups(kind, splits):
    from gpu_util import DevCase
    c = packing_case(kind)
    d = DevCase(c, splits)
    a = d.result(counters=True)
    check_parity(c, a, f"{kind} s{splits}")
    assert np.array_equal(a, d.result(counters=False))


def test_nan_outside_windows_never_reaches_output():
    """Slots of read pages outside every row's [lo, hi] and whole unread pages hold NaN."""
    from gpu_util import DevCase, first_difference
    c = wl.page_case(16, 8, 256, 1024, 1500, 5, dist="sym", seed=3)
    d = DevCase(c, 6)
    clean = d.result()
    poisoned_k = c.k_pool.copy().reshape(c.npg, c.nkv, 16, c.hd)
    poisoned_v = c.v_pool.copy().reshape(c.npg, c.nkv, 16, c.hd)
    lo_min = min(wl.window_lo(int(x), c.window) for x in c.qpos)
    hi_max = int(c.qpos.max())
    for pos in range(c.npg * 16):
        if pos < lo_min or pos > hi_max:
            poisoned_k[pos // 16, :, pos % 16, :] = wl.BF16_NAN
            poisoned_v[pos // 16, :, pos % 16, :] = wl.BF16_NAN
    import dataclasses
    pc = dataclasses.replace(c, k_pool=poisoned_k.reshape(-1), v_pool=poisoned_v.reshape(-1))
    dp = DevCase(pc, 6)
    for counters in (True, False):
        got = dp.result(counters=counters)
        assert np.array_equal(got, clean), first_difference(got, clean)


def test_repeated_calls_and_streams_are_deterministic():
    import torch
    from gpu_util import DevCase
    c = wl.page_case(32, 4, 512, 0, 3000, 2, dist="sym", seed=8)
    d = DevCase(c)
    first = d.result()
    for _ in range(5):
        assert np.array_equal(d.result(), first)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o = d.run(stream=s)
    s.synchronize()
    assert np.array_equal(o.cpu().numpy().view(np.uint16).reshape(first.shape), first)
    assert int(d.cnt.abs().sum().item()) == 0


@pytest.mark.parametrize("make,splits,counters", [
    (lambda: wl.sliding(), 8, True),                                            # cluster merge
    (lambda: wl.page_case(32, 4, 512, 0, 3000, 1, dist="sym", seed=9), 19, False),   # combine kernel
    (lambda: wl.page_case(32, 4, 512, 0, 3000, 1, dist="sym", seed=9), 6, True),     # last-CTA merge
], ids=["cluster8", "combine19", "lastcta6"])
def test_independent_calls_on_several_streams_match_one_stream(make, splits, counters):
    """Independent calls taken in turn by four streams, each stream with its own output, scratch and
    counters and nothing between the launches (as the bench's concurrent and end-to-end runs issue
    them), give the bits of one call on one stream; every stream's counters end at zero."""
    import torch
    import paged_gqa_decode_attn_gb300 as pgqa
    from gpu_util import DevCase, first_difference
    c = make()
    d = DevCase(c, splits)
    ref = d.result(counters=counters)
    streams = [torch.cuda.Stream() for _ in range(4)]
    sets = [(torch.empty_like(d.o), torch.zeros_like(d.part), torch.zeros_like(d.cnt)) for _ in streams]
    torch.cuda.synchronize()
    for i in range(12):
        s = streams[i % 4]
        o, part, cnt = sets[i % 4]
        with torch.cuda.stream(s):
            pgqa.attn_decode(o, part, d.q, d.k, d.v, d.bt, d.off, d.qpos, d.kvpos, c.rows, c.nh, c.nkv, c.hd,
                             c.window, splits, cnt if counters else None, d.pm, s)
    torch.cuda.synchronize()
    pgqa.device_status()
    for o, _, cnt in sets:
        got = o.cpu().numpy().view(np.uint16).reshape(ref.shape)
        assert np.array_equal(got, ref), first_difference(got, ref)
        assert int(cnt.abs().sum().item()) == 0


def test_zero_rows_is_a_no_op():
    import torch
    import paged_gqa_decode_attn_gb300 as pgqa
    x = torch.zeros(16, dtype=torch.int16, device="cuda")
    pgqa.attn_decode(x, None, x, x, x, x, x, x, None, 0, 8, 2, 128, 0, 1)
    torch.cuda.synchronize()
    assert int(x.abs().sum().item()) == 0


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    """A wait that nothing ends (the library's self-test kernel, the kernels' own bounded wait) gives up
    after about a second: device_status reports the timeout once, and the next decode passes the gates."""
    import torch
    import paged_gqa_decode_attn_gb300 as pgqa
    from paged_gqa_decode_attn_gb300 import _lib
    pgqa.device_status()
    pgqa.selftest_bounded_wait()
    torch.cuda.synchronize()
    with pytest.raises(pgqa.PgqaError) as ei:
        pgqa.device_status()
    assert ei.value.status == _lib.PGQA_ERR_DEVICE_TIMEOUT
    pgqa.device_status()              # read once, then clear
    full_gates(wl.page_case(8, 2, 128, 0, 300, 3, dist="sym", seed=11), splits=3, mapped=False)
    pgqa.device_status()


def test_device_status_clean_after_runs():
    import paged_gqa_decode_attn_gb300 as pgqa
    from gpu_util import DevCase
    DevCase(wl.tiny()).result()
    pgqa.device_status()
