"""GPU parity of libpgqa's paged causal prefill against the f64 oracle.

The gates follow the prefill part of `run` in span-02
``engine/crates/kernels/tests/gpu.rs``: every row of the sequence, tiled by
``make_tiles`` with ``prefill_rows_per_tile``, is within rel-RMS 1e-2 of the
reference, and the permuted pool behind a page map (and the map folded into
the block table) gives the same bits.  Every element is also held to the
arithmetic bound of ``parity.py`` (c = 2^-6: the tcgen05 kernel, at every head
dim, lets P grow to 2^8 before rescaling).  A prefill row is a decode row at the
same position, so the oracle is the decode oracle over all rows.
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


def prefill_gates(case, mapped=True, seq=None):
    """Parity, then the page-map gate both ways; returns the identity-pool output."""
    from gpu_util import PrefillDev, check_parity, first_difference
    d = PrefillDev(case, seq)
    a = d.result()
    check_parity(case, a, case.name, tiled=True)
    if mapped:
        for fold in (False, True):
            m = wl.with_mapped_pool(case, fold_into_table=fold)
            am = PrefillDev(m, seq).result()
            assert np.array_equal(am, a), f"page map (fold={fold}) differs: " + first_difference(am, a)
    return a, d


@pytest.mark.parametrize("args", [(16, 8, 256, 1024, 1500, 5), (16, 2, 512, 0, 700, 1)],
                         ids=["hd256_w1024_T1500", "hd512_w0_T700"])
def test_page_prefill_cases(args):
    nh, nkv, hd, window, ctx, rows = args
    prefill_gates(wl.prefill_case(nh, nkv, hd, window, ctx, decode_rows=rows))


@pytest.mark.parametrize("hd", [64, 128, 256, 512])
@pytest.mark.parametrize("nh,nkv", [(4, 4), (8, 1), (32, 2), (24, 2), (6, 2)])
def test_head_dims_and_group_sizes(hd, nh, nkv):
    """g = 1, 8, 16, 12 and 3: chunks of 128 query rows cut rows' heads apart for g = 3 and 12; at hd 512
    each chunk runs on a CTA pair, each CTA over half of the head dims."""
    c = wl.prefill_case(nh, nkv, hd, 0, 150, dist="sym", seed=hd + nh)
    prefill_gates(c, mapped=False)


@pytest.mark.parametrize("window", [1, 5, 17, 100, 5000])
def test_windows(window):
    c = wl.prefill_case(16, 4, 128, window, 300, dist="sym", seed=window)
    prefill_gates(c)


def multi_sequence_case(seed=41, nh=16, nkv=4, hd=128, window=0):
    """Three sequences in one call, each with its own span of a permuted block table:
    a 70-row prompt, a 1-row prompt, and a 50-row continuation at positions 80..129
    whose first 80 positions are already in the cache (chunked prefill)."""
    rng = wl.Lcg(seed)
    npages = 40
    n = npages * nkv * 16 * hd
    k = wl.draw_bf16(rng, n, "sym")
    v = wl.draw_bf16(rng, n, "sym")
    perm = wl.lcg_permutation(npages, seed + 1)
    bt = np.concatenate([perm[:5], perm[5:6], perm[6:15]]).astype(np.int32)
    lens = [(0, 70, 0), (5, 1, 0), (6, 50, 80)]          # (off, rows, first position)
    off = np.concatenate([np.full(r, o, np.int32) for o, r, _ in lens])
    qpos = np.concatenate([np.arange(p0, p0 + r, dtype=np.int32) for _, r, p0 in lens])
    rows = len(qpos)
    q = wl.draw_bf16(rng, rows * nh * hd, "sym")
    return wl.Case("prefill_multiseq", nh, nkv, hd, window, rows, q, k, v, bt, off, qpos, ctx=130, npg=npages)


@pytest.mark.parametrize("window", [0, 33])
def test_several_sequences_and_a_continuation(window):
    prefill_gates(multi_sequence_case(window=window), mapped=False)


def many_sequence_case(lens, nh, nkv, hd, window, seed):
    """Sequences given as (rows, first position) in one call, each through its own span
    of one permuted block table."""
    rng = wl.Lcg(seed)
    spans = [(p0 + r + 15) // 16 for r, p0 in lens]
    npages = sum(spans) + 1
    n = npages * nkv * 16 * hd
    k = wl.draw_bf16(rng, n, "sym")
    v = wl.draw_bf16(rng, n, "sym")
    bt = wl.lcg_permutation(npages, seed + 1)[:sum(spans)].astype(np.int32)
    starts = np.cumsum([0] + spans[:-1])
    off = np.concatenate([np.full(r, o, np.int32) for (r, _), o in zip(lens, starts)])
    qpos = np.concatenate([np.arange(p0, p0 + r, dtype=np.int32) for r, p0 in lens])
    rows = len(qpos)
    q = wl.draw_bf16(rng, rows * nh * hd, "sym")
    return wl.Case(f"prefill_{len(lens)}seq_nh{nh}_nkv{nkv}_hd{hd}_w{window}", nh, nkv, hd, window, rows, q, k, v,
                   bt, off, qpos, ctx=int(max(p0 + r for r, p0 in lens)), npg=npages)


@pytest.mark.parametrize("hd,nh,nkv,window", [(64, 16, 16, 0), (128, 32, 16, 300), (256, 16, 8, 700),
                                              (512, 16, 4, 300)])
def test_persistent_grid_many_items(hd, nh, nkv, window):
    """More (tile, kv head, chunk) items than two per SM: each CTA (CTA pair at hd 512)
    serves several items in turn, its ring, S buffers and barriers -- at hd 512 also
    the S exchange buffers -- running across them.  Four sequences -- a 1-row prompt
    (an empty second chunk) and a continuation at position 300 among them -- give
    ragged tiles."""
    import torch
    from gpu_util import PrefillDev
    c = many_sequence_case([(1500, 0), (1, 0), (900, 300), (1700, 0)], nh, nkv, hd, window, seed=hd + window)
    d = PrefillDev(c)
    chunks = (pgqa_rows_per_tile(hd) * (nh // nkv) + 127) // 128
    items = d.ntiles * nkv * chunks
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert items > 2 * sms, f"{items} items do not reach the persistent grid on {sms} SMs"
    prefill_gates(c)


def pgqa_rows_per_tile(hd):
    import paged_gqa_decode_attn_gb300 as pgqa
    return pgqa.prefill_rows_per_tile(hd)


def test_prefill_long_full_size():
    """The benchmark's workload in its launch configuration: 8192 rows, nh16 nkv8 hd256,
    window 1024 (1024 items on the persistent grid), every element against the oracle,
    and the page-map gate."""
    prefill_gates(wl.prefill_long())


def run_split(case, splits, seq=None):
    """pgqa_attn_prefill_split over make_tiles' tiles; bf16 bits [rows][nh][hd]."""
    import torch
    import paged_gqa_decode_attn_gb300 as pgqa
    from gpu_util import PrefillDev
    d = PrefillDev(case, seq)
    part = torch.empty(pgqa.decode_part_bytes(case.rows, case.nh, splits, case.hd) // 4 + 4, dtype=torch.float32,
                       device="cuda")
    d.o.fill_(0x5555)
    pgqa.attn_prefill_split(d.o, part, d.q, d.k, d.v, d.bt, d.off, d.qpos, d.kvpos, d.t0, d.tn, d.ntiles,
                            case.rows, case.nh, case.nkv, case.hd, case.window, splits, d.pm)
    torch.cuda.synchronize()
    assert pgqa.device_status() is None or pgqa.device_status() == 0
    return d.o.cpu().numpy().view(np.uint16).reshape(case.rows, case.nh, case.hd)


@pytest.mark.parametrize("splits", [1, 2, 5, 16])
@pytest.mark.parametrize("hd,window", [(64, 0), (128, 1024), (256, 0), (256, 1024), (512, 0), (512, 1024)])
def test_split_kv_multi_row_decode(hd, window, splits):
    """The tcgen05 large-M path for multi-row decode: 16 rows of one sequence at the
    end of a 3000-token context (32 query rows per kv head, beyond the decode kernel's
    8), each work item cut into `splits` page ranges and merged by the combine kernel:
    against the oracle, and the page-map gate at fixed splits."""
    from gpu_util import check_parity, first_difference
    c = many_sequence_case([(16, 2984)], 32, 16, hd, window, seed=hd + splits)
    a = run_split(c, splits)
    check_parity(c, a, f"{c.name} splits {splits}", tiled=True)
    for fold in (False, True):
        m = wl.with_mapped_pool(c, fold_into_table=fold)
        am = run_split(m, splits)
        assert np.array_equal(am, a), f"page map (fold={fold}) differs: " + first_difference(am, a)


SWEEP_TILED = [(128, 16384, 16, 4096), (128, 65536, 16, 0), (128, 65536, 16, 1024), (256, 4096, 16, 1024),
               (256, 16384, 16, 0), (256, 65536, 16, 4096), (512, 16384, 16, 0), (512, 65536, 16, 4096)]


@pytest.mark.parametrize("pt", SWEEP_TILED, ids=lambda p: "hd%d_ctx%d_r%d_w%d" % p)
def test_sweep_rows16_points_on_the_tiled_split_path(pt):
    """The sweep's 16-row points that the benchmark sends down the tiled tcgen05 path (rows x g > 8;
    CTA pairs at hd 512), routed exactly as it routes them -- make_tiles over one sequence, splits from
    prefill_split_count, the combine kernel merging -- on the sweep's inputs: Gaussian Q/K/V with 5% of
    keys x8, served from the permuted pool with the NaN null page, at 4K to 64K positions."""
    import paged_gqa_decode_attn_gb300 as pgqa
    from gpu_util import check_parity
    hd, ctx, rows, window = pt
    c = wl.sweep(*pt, mapped=True)
    assert rows * (c.nh // c.nkv) > 8
    t0, _ = pgqa.make_tiles(np.zeros(rows, np.int32), pgqa.prefill_rows_per_tile(hd))
    splits = pgqa.prefill_split_count(c.kv_len_eff(), rows, len(t0), c.nh, c.nkv, hd=c.hd)
    assert splits > 1
    check_parity(c, run_split(c, splits), f"{c.name} splits {splits}", tiled=True)


def test_split_kv_several_sequences_and_empty_splits():
    """Three sequences (16 rows at the end of 2000 tokens, a 1-row prompt, 40 rows of a
    continuation) in one call; 13 splits leave the short windows' later splits empty."""
    from gpu_util import check_parity
    c = many_sequence_case([(16, 1984), (1, 0), (40, 500)], 16, 8, 256, 0, seed=7)
    for splits in (4, 13):
        check_parity(c, run_split(c, splits), f"{c.name} splits {splits}", tiled=True)


def test_split_kv_bad_arguments():
    import torch
    import paged_gqa_decode_attn_gb300 as pgqa
    x = torch.zeros(64, dtype=torch.int16, device="cuda")
    with pytest.raises(pgqa.PgqaError):          # no scratch with splits > 1
        pgqa.attn_prefill_split(x, None, x, x, x, x, x, x, None, x, x, 1, 1, 8, 2, 128, 0, 2)
    with pytest.raises(pgqa.PgqaError):          # a head dim the kernels do not take
        pgqa.attn_prefill_split(x, x, x, x, x, x, x, x, None, x, x, 1, 1, 8, 2, 96, 0, 2)


def test_kvpos_below_qpos_and_an_empty_row():
    """Rows that see only up to kvpos < qpos, and one row whose window holds nothing."""
    c = wl.prefill_case(8, 2, 256, 20, 90, dist="sym", seed=5)
    kvpos = c.qpos.copy()
    kvpos[10:40] -= 3
    kvpos[50] = c.qpos[50] - 25         # below lo = qpos - 19: nothing visible
    c = dataclasses.replace(c, kvpos=kvpos)
    a, _ = prefill_gates(c, mapped=False)
    assert np.all(a[50] == 0), "a row with no visible position must be zero"


def test_output_16_byte_aligned_gives_the_same_bits():
    """o needs only 16-byte alignment; the epilogue's whole-sector stores take 32-byte-aligned outputs, and a
    16-byte-aligned one takes the two-store path: the bits must not depend on which."""
    import torch
    import paged_gqa_decode_attn_gb300 as pgqa
    from gpu_util import PrefillDev, first_difference
    c = wl.prefill_case(16, 8, 256, 1024, 300, dist="sym", seed=9)
    d = PrefillDev(c)
    ref = d.result()
    n = c.rows * c.nh * c.hd
    big = torch.full((n + 16,), 0x5555, dtype=torch.int16, device="cuda")
    o16 = big[8:8 + n]                       # 16 bytes past a 32-byte boundary
    assert o16.data_ptr() % 32 == 16
    pgqa.attn_prefill(o16, d.q, d.k, d.v, d.bt, d.off, d.qpos, d.kvpos, d.t0, d.tn, d.ntiles, c.nh, c.nkv, c.hd,
                      c.window, d.pm)
    torch.cuda.synchronize()
    got = o16.cpu().numpy().view(np.uint16).reshape(ref.shape)
    assert np.array_equal(got, ref), first_difference(got, ref)


def test_split_scratch_16_byte_aligned_gives_the_same_bits():
    """The split path's partials go out as whole sectors when part is 32-byte aligned, else in 16-byte
    pieces (the API asks for 16): the merged output must not depend on which."""
    import torch
    import paged_gqa_decode_attn_gb300 as pgqa
    from gpu_util import PrefillDev, first_difference
    c = many_sequence_case([(16, 2984)], 32, 16, 128, 0, seed=5)
    splits = 5
    ref = run_split(c, splits)
    d = PrefillDev(c)
    nf = pgqa.decode_part_bytes(c.rows, c.nh, splits, c.hd) // 4
    big = torch.empty(nf + 8, dtype=torch.float32, device="cuda")
    part = big[4:4 + nf]                     # 16 bytes past a 32-byte boundary
    assert part.data_ptr() % 32 == 16
    d.o.fill_(0x5555)
    pgqa.attn_prefill_split(d.o, part, d.q, d.k, d.v, d.bt, d.off, d.qpos, d.kvpos, d.t0, d.tn, d.ntiles, c.rows,
                            c.nh, c.nkv, c.hd, c.window, splits, d.pm)
    torch.cuda.synchronize()
    got = d.o.cpu().numpy().view(np.uint16).reshape(ref.shape)
    assert np.array_equal(got, ref), first_difference(got, ref)


def test_kvpos_past_qpos_changes_nothing():
    """Causal prefill: kvpos past qpos gives the bits of kvpos = qpos, on the tiled kernel
    (hd 128, 256; hd 512 on CTA pairs) and the split-KV path, with NaN in every slot past
    the last row's position."""
    from gpu_util import PrefillDev, first_difference
    for hd, splits in ((128, 1), (256, 1), (512, 1), (256, 3), (512, 3)):
        c = wl.prefill_case(16, 8, hd, 0, 200, dist="sym", seed=hd)
        rows = 150
        c = dataclasses.replace(c, rows=rows, q=c.q[:rows * c.nh * c.hd], qpos=c.qpos[:rows], off=c.off[:rows])
        ref = PrefillDev(c).result() if splits == 1 else run_split(c, splits)
        pk = c.k_pool.copy().reshape(c.npg, c.nkv, 16, c.hd)
        pv = c.v_pool.copy().reshape(c.npg, c.nkv, 16, c.hd)
        for pos in range(rows, c.npg * 16):
            pk[pos // 16, :, pos % 16, :] = wl.BF16_NAN
            pv[pos // 16, :, pos % 16, :] = wl.BF16_NAN
        ahead = dataclasses.replace(c, k_pool=pk.reshape(-1), v_pool=pv.reshape(-1),
                                    kvpos=c.qpos + 1 + (np.arange(rows, dtype=np.int32) % 30))
        got = PrefillDev(ahead).result() if splits == 1 else run_split(ahead, splits)
        assert np.array_equal(got, ref), f"hd {hd} splits {splits}: " + first_difference(got, ref)


def test_nan_outside_the_union_window_never_reaches_output():
    """Slots before the first row's window and after the last row's position hold NaN."""
    from gpu_util import PrefillDev, first_difference
    c = wl.prefill_case(16, 8, 256, 64, 200, dist="sym", seed=3)
    rows = 150                        # positions 0..149 of a 200-token cache, window 64
    c = dataclasses.replace(c, rows=rows, q=c.q[:rows * c.nh * c.hd], qpos=c.qpos[:rows], off=c.off[:rows])
    clean = PrefillDev(c).result()
    pk = c.k_pool.copy().reshape(c.npg, c.nkv, 16, c.hd)
    pv = c.v_pool.copy().reshape(c.npg, c.nkv, 16, c.hd)
    for pos in range(c.npg * 16):
        if pos > rows - 1:
            pk[pos // 16, :, pos % 16, :] = wl.BF16_NAN
            pv[pos // 16, :, pos % 16, :] = wl.BF16_NAN
    poisoned = dataclasses.replace(c, k_pool=pk.reshape(-1), v_pool=pv.reshape(-1))
    got = PrefillDev(poisoned).result()
    assert np.array_equal(got, clean), first_difference(got, clean)
    # and tiles late in the sequence never read before their window: poison early slots too
    late = dataclasses.replace(c, rows=20, q=c.q[130 * c.nh * c.hd:150 * c.nh * c.hd], qpos=c.qpos[130:150],
                               off=c.off[130:150])
    clean_late = PrefillDev(late).result()
    pk2, pv2 = pk.copy(), pv.copy()
    for pos in range(0, 130 + 1 - 64):
        pk2[pos // 16, :, pos % 16, :] = wl.BF16_NAN
        pv2[pos // 16, :, pos % 16, :] = wl.BF16_NAN
    got_late = PrefillDev(dataclasses.replace(late, k_pool=pk2.reshape(-1), v_pool=pv2.reshape(-1))).result()
    assert np.array_equal(got_late, clean_late), first_difference(got_late, clean_late)


def test_prefill_rows_match_decode_rows():
    """Decode-equals-prefill: the last rows of a prefill, decoded on their own, agree
    within the gate (the two kernels reduce in different orders, so not bit for bit)."""
    from gpu_util import DevCase, PrefillDev
    import oracle
    c = wl.prefill_case(16, 4, 256, 0, 400, dist="sym", seed=9)
    pre = PrefillDev(c).result()
    tail = 8
    dec_case = dataclasses.replace(c, rows=tail, q=c.q[(400 - tail) * c.nh * c.hd:], qpos=c.qpos[-tail:],
                                   off=c.off[-tail:])
    dec = DevCase(dec_case, 4).result(counters=True)
    assert oracle.rel_rms(pre[-tail:], dec) < 1e-2
    assert oracle.rel_rms(dec, pre[-tail:]) < 1e-2


def test_tile_longer_than_rows_per_tile_is_reported_and_skipped():
    import torch
    import paged_gqa_decode_attn_gb300 as pgqa
    from gpu_util import PrefillDev
    rpt = pgqa.prefill_rows_per_tile(128)
    rows = rpt + 1 + 40
    c = wl.prefill_case(8, 2, 128, 0, rows, dist="sym", seed=2)
    d = PrefillDev(c)
    pgqa.device_status()
    d.t0 = torch.tensor([0, rpt + 1], dtype=torch.int32, device="cuda")
    d.tn = torch.tensor([rpt + 1, rows - rpt - 1], dtype=torch.int32, device="cuda")
    d.ntiles = 2
    out = d.result(fill=0x5555)
    with pytest.raises(pgqa.PgqaError) as ei:
        pgqa.device_status()
    assert ei.value.status == pgqa._lib.PGQA_ERR_TILE_TOO_LONG
    assert np.all(out[:rpt + 1] == 0x5555), "the over-long tile must be skipped"
    assert not np.all(out[rpt + 1:] == 0x5555)
    pgqa.device_status()


def test_repeated_calls_and_streams_are_deterministic():
    import torch
    from gpu_util import PrefillDev
    c = wl.prefill_case(32, 4, 512, 0, 130, dist="sym", seed=8)
    d = PrefillDev(c)
    first = d.result()
    for _ in range(3):
        assert np.array_equal(d.result(), first)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o = d.run(stream=s)
    s.synchronize()
    assert np.array_equal(o.cpu().numpy().view(np.uint16).reshape(first.shape), first)


def test_zero_tiles_is_a_no_op():
    import torch
    import paged_gqa_decode_attn_gb300 as pgqa
    x = torch.zeros(16, dtype=torch.int16, device="cuda")
    pgqa.attn_prefill(x, x, x, x, x, x, x, None, x, x, 0, 8, 2, 128, 0)
    torch.cuda.synchronize()
    assert int(x.abs().sum().item()) == 0
