"""Host-side checks of libpgqa.so that need no GPU: it builds, loads, exports every
symbol include/pgqa.h declares, sizes its scratch, picks splits, and rejects bad
arguments before touching CUDA.  Also pins constants that the header, the
kernels and the Python binding must agree on (a structural source test)."""
import ctypes
import os
import re
import sys

import numpy as np

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import paged_gqa_decode_attn_gb300 as pgqa  # noqa: E402
from paged_gqa_decode_attn_gb300 import _lib  # noqa: E402

HEADER = os.path.join(ROOT, "include", "pgqa.h")
DEVICE = os.path.join(ROOT, "paged_gqa_decode_attn_gb300", "csrc", "pgqa_device.cuh")


@pytest.fixture(scope="module")
def lib():
    pgqa.build()
    return pgqa.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w ]+?\*?\s*(pgqa_\w+)\s*\(", text, re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("pgqa_attn_decode", "pgqa_choose_splits", "pgqa_decode_part_bytes"):
        assert n in names
    assert set(names) <= set(_lib.SIGNATURES), "binding lacks a declared function"


def test_every_declaration_has_its_own_doc_comment():
    """Each function of the boundary is documented where it is declared: the nearest non-blank,
    non-#define line above the declaration closes a comment."""
    lines = open(HEADER).read().splitlines()
    in_comment = False
    checked = []
    for i, ln in enumerate(lines):
        s = ln.strip()
        if in_comment:
            in_comment = "*/" not in s
            continue
        if s.startswith("/*"):
            in_comment = "*/" not in s
            continue
        m = re.match(r"(?:const\s+)?[\w ]+?\*?\s*(pgqa_\w+)\s*\(", s)
        if not m or s.startswith("#"):
            continue
        j = i - 1
        while j >= 0 and (not lines[j].strip() or lines[j].strip().startswith("#define")):
            j -= 1
        assert j >= 0 and lines[j].strip().endswith("*/"), f"{m.group(1)} has no doc comment above it"
        checked.append(m.group(1))
    assert set(checked) == set(declared_functions())


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n
        assert isinstance(getattr(lib, n), ctypes._CFuncPtr)


def test_constants_agree_between_header_kernels_and_binding():
    h = open(HEADER).read()
    dev = open(DEVICE).read()
    hdr = {k: int(v) for k, v in re.findall(r"#define (PGQA_\w+) \(?(-?\d+)\)?", h)}
    assert hdr["PGQA_PAGE_TOKENS"] == int(re.search(r"kPage = (\d+);", dev).group(1)) == _lib.PAGE_TOKENS
    assert hdr["PGQA_MAX_SPLITS"] == int(re.search(r"kMaxSplits = (\d+);", dev).group(1)) == _lib.MAX_SPLITS
    for name in ("OK", "ERR_INVALID_ARGUMENT", "ERR_UNSUPPORTED_HD", "ERR_MISALIGNED", "ERR_CUDA",
                 "ERR_TENSOR_MAP", "ERR_DEVICE_TIMEOUT", "ERR_TOO_MANY_SPLITS", "ERR_NOALLOC_TOO_LARGE",
                 "ERR_TILE_TOO_LONG"):
        assert hdr["PGQA_" + name] == getattr(_lib, "PGQA_" + name)


def test_part_bytes_and_counter_count(lib):
    assert pgqa.decode_part_bytes(4, 16, 8, 256) == 4 * 16 * 8 * 258 * 4     # f32 O, max and sum per split
    assert pgqa.decode_part_bytes(4, 16, 9, 256) == 4 * 16 * 9 * 258 * 4
    assert pgqa.decode_part_bytes(1, 32, 38, 512) == 32 * 38 * 514 * 4
    assert pgqa.decode_part_bytes(1, 32, 1, 512) == 32 * 514 * 4
    assert pgqa.decode_part_bytes(0, 16, 9, 256) == 0
    assert pgqa.decode_counter_count(4, 16, 8) == 32          # g = 2: one subgroup per kv head
    assert pgqa.decode_counter_count(1, 32, 2) == 4           # g = 16: two subgroups of 8 heads
    assert pgqa.decode_counter_count(2, 24, 2) == 8           # g = 12: two subgroups
    assert pgqa.decode_counter_count(2, 10, 3) == 0           # nh % nkv != 0


def test_decode_kernel_count(lib):
    """The in-kernel merges take up to 8 splits; more, or no counters, add the combine kernel."""
    assert pgqa.decode_kernel_count(1, False) == 1 and pgqa.decode_kernel_count(1, True) == 1
    for s in (2, 4, 5, 8):
        assert pgqa.decode_kernel_count(s, True) == 1
        assert pgqa.decode_kernel_count(s, False) == 2
    for s in (9, 38, 256):
        assert pgqa.decode_kernel_count(s, True) == 2
        assert pgqa.decode_kernel_count(s, False) == 2
    assert pgqa.decode_kernel_count(0, True) == 0 and pgqa.decode_kernel_count(257, False) == 0


def test_choose_splits_rule(lib):
    for kv in (1, 15, 16, 64, 1000, 1024, 4096, 32768, 1 << 20):
        for rows in (1, 4, 16, 64):
            for nkv in (1, 2, 4, 8, 16):
                s = pgqa.choose_splits(kv, rows, nkv, rows, num_sms=152)
                pages = (kv + 15) // 16
                assert 1 <= s <= pgqa.MAX_SPLITS
                assert s == 1 or s <= pages // 2           # at least two pages per split
                assert s == 1 or rows * nkv * (s - 1) < 4 * 152   # no more splits than needed
    # the named workloads (152 SMs): one wave for few tiles, ~4 CTAs per SM for many
    assert pgqa.choose_splits(256, 1, 2, 1, num_sms=152) == 8           # capped at 2 pages per split
    assert pgqa.choose_splits(1024, 4, 8, 1, num_sms=152) == 8          # 4 rows of one sequence packed; 19 -> 8
    assert pgqa.choose_splits(1024, 4, 8, 4, num_sms=152) == 4          # 4 independent rows; 5 -> 4
    assert pgqa.choose_splits(32768, 1, 4, 1, num_sms=152) == 38
    assert pgqa.choose_splits(4096, 64, 8, 64, num_sms=152) == 2
    # up to 24 the count is a power of two of at most 8 (on-chip merge), above it is not rounded
    # GB300 residency: 76 clusters of 2, 36 of 4, 15 of 8.  A count whose clusters
    # are not all resident (merged by the last CTA instead) is taken only when a
    # smaller resident cluster would leave each CTA more than 16 pages longer.
    res = {2: 76, 4: 36, 8: 15}
    for kv in (256, 1024, 4096, 1 << 16):
        pages = (kv + 15) // 16
        for tiles in range(1, 160):
            s = pgqa.choose_splits(kv, tiles, 1, tiles, num_sms=152)
            assert s > 24 or (s in (1, 2, 4, 8))
            if s in (2, 4, 8) and tiles <= 76 and res[s] < tiles:
                fit = max([c for c in (2, 4) if c < s and res[c] >= tiles], default=0)
                assert fit and pages // fit - pages // s > 16 and tiles * s <= 152, (kv, tiles, s)
    assert pgqa.choose_splits(1 << 16, 15, 1, 15, num_sms=152) == 8
    # 16 clusters of 8 would take 2 waves: on chip, 4 splits; the 4096-page loop
    # makes 8 splits merged by the last CTA worth it (128 CTAs: one wave)
    assert pgqa.choose_splits(1 << 16, 16, 1, 16, num_sms=152) == 8
    assert pgqa.choose_splits(1 << 16, 1, 16, 1, num_sms=152) == 8      # one row, 16 kv heads
    assert pgqa.choose_splits(1024, 16, 1, 16, num_sms=152) == 4       # 64 pages: the short loop stays on chip
    assert pgqa.choose_splits(1 << 16, 16, 16, 1, num_sms=152) == 4    # 16 rows: unpacked, 8 splits need 13 waves
    # nseq outside [1, rows] means every row is its own sequence
    assert pgqa.choose_splits(1024, 4, 8, 0, num_sms=152) == pgqa.choose_splits(1024, 4, 8, 4, num_sms=152)
    # without a device the current-device form falls back to 152 SMs
    assert pgqa.choose_splits(32768, 1, 4, 1) >= 1


def test_choose_splits_ex_rule(lib):
    """The head-aware rule on a 152-SM GB300 (one CTA per SM and 76/36/15 clusters of 2/4/8 at hd 256 and
    512; three per SM at hd 64 and 128, with three times the clusters), against its statement in pgqa.h."""
    d1 = dict(num_sms=152, ctas_per_sm=1, clusters2=76, clusters4=36, clusters8=15)
    d3 = dict(num_sms=152, ctas_per_sm=3, clusters2=228, clusters4=108, clusters8=45)
    f = pgqa.choose_splits_ex_for
    # the named workloads keep their counts
    assert f(1024, 4, 8, 1, 16, 256, **d1) == 8          # sliding: 8 pages a CTA, on chip
    assert f(32768, 1, 4, 1, 32, 512, **d1) == 38        # long: fills 152 SMs, combine kernel
    assert f(256, 1, 2, 1, 8, 128, **d3) == 8            # tiny: capped at two pages per split
    assert f(4096, 64, 8, 64, 32, 128, **d3) == 2        # batched: many tiles, the page-signature rule
    assert f(4096, 64, 8, 64, 32, 128, **d3) == pgqa.choose_splits(4096, 64, 8, 64, num_sms=152)
    # rows of one sequence pack: 4 rows at g = 2 launch the CTAs one row does (and long loops take the same count)
    for hd, d in ((128, d3), (256, d1), (512, d1)):
        assert f(65536, 4, 16, 1, 32, hd, **d) == f(65536, 1, 16, 1, 32, hd, **d)
    # long loops fill the GPU in one wave: one CTA per SM at hd 256 and 512, ~2.5 per SM at hd 128
    for nkv in (2, 4, 8, 16, 32):
        assert f(65536, 1, nkv, 1, 2 * nkv, 256, **d1) == 152 // nkv
        assert f(65536, 1, nkv, 1, 2 * nkv, 512, **d1) == 152 // nkv
        assert f(65536, 1, nkv, 1, 2 * nkv, 128, **d3) == min(380 // nkv, 256)
    # a short loop (each CTA <= 128 KB of K and V with the largest cluster that fits) merges on chip
    assert f(1024, 1, 8, 1, 16, 256, **d1) == 8           # 8 pages x 16 KB
    assert f(1024, 1, 16, 1, 32, 128, **d3) == 8          # 8 pages x 8 KB; 16 clusters of 8 fit at 3 per SM
    assert f(1024, 1, 16, 1, 32, 256, **d1) == 9          # 16 clusters of 8 do not fit; 4 leaves 256 KB
    assert f(4096, 1, 8, 1, 16, 256, **d1) == 19          # 32 pages x 16 KB > 128 KB
    # the budget grows with the query rows a CTA serves: 4 packed rows x g = 2 -> 8 rows -> 512 KB
    assert f(1024, 4, 16, 1, 32, 256, **d1) == 4          # 16 pages x 16 KB on chip, not 9 through the combine
    assert f(1024, 4, 16, 1, 32, 512, **d1) == 4          # 16 pages x 32 KB
    assert f(4096, 4, 16, 1, 32, 256, **d1) == 9          # 64 pages x 16 KB = 1 MB > 512 KB
    assert f(4096, 4, 16, 1, 32, 128, **d3) == 23         # 32 pages: more than 16 a CTA, though 256 KB
    assert f(1024, 4, 16, 1, 32, 128, **d3) == 8          # 8 pages
    # bounds: >= 1, at least two pages per split, at most PGQA_MAX_SPLITS; every g and group size
    for hd, d in ((64, d3), (128, d3), (256, d1), (512, d1)):
        for kv in (1, 16, 100, 1024, 1 << 20):
            for rows, nseq in ((1, 1), (4, 1), (16, 1), (16, 16), (64, 64)):
                for nkv, nh in ((1, 1), (2, 16), (8, 8), (4, 96), (16, 32)):
                    s = f(kv, rows, nkv, nseq, nh, hd, **d)
                    pages = (kv + 15) // 16
                    assert 1 <= s <= pgqa.MAX_SPLITS and (s == 1 or s <= pages // 2), (hd, kv, rows, nkv, nh, s)
    # arguments the rule cannot take
    from paged_gqa_decode_attn_gb300 import _lib
    assert f(1024, 1, 2, 1, 8, 96, **d1) == _lib.PGQA_ERR_UNSUPPORTED_HD
    assert f(1024, 1, 3, 1, 8, 128, **d1) == _lib.PGQA_ERR_INVALID_ARGUMENT
    assert f(1024, 1, 0, 1, 8, 128, **d1) == _lib.PGQA_ERR_INVALID_ARGUMENT


def test_prefill_split_count_ex_errors_and_other_head_dims(lib):
    """The hd form is the base count at hd 64, 128 and 256 (it asks the device only at hd 512), and rejects
    other head dims and the base count's bad sizes."""
    from paged_gqa_decode_attn_gb300 import _lib
    for hd in (64, 128, 256):
        for kv in (100, 1024, 65536):
            assert pgqa.prefill_split_count(kv, 16, 1, 32, 16, hd=hd) == pgqa.prefill_split_count(kv, 16, 1, 32, 16)
    with pytest.raises(pgqa.PgqaError):
        pgqa.prefill_split_count(1024, 16, 1, 32, 16, hd=96)
    assert pgqa.load().pgqa_prefill_split_count_ex(1024, 16, 1, 32, 16, 96) == _lib.PGQA_ERR_UNSUPPORTED_HD
    assert pgqa.load().pgqa_prefill_split_count_ex(1024, 16, 1, 32, 5, 128) == _lib.PGQA_ERR_INVALID_ARGUMENT


def test_prefill_split_count(lib):
    """One wave of live items over the SMs (152 without a device), at least two 64-token blocks a split."""
    assert pgqa.prefill_split_count(65536, 16, 1, 32, 16) == 152 // 16     # 16 rows of one sequence: 16 items
    assert pgqa.prefill_split_count(1024, 16, 1, 32, 16) == 8              # 16 blocks: at most 8 splits
    assert pgqa.prefill_split_count(100, 16, 1, 32, 16) == 1
    assert pgqa.prefill_split_count(8192, 8192, 64, 16, 8) == 1            # many items already fill the SMs
    for bad in ((0, 1, 1, 8, 2), (64, 0, 1, 8, 2), (64, 1, 0, 8, 2), (64, 1, 1, 8, 3)):
        with pytest.raises(pgqa.PgqaError):
            pgqa.prefill_split_count(*bad)


def test_strerror_names_every_code(lib):
    for code in range(-9, 1):
        assert pgqa.strerror(code) != "unknown status"
    assert pgqa.strerror(-99) == "unknown status"


FAKE = 0x10000   # never dereferenced: validation fails first


def call(lib, rows=1, nh=8, nkv=2, hd=128, window=0, splits=1, o=FAKE, part=FAKE, q=FAKE, k=FAKE, v=FAKE,
         bt=FAKE, off=FAKE, qpos=FAKE):
    return lib.pgqa_attn_decode(o, part, q, k, v, bt, off, qpos, None, rows, nh, nkv, hd, window, splits,
                                None, None, None)


@pytest.mark.parametrize("kw,code", [
    (dict(rows=-1), -1), (dict(nh=0), -1), (dict(nkv=0), -1), (dict(nh=10, nkv=4), -1),
    (dict(window=-1), -1), (dict(splits=0), -1), (dict(hd=96), -2), (dict(hd=1024), -2),
    (dict(splits=257), -7), (dict(o=None), -1), (dict(q=None), -1), (dict(k=None), -1),
    (dict(v=None), -1), (dict(bt=None), -1), (dict(off=None), -1), (dict(qpos=None), -1),
    (dict(splits=2, part=None), -1), (dict(k=FAKE + 8), -3), (dict(v=FAKE + 2), -3),
    (dict(q=FAKE + 4), -3), (dict(o=FAKE + 8), -3), (dict(splits=2, part=FAKE + 4), -3),
    (dict(rows=70000), -1),
    (dict(rows=65535, nh=65536, nkv=8192, splits=2), -1),   # rows * nh > INT_MAX: the combine grid
])
def test_bad_arguments_are_rejected_before_any_cuda_call(lib, kw, code):
    assert call(lib, **kw) == code


def test_zero_rows_is_ok_without_a_device(lib):
    assert call(lib, rows=0, o=None, q=None) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(rows=-1), -1), (dict(nh=10, nkv=4), -1), (dict(window=-1), -1), (dict(splits=0), -1),
    (dict(hd=96), -2), (dict(splits=257), -7), (dict(o=None), -1), (dict(q=None), -1), (dict(k=None), -1),
    (dict(v=None), -1), (dict(bt=None), -1), (dict(off=None), -1), (dict(qpos=None), -1),
    (dict(k=FAKE + 8), -3), (dict(v=FAKE + 2), -3), (dict(q=FAKE + 4), -3), (dict(o=FAKE + 8), -3),
    (dict(rows=70000), -8),
])
def test_noalloc_rejects_bad_arguments_before_any_cuda_call(lib, kw, code):
    """The no-allocation entry point runs pgqa_attn_decode's checks before it clears its counters, so a
    rejected call enqueues nothing (here: no device at all, and no CUDA call is reached)."""
    a = dict(rows=1, nh=8, nkv=2, hd=128, window=0, splits=1, o=FAKE, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, off=FAKE,
             qpos=FAKE)
    a.update(kw)
    st = lib.pgqa_attn_decode_noalloc(a["o"], a["q"], a["k"], a["v"], a["bt"], a["off"], a["qpos"], None,
                                      a["rows"], a["nh"], a["nkv"], a["hd"], a["window"], a["splits"], None, None)
    assert st == code


def test_python_binding_raises_on_error(lib):
    with pytest.raises(pgqa.PgqaError) as ei:
        pgqa.attn_decode(FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 1, 8, 2, 96, 0, 1, stream=0)
    assert ei.value.status == -2


# ---------------------------------------------------------------- prefill host side

def test_prefill_rows_per_tile(lib):
    assert [pgqa.prefill_rows_per_tile(h) for h in (64, 128, 256, 512)] == [128, 128, 128, 128]
    assert lib.pgqa_prefill_rows_per_tile(96) == -2


def brute_tiles(seq, rpt):
    t0, tn = [], []
    for r, k in enumerate(seq):
        if r == 0 or k != seq[r - 1] or tn[-1] == rpt:
            t0.append(r)
            tn.append(0)
        tn[-1] += 1
    return t0, tn


@pytest.mark.parametrize("seq,rpt", [([0] * 130, 64), ([0, 0, 1, 1, 1, 2], 2), ([], 4), ([7], 1),
                                     ([3] * 64, 64), ([3] * 65, 64), ([0, 1, 0, 1], 8),
                                     (list(np.repeat([5, 9, 5, 2], [100, 1, 33, 64])), 32)])
def test_make_tiles_matches_brute_force(lib, seq, rpt):
    t0, tn = pgqa.make_tiles(seq, rpt)
    e0, en = brute_tiles(list(seq), rpt)
    assert list(t0) == e0 and list(tn) == en
    assert sum(tn) == len(seq) and all(1 <= n <= rpt for n in tn)


def test_make_tiles_rejects_bad_arguments(lib):
    import ctypes
    seq = (ctypes.c_int32 * 4)(0, 0, 1, 1)
    t0 = (ctypes.c_int32 * 1)()
    tn = (ctypes.c_int32 * 1)()
    assert lib.pgqa_make_tiles(seq, 4, 2, None, None, 0) == 2
    assert lib.pgqa_make_tiles(seq, 4, 2, t0, tn, 1) == -1          # arrays too small
    assert lib.pgqa_make_tiles(seq, 4, 0, None, None, 0) == -1       # rows_per_tile < 1
    assert lib.pgqa_make_tiles(seq, -1, 2, None, None, 0) == -1
    assert lib.pgqa_make_tiles(None, 3, 2, None, None, 0) == -1


def prefill_call(lib, ntiles=1, nh=8, nkv=2, hd=128, window=0, o=FAKE, q=FAKE, k=FAKE, v=FAKE, bt=FAKE,
                 off=FAKE, qpos=FAKE, t0=FAKE, tn=FAKE):
    return lib.pgqa_attn_prefill(o, q, k, v, bt, off, qpos, None, t0, tn, ntiles, nh, nkv, hd, window, None, None)


@pytest.mark.parametrize("kw,code", [
    (dict(ntiles=-1), -1), (dict(nh=0), -1), (dict(nkv=0), -1), (dict(nh=10, nkv=4), -1), (dict(window=-1), -1),
    (dict(hd=96), -2), (dict(o=None), -1), (dict(q=None), -1), (dict(k=None), -1), (dict(v=None), -1),
    (dict(bt=None), -1), (dict(off=None), -1), (dict(qpos=None), -1), (dict(t0=None), -1), (dict(tn=None), -1),
    (dict(k=FAKE + 8), -3), (dict(q=FAKE + 2), -3), (dict(o=FAKE + 4), -3), (dict(nkv=70000, nh=70000), -1),
])
def test_prefill_bad_arguments_are_rejected_before_any_cuda_call(lib, kw, code):
    assert prefill_call(lib, **kw) == code


def split_call(lib, splits=2, rows=4, hd=128, part=FAKE, ntiles=1, nh=8, nkv=2):
    return lib.pgqa_attn_prefill_split(FAKE, part, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, ntiles, rows,
                                       nh, nkv, hd, 0, splits, None, None)


@pytest.mark.parametrize("kw,code", [
    ({"splits": 0}, -1), ({"splits": 257}, -7), ({"hd": 32}, -2), ({"hd": 96}, -2), ({"part": None}, -1),
    ({"rows": 0}, -1), ({"part": FAKE + 4}, -3), ({"nh": 6, "nkv": 4}, -1),
    ({"rows": 65535, "nh": 65536, "nkv": 8192}, -1)])
def test_prefill_split_bad_arguments_are_rejected_before_any_cuda_call(lib, kw, code):
    """splits 1..256; head dims 64..512 only; scratch and a row count with splits > 1; 16-byte alignment."""
    assert split_call(lib, **kw) == code


def test_prefill_zero_tiles_is_ok_without_a_device(lib):
    assert prefill_call(lib, ntiles=0, o=None, q=None) == 0


# ---------------------------------------------------------------- QK-RMSNorm / RoPE / paged write host side

def prep_call(lib, rows=1, nh=8, nkv=2, hd=128, rd=128, theta=10000.0, eps=1e-6, qo=FAKE, kp=FAKE, vp=FAKE,
              qi=FAKE, ki=FAKE, vi=FAKE, wq=FAKE, wk=FAKE, pos=FAKE, bt=FAKE, off=FAKE):
    return lib.pgqa_qk_norm_rope_write(qo, kp, vp, qi, ki, vi, wq, wk, pos, bt, off, None, rows, nh, nkv, hd, rd,
                                       theta, eps, 1, None)


@pytest.mark.parametrize("kw,code", [
    (dict(rows=-1), -1), (dict(nh=0), -1), (dict(nkv=0), -1), (dict(nh=10, nkv=4), -1), (dict(hd=96), -2),
    (dict(rd=130), -1), (dict(rd=-8), -1), (dict(rd=12), -1), (dict(theta=0.0), -1), (dict(theta=float("inf")), -1),
    (dict(eps=-1.0), -1), (dict(qo=None), -1), (dict(kp=None), -1), (dict(vp=None), -1), (dict(qi=None), -1),
    (dict(wk=None), -1), (dict(pos=None), -1), (dict(bt=None), -1), (dict(off=None), -1),
    (dict(ki=FAKE + 8), -3), (dict(vp=FAKE + 2), -3), (dict(wq=FAKE + 4), -3),
])
def test_prep_bad_arguments_are_rejected_before_any_cuda_call(lib, kw, code):
    assert prep_call(lib, **kw) == code


def test_prep_zero_rows_is_ok_without_a_device(lib):
    assert prep_call(lib, rows=0, qo=None) == 0
    assert prep_call(lib, rows=0, rd=0) == 0
