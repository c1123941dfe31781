"""Seeded synthetic inputs for paged GQA decode attention.

This module only *draws* inputs: a 64-bit LCG, its bf16 conversion, Box-Muller
Gaussians, and the paged-pool / block-table / page-map construction.  It holds
none of the attention arithmetic, so both the CUDA path's tests and the CPU
oracle can be fed from it without sharing any of the method.

Sources (span-02 ``engine/crates/kernels/tests/gpu.rs``, the kernels crate's
GPU test file):

* ``Rng``: state update ``s = s*6364136223846793005 + 1442695040888963407``
  (wrapping u64) and output ``u32(s >> 33) as f32 / 2^31 - 1``.  The output
  therefore lies in [-1, 0], not [-1, 1); :func:`uniform_page` reproduces it
  bit for bit.
* ``bf``: f32 -> bf16 by keeping the top 16 bits (truncation).
* ``run``: draw order K pool, V pool, Q; ``npg = ceil(ctx/16) + 1`` pages;
  identity block table of ``ceil(ctx/16)`` entries; rows at
  ``qpos = ctx-rows .. ctx-1``; ``off = 0``; seed ``12345 + hd``.
* ``mapped_pool``: logical page ``p >= first_live`` moves to physical page
  ``npg - p`` of an ``npg + 1``-page pool whose other pages hold the bf16 NaN
  ``0x7fc0``; pages below ``first_live`` map to the null page 0.  With a
  permuted block table or several sequences, the live pages are those some
  row's window reads (:func:`live_pages`): the same pages for the page's case.

Readings where the page says nothing (each is stated where it is used):

* "uniform[-1,1)" workloads keep the page's LCG state update but map the top
  24 bits symmetrically: ``x = 2*(s >> 40)/2^24 - 1``.
* Gaussians: Box-Muller on two successive symmetric-LCG uniforms, in f64,
  then f32 and the page's bf16 truncation.  "5% of keys x8": one extra LCG
  stream draws, per (page, kv head, slot), whether that key vector is
  multiplied by 8 (exact in bf16).
* The batched workload's shared table is a Fisher-Yates permutation driven
  by the LCG.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

PAGE = 16                      # tokens per KV page
LCG_A = 6364136223846793005
LCG_C = 1442695040888963407
_M64 = (1 << 64) - 1
BF16_NAN = 0x7FC0              # fill of the null page

_BLOCK = 1 << 16
_JUMP_A: Optional[np.ndarray] = None   # A^k mod 2^64, k = 1.._BLOCK
_JUMP_C: Optional[np.ndarray] = None   # state after k steps from 0


def _jump_tables():
    global _JUMP_A, _JUMP_C
    if _JUMP_A is None:
        a = np.empty(_BLOCK, dtype=np.uint64)
        c = np.empty(_BLOCK, dtype=np.uint64)
        ak, ck = 1, 0
        for k in range(_BLOCK):
            ak = (ak * LCG_A) & _M64
            ck = (ck * LCG_A + LCG_C) & _M64
            a[k] = ak
            c[k] = ck
        _JUMP_A, _JUMP_C = a, c
    return _JUMP_A, _JUMP_C


class Lcg:
    """The page's 64-bit LCG, drawn in vectorised blocks via jump-ahead."""

    def __init__(self, seed: int):
        self.state = seed & _M64

    def step_scalar(self) -> int:
        self.state = (self.state * LCG_A + LCG_C) & _M64
        return self.state

    def states(self, n: int) -> np.ndarray:
        """The next ``n`` states (each taken after its update), as uint64."""
        ja, jc = _jump_tables()
        out = np.empty(n, dtype=np.uint64)
        a_blk, c_blk = int(ja[-1]), int(jc[-1])
        pos = 0
        s = self.state
        while pos < n:
            m = min(_BLOCK, n - pos)
            out[pos:pos + m] = ja[:m] * np.uint64(s) + jc[:m]
            pos += m
            if m == _BLOCK:
                s = (s * a_blk + c_blk) & _M64
            else:
                s = int(out[pos - 1])
        self.state = s
        return out


def bf16_trunc(x: np.ndarray) -> np.ndarray:
    """f32 -> bf16 bits by truncation (the page's ``bf``)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bits -> f32 (the page's ``f``)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def uniform_page(states: np.ndarray) -> np.ndarray:
    """The page's ``Rng::next`` output as f32, in [-1, 0]."""
    hi31 = (states >> np.uint64(33)).astype(np.uint32)
    return hi31.astype(np.float32) / np.float32(2147483648.0) - np.float32(1.0)


def uniform_sym(states: np.ndarray) -> np.ndarray:
    """Symmetric reading of "uniform[-1,1)": 2*(s>>40)/2^24 - 1, exact in f32."""
    u24 = (states >> np.uint64(40)).astype(np.float32)
    return u24 * np.float32(2.0 ** -23) - np.float32(1.0)


_CHUNK = 1 << 24


def draw_bf16(rng: Lcg, n: int, dist: str) -> np.ndarray:
    """``n`` bf16 values (bits) from ``rng`` in the given distribution."""
    out = np.empty(n, dtype=np.uint16)
    pos = 0
    while pos < n:
        m = min(_CHUNK, n - pos)
        if dist == "page":
            out[pos:pos + m] = bf16_trunc(uniform_page(rng.states(m)))
        elif dist == "sym":
            out[pos:pos + m] = bf16_trunc(uniform_sym(rng.states(m)))
        elif dist == "gauss":
            st = rng.states(2 * ((m + 1) // 2))
            u1 = ((st[0::2] >> np.uint64(40)).astype(np.float64) + 1.0) * 2.0 ** -24
            u2 = (st[1::2] >> np.uint64(40)).astype(np.float64) * 2.0 ** -24
            r = np.sqrt(-2.0 * np.log(u1))
            z = np.empty(2 * r.size, dtype=np.float64)
            z[0::2] = r * np.cos(2.0 * math.pi * u2)
            z[1::2] = r * np.sin(2.0 * math.pi * u2)
            out[pos:pos + m] = bf16_trunc(z[:m].astype(np.float32))
        else:
            raise ValueError(f"unknown distribution {dist!r}")
        pos += m
    return out


def scale_peaky_keys(k_pool: np.ndarray, nkv: int, hd: int, seed: int, frac: float = 0.05,
                     factor: float = 8.0) -> np.ndarray:
    """Multiply a seeded ``frac`` of key vectors (one per page, kv head, slot) by ``factor``."""
    rows = k_pool.size // hd
    pick = uniform_sym(Lcg(seed).states(rows)) * np.float32(0.5) + np.float32(0.5) < np.float32(frac)
    kf = bf16_to_f32(k_pool).reshape(rows, hd)
    kf[pick] *= np.float32(factor)
    return bf16_trunc(kf).reshape(k_pool.shape)


def lcg_permutation(n: int, seed: int) -> np.ndarray:
    """Fisher-Yates permutation of 0..n-1 driven by the LCG (top 31 bits)."""
    rng = Lcg(seed)
    perm = list(range(n))
    for i in range(n - 1, 0, -1):
        j = (rng.step_scalar() >> 33) % (i + 1)
        perm[i], perm[j] = perm[j], perm[i]
    return np.asarray(perm, dtype=np.int32)


def mapped_pool(k: np.ndarray, v: np.ndarray, npg: int, nkv: int, hd: int, first_live):
    """Permuted copy of a ``[npg][nkv][16][hd]`` pool with a NaN null page 0.

    A live page ``p`` (``first_live``: an int, meaning pages ``>= first_live``,
    or a boolean mask over the ``npg`` pages) sits at page ``npg - p``; the
    others map to page 0, which (like every unused page) holds bf16 NaN.
    Returns ``(k_mapped, v_mapped, page_map)``.
    """
    if isinstance(first_live, (int, np.integer)):
        mask = np.arange(npg) >= int(first_live)
    else:
        mask = np.asarray(first_live, dtype=bool)
    pe = nkv * PAGE * hd
    mk = np.full((npg + 1) * pe, BF16_NAN, dtype=np.uint16)
    mv = np.full((npg + 1) * pe, BF16_NAN, dtype=np.uint16)
    pmap = np.zeros(npg, dtype=np.int32)
    kf = k.reshape(-1)
    vf = v.reshape(-1)
    for p in np.flatnonzero(mask):
        p = int(p)
        s = npg - p
        pmap[p] = s
        mk[s * pe:(s + 1) * pe] = kf[p * pe:(p + 1) * pe]
        mv[s * pe:(s + 1) * pe] = vf[p * pe:(p + 1) * pe]
    return mk, mv, pmap


def window_lo(qpos: int, window: int) -> int:
    """First visible KV position of a row (saturating ``qpos + 1 - window``)."""
    return max(0, qpos + 1 - window) if window > 0 else 0


@dataclasses.dataclass
class Case:
    """One decode problem: host arrays (bf16 as uint16 bits, int32 metadata)."""
    name: str
    nh: int
    nkv: int
    hd: int
    window: int
    rows: int
    q: np.ndarray
    k_pool: np.ndarray
    v_pool: np.ndarray
    block_table: np.ndarray
    off: np.ndarray
    qpos: np.ndarray
    kvpos: Optional[np.ndarray] = None
    page_map: Optional[np.ndarray] = None
    ctx: int = 0
    npg: int = 0

    def kv_len_eff(self) -> int:
        return min(self.ctx, self.window) if self.window > 0 else self.ctx

    def algorithmic_bytes(self) -> int:
        return algorithmic_bytes(self.nh, self.nkv, self.hd, self.window, self.qpos, self.off,
                                 self.kvpos)


def algorithmic_bytes(nh: int, nkv: int, hd: int, window: int, qpos, off, kvpos=None) -> int:
    """Compulsory bytes of one decode call: in-window KV, Q and O.

    Rows that share a block-table span (equal ``off``) count the union of
    their windows once per kv head; partial-page over-fetch is not counted.
    """
    rows = len(qpos)
    spans = {}
    for r in range(rows):
        qp = int(qpos[r])
        hi = min(qp, int(kvpos[r])) if kvpos is not None else qp     # causal
        lo = window_lo(qp, window)
        if hi < lo:
            continue
        spans.setdefault(int(off[r]), []).append((lo, hi))
    tokens = 0
    for ivs in spans.values():
        ivs.sort()
        cur_lo, cur_hi = ivs[0]
        for lo, hi in ivs[1:]:
            if lo > cur_hi + 1:
                tokens += cur_hi - cur_lo + 1
                cur_lo, cur_hi = lo, hi
            else:
                cur_hi = max(cur_hi, hi)
        tokens += cur_hi - cur_lo + 1
    return tokens * nkv * hd * 2 * 2 + 2 * rows * nh * hd * 2


def page_case(nh: int, nkv: int, hd: int, window: int, ctx: int, rows: int,
              dist: str = "page", seed: Optional[int] = None, name: str = "") -> Case:
    """The page's decode fixture: K pool, V pool, then Q from one LCG stream."""
    rng = Lcg(12345 + hd if seed is None else seed)
    npg = (ctx + PAGE - 1) // PAGE + 1
    n = npg * nkv * PAGE * hd
    k = draw_bf16(rng, n, dist)
    v = draw_bf16(rng, n, dist)
    q = draw_bf16(rng, rows * nh * hd, dist)
    bt = np.arange((ctx + PAGE - 1) // PAGE, dtype=np.int32)
    qpos = np.arange(ctx - rows, ctx, dtype=np.int32)
    off = np.zeros(rows, dtype=np.int32)
    return Case(name or f"page_nh{nh}_nkv{nkv}_hd{hd}_w{window}_ctx{ctx}_r{rows}", nh, nkv, hd,
                window, rows, q, k, v, bt, off, qpos, ctx=ctx, npg=npg)


def prefill_case(nh: int, nkv: int, hd: int, window: int, ctx: int, decode_rows: int = 0,
                 dist: str = "page", seed: Optional[int] = None, name: str = "") -> Case:
    """The page's prefill fixture: rows at positions 0..ctx-1, off 0, identity table.

    One LCG stream gives the K pool, the V pool, the decode rows' Q (drawn and
    dropped when ``decode_rows`` > 0, so the stream matches the page's test,
    which runs the decode first) and then the ctx rows' Q.
    """
    rng = Lcg(12345 + hd if seed is None else seed)
    npg = (ctx + PAGE - 1) // PAGE + 1
    n = npg * nkv * PAGE * hd
    k = draw_bf16(rng, n, dist)
    v = draw_bf16(rng, n, dist)
    if decode_rows:
        draw_bf16(rng, decode_rows * nh * hd, dist)
    q = draw_bf16(rng, ctx * nh * hd, dist)
    bt = np.arange((ctx + PAGE - 1) // PAGE, dtype=np.int32)
    qpos = np.arange(ctx, dtype=np.int32)
    off = np.zeros(ctx, dtype=np.int32)
    return Case(name or f"prefill_nh{nh}_nkv{nkv}_hd{hd}_w{window}_ctx{ctx}", nh, nkv, hd, window, ctx, q, k, v,
                bt, off, qpos, ctx=ctx, npg=npg)


def live_pages(c: Case) -> np.ndarray:
    """Mask of the physical pages some row's visible window reads, through the block table."""
    mask = np.zeros(c.npg, dtype=bool)
    q = np.asarray(c.qpos, dtype=np.int64)
    hi = q if c.kvpos is None else np.minimum(q, np.asarray(c.kvpos, dtype=np.int64))
    lo = np.maximum(0, q + 1 - c.window) if c.window > 0 else np.zeros_like(q)
    bt = np.asarray(c.block_table)
    for r in np.flatnonzero(hi >= lo):
        o = int(c.off[r])
        mask[bt[o + int(lo[r]) // PAGE:o + int(hi[r]) // PAGE + 1]] = True
    return mask


def with_mapped_pool(c: Case, fold_into_table: bool = False) -> Case:
    """The same KV behind the permuted / NaN-null-page pool.

    Pages no row's window reads map to the NaN page: for the page's one
    sequence with an identity table, those below ``lo(row 0) / 16`` (its
    ``first_live``) and past the last row.  With ``fold_into_table`` the page
    map is composed into the block table instead of being passed separately.
    """
    mk, mv, pmap = mapped_pool(c.k_pool, c.v_pool, c.npg, c.nkv, c.hd, live_pages(c))
    if fold_into_table:
        return dataclasses.replace(c, name=c.name + "_mappedbt", k_pool=mk, v_pool=mv,
                                   block_table=pmap[c.block_table].astype(np.int32), page_map=None)
    return dataclasses.replace(c, name=c.name + "_mapped", k_pool=mk, v_pool=mv, page_map=pmap)


# --- the named workloads ---------------------------------------------------

def tiny() -> Case:
    """nh8 nkv2 hd128, ctx256, one row at qpos 255, full attention; the page's LCG verbatim."""
    return page_case(8, 2, 128, 0, 256, 1, dist="page", name="tiny_nh8_nkv2_hd128_ctx256")


def sliding(mapped: bool = False) -> Case:
    """nh16 nkv8 hd256, ctx8192, rows at qpos 8188..8191, window 1024, symmetric uniform."""
    c = page_case(16, 8, 256, 1024, 8192, 4, dist="sym", name="sliding_nh16_nkv8_hd256_ctx8192_r4_w1024")
    return with_mapped_pool(c) if mapped else c


def long_ctx() -> Case:
    """nh32 nkv4 hd512, ctx32768, one row, full attention, symmetric uniform."""
    return page_case(32, 4, 512, 0, 32768, 1, dist="sym", name="long_nh32_nkv4_hd512_ctx32768")


def batched(rows: int = 64, ctx: int = 4096) -> Case:
    """64 rows x ctx4096, nh32 nkv8 hd128; one shared table (LCG permutation), off[r] = r*ctx/16."""
    nh, nkv, hd = 32, 8, 128
    ppr = ctx // PAGE
    npages = rows * ppr
    rng = Lcg(12345 + hd)
    n = npages * nkv * PAGE * hd
    k = draw_bf16(rng, n, "sym")
    v = draw_bf16(rng, n, "sym")
    q = draw_bf16(rng, rows * nh * hd, "sym")
    bt = lcg_permutation(npages, 12345 + hd + 1)
    off = (np.arange(rows, dtype=np.int32) * ppr).astype(np.int32)
    qpos = np.full(rows, ctx - 1, dtype=np.int32)
    return Case(f"batched_nh32_nkv8_hd128_ctx{ctx}_r{rows}", nh, nkv, hd, 0, rows, q, k, v, bt, off,
                qpos, ctx=ctx, npg=npages)


SWEEP_HD = (128, 256, 512)
SWEEP_CTX = (1024, 4096, 16384, 65536)
SWEEP_ROWS = (1, 4, 16)
SWEEP_WINDOW = (0, 1024, 4096)


def prefill_page() -> Case:
    """The page's first prefill: nh16 nkv8 hd256, window 1024, 1500 rows (after its 5-row decode)."""
    return prefill_case(16, 8, 256, 1024, 1500, decode_rows=5, name="prefill_nh16_nkv8_hd256_w1024_ctx1500")


def prefill_long() -> Case:
    """A measured prefill: nh16 nkv8 hd256, window 1024, 8192 rows (the sliding decode's sequence)."""
    return prefill_case(16, 8, 256, 1024, 8192, dist="sym", name="prefill_nh16_nkv8_hd256_w1024_ctx8192")


def prefill_hd512() -> Case:
    """A measured prefill in the page's second case shape: nh16 nkv2 hd512, full causal, 4096 rows."""
    return prefill_case(16, 2, 512, 0, 4096, dist="sym", name="prefill_nh16_nkv2_hd512_w0_ctx4096")


@dataclasses.dataclass
class PrepCase:
    """One QK-RMSNorm / RoPE / paged K-V write problem (bf16 bits, int32 metadata).

    Row t's K and V land in page block_table[off[t] + pos[t]/16] (through
    page_map when given), slot pos[t] % 16, of [npg][nkv][16][hd] pools.
    """
    name: str
    nh: int
    nkv: int
    hd: int
    rotary_dim: int
    theta: float
    eps: float
    norm_v: bool
    rows: int
    q_in: np.ndarray
    k_in: np.ndarray
    v_in: np.ndarray
    q_weight: np.ndarray
    k_weight: np.ndarray
    pos: np.ndarray
    block_table: np.ndarray
    off: np.ndarray
    page_map: Optional[np.ndarray] = None
    npg: int = 0

    def bytes_moved(self) -> int:
        """Compulsory bytes of one call: the head vectors read and written, weights and metadata aside."""
        return 2 * self.rows * (self.nh + 2 * self.nkv) * self.hd * 2


def prep_case(nh: int, nkv: int, hd: int, rotary_dim: int, rows: int, ctx: int, positions: str = "prefill",
              theta: float = 10000.0, eps: float = 1e-6, norm_v: bool = True, dist: str = "sym",
              seed: int = 77, mapped: bool = False, name: str = "") -> PrepCase:
    """Seeded inputs: Q/K/V rows from one LCG stream, weights around 1, positions
    0..rows-1 ("prefill"), ctx-rows..ctx-1 ("decode") or a seeded shuffle of
    distinct positions below ctx ("scattered"), one sequence whose block table
    is the identity or, with ``mapped``, a seeded permutation of the pool."""
    rng = Lcg(seed)
    q_in = draw_bf16(rng, rows * nh * hd, dist)
    k_in = draw_bf16(rng, rows * nkv * hd, dist)
    v_in = draw_bf16(rng, rows * nkv * hd, dist)
    wq = bf16_trunc(np.float32(1.0) + np.float32(0.5) * uniform_sym(rng.states(hd)))
    wk = bf16_trunc(np.float32(1.0) + np.float32(0.5) * uniform_sym(rng.states(hd)))
    if positions == "prefill":
        pos = np.arange(rows, dtype=np.int32)
    elif positions == "decode":
        pos = np.arange(ctx - rows, ctx, dtype=np.int32)
    else:
        pos = lcg_permutation(ctx, seed + 3)[:rows].astype(np.int32)
    npages = (ctx + PAGE - 1) // PAGE
    bt = lcg_permutation(npages, seed + 5).astype(np.int32) if mapped else np.arange(npages, dtype=np.int32)
    off = np.zeros(rows, dtype=np.int32)
    return PrepCase(name or f"prep_nh{nh}_nkv{nkv}_hd{hd}_rd{rotary_dim}_r{rows}", nh, nkv, hd, rotary_dim,
                    float(theta), float(eps), bool(norm_v), rows, q_in, k_in, v_in, wq, wk, pos, bt, off,
                    npg=npages)


def prep_long() -> PrepCase:
    """A measured prep: the 8192 prompt rows of the sliding sequence, nh16 nkv8 hd256, full rotation."""
    return prep_case(16, 8, 256, 256, 8192, 8192, positions="prefill", name="prep_nh16_nkv8_hd256_rd256_r8192")


def multirow(ctx: int = 32768, rows: int = 16) -> Case:
    """A multi-token decode: ``rows`` rows of one sequence at its last positions
    (speculative verification), nh32 nkv16 hd256, full attention over ``ctx``,
    symmetric uniform; 32 query rows per kv head."""
    return page_case(32, 16, 256, 0, ctx, rows, dist="sym", name=f"multirow_nh32_nkv16_hd256_ctx{ctx}_r{rows}")


def sweep_points():
    """The 108 hybrid-sweep points (hd, ctx, rows, window), in a fixed order."""
    return [(hd, ctx, rows, w) for hd in SWEEP_HD for ctx in SWEEP_CTX
            for rows in SWEEP_ROWS for w in SWEEP_WINDOW]


def sweep(hd: int, ctx: int, rows: int, window: int, mapped: bool = True) -> Case:
    """nh32 nkv16 Gaussian point, 5% of keys x8, permuted pool with the NaN null page."""
    idx = sweep_points().index((hd, ctx, rows, window))
    seed = 12345 + hd + 7919 * idx
    c = page_case(32, 16, hd, window, ctx, rows, dist="gauss", seed=seed,
                  name=f"sweep_hd{hd}_ctx{ctx}_r{rows}_w{window}")
    c.k_pool = scale_peaky_keys(c.k_pool, c.nkv, hd, seed + 1)
    return with_mapped_pool(c) if mapped else c


WORKLOADS = {
    "tiny": tiny,
    "sliding": sliding,
    "long": long_ctx,
    "batched": batched,
}
