"""Helpers for the GPU parity tests: upload a workloads.Case and run the library on it.

Only marshalling: the decode and the prefill run in libpgqa.so's kernels.
"""
import json
import os

import numpy as np
import torch

import oracle
import paged_gqa_decode_attn_gb300 as pgqa
import parity
from paged_gqa_decode_attn_gb300 import workloads as wl

REL_RMS_GATE = 1e-2


def bits_to_f64(b):
    return wl.bf16_to_f32(b).astype(np.float64)


def parity_verdict(case, got, label="", tiled=False, oracle_case=None):
    """The page's gate (rel-RMS of the bf16 output against the oracle's bf16 output
    < 1e-2) plus two checks of ``parity.py`` against the oracle's f64 values: the
    element bound |o - o64| <= 2^-8 |o64| + c rms_h(o64), c = 2^-7 (decode, hd-512
    prefill) or 2^-6 (``tiled``: the tcgen05 kernels), and rel-RMS against the f64
    values < 2^-8.  The oracle runs on ``oracle_case`` (default:
    ``case``).  Returns (passed, message naming the first element out of bounds), and
    the rel-RMS."""
    ref64, ref16 = oracle.decode_case(oracle_case or case)
    e = oracle.rel_rms(got, ref16)
    g = bits_to_f64(got)
    coef = parity.COEF_TILED if tiled else parity.COEF_DECODE
    bad = parity.beyond_bound(got, ref64, coef)
    if bad.any():
        i = tuple(int(x) for x in np.argwhere(bad)[0])
        return False, (f"{label}: rel_rms {e:.3e}, {int(bad.sum())} elements beyond the bound; first (row, head, "
                       f"dim) {i}: got {g[i]!r}, oracle {ref64[i]!r}"), e
    if not e < REL_RMS_GATE:
        return False, f"{label}: rel_rms {e:.3e} >= {REL_RMS_GATE}", e
    e64 = parity.rel_rms_f64(got, ref64)
    if not e64 < parity.REL_RMS_F64_GATE:
        return False, f"{label}: rel_rms against the f64 values {e64:.3e} >= {parity.REL_RMS_F64_GATE}", e
    _log_error_profile(label, g, ref64, e)
    return True, f"{label}: rel_rms {e:.3e}", e


def check_parity(case, got, label="", tiled=False):
    ok, msg, e = parity_verdict(case, got, label, tiled)
    assert ok, msg
    return e


def _log_error_profile(label, g, ref64, e):
    """With PGQA_PARITY_LOG set, append one JSON line per checked output: the largest error beyond output
    rounding, in units of its (row, head)'s RMS output (the scale of the random rounding of P)."""
    path = os.environ.get("PGQA_PARITY_LOG")
    if not path:
        return
    r = ref64.reshape(-1, ref64.shape[-1])
    d = np.abs(g.reshape(r.shape) - r)
    rms = np.sqrt(np.mean(r * r, axis=-1, keepdims=True))
    excess = d - 2.0 ** -8 * np.abs(r)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(rms > 0, excess / rms, np.where(excess > 0, np.inf, 0.0))
        rel_h = np.sqrt(np.sum(d * d, axis=-1) / np.maximum(np.sum(r * r, axis=-1), 1e-300))
    rec = {"label": str(label), "rel_rms": float(e), "elements": int(d.size),
           "max_excess_over_rms": float(np.max(ratio)),
           "rel_rms_f64": float(np.sqrt(np.sum(d * d) / max(float(np.sum(r * r)), 1e-300))),
           "max_rel_rms_f64_per_head": float(np.max(np.where(np.sum(r * r, axis=-1) > 0, rel_h, 0.0)))}
    with open(path, "a") as f:
        f.write(json.dumps(rec) + "\n")


def dev_i16(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device)


def dev_i32(a, device="cuda"):
    if a is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


class DevCase:
    """A Case resident on the GPU, plus scratch sized for `splits`."""

    def __init__(self, case, splits=None, device="cuda"):
        self.c = case
        self.q = dev_i16(case.q, device)
        self.k = dev_i16(case.k_pool, device)
        self.v = dev_i16(case.v_pool, device)
        self.bt = dev_i32(case.block_table, device)
        self.off = dev_i32(case.off, device)
        self.qpos = dev_i32(case.qpos, device)
        self.kvpos = dev_i32(case.kvpos, device)
        self.pm = dev_i32(case.page_map, device)
        if splits is None:
            rows = case.rows
            nseq = len(set(int(x) for x in case.off))
            splits = pgqa.choose_splits(case.kv_len_eff(), rows, case.nkv, nseq, nh=case.nh, hd=case.hd)
        self.splits = splits
        self.part = torch.zeros(max(1, pgqa.decode_part_bytes(case.rows, case.nh, splits, case.hd)) // 4 + 4,
                                dtype=torch.float32, device=device)
        self.cnt = torch.zeros(max(4096, pgqa.decode_counter_count(case.rows, case.nh, case.nkv)),
                               dtype=torch.int32, device=device)
        self.o = torch.empty(case.rows * case.nh * case.hd, dtype=torch.int16, device=device)

    def run(self, counters=True, stream=None, o=None, splits=None):
        c = self.c
        out = self.o if o is None else o
        out.fill_(0x5555)
        pgqa.attn_decode(out, self.part, self.q, self.k, self.v, self.bt, self.off, self.qpos, self.kvpos,
                         c.rows, c.nh, c.nkv, c.hd, c.window, self.splits if splits is None else splits,
                         self.cnt if counters else None, self.pm, stream)
        return out

    def result(self, **kw) -> np.ndarray:
        out = self.run(**kw)
        torch.cuda.synchronize()
        return out.cpu().numpy().view(np.uint16).reshape(self.c.rows, self.c.nh, self.c.hd)


def first_difference(a: np.ndarray, b: np.ndarray) -> str:
    """Label of the first differing element (flat index and both bit patterns)."""
    fa, fb = a.reshape(-1), b.reshape(-1)
    idx = np.nonzero(fa != fb)[0]
    if idx.size == 0:
        return "identical"
    i = int(idx[0])
    return f"{idx.size} differ; first at {i}: got 0x{int(fa[i]):04x}, expected 0x{int(fb[i]):04x}"


class PrefillDev:
    """A Case resident on the GPU for pgqa_attn_prefill, tiled by the library's make_tiles
    over the per-row keys ``seq`` (default: off)."""

    def __init__(self, case, seq=None, device="cuda"):
        self.c = case
        self.q = dev_i16(case.q, device)
        self.k = dev_i16(case.k_pool, device)
        self.v = dev_i16(case.v_pool, device)
        self.bt = dev_i32(case.block_table, device)
        self.off = dev_i32(case.off, device)
        self.qpos = dev_i32(case.qpos, device)
        self.kvpos = dev_i32(case.kvpos, device)
        self.pm = dev_i32(case.page_map, device)
        t0, tn = pgqa.make_tiles(case.off if seq is None else seq, pgqa.prefill_rows_per_tile(case.hd))
        self.ntiles = len(t0)
        self.t0 = dev_i32(t0 if len(t0) else np.zeros(1, np.int32), device)
        self.tn = dev_i32(tn if len(tn) else np.zeros(1, np.int32), device)
        self.o = torch.empty(case.rows * case.nh * case.hd, dtype=torch.int16, device=device)

    def run(self, stream=None, fill=0x5555):
        c = self.c
        self.o.fill_(fill)
        pgqa.attn_prefill(self.o, self.q, self.k, self.v, self.bt, self.off, self.qpos, self.kvpos, self.t0,
                          self.tn, self.ntiles, c.nh, c.nkv, c.hd, c.window, self.pm, stream)
        return self.o

    def result(self, **kw) -> np.ndarray:
        out = self.run(**kw)
        torch.cuda.synchronize()
        return out.cpu().numpy().view(np.uint16).reshape(self.c.rows, self.c.nh, self.c.hd)
