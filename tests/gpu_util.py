"""Helpers for the GPU parity tests: upload a workloads.Case and run the library on it.

Only marshalling: the decode itself runs in libpgqa.so's kernels.
"""
import numpy as np
import torch

import paged_gqa_decode_attn_gb300 as pgqa


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
            splits = pgqa.choose_splits(case.kv_len_eff(), rows, case.nkv, nseq)
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
