"""Python handle on the f64 oracle of the QK-RMSNorm / RoPE / paged K-V write
(``pgqa_prep_oracle.c``), the step before paged attention.

TEST INFRASTRUCTURE ONLY: only ``tests/`` and ``bench.py``'s CPU-baseline leg
load it; the library in ``paged_gqa_decode_attn_gb300/`` shares no code with it.
``pgqa_prep_oracle.c`` states the definition and the reading taken of pegainfer
PR #1002, which describes the step's device gates but prints no formula.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pgqa_prep_oracle.c")
_LIB = os.path.join(_HERE, "libpgqa_prep_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        # PGQA_PREP_ORACLE_LIB lets the negative-control test load a deliberately broken build.
        lib = ctypes.CDLL(os.environ.get("PGQA_PREP_ORACLE_LIB") or build())
        p, i, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        lib.pgqa_prep_oracle.argtypes = [p, p, p, p, p, p, p, p, p, i, i, i, i, i, dbl, dbl, i, p, p, p, p]
        lib.pgqa_prep_oracle.restype = ctypes.c_int
        _lib = lib
    return _lib


def _arr(a, dtype):
    if a is None:
        return None, None
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


def prep(q_in, k_in, v_in, q_weight, k_weight, pos, block_table, off, page_map, nh: int, nkv: int, hd: int,
         rotary_dim: int, theta: float, eps: float, norm_v: bool):
    """f64 (q_out [rows][nh][hd], k_out [rows][nkv][hd], v_out [rows][nkv][hd], slot [rows])."""
    pos, pp = _arr(pos, np.int32)
    rows = int(pos.size)
    keep = []
    ptrs = []
    for a, dt in ((q_in, np.uint16), (k_in, np.uint16), (v_in, np.uint16), (q_weight, np.uint16),
                  (k_weight, np.uint16)):
        arr, ptr = _arr(a, dt)
        keep.append(arr)
        ptrs.append(ptr)
    bt, bp = _arr(block_table, np.int32)
    of, op = _arr(off, np.int32)
    pm, mp = _arr(page_map, np.int32)
    q_out = np.zeros((rows, nh, hd), np.float64)
    k_out = np.zeros((rows, nkv, hd), np.float64)
    v_out = np.zeros((rows, nkv, hd), np.float64)
    slot = np.zeros(rows, np.int64)
    st = _load().pgqa_prep_oracle(*ptrs, pp, bp, op, mp, rows, nh, nkv, hd, rotary_dim, float(theta), float(eps),
                                  1 if norm_v else 0, q_out.ctypes.data, k_out.ctypes.data, v_out.ctypes.data,
                                  slot.ctypes.data)
    if st != 0:
        raise ValueError("pgqa_prep_oracle: bad sizes")
    return q_out, k_out, v_out, slot


def prep_case(c, pairs_unused=None):
    """The oracle on a workloads.PrepCase."""
    return prep(c.q_in, c.k_in, c.v_in, c.q_weight, c.k_weight, c.pos, c.block_table, c.off, c.page_map, c.nh,
                c.nkv, c.hd, c.rotary_dim, c.theta, c.eps, c.norm_v)
