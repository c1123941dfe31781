"""Python handle on the f64 CPU oracle (``pgqa_oracle.c``).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference arm load this package.  The library
in ``paged_gqa_decode_attn_gb300/`` neither imports it nor shares code with it.

The oracle follows the f64 ``reference`` function of span-02
``engine/crates/kernels/tests/gpu.rs``; ``pgqa_oracle.c`` states the
definition and the readings taken where the page is silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pgqa_oracle.c")
_LIB = os.path.join(_HERE, "libpgqa_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, so f64 semantics hold)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-fno-fast-math", "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        # PGQA_ORACLE_LIB lets the negative-control test load a deliberately broken build.
        path = os.environ.get("PGQA_ORACLE_LIB") or build()
        lib = ctypes.CDLL(path)
        p = ctypes.c_void_p
        i = ctypes.c_int
        lib.pgqa_oracle_decode.argtypes = [p, p, p, p, p, p, p, p, i, i, i, i, i, p, i, p, p, i]
        lib.pgqa_oracle_decode.restype = ctypes.c_int
        lib.pgqa_oracle_default_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def default_threads() -> int:
    return int(_load().pgqa_oracle_default_threads())


def _ptr(a: Optional[np.ndarray], dtype) -> Optional[int]:
    if a is None:
        return None
    assert a.dtype == dtype and a.flags.c_contiguous, (a.dtype, dtype)
    return a.ctypes.data


def decode(q, k_pool, v_pool, block_table, off, qpos, nh: int, nkv: int, hd: int, window: int,
           kvpos=None, page_map=None, pairs: Optional[Sequence] = None, nthreads: int = 0,
           want_f64: bool = True, want_bf16: bool = True):
    """Run the oracle.

    Arrays are numpy: bf16 as uint16 bits, metadata as int32.  Returns
    ``(f64, bf16)`` shaped ``[rows, nh, hd]`` (or ``[len(pairs), hd]`` when
    ``pairs`` lists (row, head) pairs); an output not asked for is None.
    """
    lib = _load()
    rows = int(np.asarray(qpos).size)
    arrs = {}
    for name, a, dt in (("q", q, np.uint16), ("k", k_pool, np.uint16), ("v", v_pool, np.uint16),
                        ("bt", block_table, np.int32), ("off", off, np.int32),
                        ("qpos", qpos, np.int32), ("kvpos", kvpos, np.int32),
                        ("pm", page_map, np.int32)):
        arrs[name] = None if a is None else np.ascontiguousarray(a, dtype=dt)
    pr = None
    if pairs is not None:
        pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
        n = pr.shape[0]
        shape = (n, hd)
    else:
        n = rows * nh
        shape = (rows, nh, hd)
    o64 = np.empty(shape, dtype=np.float64) if want_f64 else None
    o16 = np.empty(shape, dtype=np.uint16) if want_bf16 else None
    st = lib.pgqa_oracle_decode(
        _ptr(arrs["q"], np.uint16), _ptr(arrs["k"], np.uint16), _ptr(arrs["v"], np.uint16),
        _ptr(arrs["bt"], np.int32), _ptr(arrs["off"], np.int32), _ptr(arrs["qpos"], np.int32),
        _ptr(arrs["kvpos"], np.int32), _ptr(arrs["pm"], np.int32), rows, nh, nkv, hd, window,
        _ptr(pr, np.int32), n, _ptr(o64, np.float64), _ptr(o16, np.uint16), nthreads)
    if st != 0:
        raise RuntimeError(f"oracle failed with status {st}")
    return o64, o16


def decode_case(case, pairs=None, nthreads: int = 0, **kw):
    """Oracle on a ``workloads.Case``-like object (any object with the same fields)."""
    return decode(case.q, case.k_pool, case.v_pool, case.block_table, case.off, case.qpos,
                  case.nh, case.nkv, case.hd, case.window, kvpos=case.kvpos,
                  page_map=case.page_map, pairs=pairs, nthreads=nthreads, **kw)


def rel_rms(a_bf16: np.ndarray, b_bf16: np.ndarray) -> float:
    """sqrt(sum (a-b)^2 / max(sum b^2, 1e-30)) over bf16 values, in f64 (the page's gate)."""
    a = (np.asarray(a_bf16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    b = (np.asarray(b_bf16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    n = float(np.sum((a - b) ** 2))
    d = float(np.sum(b * b))
    return float(np.sqrt(n / max(d, 1e-30)))
