"""ctypes binding of libpgqa.so (include/pgqa.h).  Argument marshalling only:
every step of the decode and the prefill runs in the library's CUDA kernels.  There is no CPU
fallback: without the built library these functions raise."""
from __future__ import annotations

import ctypes
import os

from . import builder as _build

PGQA_OK = 0
PGQA_ERR_INVALID_ARGUMENT = -1
PGQA_ERR_UNSUPPORTED_HD = -2
PGQA_ERR_MISALIGNED = -3
PGQA_ERR_CUDA = -4
PGQA_ERR_TENSOR_MAP = -5
PGQA_ERR_DEVICE_TIMEOUT = -6
PGQA_ERR_TOO_MANY_SPLITS = -7
PGQA_ERR_NOALLOC_TOO_LARGE = -8
PGQA_ERR_TILE_TOO_LONG = -9
NOALLOC_MAX_COUNTERS = 16384
NOALLOC_MAX_PART_BYTES = 8 * 1024 * 1024
PAGE_TOKENS = 16
MAX_SPLITS = 256

# name -> (restype, argtypes)
_P, _I = ctypes.c_void_p, ctypes.c_int
SIGNATURES = {
    "pgqa_attn_decode": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P]),
    "pgqa_choose_splits": (_I, [_I, _I, _I, _I]),
    "pgqa_choose_splits_for": (_I, [_I, _I, _I, _I, _I]),
    "pgqa_choose_splits_ex": (_I, [_I, _I, _I, _I, _I, _I]),
    "pgqa_choose_splits_ex_for": (_I, [_I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I]),
    "pgqa_decode_part_bytes": (ctypes.c_size_t, [_I, _I, _I, _I]),
    "pgqa_decode_counter_count": (ctypes.c_size_t, [_I, _I, _I]),
    "pgqa_decode_kernel_count": (_I, [_I, _I]),
    "pgqa_selftest_bounded_wait": (_I, [_P]),
    "pgqa_device_status": (_I, []),
    "pgqa_strerror": (ctypes.c_char_p, [_I]),
    "pgqa_version": (_I, []),
    "pgqa_trace_buffer": (_I, [_P, ctypes.c_size_t]),
    "pgqa_attn_decode_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P]),
    "pgqa_attn_prefill": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P]),
    "pgqa_attn_prefill_split": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I,
                                     _P, _P]),
    "pgqa_prefill_split_count": (_I, [_I, _I, _I, _I, _I]),
    "pgqa_prefill_split_count_ex": (_I, [_I, _I, _I, _I, _I, _I]),
    "pgqa_prefill_rows_per_tile": (_I, [_I]),
    "pgqa_make_tiles": (_I, [_P, _I, _I, _P, _P, _I]),
    "pgqa_qk_norm_rope_write": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                                     ctypes.c_float, ctypes.c_float, _I, _P]),
}


class PgqaError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {strerror(status)} ({status})" if what else f"{strerror(status)} ({status})")


_lib = None


def lib_path() -> str:
    return _build.lib_path(os.environ.get("PGQA_VARIANT", ""))


def load() -> ctypes.CDLL:
    """Load libpgqa.so (it must have been built: ``paged_gqa_decode_attn_gb300.build.build()``).

    With PGQA_VARIANT=trace in the environment the trace build is loaded instead."""
    global _lib
    if _lib is None:
        path = _build.lib_path(os.environ.get("PGQA_VARIANT", ""))
        if not os.path.exists(path):
            raise ImportError(f"{os.path.basename(path)} is not built ({path}); "
                              "run paged_gqa_decode_attn_gb300.build.build()")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def strerror(status: int) -> str:
    return load().pgqa_strerror(int(status)).decode()


def _ptr(x):
    """A device/host pointer from a torch tensor, an int address, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def attn_decode(o, part, q, k_pool, v_pool, block_table, off, qpos, kvpos, rows: int, nh: int, nkv: int,
                hd: int, window: int, splits: int, counters=None, page_map=None, stream=None) -> None:
    """Split-KV paged GQA decode attention (``pgqa_attn_decode``), enqueued on ``stream``
    (default: torch's current stream).  Tensors are passed by device pointer;
    bf16 buffers may be any 2-byte dtype holding bf16 bits."""
    st = load().pgqa_attn_decode(_ptr(o), _ptr(part), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table),
                                 _ptr(off), _ptr(qpos), _ptr(kvpos), int(rows), int(nh), int(nkv), int(hd),
                                 int(window), int(splits), _ptr(counters), _ptr(page_map), _stream(stream))
    if st != PGQA_OK:
        raise PgqaError(st, "attn_decode")


def attn_decode_noalloc(o, q, k_pool, v_pool, block_table, off, qpos, kvpos, rows: int, nh: int, nkv: int,
                        hd: int, window: int, splits: int, page_map=None, stream=None) -> None:
    """``pgqa_attn_decode_noalloc``: the decode with its scratch in the library's
    static device array, for callers that cannot allocate device memory."""
    st = load().pgqa_attn_decode_noalloc(_ptr(o), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table), _ptr(off),
                                         _ptr(qpos), _ptr(kvpos), int(rows), int(nh), int(nkv), int(hd), int(window),
                                         int(splits), _ptr(page_map), _stream(stream))
    if st != PGQA_OK:
        raise PgqaError(st, "attn_decode_noalloc")


def attn_prefill(o, q, k_pool, v_pool, block_table, off, qpos, kvpos, tile_t0, tile_tn, ntiles: int, nh: int,
                 nkv: int, hd: int, window: int, page_map=None, stream=None) -> None:
    """Paged causal prefill (``pgqa_attn_prefill``) over the tiles ``tile_t0``/``tile_tn``
    (device int32 arrays, e.g. from ``make_tiles``), enqueued on ``stream``."""
    st = load().pgqa_attn_prefill(_ptr(o), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table), _ptr(off),
                                  _ptr(qpos), _ptr(kvpos), _ptr(tile_t0), _ptr(tile_tn), int(ntiles), int(nh),
                                  int(nkv), int(hd), int(window), _ptr(page_map), _stream(stream))
    if st != PGQA_OK:
        raise PgqaError(st, "attn_prefill")


def attn_prefill_split(o, part, q, k_pool, v_pool, block_table, off, qpos, kvpos, tile_t0, tile_tn, ntiles: int,
                       rows: int, nh: int, nkv: int, hd: int, window: int, splits: int, page_map=None,
                       stream=None) -> None:
    """Split-KV tiled attention (``pgqa_attn_prefill_split``): partials in ``part``
    (``decode_part_bytes(rows, nh, splits, hd)`` bytes), merged into ``o``."""
    st = load().pgqa_attn_prefill_split(_ptr(o), _ptr(part), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table),
                                        _ptr(off), _ptr(qpos), _ptr(kvpos), _ptr(tile_t0), _ptr(tile_tn),
                                        int(ntiles), int(rows), int(nh), int(nkv), int(hd), int(window),
                                        int(splits), _ptr(page_map), _stream(stream))
    if st != PGQA_OK:
        raise PgqaError(st, "attn_prefill_split")


def prefill_split_count(kv_len_eff: int, rows: int, ntiles: int, nh: int, nkv: int, hd: int | None = None) -> int:
    """``pgqa_prefill_split_count``, or with ``hd`` given ``pgqa_prefill_split_count_ex``."""
    if hd is None:
        n = int(load().pgqa_prefill_split_count(int(kv_len_eff), int(rows), int(ntiles), int(nh), int(nkv)))
    else:
        n = int(load().pgqa_prefill_split_count_ex(int(kv_len_eff), int(rows), int(ntiles), int(nh), int(nkv),
                                                   int(hd)))
    if n < 0:
        raise PgqaError(n, "prefill_split_count")
    return n


def prefill_rows_per_tile(hd: int) -> int:
    n = int(load().pgqa_prefill_rows_per_tile(int(hd)))
    if n < 0:
        raise PgqaError(n, "prefill_rows_per_tile")
    return n


def make_tiles(seq, rows_per_tile: int):
    """``pgqa_make_tiles`` on a host sequence of per-row keys: (tile_t0, tile_tn) as int32 numpy arrays."""
    import numpy as np
    key = np.ascontiguousarray(np.asarray(seq, dtype=np.int32))
    lib = load()
    n = int(lib.pgqa_make_tiles(key.ctypes.data if key.size else None, int(key.size), int(rows_per_tile),
                                None, None, 0))
    if n < 0:
        raise PgqaError(n, "make_tiles")
    t0 = np.zeros(max(n, 1), dtype=np.int32)
    tn = np.zeros(max(n, 1), dtype=np.int32)
    m = int(lib.pgqa_make_tiles(key.ctypes.data if key.size else None, int(key.size), int(rows_per_tile),
                                t0.ctypes.data, tn.ctypes.data, n))
    if m != n:
        raise PgqaError(m if m < 0 else PGQA_ERR_INVALID_ARGUMENT, "make_tiles")
    return t0[:n], tn[:n]


def qk_norm_rope_write(q_out, k_pool, v_pool, q_in, k_in, v_in, q_weight, k_weight, pos, block_table, off,
                       page_map, rows: int, nh: int, nkv: int, hd: int, rotary_dim: int, theta: float, eps: float,
                       norm_v: bool = True, stream=None) -> None:
    """QK-RMSNorm, rotary embedding and the paged K/V write (``pgqa_qk_norm_rope_write``)."""
    st = load().pgqa_qk_norm_rope_write(_ptr(q_out), _ptr(k_pool), _ptr(v_pool), _ptr(q_in), _ptr(k_in), _ptr(v_in),
                                        _ptr(q_weight), _ptr(k_weight), _ptr(pos), _ptr(block_table), _ptr(off),
                                        _ptr(page_map), int(rows), int(nh), int(nkv), int(hd), int(rotary_dim),
                                        float(theta), float(eps), 1 if norm_v else 0, _stream(stream))
    if st != PGQA_OK:
        raise PgqaError(st, "qk_norm_rope_write")


def choose_splits(kv_len_eff: int, rows: int, nkv: int, nseq: int, num_sms: int | None = None,
                  nh: int | None = None, hd: int | None = None) -> int:
    """Splits per tile: ``pgqa_choose_splits`` (the page's arguments), or, given ``nh`` and ``hd``,
    ``pgqa_choose_splits_ex`` (which knows how rows pack and the hd kernel's residency)."""
    if nh is not None and hd is not None:
        st = int(load().pgqa_choose_splits_ex(int(kv_len_eff), int(rows), int(nkv), int(nseq), int(nh), int(hd)))
        if st < 1:
            raise PgqaError(st, "choose_splits_ex")
        return st
    if num_sms is None:
        return int(load().pgqa_choose_splits(int(kv_len_eff), int(rows), int(nkv), int(nseq)))
    return int(load().pgqa_choose_splits_for(int(kv_len_eff), int(rows), int(nkv), int(nseq), int(num_sms)))


def choose_splits_ex_for(kv_len_eff: int, rows: int, nkv: int, nseq: int, nh: int, hd: int, num_sms: int,
                         ctas_per_sm: int, clusters2: int, clusters4: int, clusters8: int) -> int:
    """``pgqa_choose_splits_ex_for``: the same rule for an explicit device (host arithmetic only)."""
    return int(load().pgqa_choose_splits_ex_for(int(kv_len_eff), int(rows), int(nkv), int(nseq), int(nh), int(hd),
                                                int(num_sms), int(ctas_per_sm), int(clusters2), int(clusters4),
                                                int(clusters8)))


def decode_part_bytes(rows: int, nh: int, splits: int, hd: int) -> int:
    return int(load().pgqa_decode_part_bytes(int(rows), int(nh), int(splits), int(hd)))


def decode_counter_count(rows: int, nh: int, nkv: int) -> int:
    return int(load().pgqa_decode_counter_count(int(rows), int(nh), int(nkv)))


def decode_kernel_count(splits: int, with_counters: bool) -> int:
    return int(load().pgqa_decode_kernel_count(int(splits), int(bool(with_counters))))


def device_status() -> None:
    """Raise PgqaError if a kernel gave up a bounded wait since the last check (synchronises)."""
    st = load().pgqa_device_status()
    if st != PGQA_OK:
        raise PgqaError(st, "device_status")


def selftest_bounded_wait(stream=None) -> None:
    """Enqueue the bounded-wait self-test; the next device_status() then raises PGQA_ERR_DEVICE_TIMEOUT."""
    st = load().pgqa_selftest_bounded_wait(_stream(stream))
    if st != PGQA_OK:
        raise PgqaError(st, "selftest_bounded_wait")


def trace_buffer(buf) -> bool:
    """Point trace builds at a device buffer (torch tensor or None); False in normal builds."""
    nbytes = 0 if buf is None else buf.numel() * buf.element_size()
    return load().pgqa_trace_buffer(_ptr(buf), nbytes) == PGQA_OK


def version() -> int:
    return int(load().pgqa_version())
