"""Split-KV paged GQA decode attention, and paged causal prefill, for NVIDIA GB300 (sm_103a).

The compute path is libpgqa.so (hand-written CUDA, C ABI in include/pgqa.h);
this package only builds it, loads it and marshals arguments.  ``workloads``
draws the seeded synthetic inputs used by the tests and the benchmark.
"""
from ._lib import (MAX_SPLITS, PAGE_TOKENS, PgqaError, attn_decode, attn_decode_noalloc, attn_prefill,
                   attn_prefill_split, choose_splits, choose_splits_ex_for, decode_counter_count, decode_kernel_count, decode_part_bytes,
                   device_status, lib_path, load, make_tiles, prefill_rows_per_tile, prefill_split_count,
                   qk_norm_rope_write, selftest_bounded_wait, strerror, trace_buffer, version)
from .builder import build

__all__ = ["attn_decode", "attn_decode_noalloc", "attn_prefill", "attn_prefill_split", "make_tiles", "prefill_rows_per_tile",
           "prefill_split_count",
           "qk_norm_rope_write",
           "choose_splits", "choose_splits_ex_for", "decode_part_bytes", "decode_counter_count", "decode_kernel_count",
           "device_status", "selftest_bounded_wait", "PgqaError", "build", "load", "lib_path", "strerror", "trace_buffer", "version",
           "PAGE_TOKENS", "MAX_SPLITS"]
