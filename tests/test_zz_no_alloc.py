"""The no-allocation entry point (pgqa_attn_decode_noalloc) against the ordinary one.

pgqa_attn_decode_noalloc serves callers that cannot allocate device memory for
the split partials and merge counters: it keeps them in one static device
array of the library.  This file is named so pytest collects it last; it must
pass on its own in a fresh process (the first call on the device looks the
array up) and after every other test (the array then holds an earlier
call's leftovers, and the counters must be cleared by each call).
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

REL_RMS_GATE = 1e-2      # the tolerance every parity test here uses


def _run_both(case, splits):
    import torch
    import paged_gqa_decode_attn_gb300 as pgqa
    from gpu_util import DevCase
    pgqa.build()
    d = DevCase(case, splits)
    ref = d.result(counters=True)          # ordinary entry point, caller-owned scratch
    outs = []
    for _ in range(2):                     # two calls in a row share the static scratch
        o = torch.full((case.rows * case.nh * case.hd,), 0x5555, dtype=torch.int16, device="cuda")
        pgqa.attn_decode_noalloc(o, d.q, d.k, d.v, d.bt, d.off, d.qpos, d.kvpos, case.rows, case.nh, case.nkv,
                                 case.hd, case.window, d.splits, d.pm)
        torch.cuda.synchronize()
        outs.append(o.cpu().numpy().view(np.uint16).reshape(case.rows, case.nh, case.hd))
    pgqa.device_status()
    return ref, outs


@pytest.mark.parametrize("make,splits", [
    (lambda: wl.page_case(16, 8, 256, 1024, 1500, 5), 6),       # the page's first decode case: last-CTA merge
    (lambda: wl.page_case(16, 8, 256, 1024, 1500, 5), 4),       # the same, merged on chip (4-CTA clusters)
    (lambda: wl.sliding(mapped=True), 8),                        # sliding window, page map: 8-CTA clusters
    (lambda: wl.tiny(), 2),                                      # 2-CTA clusters
    (lambda: wl.sliding(mapped=True), 19),                       # the combine kernel
    (lambda: wl.long_ctx(), 38),                                 # 32K context, hd 512, two-level combine
], ids=["page_case_hd256_s6", "page_case_hd256_s4", "sliding_mapped_s8", "tiny_s2", "sliding_mapped_s19",
        "long_32k_s38"])
def test_noalloc_matches_allocating_entry_point_twice(make, splits):
    case = make()
    ref, outs = _run_both(case, splits)
    _, ref16 = oracle.decode_case(case)
    assert oracle.rel_rms(ref, ref16) < REL_RMS_GATE
    for o in outs:
        assert oracle.rel_rms(o, ref) < REL_RMS_GATE
        assert oracle.rel_rms(o, ref16) < REL_RMS_GATE
        assert np.array_equal(o, ref), "same kernel and splits: expected identical bits"


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import paged_gqa_decode_attn_gb300 as pgqa
    from paged_gqa_decode_attn_gb300 import _lib
    pgqa.build()
    lib = pgqa.load()
    fake = 0x10000        # never dereferenced: the size check comes first
    # 64 rows x 64 heads x 256 splits x (512 + 2) x 4 bytes is far above 8 MiB
    st = lib.pgqa_attn_decode_noalloc(fake, fake, fake, fake, fake, fake, fake, None, 64, 64, 8, 512, 0, 256,
                                      None, None)
    assert st == _lib.PGQA_ERR_NOALLOC_TOO_LARGE
    assert "scratch" in pgqa.strerror(st)
