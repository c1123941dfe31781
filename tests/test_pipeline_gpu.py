"""The step before the path and the path together on the GPU.

pegainfer PR #1002 chains its device gates as "anchor -> flat kernel -> paged
prefill -> paged decode": the QK-RMSNorm / RoPE write fills the paged pools, and
attention reads them.  Here the library's K/V write fills the pools and writes
the normed, rotated Q; the decode then reads both, queued behind it on the same
stream with no host round trip.  The reference chains the two f64 oracles on
the host: the prep oracle's Q, K and V, rounded to bf16 (nearest, as the write
stores them), placed at the oracle's slots, then the decode oracle.  No input of
either oracle comes from the GPU.

The decode runs both with more than 8 splits (the combine kernel, whose split
CTAs prefetch K/V into L2 before their dependency wait) and with 4 (the on-chip
cluster merge).  The gates are the decode parity gates: the page's rel-RMS,
the f64 rel-RMS and the per-(row, head) element bound.  The GPU's bf16 Q, K
and V can differ from the rounded oracle values by one unit in the last place
where the f32 arithmetic lands within ~1e-6 of a rounding midpoint (a few in
10^4 elements); that moves a score by far less than the bound allows.
"""
import os
import sys

import numpy as np
import pytest

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from paged_gqa_decode_attn_gb300 import workloads as wl  # noqa: E402

pytestmark = pytest.mark.gpu

SENTINEL = 0x5555


def bf16_rne(x: np.ndarray) -> np.ndarray:
    """bf16 bits of x, rounded to nearest even (finite inputs)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


def reference_case(pc, last: int, window: int):
    """The decode case the two oracles chain to: the last `last` prompt rows attend over the pools the prep
    oracle fills (every position of the prompt is written)."""
    from oracle import prep as op
    q64, k64, v64, slot = op.prep_case(pc)
    npool = pc.npg
    kpool = np.full(npool * pc.nkv * 16 * pc.hd, SENTINEL, dtype=np.uint16)
    vpool = kpool.copy()
    for kh in range(pc.nkv):
        idx = slot[:, None] + kh * 16 * pc.hd + np.arange(pc.hd)[None, :]
        kpool[idx] = bf16_rne(k64[:, kh])
        vpool[idx] = bf16_rne(v64[:, kh])
    rows = np.arange(pc.rows - last, pc.rows)
    return wl.Case(f"pipeline_{pc.name}_last{last}_w{window}", pc.nh, pc.nkv, pc.hd, window, last,
                   bf16_rne(q64[rows]).reshape(-1), kpool, vpool, pc.block_table.astype(np.int32),
                   np.zeros(last, dtype=np.int32), pc.pos[rows].astype(np.int32), ctx=pc.rows, npg=npool)


def run_device(pc, last: int, window: int, splits: int, counters: bool):
    """K/V write of the whole prompt, then the decode of its last rows, on one stream."""
    import torch
    import paged_gqa_decode_attn_gb300 as pgqa
    from gpu_util import dev_i16, dev_i32
    pgqa.build()
    k_pool = torch.full((pc.npg * pc.nkv * 16 * pc.hd,), SENTINEL, dtype=torch.int16, device="cuda")
    v_pool = torch.full_like(k_pool, SENTINEL)
    q_out = torch.full((pc.rows * pc.nh * pc.hd,), SENTINEL, dtype=torch.int16, device="cuda")
    bt = dev_i32(pc.block_table)
    pgqa.qk_norm_rope_write(q_out, k_pool, v_pool, dev_i16(pc.q_in), dev_i16(pc.k_in), dev_i16(pc.v_in),
                            dev_i16(pc.q_weight), dev_i16(pc.k_weight), dev_i32(pc.pos), bt, dev_i32(pc.off),
                            None, pc.rows, pc.nh, pc.nkv, pc.hd, pc.rotary_dim, pc.theta, pc.eps, pc.norm_v)
    q = q_out[(pc.rows - last) * pc.nh * pc.hd:]          # the last rows' Q, as written
    qpos = dev_i32(pc.pos[pc.rows - last:])
    off = dev_i32(np.zeros(last, dtype=np.int32))
    o = torch.full((last * pc.nh * pc.hd,), SENTINEL, dtype=torch.int16, device="cuda")
    part = torch.empty(pgqa.decode_part_bytes(last, pc.nh, splits, pc.hd), dtype=torch.uint8, device="cuda")
    cnt = (torch.zeros(pgqa.decode_counter_count(last, pc.nh, pc.nkv), dtype=torch.int32, device="cuda")
           if counters else None)
    pgqa.attn_decode(o, part, q, k_pool, v_pool, bt, off, qpos, None, last, pc.nh, pc.nkv, pc.hd, window,
                     splits, cnt)
    torch.cuda.synchronize()
    pgqa.device_status()                                  # raises if a kernel gave up a wait
    if cnt is not None:
        assert int(cnt.abs().sum()) == 0, "merge counters must end at zero"
    return o.cpu().numpy().view(np.uint16).reshape(last, pc.nh, pc.hd)


@pytest.mark.parametrize("splits,counters", [(13, True), (13, False), (4, True)],
                         ids=["combine_13_counters", "combine_13", "cluster_4"])
@pytest.mark.parametrize("window", [0, 300])
def test_kv_write_then_decode_on_one_stream(splits, counters, window):
    from gpu_util import check_parity
    pc = wl.prep_case(16, 2, 128, 128, rows=1000, ctx=1000, positions="prefill", mapped=True, seed=91)
    got = run_device(pc, 3, window, splits, counters)
    check_parity(reference_case(pc, 3, window), got, label=f"pipeline splits {splits} window {window}")


def test_kv_write_then_decode_hd256_partial_rotation():
    """hd 256, half the dims rotated, V without the norm: the sliding workload's head shape."""
    from gpu_util import check_parity
    pc = wl.prep_case(16, 8, 256, 128, rows=600, ctx=600, positions="prefill", mapped=True, seed=92, norm_v=False)
    got = run_device(pc, 4, 256, 19, True)
    check_parity(reference_case(pc, 4, 256), got, label="pipeline hd256")
