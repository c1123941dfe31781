"""The benchmark's algorithmic byte and FLOP counts against brute-force enumeration.

Every roofline number divides one of these counts by a measured time, so each
is checked here on the CPU against a count that enumerates what the call has
to touch: every (block-table span, position) some row sees, read once per kv
head for K and V, plus Q in and O out; every (row, visible position) pair for
prefill; every head vector read and written for the QK-norm / RoPE write.
The reference arm, which needs no GPU, is run here too, for the keys of its line.
"""
import importlib.util
import os
import random
import sys

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
sys.path.insert(0, ROOT)

from paged_gqa_decode_attn_gb300 import workloads as wl  # noqa: E402


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def visible(qp, kv, window):
    lo = max(0, qp + 1 - window) if window > 0 else 0
    return range(lo, kv + 1)


def brute_decode_bytes(nh, nkv, hd, window, qpos, off, kvpos=None):
    seen = set()
    for r, qp in enumerate(qpos):
        kv = qp if kvpos is None else kvpos[r]
        for t in visible(qp, kv, window):
            if t > qp:               # causal: a second position past qpos adds nothing
                continue
            seen.add((off[r], t))
    return len(seen) * nkv * hd * 2 * 2 + 2 * len(qpos) * nh * hd * 2


@pytest.mark.parametrize("seed", range(40))
def test_decode_bytes_match_brute_force(seed):
    rng = random.Random(seed)
    nkv = rng.choice([1, 2, 4, 8])
    nh = nkv * rng.choice([1, 2, 3, 8])
    hd = rng.choice([64, 128, 256, 512])
    window = rng.choice([0, 0, 1, 5, 17, 64, 300])
    rows = rng.randint(1, 9)
    spans = [0, 100, 250][:rng.randint(1, 3)]
    off = [rng.choice(spans) for _ in range(rows)]
    qpos = [rng.randint(0, 400) for _ in range(rows)]
    kvpos = None
    if rng.random() < 0.4:       # some rows see less than their query position (or nothing), some more
        kvpos = [max(-1, q - rng.randint(-5, 50)) for q in qpos]
    got = wl.algorithmic_bytes(nh, nkv, hd, window, qpos, off, kvpos)
    assert got == brute_decode_bytes(nh, nkv, hd, window, qpos, off, kvpos)


def test_sweep_bytes_equal_the_decode_count_at_every_point():
    b = _bench()
    for hd, ctx, rows, window in wl.sweep_points():
        qpos = list(range(ctx - rows, ctx))
        assert b.sweep_bytes(hd, ctx, rows, window) == wl.algorithmic_bytes(32, 16, hd, window, qpos, [0] * rows)


@pytest.mark.parametrize("seed", range(12))
def test_prefill_flops_match_brute_force(seed):
    b = _bench()
    rng = random.Random(100 + seed)
    nkv = rng.choice([1, 2, 8])
    nh = nkv * rng.choice([1, 2, 4])
    hd = rng.choice([64, 128, 256])
    window = rng.choice([0, 3, 64, 1000])
    rows = rng.randint(1, 40)
    qpos = np.array([rng.randint(0, 300) for _ in range(rows)], dtype=np.int32)
    kvpos = None
    if seed % 2:
        kvpos = np.array([q - rng.randint(-5, 20) for q in qpos], dtype=np.int32)

    class C:
        pass
    c = C()
    c.qpos, c.kvpos, c.window, c.nh, c.hd = qpos, kvpos, window, nh, hd
    pairs = 0
    for r in range(rows):
        hi = int(qpos[r]) if kvpos is None else min(int(qpos[r]), int(kvpos[r]))
        pairs += sum(1 for _ in visible(int(qpos[r]), hi, window))
    assert b.prefill_flops(c) == pairs * 4 * nh * hd


def test_prep_bytes_count_every_head_vector_once_each_way():
    c = wl.prep_case(8, 2, 128, 64, 33, 200, positions="scattered", seed=1)
    read = c.q_in.size + c.k_in.size + c.v_in.size          # bf16 elements read
    written = c.rows * c.nh * c.hd + 2 * c.rows * c.nkv * c.hd   # q_out, and K and V into the pools
    assert c.bytes_moved() == 2 * (read + written)


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` runs the oracle on the host cores alone and prints one JSON line with the
    contract's keys; its cpu_baseline and e2e repeat the line's own value, with no host-device bytes."""
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "2", "--warmup", "1", "--ref-budget", "1"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["e2e"]["d2h_bytes_per_step"] == 0 and d["config"]["workload"].startswith("tiny")
    # the config describes the workload alone, with the keys and values the GPU arm prints for it
    # (run details such as splits and timing go under "run"), so the two lines match
    b = _bench()
    assert d["config"] == json.loads(json.dumps(b.config_of(b.build_case("tiny"))))
    assert not {"splits", "merge", "l2", "timing"} & set(d["config"])


def test_the_default_line_summarises_each_other_workload():
    """The default run times the tiled paths and the K/V write beside the decode workloads: each of their
    workloads builds on the host, and a full line of theirs reduces to the record the default line lists
    (its metric, rate, roofline fraction, launches per call and every spot-check key)."""
    b = _bench()
    assert set(b.EXTRA_OTHER) <= {"prefill_long", "prefill_hd512", "multirow", "prep_long", "prefill_page"}
    for name in b.EXTRA_OTHER:
        assert b.build_case(name).name
    line = {"metric": "paged causal prefill attention TFLOP/s", "value": 700.0, "unit": "TFLOP/s", "steps": 20,
            "ms_per_step": 0.1845, "gpu_launches": 40,
            "config": {"workload": "prefill_nh16_nkv8_hd256_w1024_ctx8192"},
            "run": {"tiles": 64, "spot_check_rel_rms": 0.004, "spot_check_worst": 0.1},
            "roofline": {"bound": "tensor", "frac": 0.37, "kernel": "prefill_tc_kernel<256>", "traffic": 1.0e8}}
    s = b.line_summary(line)
    assert s["workload"] == "prefill_nh16_nkv8_hd256_w1024_ctx8192" and s["us_per_call"] == 184.5
    assert s["value"] == 700.0 and s["unit"] == "TFLOP/s" and s["frac"] == 0.37 and s["bound"] == "tensor"
    assert s["kernels_per_call"] == 2 and s["steps"] == 20 and s["traffic"] == 1.0e8
    assert s["spot_check"] == {"spot_check_rel_rms": 0.004, "spot_check_worst": 0.1}
    line["run"] = {"tiles": 64}
    assert b.line_summary(line)["spot_check"] is None


def test_l2_note_claims_hbm_only_past_three_l2():
    """A run's L2 note says its reads come from HBM only when one rotation of its copies moves at least
    3x L2 (129 MB); a smaller rotation (``--copies 1`` on the sliding workload) is marked a diagnostic."""
    b = _bench()
    big = b.l2_note(48, "pool copies", 48 * 8478720, "every step reads KV from HBM")
    assert big.endswith("every step reads KV from HBM") and "> 3x L2" in big
    small = b.l2_note(1, "pool copies", 8478720, "every step reads KV from HBM")
    assert "HBM" not in small and "<= 3x L2" in small and "diagnostic" in small
    edge = b.l2_note(3, "pool copies", 3 * b.L2_BYTES, "from HBM")
    assert edge.endswith("from HBM")


def test_decode_summary_carries_single_call_latency_and_repeats():
    """Each extra decode workload's record keeps the protocol's other two numbers beside the per-call period:
    the latency of one call alone, and the per-call time of repeated timed regions (median and each)."""
    import types
    b = _bench()
    case = b.build_case("tiny")
    rig = types.SimpleNamespace(case=case, bpc=case.algorithmic_bytes(), splits=8, launches_per_call=1)
    rec = b.decode_summary(rig, 0.08, 20, 0.004, 6788.3, single_us=3.21,
                           repeats={"median": 3.95, "each": [3.95, 3.94, 3.96]})
    assert rec["us_per_call"] == 4.0 and rec["single_call_us"] == 3.21
    assert rec["us_per_call_repeats"]["median"] == 3.95 and len(rec["us_per_call_repeats"]["each"]) == 3
    assert "single_call_us" not in b.decode_summary(rig, 0.08, 20, None, 6788.3)
