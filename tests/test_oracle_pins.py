"""Pins of the f64 oracle against facts that do not come from the oracle itself.

Each test targets a mistake the oracle could plausibly make (a dropped
max-subtraction, a wrong kv-head mapping, an off-by-one window, a page index
that swaps slot and page, a page map applied in the wrong place, RNE instead
of the page's truncating bf16) and checks it against a closed form, a
textbook routine (``scipy.special.softmax``), or a high-precision brute force
written from the definition of the visible set rather than from ``lo``.

The semantics pinned are those of the f64 ``reference`` in span-02
``engine/crates/kernels/tests/gpu.rs`` (scaling 1.0, causal, sliding windows
``qpos - kvpos < window``, pool ``[page][nkv][16][hd]``, output ``bf(o as f32)``).
"""
import math
import os
import sys

import numpy as np
import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import oracle  # noqa: E402
from paged_gqa_decode_attn_gb300 import workloads as wl  # noqa: E402

PAGE = 16


def bf(x):
    """Exact bf16 bits of a value that is representable in bf16."""
    x = np.asarray(x, dtype=np.float32)
    b = wl.bf16_trunc(x).reshape(x.shape)
    assert np.array_equal(wl.bf16_to_f32(b), x), "not bf16-exact"
    return b


def build_pool(dense_k, dense_v, perm=None, extra_pages=0, fill=wl.BF16_NAN):
    """Scatter dense per-position KV ``[ctx][nkv][hd]`` into a paged pool.

    Logical page j goes to physical page ``perm[j]``; other physical pages hold ``fill``.
    Returns (k_pool, v_pool, block_table_for_logical_pages).
    """
    ctx, nkv, hd = dense_k.shape
    npg = (ctx + PAGE - 1) // PAGE
    if perm is None:
        perm = np.arange(npg, dtype=np.int32)
    nphys = int(max(perm)) + 1 + extra_pages
    kp = np.full((nphys, nkv, PAGE, hd), fill, dtype=np.uint16)
    vp = np.full((nphys, nkv, PAGE, hd), fill, dtype=np.uint16)
    for p in range(ctx):
        kp[perm[p // PAGE], :, p % PAGE, :] = dense_k[p]
        vp[perm[p // PAGE], :, p % PAGE, :] = dense_v[p]
    return kp.reshape(-1), vp.reshape(-1), np.asarray(perm, dtype=np.int32)


def small_ints(rng, shape, lo=-3, hi=3):
    return bf(rng.integers(lo, hi + 1, size=shape).astype(np.float32))


def run_oracle(q, kp, vp, bt, off, qpos, nh, nkv, hd, window, kvpos=None, page_map=None):
    o64, o16 = oracle.decode(q, kp, vp, bt, off, np.asarray(qpos, np.int32), nh, nkv, hd, window,
                             kvpos=None if kvpos is None else np.asarray(kvpos, np.int32),
                             page_map=page_map, nthreads=2)
    return o64, o16


def test_one_token_context_returns_v0():
    rng = np.random.default_rng(1)
    nh, nkv, hd = 4, 2, 32
    dk = wl.bf16_trunc(rng.standard_normal((1, nkv, hd)).astype(np.float32))
    dv = wl.bf16_trunc(rng.standard_normal((1, nkv, hd)).astype(np.float32))
    kp, vp, bt = build_pool(dk, dv)
    q = wl.bf16_trunc(rng.standard_normal(nh * hd).astype(np.float32))
    o64, o16 = run_oracle(q, kp, vp, bt, np.zeros(1, np.int32), [0], nh, nkv, hd, 0)
    for h in range(nh):
        v0 = wl.bf16_to_f32(dv[0, h // (nh // nkv)]).astype(np.float64)
        assert np.array_equal(o64[0, h], v0)
        assert np.array_equal(o16[0, h], dv[0, h // (nh // nkv)])


@pytest.mark.parametrize("window", [0, 7, 33])
def test_constant_scores_give_mean_of_window(window):
    rng = np.random.default_rng(2)
    nh, nkv, hd, ctx = 2, 1, 8, 50
    dk = wl.bf16_trunc(rng.standard_normal((ctx, nkv, hd)).astype(np.float32))
    dv = wl.bf16_trunc(rng.standard_normal((ctx, nkv, hd)).astype(np.float32))
    kp, vp, bt = build_pool(dk, dv)
    q = np.zeros(nh * hd, dtype=np.uint16)         # Q = 0: every score is 0
    qp = 41
    o64, _ = run_oracle(q, kp, vp, bt, np.zeros(1, np.int32), [qp], nh, nkv, hd, window)
    first = 0 if window == 0 else max(0, qp + 1 - window)
    vis = wl.bf16_to_f32(dv[first:qp + 1, 0]).astype(np.float64)
    for d in range(hd):
        mean = math.fsum(vis[:, d]) / vis.shape[0]
        assert o64[0, 0, d] == pytest.approx(mean, rel=1e-14, abs=1e-15)


def test_window_one_returns_v_at_qpos():
    rng = np.random.default_rng(3)
    nh, nkv, hd, ctx = 4, 4, 16, 70
    dk = wl.bf16_trunc(rng.standard_normal((ctx, nkv, hd)).astype(np.float32))
    dv = wl.bf16_trunc(rng.standard_normal((ctx, nkv, hd)).astype(np.float32))
    kp, vp, bt = build_pool(dk, dv)
    qpos = [0, 15, 16, 69]
    q = wl.bf16_trunc(rng.standard_normal(len(qpos) * nh * hd).astype(np.float32))
    o64, o16 = run_oracle(q, kp, vp, bt, np.zeros(len(qpos), np.int32), qpos, nh, nkv, hd, 1)
    for r, qp in enumerate(qpos):
        for h in range(nh):
            assert np.array_equal(o16[r, h], dv[qp, h])
            assert np.array_equal(o64[r, h], wl.bf16_to_f32(dv[qp, h]).astype(np.float64))


@pytest.mark.parametrize("nh,nkv", [(8, 2), (16, 8), (32, 4), (6, 3)])
def test_gqa_head_reads_kv_head_h_over_group(nh, nkv):
    rng = np.random.default_rng(4)
    hd, ctx = 8, 40
    dk = wl.bf16_trunc(rng.standard_normal((ctx, nkv, hd)).astype(np.float32))
    consts = np.arange(1, nkv + 1, dtype=np.float32) * 2.0          # distinct per kv head
    dv = np.empty((ctx, nkv, hd), dtype=np.uint16)
    for j in range(nkv):
        dv[:, j, :] = bf(consts[j])
    kp, vp, bt = build_pool(dk, dv)
    q = wl.bf16_trunc(rng.standard_normal(nh * hd).astype(np.float32))
    o64, _ = run_oracle(q, kp, vp, bt, np.zeros(1, np.int32), [ctx - 1], nh, nkv, hd, 0)
    g = nh // nkv
    for h in range(nh):
        np.testing.assert_allclose(o64[0, h], consts[h // g], rtol=1e-14)


def _two_token_expect(qv, k0, k1, v0, v1):
    s0 = math.fsum(float(a) * float(b) for a, b in zip(qv, k0))
    s1 = math.fsum(float(a) * float(b) for a, b in zip(qv, k1))
    delta = s1 - s0
    # O = (v0 + e^delta v1) / (1 + e^delta), written in the overflow-safe form
    if delta > 0:
        w1 = 1.0 / (1.0 + math.exp(-delta))
    else:
        w1 = math.exp(delta) / (1.0 + math.exp(delta))
    return (1.0 - w1) * v0 + w1 * v1, s0, s1


@pytest.mark.parametrize("scale", [1.0, 64.0])
def test_two_token_closed_form(scale):
    """Two visible tokens: O = (v0 + e^d v1)/(1 + e^d), d = s1 - s0.

    With ``scale`` 64 the scores reach the thousands, where exp() without the
    max-subtraction overflows f64.
    """
    rng = np.random.default_rng(5)
    nh, nkv, hd = 2, 1, 16
    biggest = 0.0
    for trial in range(20):
        dk = wl.bf16_trunc((rng.standard_normal((2, nkv, hd)) * scale).astype(np.float32))
        dv = wl.bf16_trunc(rng.standard_normal((2, nkv, hd)).astype(np.float32))
        kp, vp, bt = build_pool(dk, dv)
        q = wl.bf16_trunc((rng.standard_normal(nh * hd) * scale).astype(np.float32))
        o64, _ = run_oracle(q, kp, vp, bt, np.zeros(1, np.int32), [1], nh, nkv, hd, 0)
        for h in range(nh):
            qv = wl.bf16_to_f32(q[h * hd:(h + 1) * hd]).astype(np.float64)
            k0, k1 = (wl.bf16_to_f32(dk[i, 0]).astype(np.float64) for i in range(2))
            v0, v1 = (wl.bf16_to_f32(dv[i, 0]).astype(np.float64) for i in range(2))
            exp_o, s0, s1 = _two_token_expect(qv, k0, k1, v0, v1)
            biggest = max(biggest, abs(s0), abs(s1))
            np.testing.assert_allclose(o64[0, h], exp_o, rtol=1e-12, atol=1e-14)
            assert np.all(np.isfinite(o64[0, h]))
    if scale > 1:
        assert biggest > 710.0          # exp(score) alone would overflow f64 here


def test_large_scores_stay_finite():
    """Scores far above the f64 exp range (~709) still give the dominant token's V."""
    nh, nkv, hd = 1, 1, 4
    dk = np.stack([bf(np.full((1, hd), 30.0, np.float32)), bf(np.full((1, hd), 31.0, np.float32))])
    dv = np.stack([bf(np.full((1, hd), -1.0, np.float32)), bf(np.full((1, hd), 2.0, np.float32))])
    kp, vp, bt = build_pool(dk, dv)
    q = bf(np.full(hd, 16.0, np.float32))         # s0 = 1920, s1 = 1984: gap 64
    o64, _ = run_oracle(q, kp, vp, bt, np.zeros(1, np.int32), [1], nh, nkv, hd, 0)
    w0 = math.exp(-64.0) / (1.0 + math.exp(-64.0))
    np.testing.assert_allclose(o64[0, 0], -1.0 * w0 + 2.0 * (1.0 - w0), rtol=1e-15)


def _brute_force_mp(qv, dense_k, dense_v, qpos, kvpos, window, kh, mp):
    """Softmax without max-subtraction, in 50-digit arithmetic, over the set
    {p : p <= qpos (causal), p <= kvpos, and (window == 0 or qpos - p < window)},
    each condition tested on its own for every position of the dense context."""
    vis = [p for p in range(dense_k.shape[0])
           if p <= qpos and p <= kvpos and (window == 0 or qpos - p < window)]
    if not vis:
        return [mp.mpf(0)] * len(qv)
    s = [mp.fsum(mp.mpf(float(a)) * mp.mpf(float(b)) for a, b in zip(qv, dense_k[p, kh]))
         for p in vis]
    e = [mp.e ** x for x in s]
    z = mp.fsum(e)
    return [mp.fsum(e[i] * mp.mpf(float(dense_v[p, kh, d])) for i, p in enumerate(vis)) / z
            for d in range(len(qv))]


def test_brute_force_tiny_cases():
    """hd <= 4, <= 40 tokens, random windows / positions / kvpos / permutations / offsets."""
    mpmath = pytest.importorskip("mpmath")
    mp = mpmath.mp
    mp.dps = 50
    rng = np.random.default_rng(6)
    for trial in range(60):
        hd = int(rng.integers(1, 5))
        nkv = int(rng.integers(1, 3))
        g = int(rng.integers(1, 3))
        nh = nkv * g
        ctx = int(rng.integers(1, 41))
        rows = int(rng.integers(1, 4))
        window = int(rng.choice([0, 1, 2, 5, 16, 17, 100]))
        dkf = rng.standard_normal((ctx, nkv, hd)).astype(np.float32)
        dvf = rng.standard_normal((ctx, nkv, hd)).astype(np.float32)
        dk, dv = wl.bf16_trunc(dkf), wl.bf16_trunc(dvf)
        npg = (ctx + PAGE - 1) // PAGE
        perm = rng.permutation(npg).astype(np.int32) + 1      # physical page 0 stays NaN
        kp, vp, table = build_pool(dk, dv, perm)
        # rows read the table through distinct offsets into one longer table
        offs = np.arange(rows, dtype=np.int32) * (npg + 1) + 1
        bt = np.zeros(rows * (npg + 1) + 1, dtype=np.int32)
        for r in range(rows):
            bt[offs[r]:offs[r] + npg] = table
        qpos = rng.integers(0, ctx, size=rows).astype(np.int32)
        # the second position array both below and past qpos (past it, causality must win)
        kvpos = np.minimum(qpos + rng.integers(-3, 4, size=rows), ctx - 1).astype(np.int32)
        q = wl.bf16_trunc(rng.standard_normal(rows * nh * hd).astype(np.float32))
        o64, _ = run_oracle(q, kp, vp, bt, offs, qpos, nh, nkv, hd, window, kvpos=kvpos)
        dkv = wl.bf16_to_f32(dk).astype(np.float64)
        dvv = wl.bf16_to_f32(dv).astype(np.float64)
        for r in range(rows):
            for h in range(nh):
                qv = wl.bf16_to_f32(q[(r * nh + h) * hd:(r * nh + h + 1) * hd]).astype(np.float64)
                ref = _brute_force_mp(qv, dkv, dvv, int(qpos[r]), int(kvpos[r]), window, h // g, mp)
                np.testing.assert_allclose(o64[r, h], [float(x) for x in ref], rtol=1e-12,
                                           atol=1e-13, err_msg=f"trial {trial} r{r} h{h}")


def test_paged_matches_dense_library_softmax():
    """A permuted pool + page map + offsets against scipy's softmax on dense rows."""
    special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(7)
    nh, nkv, hd, ctx = 8, 2, 64, 300
    g = nh // nkv
    dk = wl.bf16_trunc(rng.standard_normal((ctx, nkv, hd)).astype(np.float32))
    dv = wl.bf16_trunc(rng.standard_normal((ctx, nkv, hd)).astype(np.float32))
    npg = (ctx + PAGE - 1) // PAGE
    phys = rng.permutation(npg).astype(np.int32) + 3
    kp, vp, _ = build_pool(dk, dv, phys)
    # table holds "virtual" ids; the page map turns them into physical pages
    virt = rng.permutation(npg).astype(np.int32) + 5
    page_map = np.zeros(int(virt.max()) + 1, dtype=np.int32)
    page_map[virt] = phys
    rows = 3
    offs = np.array([0, npg, 2 * npg], dtype=np.int32)
    bt = np.concatenate([virt] * rows).astype(np.int32)
    qpos = np.array([299, 150, 17], dtype=np.int32)
    window = 100
    q = wl.bf16_trunc(rng.standard_normal(rows * nh * hd).astype(np.float32))
    o64, _ = run_oracle(q, kp, vp, bt, offs, qpos, nh, nkv, hd, window, page_map=page_map)
    kd = wl.bf16_to_f32(dk).astype(np.float64)
    vd = wl.bf16_to_f32(dv).astype(np.float64)
    for r in range(rows):
        lo = max(0, int(qpos[r]) + 1 - window)
        for h in range(nh):
            qv = wl.bf16_to_f32(q[(r * nh + h) * hd:(r * nh + h + 1) * hd]).astype(np.float64)
            s = kd[lo:qpos[r] + 1, h // g] @ qv
            ref = special.softmax(s) @ vd[lo:qpos[r] + 1, h // g]
            np.testing.assert_allclose(o64[r, h], ref, rtol=1e-11, atol=1e-13)


def test_key_shift_leaves_output_unchanged():
    """K + c for every key adds q.c to every score of a row: softmax is unchanged."""
    rng = np.random.default_rng(8)
    nh, nkv, hd, ctx = 4, 2, 16, 90
    dk = small_ints(rng, (ctx, nkv, hd))
    dv = wl.bf16_trunc(rng.standard_normal((ctx, nkv, hd)).astype(np.float32))
    c = rng.integers(-2, 3, size=(nkv, hd)).astype(np.float32)
    dk2 = bf(wl.bf16_to_f32(dk) + c[None])
    q = small_ints(rng, (2 * nh * hd,), -2, 2)
    a, _ = run_oracle(q, *build_pool(dk, dv), np.zeros(2, np.int32), [89, 50], nh, nkv, hd, 30)
    b, _ = run_oracle(q, *build_pool(dk2, dv), np.zeros(2, np.int32), [89, 50], nh, nkv, hd, 30)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)


def test_value_shift_shifts_output():
    """V + c gives O + c (the weights sum to one)."""
    rng = np.random.default_rng(9)
    nh, nkv, hd, ctx = 4, 2, 16, 90
    dk = wl.bf16_trunc(rng.standard_normal((ctx, nkv, hd)).astype(np.float32))
    dv = small_ints(rng, (ctx, nkv, hd))
    c = rng.integers(-4, 5, size=(nkv, hd)).astype(np.float32)
    dv2 = bf(wl.bf16_to_f32(dv) + c[None])
    q = wl.bf16_trunc(rng.standard_normal(nh * hd).astype(np.float32))
    a, _ = run_oracle(q, *build_pool(dk, dv), np.zeros(1, np.int32), [70], nh, nkv, hd, 0)
    b, _ = run_oracle(q, *build_pool(dk, dv2), np.zeros(1, np.int32), [70], nh, nkv, hd, 0)
    g = nh // nkv
    for h in range(nh):
        np.testing.assert_allclose(b[0, h], a[0, h] + c[h // g], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("args", [(16, 8, 256, 1024, 1500, 5), (16, 2, 512, 0, 700, 1)])
def test_page_cases_permuted_pool_is_bit_identical(args):
    """The page's own two decode cases: identity pool == page-map pool == folded table, and no
    NaN from the null page reaches the output."""
    c = wl.page_case(*args)
    a64, a16 = oracle.decode_case(c)
    m = wl.with_mapped_pool(c)
    b64, b16 = oracle.decode_case(m)
    f = wl.with_mapped_pool(c, fold_into_table=True)
    c64, c16 = oracle.decode_case(f)
    assert np.all(np.isfinite(a64))
    assert np.array_equal(a64, b64) and np.array_equal(a64, c64)
    assert np.array_equal(a16, b16) and np.array_equal(a16, c16)
    if c.window > 0:
        assert int((m.page_map == 0).sum()) > 0          # some pages really are on the NaN page


def test_bf16_output_truncates():
    """o = 1 + 3*2^-8 is a bf16 tie: the page's bf() truncates it to 0x3f81 (RNE would give 0x3f82)."""
    nh, nkv, hd = 1, 1, 2
    dk = bf(np.zeros((2, 1, hd), np.float32))
    dv = np.stack([bf(np.full((1, hd), 1.0, np.float32)),
                   bf(np.full((1, hd), 1.0 + 3 * 2.0 ** -7, np.float32))])
    kp, vp, bt = build_pool(dk, dv)
    q = bf(np.zeros(hd, np.float32))
    o64, o16 = run_oracle(q, kp, vp, bt, np.zeros(1, np.int32), [1], nh, nkv, hd, 0)
    assert o64[0, 0, 0] == 1.0 + 3 * 2.0 ** -8
    assert int(o16[0, 0, 0]) == 0x3F81
    # a negative value truncates toward zero in magnitude
    kp, vp, bt = build_pool(dk, bf(-wl.bf16_to_f32(dv)))
    _, o16 = run_oracle(q, kp, vp, bt, np.zeros(1, np.int32), [1], nh, nkv, hd, 0)
    assert int(o16[0, 0, 0]) == 0xBF81


def test_row_with_no_visible_position_is_zero():
    rng = np.random.default_rng(10)
    nh, nkv, hd, ctx = 2, 1, 8, 40
    dk = wl.bf16_trunc(rng.standard_normal((ctx, nkv, hd)).astype(np.float32))
    dv = wl.bf16_trunc(rng.standard_normal((ctx, nkv, hd)).astype(np.float32))
    kp, vp, bt = build_pool(dk, dv)
    q = wl.bf16_trunc(rng.standard_normal(nh * hd).astype(np.float32))
    # window 4 at qpos 30 starts at 27; kvpos 20 < 27 leaves nothing visible
    o64, o16 = run_oracle(q, kp, vp, bt, np.zeros(1, np.int32), [30], nh, nkv, hd, 4, kvpos=[20])
    assert np.all(o64 == 0.0) and np.all(o16 == 0)


def test_kvpos_past_qpos_is_causal():
    """The page's ``reference`` attends over ``lo..=qp``: the attention is causal, so a second
    position array past qpos must give exactly the result of kvpos = qpos, and a distinct V at the
    positions past qpos must not leak into the output."""
    rng = np.random.default_rng(11)
    nh, nkv, hd, ctx = 4, 2, 8, 64
    dk = wl.bf16_trunc(rng.standard_normal((ctx, nkv, hd)).astype(np.float32))
    dv = wl.bf16_trunc(rng.standard_normal((ctx, nkv, hd)).astype(np.float32))
    dv[41:] = bf(np.full((ctx - 41, nkv, hd), 1000.0, np.float32))      # loud V past every qpos
    dk[41:] = bf(np.full((ctx - 41, nkv, hd), 4.0, np.float32))         # and keys that would win
    kp, vp, bt = build_pool(dk, dv)
    qpos = [40, 33, 7]
    q = bf(np.abs(wl.bf16_to_f32(wl.bf16_trunc(rng.standard_normal(3 * nh * hd).astype(np.float32)))))
    for window in (0, 5):
        a64, a16 = run_oracle(q, kp, vp, bt, np.zeros(3, np.int32), qpos, nh, nkv, hd, window,
                              kvpos=qpos)
        b64, b16 = run_oracle(q, kp, vp, bt, np.zeros(3, np.int32), qpos, nh, nkv, hd, window,
                              kvpos=[63, 40, 9])
        assert np.array_equal(a64, b64) and np.array_equal(a16, b16)
        assert np.all(np.abs(b64) < 10.0)          # nothing of the loud V past qpos
        n64, _ = run_oracle(q, kp, vp, bt, np.zeros(3, np.int32), qpos, nh, nkv, hd, window)
        assert np.array_equal(a64, n64)            # NULL kvpos means kvpos = qpos


def test_kvpos_below_qpos_shortens_the_range():
    """kvpos < qpos: the row sees [lo, kvpos] only; with Q = 0 the output is that range's mean of V."""
    rng = np.random.default_rng(12)
    nh, nkv, hd, ctx = 2, 1, 8, 50
    dk = wl.bf16_trunc(rng.standard_normal((ctx, nkv, hd)).astype(np.float32))
    dv = wl.bf16_trunc(rng.standard_normal((ctx, nkv, hd)).astype(np.float32))
    kp, vp, bt = build_pool(dk, dv)
    q = np.zeros(nh * hd, dtype=np.uint16)
    for window, qp, kv in ((0, 45, 30), (20, 45, 30), (20, 45, 26)):
        o64, _ = run_oracle(q, kp, vp, bt, np.zeros(1, np.int32), [qp], nh, nkv, hd, window, kvpos=[kv])
        first = 0 if window == 0 else qp + 1 - window
        vis = wl.bf16_to_f32(dv[first:kv + 1, 0]).astype(np.float64)
        for d in range(hd):
            assert o64[0, 0, d] == pytest.approx(math.fsum(vis[:, d]) / vis.shape[0], rel=1e-14, abs=1e-15)


def test_pairs_and_threads_do_not_change_results():
    c = wl.page_case(8, 2, 64, 100, 333, 3, dist="sym", seed=77)
    full64, full16 = oracle.decode_case(c, nthreads=1)
    par64, _ = oracle.decode_case(c, nthreads=5)
    assert np.array_equal(full64, par64)
    pairs = [(2, 7), (0, 0), (1, 3)]
    p64, p16 = oracle.decode_case(c, pairs=pairs)
    for i, (r, h) in enumerate(pairs):
        assert np.array_equal(p64[i], full64[r, h]) and np.array_equal(p16[i], full16[r, h])


def test_rel_rms_definition_values():
    one = bf(np.array([1.0, 2.0], np.float32))
    assert oracle.rel_rms(one, one) == 0.0
    a = bf(np.array([1.0, 0.0], np.float32))
    b = bf(np.array([0.0, 1.0], np.float32))
    assert oracle.rel_rms(a, b) == pytest.approx(math.sqrt(2.0))
    z = bf(np.zeros(2, np.float32))
    assert oracle.rel_rms(a, z) == pytest.approx(math.sqrt(1.0 / 1e-30))
