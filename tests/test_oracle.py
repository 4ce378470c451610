"""Pins of the CPU oracle against what the pages and the mathematics fix.

CPU only.  Each test pins the oracle to something other than itself:
closed forms, invariants, a pure-Python brute force, a library routine
(scipy's logsumexp / softmax), finite differences, and the page's own
printed numbers (tests/golden/fa4_pages.json).
"""
import json
import math
import os

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

from oracle import attention as A
from oracle import online_softmax as OS

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "fa4_pages.json")))


def rnd(shape, seed, std=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * std


# ----------------------------------------------------------------- forward

def test_softmax_rows_sum_to_one():
    s = A._scores(rnd((37, 16), 0), rnd((53, 16), 1), 0.25, causal=False, row0=0)
    p, _ = A._softmax_rows(s)
    assert np.abs(p.sum(1) - 1).max() < 1e-12
    sc = A._scores(rnd((53, 16), 0), rnd((53, 16), 1), 0.25, causal=True, row0=0)
    pc, _ = A._softmax_rows(sc)
    assert np.abs(pc.sum(1) - 1).max() < 1e-12
    assert np.all(np.triu(pc, 1) == 0)  # nothing above the diagonal


@pytest.mark.parametrize("causal", [False, True])
def test_constant_v_gives_v(causal):
    B, N, H, d = 2, 45, 3, 8
    q, k = rnd((B, N, H, d), 2, 3.0), rnd((B, N, H, d), 3)
    v = np.broadcast_to(rnd((1, 1, H, d), 4), (B, N, H, d)).copy()
    o, _ = A.forward(q, k, v, 0.3, causal)
    assert np.abs(o - v).max() < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_zero_q_gives_mean_of_visible_v(causal):
    B, N, H, d = 1, 33, 2, 8
    q = np.zeros((B, N, H, d))
    k, v = rnd((B, N, H, d), 5), rnd((B, N, H, d), 6)
    o, lse = A.forward(q, k, v, 0.125, causal)
    for i in range(N):
        cnt = i + 1 if causal else N
        assert np.abs(o[0, i] - v[0, :cnt].mean(0)).max() < 1e-12
        assert abs(lse[0, 0, i] - math.log(cnt)) < 1e-12


def test_causal_row0_is_v0():
    q, k, v = rnd((1, 20, 2, 8), 7), rnd((1, 20, 2, 8), 8), rnd((1, 20, 2, 8), 9)
    o, _ = A.forward(q, k, v, 0.5, True)
    assert np.abs(o[0, 0] - v[0, 0]).max() < 1e-14


@pytest.mark.parametrize("N,d,causal", [(1, 4, False), (2, 4, True), (17, 8, False), (17, 8, True),
                                        (64, 8, True), (9, 128, False), (9, 64, True), (33, 64, False),
                                        (7, 256, True), (12, 256, False)])
def test_bruteforce_agrees(N, d, causal):
    alpha = 1 / math.sqrt(d)
    q, k, v = rnd((N, d), 10), rnd((N, d), 11), rnd((N, d), 12)
    o_bf, lse_bf = A.bruteforce_forward(q, k, v, alpha, causal)
    o, lse = A.head_forward(q, k, v, alpha, causal)
    assert np.abs(o - np.array(o_bf)).max() < 1e-12
    assert np.abs(lse - np.array(lse_bf)).max() < 1e-12


def test_lse_and_p_match_scipy():
    N, d, alpha = 70, 16, 0.2
    q, k, v = rnd((N, d), 13, 2.0), rnd((N, d), 14), rnd((N, d), 15)
    o, lse = A.head_forward(q, k, v, alpha, causal=False)
    s = alpha * q @ k.T
    assert np.abs(lse - logsumexp(s, axis=1)).max() < 1e-12
    assert np.abs(o - softmax(s, axis=1) @ v).max() < 1e-12


def test_gqa_equals_repeated_heads():
    B, N, Hq, Hkv, d = 2, 19, 6, 2, 8
    q, k, v = rnd((B, N, Hq, d), 16), rnd((B, N, Hkv, d), 17), rnd((B, N, Hkv, d), 18)
    o, lse = A.forward(q, k, v, 0.3, True)
    g = Hq // Hkv
    o2, lse2 = A.forward(q, np.repeat(k, g, axis=2), np.repeat(v, g, axis=2), 0.3, True)
    assert np.abs(o - o2).max() < 1e-14 and np.abs(lse - lse2).max() < 1e-14
    # head 3 must read kv head 1 (contiguous groups), not kv head 3 % 2
    oh, _ = A.head_forward(q[0, :, 3], k[0, :, 1], v[0, :, 1], 0.3, True)
    assert np.abs(o[0, :, 3] - oh).max() < 1e-14


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_equals_separate_sequences(causal):
    lens = [5, 0, 17, 1, 9]
    cu = np.cumsum([0] + lens)
    T, Hq, Hkv, d = cu[-1], 4, 2, 8
    q, k, v = rnd((T, Hq, d), 19), rnd((T, Hkv, d), 20), rnd((T, Hkv, d), 21)
    o, lse = A.forward(q, k, v, 0.4, causal, cu_seqlens=cu)
    for s, L in enumerate(lens):
        if L == 0:
            continue
        a, b = cu[s], cu[s + 1]
        os_, ls = A.forward(q[None, a:b], k[None, a:b], v[None, a:b], 0.4, causal)
        assert np.abs(o[a:b] - os_[0]).max() < 1e-14
        assert np.abs(lse[:, a:b] - ls[0]).max() < 1e-14


def test_forward_rows_matches_full():
    B, N, Hq, Hkv, d = 2, 40, 4, 1, 8
    q, k, v = rnd((B, N, Hq, d), 22), rnd((B, N, Hkv, d), 23), rnd((B, N, Hkv, d), 24)
    o, lse = A.forward(q, k, v, 0.3, True)
    picks = [(0, 0, 0), (1, 3, 39), (0, 2, 17)]
    ro, rl = A.forward_rows(q, k, v, 0.3, True, picks)
    for n, (b, h, i) in enumerate(picks):
        assert np.abs(ro[n] - o[b, i, h]).max() < 1e-13
        assert abs(rl[n] - lse[b, h, i]) < 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_dq_rows_match_full_backward(causal):
    """Sampled dQ rows equal the full backward's rows (fixed length, grouped
    heads), and the packed layout's rows equal each sequence's own."""
    B, N, Hq, Hkv, d = 2, 40, 4, 2, 8
    q, k, v, do = (rnd((B, N, h, d), 30 + n) for n, h in enumerate((Hq, Hkv, Hkv, Hq)))
    dq, _, _ = A.backward(q, k, v, do, 0.3, causal)
    picks = [(0, 0, 0), (1, 3, 39), (0, 2, 17), (1, 1, 1)]
    rq = A.dq_rows(q, k, v, do, 0.3, causal, picks)
    for n, (b, h, i) in enumerate(picks):
        assert np.abs(rq[n] - dq[b, i, h]).max() < 1e-12
    lengths = [5, 0, 1, 33]
    cu = np.cumsum([0] + lengths).astype(np.int32)
    T = int(cu[-1])
    qv, kv, vv, dov = (rnd((T, h, d), 40 + n) for n, h in enumerate((Hq, Hkv, Hkv, Hq)))
    dqv, _, _ = A.backward(qv, kv, vv, dov, 0.3, causal, cu_seqlens=cu)
    picks = [(0, 0, 4), (2, 1, 0), (3, 3, 32), (3, 0, 0)]
    rq = A.dq_rows(qv, kv, vv, dov, 0.3, causal, picks, cu_seqlens=cu)
    for n, (b, h, i) in enumerate(picks):
        assert np.abs(rq[n] - dqv[cu[b] + i, h]).max() < 1e-12


# ---------------------------------------------------------------- backward

@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_finite_differences(causal):
    B, N, Hq, Hkv, d, alpha = 1, 6, 2, 1, 4, 0.7
    q, k, v = rnd((B, N, Hq, d), 25), rnd((B, N, Hkv, d), 26), rnd((B, N, Hkv, d), 27)
    do = rnd((B, N, Hq, d), 28)

    def loss(q_, k_, v_):
        o, _ = A.forward(q_, k_, v_, alpha, causal)
        return float((o * do).sum())

    dq, dk, dv = A.backward(q, k, v, do, alpha, causal)
    h = 1e-6
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = [xp if t is x else t for t in (q, k, v)]
            args_m = [xm if t is x else t for t in (q, k, v)]
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        assert np.abs(num - g).max() < 1e-7 * max(1.0, np.abs(g).max())


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_backward_matches_finite_differences(causal):
    """The packed-sequence branch of the backward against central differences
    of L = sum(O * dO) taken through the packed forward, with empty and
    one-token sequences in the batch and grouped heads: every element of
    dQ, dK, dV, including that no gradient leaks across sequences."""
    lens = [3, 0, 1, 5, 0]
    cu = np.cumsum([0] + lens)
    T, Hq, Hkv, d, alpha = int(cu[-1]), 4, 2, 3, 0.6
    q, k, v = rnd((T, Hq, d), 40), rnd((T, Hkv, d), 41), rnd((T, Hkv, d), 42)
    do = rnd((T, Hq, d), 43)

    def loss(q_, k_, v_):
        o, _ = A.forward(q_, k_, v_, alpha, causal, cu_seqlens=cu)
        return float((o * do).sum())

    dq, dk, dv = A.backward(q, k, v, do, alpha, causal, cu_seqlens=cu)
    h = 1e-6
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = [xp if t is x else t for t in (q, k, v)]
            args_m = [xm if t is x else t for t in (q, k, v)]
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        assert np.abs(num - g).max() < 1e-7 * max(1.0, np.abs(g).max())


def test_varlen_backward_one_token_sequence_closed_form():
    """A one-token sequence attends to itself alone: P = 1, so dS = 0 and
    dQ = dK = 0, while dV is dO summed over the key/value head's group."""
    lens = [4, 1, 0, 1, 3]
    cu = np.cumsum([0] + lens)
    T, Hq, Hkv, d = int(cu[-1]), 6, 2, 5
    q, k, v, do = rnd((T, Hq, d), 44), rnd((T, Hkv, d), 45), rnd((T, Hkv, d), 46), rnd((T, Hq, d), 47)
    for causal in (False, True):
        dq, dk, dv = A.backward(q, k, v, do, 0.5, causal, cu_seqlens=cu)
        for s in (1, 3):
            r = int(cu[s])
            assert np.abs(dq[r]).max() < 1e-15 and np.abs(dk[r]).max() < 1e-15
            expect = do[r].reshape(Hkv, Hq // Hkv, d).sum(axis=1)
            assert np.abs(dv[r] - expect).max() < 1e-14


def test_parallel_driver_matches_serial():
    """The process-pool driver evaluates the same per-head problems: outputs
    agree with the serial loop to the last bits BLAS may change."""
    lens = [70, 0, 1, 130]
    cu = np.cumsum([0] + lens)
    T, Hq, Hkv, d = int(cu[-1]), 4, 2, 16
    q, k, v, do = rnd((T, Hq, d), 48), rnd((T, Hkv, d), 49), rnd((T, Hkv, d), 50), rnd((T, Hq, d), 51)
    o1, l1 = A.forward(q, k, v, 0.3, True, cu_seqlens=cu)
    o2, l2 = A.forward(q, k, v, 0.3, True, cu_seqlens=cu, workers=2)
    assert np.abs(o1 - o2).max() < 1e-12 and np.abs(l1 - l2).max() < 1e-12
    g1 = A.backward(q, k, v, do, 0.3, True, cu_seqlens=cu)
    g2 = A.backward(q, k, v, do, 0.3, True, cu_seqlens=cu, workers=2)
    for a, b in zip(g1, g2):
        assert np.abs(a - b).max() < 1e-12


def test_delta_identity():
    N, d, alpha = 31, 8, 0.35
    q, k, v, do = rnd((N, d), 29), rnd((N, d), 30), rnd((N, d), 31), rnd((N, d), 32)
    o, _ = A.head_forward(q, k, v, alpha, True)
    p, _ = A._softmax_rows(A._scores(q, k, alpha, True, 0))
    dp = do @ v.T
    assert np.abs((do * o).sum(1) - (p * dp).sum(1)).max() < 1e-12
    assert np.abs(A.delta(o, do) - (do * o).sum(1)).max() < 1e-15


def test_backward_gqa_sums_group():
    B, N, Hq, Hkv, d = 1, 11, 4, 2, 8
    q, k, v, do = rnd((B, N, Hq, d), 33), rnd((B, N, Hkv, d), 34), rnd((B, N, Hkv, d), 35), rnd((B, N, Hq, d), 36)
    dq, dk, dv = A.backward(q, k, v, do, 0.3, True)
    dq2, dk2, dv2 = A.backward(q, np.repeat(k, 2, 2), np.repeat(v, 2, 2), do, 0.3, True)
    assert np.abs(dq - dq2).max() < 1e-13
    assert np.abs(dk - (dk2[:, :, 0::2] + dk2[:, :, 1::2])).max() < 1e-13
    assert np.abs(dv - (dv2[:, :, 0::2] + dv2[:, :, 1::2])).max() < 1e-13


# ------------------------------------------- online softmax with rescale tau

@pytest.mark.parametrize("N,causal,std", [(300, False, 1.0), (300, True, 3.0), (517, True, 1.0), (129, False, 5.0)])
def test_conditional_rescale_identity(N, causal, std):
    d = 128
    alpha = 1 / math.sqrt(d)
    q, k, v = rnd((N, d), 37, std), rnd((N, d), 38), rnd((N, d), 39)
    o_ref, lse_ref = A.head_forward(q, k, v, alpha, causal)
    for tau in (0.0, GOLDEN["rescale"]["tau"], 1e9):
        o, lse, _ = OS.blockwise_forward(q, k, v, alpha, causal, tau=tau)
        assert np.abs(o - o_ref).max() < 1e-12
        assert np.abs(lse - lse_ref).max() < 1e-12


def test_rescale_branches_both_taken_and_bounded():
    N, d = 1024, 128
    alpha = 1 / math.sqrt(d)
    q, k, v = rnd((N, d), 40, 3.0), rnd((N, d), 41), rnd((N, d), 42)
    _, _, n8 = OS.blockwise_forward(q, k, v, alpha, True, tau=8.0)
    _, _, n0 = OS.blockwise_forward(q, k, v, alpha, True, tau=0.0)
    assert 0 < n8 < n0  # tau = 8 skips some rescales but not all
    worst = OS.max_unnormalised_term(q, k, alpha, True, tau=8.0)
    assert 1.0 <= worst <= GOLDEN["rescale"]["tau_as_ratio"]
    assert OS.TAU == math.log2(GOLDEN["rescale"]["tau_as_ratio"])


# ------------------------------------------------ the pages' cost model

def test_feeds_and_speeds_arithmetic():
    f = GOLDEN["feeds_per_sm_b200"]
    c = GOLDEN["cycles_per_tile_m_n_d_128"]
    M = N = d = 128
    tile = M * d * 2  # one bf16 128x128 operand tile, bytes
    assert 4 * M * N * d / f["mma_bf16_ops_per_clock"] == c["fwd"]["mma"]
    assert M * N / f["mufu_exp_ops_per_clock"] == c["fwd"]["exp"]
    assert 3 * tile / f["smem_bytes_per_clock"] == c["fwd"]["smem"]
    assert 10 * M * N * d / f["mma_bf16_ops_per_clock"] == c["bwd_1cta"]["mma"]
    assert 13 * tile / f["smem_bytes_per_clock"] == c["bwd_1cta"]["smem"]
    assert 10.5 * tile / f["smem_bytes_per_clock"] == c["bwd_2cta"]["smem"]
