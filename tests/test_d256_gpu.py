"""Head dim d = 256: forward parity against the fp64 oracle.

The d = 256 forward (one 128-row query tile per CTA, 64-key blocks, O in
256 tensor-memory columns, the query tile in 128 more) takes
fixed-length and packed variable-length inputs; the backward is not built for
d = 256 (dK and dV alone would fill the 512 tensor-memory columns).
Tolerances as for d = 128: O max |err| <= 2e-2, mean |err| <= 1e-3, LSE abs
err <= 1e-3.  alpha = 1/sqrt(256).
"""
import math

import numpy as np
import pytest
import torch

from attention_blackwell_gb300 import workloads as W
from oracle import attention as A

pytestmark = pytest.mark.gpu

D = 256
ALPHA = 1 / math.sqrt(D)
O_MAX, O_MEAN, LSE_ABS = 2e-2, 1e-3, 1e-3


@pytest.fixture(scope="module")
def fa():
    import attention_blackwell_gb300 as fa
    fa.lib()
    fa.set_tuning(0, 8.0)
    return fa


def inputs(B, N, Hq, Hkv, seed=0, q_std=1.0, lengths=None):
    if lengths is not None:   # packed varlen: N is ignored, T = sum(lengths)
        cu = W.cu_seqlens_of(lengths)
        T = int(cu[-1])
        sq, sk = (T, Hq, D), (T, Hkv, D)
    else:
        cu = None
        sq, sk = (B, N, Hq, D), (B, N, Hkv, D)
    return {"q": W.normal_bf16(sq, seed, q_std), "k": W.normal_bf16(sk, seed + 1), "v": W.normal_bf16(sk, seed + 2),
            "cu_seqlens": cu, "lengths": lengths}


def run(fa, inp, causal):
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    if inp.get("cu_seqlens") is not None:
        o, lse = fa.fwd(q, k, v, causal=causal, cu_seqlens=inp["cu_seqlens"].cuda(), max_seqlen=max(inp["lengths"]))
    else:
        o, lse = fa.fwd(q, k, v, causal=causal)
    assert fa.device_status() == 0
    return o.float().cpu().numpy(), lse.cpu().numpy()


def check(o, lse, inp, causal):
    o_ref, lse_ref = A.forward(inp["q"], inp["k"], inp["v"], ALPHA, causal, cu_seqlens=inp.get("cu_seqlens"))
    err = np.abs(o - o_ref)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    assert err.max() <= O_MAX, err.max()
    assert err.mean() <= O_MEAN, err.mean()
    assert np.abs(lse - lse_ref).max() <= LSE_ABS


@pytest.mark.parametrize("N", [1, 63, 64, 100, 128, 257, 640, 1000])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged(fa, N, causal):
    inp = inputs(2, N, 2, 2, seed=N + 7)
    check(*run(fa, inp, causal), inp, causal)


@pytest.mark.parametrize("causal", [False, True])
def test_grouped_heads(fa, causal):
    inp = inputs(1, 300, 8, 2, seed=3)
    check(*run(fa, inp, causal), inp, causal)


def test_large_q_logits(fa):
    """Q ~ N(0, 9): large row-max jumps exercise the rescale of the 256-wide O row."""
    inp = inputs(1, 1024, 2, 2, seed=11, q_std=3.0)
    check(*run(fa, inp, True), inp, True)


@pytest.mark.parametrize("tau", [0.0, 64.0])
def test_rescale_threshold_extremes(fa, tau):
    """tau = 0 rescales O whenever a row maximum grows (the wait for the
    previous block's P V on almost every block); tau = 64 keeps the first
    maximum unless it is beaten by 2^64.  Both give the same attention."""
    fa.set_tuning(0, tau)
    try:
        inp = inputs(1, 1000, 4, 2, seed=17, q_std=3.0)
        check(*run(fa, inp, True), inp, True)
        inp = inputs(0, 0, 2, 1, seed=18, q_std=3.0, lengths=[700, 5, 257])
        check(*run(fa, inp, False), inp, False)
    finally:
        fa.set_tuning(0, 8.0)


def test_many_units_sampled_rows(fa):
    """B=2, Hq=8, N=4096, causal: more units than CTAs, rows checked one by one."""
    inp = inputs(2, 4096, 8, 8, seed=33)
    o, lse = run(fa, inp, True)
    rng = np.random.default_rng(9)
    picks = [(int(rng.integers(2)), int(rng.integers(8)), int(rng.integers(4096))) for _ in range(40)]
    picks += [(0, 0, 0), (1, 7, 4095), (0, 5, 127), (1, 2, 128)]   # (sequence, query head, row)
    ro, rl = A.forward_rows(inp["q"], inp["k"], inp["v"], ALPHA, True, picks)
    for n, (b, h, i) in enumerate(picks):
        assert np.abs(o[b, i, h] - ro[n]).max() <= O_MAX
        assert abs(lse[b, h, i] - rl[n]) <= LSE_ABS


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_ragged_and_empty_sequences(fa, causal):
    """Lengths straddling the 64-key block and 128-row tile edges, empty and
    one-token sequences, grouped heads."""
    inp = inputs(0, 0, 4, 2, seed=61, lengths=[130, 1, 0, 300, 64, 257, 1000, 128, 63])
    check(*run(fa, inp, causal), inp, causal)


def test_varlen_many_short_sequences(fa):
    """1000 sequences of 0-300 tokens: many levels of units per CTA."""
    rng = np.random.default_rng(81)
    inp = inputs(0, 0, 2, 1, seed=62, lengths=[int(x) for x in rng.integers(0, 301, size=1000)])
    check(*run(fa, inp, True), inp, True)


def test_varlen_mqa_full_size_sampled_rows(fa):
    """16 sequences of 512-8192 tokens, Hq = 8, one key/value head, causal:
    more units than CTAs at every level; rows checked one by one."""
    rng = np.random.default_rng(4)
    lengths = [int(x) for x in rng.integers(512, 8193, size=16)]
    inp = inputs(0, 0, 8, 1, seed=71, lengths=lengths)
    o, lse = run(fa, inp, True)
    cu = [int(c) for c in inp["cu_seqlens"]]
    picks = [(int(b), int(rng.integers(8)), int(rng.integers(lengths[b]))) for b in rng.integers(16, size=40)]
    picks += [(0, 0, 0), (15, 7, lengths[15] - 1), (3, 2, 127), (9, 5, 128)]   # (sequence, query head, row)
    ro, rl = A.forward_rows(inp["q"], inp["k"], inp["v"], ALPHA, True, picks, cu_seqlens=inp["cu_seqlens"])
    for n, (b, h, i) in enumerate(picks):
        assert np.abs(o[cu[b] + i, h] - ro[n]).max() <= O_MAX
        assert abs(lse[h, cu[b] + i] - rl[n]) <= LSE_ABS


def test_unsupported_forms_are_rejected_on_the_host(fa):
    with pytest.raises(ValueError):
        fa.bwd_workspace(1, 2, 300, d=D)                        # no d = 256 backward
