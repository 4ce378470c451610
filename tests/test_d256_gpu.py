"""Head dim d = 256: forward and backward parity against the fp64 oracle.

The d = 256 forward (one 128-row query tile per CTA, 64-key blocks, O in
256 tensor-memory columns, the query tile in 128 more) and backward (each
128-key unit once per head-dim half of the gradients, 64-row query steps)
take fixed-length and packed variable-length inputs.
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


# ------------------------------------------------------------------ backward
#
# The d = 256 backward (fa_bwd256.cu): each 128-key unit runs once per
# head-dim half of dK / dV / dQ, queries in 64-row steps.  Tolerance as for
# d = 128: max |err| <= 2e-2 * max |grad| for each of dQ, dK, dV.

REL = 2e-2


def bwd_inputs(B, N, Hq, Hkv, seed=0, lengths=None, q_std=1.0):
    inp = inputs(B, N, Hq, Hkv, seed=seed, q_std=q_std, lengths=lengths)
    inp["do"] = W.normal_bf16(inp["q"].shape, seed + 3)
    if lengths is None:
        inp["lengths"] = [N] * B
    return inp


def gpu_grads(fa, inp, causal, deterministic=False, repeats=1):
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    cu = inp["cu_seqlens"].cuda() if inp.get("cu_seqlens") is not None else None
    ms = max(inp["lengths"]) if cu is not None else None
    o, lse = fa.fwd(q, k, v, causal=causal, cu_seqlens=cu, max_seqlen=ms)
    B = len(inp["lengths"])
    N = q.shape[0] if cu is not None else q.shape[1]
    ws = fa.bwd_workspace(B, q.shape[-2], N, deterministic, cu is not None, d=D)
    outs = []
    for _ in range(repeats):
        g = fa.bwd(q, k, v, o, lse, do, causal=causal, cu_seqlens=cu, max_seqlen=ms, deterministic=deterministic,
                   workspace=ws)
        assert fa.device_status(ws) == 0
        outs.append(tuple(t.float().cpu().numpy() for t in g))
    return outs


def check_bwd(got, ref):
    """max |err| <= 2e-2 * max |grad|.  Where a gradient is exactly zero in
    exact arithmetic (N = 1: P = 1, so dS = dP - D = 0 and dQ = dK = 0) the
    relative bound has no scale; there it is read with the scale floored at
    1e-3 (2e-5 absolute, rounding noise of the fp32 dP and D against O(1)
    inputs)."""
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        assert np.isfinite(g).all(), name
        err, scale = np.abs(g - r).max(), np.abs(r).max()
        assert err <= REL * max(scale, 1e-3), (name, err, scale)


def oracle_bwd(inp, causal):
    return A.backward(inp["q"], inp["k"], inp["v"], inp["do"], ALPHA, causal, cu_seqlens=inp.get("cu_seqlens"))


@pytest.mark.parametrize("N", [1, 63, 64, 65, 128, 200, 513])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_ragged(fa, N, causal):
    inp = bwd_inputs(2, N, 2, 2, seed=N + 100)
    check_bwd(gpu_grads(fa, inp, causal)[0], oracle_bwd(inp, causal))


@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (8, 1)])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_grouped_heads(fa, Hq, Hkv, causal):
    inp = bwd_inputs(1, 300, Hq, Hkv, seed=5)
    check_bwd(gpu_grads(fa, inp, causal)[0], oracle_bwd(inp, causal))


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_varlen(fa, causal):
    inp = bwd_inputs(0, 0, 4, 2, seed=9, lengths=[130, 1, 0, 300, 64, 257, 63])
    check_bwd(gpu_grads(fa, inp, causal)[0], oracle_bwd(inp, causal))


def test_bwd_large_q_logits(fa):
    inp = bwd_inputs(1, 384, 2, 2, seed=17, q_std=3.0)
    check_bwd(gpu_grads(fa, inp, True)[0], oracle_bwd(inp, True))


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_deterministic_bit_identical(fa, causal):
    inp = bwd_inputs(2, 640, 4, 2, seed=13)
    runs = gpu_grads(fa, inp, causal, deterministic=True, repeats=10)
    for r in runs[1:]:
        for a_, b_ in zip(runs[0], r):
            assert np.array_equal(a_.view(np.uint32), b_.view(np.uint32))
    check_bwd(runs[0], oracle_bwd(inp, causal))


def test_bwd_deterministic_many_waves(fa):
    """More units (2 x 40 key tiles x heads) than two waves of CTAs: the
    fixed-order semaphores must never wait on a unit that has not started."""
    import attention_blackwell_gb300 as fa_mod
    N = 128 * 40
    H = max(4, (2 * fa_mod.num_sms()) // 80 + 1)
    inp = bwd_inputs(1, N, H, H, seed=31)
    runs = gpu_grads(fa, inp, False, deterministic=True, repeats=2)
    for a_, b_ in zip(runs[0], runs[1]):
        assert np.array_equal(a_.view(np.uint32), b_.view(np.uint32))
    ref = A.head_backward(*(inp[n][0, :, 0].float().numpy().astype(np.float64) for n in ("q", "k", "v", "do")),
                          ALPHA, False)
    check_bwd([g[0, :, 0] for g in runs[0]], ref)


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_varlen_deterministic_many_units(fa, causal):
    lengths = [2500, 2000, 1500, 1000, 700, 300, 129, 0, 1]
    inp = bwd_inputs(0, 0, 8, 8, seed=41, lengths=lengths)
    runs = gpu_grads(fa, inp, causal, deterministic=True, repeats=3)
    for r in runs[1:]:
        for a_, b_ in zip(runs[0], r):
            assert np.array_equal(a_.view(np.uint32), b_.view(np.uint32))
    check_bwd(runs[0], oracle_bwd(inp, causal))


@pytest.mark.parametrize("name", ["large_d256", "varlen_d256"])
def test_bwd_full_size_every_element(fa, name):
    """The benchmarked d = 256 shapes: every element of dQ, dK, dV against the
    float64 oracle over the whole workload."""
    import full_size as FS
    w, inp = FS.inputs(name)
    got = gpu_grads(fa, inp, w.causal)[0]
    ref = FS.backward_reference(name)
    for name_, g, r in zip(("dq", "dk", "dv"), got, ref):
        assert np.isfinite(g).all(), name_
        err, _ = FS.abs_err_stats(g, r)
        assert err <= REL * FS.max_abs(r), (name_, err)


def test_unsupported_forms_are_rejected_on_the_host(fa):
    import attention_blackwell_gb300 as fa_mod
    assert fa_mod.lib().fa_bwd_workspace_size(1, 2, 300, 96, 0, 0) == 0   # d = 96 is not built
