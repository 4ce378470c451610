"""Head dim d = 64: forward and backward parity against the fp64 oracle.

The d = 64 calls run on the ping-pong forward kernel and the one-CTA
backward kernel (both templated on the head dim); the tolerances are the
d = 128 ones: forward O max |err| <= 2e-2, mean |err| <= 1e-3, LSE abs err
<= 1e-3; backward max |err| <= 2e-2 * max |grad| per gradient; deterministic
mode bit-identical across runs.  alpha = 1/sqrt(64).
"""
import math

import numpy as np
import pytest
import torch

from attention_blackwell_gb300 import workloads as W
from oracle import attention as A

pytestmark = pytest.mark.gpu

D = 64
ALPHA = 1 / math.sqrt(D)
O_MAX, O_MEAN, LSE_ABS, REL = 2e-2, 1e-3, 1e-3, 2e-2


@pytest.fixture(scope="module")
def fa():
    import attention_blackwell_gb300 as fa
    fa.lib()
    fa.set_tuning(0, 8.0)
    yield fa
    fa.set_tuning(0, 8.0)


def inputs(B, N, Hq, Hkv, seed=0, lengths=None, q_std=1.0):
    if lengths is not None:
        cu = W.cu_seqlens_of(lengths)
        T = int(cu[-1])
        sq, sk = (T, Hq, D), (T, Hkv, D)
    else:
        cu, lengths = None, [N] * B
        sq, sk = (B, N, Hq, D), (B, N, Hkv, D)
    return {"q": W.normal_bf16(sq, seed, q_std), "k": W.normal_bf16(sk, seed + 1), "v": W.normal_bf16(sk, seed + 2),
            "do": W.normal_bf16(sq, seed + 3), "cu_seqlens": cu, "lengths": lengths}


def gpu_fwd(fa, inp, causal):
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    cu = inp["cu_seqlens"].cuda() if inp["cu_seqlens"] is not None else None
    ms = max(inp["lengths"]) if cu is not None else None
    o, lse = fa.fwd(q, k, v, causal=causal, cu_seqlens=cu, max_seqlen=ms)
    assert fa.device_status() == 0
    return q, k, v, cu, ms, o, lse


def check_fwd(o, lse, inp, causal):
    o_ref, lse_ref = A.forward(inp["q"], inp["k"], inp["v"], ALPHA, causal, cu_seqlens=inp["cu_seqlens"])
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    err = np.abs(o - o_ref)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    assert err.max() <= O_MAX, err.max()
    assert err.mean() <= O_MEAN, err.mean()
    assert np.abs(lse - lse_ref).max() <= LSE_ABS


def gpu_grads(fa, inp, causal, deterministic=False, repeats=1):
    q, k, v, cu, ms, o, lse = gpu_fwd(fa, inp, causal)
    do = inp["do"].cuda()
    B, Hq = len(inp["lengths"]), q.shape[-2]
    N = q.shape[0] if cu is not None else q.shape[1]
    ws = fa.bwd_workspace(B, Hq, N, deterministic, cu is not None, d=D)
    outs = []
    for _ in range(repeats):
        dq, dk, dv = fa.bwd(q, k, v, o, lse, do, causal=causal, cu_seqlens=cu, max_seqlen=ms,
                            deterministic=deterministic, workspace=ws)
        assert fa.device_status(ws) == 0
        outs.append(tuple(t.float().cpu().numpy() for t in (dq, dk, dv)))
    return outs


def check_bwd(got, ref):
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        assert np.isfinite(g).all(), name
        assert np.abs(g - r).max() <= REL * np.abs(r).max(), name


# ---------------------------------------------------------------- forward

@pytest.mark.parametrize("N", [1, 100, 128, 257, 640, 1000])
@pytest.mark.parametrize("causal", [False, True])
def test_fwd_ragged(fa, N, causal):
    inp = inputs(2, N, 2, 2, seed=N)
    o, lse = gpu_fwd(fa, inp, causal)[5:]
    check_fwd(o, lse, inp, causal)


@pytest.mark.parametrize("causal", [False, True])
def test_fwd_grouped_and_varlen(fa, causal):
    inp = inputs(1, 300, 8, 2, seed=3)
    check_fwd(*gpu_fwd(fa, inp, causal)[5:], inp, causal)
    inp = inputs(0, 0, 4, 2, seed=9, lengths=[130, 1, 0, 300, 64, 257])
    check_fwd(*gpu_fwd(fa, inp, causal)[5:], inp, causal)


@pytest.mark.parametrize("emu", [1, 2, 3, 4])
def test_fwd_exp2_split(fa, emu):
    fa.set_tuning(emu, 8.0)
    try:
        inp = inputs(1, 640, 2, 2, seed=21, q_std=3.0)
        check_fwd(*gpu_fwd(fa, inp, True)[5:], inp, True)
    finally:
        fa.set_tuning(0, 8.0)


def test_fwd_large_q_logits_sampled_rows(fa):
    """B=2, Hq=8, N=4096, causal, Q ~ N(0, 9): rows checked one by one."""
    inp = inputs(2, 4096, 8, 8, seed=33, q_std=3.0)
    o, lse = gpu_fwd(fa, inp, True)[5:]
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    rng = np.random.default_rng(5)
    picks = [(int(rng.integers(2)), int(rng.integers(8)), int(rng.integers(4096))) for _ in range(48)]
    picks += [(0, 0, 0), (1, 7, 4095), (0, 3, 4095)]   # (sequence, query head, row)
    ro, rl = A.forward_rows(inp["q"], inp["k"], inp["v"], ALPHA, True, picks)
    for n, (b, h, i) in enumerate(picks):
        assert np.abs(o[b, i, h] - ro[n]).max() <= O_MAX
        assert abs(lse[b, h, i] - rl[n]) <= LSE_ABS


# ---------------------------------------------------------------- backward

@pytest.mark.parametrize("N", [128, 200, 513])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_small(fa, N, causal):
    inp = inputs(2, N, 2, 2, seed=N + 1)
    check_bwd(gpu_grads(fa, inp, causal)[0],
              A.backward(inp["q"], inp["k"], inp["v"], inp["do"], ALPHA, causal))


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_grouped_and_varlen(fa, causal):
    inp = inputs(1, 300, 8, 1, seed=5)
    check_bwd(gpu_grads(fa, inp, causal)[0],
              A.backward(inp["q"], inp["k"], inp["v"], inp["do"], ALPHA, causal))
    inp = inputs(0, 0, 4, 2, seed=9, lengths=[130, 1, 0, 300, 64, 257])
    check_bwd(gpu_grads(fa, inp, causal)[0],
              A.backward(inp["q"], inp["k"], inp["v"], inp["do"], ALPHA, causal, cu_seqlens=inp["cu_seqlens"]))


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_deterministic(fa, causal):
    inp = inputs(2, 640, 4, 2, seed=13)
    runs = gpu_grads(fa, inp, causal, deterministic=True, repeats=5)
    for r in runs[1:]:
        for a_, b_ in zip(runs[0], r):
            assert np.array_equal(a_.view(np.uint32), b_.view(np.uint32))
    check_bwd(runs[0], A.backward(inp["q"], inp["k"], inp["v"], inp["do"], ALPHA, causal))


def test_bwd_many_tiles_one_head(fa):
    """N = 2048 causal, more units than one wave of CTAs: head (0, 0) checked whole."""
    inp = inputs(2, 2048, 16, 16, seed=41)
    dq, dk, dv = gpu_grads(fa, inp, True)[0]
    ref = A.head_backward(*(inp[n][0, :, 0].float().numpy().astype(np.float64) for n in ("q", "k", "v", "do")),
                          ALPHA, True)
    check_bwd([g[0, :, 0] for g in (dq, dk, dv)], ref)



@pytest.mark.parametrize("causal", [False, True])
def test_bwd_varlen_head_group_units(fa, causal):
    """16 query heads on one key/value head, packed: atomic-mode units of 8
    query heads with fp32 partial dK and dV, as at d = 128."""
    inp = inputs(0, 0, 16, 1, seed=63, lengths=[700, 0, 1, 300, 129, 257])
    check_bwd(gpu_grads(fa, inp, causal)[0],
              A.backward(inp["q"], inp["k"], inp["v"], inp["do"], ALPHA, causal, cu_seqlens=inp["cu_seqlens"]))


def test_varlen_many_short_sequences_d64(fa):
    rng = np.random.default_rng(78)
    lengths = [int(x) for x in rng.integers(0, 301, size=1000)]
    inp = inputs(0, 0, 4, 2, seed=52, lengths=lengths)
    check_fwd(*gpu_fwd(fa, inp, True)[5:], inp, True)
    check_bwd(gpu_grads(fa, inp, True)[0],
              A.backward(inp["q"], inp["k"], inp["v"], inp["do"], ALPHA, True, cu_seqlens=inp["cu_seqlens"]))
