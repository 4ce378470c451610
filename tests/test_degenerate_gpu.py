"""Degenerate inputs whose results have closed forms, at full tile counts.

* Q = 0: every logit is 0, so each row of P is uniform over the keys the row
  sees (c_i of them: all N, or i + 1 under the causal mask).  Then
  O_i = mean of those V rows, LSE_i = ln c_i, dK = alpha dS^T Q = 0 exactly,
  and dV_j = sum over the queries i that see key j of dO_i / c_i (for grouped
  heads, summed over the group's query heads).
* V constant: O_i = that constant for every row, whatever Q and K are.
* dO = 0: D = 0 and dP = 0, so dS = 0 and dQ = dK = dV = 0 exactly.
Checked on every forward kernel and both backward kernels, at d = 64, 128 and
256, with grouped heads and ragged lengths.
"""
import math

import numpy as np
import pytest
import torch

from attention_blackwell_gb300 import workloads as W

pytestmark = pytest.mark.gpu

B, N, HQ, HKV = 2, 1500, 4, 2
O_ABS, LSE_ABS, REL = 2e-2, 1e-3, 2e-2


@pytest.fixture(scope="module")
def fa():
    import attention_blackwell_gb300 as fa
    fa.lib()
    fa.set_tuning(0, 8.0)
    yield fa
    fa.set_fwd_kernel(2)
    fa.set_bwd_kernel(0)


CASES = [(128, 2, 0), (128, 0, 1), (64, 0, 0), (256, 2, 0)]
IDS = ["d128", "d128_pingpong_pairbwd", "d64", "d256"]


def counts(causal):
    """c_i: keys row i sees."""
    return np.arange(1, N + 1, dtype=np.float64) if causal else np.full(N, float(N))


def grads(fa, q, k, v, do, causal, d):
    alpha = 1 / math.sqrt(d)
    o, lse = fa.fwd(q, k, v, causal=causal, alpha=alpha)
    ws = fa.bwd_workspace(B, HQ, N, False, False, d=d)
    out = fa.bwd(q, k, v, o, lse, do, causal=causal, alpha=alpha, workspace=ws)
    assert fa.device_status(ws) == 0
    return o, lse, out


def with_kernels(fa, fk, bk, fn):
    fa.set_fwd_kernel(fk)
    fa.set_bwd_kernel(bk)
    try:
        return fn()
    finally:
        fa.set_fwd_kernel(2)
        fa.set_bwd_kernel(0)


@pytest.mark.parametrize("d,fk,bk", CASES, ids=IDS)
@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries(fa, d, fk, bk, causal):
    q = torch.zeros(B, N, HQ, d, dtype=torch.bfloat16)
    k, v = W.normal_bf16((B, N, HKV, d), 1), W.normal_bf16((B, N, HKV, d), 2)
    do = W.normal_bf16((B, N, HQ, d), 3)
    o, lse, (dq, dk, dv) = with_kernels(fa, fk, bk, lambda: grads(
        fa, q.cuda(), k.cuda(), v.cuda(), do.cuda(), causal, d))
    c = counts(causal)
    v64, do64 = v.double().numpy(), do.double().numpy()
    g = HQ // HKV
    # O: running (causal) or full mean of V per key/value head.
    if causal:
        want_o = np.cumsum(v64, axis=1) / c[None, :, None, None]
    else:
        want_o = np.broadcast_to(v64.mean(axis=1, keepdims=True), v64.shape)
    got_o = o.float().cpu().numpy()
    for h in range(HQ):
        err = np.abs(got_o[:, :, h] - want_o[:, :, h // g])
        assert err.max() <= O_ABS and err.mean() <= 1e-3, (h, err.max(), err.mean())
    assert np.abs(lse.cpu().numpy() - np.log(c)[None, None, :]).max() <= LSE_ABS
    # dK exactly zero.
    assert torch.count_nonzero(dk).item() == 0
    # dV_j = sum over the group's heads and the rows i that see j of dO_i / c_i.
    w = do64 / c[None, :, None, None]
    if causal:
        tail = np.flip(np.cumsum(np.flip(w, axis=1), axis=1), axis=1)   # sum over i >= j
    else:
        tail = np.broadcast_to(w.sum(axis=1, keepdims=True), w.shape)
    want_dv = tail.reshape(B, N, HKV, g, d).sum(axis=3)
    got_dv = dv.float().cpu().numpy()
    assert np.abs(got_dv - want_dv).max() <= REL * np.abs(want_dv).max()
    assert torch.isfinite(dq.float()).all()


@pytest.mark.parametrize("d,fk,bk", CASES, ids=IDS)
@pytest.mark.parametrize("causal", [False, True])
def test_constant_values(fa, d, fk, bk, causal):
    q = W.normal_bf16((B, N, HQ, d), 4, 2.0)
    k = W.normal_bf16((B, N, HKV, d), 5)
    v = torch.full((B, N, HKV, d), 0.75, dtype=torch.bfloat16)
    o, _ = with_kernels(fa, fk, bk, lambda: fa.fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal,
                                                   alpha=1 / math.sqrt(d)))
    assert fa.device_status() == 0
    assert (o.float() - 0.75).abs().max().item() <= 1e-2


@pytest.mark.parametrize("d,fk,bk", CASES, ids=IDS)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("deterministic", [False, True])
def test_zero_upstream_gradient(fa, d, fk, bk, causal, deterministic):
    q = W.normal_bf16((B, N, HQ, d), 6)
    k, v = W.normal_bf16((B, N, HKV, d), 7), W.normal_bf16((B, N, HKV, d), 8)
    do = torch.zeros(B, N, HQ, d, dtype=torch.bfloat16)

    def run():
        alpha = 1 / math.sqrt(d)
        qg, kg, vg, dog = q.cuda(), k.cuda(), v.cuda(), do.cuda()
        o, lse = fa.fwd(qg, kg, vg, causal=causal, alpha=alpha)
        ws = fa.bwd_workspace(B, HQ, N, deterministic, False, d=d)
        out = fa.bwd(qg, kg, vg, o, lse, dog, causal=causal, alpha=alpha, deterministic=deterministic, workspace=ws)
        assert fa.device_status(ws) == 0
        return out
    for name, t in zip(("dq", "dk", "dv"), with_kernels(fa, fk, bk, run)):
        assert torch.count_nonzero(t).item() == 0, name
