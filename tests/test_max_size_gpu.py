"""The largest supported sequence length, forward and backward, on every
kernel family.

131072 tokens is the longest sequence a packed varlen call accepts
(max_seqlen, include/fa.h); the fixed-length path has no such bound and is
run at the same length.  The whole oracle is out of reach there (S alone is
2^34 entries per head), so the checks are ones that hold at any size:
* O, LSE and dQ of sampled query rows against the oracle's row functions:
  each depends only on its own query row and the keys it sees, so sampled
  rows are exact (oracle.attention.forward_rows and dq_rows, pinned against
  the full oracle in tests/test_oracle.py).  The rows straddle tile and
  block boundaries and include the first and last rows of every sequence;
* two identities of the backward, for every key/value head and sequence:
  sum_j dV_j = sum over the group's query heads of sum_i dO_i (each row of P
  sums to 1), and sum_j dK_j = 0 (each row of dS sums to 0, as
  sum_j P_ij (dP_ij - D_i) = D_i - D_i).  Dropping, duplicating or
  mis-scaling a tile of dK or dV breaks them by more than the tolerance,
  which is 1 % of the root-sum-square of the rows being summed (bf16
  rounding of the rows contributes about 0.2 %).
"""
import math

import numpy as np
import pytest
import torch

from attention_blackwell_gb300 import workloads as W
from oracle import attention as A

pytestmark = pytest.mark.gpu

NMAX = 131072
O_ABS, LSE_ABS, REL = 2e-2, 1e-3, 2e-2


@pytest.fixture(scope="module")
def fa():
    import attention_blackwell_gb300 as fa
    fa.lib()
    fa.set_tuning(0, 8.0)
    yield fa
    fa.set_fwd_kernel(2)
    fa.set_bwd_kernel(0)


def make(d, Hq, Hkv, lengths=None, N=None):
    if lengths is not None:
        cu = W.cu_seqlens_of(lengths)
        T = int(cu[-1])
        sq, sk = (T, Hq, d), (T, Hkv, d)
    else:
        cu = None
        sq, sk = (1, N, Hq, d), (1, N, Hkv, d)
    host = {"q": W.normal_bf16(sq, 70), "k": W.normal_bf16(sk, 71), "v": W.normal_bf16(sk, 72),
            "do": W.normal_bf16(sq, 73)}
    return host, cu


def sample_rows(L, rng, n=8):
    """First and last rows, rows around the 128- and 256-row boundaries,
    and a few at random."""
    if L == 0:
        return []
    base = {0, 1, 127, 128, 255, 256, L // 2, L - 129, L - 128, L - 2, L - 1}
    rows = sorted(r for r in base if 0 <= r < L)
    return rows + sorted(int(x) for x in rng.integers(0, L, size=n))


def run(fa, host, cu, causal, d):
    g = {n: t.cuda() for n, t in host.items()}
    cu_d = cu.cuda() if cu is not None else None
    lengths = None if cu is None else [int(cu[i + 1] - cu[i]) for i in range(len(cu) - 1)]
    ms = max(lengths) if lengths else None
    alpha = 1 / math.sqrt(d)
    o, lse = fa.fwd(g["q"], g["k"], g["v"], causal=causal, alpha=alpha, cu_seqlens=cu_d, max_seqlen=ms)
    assert fa.device_status() == 0
    B = len(lengths) if lengths else 1
    N = g["q"].shape[0] if cu is not None else g["q"].shape[1]
    ws = fa.bwd_workspace(B, g["q"].shape[-2], N, False, cu is not None, d=d)
    dq, dk, dv = fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal=causal, alpha=alpha, cu_seqlens=cu_d,
                        max_seqlen=ms, workspace=ws)
    assert fa.device_status(ws) == 0
    return [t.float().cpu().numpy() for t in (o, lse, dq, dk, dv)], alpha, lengths


def check(host, cu, causal, outs, alpha, lengths):
    o, lse, dq, dk, dv = outs
    q, k, v, do = (host[n] for n in ("q", "k", "v", "do"))
    Hq, Hkv = q.shape[-2], k.shape[-2]
    rng = np.random.default_rng(5)
    seqs = range(len(lengths)) if lengths else [0]
    picks = []
    for b in seqs:
        L = lengths[b] if lengths else q.shape[1]
        for i in sample_rows(L, rng):
            picks.append((b, int(rng.integers(0, Hq)), i))
    ro, rl = A.forward_rows(q, k, v, alpha, causal, picks, cu_seqlens=cu)
    rq = A.dq_rows(q, k, v, do, alpha, causal, picks, cu_seqlens=cu)
    dq_scale = max(np.abs(rq).max(), 1e-6)
    for n, (b, h, i) in enumerate(picks):
        if cu is not None:
            row = int(cu[b]) + i
            go, gl, gq = o[row, h], lse[h, row], dq[row, h]
        else:
            go, gl, gq = o[0, i, h], lse[0, h, i], dq[0, i, h]
        assert np.abs(go - ro[n]).max() <= O_ABS, (b, h, i)
        assert abs(gl - rl[n]) <= LSE_ABS, (b, h, i)
        assert np.abs(gq - rq[n]).max() <= REL * dq_scale, (b, h, i)
    # Column sums of dV and dK per sequence and key/value head.
    g = Hq // Hkv
    do64 = do.double().numpy()
    for b in seqs:
        if cu is not None:
            a0, a1 = int(cu[b]), int(cu[b + 1])
            dvs, dks, dos = dv[a0:a1], dk[a0:a1], do64[a0:a1]
        else:
            dvs, dks, dos = dv[0], dk[0], do64[0]
        if dvs.shape[0] == 0:
            continue
        for hk in range(Hkv):
            want = dos[:, hk * g:(hk + 1) * g].sum(axis=(0, 1))
            got_v = dvs[:, hk].astype(np.float64).sum(axis=0)
            tol_v = 1e-2 * math.sqrt((dvs[:, hk].astype(np.float64) ** 2).sum()) + 1e-3
            assert np.abs(got_v - want).max() <= tol_v, (b, hk, np.abs(got_v - want).max(), tol_v)
            got_k = dks[:, hk].astype(np.float64).sum(axis=0)
            tol_k = 1e-2 * math.sqrt((dks[:, hk].astype(np.float64) ** 2).sum()) + 1e-3
            assert np.abs(got_k).max() <= tol_k, (b, hk, np.abs(got_k).max(), tol_k)


@pytest.mark.parametrize("d,fwd_kernel,bwd_kernel", [(128, 2, 0), (128, 0, 1), (64, 0, 0), (256, 2, 0)],
                         ids=["d128", "d128_pingpong_pairbwd", "d64", "d256"])
def test_varlen_longest_sequence(fa, d, fwd_kernel, bwd_kernel):
    """One sequence at the varlen limit packed with an empty, a one-token and
    two ragged ones; causal, grouped heads."""
    host, cu = make(d, 2, 1, lengths=[NMAX, 0, 1, 300, 4097])
    fa.set_fwd_kernel(fwd_kernel)
    fa.set_bwd_kernel(bwd_kernel)
    try:
        outs, alpha, lengths = run(fa, host, cu, True, d)
    finally:
        fa.set_fwd_kernel(2)
        fa.set_bwd_kernel(0)
    check(host, cu, True, outs, alpha, lengths)


@pytest.mark.parametrize("bwd_kernel", [0, 1], ids=["one_cta", "pair"])
def test_fixed_length_at_the_same_length(fa, bwd_kernel):
    """Fixed length, N = 131072, non-causal, one query head per key/value head."""
    host, _ = make(128, 1, 1, N=NMAX)
    fa.set_bwd_kernel(bwd_kernel)
    try:
        outs, alpha, _ = run(fa, host, None, False, 128)
    finally:
        fa.set_bwd_kernel(0)
    check(host, None, False, outs, alpha, None)
