"""Malformed cu_seqlens: every kernel applies one sanitising rule.

fa.h states the rule: c'_0 = clamp(c_0, 0, T), c'_s = max(c'_{s-1},
clamp(c_s, 0, T)); sequence s is rows [c'_s, c'_{s+1}).  Offsets that are
negative, above T or decreasing must therefore (a) touch nothing outside the
tensors (guard rows around each buffer keep their sentinel), (b) leave rows
outside every sequence unwritten (o, lse, dk, dv) or zero (dq), (c) give,
on the rows they do cover, the oracle's attention for the sanitised offsets,
and (d) report FA_OK.  Checked on every kernel that reads offsets: the
pair and ping-pong forwards (d = 128), the ping-pong forward at d = 64, the
d = 256 forward, and the backward (d = 128 on both main kernels, and 64;
the plan stage and the main kernel share one sanitised copy).
"""
import math

import numpy as np
import pytest
import torch

from attention_blackwell_gb300 import workloads as W
from oracle import attention as A

pytestmark = pytest.mark.gpu

GUARD = 64            # guard rows before and after every buffer
SENT = 1232.0         # sentinel (exact in bf16 and fp32)
O_MAX, O_MEAN, LSE_ABS, REL = 2e-2, 1e-3, 1e-3, 2e-2

# (raw offsets, T): negative, decreasing, above T, rows before the first and
# after the last sequence, empty and one-token sequences.
CASES = [
    ([20, 300, 200, -50, 650, 900, 640, 901, 905], 1000),
    ([0, 5000, 10, 1000], 1000),
    ([-9, 1, 1, 0, 513, 400, 700], 700),
]


def sanitise(raw, T):
    """The documented rule, restated for the test (not the kernels' code)."""
    out, run = [], 0
    for i, c in enumerate(raw):
        c = min(max(int(c), 0), T)
        run = c if i == 0 else max(run, c)
        out.append(run)
    return out


def guarded(shape, dtype):
    """A tensor of `shape` in the middle of a buffer with GUARD rows of
    sentinel on each side; returns (view, whole buffer)."""
    row = int(np.prod(shape[1:]))
    buf = torch.full(((shape[0] + 2 * GUARD) * row,), SENT, dtype=dtype, device="cuda")
    return buf[GUARD * row:(GUARD + shape[0]) * row].view(shape), buf, row


def guards_intact(buf, row, n):
    g = buf.view(n + 2 * GUARD, row)
    return bool((g[:GUARD] == SENT).all()) and bool((g[GUARD + n:] == SENT).all())


def covered_rows(cs, T):
    m = np.zeros(T, dtype=bool)
    for s in range(len(cs) - 1):
        m[cs[s]:cs[s + 1]] = True
    return m


@pytest.fixture(scope="module")
def fa():
    import attention_blackwell_gb300 as fa
    fa.lib()
    fa.set_tuning(0, 8.0)
    yield fa
    fa.set_fwd_kernel(2)


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("kernel,d", [(2, 128), (0, 128), (0, 64), (2, 256)], ids=["pair", "pingpong", "d64", "d256"])
@pytest.mark.parametrize("causal", [False, True])
def test_forward_malformed_offsets(fa, case, kernel, d, causal):
    raw, T = CASES[case]
    cs = sanitise(raw, T)
    Hq, Hkv = 4, 2
    q, k, v = (W.normal_bf16((T, h, d), 70 + i) for i, h in enumerate((Hq, Hkv, Hkv)))
    fa.set_fwd_kernel(kernel)
    o, obuf, orow = guarded((T, Hq, d), torch.bfloat16)
    lse_buf = torch.full(((Hq + 2) * T,), SENT, dtype=torch.float32, device="cuda")
    lse = lse_buf[T:(Hq + 1) * T].view(Hq, T)
    cu = torch.tensor(raw, dtype=torch.int32, device="cuda")
    fa.fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, alpha=1 / math.sqrt(d), cu_seqlens=cu, max_seqlen=T,
           out=o, lse=lse)
    assert fa.device_status() == 0
    assert guards_intact(obuf, orow, T)
    assert bool((lse_buf[:T] == SENT).all()) and bool((lse_buf[(Hq + 1) * T:] == SENT).all())
    cov = covered_rows(cs, T)
    on, ln = o.float().cpu().numpy(), lse.cpu().numpy()
    assert (on[~cov] == SENT).all() and (ln[:, ~cov] == SENT).all()
    o_ref, lse_ref = A.forward(q, k, v, 1 / math.sqrt(d), causal, cu_seqlens=np.array(cs))
    err = np.abs(on[cov] - o_ref[cov])
    assert err.max() <= O_MAX and err.mean() <= O_MEAN, (err.max(), err.mean())
    assert np.abs(ln[:, cov] - lse_ref[:, cov]).max() <= LSE_ABS


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("kernel,d,heads", [(0, 128, (4, 2)), (1, 128, (4, 2)), (0, 64, (4, 2)), (0, 128, (16, 1))],
                         ids=["one_cta", "pair", "d64", "one_cta_head_groups"])
@pytest.mark.parametrize("causal,deterministic", [(False, False), (True, False), (True, True)])
def test_backward_malformed_offsets(fa, case, kernel, d, heads, causal, deterministic):
    """16 query heads on one key/value head: in atomic mode units of 8
    query heads whose fp32 partial dK and dV the last stage converts, for
    the sequences' rows only."""
    fa.set_bwd_kernel(kernel)
    try:
        _backward_malformed_offsets(fa, case, d, causal, deterministic, heads)
    finally:
        fa.set_bwd_kernel(0)


def _backward_malformed_offsets(fa, case, d, causal, deterministic, heads=(4, 2)):
    raw, T = CASES[case]
    cs = sanitise(raw, T)
    Hq, Hkv = heads
    q, k, v = (W.normal_bf16((T, h, d), 80 + i) for i, h in enumerate((Hq, Hkv, Hkv)))
    do = W.normal_bf16((T, Hq, d), 83)
    qg, kg, vg, dog = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    alpha = 1 / math.sqrt(d)
    # The forward on the sanitised offsets gives the O and LSE the backward reads.
    fa.set_fwd_kernel(2)
    o, lse = fa.fwd(qg, kg, vg, causal=causal, alpha=alpha, cu_seqlens=torch.tensor(cs, dtype=torch.int32).cuda(),
                    max_seqlen=T)
    dq, dqbuf, qrow = guarded((T, Hq, d), torch.bfloat16)
    dk, dkbuf, krow = guarded((T, Hkv, d), torch.bfloat16)
    dv, dvbuf, _ = guarded((T, Hkv, d), torch.bfloat16)
    ws = fa.bwd_workspace(len(raw) - 1, Hq, T, deterministic, varlen=True, d=d)
    cu = torch.tensor(raw, dtype=torch.int32, device="cuda")
    fa.bwd(qg, kg, vg, o, lse, dog, causal=causal, alpha=alpha, cu_seqlens=cu, max_seqlen=T,
           deterministic=deterministic, workspace=ws, dq=dq, dk=dk, dv=dv)
    assert fa.device_status(ws) == 0
    for buf, row in ((dqbuf, qrow), (dkbuf, krow), (dvbuf, krow)):
        assert guards_intact(buf, row, T)
    cov = covered_rows(cs, T)
    g = [t.float().cpu().numpy() for t in (dq, dk, dv)]
    assert (g[0][~cov] == 0).all()
    assert (g[1][~cov] == SENT).all() and (g[2][~cov] == SENT).all()
    ref = A.backward(q, k, v, do, alpha, causal, cu_seqlens=np.array(cs))
    for name, gg, r in zip(("dq", "dk", "dv"), g, ref):
        err = np.abs(gg[cov] - r[cov]).max()
        assert err <= REL * np.abs(r).max(), (name, err)
