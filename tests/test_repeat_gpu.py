"""Repeated runs at full size: races that corrupt a tile only now and then.

The kernels hand tensor-memory columns and shared-memory buffers between
threads with mbarriers; a hand-off that waits on the wrong phase, or relies
on an ordering the hardware does not give, can corrupt a tile in a few
percent of launches, and a single parity run then usually passes.  These
tests repeat each benchmarked workload on the same inputs:

* forward: every kernel is deterministic (each output tile is written by one
  CTA, in a fixed order), so O and LSE must be bitwise identical over 20
  launches;
* backward, atomic mode: dQ accumulates in whatever order the key tiles
  finish, so runs differ by summation order only; every run must agree with
  the deterministic mode's result (checked against the oracle elsewhere) to
  1e-2 of each gradient's scale, where a corrupted tile measured 3-30 %.
"""
import pytest
import torch

import full_size as FS

pytestmark = pytest.mark.gpu

REPS = 20


@pytest.fixture(scope="module")
def fa():
    import attention_blackwell_gb300 as fa
    fa.lib()
    fa.set_tuning(0, 8.0)
    yield fa
    fa.set_fwd_kernel(2)
    fa.set_bwd_kernel(0)


def _dev(inp):
    g = {n: inp[n].cuda() for n in ("q", "k", "v", "do")}
    cu = inp["cu_seqlens"]
    g["cu"] = cu.cuda() if cu is not None else None
    g["ms"] = max(inp["lengths"]) if cu is not None else None
    return g


@pytest.mark.parametrize("name,kernel", [
    ("large", 2), ("causal", 2), ("varlen", 2), ("large", 0), ("causal", 0), ("large_d64", 0),
    ("large_d256", 2), ("causal_d256", 2), ("varlen_d256", 2)])
def test_forward_bitwise_identical(fa, name, kernel):
    """kernel: 2 = CTA pairs, 0 = ping-pong (d = 64 always runs ping-pong and
    d = 256 its own kernel, whatever the selector says)."""
    w, inp = FS.inputs(name)
    g = _dev(inp)
    fa.set_fwd_kernel(kernel)
    try:
        o0, l0 = fa.fwd(g["q"], g["k"], g["v"], causal=w.causal, cu_seqlens=g["cu"], max_seqlen=g["ms"])
        o, l = torch.empty_like(o0), torch.empty_like(l0)
        bad = []
        for rep in range(REPS):
            fa.fwd(g["q"], g["k"], g["v"], causal=w.causal, cu_seqlens=g["cu"], max_seqlen=g["ms"], out=o, lse=l)
            if not (torch.equal(o.view(torch.int16), o0.view(torch.int16)) and
                    torch.equal(l.view(torch.int32), l0.view(torch.int32))):
                bad.append((rep, (o.float() - o0.float()).abs().max().item(), (l - l0).abs().max().item()))
        assert fa.device_status() == 0
    finally:
        fa.set_fwd_kernel(2)
    assert not bad, bad[:3]


@pytest.mark.parametrize("name", ["large", "causal_bwd", "varlen", "large_d64", "large_d256", "causal_d256"])
def test_backward_atomic_runs_match_deterministic(fa, name):
    """The one-CTA kernel at d = 64 / 128 and the d = 256 kernel: every atomic
    run against the deterministic result."""
    w, inp = FS.inputs(name)
    g = _dev(inp)
    varlen = g["cu"] is not None
    B, T = len(inp["lengths"]), inp["T"]
    N = T if varlen else w.N
    o, lse = fa.fwd(g["q"], g["k"], g["v"], causal=w.causal, cu_seqlens=g["cu"], max_seqlen=g["ms"])
    kw = dict(causal=w.causal, cu_seqlens=g["cu"], max_seqlen=g["ms"])
    wsd = fa.bwd_workspace(B, w.Hq, N, True, varlen, d=w.d)
    ref = [t.float() for t in fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], deterministic=True, workspace=wsd, **kw)]
    assert fa.device_status(wsd) == 0
    tol = [1e-2 * r.abs().max().item() for r in ref]
    ws = fa.bwd_workspace(B, w.Hq, N, False, varlen, d=w.d)
    bad = []
    for rep in range(REPS):
        got = fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], workspace=ws, **kw)
        err = [(x.float() - r).abs().max().item() for x, r in zip(got, ref)]
        if any(e > t for e, t in zip(err, tol)):
            bad.append((rep, err))
    assert fa.device_status(ws) == 0
    assert not bad, (tol, bad[:3])
