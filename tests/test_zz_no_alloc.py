"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory.

Called through the C ABI; its gradients must match the regular entry point
(fa_bwd with a caller-allocated workspace) within the backward tolerance,
on two calls in a row (the second call reuses the scratch the first left).
Collected last so that a failure here cannot hide any other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from attention_blackwell_gb300 import workloads as W

pytestmark = pytest.mark.gpu

REL = 2e-2


def _noalloc(L):
    f = L.fa_bwd_noalloc
    vp, i, fl = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.restype = i
    f.argtypes = [vp] * 9 + [i, i, i, i, i, fl, i, vp, i, i, vp]
    return f


def _check_against_workspace_entry_point(fa, f, q, k, v, do, causal, deterministic, cu=None, lengths=None):
    """Two no-allocation calls in a row against fa_bwd with a workspace."""
    d = q.shape[-1]
    alpha = 1 / d ** 0.5
    ms = max(lengths) if cu is not None else None
    o, lse = fa.fwd(q, k, v, causal=causal, cu_seqlens=cu, max_seqlen=ms)
    ref = fa.bwd(q, k, v, o, lse, do, causal=causal, cu_seqlens=cu, max_seqlen=ms, deterministic=deterministic)
    if cu is None:
        B, N, Hq, _ = q.shape
        Hkv = k.shape[2]
    else:
        B, N, Hq, Hkv = cu.numel() - 1, q.shape[0], q.shape[1], k.shape[1]
    s = torch.cuda.current_stream().cuda_stream
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
    for call in range(2):
        dq, dk, dv = torch.full_like(q, float("nan")), torch.full_like(k, float("nan")), torch.full_like(v, float("nan"))
        rc = f(p(q), p(k), p(v), p(o), p(lse), p(do), p(dq), p(dk), p(dv), B, Hq, Hkv, N, d,
               alpha, int(causal), p(cu), ms or 0, int(deterministic), ctypes.c_void_p(s))
        assert rc == 0, (call, rc)
        torch.cuda.synchronize()
        for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
            g, r = g.float().cpu().numpy(), r.float().cpu().numpy()
            assert np.isfinite(g).all(), (call, name)
            assert np.abs(g - r).max() <= REL * np.abs(r).max(), (call, name)
            if deterministic:
                assert np.array_equal(g, r), (call, name)
    assert fa.device_status() == 0


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("causal,deterministic", [(True, False), (False, True)])
def test_noalloc_matches_workspace_entry_point(d, causal, deterministic):
    import attention_blackwell_gb300 as fa
    f = _noalloc(fa.lib())
    B, N, Hq, Hkv = 2, 384, 4, 2
    q = W.normal_bf16((B, N, Hq, d), 30).cuda()
    k = W.normal_bf16((B, N, Hkv, d), 31).cuda()
    v = W.normal_bf16((B, N, Hkv, d), 32).cuda()
    do = W.normal_bf16((B, N, Hq, d), 33).cuda()
    _check_against_workspace_entry_point(fa, f, q, k, v, do, causal, deterministic)


@pytest.mark.parametrize("deterministic", [False, True])
def test_noalloc_varlen_matches_workspace_entry_point(deterministic):
    import attention_blackwell_gb300 as fa
    f = _noalloc(fa.lib())
    lengths = [300, 0, 1, 129, 700]
    cu = W.cu_seqlens_of(lengths).cuda()
    T, Hq, Hkv = sum(lengths), 4, 1
    q = W.normal_bf16((T, Hq, 128), 34).cuda()
    k = W.normal_bf16((T, Hkv, 128), 35).cuda()
    v = W.normal_bf16((T, Hkv, 128), 36).cuda()
    do = W.normal_bf16((T, Hq, 128), 37).cuda()
    _check_against_workspace_entry_point(fa, f, q, k, v, do, True, deterministic, cu=cu, lengths=lengths)


def test_noalloc_device_status_is_reported_once_and_cleared():
    """A failure recorded in the scratch area's own status word reaches the
    caller through fa_get_device_status, once.  The failure used is one the
    plan stage detects on the device without faulting: a packed sequence
    longer than the 131072-token limit (max_seqlen understated), for which
    nothing is computed.  A later call on the same scratch then works."""
    import attention_blackwell_gb300 as fa
    f = _noalloc(fa.lib())
    T, d = 140000, 64
    q = torch.zeros(T, 1, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, T, dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    cu = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert fa.device_status() == 0
    rc = f(p(q), p(q), p(q), p(q), p(lse), p(q), p(dq), p(dk), p(dv), 1, 1, 1, T, d, 0.125, 1, p(cu), 1000, 0, s)
    assert rc == 0
    assert fa.device_status() == -1          # reported ...
    assert fa.device_status() == 0           # ... once: reading cleared it
    assert bool((dq == 0).all())             # nothing was added into dQ
    del q, dq, dk, dv
    test_noalloc_matches_workspace_entry_point(128, True, False)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import attention_blackwell_gb300 as fa
    f = _noalloc(fa.lib())
    t = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    P = ctypes.c_void_p(t.data_ptr())
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # B=4, Hq=16, N=4096 needs ~135 MB of workspace: rejected, nothing launched.
    assert f(P, P, P, P, P, P, P, P, P, 4, 16, 16, 4096, 128, 0.088, 0, None, 0, 0, s) == -6
