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


@pytest.mark.parametrize("causal,deterministic", [(True, False), (False, True)])
def test_noalloc_matches_workspace_entry_point(causal, deterministic):
    import attention_blackwell_gb300 as fa
    L = fa.lib()
    f = _noalloc(L)
    B, N, Hq, Hkv = 2, 384, 4, 2
    q = W.normal_bf16((B, N, Hq, 128), 30).cuda()
    k = W.normal_bf16((B, N, Hkv, 128), 31).cuda()
    v = W.normal_bf16((B, N, Hkv, 128), 32).cuda()
    do = W.normal_bf16((B, N, Hq, 128), 33).cuda()
    o, lse = fa.fwd(q, k, v, causal=causal)
    ref = fa.bwd(q, k, v, o, lse, do, causal=causal, deterministic=deterministic)
    s = torch.cuda.current_stream().cuda_stream
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    for call in range(2):
        dq, dk, dv = torch.full_like(q, float("nan")), torch.full_like(k, float("nan")), torch.full_like(v, float("nan"))
        rc = f(p(q), p(k), p(v), p(o), p(lse), p(do), p(dq), p(dk), p(dv), B, Hq, Hkv, N, 128,
               1 / 128 ** 0.5, int(causal), None, 0, int(deterministic), ctypes.c_void_p(s))
        assert rc == 0, (call, rc)
        torch.cuda.synchronize()
        for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
            g, r = g.float().cpu().numpy(), r.float().cpu().numpy()
            assert np.isfinite(g).all(), (call, name)
            assert np.abs(g - r).max() <= REL * np.abs(r).max(), (call, name)
            if deterministic:
                assert np.array_equal(g, r), (call, name)
    assert fa.device_status() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import attention_blackwell_gb300 as fa
    f = _noalloc(fa.lib())
    t = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    P = ctypes.c_void_p(t.data_ptr())
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # B=4, Hq=16, N=4096 needs ~135 MB of workspace: rejected, nothing launched.
    assert f(P, P, P, P, P, P, P, P, P, 4, 16, 16, 4096, 128, 0.088, 0, None, 0, 0, s) == -6
