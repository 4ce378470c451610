"""Oracle results for the full-size workloads, computed once per test session.

Helper for the GPU parity tests (not a test module).  The float64 oracle is
evaluated whole -- every (sequence, head) problem of the workload -- in a
pool of processes (``oracle.attention``'s ``workers``), and kept in memory so
that every kernel variant is compared against the same result.  The
references are stored as float32 once computed: that rounding (relative
6e-8) is five orders of magnitude below every tolerance they are compared
with.

Comparisons are made in slices along the leading axis to bound the memory
the temporaries take (the varlen workload's O has 238 M elements).
"""
import functools
import os

import numpy as np

from attention_blackwell_gb300 import workloads as W
from oracle import attention as A

WORKERS = max(1, min(32, os.cpu_count() or 1))


@functools.lru_cache(maxsize=None)
def inputs(name):
    w = W.WORKLOADS[name]
    return w, W.make_inputs(w, with_grad=True)


@functools.lru_cache(maxsize=None)
def forward_reference(name):
    """(o [.., Hq, d] float32, lse float64) of the whole workload."""
    w, inp = inputs(name)
    o, lse = A.forward(inp["q"], inp["k"], inp["v"], w.alpha, w.causal, cu_seqlens=inp["cu_seqlens"],
                       workers=WORKERS)
    return o.astype(np.float32), lse


@functools.lru_cache(maxsize=None)
def backward_reference(name):
    """(dq, dk, dv) float32 of the whole workload."""
    w, inp = inputs(name)
    g = A.backward(inp["q"], inp["k"], inp["v"], inp["do"], w.alpha, w.causal, cu_seqlens=inp["cu_seqlens"],
                   workers=WORKERS)
    return tuple(x.astype(np.float32) for x in g)


def abs_err_stats(got, ref, step=2048):
    """(max |got - ref|, mean |got - ref|) over every element, in slices."""
    mx, total, n = 0.0, 0.0, 0
    for i in range(0, got.shape[0], step):
        e = np.abs(got[i:i + step].astype(np.float64) - ref[i:i + step])
        mx = max(mx, float(e.max()) if e.size else 0.0)
        total += float(e.sum())
        n += e.size
    return mx, total / max(n, 1)


def max_abs(x, step=2048):
    return max((float(np.abs(x[i:i + step]).max()) for i in range(0, x.shape[0], step)), default=0.0)
