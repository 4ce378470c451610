"""Exact scaled-dot-product attention, forward and backward, in float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): the product path never
imports this module.

What is computed (the plain definition that every optimisation in the
FlashAttention-4 pages reaches exactly, up to rounding):

* FlashAttention-4 blog, opening section: attention is the two GEMMs
  S = Q K^T and O = P V with a softmax between them; the paper summary's
  notation table fixes the scale alpha = 1/sqrt(d) (passed in here).
* FlashAttention-4 blog, "Forward pass" section: the output is normalised by
  the true final row statistics, O_final = O / l_final, and the kernel may store
  the log-sum-exp (LSE).  Here LSE_i = ln sum_j exp(alpha * q_i . k_j), natural
  log, including alpha.
* Causal mask: key j is visible to query i iff j <= i (top-left aligned; query
  and key lengths are equal in every workload, so there is no ambiguity).
* Grouped / multi-query heads: query head hq reads key/value head
  hq // (Hq / Hkv) (contiguous groups; the pages are silent, this is the
  plainest reading).
* Backward (FlashAttention-4 blog, "Backward pass" section names the five
  products S, dP, dV, dK, dQ and the elementwise work for P and dS): with
  upstream gradient dO, dV = P^T dO, dP = dO V^T, D_i = sum_j P_ij dP_ij,
  dS = P * (dP - D), dQ = alpha dS K, dK = alpha dS^T Q.  For grouped heads dK
  and dV sum over the query heads of the group.

Layouts: fixed-length tensors are [B, N, H, d]; variable-length tensors are
packed [T, H, d] with int32 ``cu_seqlens`` of length B+1 (sequence s owns rows
cu[s] .. cu[s+1]-1).  LSE is [B, Hq, N] (fixed length) or [Hq, T] (varlen).

Rows of S are independent, so the forward and the dQ part of the backward are
evaluated over chunks of query rows only to bound memory; no other blocking,
fusion or reordering is applied.

``workers`` (forward / backward): the (sequence, head) problems are
independent, so they may be evaluated by a pool of processes (started with
``spawn``, safe after CUDA has been initialised in the caller).  Each task
runs the same per-head function on the same inputs; the results are
assembled in the serial loop's order (dK/dV group sums included).  The output
equals ``workers=None`` up to the BLAS library's own summation order inside
each matrix product, which depends on its thread count (each worker runs it
single-threaded).
"""
import math
import multiprocessing as mp
import os
from concurrent.futures import ProcessPoolExecutor

import numpy as np

_ROW_CHUNK = 2048


def kv_head_of(hq, Hq, Hkv):
    """Key/value head read by query head ``hq`` (contiguous groups)."""
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    return hq // (Hq // Hkv)


def _as_f64(x):
    if hasattr(x, "detach"):  # torch tensor (bf16 upcast is exact)
        x = x.detach().float().cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def _sequences(B_or_T_shape, cu_seqlens):
    """Yield (seq index, row offset, length) for fixed-length or packed input."""
    if cu_seqlens is None:
        B, N = B_or_T_shape
        for b in range(B):
            yield b, None, N
    else:
        cu = [int(c) for c in np.asarray(cu_seqlens).reshape(-1)]
        for s in range(len(cu) - 1):
            yield s, cu[s], cu[s + 1] - cu[s]


def _seq_slice(x, b, off, L):
    """[L, H, d] view of sequence b of a [B,N,H,d] or packed [T,H,d] tensor."""
    return x[b] if off is None else x[off:off + L]


def _scores(qh, kh, alpha, causal, row0):
    """S = alpha * q k^T for query rows row0.. (absolute indices), causal mask."""
    s = alpha * (qh @ kh.T)
    if causal:
        rows = np.arange(row0, row0 + qh.shape[0])[:, None]
        cols = np.arange(kh.shape[0])[None, :]
        s = np.where(cols > rows, -np.inf, s)
    return s


def _softmax_rows(s):
    """Row softmax and log-sum-exp; a row with every key masked gives P=0, LSE=-inf."""
    m = s.max(axis=1, keepdims=True)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - m_safe)
    l = e.sum(axis=1, keepdims=True)
    with np.errstate(divide="ignore", invalid="ignore"):
        p = np.where(l > 0, e / np.where(l > 0, l, 1.0), 0.0)
        lse = np.where(l[:, 0] > 0, m_safe[:, 0] + np.log(np.where(l[:, 0] > 0, l[:, 0], 1.0)), -np.inf)
    return p, lse


def head_forward(qh, kh, vh, alpha, causal=False):
    """One head of one sequence: qh [L,d], kh/vh [L,d] -> (O [L,d], LSE [L])."""
    L = qh.shape[0]
    o = np.zeros((L, vh.shape[1]))
    lse = np.full(L, -np.inf)
    for r0 in range(0, L, _ROW_CHUNK):
        r1 = min(L, r0 + _ROW_CHUNK)
        p, lse[r0:r1] = _softmax_rows(_scores(qh[r0:r1], kh, alpha, causal, r0))
        o[r0:r1] = p @ vh
    return o, lse


_ONE_THREAD = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")


def _pool(workers):
    """A spawn pool whose workers each run single-threaded BLAS (the pool
    itself supplies the parallelism)."""
    saved = {k: os.environ.get(k) for k in _ONE_THREAD}
    os.environ.update({k: "1" for k in _ONE_THREAD})
    try:
        ex = ProcessPoolExecutor(max_workers=workers, mp_context=mp.get_context("spawn"))
        # Start every worker now, while the variables are set.
        list(ex.map(int, range(workers)))
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    return ex


def _head_tasks(shape, cu_seqlens, heads, Hq, Hkv):
    """(b, off, L, hq, hk) in the serial loop's order, empty sequences skipped."""
    return [(b, off, L, hq, kv_head_of(hq, Hq, Hkv))
            for b, off, L in _sequences(shape, cu_seqlens) if L > 0 for hq in heads]


def _run_heads(fn, tasks, operands, extra, workers):
    """fn(*[t[seq][:, head] for each operand], *extra) for every task, in order.

    operands: list of (tensor, 'q' | 'k') -- the head index used is hq or hk.
    """
    def args(task):  # contiguous copies in both modes, so both see identical inputs
        b, off, L, hq, hk = task
        return [np.ascontiguousarray(_seq_slice(t, b, off, L)[:, hq if which == "q" else hk])
                for t, which in operands] + list(extra)

    if not workers or workers <= 1 or len(tasks) <= 1:
        for task in tasks:
            yield task, fn(*args(task))
        return
    with _pool(min(workers, len(tasks))) as ex:
        # Bounded look-ahead keeps at most ~2 tasks per worker in flight.
        pending = []
        for task in tasks:
            pending.append((task, ex.submit(fn, *args(task))))
            if len(pending) >= 2 * workers:
                t0, f0 = pending.pop(0)
                yield t0, f0.result()
        for t0, f0 in pending:
            yield t0, f0.result()


def forward(q, k, v, alpha, causal=False, cu_seqlens=None, heads=None, workers=None):
    """O and LSE of exact attention.

    q: [B,N,Hq,d] or packed [T,Hq,d]; k, v: same with Hkv heads.
    heads: optional iterable of query heads to compute (others are left 0 /
    -inf), used to sample large workloads head by head (heads are independent).
    workers: evaluate the (sequence, head) problems in that many processes.
    Returns (o float64 like q, lse float64 [B,Hq,N] or [Hq,T]).
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    varlen = cu_seqlens is not None
    Hq, Hkv = q.shape[-2], k.shape[-2]
    o = np.zeros(q.shape[:-1] + (v.shape[-1],))
    if varlen:
        lse = np.full((Hq, q.shape[0]), -np.inf)
        shape = None
    else:
        lse = np.full((q.shape[0], Hq, q.shape[1]), -np.inf)
        shape = q.shape[:2]
    heads = range(Hq) if heads is None else list(heads)
    tasks = _head_tasks(shape, cu_seqlens, heads, Hq, Hkv)
    ops = [(q, "q"), (k, "k"), (v, "k")]
    for (b, off, L, hq, hk), (oh, lh) in _run_heads(head_forward, tasks, ops, (alpha, causal), workers):
        _seq_slice(o, b, off, L)[:, hq] = oh
        if varlen:
            lse[hq, off:off + L] = lh
        else:
            lse[b, hq] = lh
    return o, lse


def forward_rows(q, k, v, alpha, causal, picks, cu_seqlens=None):
    """O rows and LSE for sampled (sequence, query head, row) triples.

    Each output row depends only on its own query row and the visible keys, so
    sampled rows are exact.  Returns (o [n, d], lse [n]).
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    Hq, Hkv = q.shape[-2], k.shape[-2]
    if cu_seqlens is not None:
        cu = [int(c) for c in np.asarray(cu_seqlens).reshape(-1)]
    out_o, out_l = [], []
    for (b, hq, i) in picks:
        hk = kv_head_of(hq, Hq, Hkv)
        if cu_seqlens is None:
            qs, ks, vs = q[b], k[b], v[b]
        else:
            o0, L = cu[b], cu[b + 1] - cu[b]
            qs, ks, vs = q[o0:o0 + L], k[o0:o0 + L], v[o0:o0 + L]
        s = _scores(qs[i:i + 1, hq], ks[:, hk], alpha, causal, i)
        p, lse = _softmax_rows(s)
        out_o.append((p @ vs[:, hk])[0])
        out_l.append(lse[0])
    return np.array(out_o), np.array(out_l)


def dq_rows(q, k, v, do, alpha, causal, picks, cu_seqlens=None):
    """dQ rows for sampled (sequence, query head, row) triples.

    dQ_i = alpha * sum_j dS_ij k_j with dS_ij = P_ij (dP_ij - D_i),
    dP_ij = do_i . v_j and D_i = sum_j P_ij dP_ij: every quantity belongs to
    query row i and the keys it sees, so sampled rows are exact (the same
    steps as ``head_backward``, for one row).  Returns dq [n, d].
    """
    q, k, v, do = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(do)
    Hq, Hkv = q.shape[-2], k.shape[-2]
    if cu_seqlens is not None:
        cu = [int(c) for c in np.asarray(cu_seqlens).reshape(-1)]
    out = []
    for (b, hq, i) in picks:
        hk = kv_head_of(hq, Hq, Hkv)
        if cu_seqlens is None:
            qs, ks, vs, ds_ = q[b], k[b], v[b], do[b]
        else:
            o0, L = cu[b], cu[b + 1] - cu[b]
            qs, ks, vs, ds_ = q[o0:o0 + L], k[o0:o0 + L], v[o0:o0 + L], do[o0:o0 + L]
        p, _ = _softmax_rows(_scores(qs[i:i + 1, hq], ks[:, hk], alpha, causal, i))
        dp = ds_[i:i + 1, hq] @ vs[:, hk].T
        D = (p * dp).sum(axis=1, keepdims=True)
        out.append((alpha * ((p * (dp - D)) @ ks[:, hk]))[0])
    return np.array(out)


def head_backward(qh, kh, vh, doh, alpha, causal=False):
    """One head: returns (dq [L,d], dk [L,d], dv [L,d]) in float64."""
    L = qh.shape[0]
    dq = np.zeros_like(qh)
    dk = np.zeros_like(kh)
    dv = np.zeros_like(vh)
    for r0 in range(0, L, _ROW_CHUNK):
        r1 = min(L, r0 + _ROW_CHUNK)
        p, _ = _softmax_rows(_scores(qh[r0:r1], kh, alpha, causal, r0))
        do = doh[r0:r1]
        dv += p.T @ do
        dp = do @ vh.T
        D = (p * dp).sum(axis=1, keepdims=True)
        ds = p * (dp - D)
        dq[r0:r1] = alpha * (ds @ kh)
        dk += alpha * (ds.T @ qh[r0:r1])
    return dq, dk, dv


def backward(q, k, v, do, alpha, causal=False, cu_seqlens=None, heads=None, workers=None):
    """dQ, dK, dV of L = sum(O * dO) for exact attention, float64.

    heads: optional query heads to include (for sampling whole heads of large
    workloads); dK/dV of a key/value head then sum only the included heads.
    workers: evaluate the (sequence, head) problems in that many processes.
    """
    q, k, v, do = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(do)
    Hq, Hkv = q.shape[-2], k.shape[-2]
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    shape = None if cu_seqlens is not None else q.shape[:2]
    heads = range(Hq) if heads is None else list(heads)
    tasks = _head_tasks(shape, cu_seqlens, heads, Hq, Hkv)
    ops = [(q, "q"), (k, "k"), (v, "k"), (do, "q")]
    for (b, off, L, hq, hk), (a, bb, c) in _run_heads(head_backward, tasks, ops, (alpha, causal), workers):
        _seq_slice(dq, b, off, L)[:, hq] = a
        _seq_slice(dk, b, off, L)[:, hk] += bb
        _seq_slice(dv, b, off, L)[:, hk] += c
    return dq, dk, dv


def delta(o, do):
    """D_i = sum_d dO_id * O_id (the row term the backward's dS needs)."""
    return (_as_f64(o) * _as_f64(do)).sum(axis=-1)


# ---------------------------------------------------------------------------
# Brute force: pure Python loops, tiny shapes only.  Written independently of
# the NumPy code above (no shared helper) so each can pin the other.
# ---------------------------------------------------------------------------

def bruteforce_forward(q, k, v, alpha, causal=False):
    """q, k, v: nested lists / arrays [N][d] for ONE head.  Returns (O, LSE) lists."""
    q = [[float(x) for x in row] for row in q]
    k = [[float(x) for x in row] for row in k]
    v = [[float(x) for x in row] for row in v]
    n, dv = len(q), len(v[0]) if v else 0
    out, lses = [], []
    for i in range(n):
        logits = []
        for j in range(len(k)):
            if causal and j > i:
                continue
            logits.append((j, alpha * sum(a * b for a, b in zip(q[i], k[j]))))
        big = max(s for _, s in logits)
        weights = [(j, math.exp(s - big)) for j, s in logits]
        total = sum(w for _, w in weights)
        row = [0.0] * dv
        for j, w in weights:
            for c in range(dv):
                row[c] += w / total * v[j][c]
        out.append(row)
        lses.append(big + math.log(total))
    return out, lses
