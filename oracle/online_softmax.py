"""Block-by-block online softmax with the conditional rescale, float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Restates, in the pages' order, what the forward pipeline does to one query
row block while streaming key/value blocks (FlashAttention-4 blog, "Forward
pass: a new softmax pipeline with conditional rescaling", the two-case
rescale equation; FlashAttention-4 paper summary §3.1.4):

  for each key block j:
      m_j = max(m_{j-1}, rowmax(S_j))
      if m_j - m_{j-1} > tau:   O <- exp(m_{j-1} - m_j) O + exp(S_j - m_j) V_j
      otherwise:                O <- O + exp(S_j - m_{j-1}) V_j   (stale max kept)
  O_final = O / l_final,  LSE from the final statistics.

Readings taken where the pages leave a step open:

* tau = log2(256) = 8 compares maxima in the log2 domain (logits scaled by
  alpha * log2(e)); a skipped rescale therefore leaves every term <= 2^8.
* "> tau" rescales, "<= tau" keeps the stale maximum; the first block always
  initialises (the running max starts at -inf).
* The decision is taken per warp of 32 rows: if any row of the warp exceeds
  tau, every row of that warp moves to its own new maximum.
* l and O accumulate against the same (possibly stale) maximum, so the final
  O / l and LSE = (m + log2 l) * ln 2 are exact.

Everything here is float64 with exact exp2, so the result must equal the
plain definition in ``attention.py`` for every tau (the rescale identity).
"""
import math

import numpy as np

LOG2E = 1.0 / math.log(2.0)
TAU = math.log2(256.0)  # = 8.0


def blockwise_forward(qh, kh, vh, alpha, causal=False, tau=TAU, block=128, warp_rows=32):
    """One head: qh [L,d], kh/vh [Lk,d] float64.

    Returns (O [L,d], LSE [L], rescales) where ``rescales`` counts, over all
    key blocks after the first, the warps that took the rescale branch.
    """
    qh, kh, vh = (np.asarray(t, dtype=np.float64) for t in (qh, kh, vh))
    L, Lk = qh.shape[0], kh.shape[0]
    scale = alpha * LOG2E
    m = np.full(L, -np.inf)   # running (possibly stale) max, log2 units
    l = np.zeros(L)
    o = np.zeros((L, vh.shape[1]))
    rescales = 0
    rows = np.arange(L)[:, None]
    for j0 in range(0, Lk, block):
        j1 = min(Lk, j0 + block)
        x = scale * (qh @ kh[j0:j1].T)
        if causal:
            cols = np.arange(j0, j1)[None, :]
            x = np.where(cols > rows, -np.inf, x)
        m_cand = np.maximum(m, x.max(axis=1))
        jump = np.where(np.isfinite(m), m_cand - m, np.inf)
        for w0 in range(0, L, warp_rows):
            w1 = min(L, w0 + warp_rows)
            if np.any(jump[w0:w1] > tau):
                if j0 > 0 and np.any(np.isfinite(m[w0:w1])):
                    rescales += 1
                fac = np.where(np.isfinite(m[w0:w1]), np.exp2(m[w0:w1] - m_cand[w0:w1]), 0.0)
                o[w0:w1] *= fac[:, None]
                l[w0:w1] *= fac
                m[w0:w1] = m_cand[w0:w1]
        m_use = np.where(np.isfinite(m), m, 0.0)
        p = np.exp2(x - m_use[:, None])
        l += p.sum(axis=1)
        o += p @ vh[j0:j1]
    with np.errstate(divide="ignore", invalid="ignore"):
        o_final = np.where(l[:, None] > 0, o / np.where(l > 0, l, 1.0)[:, None], 0.0)
        lse = np.where(l > 0, (m + np.log2(np.where(l > 0, l, 1.0))) / LOG2E, -np.inf)
    return o_final, lse, rescales


def max_unnormalised_term(qh, kh, alpha, causal=False, tau=TAU, block=128, warp_rows=32):
    """Largest exp2(x - m_ref) the pipeline ever forms (bounded by 2^tau)."""
    qh, kh = np.asarray(qh, np.float64), np.asarray(kh, np.float64)
    L, Lk = qh.shape[0], kh.shape[0]
    scale = alpha * LOG2E
    m = np.full(L, -np.inf)
    worst = 0.0
    rows = np.arange(L)[:, None]
    for j0 in range(0, Lk, block):
        j1 = min(Lk, j0 + block)
        x = scale * (qh @ kh[j0:j1].T)
        if causal:
            x = np.where(np.arange(j0, j1)[None, :] > rows, -np.inf, x)
        m_cand = np.maximum(m, x.max(axis=1))
        jump = np.where(np.isfinite(m), m_cand - m, np.inf)
        for w0 in range(0, L, warp_rows):
            w1 = min(L, w0 + warp_rows)
            if np.any(jump[w0:w1] > tau):
                m[w0:w1] = m_cand[w0:w1]
        fin = np.isfinite(x)
        if fin.any():
            worst = max(worst, float(np.exp2((x - np.where(np.isfinite(m), m, 0.0)[:, None])[fin]).max()))
    return worst
