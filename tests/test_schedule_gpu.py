"""The persistent schedulers hand out every work tile exactly once.

A tile visited twice writes the same output again, so parity alone cannot
see it (FlashAttention-4 blog, "Scheduling": each worker takes units from a
fixed order or a counter; nothing may be skipped or repeated).  The kernels'
debug counters (fa_set_debug_counters) count, per tile, the times its work
was finished:

* forward: every 128-row query tile of every (sequence, query head) once, on
  the benchmarked workloads and every forward kernel;
* backward: every work unit (128-key tile of a key/value head) once, and
  every query tile's dQ receiving exactly one contribution per key tile that
  sees it (all key tiles of its sequence, or under the causal mask the tiles
  at or before it) -- on the headline workload, whose 2048 units are claimed
  from the workspace counter over more than ten waves of CTAs, on the causal
  one in both modes, and on the packed MQA one (whose atomic units on the
  one-CTA kernel cover 8 of the 32 query heads each: one visit per head
  group);
* the conditional rescale's branch counter (paper summary §3.1.4): on the
  causal workload (Q ~ N(0, 9)) tau = 8 takes the rescale branch on some
  but not all warp decisions, tau = 0 on at least as many, tau = 64 on none.
"""
import numpy as np
import pytest
import torch

import full_size as FS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import attention_blackwell_gb300 as fa
    fa.lib()
    fa.set_tuning(0, 8.0)
    yield fa
    fa.set_debug_counters(None, None, None)
    fa.set_tuning(0, 8.0)
    fa.set_fwd_kernel(2)
    fa.set_bwd_kernel(0)
    fa.set_schedule_order(0)


def _dev(inp):
    g = {n: inp[n].cuda() for n in ("q", "k", "v", "do")}
    cu = inp["cu_seqlens"]
    g["cu"] = cu.cuda() if cu is not None else None
    g["ms"] = max(inp["lengths"]) if cu is not None else None
    return g


def _tile_starts(inp):
    """(start row, tile index within its sequence, tiles in the sequence) of
    every 128-row tile, in token-row coordinates."""
    out, row = [], 0
    for L in inp["lengths"]:
        n = (L + 127) // 128
        out += [(row + 128 * i, i, n) for i in range(n)]
        row += L
    return out


def _expected_visits(inp, H):
    T = inp["T"]
    e = np.zeros((H, T), dtype=np.int64)
    for r, _, _ in _tile_starts(inp):
        e[:, r] = 1
    return e


def _split_groups(w, kernel, deterministic):
    """Head groups per key tile of a packed batch's backward: in atomic mode
    the one-CTA kernel (d = 64 or 128) splits a key/value head's query heads
    into units of 8 when there are at least 16 of them, a multiple of 8
    (include/fa.h, fa_bwd_workspace_size); each unit counts one visit."""
    G = w.Hq // w.Hkv
    split = w.varlen and not deterministic and kernel == 0 and w.d != 256 and G >= 16 and G % 8 == 0
    return G // 8 if split else 1


def _expected_inner(inp, H, causal):
    T = inp["T"]
    e = np.zeros((H, T), dtype=np.int64)
    for r, i, n in _tile_starts(inp):
        e[:, r] = i + 1 if causal else n
    return e


@pytest.mark.parametrize("kernel", [2, 0], ids=["pair", "pingpong"])
@pytest.mark.parametrize("name", ["large", "causal", "varlen"])
def test_forward_tiles_exactly_once(fa, kernel, name):
    w, inp = FS.inputs(name)
    g = _dev(inp)
    visits = torch.zeros(w.Hq * inp["T"], dtype=torch.int32, device="cuda")
    fa.set_fwd_kernel(kernel)
    fa.set_debug_counters(visits, None, None)
    try:
        fa.fwd(g["q"], g["k"], g["v"], causal=w.causal, cu_seqlens=g["cu"], max_seqlen=g["ms"])
        assert fa.device_status() == 0
    finally:
        fa.set_debug_counters(None, None, None)
    got = visits.view(w.Hq, inp["T"]).cpu().numpy()
    assert np.array_equal(got, _expected_visits(inp, w.Hq)), (got.max(), got.sum())


@pytest.mark.parametrize("name", ["causal_d256", "varlen_d256"])
def test_forward_d256_tiles_exactly_once(fa, name):
    w, inp = FS.inputs(name)
    g = _dev(inp)
    visits = torch.zeros(w.Hq * inp["T"], dtype=torch.int32, device="cuda")
    fa.set_debug_counters(visits, None, None)
    try:
        fa.fwd(g["q"], g["k"], g["v"], causal=w.causal, cu_seqlens=g["cu"], max_seqlen=g["ms"])
        assert fa.device_status() == 0
    finally:
        fa.set_debug_counters(None, None, None)
    got = visits.view(w.Hq, inp["T"]).cpu().numpy()
    assert np.array_equal(got, _expected_visits(inp, w.Hq))


@pytest.mark.parametrize("name,kernel,deterministic", [
    ("large", 0, False), ("large", 1, False), ("causal_bwd", 0, False), ("causal_bwd", 1, False),
    ("causal_bwd", 0, True), ("causal_bwd", 1, True), ("varlen", 0, False), ("varlen", 1, False),
    ("varlen", 1, True)])
def test_backward_units_and_tiles_exactly_once(fa, name, kernel, deterministic):
    w, inp = FS.inputs(name)
    g = _dev(inp)
    T = inp["T"]
    fa.set_fwd_kernel(2)
    o, lse = fa.fwd(g["q"], g["k"], g["v"], causal=w.causal, cu_seqlens=g["cu"], max_seqlen=g["ms"])
    visits = torch.zeros(w.Hkv * T, dtype=torch.int32, device="cuda")
    inner = torch.zeros(w.Hq * T, dtype=torch.int32, device="cuda")
    fa.set_bwd_kernel(kernel)
    fa.set_debug_counters(visits, inner, None)
    try:
        ws = fa.bwd_workspace(len(inp["lengths"]), w.Hq, T if g["cu"] is not None else w.N, deterministic,
                              g["cu"] is not None)
        fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal=w.causal, cu_seqlens=g["cu"], max_seqlen=g["ms"],
               deterministic=deterministic, workspace=ws)
        assert fa.device_status(ws) == 0
    finally:
        fa.set_debug_counters(None, None, None)
        fa.set_bwd_kernel(0)
    gv = visits.view(w.Hkv, T).cpu().numpy()
    gi = inner.view(w.Hq, T).cpu().numpy()
    want_v = _expected_visits(inp, w.Hkv) * _split_groups(w, kernel, deterministic)
    assert np.array_equal(gv, want_v), (gv.max(), gv.sum())
    assert np.array_equal(gi, _expected_inner(inp, w.Hq, w.causal)), (gi.max(), gi.sum())


@pytest.mark.parametrize("kernel", [2, 0], ids=["pair", "pingpong"])
def test_rescale_branch_counts_on_the_causal_workload(fa, kernel):
    w, inp = FS.inputs("causal")
    g = _dev(inp)
    fa.set_fwd_kernel(kernel)
    counts = {}
    for tau in (0.0, 8.0, 64.0):
        c = torch.zeros(2, dtype=torch.int64, device="cuda")
        fa.set_tuning(0, tau)
        fa.set_debug_counters(None, None, c)
        try:
            fa.fwd(g["q"], g["k"], g["v"], causal=True)
            assert fa.device_status() == 0
        finally:
            fa.set_debug_counters(None, None, None)
            fa.set_tuning(0, 8.0)
        counts[tau] = [int(x) for x in c.cpu()]
    taken8, total8 = counts[8.0]
    print("rescale branch taken (kernel %d): tau=0 %d/%d, tau=8 %d/%d (%.2f %%), tau=64 %d/%d" % (
        kernel, *counts[0.0], taken8, total8, 100.0 * taken8 / max(total8, 1), *counts[64.0]))
    assert total8 > 0 and counts[0.0][1] == total8 == counts[64.0][1]
    assert 0 < taken8 < total8
    assert counts[0.0][0] >= taken8
    assert counts[64.0][0] == 0


# ------------------------------------------------ the naive order as well
# (fa_set_schedule_order(1): plain enumeration instead of the cost order;
# tests/test_schedule_order_gpu.py checks that the results do not change).

@pytest.mark.parametrize("kernel,name", [(2, "causal"), (2, "varlen"), (0, "varlen")])
def test_forward_tiles_exactly_once_naive_order(fa, kernel, name):
    fa.set_schedule_order(1)
    try:
        test_forward_tiles_exactly_once(fa, kernel, name)
    finally:
        fa.set_schedule_order(0)


def test_forward_d256_tiles_exactly_once_naive_order(fa):
    fa.set_schedule_order(1)
    try:
        test_forward_d256_tiles_exactly_once(fa, "varlen_d256")
    finally:
        fa.set_schedule_order(0)


@pytest.mark.parametrize("name,kernel,deterministic", [
    ("causal_bwd", 0, True), ("causal_bwd", 1, True), ("varlen", 0, False)])
def test_backward_units_and_tiles_exactly_once_naive_order(fa, name, kernel, deterministic):
    fa.set_schedule_order(1)
    try:
        test_backward_units_and_tiles_exactly_once(fa, name, kernel, deterministic)
    finally:
        fa.set_schedule_order(0)


# ------------------------------------------- backward at d = 64 and d = 256

def _expected_inner_steps(inp, H, causal, step):
    """Key tiles contributing to each `step`-row query step (d = 256: 64-row
    steps; a 128-key tile k reaches the steps from row 128 k on)."""
    T = inp["T"]
    e = np.zeros((H, T), dtype=np.int64)
    row = 0
    for L in inp["lengths"]:
        nk = (L + 127) // 128
        for i in range((L + step - 1) // step):
            e[:, row + step * i] = (step * i) // 128 + 1 if causal else nk
        row += L
    return e


@pytest.mark.parametrize("name,deterministic", [
    ("large_d64", False), ("causal_bwd_d64", False), ("causal_bwd_d64", True),
    ("large_d256", False), ("causal_d256", False), ("causal_d256", True), ("varlen_d256", False)])
def test_backward_other_head_dims_exactly_once(fa, name, deterministic):
    """Every 128-key unit once; every query tile (d = 64) or 64-row query
    step (d = 256, counted on the first head-dim pass) receives one
    contribution per key tile that sees it."""
    w, inp = FS.inputs(name)
    g = _dev(inp)
    T = inp["T"]
    o, lse = fa.fwd(g["q"], g["k"], g["v"], causal=w.causal, cu_seqlens=g["cu"], max_seqlen=g["ms"])
    visits = torch.zeros(w.Hkv * T, dtype=torch.int32, device="cuda")
    inner = torch.zeros(w.Hq * T, dtype=torch.int32, device="cuda")
    fa.set_debug_counters(visits, inner, None)
    try:
        ws = fa.bwd_workspace(len(inp["lengths"]), w.Hq, T if g["cu"] is not None else w.N, deterministic,
                              g["cu"] is not None, d=w.d)
        fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal=w.causal, cu_seqlens=g["cu"], max_seqlen=g["ms"],
               deterministic=deterministic, workspace=ws)
        assert fa.device_status(ws) == 0
    finally:
        fa.set_debug_counters(None, None, None)
    gv = visits.view(w.Hkv, T).cpu().numpy()
    gi = inner.view(w.Hq, T).cpu().numpy()
    assert np.array_equal(gv, _expected_visits(inp, w.Hkv)), (gv.max(), gv.sum())
    want = (_expected_inner_steps(inp, w.Hq, w.causal, 64) if w.d == 256
            else _expected_inner(inp, w.Hq, w.causal))
    assert np.array_equal(gi, want), (gi.max(), gi.sum(), want.sum())
