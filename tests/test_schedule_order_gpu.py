"""The order of the work units does not change the result.

The schedulers only decide which worker computes a tile and when
(FlashAttention-4 blog, "Scheduling"); each tile's arithmetic is its own.
fa_set_schedule_order(1) makes every kernel take its units in plain
enumeration order -- (sequence, head) major, tiles ascending, sequences in
index order -- instead of the cost-ordered schedule (longest first, L2-sized
sections, zig-zag couples, packed sequences sorted by length).  Under both
orders
* every forward kernel's O and LSE are bitwise identical;
* the deterministic backward's dQ, dK and dV are bitwise identical: its dQ
  additions follow the key-tile order at every query tile whatever order
  the units are claimed in;
* the atomic backward's agree to within the order of the fp32 dQ additions.
The shapes take both causal paths of the fixed-length forward order (zig-zag
couples for an even number of 256-row blocks, L2 sections for an odd one),
grouped heads, and packed batches with empty, one-token and ragged
sequences, whose unit tables the order changes the most.
"""
import numpy as np
import pytest
import torch

from attention_blackwell_gb300 import workloads as W

pytestmark = pytest.mark.gpu

LENGTHS = [700, 0, 1, 2049, 129, 513, 3000, 257]


@pytest.fixture(scope="module")
def fa():
    import attention_blackwell_gb300 as fa
    fa.lib()
    fa.set_tuning(0, 8.0)
    yield fa
    fa.set_schedule_order(0)
    fa.set_fwd_kernel(2)
    fa.set_bwd_kernel(0)


def make(B, N, Hq, Hkv, d, lengths=None, seed=0):
    if lengths is not None:
        cu = W.cu_seqlens_of(lengths)
        T = int(cu[-1])
        sq, sk = (T, Hq, d), (T, Hkv, d)
    else:
        cu = None
        sq, sk = (B, N, Hq, d), (B, N, Hkv, d)
    g = {"q": W.normal_bf16(sq, seed, 2.0), "k": W.normal_bf16(sk, seed + 1), "v": W.normal_bf16(sk, seed + 2),
         "do": W.normal_bf16(sq, seed + 3)}
    g = {n: t.cuda() for n, t in g.items()}
    g["cu"] = cu.cuda() if cu is not None else None
    g["ms"] = max(lengths) if lengths is not None else None
    g["B"] = len(lengths) if lengths is not None else B
    g["N"] = T if lengths is not None else N
    g["d"] = d
    return g


def fwd(fa, g, causal, order, out=None):
    fa.set_schedule_order(order)
    try:
        o, lse = fa.fwd(g["q"], g["k"], g["v"], causal=causal, cu_seqlens=g["cu"], max_seqlen=g["ms"])
        assert fa.device_status() == 0
    finally:
        fa.set_schedule_order(0)
    return o, lse


def same_bits(a, b):
    if a.dtype == torch.bfloat16:
        return torch.equal(a.view(torch.int16), b.view(torch.int16))
    return torch.equal(a.view(torch.int32), b.view(torch.int32))


FWD_CASES = {
    "causal_even_blocks": dict(B=2, N=2048, Hq=4, Hkv=4, causal=True),
    "causal_odd_blocks": dict(B=3, N=1792, Hq=4, Hkv=2, causal=True),
    "noncausal_ragged": dict(B=2, N=1000, Hq=4, Hkv=1, causal=False),
    "varlen_causal": dict(lengths=LENGTHS, Hq=4, Hkv=2, causal=True),
    "varlen": dict(lengths=LENGTHS, Hq=4, Hkv=1, causal=False),
}


def _fwd_case(fa, name, d):
    c = dict(FWD_CASES[name])
    causal = c.pop("causal")
    g = make(c.get("B", 0), c.get("N", 0), c["Hq"], c["Hkv"], d, lengths=c.get("lengths"))
    o0, l0 = fwd(fa, g, causal, 0)
    o1, l1 = fwd(fa, g, causal, 1)
    assert torch.isfinite(o0.float()).all()
    assert same_bits(o0, o1), (o0.float() - o1.float()).abs().max().item()
    assert same_bits(l0, l1), (l0 - l1).abs().max().item()


@pytest.mark.parametrize("kernel", [2, 0], ids=["pair", "pingpong"])
@pytest.mark.parametrize("name", list(FWD_CASES))
def test_forward_d128_bitwise_under_both_orders(fa, kernel, name):
    fa.set_fwd_kernel(kernel)
    try:
        _fwd_case(fa, name, 128)
    finally:
        fa.set_fwd_kernel(2)


@pytest.mark.parametrize("d", [64, 256])
@pytest.mark.parametrize("name", ["causal_odd_blocks", "varlen_causal", "varlen"])
def test_forward_other_head_dims_bitwise_under_both_orders(fa, d, name):
    _fwd_case(fa, name, d)


BWD_CASES = {
    "causal": dict(B=2, N=1100, Hq=4, Hkv=2, causal=True),
    "noncausal": dict(B=2, N=700, Hq=2, Hkv=2, causal=False),
    "varlen_causal": dict(lengths=LENGTHS, Hq=4, Hkv=1, causal=True),
}


def bwd(fa, g, causal, o, lse, deterministic, order):
    ws = fa.bwd_workspace(g["B"], g["q"].shape[-2], g["N"], deterministic, g["cu"] is not None, d=g["d"])
    fa.set_schedule_order(order)
    try:
        out = fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal=causal, cu_seqlens=g["cu"],
                     max_seqlen=g["ms"], deterministic=deterministic, workspace=ws)
        assert fa.device_status(ws) == 0
    finally:
        fa.set_schedule_order(0)
    return out


@pytest.mark.parametrize("d,kernel", [(128, 0), (128, 1), (64, 0), (256, 0)],
                         ids=["d128_one_cta", "d128_pair", "d64", "d256"])
@pytest.mark.parametrize("name", list(BWD_CASES))
def test_deterministic_backward_bitwise_under_both_orders(fa, d, kernel, name):
    c = dict(BWD_CASES[name])
    causal = c.pop("causal")
    g = make(c.get("B", 0), c.get("N", 0), c["Hq"], c["Hkv"], d, lengths=c.get("lengths"), seed=10)
    o, lse = fwd(fa, g, causal, 0)
    fa.set_bwd_kernel(kernel)
    try:
        ref = bwd(fa, g, causal, o, lse, True, 0)
        got = bwd(fa, g, causal, o, lse, True, 1)
    finally:
        fa.set_bwd_kernel(0)
    for n, a, b in zip(("dq", "dk", "dv"), ref, got):
        assert torch.isfinite(a.float()).all(), n
        assert same_bits(a, b), (n, (a.float() - b.float()).abs().max().item())


@pytest.mark.parametrize("kernel", [0, 1], ids=["one_cta", "pair"])
@pytest.mark.parametrize("name", ["causal", "noncausal"])
def test_atomic_backward_within_summation_order_under_both_orders(fa, kernel, name):
    c = dict(BWD_CASES[name])
    causal = c.pop("causal")
    g = make(c["B"], c["N"], c["Hq"], c["Hkv"], 128, seed=20)
    o, lse = fwd(fa, g, causal, 0)
    ref = bwd(fa, g, causal, o, lse, True, 0)
    fa.set_bwd_kernel(kernel)
    try:
        got = bwd(fa, g, causal, o, lse, False, 1)
    finally:
        fa.set_bwd_kernel(0)
    for n, a, b in zip(("dq", "dk", "dv"), ref, got):
        a, b = a.float(), b.float()
        tol = 1e-2 * max(a.abs().max().item(), 1e-6)
        assert (a - b).abs().max().item() <= tol, n


def test_varlen_plan_for_the_other_backward_kernel_is_refused(fa):
    """Stage 1 of a packed batch plans the work list for the backward kernel
    selected at that time (128-key units for the one-CTA kernel, 256-key
    blocks for CTA pairs).  A stage 2 run under the other selection must
    compute nothing and report FA_ERR_INVALID, never read the list with the
    wrong unit size; a consistent pair of stages then works again."""
    g = make(0, 0, 2, 1, 128, lengths=[300, 129, 513], seed=41)
    o, lse = fwd(fa, g, True, 0)
    ws = fa.bwd_workspace(g["B"], 2, g["N"], False, True)
    dq, dk, dv = (torch.zeros_like(t) for t in (g["q"], g["k"], g["v"]))
    kw = dict(causal=True, cu_seqlens=g["cu"], max_seqlen=g["ms"], workspace=ws, dq=dq, dk=dk, dv=dv)
    try:
        for first, second in ((0, 1), (1, 0)):
            fa.set_bwd_kernel(first)
            fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], stages=1, **kw)
            fa.set_bwd_kernel(second)
            fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], stages=2, **kw)
            assert fa.device_status(ws) == -1   # FA_ERR_INVALID
            fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], stages=1, **kw)
            fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], stages=2, **kw)
            assert fa.device_status(ws) == 0
    finally:
        fa.set_bwd_kernel(0)


def test_varlen_plan_for_the_other_mode_is_refused(fa):
    """With 16 query heads per key/value head, stage 1 in atomic mode plans
    units of 8 query heads (their dK and dV partial sums in fp32) and in
    deterministic mode one unit per key tile.  A stage 2 in the other mode
    must compute nothing and report FA_ERR_INVALID; a consistent pair of
    stages then works again."""
    g = make(0, 0, 16, 1, 128, lengths=[300, 129, 513], seed=42)
    o, lse = fwd(fa, g, True, 0)
    ws = fa.bwd_workspace(g["B"], 16, g["N"], True, True)   # sized for both modes
    dq, dk, dv = (torch.zeros_like(t) for t in (g["q"], g["k"], g["v"]))
    kw = dict(causal=True, cu_seqlens=g["cu"], max_seqlen=g["ms"], workspace=ws, dq=dq, dk=dk, dv=dv)
    for first, second in ((False, True), (True, False)):
        fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], stages=1, deterministic=first, **kw)
        fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], stages=2, deterministic=second, **kw)
        assert fa.device_status(ws) == -1   # FA_ERR_INVALID
        fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], stages=1, deterministic=second, **kw)
        fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], stages=2, deterministic=second, **kw)
        assert fa.device_status(ws) == 0
