"""Seeded synthetic inputs for the attention workloads.

This module holds no attention arithmetic: it only draws inputs (and counts
the FLOPs the throughput metric credits).  Both the CUDA path (bench, tests)
and the CPU oracle (tests, bench's CPU baseline) take their inputs from here.

Recipe: ``torch.Generator('cpu').manual_seed(seed)``, float32 normal samples
times the stated standard deviation, rounded to bfloat16 (round to nearest
even).  Seeds: Q=0, K=1, V=2, dO=3, sequence lengths=4.

Workloads (FlashAttention-4 pages give no public dataset; these shapes are
the workloads the pages' analysis is about: d = 128, BF16, long sequences):

* tiny:   B=1, Hq=Hkv=2, N=256, non-causal.
* large:  B=4, Hq=Hkv=16, N=4096, non-causal (the compute-bound headline).
* causal: B=2, Hq=Hkv=16, N=8192, causal, Q ~ N(0, 3^2) so logits have large
  row-max jumps (exercises the conditional rescale).
* varlen: 16 packed sequences, lengths uniform integers in [512, 8192],
  Hq=32, Hkv=1 (multi-query), causal.
* causal_bwd: B=2, Hq=Hkv=16, N=8192, causal, Q, K, V, dO ~ N(0, 1).
* large_d64, causal_bwd_d64: large and causal_bwd at head dim 64 (the
  exponential-bound end of the balance between MUFU and tensor work).
* large_d256, causal_d256: large and causal at head dim 256 (the
  product-bound end).
* varlen_d256: the varlen workload's sequences and heads at head dim 256.
"""
from dataclasses import dataclass, field

import torch

HEAD_DIM = 128
SEED_Q, SEED_K, SEED_V, SEED_DO, SEED_LENS = 0, 1, 2, 3, 4


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    N: int                       # per-sequence length (fixed-length workloads)
    causal: bool
    q_std: float = 1.0
    varlen: bool = False
    len_range: tuple = (0, 0)    # varlen: inclusive range of lengths
    backward: bool = False
    d: int = HEAD_DIM
    extra: dict = field(default_factory=dict)

    @property
    def alpha(self):
        return 1.0 / (self.d ** 0.5)


WORKLOADS = {
    "tiny": Workload("tiny", B=1, Hq=2, Hkv=2, N=256, causal=False),
    "large": Workload("large", B=4, Hq=16, Hkv=16, N=4096, causal=False),
    "causal": Workload("causal", B=2, Hq=16, Hkv=16, N=8192, causal=True, q_std=3.0),
    "varlen": Workload("varlen", B=16, Hq=32, Hkv=1, N=0, causal=True, varlen=True,
                       len_range=(512, 8192)),
    "causal_bwd": Workload("causal_bwd", B=2, Hq=16, Hkv=16, N=8192, causal=True, backward=True),
    "large_d64": Workload("large_d64", B=4, Hq=16, Hkv=16, N=4096, causal=False, d=64),
    "causal_bwd_d64": Workload("causal_bwd_d64", B=2, Hq=16, Hkv=16, N=8192, causal=True, backward=True, d=64),
    "large_d256": Workload("large_d256", B=4, Hq=16, Hkv=16, N=4096, causal=False, d=256),
    "causal_d256": Workload("causal_d256", B=2, Hq=16, Hkv=16, N=8192, causal=True, d=256),
    "varlen_d256": Workload("varlen_d256", B=16, Hq=32, Hkv=1, N=0, causal=True, varlen=True,
                            len_range=(512, 8192), d=256),
}


def seq_lengths(B, lo, hi, seed=SEED_LENS):
    """B integer lengths drawn uniformly from [lo, hi] (inclusive)."""
    g = torch.Generator("cpu").manual_seed(seed)
    return [int(x) for x in torch.randint(lo, hi + 1, (B,), generator=g)]


def cu_seqlens_of(lengths):
    """int32 prefix offsets [0, L0, L0+L1, ...] of length B+1."""
    out = [0]
    for L in lengths:
        out.append(out[-1] + int(L))
    return torch.tensor(out, dtype=torch.int32)


def normal_bf16(shape, seed, std=1.0):
    """float32 N(0, std^2) samples from ``seed`` rounded to bfloat16."""
    g = torch.Generator("cpu").manual_seed(seed)
    x = torch.randn(shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        x = x * std
    return x.to(torch.bfloat16)


def make_inputs(w, lengths=None, with_grad=None):
    """CPU bf16 tensors for workload ``w``.

    Returns dict with q, k, v (and do when ``with_grad`` or w.backward),
    cu_seqlens (int32 or None), lengths, and the row count T.
    Fixed-length tensors are [B, N, H, d]; varlen tensors are packed [T, H, d].
    """
    if w.varlen:
        lengths = lengths or seq_lengths(w.B, *w.len_range)
        cu = cu_seqlens_of(lengths)
        T = int(cu[-1])
        qs, ks = (T, w.Hq, w.d), (T, w.Hkv, w.d)
    else:
        lengths = [w.N] * w.B
        cu = None
        T = w.B * w.N
        qs, ks = (w.B, w.N, w.Hq, w.d), (w.B, w.N, w.Hkv, w.d)
    out = {
        "q": normal_bf16(qs, SEED_Q, w.q_std),
        "k": normal_bf16(ks, SEED_K),
        "v": normal_bf16(ks, SEED_V),
        "cu_seqlens": cu,
        "lengths": lengths,
        "T": T,
    }
    if with_grad or (with_grad is None and w.backward):
        out["do"] = normal_bf16(qs, SEED_DO)
    return out


def attention_flops(Hq, lengths, causal, d=HEAD_DIM, backward=False):
    """FLOPs credited by the metric: 4*Hq*L^2*d per sequence for the forward,
    2.5x that for the backward, halved for causal."""
    f = sum(4.0 * Hq * L * L * d for L in lengths)
    if causal:
        f *= 0.5
    if backward:
        f *= 2.5
    return f
