"""The per-tile cycle model (bench.tile_budget) against the figures the pages
print for it.

FA4 blog, "Feeds and speeds", and FA4 paper summary, Tables 1 and 3: per
B200 SM (8192 BF16 FLOP, 16 exponentials and 128 shared-memory bytes per
clock) one 128 x 128 tile at d = 128 costs
  forward:  1024 tensor-core, 1024 exponential, 768 shared-memory cycles;
  backward: 2560 tensor-core, 1024 exponential, 3328 shared-memory cycles on
            one CTA, 2688 on a CTA pair.
The model counts each byte source separately, so a dropped term (the dQ
round trip, the dS store) or one counted on the wrong side (dK's dS^T from
shared memory instead of tensor memory, a halved A operand on the pair)
misses one of these numbers.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_forward_tile_b200():
    assert bench.tile_budget("fwd") == {"mma": 1024, "exp": 1024, "smem": 768}


def test_backward_tile_b200_one_cta_and_pair():
    assert bench.tile_budget("bwd") == {"mma": 2560, "exp": 1024, "smem": 3328}
    assert bench.tile_budget("bwd", pair=True) == {"mma": 2560, "exp": 1024, "smem": 2688}
    # The pages' margins: shared memory 30 % above the tensor core on one
    # CTA, 5 % on a pair.
    one, two = bench.tile_budget("bwd"), bench.tile_budget("bwd", pair=True)
    assert one["smem"] / one["mma"] == pytest.approx(1.3, abs=0.005)
    assert two["smem"] / two["mma"] == pytest.approx(1.05, abs=0.0001)


def test_balance_moves_with_head_dim():
    """FA4 paper summary, remark after Table 1: the exponentials do not
    depend on d while the products grow with it, so d = 128 is where they
    balance; below it the exponentials bound the forward, above it the
    products do."""
    for d, rel in ((64, "lt"), (128, "eq"), (256, "gt")):
        t = bench.tile_budget("fwd", d=d)
        assert t["exp"] == 1024
        assert t["mma"] == 8 * d
        assert {"lt": t["mma"] < t["exp"], "eq": t["mma"] == t["exp"], "gt": t["mma"] > t["exp"]}[rel]


def test_gb300_exponential_rate():
    """FA4 synthesis page: B300 / GB300 run 32 exponentials per clock per SM,
    which halves the forward's exponential time and leaves the products as
    its bound at d = 128."""
    t = bench.tile_budget("fwd", exp_per_clk=32)
    assert t["exp"] == 512 and t["mma"] == 1024


def test_this_builds_one_cta_backward_accounting():
    """The one-CTA backward here lands Q and dO in shared memory by TMA and
    dK takes dS^T from tensor memory: 480 KB per tile at d = 128, 3840
    cycles at 128 bytes per clock; with dS^T read from shared memory instead
    (the earlier layout) the same tile is 512 KB, 4096 cycles.  The CTA-pair
    forward moves 1024 cycles' worth per SM with its copies included, the
    one-CTA forward 1536."""
    t = bench.tile_budget("bwd", tma_writes=True)
    assert t["smem"] * 128 == 480 * 1024 and t["smem"] == 3840
    t = bench.tile_budget("bwd", ds_t_in_tmem=False, tma_writes=True)
    assert t["smem"] * 128 == 512 * 1024 and t["smem"] == 4096
    # d = 64: 16 KB tiles, dS^T 32 KB, fp32 dQ 32 KB -> 272 KB per tile
    # (304 KB with dK reading dS^T from shared memory)
    assert bench.tile_budget("bwd", d=64, tma_writes=True)["smem"] * 128 == 272 * 1024
    assert bench.tile_budget("bwd", d=64, ds_t_in_tmem=False, tma_writes=True)["smem"] * 128 == 304 * 1024
    assert bench.tile_budget("fwd", pair=True, tma_writes=True)["smem"] == 1024
    assert bench.tile_budget("fwd", tma_writes=True)["smem"] == 1536


def test_unknown_kind_rejected():
    with pytest.raises(ValueError):
        bench.tile_budget("both")
