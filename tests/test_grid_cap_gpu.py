"""GPU parity with the launches' grids cut short by a test hook, so that small
layouts give every block many work items.

The kernel treats a block's items differently by their number:
- In a single launch of at most 64 items per block, the producer warp's lanes resolve up to 32 of the block's fixed-order items at once, before the dependent-launch wait, and after it stage the first four themselves (one fewer in a block that shares its last items).
- A block with more fixed-order items than its 4-stage ring prefetches the first 4 into L2; a block whose whole work fits the ring prefetches its first.
- Longer launches and batched launches look up their first 1 or 4 items one by one (4 from 16 items per block), and the lanes stage all but the last of them at once.
- A launch with at least 8 items per block (per layout, when batched) shares its last quarter through the work-sharing word.

At their planned grids, full-size groups reach these paths only at a few
points.  Here layouts of a few hundred items run on grids chosen so that the
blocks hold counts on both sides of each boundary, in every schedule and
batched, against the oracle bit for bit.
"""
import math

import pytest

from fsdp2_gradient_packing_gb300 import workloads as wl
from gpu_util import GroupRun, assert_batched_parity, assert_group_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp():
    from fsdp2_gradient_packing_gb300 import _build
    _build.build()
    from fsdp2_gradient_packing_gb300 import fsdp_pack
    return fsdp_pack


@pytest.fixture
def cap(fp):
    """Set a grid cap for one test; planned grids and the default schedule
    are restored afterwards."""
    yield fp.fsdp_debug_set_grid_cap
    fp.fsdp_debug_set_grid_cap(0)
    fp.fsdp_debug_set_schedule(fp.FSDP_SCHEDULE_DEFAULT)


def _layout(seed):
    return wl.random_layout(43000 + seed, max_params=12, max_numel=400000, W_choices=(3, 8, 13))


def _pack_items(fp, work):
    L = fp.fsdp_plan_layout_host(work.groups[0], work.W)
    try:
        return fp.fsdp_layout_query(L).pack_items
    finally:
        L.close()


# Pack items per block: around the ring size (4), the sharing threshold (8),
# the batched look-ahead threshold (16), the lanes of one warp (32) and the
# parallel-prologue limit (64), plus one block for everything.
PER_BLOCK = (2, 4, 5, 8, 9, 16, 17, 32, 33, 64, 65, 1000)


@pytest.mark.parametrize("seed", [0, 3, 5])
@pytest.mark.parametrize("k", PER_BLOCK)
def test_every_entry_point_with_k_items_per_block(fp, cap, seed, k):
    work = _layout(seed)
    n = _pack_items(fp, work)
    assert n > 150
    cap(max(1, math.ceil(n / k)))
    assert_group_parity(fp, work.groups[0], work.W, work, 0, misalign_seed=seed * 100 + k, specials=0.03)


@pytest.mark.parametrize("mode", ["FIXED", "SHARED", "MIXED"])
@pytest.mark.parametrize("k", [5, 33, 65])
def test_each_schedule_with_many_items_per_block(fp, cap, mode, k):
    fp.fsdp_debug_set_schedule(getattr(fp, f"FSDP_SCHEDULE_{mode}"))
    work = _layout(0)
    cap(max(1, math.ceil(_pack_items(fp, work) / k)))
    assert_group_parity(fp, work.groups[0], work.W, work, 0, misalign_seed=k, specials=0.03)


@pytest.mark.parametrize("blocks", [1, 3, 17, 60])
def test_batched_launches_on_few_blocks(fp, cap, blocks):
    cap(blocks)
    runs = []
    try:
        for seed in (1, 4, 7, 9):
            work = _layout(seed)
            runs.append(GroupRun(fp, work.groups[0], work.W, work, 0, misalign_seed=seed, specials=0.02))
        assert_batched_parity(fp, runs)
    finally:
        for run in runs:
            run.close()


def test_cap_above_the_planned_grid_changes_nothing(fp, cap):
    """A cap larger than every planned grid leaves the launches as planned."""
    cap(1 << 30)
    work = _layout(8)
    assert_group_parity(fp, work.groups[0], work.W, work, 0, misalign_seed=8)
