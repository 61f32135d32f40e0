"""GPU parity of the kernel's work schedules, through the C ABI, against the
oracle.

A launch hands out its work items in a fixed order (block b takes items b,
b + G, ...) or, for its last items, to whichever block asks first through a
work-sharing word in the layout's device memory.  The bytes written must not
depend on that choice, so every entry point is checked bit-exactly in each
schedule the test hook offers: the fixed order, every item but each block's
first through the word, and a mix in which odd blocks keep the fixed order while even blocks share
the word (some items are then written twice, with the same bytes).  Then
launches of one layout that overlap on the GPU, on two streams, must each
give the oracle's bytes: the word is held by one launch at a time and the
other launch keeps the fixed order.
"""
import numpy as np
import pytest
import torch

import oracle
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
def schedule(fp):
    """Set a schedule for one test; the default is restored afterwards."""
    yield fp.fsdp_debug_set_schedule
    fp.fsdp_debug_set_schedule(fp.FSDP_SCHEDULE_DEFAULT)


ODD_WORLD_SIZES = (1, 3, 5, 8, 12, 13, 31, 64)


@pytest.mark.parametrize("mode", ["FIXED", "SHARED", "MIXED"])
def test_every_entry_point_in_each_schedule(fp, schedule, mode):
    schedule(getattr(fp, f"FSDP_SCHEDULE_{mode}"))
    for seed in range(40):
        work = wl.random_layout(41000 + seed, max_params=12, max_numel=40000, W_choices=ODD_WORLD_SIZES)
        assert_group_parity(fp, work.groups[0], work.W, work, 0, misalign_seed=seed, specials=0.05)
    work = wl.transformer_500(W=8, layers=1)
    assert_group_parity(fp, work.groups[0], 8, work, 0)
    work = wl.kda_block(W=64, reduce="grad", d=512, ffn=1536)
    assert_group_parity(fp, work.groups[0], 64, work, 0, misalign_seed=3)
    runs = []
    try:
        for k in range(6):
            work = wl.random_layout(42000 + k, max_params=8, max_numel=30000, W_choices=ODD_WORLD_SIZES)
            runs.append(GroupRun(fp, work.groups[0], work.W, work, 0, misalign_seed=k, specials=0.02))
        assert_batched_parity(fp, runs)
    finally:
        for run in runs:
            run.close()


def test_default_schedule_shares_the_last_items(fp):
    """Two layers of the 50.3M-element layout at W = 12: 6,000+ pack items,
    more than 8 per block, so the default schedule shares its last quarter;
    every bucket row starts at a different 16-byte phase."""
    work = wl.mixed_50m(W=12, layers=2)
    L = fp.fsdp_plan_layout(work.groups[0], work.W)
    try:
        info = fp.fsdp_layout_query(L)
        assert info.pack_items >= 8 * 152 * 3
    finally:
        L.close()
    assert_group_parity(fp, work.groups[0], work.W, work, 0)


def _upload(bits):
    return torch.from_numpy(bits.view(np.uint8).copy()).cuda()


@pytest.mark.parametrize("mode", ["DEFAULT", "SHARED"])
def test_overlapping_launches_on_two_streams(fp, schedule, mode):
    """Packs and copy-outs of one layout issued alternately on two streams,
    eight of each per stream, each into its own output: every output must
    equal the oracle's, and no wait may have timed out."""
    schedule(getattr(fp, f"FSDP_SCHEDULE_{mode}"))
    work = wl.mixed_50m(W=8, layers=2)
    specs, W = work.groups[0], work.W
    pl = oracle.plan(oracle.params_from_specs(specs), W)
    grads_h = [wl.grad_values(work, 0, i) for i in range(len(specs))]
    want_pack = oracle.pack_reduce_scatter(pl, grads_h)
    gathered_h = np.concatenate([oracle.allgather_copy_in(
        pl, [wl.shard_values(work, 0, i, r, c, max(0, min(c, s.numel - r * c))) for i, (s, c) in
             enumerate(zip(specs, pl.chunk))]) for r in range(W)])
    want_full = oracle.allgather_copy_out(pl, gathered_h)
    L = fp.fsdp_plan_layout(specs, W)
    try:
        grads = [_upload(g) for g in grads_h]
        gathered = _upload(gathered_h)
        want_pack_d = [_upload(x) for x in want_pack]
        want_full_d = [_upload(x) for x in want_full]
        streams = [torch.cuda.Stream(), torch.cuda.Stream()]
        rounds = 8
        packs = [[[torch.full_like(x, 0xA5) for x in want_pack_d] for _ in range(rounds)] for _ in streams]
        fulls = [[[torch.full_like(x, 0xA5) for x in want_full_d] for _ in range(rounds)] for _ in streams]
        torch.cuda.synchronize()
        for it in range(rounds):
            for k, s in enumerate(streams):
                fp.fsdp_pack_reduce_scatter(L, grads, packs[k][it], stream=s)
                fp.fsdp_allgather_copy_out(L, gathered, fulls[k][it], stream=s)
        torch.cuda.synchronize()
        fp.fsdp_sync_status(L)
        for k in range(len(streams)):
            for it in range(rounds):
                for b, (got, want) in enumerate(zip(packs[k][it], want_pack_d)):
                    assert torch.equal(got, want), f"stream {k} round {it}: pack bucket {b} differs"
                for p, (got, want) in enumerate(zip(fulls[k][it], want_full_d)):
                    assert torch.equal(got, want), f"stream {k} round {it}: copy-out param {p} differs"
    finally:
        L.close()


@pytest.mark.parametrize("mode", ["DEFAULT", "SHARED", "MIXED"])
def test_batched_and_single_launches_share_one_word(fp, schedule, mode):
    """A batched pack of [L, L] takes its work-sharing word from its first
    layout, the same word a single pack of L uses.  Batched packs on one
    stream and single packs on another, issued alternately, must each give
    the oracle's bytes whichever launch holds the word."""
    schedule(getattr(fp, f"FSDP_SCHEDULE_{mode}"))
    work = wl.mixed_50m(W=8, layers=2)
    specs, W = work.groups[0], work.W
    pl = oracle.plan(oracle.params_from_specs(specs), W)
    grads_h = [wl.grad_values(work, 0, i, specials=0.01) for i in range(len(specs))]
    want = oracle.pack_reduce_scatter(pl, grads_h)
    L = fp.fsdp_plan_layout(specs, W)
    try:
        if mode == "DEFAULT":
            # Twice the layout's items reach the sharing threshold of a batch of two.
            assert 2 * fp.fsdp_layout_query(L).pack_items >= 8 * 2 * 152 * 3
        grads = [_upload(g) for g in grads_h]
        want_d = [_upload(x) for x in want]
        s_batched, s_single = torch.cuda.Stream(), torch.cuda.Stream()
        rounds = 6
        batched = [[torch.full_like(x, 0x5A) for _ in range(2) for x in want_d] for _ in range(rounds)]
        single = [[torch.full_like(x, 0xA5) for x in want_d] for _ in range(rounds)]
        torch.cuda.synchronize()
        for it in range(rounds):
            fp.fsdp_pack_reduce_scatter_batched([L, L], grads + grads, batched[it], stream=s_batched)
            fp.fsdp_pack_reduce_scatter(L, grads, single[it], stream=s_single)
        torch.cuda.synchronize()
        fp.fsdp_sync_status(L)
        for it in range(rounds):
            for b, got in enumerate(batched[it]):
                assert torch.equal(got, want_d[b % len(want_d)]), f"round {it}: batched bucket {b} differs"
            for b, got in enumerate(single[it]):
                assert torch.equal(got, want_d[b]), f"round {it}: single bucket {b} differs"
    finally:
        L.close()
