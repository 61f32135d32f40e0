"""GPU parity for a parameter of more than 2**31 elements.

A BF16 gradient / parameter of 2**31 + 2**20 + 37 elements is followed by a small FP32
one. At W = 1 the small parameter's bucket offset and the big parameter's source offsets
pass 2**31 elements. At W = 8 the bucket passes 2**32 bytes, and the gathered buffer's
rows and the full parameter's rank chunks start past 2**31 bytes. So every element and
byte offset of planning, the work table and the kernel must be 64-bit. An offset
truncated to 32 bits lands a multiple of 2**31 elements (or 2**32 bytes) away, so the
inputs are random bit patterns without any period (drawn on the device).

The checks:
- outputs the oracle computes one by one or segment by segment (pack samples including
  every run edge, the whole copy-in row, the copy-out chunks of ranks 0, 4 and 7 of the
  big parameter and every rank of the small one, the whole reduce-scatter copy-out at
  W = 8);
- each operation's definition restated with torch slicing over the whole device output
  (a BF16 -> FP32 cast is the bits shifted left by 16).
"""
import numpy as np
import pytest
import torch

import oracle
from fsdp2_gradient_packing_gb300 import workloads as wl
from gpu_util import DevBuf, first_mismatch

pytestmark = pytest.mark.gpu

N_BIG = 2**31 + 2**20 + 37
N_SMALL = 1003
SPECS = [wl.ParamSpec("big", (N_BIG,), "bf16", "f32", "f32", "bf16"),
         wl.ParamSpec("small", (N_SMALL,), "f32", "f32", "f32", "f32")]
SEED = 7000


@pytest.fixture(scope="module")
def fp():
    from fsdp2_gradient_packing_gb300 import _build
    _build.build()
    from fsdp2_gradient_packing_gb300 import fsdp_pack
    return fsdp_pack


def _dev_input(nbytes, *key):
    """A guard-banded device buffer holding seeded random bytes, and their host copy."""
    t = wl.device_random_bytes(nbytes, SEED, *key)
    buf = DevBuf(nbytes)
    buf.raw[buf.off:buf.off + nbytes].copy_(t)
    host = t.cpu().numpy()
    del t
    return buf, host


def _payload(buf, dtype):
    return buf.raw[buf.off:buf.off + buf.nbytes].view(dtype)


def _edge_samples(pl, b, rng, n_random):
    """Random flat bucket indices, every run's edges, and the indices around
    2**29, 2**30, 2**31 and 2**32 elements (the 2**31- and 2**32-byte marks)."""
    S = pl.bucket_S[b]
    total = pl.W * S
    idx = [rng.integers(0, total, n_random)]
    edges = []
    for p, spec in enumerate(pl.params):
        if pl.bucket_of[p] != b:
            continue
        c, o = pl.chunk[p], pl.bucket_off[p]
        for r in range(pl.W):
            valid = max(0, min(c, spec.numel - r * c))
            for i in (0, 1, c - 2, c - 1, valid - 1, valid, valid + 1):
                if 0 <= i < c:
                    edges.append(r * S + o + i)
    for mark in (2**29, 2**30, 2**31, 2**32):
        edges += [mark + d for d in range(-3, 4)]
    idx.append(np.array(edges, np.int64))
    idx = np.unique(np.concatenate(idx))
    return idx[(idx >= 0) & (idx < total)]


@pytest.fixture(scope="module")
def grads():
    big, big_h = _dev_input(N_BIG * 2, 0)
    small, small_h = _dev_input(N_SMALL * 4, 1)
    yield [big, small], [big_h.view(np.uint16), small_h.view(np.uint32)]
    del big, small
    torch.cuda.empty_cache()


@pytest.mark.parametrize("W", [1, 8])
def test_pack_beyond_2_31_elements(fp, grads, W):
    dev, host = grads
    pl = oracle.plan(oracle.params_from_specs(SPECS), W)
    S, c0, c1 = pl.bucket_S[0], pl.chunk[0], pl.chunk[1]
    assert W * S * 4 > 2**32 or N_BIG > 2**31
    with fp.fsdp_plan_layout(SPECS, W) as L:
        bucket = DevBuf(W * S * 4)
        fp.fsdp_pack_reduce_scatter(L, [b.ptr for b in dev], [bucket.ptr])
        torch.cuda.synchronize()
        fp.fsdp_sync_status(L)
    assert bucket.guards_ok() and all(b.guards_ok() for b in dev)
    out = _payload(bucket, torch.int32)

    idx = _edge_samples(pl, 0, np.random.default_rng(W), 2_000_000)
    got = out[torch.from_numpy(idx).cuda()].cpu().numpy().view(np.uint32)
    want = oracle.pack_samples(pl, host, 0, idx)
    assert np.array_equal(got, want), first_mismatch(got, want)

    # The whole buffer from the definition: row r holds chunk r of each
    # parameter, then zeros.  BF16 -> FP32 keeps the 16 bits as the upper
    # half of the FP32 word and zeros the lower half (little-endian halves).
    rows = out.view(W, S)
    big = _payload(dev[0], torch.int16)
    small = _payload(dev[1], torch.int32)
    for r in range(W):
        valid = max(0, min(c0, N_BIG - r * c0))
        halves = rows[r, :valid].view(torch.int16).view(valid, 2)
        assert torch.equal(halves[:, 1], big[r * c0:r * c0 + valid]), r
        assert not halves[:, 0].any()
        assert not rows[r, valid:c0].any()
        v1 = max(0, min(c1, N_SMALL - r * c1))
        assert torch.equal(rows[r, c0:c0 + v1], small[r * c1:r * c1 + v1])
        assert not rows[r, c0 + v1:c0 + c1].any()
    del rows, out, bucket
    torch.cuda.empty_cache()


def test_allgather_copy_in_and_copy_out_beyond_2_31_bytes(fp):
    W = 8
    pl = oracle.plan(oracle.params_from_specs(SPECS), W)
    c0, c1, S_ag = pl.chunk[0], pl.chunk[1], pl.S_ag
    assert W * S_ag > 2**32
    with fp.fsdp_plan_layout(SPECS, W) as L:
        # Copy-in of one rank: the whole row against the oracle.
        shards, shards_h = zip(*(_dev_input(c * 4, 2, p) for p, c in enumerate((c0, c1))))
        row = DevBuf(S_ag)
        fp.fsdp_allgather_copy_in(L, [b.ptr for b in shards], row.ptr)
        torch.cuda.synchronize()
        fp.fsdp_sync_status(L)
        assert row.guards_ok()
        want_row = oracle.allgather_copy_in(pl, [h.view(np.uint32) for h in shards_h])
        got_row = row.read()
        assert np.array_equal(got_row, want_row), first_mismatch(got_row, want_row)
        del shards, shards_h, row, got_row, want_row

        # Copy-out from W random rows (what an all-gather would deliver).
        gathered, gathered_h = _dev_input(W * S_ag, 3)
        full = [DevBuf(N_BIG * 2), DevBuf(N_SMALL * 4)]
        fp.fsdp_allgather_copy_out(L, gathered.ptr, [b.ptr for b in full])
        torch.cuda.synchronize()
        fp.fsdp_sync_status(L)
    assert all(b.guards_ok() for b in full)

    # Oracle segments: the big parameter's chunks from ranks 0, 4 (first past
    # 2**31 bytes in both buffers) and 7 (the short last chunk); the small
    # parameter from every rank.
    want = [np.zeros(N_BIG, np.uint16), np.zeros(N_SMALL, np.uint32)]
    for r in (0, 4, 7):
        oracle.allgather_copy_out_segment(pl, gathered_h, want, 0, r)
        lo, hi = r * c0, min(N_BIG, (r + 1) * c0)
        got = _payload(full[0], torch.int16)[lo:hi].cpu().numpy().view(np.uint16)
        assert np.array_equal(got, want[0][lo:hi]), (r, first_mismatch(got, want[0][lo:hi]))
    for r in range(W):
        oracle.allgather_copy_out_segment(pl, gathered_h, want, 1, r)
    got = full[1].read(np.uint32)
    assert np.array_equal(got, want[1]), first_mismatch(got, want[1])

    # The whole big parameter from the definition: chunk r is read from row r
    # at the group's start plus the parameter's offset in the group.
    g0 = pl.group_byte_off[pl.group_of[0]] + pl.group_elem_off[0] * 2
    src = _payload(gathered, torch.uint8)
    dst = _payload(full[0], torch.uint8)
    for r in range(W):
        valid = max(0, min(c0, N_BIG - r * c0))
        a = src[r * S_ag + g0:r * S_ag + g0 + valid * 2]
        assert torch.equal(dst[r * c0 * 2:(r * c0 + valid) * 2], a), r
    del gathered, gathered_h, full, src, dst
    torch.cuda.empty_cache()


@pytest.mark.parametrize("W", [1, 8])
def test_reduce_scatter_copy_out_beyond_2_31_elements(fp, W):
    pl = oracle.plan(oracle.params_from_specs(SPECS), W)
    S, c0, c1, o1 = pl.bucket_S[0], pl.chunk[0], pl.chunk[1], pl.bucket_off[1]
    with fp.fsdp_plan_layout(SPECS, W) as L:
        row, row_h = _dev_input(S * 4, 4, W)
        sharded = [DevBuf(c0 * 4), DevBuf(c1 * 4)]
        fp.fsdp_reduce_scatter_copy_out(L, [row.ptr], [b.ptr for b in sharded])
        torch.cuda.synchronize()
        fp.fsdp_sync_status(L)
    assert all(b.guards_ok() for b in sharded)
    # FP32 -> FP32: each shard is its slice of the row, whole, on the device.
    r32 = _payload(row, torch.int32)
    assert torch.equal(_payload(sharded[0], torch.int32), r32[:c0])
    assert torch.equal(_payload(sharded[1], torch.int32), r32[o1:o1 + c1])
    if W == 8:  # the oracle's whole output (1 GB) at this world size
        want = oracle.reduce_scatter_copy_out(pl, [row_h.view(np.uint32)])
        for b, w in zip(sharded, want):
            got = b.read(np.uint32)
            assert np.array_equal(got, w), first_mismatch(got, w)
    del row, row_h, sharded, r32
    torch.cuda.empty_cache()
