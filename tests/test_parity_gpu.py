"""GPU parity: every entry point of the CUDA library, called through the C
ABI, against the CPU oracle on the same seeded inputs.  Every comparison is
bit-exact (the path only moves and casts bits, so the oracle's result is the
only correct one).  Output buffers sit between canary bands and start filled
with a non-zero pattern, so stray writes and skipped padding both show up;
inputs and outputs are placed at byte offsets that break 16-byte alignment in
the fuzz cases, to exercise the scalar heads and tails and the shifted reads.
"""
import numpy as np
import pytest
import torch

import oracle
from fsdp2_gradient_packing_gb300 import workloads as wl
from gpu_util import DevBuf, ESZ, NP, GroupRun, assert_batched_parity, assert_group_parity, first_mismatch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp():
    from fsdp2_gradient_packing_gb300 import _build
    _build.build()
    from fsdp2_gradient_packing_gb300 import fsdp_pack
    return fsdp_pack


@pytest.mark.parametrize("grouping", ["linear", "block", "model"])
def test_tiny_two_blocks(fp, grouping):
    work = wl.tiny_two_blocks(W=4, grouping=grouping)
    for g, specs in enumerate(work.groups):
        assert_group_parity(fp, specs, work.W, work, g)
        assert_group_parity(fp, specs, work.W, work, g, misalign_seed=g + 1, specials=0.2)


@pytest.mark.parametrize("chunk", range(6))
def test_random_layouts_misaligned_with_special_values(fp, chunk):
    for seed in range(chunk * 60, (chunk + 1) * 60):
        work = wl.random_layout(seed, max_params=8, max_numel=5000)
        assert_group_parity(fp, work.groups[0], work.W, work, 0, misalign_seed=seed, specials=0.05)


ODD_WORLD_SIZES = (1, 2, 3, 5, 6, 7, 8, 9, 12, 13, 16, 31, 64, 100, 128)


@pytest.mark.parametrize("chunk", range(4))
def test_random_layouts_odd_world_sizes(fp, chunk):
    """Wider random layouts (up to 12 parameters of up to 40,000 elements, so
    runs span several work items) at world sizes that divide nothing, both
    chunking rules, every buffer at a random phase, special values."""
    for seed in range(20000 + chunk * 100, 20000 + (chunk + 1) * 100):
        work = wl.random_layout(seed, max_params=12, max_numel=40000, W_choices=ODD_WORLD_SIZES)
        assert_group_parity(fp, work.groups[0], work.W, work, 0, misalign_seed=seed, specials=0.05)
    for seed in range(30000 + chunk * 40, 30000 + (chunk + 1) * 40):
        work = wl.random_layout_2d(seed, max_params=8, max_rows=400, max_row=96, W_choices=ODD_WORLD_SIZES)
        assert_group_parity(fp, work.groups[0], work.W, work, 0, misalign_seed=seed, specials=0.05, rows=True)


@pytest.mark.parametrize("batch", range(8))
def test_batched_random_layouts_odd_world_sizes(fp, batch):
    rnd = np.random.default_rng(40000 + batch)
    runs = []
    try:
        for k in range(int(rnd.integers(2, 20))):
            work = wl.random_layout(50000 + 32 * batch + k, max_params=8, max_numel=30000, W_choices=ODD_WORLD_SIZES)
            runs.append(GroupRun(fp, work.groups[0], work.W, work, 0, misalign_seed=batch * 32 + k, specials=0.02))
        assert_batched_parity(fp, runs)
    finally:
        for run in runs:
            run.close()


def test_random_long_runs_misaligned(fp):
    # runs long enough to span several work items and pipeline stages
    for seed in range(12):
        work = wl.random_layout(1000 + seed, max_params=5, max_numel=200_000, W_choices=(1, 3, 8, 64))
        assert_group_parity(fp, work.groups[0], work.W, work, 0, misalign_seed=seed, specials=0.01)


def test_transformer500_every_layer(fp):
    work = wl.transformer_500(W=8)
    assert work.n_params == 408
    for g, specs in enumerate(work.groups):
        assert_group_parity(fp, specs, work.W, work, g)


def test_world_size_one_and_sixty_four(fp):
    for W in (1, 64):
        work = wl.transformer_500(W=W, layers=2)
        for g, specs in enumerate(work.groups):
            assert_group_parity(fp, specs, W, work, g, misalign_seed=W + g, specials=0.01)


def test_mixed50m_full_size(fp):
    """The 50.3M-element group at W=8: all three entry points at full size,
    compared whole, in the launch configuration the benchmark times."""
    work = wl.mixed_50m(W=8)
    assert_group_parity(fp, work.groups[0], 8, work, 0)


def _sample_indices(pl, b, rng, n_random):
    """Random flat indices plus every (rank, parameter) run's first, last and
    first-padding positions in bucket b."""
    S = pl.bucket_S[b]
    idx = [rng.integers(0, pl.W * S, n_random)]
    edges = []
    for p, spec in enumerate(pl.params):
        if pl.bucket_of[p] != b or pl.chunk[p] == 0:
            continue
        c, o = pl.chunk[p], pl.bucket_off[p]
        for r in range(pl.W):
            valid = max(0, min(c, spec.numel - r * c))
            for i in (0, 1, c - 2, c - 1, valid - 1, valid, valid + 1):
                if 0 <= i < c:
                    edges.append(r * S + o + i)
    idx.append(np.array(edges, np.int64))
    return np.unique(np.concatenate(idx))


@pytest.mark.parametrize("W,reduce", [(8, "f32"), (64, "f32"), (8, "grad"), (64, "grad"), (8, "bf16")])
def test_kda_block_full_size(fp, W, reduce):
    """One block of the 1.75B-parameter KDA-style layout at full size, in the
    launch configuration the benchmark times.  Every bucket of the pack (up
    to 872 MB) is compared whole with the oracle's pack, element by element.
    At W = 64 the FP32 bucket row holds an odd number of elements, so every
    rank's row starts at a different 16-byte phase and most items take the
    shifted path.  The pack runs twice, into buffers pre-filled with two
    different bytes, and both must equal the oracle: every output byte was
    written.  The all-gather copy-in and copy-out are compared whole too."""
    work = wl.kda_block(W=W, reduce=reduce)
    specs = work.groups[0]
    run = GroupRun(fp, specs, W, work, 0)
    try:
        want = run.pack_expected()
        for fill in (0xA5, 0x5A):
            got, ok = run.pack(fill=fill)
            assert ok
            for b, (x, y) in enumerate(zip(got, want)):
                assert np.array_equal(x, y), f"fill {fill:#x}, bucket {b}: {first_mismatch(x, y)}"
            del got
        del want
        got, ok = run.rs_copy_out()
        assert ok
        for x, y in zip(got, run.rs_copy_out_expected()):
            assert np.array_equal(x, y), first_mismatch(x, y)
        del got
        if reduce == "f32":
            rows, full, ok = run.gather()
            assert ok
            want_rows, want_full = run.gather_expected()
            assert np.array_equal(rows, want_rows), first_mismatch(rows, want_rows)
            for x, y in zip(full, want_full):
                assert np.array_equal(x, y), first_mismatch(x, y)
    finally:
        run.close()


@pytest.mark.parametrize("reduce", ["f32", "bf16"])
def test_kda_eight_blocks_batched_full_size(fp, reduce):
    """The whole 1.75B-parameter KDA-style layout at W = 8, one fully_shard
    group per block, packed in one batched launch as the benchmark's
    eight-block run does: 3.5 GB of gradients into 7 GB (FP32) or 3.5 GB
    (BF16) of bucket rows.  The gradients are seeded random bit patterns, so
    NaN payloads, infinities and subnormals pass through every cast.  Each
    bucket is checked on random elements plus every run's edges, computed one
    by one by the oracle.  The pack runs twice, into buffers pre-filled with
    two different bytes, and the two results must be equal: every output byte
    was written."""
    W, blocks = 8, 8
    work = wl.kda_block(W=W, reduce=reduce, blocks=blocks)
    assert len(work.groups) == blocks
    layouts, plans, grads_d, grads_h, outs = [], [], [], [], []
    try:
        for g, specs in enumerate(work.groups):
            plans.append(oracle.plan(oracle.params_from_specs(specs), W))
            layouts.append(fp.fsdp_plan_layout(specs, W))
            row_d, row_h = [], []
            for i, s in enumerate(specs):
                t = wl.device_random_bytes(s.numel * ESZ[s.grad_dtype], 9100, g, i)
                row_d.append(t)
                row_h.append(t.cpu().numpy().view(NP[s.grad_dtype]))
            grads_d.append(row_d)
            grads_h.append(row_h)
        names = [["f32" if d == oracle.F32 else "bf16" for d in pl.bucket_dtype] for pl in plans]
        flat_grads = [t for row in grads_d for t in row]
        for fill in (0xA5, 0x5A):
            bufs = [[torch.full((W * S * ESZ[n],), fill, dtype=torch.uint8, device="cuda")
                     for n, S in zip(nm, pl.bucket_S)] for nm, pl in zip(names, plans)]
            fp.fsdp_pack_reduce_scatter_batched(layouts, flat_grads, [b for row in bufs for b in row])
            fp.fsdp_sync_status(layouts[0])
            outs.append(bufs)
        for g in range(blocks):
            for b, (x, y) in enumerate(zip(*(o[g] for o in outs))):
                assert torch.equal(x, y), f"block {g} bucket {b}: bytes left unwritten"
        del outs[1]
        rng = np.random.default_rng(9100)
        for g in range(blocks):
            for b, (buf, n) in enumerate(zip(outs[0][g], names[g])):
                idx = _sample_indices(plans[g], b, rng, 250_000)
                view = buf.view(torch.int32 if n == "f32" else torch.int16)
                got = view[torch.from_numpy(idx).cuda()].cpu().numpy().view(NP[n])
                want = oracle.pack_samples(plans[g], grads_h[g], b, idx)
                assert np.array_equal(got, want), f"block {g} bucket {b}: {first_mismatch(got, want)}"
    finally:
        for L in layouts:
            L.close()


def test_many_parameters_use_the_larger_parameter_blocks(fp):
    rnd = np.random.default_rng(5)
    for n in (70, 600, 4000):
        specs = tuple(wl.ParamSpec(f"p{i}", (int(rnd.integers(0, 40)),), ("f32", "bf16")[i % 2],
                                   ("f32", "bf16")[(i // 2) % 2], "f32", ("f32", "bf16")[(i // 3) % 2])
                      for i in range(n))
        work = wl.Workload(f"many{n}", 4, (specs,), std=1.0, seed=77)
        assert_group_parity(fp, specs, 4, work, 0, misalign_seed=n)


@pytest.mark.parametrize("chunk", range(4))
def test_row_chunk_mode_random_2d_layouts(fp, chunk):
    """Dim-0 row chunks (FSDP2's own sharding) with world sizes that often do
    not divide d0: all four operations against the oracle's row rule."""
    for seed in range(chunk * 40, (chunk + 1) * 40):
        work = wl.random_layout_2d(seed, max_rows=400, max_row=96)
        assert_group_parity(fp, work.groups[0], work.W, work, 0, misalign_seed=seed, specials=0.03, rows=True)


def test_row_chunk_mode_batched(fp):
    runs = []
    try:
        for k in range(6):
            work = wl.random_layout_2d(500 + k)
            runs.append(GroupRun(fp, work.groups[0], work.W, work, 0, misalign_seed=k, specials=0.03, rows=True))
        assert_batched_parity(fp, runs)
    finally:
        for run in runs:
            run.close()


def _end_to_end(fp, specs, W, work, seed, same_phase):
    """W ranks: pack each rank's gradients, emulated reduce-scatter, then each
    rank's reduce-scatter copy-out -- all on the GPU, against the oracle."""
    rng = np.random.default_rng(seed)
    pl = oracle.plan(oracle.params_from_specs(specs), W)
    grads = []
    for q in range(W):
        row = []
        for i, s in enumerate(specs):
            bits = wl.normal_bits(s.numel, s.grad_dtype, work.std, work.seed, 0, i, 20 + q)
            wl.inject_specials(bits, s.grad_dtype, 0.05, work.seed, 0, i, 20 + q)
            row.append(bits)
        grads.append(row)
    rho = ["f32" if d == oracle.F32 else "bf16" for d in pl.bucket_dtype]
    phase = {r: int(rng.integers(0, 16 // ESZ[r])) * ESZ[r] for r in ("f32", "bf16")}
    off = (lambda r: phase[r]) if same_phase else (lambda r: int(rng.integers(0, 16 // ESZ[r])) * ESZ[r])
    with fp.fsdp_plan_layout(specs, W) as L:
        packed, keep = [], []
        for q in range(W):
            g = [DevBuf(x.nbytes, 0, x) for x in grads[q]]
            out = [DevBuf(W * S * ESZ[r], off(r)) for r, S in zip(rho, pl.bucket_S)]
            fp.fsdp_pack_reduce_scatter(L, [b.ptr for b in g], [b.ptr for b in out])
            keep += g
            packed.append(out)
        red = [DevBuf(W * S * ESZ[r], off(r)) for r, S in zip(rho, pl.bucket_S)]
        fp.fsdp_emulated_reduce_scatter(L, [packed[q][b].ptr for b in range(len(rho)) for q in range(W)],
                                        [b.ptr for b in red])
        fp.fsdp_sync_status(L)
        want_red = oracle.emulated_reduce_scatter(pl, [oracle.pack_reduce_scatter(pl, grads[q]) for q in range(W)])
        for b, (buf, r, want) in enumerate(zip(red, rho, want_red)):
            got = buf.read(NP[r])
            assert np.array_equal(got, want), f"emulated reduce-scatter, bucket {b}: {first_mismatch(got, want)}"
            assert buf.guards_ok()
        for r in range(W):
            sharded = [DevBuf(c * ESZ[s.shard_dtype], 0) for s, c in zip(specs, pl.chunk)]
            fp.fsdp_reduce_scatter_copy_out(L, [buf.ptr + r * S * ESZ[rr] for buf, S, rr in zip(red, pl.bucket_S, rho)],
                                            [b.ptr for b in sharded])
            fp.fsdp_sync_status(L)
            rows = [w[r * S:(r + 1) * S] for w, S in zip(want_red, pl.bucket_S)]
            for p, (buf, s, want) in enumerate(zip(sharded, specs, oracle.reduce_scatter_copy_out(pl, rows))):
                got = buf.read(NP[s.shard_dtype])
                assert np.array_equal(got, want), f"rank {r} sharded grad {p}: {first_mismatch(got, want)}"


@pytest.mark.parametrize("same_phase", [True, False])
def test_end_to_end_pack_emulated_reduce_scatter_copy_out(fp, same_phase):
    for seed in range(40):
        work = wl.random_layout(8000 + seed, max_params=5, max_numel=3000, W_choices=(1, 2, 3, 4, 8))
        _end_to_end(fp, work.groups[0], work.W, work, seed, same_phase)
    work = wl.transformer_500(W=8, layers=1)
    _end_to_end(fp, work.groups[0], 8, work, 99, same_phase)
    work = wl.kda_block(W=8, reduce="grad", d=512, ffn=1536)
    _end_to_end(fp, work.groups[0], 8, work, 98, same_phase)


# BF16 partners for the rounding sweep below: signed zeros, subnormals, the
# smallest normal, values that put the FP32 sum exactly on, just below and just
# above a BF16 rounding tie (2**-8, 2**-9, 1.5 * 2**-8, 2**-16 against 1.0 and
# its neighbours), the largest finite values (sums that overflow to infinity),
# infinities (inf - inf) and NaNs with payloads.
BF16_PARTNERS = [0x0000, 0x8000, 0x0001, 0x8001, 0x007F, 0x807F, 0x0080, 0x8080,
                 0x3F80, 0xBF80, 0x3B80, 0xBB80, 0x3B00, 0x3BC0, 0x3780, 0x37C0, 0x3B40,
                 0x7F7F, 0xFF7F, 0x7F00, 0x7EFF, 0x4000, 0xC000, 0x7F80, 0xFF80,
                 0x7FC0, 0xFFC1, 0x7F81, 0x4B00, 0x3400]


@pytest.mark.parametrize("phase", [0, 2])
def test_emulated_rs_bf16_rounding_on_every_first_operand(fp, phase):
    """Two-rank BF16 sums of every one of the 65,536 BF16 patterns with each
    partner (plus seeded random partners): every pair's FP32 sum rounded to
    BF16 bit for bit against the oracle, through the vector path (equal phases)
    and the element path (phase 2 on one input)."""
    partners = np.array(BF16_PARTNERS + list(wl.normal_bits(34, "bf16", 1.0, 7100, 0)), np.uint16)
    K = partners.size
    n = K * 65536
    specs = [wl.ParamSpec("p", (n,), "bf16", "bf16", "f32", "bf16")]
    pl = oracle.plan(oracle.params_from_specs(specs), 2)
    assert 2 * pl.bucket_S[0] == n
    a = np.tile(np.arange(65536, dtype=np.uint32).astype(np.uint16), K)
    b = np.repeat(partners, 65536)
    want, = oracle.emulated_reduce_scatter(pl, [[a], [b]])
    with fp.fsdp_plan_layout(specs, 2) as L:
        ins = [DevBuf(2 * n, 0, a), DevBuf(2 * n, phase, b)]
        out = DevBuf(2 * n)
        fp.fsdp_emulated_reduce_scatter(L, [x.ptr for x in ins], [out.ptr])
        fp.fsdp_sync_status(L)
        got = out.read(np.uint16)
    assert out.guards_ok()
    assert np.array_equal(got, want), first_mismatch(got, want)


@pytest.mark.parametrize("phase", [0, 2])
def test_emulated_rs_at_the_rank_limit(fp, phase):
    """256 ranks, the limit: every element is the rank-ordered sum of 256
    inputs, in an FP32 and a BF16 bucket with special values, against the
    oracle (phase 2 on one input takes the element path).  257 ranks are
    refused before anything is launched."""
    specs = [wl.ParamSpec("a", (1000,), "f32", "f32", "f32", "f32"),
             wl.ParamSpec("b", (700,), "bf16", "bf16", "f32", "bf16")]
    for W in (256, 257):
        pl = oracle.plan(oracle.params_from_specs(specs), W)
        names = ["f32" if d == oracle.F32 else "bf16" for d in pl.bucket_dtype]
        packed = []
        for q in range(W):
            row = []
            for b, (name, S) in enumerate(zip(names, pl.bucket_S)):
                bits = wl.normal_bits(W * S, name, 1.0, 7200, q, b)
                wl.inject_specials(bits, name, 0.002, 7200, q, b)
                row.append(bits)
            packed.append(row)
        with fp.fsdp_plan_layout(specs, W) as L:
            ins = [DevBuf(packed[q][b].nbytes, phase if (q == 1 and b == 1) else 0, packed[q][b])
                   for b in range(len(names)) for q in range(W)]
            outs = [DevBuf(W * S * ESZ[name]) for name, S in zip(names, pl.bucket_S)]
            if W > 256:
                with pytest.raises(fp.FsdpError) as e:
                    fp.fsdp_emulated_reduce_scatter(L, [x.ptr for x in ins], [o.ptr for o in outs])
                assert e.value.status == fp.FSDP_EUNSUPPORTED
                torch.cuda.synchronize()
                assert all(bool((o.raw == 0xA5).all()) for o in outs)
                continue
            fp.fsdp_emulated_reduce_scatter(L, [x.ptr for x in ins], [o.ptr for o in outs])
            fp.fsdp_sync_status(L)
            want = oracle.emulated_reduce_scatter(pl, packed)
            for b, (o, name) in enumerate(zip(outs, names)):
                got = o.read(NP[name])
                assert o.guards_ok()
                assert np.array_equal(got, want[b]), f"bucket {b}: {first_mismatch(got, want[b])}"


def test_batched_transformer500_all_layers_in_one_launch(fp):
    work = wl.transformer_500(W=8)
    runs = [GroupRun(fp, specs, work.W, work, g) for g, specs in enumerate(work.groups)]
    try:
        assert_batched_parity(fp, runs)
    finally:
        for run in runs:
            run.close()


@pytest.mark.parametrize("batch", range(8))
def test_batched_random_layouts_mixed_world_sizes(fp, batch):
    rnd = np.random.default_rng(900 + batch)
    n = int(rnd.integers(2, 9))
    runs = []
    try:
        for k in range(n):
            work = wl.random_layout(3000 + 16 * batch + k, max_params=6, max_numel=20000)
            runs.append(GroupRun(fp, work.groups[0], work.W, work, 0, misalign_seed=batch * 16 + k, specials=0.02))
        assert_batched_parity(fp, runs)
    finally:
        for run in runs:
            run.close()


def _many_params_workload(seed: int, n: int, W: int = 4) -> wl.Workload:
    """n small parameters of random length and dtypes, one group, reduce FP32."""
    rnd = np.random.default_rng(seed)
    dts = ["f32", "bf16"]
    specs = tuple(wl.ParamSpec(f"p{i}", (int(rnd.integers(1, 40)),), dts[int(rnd.integers(0, 2))], "f32", "f32",
                               dts[int(rnd.integers(0, 2))]) for i in range(n))
    return wl.Workload(f"many{seed}", W, (specs,), 1.0, seed)


def test_batched_at_the_layout_and_pointer_limits(fp):
    """64 layouts in one batched call (the limit), and two layouts of 1,919
    parameters whose calls pass exactly 3,840 pointers (the largest parameter
    block), each against the oracle; one pointer more is refused before
    anything is launched."""
    for works in ([wl.random_layout(4100 + k, max_params=4, max_numel=3000) for k in range(64)],
                  [_many_params_workload(7300 + k, 1919) for k in range(2)]):
        runs = []
        try:
            for k, work in enumerate(works):
                runs.append(GroupRun(fp, work.groups[0], work.W, work, 0, misalign_seed=5000 + k, specials=0.02))
            assert_batched_parity(fp, runs)
        finally:
            for run in runs:
                run.close()
    works = [_many_params_workload(7400 + k, 1920) for k in range(2)]
    layouts = [fp.fsdp_plan_layout(w.groups[0], w.W) for w in works]
    try:
        mem = DevBuf(1 << 20)            # every pointer below points into it
        grads = [mem.ptr + 256 * i for i in range(2 * 1920)]
        buckets = [mem.ptr + (1 << 19), mem.ptr + (3 << 18)]
        with pytest.raises(fp.FsdpError) as e:
            fp.fsdp_pack_reduce_scatter_batched(layouts, grads, buckets)
        assert e.value.status == fp.FSDP_EUNSUPPORTED
        torch.cuda.synchronize()
        assert bool((mem.raw == 0xA5).all())
    finally:
        for L in layouts:
            L.close()


def test_batched_with_empty_layouts(fp):
    works = [wl.Workload("e0", 4, ((),), seed=1),
             wl.tiny_two_blocks(W=4, grouping="model"),
             wl.Workload("z", 2, ((wl.ParamSpec("z", (0,)), wl.ParamSpec("x", (7,), "bf16")),), seed=2)]
    runs = [GroupRun(fp, w.groups[0], w.W, w, 0) for w in works]
    try:
        assert_batched_parity(fp, runs)
        fp.fsdp_pack_reduce_scatter_batched([], [], [])
    finally:
        for run in runs:
            run.close()


def test_many_ranks_and_ranks_past_the_end(fp):
    # W far above the parameters' sizes: most ranks hold pure padding.
    specs = (wl.ParamSpec("a", (5,), "bf16"), wl.ParamSpec("b", (3, 7), "f32", "bf16"), wl.ParamSpec("c", (1,)))
    for W in (9, 100, 1000):
        work = wl.Workload(f"wide{W}", W, (specs,), seed=W)
        assert_group_parity(fp, specs, W, work, 0, misalign_seed=W, specials=0.1)
        assert_group_parity(fp, specs, W, work, 0, misalign_seed=W + 1, specials=0.1, rows=True)


def test_one_layout_from_several_host_threads(fp):
    """A layout is only read after planning: threads may share it, each on
    its own stream."""
    import threading
    work = wl.transformer_500(W=8, layers=1)
    specs = work.groups[0]
    run = GroupRun(fp, specs, 8, work, 0)
    want = run.pack_expected()[0]
    grads = [DevBuf(g.nbytes, 0, g) for g in run.grads]
    outs = [DevBuf(8 * run.pl.bucket_S[0] * 4) for _ in range(6)]
    errors = []

    def worker(k):
        try:
            s = torch.cuda.Stream()
            for _ in range(20):
                fp.fsdp_pack_reduce_scatter(run.L, [g.ptr for g in grads], [outs[k].ptr], s)
            s.synchronize()
        except Exception as e:  # pragma: no cover - reported below
            errors.append(e)
    try:
        threads = [threading.Thread(target=worker, args=(k,)) for k in range(6)]
        for t in threads:
            t.start()
        for t in threads:
            t.join()
        assert not errors, errors
        fp.fsdp_sync_status(run.L)
        for o in outs:
            assert np.array_equal(o.read(np.uint32), want)
    finally:
        run.close()


def test_calls_replay_from_a_cuda_graph(fp):
    """The entry points only launch kernels (planning and its allocation come
    first), so a step can be captured in a CUDA graph and replayed."""
    work = wl.transformer_500(W=4, layers=1)
    specs = work.groups[0]
    run = GroupRun(fp, specs, 4, work, 0, specials=0.02)
    try:
        pl = run.pl
        grads = [DevBuf(g.nbytes, 0, g) for g in run.grads]
        bucket = DevBuf(4 * pl.bucket_S[0] * 4)
        shards = [[DevBuf(x.nbytes, 0, x) for x in row] for row in run.shards]
        gathered = DevBuf(4 * pl.S_ag)
        full = [DevBuf(s.numel * ESZ[s.param_dtype]) for s in specs]
        rows = [DevBuf(x.nbytes, 0, x) for x in run.rows]
        sharded = [DevBuf(c * ESZ[s.shard_dtype]) for s, c in zip(specs, pl.chunk)]

        def step():
            fp.fsdp_pack_reduce_scatter(run.L, [g.ptr for g in grads], [bucket.ptr])
            for r in range(4):
                fp.fsdp_allgather_copy_in(run.L, [b.ptr for b in shards[r]], gathered.ptr + r * pl.S_ag)
            fp.fsdp_allgather_copy_out(run.L, gathered.ptr, [b.ptr for b in full])
            fp.fsdp_reduce_scatter_copy_out(run.L, [b.ptr for b in rows], [b.ptr for b in sharded])

        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            step()                                   # warm-up outside the capture
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        for buf in [bucket, gathered] + full + sharded:
            buf.raw[buf.off:buf.off + buf.nbytes].fill_(0x5A)
        torch.cuda.synchronize()
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        fp.fsdp_sync_status(run.L)
        assert np.array_equal(bucket.read(np.uint32), run.pack_expected()[0])
        want_rows, want_full = run.gather_expected()
        assert np.array_equal(gathered.read(), want_rows)
        for b, s_, w in zip(full, specs, want_full):
            assert np.array_equal(b.read(NP[s_.param_dtype]), w)
        for b, s_, w in zip(sharded, specs, run.rs_copy_out_expected()):
            assert np.array_equal(b.read(NP[s_.shard_dtype]), w)
    finally:
        run.close()


def test_torch_tensors_of_the_layout_dtypes_are_accepted_and_checked(fp):
    """Callers may pass float32 / bfloat16 tensors (and byte tensors for the
    all-gather buffers): correct ones give the oracle's results, a tensor
    smaller than its slot is refused before anything is launched."""
    work = wl.tiny_two_blocks(grouping="model")
    specs, W = work.groups[0], 4
    pl = oracle.plan(oracle.params_from_specs(specs), W)
    tdt = {"f32": (np.int32, torch.float32), "bf16": (np.int16, torch.bfloat16)}

    def dev(bits, dt):
        return torch.from_numpy(bits.view(tdt[dt][0]).copy()).cuda().view(tdt[dt][1])

    grads_np = [wl.grad_values(work, 0, i) for i in range(len(specs))]
    grads = [dev(g, s.grad_dtype) for g, s in zip(grads_np, specs)]
    S = pl.bucket_S[0]
    with fp.fsdp_plan_layout(specs, W) as L:
        bucket = torch.full((W * S,), float("nan"), device="cuda")
        fp.fsdp_pack_reduce_scatter(L, grads, [bucket])
        got = bucket.view(torch.int32).cpu().numpy().view(np.uint32)
        want, = oracle.pack_reduce_scatter(pl, grads_np)
        assert np.array_equal(got, want), first_mismatch(got, want)

        short = torch.full((W * S - 1,), 7.0, device="cuda")
        with pytest.raises(ValueError, match="holds"):
            fp.fsdp_pack_reduce_scatter(L, grads, [short])
        torch.cuda.synchronize()
        assert bool((short == 7.0).all())

        shards_np = [[wl.shard_values(work, 0, i, r, c, min(c, s.numel - r * c))
                      for i, (c, s) in enumerate(zip(pl.chunk, specs))] for r in range(W)]
        gathered = torch.full((W * pl.S_ag,), 0xA5, dtype=torch.uint8, device="cuda")
        for r in range(W):
            fp.fsdp_allgather_copy_in(L, [dev(x, s.shard_dtype) for x, s in zip(shards_np[r], specs)],
                                      gathered[r * pl.S_ag:(r + 1) * pl.S_ag])
        want_rows = np.concatenate([oracle.allgather_copy_in(pl, shards_np[r]) for r in range(W)])
        assert np.array_equal(gathered.cpu().numpy(), want_rows)
        full = [torch.empty(s.numel, dtype=tdt[s.param_dtype][1], device="cuda") for s in specs]
        fp.fsdp_allgather_copy_out(L, gathered, full)
        for t, s, w in zip(full, specs, oracle.allgather_copy_out(pl, want_rows)):
            got = t.view({"f32": torch.int32, "bf16": torch.int16}[s.param_dtype]).cpu().numpy().view(NP[s.param_dtype])
            assert np.array_equal(got, w), first_mismatch(got, w)


def test_flow_around_torch_collectives(fp):
    """The calls around torch.distributed's collectives, as a user makes them,
    on a one-rank NCCL process group (the collectives are then copies): pack,
    reduce_scatter_tensor, reduce-scatter copy-out; copy-in,
    all_gather_into_tensor, copy-out; every output against the oracle."""
    import socket
    import torch.distributed as dist
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    try:
        W = dist.get_world_size()
        F32, BF16 = fp.FSDP_DTYPE_F32, fp.FSDP_DTYPE_BF16
        specs = [wl.ParamSpec("w", (1024, 1024), "bf16", "f32", "f32", "bf16"),
                 wl.ParamSpec("n", (1024,), "f32", "f32", "f32", "f32")]
        work = wl.Workload("flow", W, (tuple(specs),), 1.0, 7500)
        params = [(s.numel, fp.DTYPE_CODES[s.grad_dtype], fp.DTYPE_CODES[s.reduce_dtype],
                   fp.DTYPE_CODES[s.shard_dtype], fp.DTYPE_CODES[s.param_dtype]) for s in specs]
        tdt = {F32: torch.float32, BF16: torch.bfloat16}
        ncode = {"f32": F32, "bf16": BF16}
        ibits = {F32: torch.int32, BF16: torch.int16}
        pl = oracle.plan(oracle.params_from_specs(specs), W)
        grads_np = [wl.grad_values(work, 0, i) for i in range(len(specs))]
        shards_np = [wl.shard_values(work, 0, i, 0, c, min(c, s.numel)) for i, (s, c) in enumerate(zip(specs, pl.chunk))]
        to_dev = lambda x, code: torch.from_numpy(x.view(np.int32 if code == F32 else np.int16).copy()).cuda().view(tdt[code])
        with fp.fsdp_plan_layout(params, W) as L:
            info = fp.fsdp_layout_query(L)
            buckets = [fp.fsdp_layout_bucket(L, b) for b in range(info.n_buckets)]
            chunk = [fp.fsdp_layout_param(L, p).chunk for p in range(info.n_params)]
            grads = [to_dev(g, ncode[s.grad_dtype]) for g, s in zip(grads_np, specs)]
            bufs = [torch.empty(W * b.row_elems, dtype=tdt[b.reduce_dtype], device="cuda") for b in buckets]
            fp.fsdp_pack_reduce_scatter(L, grads, bufs)
            rows = [torch.empty(b.row_elems, dtype=tdt[b.reduce_dtype], device="cuda") for b in buckets]
            for buf, row in zip(bufs, rows):
                dist.reduce_scatter_tensor(row, buf)
            sharded = [torch.empty(c, dtype=tdt[ncode[s.shard_dtype]], device="cuda") for s, c in zip(specs, chunk)]
            fp.fsdp_reduce_scatter_copy_out(L, rows, sharded)
            shards = [to_dev(x, ncode[s.shard_dtype]) for x, s in zip(shards_np, specs)]
            ag_in = torch.empty(info.ag_bytes, dtype=torch.uint8, device="cuda")
            fp.fsdp_allgather_copy_in(L, shards, ag_in)
            ag_out = torch.empty(W * info.ag_bytes, dtype=torch.uint8, device="cuda")
            dist.all_gather_into_tensor(ag_out, ag_in)
            full = [torch.empty(s.numel, dtype=tdt[ncode[s.param_dtype]], device="cuda") for s in specs]
            fp.fsdp_allgather_copy_out(L, ag_out, full)
            fp.fsdp_sync_status(L)
        bits = lambda t, code: t.view(ibits[code]).cpu().numpy().view(np.uint32 if code == F32 else np.uint16)
        want_b = oracle.pack_reduce_scatter(pl, grads_np)
        for t, w, b in zip(bufs, want_b, buckets):
            assert np.array_equal(bits(t, b.reduce_dtype), w)
        for t, w, s in zip(sharded, oracle.reduce_scatter_copy_out(pl, want_b), specs):
            assert np.array_equal(bits(t, ncode[s.shard_dtype]), w)
        want_row = oracle.allgather_copy_in(pl, shards_np)
        assert np.array_equal(ag_out.cpu().numpy(), want_row)
        for t, w, s in zip(full, oracle.allgather_copy_out(pl, want_row), specs):
            assert np.array_equal(bits(t, ncode[s.param_dtype]), w)
    finally:
        dist.destroy_process_group()


def test_empty_layout_and_empty_parameters(fp):
    with fp.fsdp_plan_layout([], 8) as L:
        fp.fsdp_pack_reduce_scatter(L, [], [])
        fp.fsdp_allgather_copy_in(L, [], None)
        fp.fsdp_allgather_copy_out(L, None, [])
        fp.fsdp_sync_status(L)
    specs = (wl.ParamSpec("z0", (0,), "bf16", "bf16"), wl.ParamSpec("x", (5,)), wl.ParamSpec("z1", (0,)))
    work = wl.Workload("zeros", 3, (specs,), seed=3)
    assert_group_parity(fp, specs, 3, work, 0)
    with fp.fsdp_plan_layout(specs, 3) as L:
        out = DevBuf(3 * 2 * 4)
        x = DevBuf(5 * 4, 0, wl.grad_values(work, 0, 1))
        fp.fsdp_pack_reduce_scatter(L, [None, x.ptr, None], [None, out.ptr])   # NULL for 0-byte tensors
        fp.fsdp_sync_status(L)
        assert out.guards_ok()


def test_argument_errors_launch_nothing(fp):
    specs = wl.tiny_two_blocks(grouping="model").groups[0]
    work = wl.tiny_two_blocks(grouping="model")
    with fp.fsdp_plan_layout(specs, 4) as L:
        grads = [DevBuf(s.numel * ESZ[s.grad_dtype], 0, wl.grad_values(work, 0, i)) for i, s in enumerate(specs)]
        out = DevBuf(4 * 36 * 4)
        cases = [
            ([grads[0].ptr + 1] + [g.ptr for g in grads[1:]], [out.ptr]),     # misaligned grad
            ([g.ptr for g in grads], [out.ptr + 2]),                          # misaligned FP32 bucket
            ([None] + [g.ptr for g in grads[1:]], [out.ptr]),                 # NULL grad
            ([g.ptr for g in grads], [None]),                                 # NULL bucket
        ]
        for gp, bp in cases:
            with pytest.raises(fp.FsdpError) as e:
                fp.fsdp_pack_reduce_scatter(L, gp, bp)
            assert e.value.status == fp.FSDP_EINVAL
        with pytest.raises(fp.FsdpError):
            fp.fsdp_allgather_copy_in(L, [g.ptr for g in grads], out.ptr + 8)   # not 16-byte aligned
        with pytest.raises(fp.FsdpError):
            fp.fsdp_allgather_copy_out(L, out.ptr + 8, [g.ptr for g in grads])
        torch.cuda.synchronize()
        assert (out.raw == 0xA5).all().item(), "a rejected call wrote to its output"


def test_calls_allocate_no_device_memory(fp):
    work = wl.mixed_50m(W=8)
    run = GroupRun(fp, work.groups[0], 8, work, 0)
    try:
        grads = [torch.from_numpy(g.view(np.int16 if g.dtype == np.uint16 else np.int32)).cuda() for g in run.grads]
        out = torch.empty(8 * run.pl.bucket_S[0], dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        free0, _ = torch.cuda.mem_get_info()
        stats0 = torch.cuda.memory_stats()["allocation.all.allocated"]
        for _ in range(3):
            fp.fsdp_pack_reduce_scatter(run.L, grads, [out])
        torch.cuda.synchronize()
        free1, _ = torch.cuda.mem_get_info()
        assert free1 == free0, "the pack call changed free device memory"
        assert torch.cuda.memory_stats()["allocation.all.allocated"] == stats0
        # The FP32 temporary a pre-cast would need: 50,331,648 * 4 B = 192 MiB.
        assert sum(g.numel() for g in grads if g.dtype == torch.int16) * 4 == 192 * 2**20
    finally:
        run.close()


def test_nondefault_stream(fp):
    work = wl.transformer_500(W=8, layers=1)
    specs = work.groups[0]
    run = GroupRun(fp, specs, 8, work, 0)
    try:
        grads = [DevBuf(g.nbytes, 0, g) for g in run.grads]
        out = DevBuf(8 * run.pl.bucket_S[0] * 4)
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            fp.fsdp_pack_reduce_scatter(run.L, [g.ptr for g in grads], [out.ptr])   # current stream = s
        s.synchronize()
        want = run.pack_expected()[0]
        assert np.array_equal(out.read(np.uint32), want)
    finally:
        run.close()


@pytest.mark.parametrize("launch", ["single", "single_on_4_blocks", "batched", "batched_on_4_blocks"])
def test_bounded_wait_reports_timeout_and_recovers(fp, launch):
    """A pipeline stage that is never armed makes its consumers hit the wait
    limit: the kernel returns, fsdp_sync_status reports FSDP_ETIMEOUT, and
    the next call runs normally.  No fault, no hang.  The unarmed stage is
    block 0's first, whichever path stages it: the producer warp's lanes
    after resolving the block's items in parallel (a single launch), lane 0
    after resolving 4 items one by one (a single launch with more than 64
    items per block, on 4 blocks; a batched launch of at least 16 items per
    block), or the producer lane's own loop (a short batched launch)."""
    work = wl.transformer_500(W=8, layers=2)
    runs = [GroupRun(fp, work.groups[g], 8, work, g) for g in range(2)]
    batched = launch.startswith("batched")
    use = runs if batched else runs[:1]
    try:
        grads = [[DevBuf(g.nbytes, 0, g) for g in run.grads] for run in use]
        outs = [DevBuf(8 * run.pl.bucket_S[0] * 4) for run in use]

        def pack():
            if batched:
                fp.fsdp_pack_reduce_scatter_batched([run.L for run in use], [g.ptr for gs in grads for g in gs],
                                                    [o.ptr for o in outs])
            else:
                fp.fsdp_pack_reduce_scatter(use[0].L, [g.ptr for g in grads[0]], [outs[0].ptr])

        if launch.endswith("on_4_blocks"):
            fp.fsdp_debug_set_grid_cap(4)
        try:
            fp.fsdp_debug_set_wait_fault(1, 50_000_000)   # 50 ms
            try:
                pack()
                with pytest.raises(fp.FsdpError) as e:
                    fp.fsdp_sync_status(use[0].L)
                assert e.value.status == fp.FSDP_ETIMEOUT
            finally:
                fp.fsdp_debug_set_wait_fault(0, 0)
            pack()
            fp.fsdp_sync_status(use[0].L)
        finally:
            fp.fsdp_debug_set_grid_cap(0)
        for run, out in zip(use, outs):
            assert np.array_equal(out.read(np.uint32), run.pack_expected()[0])
            assert out.guards_ok()
    finally:
        for run in runs:
            run.close()


def test_device_table_allocation_failure_reports_enomem(fp):
    """A failed allocation of the device work table (simulated by the test
    hook at the point of the cudaMalloc, so nothing is exhausted) gives
    FSDP_ENOMEM and no layout; a layout planned before keeps working, and
    planning works again once the hook is off."""
    work = wl.transformer_500(W=8, layers=1)
    specs = work.groups[0]
    run = GroupRun(fp, specs, 8, work, 0)
    try:
        grads = [DevBuf(g.nbytes, 0, g) for g in run.grads]
        out = DevBuf(8 * run.pl.bucket_S[0] * 4)
        torch.cuda.synchronize()
        free0, _ = torch.cuda.mem_get_info()
        fp.fsdp_debug_set_upload_fault(True)
        try:
            for plan in (lambda: fp.fsdp_plan_layout(specs, 8),
                         lambda: fp.fsdp_plan_layout_ex(specs, 8, fp.row_elems_of(specs))):
                with pytest.raises(fp.FsdpError) as e:
                    plan()
                assert e.value.status == fp.FSDP_ENOMEM
                assert "simulated" in fp.fsdp_last_error()
            with fp.fsdp_plan_layout_host(specs, 8):  # host-only planning allocates no device table
                pass
            fp.fsdp_pack_reduce_scatter(run.L, [g.ptr for g in grads], [out.ptr])
            fp.fsdp_sync_status(run.L)
        finally:
            fp.fsdp_debug_set_upload_fault(False)
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0, "a refused plan kept device memory"
        assert np.array_equal(out.read(np.uint32), run.pack_expected()[0])
        with fp.fsdp_plan_layout(specs, 8) as L:
            assert fp.fsdp_layout_query(L).has_device_table
    finally:
        run.close()


def test_stream_widen_matches_oracle(fp):
    """The plain BF16 -> FP32 streaming widen that the benchmark times beside
    the pack: every BF16 bit pattern, then a seeded array long enough for
    several grid-stride rounds, against the oracle's widening."""
    every = np.arange(65536, dtype=np.uint16)
    big = wl.normal_bits(152 * 32 * 256 * 8 * 3 + 8, "bf16", 1.0, 77, 1)
    wl.inject_specials(big, "bf16", 0.01, 77, 2)
    for bits in (every, big):
        src = torch.from_numpy(bits.view(np.int16).copy()).cuda()
        dst = torch.full((bits.size,), -1, dtype=torch.int32, device="cuda")
        fp.fsdp_debug_stream_widen(src, bits.size, dst)
        torch.cuda.synchronize()
        got = dst.cpu().numpy().view(np.uint32)
        want = oracle.bf16_to_f32(bits)
        assert np.array_equal(got, want), first_mismatch(got, want)


def test_entry_points_replay_from_a_cuda_graph(fp):
    """Every per-call entry point captured in one CUDA graph and replayed:
    the pack, the reduce-scatter copy-out, the copy-in of every rank, the
    copy-out and a batched pack of two layouts.  Each replay writes outputs
    refilled with a different byte beforehand, and each must equal the
    oracle: the launches (with their programmatic dependent launch edges)
    are recorded with their arguments and replay exactly."""
    work = wl.transformer_500(W=8, layers=2)
    runs = [GroupRun(fp, specs, work.W, work, g, misalign_seed=g + 7, specials=0.02)
            for g, specs in enumerate(work.groups)]
    try:
        r0 = runs[0]
        rho = ["f32" if d == oracle.F32 else "bf16" for d in r0.pl.bucket_dtype]
        g_bufs = [DevBuf(g.nbytes, 0, g) for g in r0.grads]
        buckets = [DevBuf(r0.W * S * ESZ[r], 0) for r, S in zip(rho, r0.pl.bucket_S)]
        rows = [DevBuf(x.nbytes, 0, x) for x in r0.rows]
        sharded = [DevBuf(c * ESZ[s.shard_dtype], 0) for s, c in zip(r0.specs, r0.pl.chunk)]
        shard_bufs = [[DevBuf(x.nbytes, 0, x) for x in r0.shards[r]] for r in range(r0.W)]
        gathered = DevBuf(r0.W * r0.pl.S_ag, 0)
        full = [DevBuf(s.numel * ESZ[s.param_dtype], 0) for s in r0.specs]
        r1 = runs[1]
        g1 = [DevBuf(g.nbytes, 0, g) for g in r1.grads]
        b_batched = [[DevBuf(run.W * S * ESZ[r], 0) for r, S in zip(rho, run.pl.bucket_S)] for run in (r0, r1)]
        outputs = buckets + sharded + [gathered] + full + [b for bs in b_batched for b in bs]

        def record():
            fp.fsdp_pack_reduce_scatter(r0.L, [b.ptr for b in g_bufs], [b.ptr for b in buckets])
            fp.fsdp_reduce_scatter_copy_out(r0.L, [b.ptr for b in rows], [b.ptr for b in sharded])
            for r in range(r0.W):
                fp.fsdp_allgather_copy_in(r0.L, [b.ptr for b in shard_bufs[r]], gathered.ptr + r * r0.pl.S_ag)
            fp.fsdp_allgather_copy_out(r0.L, gathered.ptr, [b.ptr for b in full])
            fp.fsdp_pack_reduce_scatter_batched([r0.L, r1.L], [b.ptr for b in g_bufs] + [b.ptr for b in g1],
                                                [b.ptr for bs in b_batched for b in bs])

        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            record()
        want_b = r0.pack_expected()
        want_b1 = r1.pack_expected()
        want_sh = r0.rs_copy_out_expected()
        want_rows, want_full = r0.gather_expected()
        for fill in (0x5A, 0xC3):
            for b in outputs:
                b.raw[b.off:b.off + b.nbytes].fill_(fill)
            graph.replay()
            torch.cuda.synchronize()
            fp.fsdp_sync_status(r0.L)
            for b, (buf, want, r) in enumerate(zip(buckets, want_b, rho)):
                got = buf.read(NP[r])
                assert np.array_equal(got, want), f"fill {fill:#x} pack bucket {b}: {first_mismatch(got, want)}"
            for p, (buf, s, want) in enumerate(zip(sharded, r0.specs, want_sh)):
                got = buf.read(NP[s.shard_dtype])
                assert np.array_equal(got, want), f"fill {fill:#x} rs copy-out {p}: {first_mismatch(got, want)}"
            got = gathered.read()
            assert np.array_equal(got, want_rows), f"fill {fill:#x} copy-in: {first_mismatch(got, want_rows)}"
            for p, (buf, s, want) in enumerate(zip(full, r0.specs, want_full)):
                got = buf.read(NP[s.param_dtype])
                assert np.array_equal(got, want), f"fill {fill:#x} copy-out {p}: {first_mismatch(got, want)}"
            for n, (bs, wants) in enumerate(zip(b_batched, (want_b, want_b1))):
                for b, (buf, want, r) in enumerate(zip(bs, wants, rho)):
                    got = buf.read(NP[r])
                    assert np.array_equal(got, want), f"fill {fill:#x} batched {n} bucket {b}: {first_mismatch(got, want)}"
            assert all(b.guards_ok() for b in outputs)
        del graph
    finally:
        for run in runs:
            run.close()


def test_one_layout_from_several_host_threads_and_streams(fp):
    """Four host threads share one layout, each with its own stream and
    buffers, and pack, copy in and copy out over and over at once (the C
    calls run without the Python lock, so they enter the library together;
    the launches overlap on the GPU and contend for the layout's
    work-sharing words).  Every thread's final outputs must equal the
    oracle's, and a host-side argument error raised in one thread must not
    leak into another thread's error message."""
    import threading

    work = wl.mixed_50m(W=8, layers=2)  # the pack's 6,176 items share their last quarter through a word
    specs, W = work.groups[0], work.W
    run = GroupRun(fp, specs, W, work, 0, specials=0.01)
    try:
        rho = ["f32" if d == oracle.F32 else "bf16" for d in run.pl.bucket_dtype]
        want_b = run.pack_expected()
        want_rows, want_full = run.gather_expected()
        g_bufs = [DevBuf(g.nbytes, 0, g) for g in run.grads]
        shard_bufs = [[DevBuf(x.nbytes, 0, x) for x in run.shards[r]] for r in range(W)]
        n_threads, iters = 4, 12
        outs = []
        for t in range(n_threads):
            outs.append(dict(buckets=[DevBuf(W * S * ESZ[r], 0) for r, S in zip(rho, run.pl.bucket_S)],
                             gathered=DevBuf(W * run.pl.S_ag, 0),
                             full=[DevBuf(s.numel * ESZ[s.param_dtype], 0) for s in specs],
                             stream=torch.cuda.Stream()))
        errors = []
        torch.cuda.synchronize()

        def worker(t):
            try:
                o = outs[t]
                for k in range(iters):
                    fp.fsdp_pack_reduce_scatter(run.L, [b.ptr for b in g_bufs], [b.ptr for b in o["buckets"]],
                                                o["stream"])
                    for r in range(W):
                        fp.fsdp_allgather_copy_in(run.L, [b.ptr for b in shard_bufs[r]],
                                                  o["gathered"].ptr + r * run.pl.S_ag, o["stream"])
                    fp.fsdp_allgather_copy_out(run.L, o["gathered"].ptr, [b.ptr for b in o["full"]], o["stream"])
                    if t == 1 and k % 3 == 0:  # a rejected call in one thread: 1-byte misaligned bucket
                        try:
                            fp.fsdp_pack_reduce_scatter(run.L, [b.ptr for b in g_bufs],
                                                        [o["buckets"][0].ptr + 1], o["stream"])
                            errors.append("misaligned bucket was accepted")
                        except fp.FsdpError as e:
                            if "bucket_bufs[0] is not 4-byte aligned" not in str(e):
                                errors.append(f"wrong error text: {e}")
                fp.fsdp_sync_status(run.L, o["stream"])
            except Exception as e:  # noqa: BLE001 - reported below
                errors.append(f"thread {t}: {e!r}")

        threads = [threading.Thread(target=worker, args=(t,)) for t in range(n_threads)]
        for th in threads:
            th.start()
        for th in threads:
            th.join()
        torch.cuda.synchronize()
        assert not errors, errors
        for t, o in enumerate(outs):
            for b, (buf, want, r) in enumerate(zip(o["buckets"], want_b, rho)):
                got = buf.read(NP[r])
                assert np.array_equal(got, want), f"thread {t} bucket {b}: {first_mismatch(got, want)}"
            got = o["gathered"].read()
            assert np.array_equal(got, want_rows), f"thread {t} copy-in: {first_mismatch(got, want_rows)}"
            for p, (buf, s, want) in enumerate(zip(o["full"], specs, want_full)):
                got = buf.read(NP[s.param_dtype])
                assert np.array_equal(got, want), f"thread {t} copy-out {p}: {first_mismatch(got, want)}"
    finally:
        run.close()
