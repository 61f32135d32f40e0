"""Helpers for the GPU parity tests: guard-banded device buffers at chosen
byte offsets, and a runner that pushes one fully_shard group through the three
entry points of the CUDA library and through the oracle on the same inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from fsdp2_gradient_packing_gb300 import workloads as wl

GUARD = 4096
FILL = 0xA5
NP = {"f32": np.uint32, "bf16": np.uint16}
ESZ = {"f32": 4, "bf16": 2}


class DevBuf:
    """``nbytes`` of device memory starting ``offset`` bytes past a 512-byte
    aligned address, with GUARD canary bytes on both sides.  Everything,
    including the payload, starts as FILL so unwritten bytes show up."""

    def __init__(self, nbytes: int, offset: int = 0, data: np.ndarray | None = None, fill: int = FILL):
        self.nbytes = int(nbytes)
        self.off = GUARD + int(offset)
        self.fill = fill
        self.raw = torch.full((self.off + self.nbytes + GUARD,), fill, dtype=torch.uint8, device="cuda")
        assert self.raw.data_ptr() % 512 == 0
        if data is not None:
            self.write(data)

    @property
    def ptr(self) -> int:
        return self.raw.data_ptr() + self.off

    def write(self, data: np.ndarray) -> None:
        b = np.ascontiguousarray(data).view(np.uint8).reshape(-1)
        assert b.size == self.nbytes
        if b.size:
            self.raw[self.off:self.off + b.size].copy_(torch.from_numpy(b.copy()))

    def read(self, dtype=np.uint8) -> np.ndarray:
        return self.raw[self.off:self.off + self.nbytes].cpu().numpy().view(dtype)

    def guards_ok(self) -> bool:
        head = self.raw[:self.off]
        tail = self.raw[self.off + self.nbytes:]
        return bool((head == self.fill).all().item()) and bool((tail == self.fill).all().item())


def _offset(rng, align: int) -> int:
    """A byte offset that keeps ``align``-byte alignment but usually breaks 16."""
    if rng is None:
        return 0
    return int(rng.integers(0, 16 // align)) * align


class GroupRun:
    """One group through the CUDA library and the oracle."""

    def __init__(self, fp, specs, W: int, work: wl.Workload, group: int, misalign_seed=None,
                 specials: float = 0.0, rows: bool = False):
        self.fp, self.specs, self.W = fp, list(specs), W
        self.work, self.group = work, group
        row_elems = fp.row_elems_of(specs) if rows else None
        self.pl = oracle.plan(oracle.params_from_specs(specs), W, row_elems=row_elems)
        self.L = fp.fsdp_plan_layout_ex(specs, W, row_elems) if rows else fp.fsdp_plan_layout(specs, W)
        self.rng = np.random.default_rng(misalign_seed) if misalign_seed is not None else None
        self.grads = [wl.grad_values(work, group, i, specials=specials) for i in range(len(specs))]
        # This rank's reduced bucket rows (the reduce-scatter output).
        self.rows = []
        for b, (dt, S) in enumerate(zip(self.pl.bucket_dtype, self.pl.bucket_S)):
            name = "f32" if dt == oracle.F32 else "bf16"
            bits = wl.normal_bits(S, name, work.std, work.seed, group, 4, b)
            if specials:
                wl.inject_specials(bits, name, specials, work.seed, group, 4, b)
            self.rows.append(bits)
        self.shards = []
        for r in range(W):
            row = []
            for i, (s, c) in enumerate(zip(specs, self.pl.chunk)):
                row.append(wl.shard_values(work, group, i, r, c, max(0, min(c, s.numel - r * c)),
                                           specials=specials))
            self.shards.append(row)

    def close(self):
        self.L.close()

    # -- reduce-scatter copy-in --------------------------------------------
    def pack(self, fill: int = FILL):
        fp, pl = self.fp, self.pl
        g_bufs = [DevBuf(g.nbytes, _offset(self.rng, ESZ[s.grad_dtype]), g) for s, g in zip(self.specs, self.grads)]
        rho = ["f32" if d == oracle.F32 else "bf16" for d in pl.bucket_dtype]
        out = [DevBuf(self.W * S * ESZ[r], _offset(self.rng, ESZ[r]), fill=fill) for r, S in zip(rho, pl.bucket_S)]
        fp.fsdp_pack_reduce_scatter(self.L, [b.ptr for b in g_bufs], [b.ptr for b in out])
        fp.fsdp_sync_status(self.L)
        got = [b.read(NP[r]) for b, r in zip(out, rho)]
        ok = all(b.guards_ok() for b in out + g_bufs)
        return got, ok

    def pack_expected(self):
        return oracle.pack_reduce_scatter(self.pl, self.grads)

    # -- reduce-scatter copy-out -------------------------------------------
    def rs_copy_out(self):
        fp, pl = self.fp, self.pl
        rho = ["f32" if d == oracle.F32 else "bf16" for d in pl.bucket_dtype]
        rows = [DevBuf(x.nbytes, _offset(self.rng, ESZ[r]), x) for x, r in zip(self.rows, rho)]
        outs = [DevBuf(c * ESZ[s.shard_dtype], _offset(self.rng, ESZ[s.shard_dtype])) for s, c in zip(self.specs, pl.chunk)]
        fp.fsdp_reduce_scatter_copy_out(self.L, [b.ptr for b in rows], [b.ptr for b in outs])
        fp.fsdp_sync_status(self.L)
        got = [b.read(NP[s.shard_dtype]) for b, s in zip(outs, self.specs)]
        return got, all(b.guards_ok() for b in rows + outs)

    def rs_copy_out_expected(self):
        return oracle.reduce_scatter_copy_out(self.pl, self.rows)

    # -- all-gather copy-in (every rank into its row) and copy-out ------------
    def gather(self):
        fp, pl = self.fp, self.pl
        gathered = DevBuf(self.W * pl.S_ag, 0)
        inputs = []
        for r in range(self.W):
            bufs = [DevBuf(x.nbytes, _offset(self.rng, ESZ[s.shard_dtype]), x) for s, x in zip(self.specs, self.shards[r])]
            inputs += bufs
            fp.fsdp_allgather_copy_in(self.L, [b.ptr for b in bufs], gathered.ptr + r * pl.S_ag)
        outs = [DevBuf(s.numel * ESZ[s.param_dtype], _offset(self.rng, ESZ[s.param_dtype])) for s in self.specs]
        fp.fsdp_allgather_copy_out(self.L, gathered.ptr, [b.ptr for b in outs])
        fp.fsdp_sync_status(self.L)
        rows = gathered.read()
        full = [b.read(NP[s.param_dtype]) for b, s in zip(outs, self.specs)]
        ok = gathered.guards_ok() and all(b.guards_ok() for b in outs + inputs)
        return rows, full, ok

    def gather_expected(self):
        rows = np.concatenate([oracle.allgather_copy_in(self.pl, self.shards[r]) for r in range(self.W)]) \
            if self.W * self.pl.S_ag else np.zeros(0, np.uint8)
        return rows, oracle.allgather_copy_out(self.pl, rows)


def first_mismatch(a: np.ndarray, b: np.ndarray) -> str:
    if a.shape != b.shape:
        return f"shape {a.shape} vs {b.shape}"
    bad = np.flatnonzero(a != b)
    if bad.size == 0:
        return "equal"
    i = int(bad[0])
    return f"{bad.size} mismatches, first at {i}: got {a[i]:#x} want {b[i]:#x}"


def assert_group_parity(fp, specs, W, work, group, misalign_seed=None, specials=0.0, rows=False):
    run = GroupRun(fp, specs, W, work, group, misalign_seed, specials, rows)
    try:
        got, ok = run.pack()
        assert ok, "guard bytes around pack buffers changed"
        for b, (x, y) in enumerate(zip(got, run.pack_expected())):
            assert np.array_equal(x, y), f"pack bucket {b}: {first_mismatch(x, y)}"
        got, ok = run.rs_copy_out()
        assert ok, "guard bytes around reduce-scatter copy-out buffers changed"
        for p, (x, y) in enumerate(zip(got, run.rs_copy_out_expected())):
            assert np.array_equal(x, y), f"rs copy-out param {p}: {first_mismatch(x, y)}"
        rows, full, ok = run.gather()
        assert ok, "guard bytes around all-gather buffers changed"
        want_rows, want_full = run.gather_expected()
        assert np.array_equal(rows, want_rows), f"copy-in: {first_mismatch(rows, want_rows)}"
        for p, (x, y) in enumerate(zip(full, want_full)):
            assert np.array_equal(x, y), f"copy-out param {p}: {first_mismatch(x, y)}"
    finally:
        run.close()


def fp_module():
    from fsdp2_gradient_packing_gb300 import fsdp_pack
    return fsdp_pack



def assert_batched_parity(fp, runs):
    """Push several GroupRuns through the batched entry points in single
    launches and compare every group's outputs with the oracle."""
    # Reduce-scatter copy-in: one launch for every group.
    g_bufs, outs, rhos = [], [], []
    for run in runs:
        g_bufs += [DevBuf(g.nbytes, _offset(run.rng, ESZ[s.grad_dtype]), g) for s, g in zip(run.specs, run.grads)]
        rho = ["f32" if d == oracle.F32 else "bf16" for d in run.pl.bucket_dtype]
        rhos.append(rho)
        outs.append([DevBuf(run.W * S * ESZ[r], _offset(run.rng, ESZ[r])) for r, S in zip(rho, run.pl.bucket_S)])
    fp.fsdp_pack_reduce_scatter_batched([run.L for run in runs], [b.ptr for b in g_bufs],
                                        [b.ptr for o in outs for b in o])
    fp.fsdp_sync_status(runs[0].L)
    for n, (run, out, rho) in enumerate(zip(runs, outs, rhos)):
        for b, (buf, want, r) in enumerate(zip(out, run.pack_expected(), rho)):
            got = buf.read(NP[r])
            assert np.array_equal(got, want), f"batched pack, group {n}, bucket {b}: {first_mismatch(got, want)}"
            assert buf.guards_ok()
    assert all(b.guards_ok() for b in g_bufs)
    # Reduce-scatter copy-out of every group in one launch.
    rows, sharded = [], []
    for run in runs:
        rho = ["f32" if d == oracle.F32 else "bf16" for d in run.pl.bucket_dtype]
        rows += [DevBuf(x.nbytes, _offset(run.rng, ESZ[r]), x) for x, r in zip(run.rows, rho)]
        sharded.append([DevBuf(c * ESZ[s.shard_dtype], _offset(run.rng, ESZ[s.shard_dtype]))
                        for s, c in zip(run.specs, run.pl.chunk)])
    fp.fsdp_reduce_scatter_copy_out_batched([run.L for run in runs], [b.ptr for b in rows],
                                            [b.ptr for sh in sharded for b in sh])
    fp.fsdp_sync_status(runs[0].L)
    for n, (run, sh) in enumerate(zip(runs, sharded)):
        for p, (buf, s, want) in enumerate(zip(sh, run.specs, run.rs_copy_out_expected())):
            got = buf.read(NP[s.shard_dtype])
            assert np.array_equal(got, want), f"batched rs copy-out, group {n} param {p}: {first_mismatch(got, want)}"
            assert buf.guards_ok()
    assert all(b.guards_ok() for b in rows)
    # All-gather copy-in, rank by rank (layouts with fewer ranks drop out),
    # then copy-out of every group in one launch.
    gathered = [DevBuf(run.W * run.pl.S_ag, 0) for run in runs]
    keep = []
    for r in range(max(run.W for run in runs)):
        sel = [k for k, run in enumerate(runs) if run.W > r]
        shards = []
        for k in sel:
            run = runs[k]
            bufs = [DevBuf(x.nbytes, _offset(run.rng, ESZ[s.shard_dtype]), x) for s, x in zip(run.specs, run.shards[r])]
            keep += bufs
            shards += [b.ptr for b in bufs]
        fp.fsdp_allgather_copy_in_batched([runs[k].L for k in sel], shards,
                                          [gathered[k].ptr + r * runs[k].pl.S_ag for k in sel])
    full = [[DevBuf(s.numel * ESZ[s.param_dtype], _offset(run.rng, ESZ[s.param_dtype])) for s in run.specs]
            for run in runs]
    fp.fsdp_allgather_copy_out_batched([run.L for run in runs], [g.ptr for g in gathered],
                                       [b.ptr for f in full for b in f])
    fp.fsdp_sync_status(runs[0].L)
    for n, run in enumerate(runs):
        want_rows, want_full = run.gather_expected()
        rows = gathered[n].read()
        assert np.array_equal(rows, want_rows), f"batched copy-in, group {n}: {first_mismatch(rows, want_rows)}"
        for p, (buf, s, want) in enumerate(zip(full[n], run.specs, want_full)):
            got = buf.read(NP[s.param_dtype])
            assert np.array_equal(got, want), f"batched copy-out, group {n} param {p}: {first_mismatch(got, want)}"
            assert buf.guards_ok()
        assert gathered[n].guards_ok()
    assert all(b.guards_ok() for b in keep)
