#!/usr/bin/env python3
"""Benchmark of the mixed-dtype FSDP buffer-packing path on GB300.

Workload: the 50.3M-element mixed group of the "FSDP2 per-parameter mixed
precision" news item's isolated packing test, as one fully_shard group at
W = 8 -- 4 layers at d = 1024 with BF16 q/k/v/o [1024, 1024], up [4096, 1024]
and down [1024, 4096] gradients (50,331,648 elements) and FP32 RMSNorm [1024]
x 2 per layer (8,192 elements); reduce dtype FP32; local shards FP32; param
dtype BF16 for the matrices and FP32 for the norms.  Values are seeded
N(0, 1) draws (synthetic: no dataset or trained weights exist for this).

One step is one pass of the whole hot path for that group on one GPU:
  1. reduce-scatter copy-in: pack every gradient into the [8, 6,292,480] FP32
     buffer (cast in flight, padding zeroed);
  2. all-gather copy-in of this rank's shards into its row of the gathered
     buffer (the other rows stand for what the all-gather brings in);
  3. all-gather copy-out of the gathered [8, S_ag] buffer into full params.
Nothing is communicated: W is a layout parameter.  With --gpus N (launched
by torchrun) every rank runs the same step on its own GPU with no collective
on the data path ("replicas"); the timing is the max over ranks.

Reported (one JSON line on rank 0): value = algorithmic bytes of all ranks'
steps / time (GB/s), per-operation device times from CUDA events, the
roofline of the dominant kernel (the pack), the SM clocks sampled during the
timed region, an end-to-end figure through the same API with host buffers,
and the CPU oracle timed on a bounded sample.  --impl reference times the
CPU oracle alone on bounded samples of the same workload.

Algorithmic bytes (reads count valid source elements, writes count every
destination slot including padding and alignment gaps):
  pack      sum_p n_p*size(g_p) + sum_b W*S_b*size(rho_b)
  copy-in   sum_p c_p*size(sigma_p) + S_ag
  copy-out  2 * sum_p n_p*size(pi_p)
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import shutil
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from fsdp2_gradient_packing_gb300 import workloads as wl  # noqa: E402

METRIC = "reduce-scatter pack GB/s and ms per fully_shard (50.3M elem, W=8) vs HBM peak"
UNIT = "GB/s"
NOMINAL_HBM_GBS = 8000.0   # the "~8 TB/s" HBM figure the metric is quoted against
FALLBACK_HBM_GBS = 6800.0  # used only when no measured copy bandwidth is available
CHUNKING = {False: "flattened: c_p = ceil(n_p / W)", True: "dim-0 rows: c_p = ceil(d0 / W) * row elements"}
ESZ = {"f32": 4, "bf16": 2}
STEP = "step = per group: reduce-scatter pack + all-gather copy-in (one rank) + all-gather copy-out"
STEP_RS = " + reduce-scatter copy-out (row 0 of each bucket as this rank's reduced row)"
STEP_ERS = " + emulated reduce-scatter after the pack (this rank's buckets + W-1 other ranks' buffers)"
WORKLOADS = {
    # name: (factory, description); the first is the benchmark's workload.
    "mixed50m": (lambda: wl.mixed_50m(W=8),
                 "mixed50m_W8: one fully_shard group of 4 layers at d=1024 (50,331,648 BF16 + 8,192 FP32 "
                 "gradients), W=8, reduce FP32, shards FP32, params BF16 matrices / FP32 norms"),
    "transformer500": (lambda: wl.transformer_500(W=8),
                       "transformer500_W8: 24 fully_shard groups (one per layer, d=512, 17 tensors each, "
                       "408 in all), W=8, reduce FP32, shards FP32, params BF16 matrices / FP32 small"),
    "transformer500_homogeneous": (lambda: wl.transformer_500(W=8, homogeneous=True),
                                   "transformer500_W8 with param dtype BF16 for every parameter (one all-gather "
                                   "dtype group): the homogeneous counterpart of transformer500"),
    "mixed50m_w12": (lambda: wl.mixed_50m(W=12),
                     "mixed50m_W12: the mixed50m group at W=12, which divides no matrix's dim 0 "
                     "(1024, 4096), so flattened and dim-0 row chunks differ"),
    "kda8": (lambda: wl.kda_block(W=8, reduce="f32", blocks=8),
             "kda8_W8: all 8 KDA-style blocks (1,744,929,024 parameters), one fully_shard group per block, W=8"),
    "kda8_homogeneous": (lambda: wl.kda_block(W=8, reduce="f32", blocks=8, homogeneous=True),
                         "kda8_W8 with param dtype BF16 for every parameter: the homogeneous counterpart of kda8"),
    "kda_w8": (lambda: wl.kda_block(W=8, reduce="f32"),
               "kda_block_W8: one KDA-style block at d=4096 (218,116,128 parameters), W=8, reduce FP32"),
    "kda_w64": (lambda: wl.kda_block(W=64, reduce="f32"),
                "kda_block_W64: one KDA-style block at d=4096 (218,116,128 parameters), W=64 (odd row "
                "length: every row misaligned), reduce FP32"),
    "kda_w8_grad": (lambda: wl.kda_block(W=8, reduce="grad"),
                    "kda_block_W8_two_buckets: one KDA-style block, W=8, reduce dtype = gradient dtype "
                    "(BF16 and FP32 buckets)"),
}
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "pack_mixed50m_w8_ncu.md")


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU work of the oracle baseline sample (rank 0, N=1)")
    ap.add_argument("--e2e-steps", type=int, default=30,
                    help="timed end-to-end steps (0: skip the end-to-end pass, e.g. for layouts too large to "
                         "stage in pinned host memory twice)")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="mixed50m",
                    help="layout to time (the benchmark's metric is quoted on mixed50m)")
    ap.add_argument("--rs-copy-out", action="store_true",
                    help="add the reduce-scatter copy-out (reduced rows to sharded gradients) to every step")
    ap.add_argument("--emulated-rs", action="store_true",
                    help="add the emulated reduce-scatter (sum of W ranks' packed buffers) after the pack")
    ap.add_argument("--precast-iters", type=int, default=200,
                    help="iterations of the pre-cast-then-pack comparison (0 = skip)")
    ap.add_argument("--row-chunks", action="store_true",
                    help="plan every parameter by dim-0 rows (c_p = ceil(d0 / W) rows) instead of flattened")
    ap.add_argument("--graph", action="store_true",
                    help="time the step as replays of a CUDA graph holding two steps (both buffer sets)")
    ap.add_argument("--batched", action="store_true",
                    help="one launch per operation for all of the workload's groups (*_batched entry points)")
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------
# Distributed plumbing (replicas only: a barrier and a max, no data exchange).
# ---------------------------------------------------------------------------
def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def init_dist(backend: str):
    import torch.distributed as dist
    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend, rank=rank, world_size=world)
    return world


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    """The largest x over all ranks (x itself without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# Workload sizes.
# ---------------------------------------------------------------------------
def row_elems(specs):
    """Elements of one dim-0 row of each parameter (1 for 1-D parameters)."""
    return [math.prod(s.shape[1:]) if len(s.shape) > 1 else 1 for s in specs]


def chunks(specs, W, rows=False):
    """c_p of every parameter: ceil(n_p / W) of the flattened parameter, or
    with ``rows`` ceil(d0 / W) whole dim-0 rows."""
    if not rows:
        return [-(-s.numel // W) for s in specs]
    return [(-(-s.shape[0] // W) * r if s.numel else 0) for s, r in zip(specs, row_elems(specs))]


def op_bytes(specs, W, bucket_bytes, S_ag, rows=False):
    c = chunks(specs, W, rows)
    pack = sum(s.numel * ESZ[s.grad_dtype] for s in specs) + sum(bucket_bytes)
    copy_in = sum(ci * ESZ[s.shard_dtype] for ci, s in zip(c, specs)) + S_ag
    copy_out = 2 * sum(s.numel * ESZ[s.param_dtype] for s in specs)
    rs_copy_out = sum(ci * (ESZ[s.reduce_dtype] + ESZ[s.shard_dtype]) for ci, s in zip(c, specs))
    emulated_rs = (W + 1) * sum(bucket_bytes)   # W packed buffers read, one reduced buffer written
    return {"pack": pack, "copy_in": copy_in, "copy_out": copy_out, "rs_copy_out": rs_copy_out,
            "emulated_rs": emulated_rs}


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    """Hash of the kernel and planner sources with comments and whitespace
    removed, so that only a change of code invalidates a profile."""
    import re
    h = hashlib.sha256()
    for rel in ("fsdp2_gradient_packing_gb300/csrc/kernels.cu", "fsdp2_gradient_packing_gb300/csrc/layout.h",
                "fsdp2_gradient_packing_gb300/csrc/plan.cpp"):
        with open(os.path.join(ROOT, rel)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update("".join(text.split()).encode())
    return h.hexdigest()[:16]


def read_traffic():
    """DRAM bytes per pack launch from the committed ncu summary, if it was
    taken on the current kernel source (else None)."""
    try:
        text = open(PROFILE_SUMMARY).read()
    except OSError:
        return None
    fields = {}
    for line in text.splitlines():
        line = line.strip().strip("`")
        if ":" in line:
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    if fields.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    try:
        return int(fields["dram_bytes_per_pack_launch"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
# Clocks during the timed region.
# ---------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.file = None

    def start(self):
        exe = shutil.which("nvidia-smi")
        if not exe:
            return
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        cmd = [exe, f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        self.proc = subprocess.Popen(cmd, stdout=self.file, stderr=subprocess.DEVNULL)

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            self.proc.wait()
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.count(",") >= 6]
        self.file.close()
        os.unlink(self.file.name)
        sm, mx, pw, reasons = [], [], [], set()
        for r in rows:
            try:
                sm.append(float(r[0]))
                mx.append(float(r[1]))
                pw.append(float(r[2]))
            except ValueError:
                continue
            for name, v in zip(self.REASONS, r[3:7]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(pw) if pw else None}


# ---------------------------------------------------------------------------
# Host inputs (seeded), packed into flat byte buffers with aligned offsets.
# ---------------------------------------------------------------------------
def flat_offsets(sizes, align=256):
    offs, at = [], 0
    for n in sizes:
        offs.append(at)
        at += -(-n // align) * align
    return offs, max(at, align)


def host_inputs(work, g, rows=False):
    """Seeded gradients and every rank's shards of group g."""
    specs, W = work.groups[g], work.W
    c = chunks(specs, W, rows)
    grads = [wl.grad_values(work, g, i) for i in range(len(specs))]
    shards = [[wl.shard_values(work, g, i, r, c[i], max(0, min(c[i], s.numel - r * c[i])))
               for i, s in enumerate(specs)] for r in range(W)]
    return grads, shards


def flatten(arrays, offs, total):
    out = np.zeros(total, np.uint8)
    for a, o in zip(arrays, offs):
        b = a.view(np.uint8)
        out[o:o + b.size] = b
    return out


# ---------------------------------------------------------------------------
# The CPU oracle on bounded samples: one (rank, parameter) run at a time.
# ---------------------------------------------------------------------------
class OracleSampler:
    """Cycles through the segments of one step of the path over every group
    (pack runs, copy-in runs of rank 0, copy-out runs), each with its
    algorithmic bytes."""

    def __init__(self, work, inputs, rows=False):
        import oracle
        self.oracle = oracle
        W = work.W
        self.segs = []
        for g, specs in enumerate(work.groups):
            grads, shards = inputs[g]
            pl = oracle.plan(oracle.params_from_specs(specs), W, row_elems=row_elems(specs) if rows else None)
            st = {
                "pl": pl, "grads": grads, "shards0": shards[0],
                "bufs": [np.empty(W * S, oracle.DTYPE_NP[d]) for d, S in zip(pl.bucket_dtype, pl.bucket_S)],
                "row": np.empty(pl.S_ag, np.uint8),
                "gathered": np.concatenate([oracle.allgather_copy_in(pl, shards[r]) for r in range(W)]),
                "full": [np.empty(p.numel, oracle.DTYPE_NP[p.param_dtype]) for p in pl.params],
            }
            sz = oracle.DTYPE_SIZE
            for b in range(len(pl.bucket_dtype)):
                for r in range(W):
                    for p, prm in enumerate(pl.params):
                        if pl.bucket_of[p] != b:
                            continue
                        valid = max(0, min(pl.chunk[p], prm.numel - r * pl.chunk[p]))
                        nbytes = valid * sz[prm.grad_dtype] + pl.chunk[p] * sz[pl.bucket_dtype[b]]
                        self.segs.append((self._pack, (st, r, p), nbytes))
            gap = pl.S_ag - sum(c * sz[p.param_dtype] for c, p in zip(pl.chunk, pl.params))
            self.segs.append((self._clear, (st,), gap))
            for p, prm in enumerate(pl.params):
                self.segs.append((self._copy_in, (st, p), pl.chunk[p] * (sz[prm.shard_dtype] + sz[prm.param_dtype])))
            for p, prm in enumerate(pl.params):
                for r in range(W):
                    valid = max(0, min(pl.chunk[p], prm.numel - r * pl.chunk[p]))
                    self.segs.append((self._copy_out, (st, p, r), 2 * valid * sz[prm.param_dtype]))
        self.step_bytes = sum(s[2] for s in self.segs)
        self.i = 0

    def _pack(self, st, r, p):
        self.oracle.pack_segment(st["pl"], st["grads"], st["bufs"], r, p)

    def _clear(self, st):
        self.oracle.allgather_copy_in_clear(st["pl"], st["row"])

    def _copy_in(self, st, p):
        self.oracle.allgather_copy_in_segment(st["pl"], st["shards0"], st["row"], p)

    def _copy_out(self, st, p, r):
        self.oracle.allgather_copy_out_segment(st["pl"], st["gathered"], st["full"], p, r)

    def next(self) -> int:
        fn, args, nbytes = self.segs[self.i]
        self.i = (self.i + 1) % len(self.segs)
        fn(*args)
        return nbytes


def host_cpu() -> dict:
    """The host the CPU legs run on: logical CPUs and the CPU model as
    /proc/cpuinfo names it (Arm hosts give implementer and part numbers)."""
    model = None
    try:
        fields = {}
        for line in open("/proc/cpuinfo"):
            if ":" in line:
                k, v = line.split(":", 1)
                fields.setdefault(k.strip(), v.strip())
        model = fields.get("model name") or (
            f"implementer {fields['CPU implementer']} part {fields['CPU part']}"
            if "CPU implementer" in fields and "CPU part" in fields else None)
    except OSError:
        pass
    import platform
    return {"host_cpus": os.cpu_count(), "cpu_model": model, "machine": platform.machine(),
            "threads_used": 1}


def cpu_baseline(sampler: OracleSampler, seconds: float) -> dict:
    """Whole steps of the oracle (all segments in order) for about `seconds`."""
    done_bytes, steps = 0, 0
    t0 = time.perf_counter()
    while True:
        for _ in range(len(sampler.segs)):
            done_bytes += sampler.next()
        steps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": done_bytes / dt / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{steps} whole step(s) of the same workload (pack, copy-in of one rank, copy-out), "
                      f"single-threaded C oracle, {dt:.1f} s", **host_cpu()}


# ---------------------------------------------------------------------------
# Our arm.
# ---------------------------------------------------------------------------
class DeviceSet:
    """One complete set of device buffers for a step (two sets rotate)."""

    def __init__(self, fp, torch, L, specs, W, info, host_grads, host_shards, rank_row, others=None, rows=False):
        dev = torch.device("cuda")
        c = chunks(specs, W, rows)
        self.S_ag = info.ag_bytes
        g_sizes = [s.numel * ESZ[s.grad_dtype] for s in specs]
        goffs, gtot = flat_offsets(g_sizes)
        self.grads = torch.from_numpy(flatten(host_grads, goffs, gtot)).to(dev)
        self.grad_ptrs = fp.pointer_array([self.grads.data_ptr() + o for o in goffs])
        self.buckets = [torch.empty(fp.fsdp_layout_bucket(L, b).bytes, dtype=torch.uint8, device=dev)
                        for b in range(info.n_buckets)]
        self.bucket_ptrs = fp.pointer_array(self.buckets)
        s_sizes = [ci * ESZ[s.shard_dtype] for ci, s in zip(c, specs)]
        soffs, stot = flat_offsets(s_sizes)
        self.shard_offs, self.shard_tot = soffs, stot
        self.shards = torch.from_numpy(flatten(host_shards[rank_row], soffs, stot)).to(dev)
        self.shard_ptrs = fp.pointer_array([self.shards.data_ptr() + o for o in soffs])
        self.gathered = torch.empty(W * self.S_ag, dtype=torch.uint8, device=dev)
        self.row_ptr = self.gathered.data_ptr() + rank_row * self.S_ag
        f_sizes = [s.numel * ESZ[s.param_dtype] for s in specs]
        foffs, ftot = flat_offsets(f_sizes)
        self.full = torch.empty(ftot, dtype=torch.uint8, device=dev)
        self.full_ptrs = fp.pointer_array([self.full.data_ptr() + o for o in foffs])
        # Emulated reduce-scatter: this rank's buckets plus the other W - 1
        # ranks' buffers (`others[b]`, shared by both sets) summed into
        # `reduced`; the reduce-scatter copy-out then reads row 0 of it.
        self.reduced = None
        if others is not None:
            self.reduced = [torch.empty_like(b) for b in self.buckets]
            self.packed_ptrs = fp.pointer_array([p for b, mine in enumerate(self.buckets)
                                                 for p in [mine.data_ptr()] + [o.data_ptr() for o in others[b]]])
            self.reduced_ptrs = fp.pointer_array(self.reduced)
        # Reduce-scatter copy-out: row 0 of each bucket (or of the reduced
        # buffer) stands for this rank's reduced row; the sharded gradients
        # go to their own buffer.
        self.row0_ptrs = fp.pointer_array([b.data_ptr() for b in (self.reduced or self.buckets)])
        h_sizes = [ci * ESZ[s.shard_dtype] for ci, s in zip(c, specs)]
        hoffs, htot = flat_offsets(h_sizes)
        self.sharded = torch.empty(htot, dtype=torch.uint8, device=dev)
        self.sharded_ptrs = fp.pointer_array([self.sharded.data_ptr() + o for o in hoffs])
        # The other ranks' rows: what the all-gather would deliver.
        for r in range(W):
            if r == rank_row:
                continue
            other = torch.from_numpy(flatten(host_shards[r], soffs, stot)).to(dev)
            fp.fsdp_allgather_copy_in(L, [other.data_ptr() + o for o in soffs],
                                      self.gathered.data_ptr() + r * self.S_ag)
            torch.cuda.synchronize()
            del other

    def step(self, fp, L, h, ev=None, rs=False):
        """pack, [emulated reduce-scatter], copy-in, copy-out, [rs copy-out];
        ev[k] is recorded after the k-th launch (ev[0] before the first)."""
        k = 0

        def mark():
            nonlocal k
            if ev is not None:
                ev[k].record()
            k += 1
        mark()
        fp.fsdp_pack_reduce_scatter(L, self.grad_ptrs, self.bucket_ptrs, h)
        mark()
        if self.reduced is not None:
            fp.fsdp_emulated_reduce_scatter(L, self.packed_ptrs, self.reduced_ptrs, h)
            mark()
        fp.fsdp_allgather_copy_in(L, self.shard_ptrs, self.row_ptr, h)
        mark()
        fp.fsdp_allgather_copy_out(L, self.gathered.data_ptr(), self.full_ptrs, h)
        mark()
        if rs:
            fp.fsdp_reduce_scatter_copy_out(L, self.row0_ptrs, self.sharded_ptrs, h)
            mark()


class Group:
    """One fully_shard group on the device: its layout and two buffer sets."""

    def __init__(self, fp, torch, work, g, inputs, emulated_rs=False, rows=False):
        self.specs = work.groups[g]
        self.L = (fp.fsdp_plan_layout_ex(self.specs, work.W, row_elems(self.specs)) if rows
                  else fp.fsdp_plan_layout(self.specs, work.W))
        self.info = fp.fsdp_layout_query(self.L)
        bucket_bytes = [fp.fsdp_layout_bucket(self.L, b).bytes for b in range(self.info.n_buckets)]
        self.nbytes = op_bytes(self.specs, work.W, bucket_bytes, self.info.ag_bytes, rows)
        grads, shards = inputs
        others = None
        if emulated_rs:   # the other ranks' packed buffers (contents do not matter for timing)
            others = [[torch.zeros(n, dtype=torch.uint8, device="cuda") for _ in range(work.W - 1)]
                      for n in bucket_bytes]
        self.sets = [DeviceSet(fp, torch, self.L, self.specs, work.W, self.info, grads, shards, 0, others, rows)
                     for _ in range(2)]


class Batch:
    """The pointer arrays of the batched entry points for both buffer sets."""

    def __init__(self, fp, groups):
        self.layouts = fp.layout_array([grp.L for grp in groups])
        self.n = len(groups)
        cat = lambda arrs: fp.pointer_array([p for a in arrs for p in a])  # noqa: E731
        self.sets = []
        for k in range(2):
            ss = [grp.sets[k] for grp in groups]
            self.sets.append(dict(
                grads=cat(s.grad_ptrs for s in ss), buckets=cat(s.bucket_ptrs for s in ss),
                shards=cat(s.shard_ptrs for s in ss), rows=fp.pointer_array([s.row_ptr for s in ss]),
                gathered=fp.pointer_array([s.gathered.data_ptr() for s in ss]), full=cat(s.full_ptrs for s in ss),
                row0=cat(s.row0_ptrs for s in ss), sharded=cat(s.sharded_ptrs for s in ss)))

    def step(self, fp, h, k, ev=None, rs=False):
        a = self.sets[k]
        if ev is not None:
            ev[0].record()
        fp.fsdp_pack_reduce_scatter_batched(self.layouts, a["grads"], a["buckets"], h)
        if ev is not None:
            ev[1].record()
        fp.fsdp_allgather_copy_in_batched(self.layouts, a["shards"], a["rows"], h)
        if ev is not None:
            ev[2].record()
        fp.fsdp_allgather_copy_out_batched(self.layouts, a["gathered"], a["full"], h)
        if ev is not None:
            ev[3].record()
        if rs:
            fp.fsdp_reduce_scatter_copy_out_batched(self.layouts, a["row0"], a["sharded"], h)
            if ev is not None:
                ev[4].record()


def precast_comparison(fp, torch, work, grp, h, iters, rows=False):
    """The sequence the fused pack replaces: every BF16 gradient that reduces in
    FP32 is first cast into one FP32 temporary, then an FP32 -> FP32 pack reads
    the temporary ("FSDP2 per-parameter mixed precision", results table:
    copy-in with the cast fused against a separate pre-cast).  Both steps run
    on this library's own kernel: the cast is a pack on a one-rank layout (one
    bucket, c_p = n_p, no padding: a plain cast and concatenation).  The
    temporary is allocated once, as a caching allocator would hand it back.
    Timed as a loop of (cast, pack) pairs beside a loop of the fused pack alone,
    both alternating the two buffer sets, CUDA events on the launching stream."""
    import dataclasses
    specs = grp.specs
    cast_idx = [i for i, s in enumerate(specs) if s.grad_dtype == "bf16" and s.reduce_dtype == "f32"]
    if not cast_idx or iters <= 0:
        return None
    cast_specs = [dataclasses.replace(specs[i], reduce_dtype="f32") for i in cast_idx]
    fp32_specs = [dataclasses.replace(s, grad_dtype="f32") if i in set(cast_idx) else s
                  for i, s in enumerate(specs)]
    L32 = (fp.fsdp_plan_layout_ex(fp32_specs, work.W, row_elems(fp32_specs)) if rows
           else fp.fsdp_plan_layout(fp32_specs, work.W))
    with fp.fsdp_plan_layout(cast_specs, 1) as L_cast, L32:
        tmp_bytes = fp.fsdp_layout_bucket(L_cast, 0).bytes
        tmp = torch.empty(tmp_bytes, dtype=torch.uint8, device="cuda")
        offs = {i: fp.fsdp_layout_param(L_cast, k).bucket_offset * 4 for k, i in enumerate(cast_idx)}
        args = []
        for st in grp.sets:
            cast_src = fp.pointer_array([st.grad_ptrs[i] for i in cast_idx])
            tmp_dst = fp.pointer_array([tmp.data_ptr()])
            grads32 = fp.pointer_array([tmp.data_ptr() + offs[i] if i in offs else st.grad_ptrs[i]
                                        for i in range(len(specs))])
            args.append((cast_src, tmp_dst, grads32, st.bucket_ptrs, st.grad_ptrs))

        def precast(k):
            a = args[k & 1]
            fp.fsdp_pack_reduce_scatter(L_cast, a[0], a[1], h)
            fp.fsdp_pack_reduce_scatter(L32, a[2], a[3], h)

        def fused(k):
            a = args[k & 1]
            fp.fsdp_pack_reduce_scatter(grp.L, a[4], a[3], h)

        def loop(fn):
            for k in range(10):
                fn(k)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record()
            for k in range(iters):
                fn(k)
            e1.record()
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / iters

        pre_ms, fused_ms = loop(precast), loop(fused)
        for L in (L_cast, L32, grp.L):
            fp.fsdp_sync_status(L)
        bucket_bytes = [fp.fsdp_layout_bucket(L32, b).bytes for b in range(fp.fsdp_layout_query(L32).n_buckets)]
        pre_bytes = (op_bytes(cast_specs, 1, [tmp_bytes], 0)["pack"]
                     + op_bytes(fp32_specs, work.W, bucket_bytes, 0, rows)["pack"])
        del tmp
    return {"what": "BF16 gradients cast into one FP32 temporary, then the FP32 -> FP32 pack, "
                    "against the fused pack; back-to-back loops of " + str(iters),
            "temporary_bytes": tmp_bytes, "precast_ms": pre_ms, "fused_ms": fused_ms,
            "precast_over_fused": pre_ms / fused_ms, "precast_bytes": pre_bytes,
            "precast_gbs": pre_bytes / (pre_ms * 1e-3) / 1e9, "launches": 2 * iters + iters}


def run_steps(fp, groups, h, first, count, evs=None, batch=None, rs=False):
    for i in range(first, first + count):
        if batch is not None:
            batch.step(fp, h, i & 1, None if evs is None else evs[i - first][0], rs)
            continue
        for gi, grp in enumerate(groups):
            grp.sets[i & 1].step(fp, grp.L, h, None if evs is None else evs[i - first][gi], rs)


def run_ours(args):
    import torch
    from fsdp2_gradient_packing_gb300 import _build
    _build.build()
    from fsdp2_gradient_packing_gb300 import fsdp_pack as fp

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    init_dist("nccl" if world > 1 else "gloo")
    factory, description = WORKLOADS[args.workload]
    work = factory()
    rows = args.row_chunks
    inputs = [host_inputs(work, g, rows) for g in range(len(work.groups))]
    groups = [Group(fp, torch, work, g, inputs[g], args.emulated_rs, rows) for g in range(len(work.groups))]
    if args.batched and args.emulated_rs:
        raise SystemExit("--emulated-rs has no batched form; drop --batched")
    OPS = (("pack",) + (("emulated_rs",) if args.emulated_rs else ()) + ("copy_in", "copy_out")
           + (("rs_copy_out",) if args.rs_copy_out else ()))
    nbytes = {k: sum(grp.nbytes[k] for grp in groups) for k in OPS}
    step_bytes = sum(nbytes.values())
    h = torch.cuda.current_stream().cuda_stream
    batch = Batch(fp, groups) if args.batched else None
    n_launch = 1 if batch is not None else len(groups)
    rs = args.rs_copy_out
    run_steps(fp, groups, h, 0, args.warmup, batch=batch, rs=rs)
    for grp in groups:
        fp.fsdp_sync_status(grp.L)

    K = args.steps
    graph = None
    if args.graph:
        # Two steps (buffer sets 0 and 1) captured once and replayed K / 2
        # times: the layers' launches go to the GPU without host involvement.
        K += K & 1
        graph = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(graph):
            run_steps(fp, groups, torch.cuda.current_stream().cuda_stream, 0, 2, batch=batch, rs=rs)
        for _ in range(max(1, args.warmup // 2)):
            graph.replay()
        torch.cuda.synchronize()
        for grp in groups:
            fp.fsdp_sync_status(grp.L)
    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:
        pass
    # Pass 1: the timed region proper.  Launches follow each other with
    # nothing in between, as in a training step.
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(gpu_id)
    torch.cuda.synchronize()
    barrier()
    sampler.start()
    time.sleep(0.3)  # let the sampler take its first sample before the load starts
    t_start.record()
    if graph is not None:
        for _ in range(K // 2):
            graph.replay()
    else:
        run_steps(fp, groups, h, 0, K, batch=batch, rs=rs)
    t_end.record()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    barrier()
    for grp in groups:
        fp.fsdp_sync_status(grp.L)
    total_ms = max_over_ranks(t_start.elapsed_time(t_end), device=torch.device("cuda"))

    # Pass 2: the same K steps with a CUDA event around every launch, for the
    # per-operation device times (events between launches serialise them).
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(len(OPS) + 1)] for _ in range(n_launch)]
           for _ in range(K)]
    torch.cuda.synchronize()
    barrier()
    run_steps(fp, groups, h, 0, K, evs, batch=batch, rs=rs)
    torch.cuda.synchronize()
    barrier()
    for grp in groups:
        fp.fsdp_sync_status(grp.L)
    per = {k: [sum(e[j].elapsed_time(e[j + 1]) for e in step) for step in evs] for j, k in enumerate(OPS)}

    precast = None
    if len(groups) == 1 and args.precast_iters > 0:
        precast = precast_comparison(fp, torch, work, groups[0], h, args.precast_iters, rows)

    e2e = None
    if args.e2e_steps > 0:
        e2e = run_e2e(args, fp, torch, groups, h, rs, step_bytes, world)

    result = None
    if rank == 0:
        result = report(args, work, description, groups, nbytes, step_bytes, total_ms, per, clocks, e2e,
                        n_launch, rs, world, K)
        if precast is not None:
            result["precast_baseline"] = precast
    for grp in groups:
        grp.L.close()
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        samp = OracleSampler(work, inputs, rows)
        result["cpu_baseline"] = cpu_baseline(samp, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(result), flush=True)
    import torch.distributed as dist
    if dist.is_initialized():
        dist.destroy_process_group()


def run_e2e(args, fp, torch, groups, h, rs, step_bytes, world):
    # End to end through the same API with host buffers: every step copies
    # its inputs from pinned host memory and reads its results back.  Steps
    # are pipelined the way a caller would run them: uploads on one stream,
    # the kernels on another, downloads on a third, two buffer sets, so step
    # i+1's uploads overlap step i's downloads.
    pin = lambda n: torch.empty(n, dtype=torch.uint8, pin_memory=True)  # noqa: E731
    host = []
    for grp in groups:
        s0 = grp.sets[0]
        hb = {"grads": pin(s0.grads.numel()), "shards": pin(s0.shards.numel()),
              "others": pin(s0.gathered.numel() - s0.S_ag),
              "out": [{"buckets": [pin(b.numel()) for b in s0.buckets], "full": pin(s0.full.numel()),
                       "sharded": pin(s0.sharded.numel()) if rs else None} for _ in range(2)]}
        hb["grads"].copy_(s0.grads.cpu())
        hb["shards"].copy_(s0.shards.cpu())
        hb["others"].copy_(s0.gathered[s0.S_ag:].cpu())
        host.append(hb)
    h2d = sum(hb["grads"].numel() + hb["shards"].numel() + hb["others"].numel() for hb in host)
    d2h = sum(sum(b.numel() for b in hb["out"][0]["buckets"]) + hb["out"][0]["full"].numel()
              + (hb["out"][0]["sharded"].numel() if rs else 0) for hb in host)
    E = max(3, args.e2e_steps)
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    main = torch.cuda.current_stream()

    def e2e_steps(n):
        uploaded = [torch.cuda.Event() for _ in range(2)]
        computed = [torch.cuda.Event() for _ in range(2)]
        downloaded = [torch.cuda.Event() for _ in range(2)]
        up.wait_stream(main)
        down.wait_stream(main)
        for i in range(n):
            k = i & 1
            with torch.cuda.stream(up):
                if i >= 2:
                    up.wait_event(downloaded[k])           # set k's outputs of step i-2 are home
                for grp, hb in zip(groups, host):
                    sk = grp.sets[k]
                    sk.grads.copy_(hb["grads"], non_blocking=True)
                    sk.shards.copy_(hb["shards"], non_blocking=True)
                    sk.gathered[sk.S_ag:].copy_(hb["others"], non_blocking=True)
                uploaded[k].record(up)
            main.wait_event(uploaded[k])
            for grp in groups:
                grp.sets[k].step(fp, grp.L, h, None, rs)
            computed[k].record(main)
            with torch.cuda.stream(down):
                down.wait_event(computed[k])
                for grp, hb in zip(groups, host):
                    sk, ho = grp.sets[k], hb["out"][k]
                    for hbuf, dbuf in zip(ho["buckets"], sk.buckets):
                        hbuf.copy_(dbuf, non_blocking=True)
                    ho["full"].copy_(sk.full, non_blocking=True)
                    if rs:
                        ho["sharded"].copy_(sk.sharded, non_blocking=True)
                downloaded[k].record(down)
        main.wait_stream(up)
        main.wait_stream(down)

    e2e_steps(max(4, args.warmup))     # untimed: touches every pinned buffer of both sets
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier()
    e_start.record(main)
    e2e_steps(E)
    e_end.record(main)
    torch.cuda.synchronize()
    barrier()
    for grp in groups:
        fp.fsdp_sync_status(grp.L)
    e2e_ms = max_over_ranks(e_start.elapsed_time(e_end), device=torch.device("cuda"))
    return {"value": world * step_bytes * E / (e2e_ms * 1e-3) / 1e9, "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": E,
            "note": "host buffers; uploads, kernels and downloads of consecutive steps pipelined "
                    "on three streams with two buffer sets"}


def report(args, work, description, groups, nbytes, step_bytes, total_ms, per, clocks, e2e, n_launch, rs,
           world, K):
    """The JSON result of our arm (rank 0)."""
    peak, peak_kind = read_peaks()
    pack_ms = statistics.mean(per["pack"])
    achieved = nbytes["pack"] / (pack_ms * 1e-3) / 1e9
    rows = {k: {"bytes": nbytes[k], "launches_per_step": n_launch, "ms_mean": statistics.mean(v),
                "ms_median": statistics.median(v), "ms_min": min(v),
                "gbs": nbytes[k] / (statistics.mean(v) * 1e-3) / 1e9}
            for k, v in per.items()}
    result = {
        "metric": METRIC,
        "value": world * step_bytes * K / (total_ms * 1e-3) / 1e9,
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": total_ms / K,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16+f32",
        "data": "synthetic",
        "config": {"workload": f"{description}; {STEP}" + (STEP_RS if rs else "")
                   + (STEP_ERS if args.emulated_rs else ""), "world_size_layout": work.W,
                   "chunking": CHUNKING[args.row_chunks],
                   "groups": len(groups), "launches_per_op": n_launch, "step_bytes": step_bytes,
                   "launch": ("CUDA graph of two steps, replayed" if args.graph
                              else "stream launches from the host") + (", batched over groups" if args.batched else ""),
                   "parallelism": f"replicas x{world} (no data-path collective)",
                   "l2": "inputs larger than L2: two rotating buffer sets of "
                         f"{2 * step_bytes / 1e9:.2f} GB of algorithmic traffic vs 129 MB L2; no flush"},
        "ops": rows,
        "ops_note": "per-operation device times from a second pass of the same K steps with CUDA "
                    "events around every launch (summed over the step's groups)",
        "roofline": {"bound": "hbm", "kernel": "walk_kernel (reduce-scatter pack launches)",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
                     "peak_source": f"{peak_kind} hbm_gbs (burst copy)" if peak_kind == "measured" else "fallback",
                     "bytes_per_launch": nbytes["pack"] / n_launch,
                     "traffic": read_traffic() if args.workload == "mixed50m" else None},
        "e2e": e2e,
        "gpu_launches": len(per) * n_launch * K,
        "clocks": clocks,
    }
    return result


# ---------------------------------------------------------------------------
# Reference arm: the CPU oracle, each step one bounded segment of the step.
# ---------------------------------------------------------------------------
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    factory, description = WORKLOADS[args.workload]
    work = factory()
    inputs = [host_inputs(work, g, args.row_chunks) for g in range(len(work.groups))]
    samp = OracleSampler(work, inputs, args.row_chunks)
    for _ in range(args.warmup):
        samp.next()
    done = 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        done += samp.next()
    dt = time.perf_counter() - t0
    value = done / dt / 1e9
    result = {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt * 1e3 / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16+f32", "data": "synthetic",
        "config": {"workload": f"{description}; {STEP}", "world_size_layout": work.W,
                   "chunking": CHUNKING[args.row_chunks],
                   "groups": len(work.groups), "step_bytes": samp.step_bytes, "parallelism": "single host thread"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": "each step = one (rank, parameter) run of the pack, copy-in or copy-out, "
                                   f"cycling through the {len(samp.segs)} runs of a whole step", **host_cpu()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(result), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
