#!/usr/bin/env python3
"""Benchmark of the mixed-dtype FSDP buffer-packing path on GB300.

Workload: the 50.3M-element mixed group of the "FSDP2 per-parameter mixed
precision" news item's isolated packing test, as one fully_shard group at
W = 8 -- 4 layers at d = 1024 with BF16 q/k/v/o [1024, 1024], up [4096, 1024]
and down [1024, 4096] gradients (50,331,648 elements) and FP32 RMSNorm [1024]
x 2 per layer (8,192 elements); reduce dtype FP32; local shards FP32; param
dtype BF16 for the matrices and FP32 for the norms.  Values are seeded
N(0, 1) draws (synthetic: no dataset or trained weights exist for this).

The metric is the reduce-scatter pack of that group, the step the news
item times in isolation: gradients -> the [8, 6,292,480] FP32 buffer, cast
in flight, padding zeroed.  The timed region is K packs back to back on one
stream, alternating two buffer sets (each larger than L2), with no event or
host synchronisation between launches; `value` is the pack's algorithmic
bytes over that time and `ms_per_step` the time of one pack.  Also reported:
  * hot_path_step: the whole path per group -- pack, all-gather copy-in of one
    rank (the other rows stand for what the all-gather brings in), all-gather
    copy-out -- timed the same way;
  * ops: per-operation device times from a pass with CUDA events around
    every launch (events serialise the launches);
  * roofline of the pack against the measured copy bandwidth and against a
    plain 1:2 streaming widen of the same bytes run in the same process;
  * e2e: the pack through the same C-ABI call with pinned host buffers (the
    gradients uploaded and the bucket downloaded every step);
  * extra_workloads: the ~500-parameter transformer layout (24 groups, one
    launch per operation) and one KDA-style block at W = 64;
  * cpu_baseline: the CPU oracle's pack on a bounded sample.
Nothing is communicated: W is a layout parameter.  With --gpus N (launched
by torchrun) every rank runs the same work on its own GPU with no collective
on the data path ("replicas"); the timing is the max over ranks.
--impl reference times the CPU oracle's pack alone on bounded samples of the
same workload.

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
STEP = "per group: reduce-scatter pack + all-gather copy-in (one rank) + all-gather copy-out"
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
# Counters of one ncu capture of the pack on mixed50m (written by hand from the
# capture; see the .md summary of the same name for the command and the reading).
PROFILE_COUNTERS = os.path.join(ROOT, "profiles", "pack_mixed50m_w8_ncu.json")


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
                    help="time packs and steps as replays of CUDA graphs holding two of each (both buffer sets)")
    ap.add_argument("--batched", action="store_true",
                    help="one launch per operation for all of the workload's groups (*_batched entry points)")
    ap.add_argument("--evented-steps", type=int, default=2000,
                    help="whole steps of the pass with CUDA events around every launch (per-operation times)")
    ap.add_argument("--reference-iters", type=int, default=400,
                    help="iterations of the same-run plain copies of the pack's bytes (0 = skip)")
    ap.add_argument("--op-seconds", type=float, default=0.2,
                    help="seconds of back-to-back launches per operation for ops_alone (0 = skip)")
    ap.add_argument("--no-extra", dest="extra", action="store_false",
                    help="skip the extra workloads (transformer layout batched, one KDA block at W = 64)")
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
    """Hash of the sources the table-walking kernel and its planner are built
    from, with comments and whitespace removed, so that only a change of
    their code invalidates a profile (reduce.cu, the emulated
    reduce-scatter, is not among them)."""
    import re
    h = hashlib.sha256()
    for rel in ("fsdp2_gradient_packing_gb300/csrc/kernels.cu", "fsdp2_gradient_packing_gb300/csrc/bf16_bits.h",
                "fsdp2_gradient_packing_gb300/csrc/layout.h", "fsdp2_gradient_packing_gb300/csrc/plan.cpp"):
        with open(os.path.join(ROOT, rel)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update("".join(text.split()).encode())
    return h.hexdigest()[:16]


def read_traffic():
    """DRAM and L2 write bytes of one pack launch from the committed ncu
    counters, if they were taken on the current kernel source (else None)."""
    try:
        with open(PROFILE_COUNTERS) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    try:
        rd, wr = int(d["dram__bytes_read.sum"]), int(d["dram__bytes_write.sum"])
        l2w = int(d["lts__t_sectors_srcunit_tex_op_write.sum"]) * 32
    except (KeyError, ValueError, TypeError):
        return None
    return {"traffic": rd + wr, "traffic_dram_read": rd, "traffic_dram_write": wr, "traffic_l2_write": l2w,
            "traffic_source": os.path.relpath(PROFILE_COUNTERS, ROOT)}


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
# Inputs (seeded), packed into flat byte buffers with aligned offsets.
# ---------------------------------------------------------------------------
def flat_offsets(sizes, align=256):
    offs, at = [], 0
    for n in sizes:
        offs.append(at)
        at += -(-n // align) * align
    return offs, max(at, align)


def host_inputs(work, g, rows=False, shards=True):
    """Seeded gradients and (unless ``shards`` is False) every rank's shards
    of group g (host arrays)."""
    specs, W = work.groups[g], work.W
    c = chunks(specs, W, rows)
    grads = [wl.grad_values(work, g, i) for i in range(len(specs))]
    if not shards:
        return grads, None
    local = [[wl.shard_values(work, g, i, r, c[i], max(0, min(c[i], s.numel - r * c[i])))
              for i, s in enumerate(specs)] for r in range(W)]
    return grads, local


def device_inputs(work, g, rows=False):
    """The same inputs drawn on the device (torch's seeded generator, the same
    distributions), for workloads too large to draw on the host quickly."""
    specs, W = work.groups[g], work.W
    c = chunks(specs, W, rows)
    grads = [wl.device_normal_bits(s.numel, s.grad_dtype, work.std, work.seed, g, i, 1) for i, s in enumerate(specs)]
    shards = []
    for r in range(W):
        row = []
        for i, s in enumerate(specs):
            t = wl.device_normal_bits(c[i], s.shard_dtype, work.std, work.seed, g, i, 3, r)
            valid = max(0, min(c[i], s.numel - r * c[i]))
            t[valid * ESZ[s.shard_dtype]:] = 0
            row.append(t)
        shards.append(row)
    return grads, shards


def flatten(arrays, offs, total, torch=None):
    """Concatenate per-parameter byte arrays at the given offsets: numpy arrays
    into a host buffer, device tensors into a device buffer."""
    if arrays and torch is not None and isinstance(arrays[0], torch.Tensor):
        out = torch.zeros(total, dtype=torch.uint8, device=arrays[0].device)
        for a, o in zip(arrays, offs):
            out[o:o + a.numel()].copy_(a)
        return out
    out = np.zeros(total, np.uint8)
    for a, o in zip(arrays, offs):
        b = a.view(np.uint8)
        out[o:o + b.size] = b
    return out


def to_device(flat, torch):
    return flat if isinstance(flat, torch.Tensor) else torch.from_numpy(flat).to("cuda")


# ---------------------------------------------------------------------------
# The CPU oracle's pack on bounded samples: one (rank, parameter) run at a time.
# ---------------------------------------------------------------------------
class OracleSampler:
    """Cycles through the runs of the reduce-scatter pack of every group --
    one (bucket, rank, parameter) run at a time, each with its algorithmic
    bytes -- on the oracle."""

    def __init__(self, work, inputs, rows=False):
        import oracle
        self.oracle = oracle
        W = work.W
        self.segs = []
        self.pack_bytes = 0
        for g, specs in enumerate(work.groups):
            grads = inputs[g][0]
            pl = oracle.plan(oracle.params_from_specs(specs), W, row_elems=row_elems(specs) if rows else None)
            st = {"pl": pl, "grads": grads,
                  "bufs": [np.empty(W * S, oracle.DTYPE_NP[d]) for d, S in zip(pl.bucket_dtype, pl.bucket_S)]}
            sz = oracle.DTYPE_SIZE
            for b in range(len(pl.bucket_dtype)):
                for r in range(W):
                    for p, prm in enumerate(pl.params):
                        if pl.bucket_of[p] != b:
                            continue
                        valid = max(0, min(pl.chunk[p], prm.numel - r * pl.chunk[p]))
                        nbytes = valid * sz[prm.grad_dtype] + pl.chunk[p] * sz[pl.bucket_dtype[b]]
                        self.segs.append((st, r, p, nbytes))
            self.pack_bytes += (sum(prm.numel * sz[prm.grad_dtype] for prm in pl.params)
                                + sum(W * S * sz[d] for d, S in zip(pl.bucket_dtype, pl.bucket_S)))
        self.i = 0

    def next(self) -> int:
        st, r, p, nbytes = self.segs[self.i]
        self.i = (self.i + 1) % len(self.segs)
        self.oracle.pack_segment(st["pl"], st["grads"], st["bufs"], r, p)
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
    """The oracle's pack, run after run, for about `seconds`."""
    done_bytes, runs = 0, 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds or runs == 0:
        done_bytes += sampler.next()
        runs += 1
    dt = time.perf_counter() - t0
    return {"value": done_bytes / dt / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{runs} (bucket, rank, parameter) runs of the reduce-scatter pack of the same workload "
                      f"({done_bytes / sampler.pack_bytes:.2f} whole packs), single-threaded C oracle, {dt:.1f} s",
            **host_cpu()}


def make_config(args, work, description, n_groups, n_launch, pack_bytes, world):
    """The `config` of both arms' JSON lines (identical for the same flags)."""
    return {"workload": f"{description}; timed: the reduce-scatter pack of every group, launches back to back",
            "world_size_layout": work.W, "chunking": CHUNKING[args.row_chunks], "groups": n_groups,
            "launches_per_op": n_launch, "pack_bytes": pack_bytes,
            "launch": ("CUDA graph of two packs, replayed" if args.graph
                       else "stream launches from the host") + (", batched over groups" if args.batched else ""),
            "parallelism": f"replicas x{world} (no data-path collective)",
            "l2": f"inputs larger than L2: two rotating buffer sets of {2 * pack_bytes / 1e9:.2f} GB of pack "
                  "traffic vs 129 MB L2; no flush"}


# ---------------------------------------------------------------------------
# Our arm.
# ---------------------------------------------------------------------------
class DeviceSet:
    """One complete set of device buffers for a step (two sets rotate)."""

    def __init__(self, fp, torch, L, specs, W, info, grads, shards, rank_row, others=None, rows=False):
        dev = torch.device("cuda")
        c = chunks(specs, W, rows)
        self.S_ag = info.ag_bytes
        g_sizes = [s.numel * ESZ[s.grad_dtype] for s in specs]
        goffs, gtot = flat_offsets(g_sizes)
        self.grads = to_device(flatten(grads, goffs, gtot, torch), torch)
        self.grad_ptrs = fp.pointer_array([self.grads.data_ptr() + o for o in goffs])
        self.buckets = [torch.empty(fp.fsdp_layout_bucket(L, b).bytes, dtype=torch.uint8, device=dev)
                        for b in range(info.n_buckets)]
        self.bucket_ptrs = fp.pointer_array(self.buckets)
        s_sizes = [ci * ESZ[s.shard_dtype] for ci, s in zip(c, specs)]
        soffs, stot = flat_offsets(s_sizes)
        self.shard_offs, self.shard_tot = soffs, stot
        self.shards = to_device(flatten(shards[rank_row], soffs, stot, torch), torch)
        self.shard_ptrs = fp.pointer_array([self.shards.data_ptr() + o for o in soffs])
        self.gathered = torch.empty(W * self.S_ag, dtype=torch.uint8, device=dev)
        self.gathered_ptr = self.gathered.data_ptr()
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
        self.W, self.sharded_offs = W, hoffs
        # The other ranks' rows: what the all-gather would deliver.
        for r in range(W):
            if r == rank_row:
                continue
            other = to_device(flatten(shards[r], soffs, stot, torch), torch)
            fp.fsdp_allgather_copy_in(L, [other.data_ptr() + o for o in soffs],
                                      self.gathered.data_ptr() + r * self.S_ag)
            torch.cuda.synchronize()
            del other

    def spare(self, fp, torch):
        """Fresh copies of what the copy-in and the reduce-scatter copy-out
        touch (shards, one all-gather row, row 0 of every bucket, sharded
        gradients), for loops of those short operations that rotate through
        more memory than L2 holds."""
        return SpareSet(fp, torch, self)

    def pack(self, fp, L, h):
        fp.fsdp_pack_reduce_scatter(L, self.grad_ptrs, self.bucket_ptrs, h)

    def emulated_rs(self, fp, L, h):
        fp.fsdp_emulated_reduce_scatter(L, self.packed_ptrs, self.reduced_ptrs, h)

    def copy_in(self, fp, L, h):
        fp.fsdp_allgather_copy_in(L, self.shard_ptrs, self.row_ptr, h)

    def copy_out(self, fp, L, h):
        fp.fsdp_allgather_copy_out(L, self.gathered_ptr, self.full_ptrs, h)

    def rs_copy_out(self, fp, L, h):
        fp.fsdp_reduce_scatter_copy_out(L, self.row0_ptrs, self.sharded_ptrs, h)

    def step(self, fp, L, h, ev=None, rs=False):
        """pack, [emulated reduce-scatter], copy-in, copy-out, [rs copy-out];
        ev[k] is recorded after the k-th launch (ev[0] before the first)."""
        ops = ["pack"] + (["emulated_rs"] if self.reduced is not None else []) + ["copy_in", "copy_out"] \
            + (["rs_copy_out"] if rs else [])
        for k, op in enumerate(ops):
            if ev is not None:
                ev[k].record()
            getattr(self, op)(fp, L, h)
        if ev is not None:
            ev[len(ops)].record()


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


class SpareSet:
    """See DeviceSet.spare."""

    def __init__(self, fp, torch, ds):
        self.shards = ds.shards.clone()
        self.shard_ptrs = fp.pointer_array([self.shards.data_ptr() + o for o in ds.shard_offs])
        self.row = torch.empty(ds.S_ag, dtype=torch.uint8, device=ds.shards.device)
        self.row_ptr = self.row.data_ptr()
        self.row0 = [b[:b.numel() // ds.W].clone() for b in (ds.reduced or ds.buckets)]
        self.row0_ptrs = fp.pointer_array(self.row0)
        self.sharded = torch.empty_like(ds.sharded)
        self.sharded_ptrs = fp.pointer_array([self.sharded.data_ptr() + o for o in ds.sharded_offs])

    def copy_in(self, fp, L, h):
        fp.fsdp_allgather_copy_in(L, self.shard_ptrs, self.row_ptr, h)

    def rs_copy_out(self, fp, L, h):
        fp.fsdp_reduce_scatter_copy_out(L, self.row0_ptrs, self.sharded_ptrs, h)


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

    @staticmethod
    def spare_args(fp, spares):
        """Batched pointer arrays of one SpareSet per group."""
        cat = lambda arrs: fp.pointer_array([p for a in arrs for p in a])  # noqa: E731
        return dict(shards=cat(s.shard_ptrs for s in spares), rows=fp.pointer_array([s.row_ptr for s in spares]),
                    row0=cat(s.row0_ptrs for s in spares), sharded=cat(s.sharded_ptrs for s in spares))

    def pack(self, fp, h, k):
        a = self.sets[k]
        fp.fsdp_pack_reduce_scatter_batched(self.layouts, a["grads"], a["buckets"], h)

    def copy_in(self, fp, h, k):
        a = self.sets[k]
        fp.fsdp_allgather_copy_in_batched(self.layouts, a["shards"], a["rows"], h)

    def copy_out(self, fp, h, k):
        a = self.sets[k]
        fp.fsdp_allgather_copy_out_batched(self.layouts, a["gathered"], a["full"], h)

    def rs_copy_out(self, fp, h, k):
        a = self.sets[k]
        fp.fsdp_reduce_scatter_copy_out_batched(self.layouts, a["row0"], a["sharded"], h)

    def step(self, fp, h, k, ev=None, rs=False):
        ops = ["pack", "copy_in", "copy_out"] + (["rs_copy_out"] if rs else [])
        for j, op in enumerate(ops):
            if ev is not None:
                ev[j].record()
            getattr(self, op)(fp, h, k)
        if ev is not None:
            ev[len(ops)].record()


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

        pre_ms, fused_ms = loop_ms(torch, precast, iters), loop_ms(torch, fused, iters)
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


def loop_ms(torch, fn, iters, warm=10):
    """Mean ms per call of fn(k), k = 0 .. iters - 1, timed back to back with
    CUDA events on the current stream after `warm` untimed calls."""
    for k in range(warm):
        fn(k)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for k in range(iters):
        fn(k)
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / iters


def same_run_references(fp, torch, nbytes, iters):
    """Plain copies of the pack's byte count in the same process and loop
    style: the library's streaming BF16 -> FP32 widen (the pack's 1 : 2 mix of
    bytes read to bytes written) and torch's 1 : 1 device copy.  Beside them,
    plain torch kernels of the copy-in's and the copy-out's own byte counts
    and read : write mixes (an FP32 -> BF16 cast, 2 : 1; a byte copy, 1 : 1),
    which show what one launch of that size reaches on this GPU."""
    pack_bytes = nbytes["pack"]
    n = pack_bytes // 6 // 8 * 8          # BF16 elements: 2n read + 4n written
    src = [torch.empty(2 * n, dtype=torch.uint8, device="cuda").random_(0, 256) for _ in range(2)]
    dst = [torch.empty(4 * n, dtype=torch.uint8, device="cuda") for _ in range(2)]
    widen_ms = loop_ms(torch, lambda k: fp.fsdp_debug_stream_widen(src[k & 1], n, dst[k & 1]), iters)
    half = pack_bytes // 2 // 16 * 16
    a = [torch.empty(half, dtype=torch.uint8, device="cuda") for _ in range(2)]
    b = [torch.empty(half, dtype=torch.uint8, device="cuda") for _ in range(2)]
    copy_ms = loop_ms(torch, lambda k: b[k & 1].copy_(a[k & 1]), iters)
    del src, dst, a, b
    out = {"plain_widen_1to2": {"what": "fsdp_debug_stream_widen, BF16 -> FP32, same bytes",
                                "bytes": 6 * n, "us": widen_ms * 1e3, "gbs": 6 * n / (widen_ms * 1e-3) / 1e9},
           "copy_1to1": {"what": "torch copy_ of uint8, half the bytes read and half written",
                         "bytes": 2 * half, "us": copy_ms * 1e3, "gbs": 2 * half / (copy_ms * 1e-3) / 1e9},
           "iters": iters}
    m = nbytes["copy_in"] // 6             # FP32 elements: 4m read + 2m written
    R = rotation_count(torch, 6 * m)
    f = [torch.empty(m, dtype=torch.float32, device="cuda").normal_() for _ in range(R)]
    g = [torch.empty(m, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    cast_ms = loop_ms(torch, lambda k: g[k % R].copy_(f[k % R]), iters)
    del f, g
    q = nbytes["copy_out"] // 2 // 16 * 16
    Q = rotation_count(torch, 2 * q)
    a = [torch.empty(q, dtype=torch.uint8, device="cuda") for _ in range(Q)]
    b = [torch.empty(q, dtype=torch.uint8, device="cuda") for _ in range(Q)]
    copy_out_ms = loop_ms(torch, lambda k: b[k % Q].copy_(a[k % Q]), iters)
    del a, b
    out["copy_in_sized_cast_2to1"] = {"what": "torch FP32 -> BF16 copy_ of the copy-in's byte count",
                                      "bytes": 6 * m, "us": cast_ms * 1e3, "gbs": 6 * m / (cast_ms * 1e-3) / 1e9,
                                      "rotating_buffer_sets": R}
    out["copy_out_sized_copy_1to1"] = {"what": "torch copy_ of uint8, the copy-out's byte count",
                                       "bytes": 2 * q, "us": copy_out_ms * 1e3,
                                       "gbs": 2 * q / (copy_out_ms * 1e-3) / 1e9, "rotating_buffer_sets": Q}
    return out


def run_packs(fp, groups, h, first, count, batch=None, op="pack"):
    """`count` calls of one operation (default the pack) for every group,
    alternating the two buffer sets."""
    for i in range(first, first + count):
        if batch is not None:
            getattr(batch, op)(fp, h, i & 1)
            continue
        for grp in groups:
            getattr(grp.sets[i & 1], op)(fp, grp.L, h)


def l2_bytes(torch):
    try:
        return int(torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size)
    except (AttributeError, RuntimeError):
        return 129 << 20


def rotation_count(torch, nbytes):
    """Buffers a back-to-back loop rotates through so that it touches at
    least three times L2 between two uses of one buffer (at least two)."""
    return max(2, -(-3 * l2_bytes(torch) // max(1, nbytes)))


def ops_alone(fp, torch, groups, batch, h, OPS, nbytes, n_launch, seconds):
    """Each operation alone: launches of that operation back to back (no
    events between them), about `seconds` of each after a short estimate.
    The pack and the copy-out alternate the two buffer sets, which hold more
    than L2; the copy-in and the reduce-scatter copy-out rotate through as
    many spare copies of their inputs and outputs as it takes to touch three
    times L2, so that no call finds the data of a recent one in L2."""
    out = {}
    for op in OPS:
        fn, R = (lambda k, op=op: run_packs(fp, groups, h, k, 1, batch, op)), 2
        spares = None
        if op in ("copy_in", "rs_copy_out") and 2 * nbytes[op] < 3 * l2_bytes(torch):
            R = rotation_count(torch, nbytes[op])
            spares = [[grp.sets[r & 1].spare(fp, torch) for grp in groups] for r in range(R)]
            if batch is not None:
                args = [Batch.spare_args(fp, sp) for sp in spares]
                if op == "copy_in":
                    fn = lambda k: fp.fsdp_allgather_copy_in_batched(  # noqa: E731
                        batch.layouts, args[k % R]["shards"], args[k % R]["rows"], h)
                else:
                    fn = lambda k: fp.fsdp_reduce_scatter_copy_out_batched(  # noqa: E731
                        batch.layouts, args[k % R]["row0"], args[k % R]["sharded"], h)
            else:
                fn = lambda k, op=op: [getattr(sp, op)(fp, grp.L, h)  # noqa: E731
                                       for sp, grp in zip(spares[k % R], groups)]
        est = loop_ms(torch, fn, 20)
        iters = max(50, int(seconds / (est * 1e-3)))
        ms = loop_ms(torch, fn, iters)
        out[op] = {"bytes": nbytes[op], "launches_per_call": n_launch, "calls": iters, "us": ms * 1e3,
                   "gbs": nbytes[op] / (ms * 1e-3) / 1e9, "rotating_buffer_sets": R,
                   "bytes_between_reuse": R * nbytes[op]}
        del spares
    for grp in groups:
        fp.fsdp_sync_status(grp.L)
    torch.cuda.empty_cache()
    return out


def run_steps(fp, groups, h, first, count, evs=None, batch=None, rs=False):
    for i in range(first, first + count):
        if batch is not None:
            batch.step(fp, h, i & 1, None if evs is None else evs[i - first][0], rs)
            continue
        for gi, grp in enumerate(groups):
            grp.sets[i & 1].step(fp, grp.L, h, None if evs is None else evs[i - first][gi], rs)


def capture(torch, fn):
    """A CUDA graph of fn(stream) on a side stream (two packs or two steps)."""
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        fn(torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return graph


def timed_passes(fp, torch, groups, batch, h, K, warmup, rs, graph, gpu_id):
    """The timed region (K packs of every group, back to back) and, right
    after it, K whole steps; clocks sampled over both.  Returns the two
    device times (max over ranks) and the clock record."""
    run_steps(fp, groups, h, 0, warmup, batch=batch, rs=rs)
    run_packs(fp, groups, h, 0, warmup, batch=batch)
    for grp in groups:
        fp.fsdp_sync_status(grp.L)
    g_pack = g_step = None
    if graph:
        g_pack = capture(torch, lambda s: run_packs(fp, groups, s, 0, 2, batch=batch))
        g_step = capture(torch, lambda s: run_steps(fp, groups, s, 0, 2, batch=batch, rs=rs))
        for _ in range(max(1, warmup // 2)):
            g_pack.replay()
            g_step.replay()
        torch.cuda.synchronize()
        for grp in groups:
            fp.fsdp_sync_status(grp.L)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    sampler = ClockSampler(gpu_id)
    torch.cuda.synchronize()
    barrier()
    sampler.start()
    time.sleep(0.3)  # let the sampler take its first sample before the load starts
    ev[0].record()
    if g_pack is not None:
        for _ in range(K // 2):
            g_pack.replay()
    else:
        run_packs(fp, groups, h, 0, K, batch=batch)
    ev[1].record()
    ev[2].record()
    if g_step is not None:
        for _ in range(K // 2):
            g_step.replay()
    else:
        run_steps(fp, groups, h, 0, K, batch=batch, rs=rs)
    ev[3].record()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    barrier()
    for grp in groups:
        fp.fsdp_sync_status(grp.L)
    dev = torch.device("cuda")
    return (max_over_ranks(ev[0].elapsed_time(ev[1]), device=dev),
            max_over_ranks(ev[2].elapsed_time(ev[3]), device=dev), clocks)


def evented_ops(fp, torch, groups, batch, h, K, OPS, rs):
    """Per-operation device times: the same steps with a CUDA event around
    every launch (events between launches serialise them)."""
    n_launch = 1 if batch is not None else len(groups)
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(len(OPS) + 1)] for _ in range(n_launch)]
           for _ in range(K)]
    torch.cuda.synchronize()
    barrier()
    run_steps(fp, groups, h, 0, K, evs, batch=batch, rs=rs)
    torch.cuda.synchronize()
    barrier()
    for grp in groups:
        fp.fsdp_sync_status(grp.L)
    return {k: [sum(e[j].elapsed_time(e[j + 1]) for e in step) for step in evs] for j, k in enumerate(OPS)}


def op_rows(nbytes, per, n_launch):
    return {k: {"bytes": nbytes[k], "launches_per_step": n_launch, "ms_mean": statistics.mean(v),
                "ms_median": statistics.median(v), "ms_min": min(v),
                "gbs": nbytes[k] / (statistics.mean(v) * 1e-3) / 1e9}
            for k, v in per.items()}


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
    K = args.steps + (args.steps & 1 if args.graph else 0)
    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:
        pass
    pack_total_ms, step_total_ms, clocks = timed_passes(fp, torch, groups, batch, h, K, args.warmup, rs,
                                                        args.graph, gpu_id)
    per = evented_ops(fp, torch, groups, batch, h, min(K, args.evented_steps), OPS, rs)
    alone = ops_alone(fp, torch, groups, batch, h, OPS, nbytes, n_launch, args.op_seconds) \
        if args.op_seconds > 0 else None

    refs = same_run_references(fp, torch, nbytes, args.reference_iters) if args.reference_iters > 0 else None
    if refs is not None and alone is not None and n_launch == 1:
        for op, key in (("copy_in", "copy_in_sized_cast_2to1"), ("copy_out", "copy_out_sized_copy_1to1")):
            alone[op]["same_size_reference_us"] = refs[key]["us"]
    precast = None
    if len(groups) == 1 and args.precast_iters > 0:
        precast = precast_comparison(fp, torch, work, groups[0], h, args.precast_iters, rows)
    e2e = step_e2e = None
    if args.e2e_steps > 0:
        e2e = run_e2e(args, fp, torch, groups, h, rs, nbytes["pack"], world, whole_step=False)
        step_e2e = run_e2e(args, fp, torch, groups, h, rs, step_bytes, world, whole_step=True)
    extra = None
    if args.extra and world == 1 and args.workload == "mixed50m":
        extra = {}
        for name, wname, batched in EXTRA_WORKLOADS:
            extra[name] = run_extra(fp, torch, h, wname, batched, gpu_id)
    elif args.extra:
        extra = {"skipped": "only with the default workload at N = 1 (the extra workloads are per-GPU "
                            "figures; replicas would repeat them)"}

    result = None
    if rank == 0:
        result = report(args, work, description, groups, nbytes, step_bytes, pack_total_ms, step_total_ms, per,
                        clocks, e2e, step_e2e, n_launch, world, K, refs)
        if alone is not None:
            result["ops_alone"] = alone
            result["ops_alone_note"] = ("each operation alone, its launches back to back with no events between "
                                        "them (programmatic dependent launch on): per-call device time; each loop "
                                        "rotates through buffer sets that hold more than L2 "
                                        "(bytes_between_reuse)")
        if precast is not None:
            result["precast_baseline"] = precast
        if extra is not None:
            result["extra_workloads"] = extra
    for grp in groups:
        grp.L.close()
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        result["cpu_baseline"] = cpu_baseline(OracleSampler(work, inputs, rows), args.cpu_seconds)
    if rank == 0:
        print(json.dumps(result), flush=True)
    import torch.distributed as dist
    if dist.is_initialized():
        dist.destroy_process_group()


# The extra workloads of the default run: (key, workload, batched).
EXTRA_WORKLOADS = (("transformer500_batched", "transformer500", True),
                   ("transformer500_per_group", "transformer500", False),
                   ("kda_block_w64", "kda_w64", False))


def run_extra(fp, torch, h, wname, batched, gpu_id, seconds=0.5):
    """One more workload, about `seconds` of packs and of whole steps each,
    with inputs drawn on the device: pack, copy-in and copy-out times and the
    pack's fraction of the measured copy bandwidth, with its own clocks."""
    factory, description = WORKLOADS[wname]
    work = factory()
    groups = [Group(fp, torch, work, g, device_inputs(work, g)) for g in range(len(work.groups))]
    batch = Batch(fp, groups) if batched else None
    n_launch = 1 if batch is not None else len(groups)
    OPS = ("pack", "copy_in", "copy_out")
    nbytes = {k: sum(grp.nbytes[k] for grp in groups) for k in OPS}
    step_bytes = sum(nbytes.values())
    probe_ms = loop_ms(torch, lambda k: run_packs(fp, groups, h, k, 1, batch=batch), 20)
    K = max(20, int(seconds / (probe_ms * 1e-3)))
    K += K & 1
    pack_ms, step_ms, clocks = timed_passes(fp, torch, groups, batch, h, K, 10, False, False, gpu_id)
    per = evented_ops(fp, torch, groups, batch, h, min(K, 500), OPS, False)
    alone = ops_alone(fp, torch, groups, batch, h, OPS, nbytes, n_launch, 0.1)
    peak, peak_kind = read_peaks()
    pack_gbs = nbytes["pack"] * K / (pack_ms * 1e-3) / 1e9
    out = {"workload": description, "groups": len(groups), "launches_per_op": n_launch, "steps": K,
           "pack": {"bytes": nbytes["pack"], "us": pack_ms * 1e3 / K, "gbs": pack_gbs, "frac": pack_gbs / peak,
                    "frac_of_nominal_8tbs": pack_gbs / NOMINAL_HBM_GBS, "peak": peak, "peak_source": peak_kind},
           "hot_path_step": {"bytes": step_bytes, "us": step_ms * 1e3 / K,
                             "gbs": step_bytes * K / (step_ms * 1e-3) / 1e9},
           "ops": op_rows(nbytes, per, n_launch), "ops_alone": alone, "clocks": clocks}
    for grp in groups:
        grp.L.close()
    del groups, batch
    torch.cuda.empty_cache()
    return out


def run_e2e(args, fp, torch, groups, h, rs, nbytes, world, whole_step):
    # End to end through the same API with host buffers.  Pack only: every
    # step uploads the gradients from pinned host memory and downloads the
    # packed buckets.  Whole step: also the shards and the other ranks' rows
    # up, the full parameters (and sharded gradients) down.  Steps are
    # pipelined the way a caller would run them: uploads on one stream, the
    # kernels on another, downloads on a third, two buffer sets, so step
    # i+1's uploads overlap step i's downloads.
    pin = lambda n: torch.empty(n, dtype=torch.uint8, pin_memory=True)  # noqa: E731
    host = []
    for grp in groups:
        s0 = grp.sets[0]
        hb = {"grads": pin(s0.grads.numel()),
              "out": [{"buckets": [pin(b.numel()) for b in s0.buckets]} for _ in range(2)]}
        hb["grads"].copy_(s0.grads.cpu())
        if whole_step:
            hb["shards"], hb["others"] = pin(s0.shards.numel()), pin(s0.gathered.numel() - s0.S_ag)
            hb["shards"].copy_(s0.shards.cpu())
            hb["others"].copy_(s0.gathered[s0.S_ag:].cpu())
            for o in hb["out"]:
                o["full"] = pin(s0.full.numel())
                o["sharded"] = pin(s0.sharded.numel()) if rs else None
        host.append(hb)
    h2d = sum(hb["grads"].numel() + (hb["shards"].numel() + hb["others"].numel() if whole_step else 0)
              for hb in host)
    d2h = sum(sum(b.numel() for b in hb["out"][0]["buckets"])
              + (hb["out"][0]["full"].numel() + (hb["out"][0]["sharded"].numel() if rs else 0) if whole_step else 0)
              for hb in host)
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
                    if whole_step:
                        sk.shards.copy_(hb["shards"], non_blocking=True)
                        sk.gathered[sk.S_ag:].copy_(hb["others"], non_blocking=True)
                uploaded[k].record(up)
            main.wait_event(uploaded[k])
            for grp in groups:
                if whole_step:
                    grp.sets[k].step(fp, grp.L, h, None, rs)
                else:
                    grp.sets[k].pack(fp, grp.L, h)
            computed[k].record(main)
            with torch.cuda.stream(down):
                down.wait_event(computed[k])
                for grp, hb in zip(groups, host):
                    sk, ho = grp.sets[k], hb["out"][k]
                    for hbuf, dbuf in zip(ho["buckets"], sk.buckets):
                        hbuf.copy_(dbuf, non_blocking=True)
                    if whole_step:
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
    what = ("whole step (pack, copy-in, copy-out" + (", rs copy-out" if rs else "") + ")") if whole_step else \
        "the reduce-scatter pack"
    return {"value": world * nbytes * E / (e2e_ms * 1e-3) / 1e9, "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": E, "ms_per_step": e2e_ms / E,
            "note": f"{what} with host buffers; uploads, kernels and downloads of consecutive steps pipelined "
                    "on three streams with two buffer sets"}


def report(args, work, description, groups, nbytes, step_bytes, pack_total_ms, step_total_ms, per, clocks, e2e,
           step_e2e, n_launch, world, K, refs):
    """The JSON result of our arm (rank 0)."""
    peak, peak_kind = read_peaks()
    pack_ms = pack_total_ms / K
    achieved = nbytes["pack"] / (pack_ms * 1e-3) / 1e9   # per GPU
    roofline = {"bound": "hbm", "kernel": "walk_kernel (the reduce-scatter pack launches)",
                "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
                "peak_source": f"{peak_kind} hbm_gbs (burst copy)" if peak_kind == "measured" else "fallback",
                "bytes_per_launch": nbytes["pack"] / n_launch,
                "timing": "mean per pack over the timed region (K packs back to back, CUDA events around the "
                          "whole region on the launching stream)",
                "traffic": None}
    if args.workload == "mixed50m" and not args.row_chunks and n_launch == 1:
        t = read_traffic()
        if t is not None:
            roofline.update(t)
            roofline["traffic_note"] = ("DRAM bytes of one cold ncu capture of the pack; "
                                        "traffic_l2_write counts L2 write sectors x 32 B")
    if refs is not None:
        for r in (refs["plain_widen_1to2"], refs["copy_1to1"]):
            r["pack_over_this"] = achieved / r["gbs"]
        roofline["same_run_references"] = refs
    result = {
        "metric": METRIC,
        "value": world * nbytes["pack"] * K / (pack_total_ms * 1e-3) / 1e9,
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": pack_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16+f32",
        "data": "synthetic",
        "config": make_config(args, work, description, len(groups), n_launch, nbytes["pack"], world),
        "step_note": "one step = the reduce-scatter pack of every group of the workload (the operation the "
                     "metric names); ms_per_step is the pack's ms per fully_shard group" +
                     (" (all groups)" if len(groups) > 1 else ""),
        "hot_path_step": {"what": STEP + (STEP_RS if args.rs_copy_out else "")
                          + (STEP_ERS if args.emulated_rs else ""),
                          "bytes": step_bytes, "steps": K, "ms_per_step": step_total_ms / K,
                          "gbs": world * step_bytes * K / (step_total_ms * 1e-3) / 1e9,
                          "timing": "K whole steps back to back right after the timed region, same clocks"},
        "ops": op_rows(nbytes, per, n_launch),
        "ops_note": "per-operation device times from a pass of whole steps with CUDA events around every "
                    "launch (summed over the step's groups); events serialise the launches, and each operation "
                    "also pays for the L2 write-back of the one before it",
        "roofline": roofline,
        "e2e": e2e,
        "hot_path_step_e2e": step_e2e,
        "gpu_launches": K * n_launch,
        "gpu_launches_note": "walk_kernel launches inside the timed region (the packs); the whole-step pass "
                             "after it launches 3 per group and step",
        "clocks": clocks,
    }
    return result


# ---------------------------------------------------------------------------
# Reference arm: the CPU oracle's pack, each step one bounded run of it.
# ---------------------------------------------------------------------------
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    factory, description = WORKLOADS[args.workload]
    work = factory()
    inputs = [host_inputs(work, g, args.row_chunks, shards=False) for g in range(len(work.groups))]
    samp = OracleSampler(work, inputs, args.row_chunks)
    for _ in range(args.warmup):
        samp.next()
    done = 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        done += samp.next()
    dt = time.perf_counter() - t0
    value = done / dt / 1e9
    n_launch = 1 if args.batched else len(work.groups)
    result = {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt * 1e3 / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16+f32", "data": "synthetic",
        "config": make_config(args, work, description, len(work.groups), n_launch, samp.pack_bytes, world),
        "step_note": "one step = one (bucket, rank, parameter) run of the reduce-scatter pack on the CPU oracle, "
                     f"cycling through the {len(samp.segs)} runs of the workload's pack; value = bytes / time",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{args.steps} runs of the reduce-scatter pack "
                                   f"({done / samp.pack_bytes:.2f} whole packs)", **host_cpu()},
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
