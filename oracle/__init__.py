"""CPU oracle for mixed-dtype FSDP communication-buffer packing.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline / reference leg
may import this package.  It shares no code with the CUDA library in
``fsdp2_gradient_packing_gb300``: its planner below is written separately from
the library's C++ planner, and its element loops (``fsdp_oracle.c``) are plain
single-threaded C that restate the definitions.

Sources (web pages, cited by title and section):

* [News] "FSDP2 per-parameter mixed precision" news item (ainewsletter.today,
  ?p=1549), paragraphs 1-2: all-gather staging copies grouped by (source,
  target) dtype with one all-gather per fully_shard; the reduce-scatter copy-in
  casts BF16 and FP32 gradients into one reduction buffer while chunking and
  padding; one bucket and reduce-scatter per distinct effective reduce dtype.
* [Unit] "The unit you wrapped" (kernels.rudrite.com): the FlatParameter
  section (parameters flattened row-major; rank r holds the r-th contiguous
  slice), the auto_wrap_policy section (per-rank counts 36 / 18 / 9), and the
  padding section (right-hand padding to a multiple of the world size).
* [NeMo] "Mixed-Precision Training" (NVIDIA NeMo AutoModel), table "Storage
  Dtype Compared to Compute Dtype": param_dtype is the all-gather / compute
  dtype, reduce_dtype the gradient-reduction dtype, model.dtype the storage
  dtype of the resident shard.

Operations: the reduce-scatter copy-in (pack), the all-gather copy-in and
copy-out, the reduce-scatter copy-out (reduced bucket rows to sharded
gradients; [Unit] collective-count section), and an emulated reduce-scatter
(elementwise sum of every rank's packed buffer in rank order, partial sums
rounded to the bucket dtype) for end-to-end tests without a network.

Pins: every function here is checked in ``tests/test_oracle_pins.py`` against
values the pages print, closed forms, invariants, brute force on tiny inputs
and an exact-rational rounding reference.  One reading stands behind them: a
multi-parameter unit is chunked per parameter (FSDP2's rule), which the brute
force and the printed per-rank counts pin; the pages print shard values only
for single-parameter units, where FSDP1's one flat vector split W ways gives
the same result.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

F32 = 0
BF16 = 1
DTYPE_SIZE = {F32: 4, BF16: 2}
DTYPE_NP = {F32: np.uint32, BF16: np.uint16}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fsdp_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle's C loops with gcc (plain -O2, no vectorisation flags)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-tree-vectorize",
             "-Wall", "-Werror", "-o", tmp, _SRC, "-lm"],
            check=True,
        )
        os.replace(tmp, _LIB)
    return _LIB


def _bind(lib):
    """Declare the C signatures on a loaded oracle library and return it."""
    P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
    lib.oracle_f32_to_bf16.argtypes = [ctypes.c_uint32]
    lib.oracle_bf16_to_f32.restype = ctypes.c_uint32
    lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.oracle_f32_to_bf16_array.argtypes = [P, P, I64]
    lib.oracle_bf16_to_f32_array.argtypes = [P, P, I64]
    lib.oracle_pack_reduce_scatter.argtypes = [I32, I32, P, P, P, P, P, I32, P, P, P, P]
    lib.oracle_pack_samples.argtypes = [I32, P, P, P, P, P, I32, I32, I64, P, P, I64, P]
    lib.oracle_allgather_copy_in.argtypes = [I32, P, P, P, P, P, I32, P, I64, P, P]
    lib.oracle_allgather_copy_out.argtypes = [I32, I32, P, P, P, P, P, P, I64, P, P]
    lib.oracle_reduce_scatter_copy_out.argtypes = [I32, P, P, P, P, P, P, P]
    lib.oracle_emulated_reduce_scatter.argtypes = [I64, I32, I32, P, P]
    lib.oracle_emulated_reduce_scatter.restype = None
    for name in ("oracle_pack_reduce_scatter", "oracle_pack_samples", "oracle_reduce_scatter_copy_out",
                 "oracle_allgather_copy_in", "oracle_allgather_copy_out",
                 "oracle_f32_to_bf16_array", "oracle_bf16_to_f32_array"):
        getattr(lib, name).restype = None
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


# ---------------------------------------------------------------------------
# Planner ([Unit] FlatParameter + padding; [News] buckets and dtype groups).
# ---------------------------------------------------------------------------
@dataclass(frozen=True)
class Param:
    """One original parameter of a fully_shard group, in registration order."""
    numel: int
    grad_dtype: int = F32
    reduce_dtype: int = F32
    shard_dtype: int = F32
    param_dtype: int = F32


@dataclass
class Plan:
    W: int
    params: list
    chunk: list = field(default_factory=list)          # c_p
    bucket_of: list = field(default_factory=list)      # bucket index of p
    bucket_off: list = field(default_factory=list)     # o_p: element offset in its bucket row
    bucket_dtype: list = field(default_factory=list)   # rho_b
    bucket_S: list = field(default_factory=list)       # S_b: elements per rank row
    group_of: list = field(default_factory=list)       # all-gather group of p
    group_elem_off: list = field(default_factory=list)  # e_p: element offset inside its group
    group_pair: list = field(default_factory=list)     # (sigma, pi) of each group
    group_elems: list = field(default_factory=list)    # elements per group (per rank)
    group_byte_off: list = field(default_factory=list)  # G_g
    S_ag: int = 0                                      # bytes of one rank's all-gather input


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def _align16(x: int) -> int:
    return _ceil_div(x, 16) * 16


def plan(params, W: int, row_elems=None) -> Plan:
    """Layout of one fully_shard group.

    c_p = ceil(n_p / W): the flattened parameter padded on the right to c_p*W
    elements and split into W equal contiguous slices ([Unit], FlatParameter
    and padding sections).  With ``row_elems`` (elements per dim-0 row of
    each parameter; 0 keeps the flattened rule for that parameter) a
    parameter of d0 = n_p / row_elems rows is instead padded along dim 0 to a
    multiple of W rows and split into W row chunks: c_p = ceil(d0 / W) *
    row_elems, and rank r's chunk is rows [r*ceil(d0/W), (r+1)*ceil(d0/W)),
    i.e. flat elements [r*c_p, (r+1)*c_p) again.  Buckets: one per distinct reduce dtype, in order of
    first appearance; inside a bucket parameters keep registration order
    ([News] paragraph 2).  All-gather groups: one per distinct (shard dtype,
    param dtype) pair, in order of first appearance ([News] paragraph 1); each
    group starts on a 16-byte boundary and S_ag is rounded up to 16 bytes.
    """
    if W < 1:
        raise ValueError("world size must be >= 1")
    pl = Plan(W=W, params=list(params))
    bucket_index = {}
    group_index = {}
    for k, p in enumerate(pl.params):
        if p.numel < 0:
            raise ValueError("numel must be >= 0")
        rows_of = row_elems[k] if row_elems is not None else 0
        if rows_of:
            if p.numel % rows_of:
                raise ValueError("numel must be a multiple of row_elems")
            c = _ceil_div(p.numel // rows_of, W) * rows_of
        else:
            c = _ceil_div(p.numel, W)
        pl.chunk.append(c)
        if p.reduce_dtype not in bucket_index:
            bucket_index[p.reduce_dtype] = len(pl.bucket_dtype)
            pl.bucket_dtype.append(p.reduce_dtype)
            pl.bucket_S.append(0)
        b = bucket_index[p.reduce_dtype]
        pl.bucket_of.append(b)
        pl.bucket_off.append(pl.bucket_S[b])
        pl.bucket_S[b] += c
        pair = (p.shard_dtype, p.param_dtype)
        if pair not in group_index:
            group_index[pair] = len(pl.group_pair)
            pl.group_pair.append(pair)
            pl.group_elems.append(0)
        g = group_index[pair]
        pl.group_of.append(g)
        pl.group_elem_off.append(pl.group_elems[g])
        pl.group_elems[g] += c
    end = 0
    for g, (_, pi) in enumerate(pl.group_pair):
        start = _align16(end)
        pl.group_byte_off.append(start)
        end = start + pl.group_elems[g] * DTYPE_SIZE[pi]
    pl.S_ag = _align16(end)
    return pl


# ---------------------------------------------------------------------------
# Element loops (C).  Buffers are numpy arrays of raw bits: uint32 for FP32,
# uint16 for BF16, uint8 for the all-gather byte buffers.
# ---------------------------------------------------------------------------
def _i64(xs):
    return np.ascontiguousarray(np.asarray(xs, dtype=np.int64).reshape(-1))


def _i32(xs):
    return np.ascontiguousarray(np.asarray(xs, dtype=np.int32).reshape(-1))


def _ptrs(arrays):
    out = (ctypes.c_void_p * max(1, len(arrays)))()
    for k, a in enumerate(arrays):
        out[k] = a.ctypes.data if a is not None and a.size else None
    return out


def _check(arr, dt, n, what):
    if arr.dtype != DTYPE_NP[dt] or not arr.flags.c_contiguous or arr.size != n:
        raise ValueError(f"{what}: expected {n} contiguous {DTYPE_NP[dt].__name__}, "
                         f"got {arr.size} {arr.dtype}")


def _check_plan(pl: Plan) -> None:
    """Refuse a plan whose offsets would reach outside the buffers the C loops
    are given (they trust the plan).  Only bounds are checked here; the
    offsets' values are what the pins check."""
    P = len(pl.params)
    if any(len(x) != P for x in (pl.chunk, pl.bucket_of, pl.bucket_off, pl.group_of, pl.group_elem_off)) \
            or len(pl.bucket_S) != len(pl.bucket_dtype) or len(pl.group_byte_off) != len(pl.group_pair) \
            or len(pl.group_elems) != len(pl.group_pair):
        raise ValueError("plan: list lengths disagree")
    for p, prm in enumerate(pl.params):
        c, b, g = pl.chunk[p], pl.bucket_of[p], pl.group_of[p]
        if c < 0 or not 0 <= b < len(pl.bucket_S) or not 0 <= g < len(pl.group_pair):
            raise ValueError(f"plan: parameter {p} has a negative chunk or no bucket / group")
        if pl.bucket_off[p] < 0 or pl.bucket_off[p] + c > pl.bucket_S[b]:
            raise ValueError(f"plan: parameter {p} does not fit its bucket row")
        end = pl.group_byte_off[g] + (pl.group_elem_off[p] + c) * DTYPE_SIZE[prm.param_dtype]
        if pl.group_elem_off[p] < 0 or pl.group_byte_off[g] < 0 or end > pl.S_ag:
            raise ValueError(f"plan: parameter {p} does not fit the all-gather row")


def f32_to_bf16(bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint32)
    out = np.empty(bits.shape, np.uint16)
    _load().oracle_f32_to_bf16_array(bits.ctypes.data, out.ctypes.data, bits.size)
    return out


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, np.uint32)
    _load().oracle_bf16_to_f32_array(bits.ctypes.data, out.ctypes.data, bits.size)
    return out


def pack_reduce_scatter(pl: Plan, grads, out=None):
    """Reduce-scatter copy-in: one [W * S_b] buffer per bucket (flat, row r at r*S_b)."""
    _check_plan(pl)
    grads = [np.ascontiguousarray(g).reshape(-1) for g in grads]
    for p, g in zip(pl.params, grads):
        _check(g, p.grad_dtype, p.numel, "grad")
    if out is None:
        out = [np.empty(pl.W * S, DTYPE_NP[dt]) for dt, S in zip(pl.bucket_dtype, pl.bucket_S)]
    for o, dt, S in zip(out, pl.bucket_dtype, pl.bucket_S):
        _check(o, dt, pl.W * S, "bucket buffer")
    keep = [_i64([p.numel for p in pl.params]), _i32([p.grad_dtype for p in pl.params]),
            _i64(pl.chunk), _i32(pl.bucket_of), _i64(pl.bucket_off),
            _i32(pl.bucket_dtype), _i64(pl.bucket_S)]
    _load().oracle_pack_reduce_scatter(
        pl.W, len(pl.params), *(a.ctypes.data for a in keep[:5]), len(pl.bucket_dtype),
        keep[5].ctypes.data, keep[6].ctypes.data, _ptrs(grads), _ptrs(out))
    return out


def pack_samples(pl: Plan, grads, b: int, idx: np.ndarray) -> np.ndarray:
    """Elements idx (flat indices into bucket b's [W * S_b] buffer), one by one."""
    _check_plan(pl)
    grads = [np.ascontiguousarray(g).reshape(-1) for g in grads]
    for p, g in zip(pl.params, grads):
        _check(g, p.grad_dtype, p.numel, "grad")
    idx = _i64(idx)
    if idx.size and (idx.min() < 0 or idx.max() >= pl.W * pl.bucket_S[b]):
        raise ValueError("sample index outside the bucket")
    out = np.empty(idx.size, DTYPE_NP[pl.bucket_dtype[b]])
    keep = [_i64([p.numel for p in pl.params]), _i32([p.grad_dtype for p in pl.params]),
            _i64(pl.chunk), _i32(pl.bucket_of), _i64(pl.bucket_off)]
    _load().oracle_pack_samples(
        len(pl.params), *(a.ctypes.data for a in keep), b, pl.bucket_dtype[b],
        pl.bucket_S[b], _ptrs(grads), idx.ctypes.data, idx.size, out.ctypes.data)
    return out


def allgather_copy_in(pl: Plan, shards, out=None) -> np.ndarray:
    """All-gather copy-in of one rank: S_ag bytes."""
    _check_plan(pl)
    shards = [np.ascontiguousarray(s).reshape(-1) for s in shards]
    for p, c, s in zip(pl.params, pl.chunk, shards):
        _check(s, p.shard_dtype, c, "shard")
    if out is None:
        out = np.empty(pl.S_ag, np.uint8)
    if out.dtype != np.uint8 or not out.flags.c_contiguous or out.size != pl.S_ag:
        raise ValueError("all-gather input must be S_ag contiguous bytes")
    keep = [_i64(pl.chunk), _i32([p.shard_dtype for p in pl.params]),
            _i32([p.param_dtype for p in pl.params]), _i32(pl.group_of),
            _i64(pl.group_elem_off), _i64(pl.group_byte_off)]
    _load().oracle_allgather_copy_in(
        len(pl.params), *(a.ctypes.data for a in keep[:5]), len(pl.group_pair),
        keep[5].ctypes.data, pl.S_ag, _ptrs(shards), out.ctypes.data)
    return out


def allgather_copy_out(pl: Plan, ag_out: np.ndarray, out=None):
    """All-gather copy-out: the gathered [W * S_ag] bytes back to full parameters."""
    _check_plan(pl)
    ag_out = np.ascontiguousarray(ag_out, dtype=np.uint8).reshape(-1)
    if ag_out.size != pl.W * pl.S_ag:
        raise ValueError("gathered buffer must hold W * S_ag bytes")
    if out is None:
        out = [np.empty(p.numel, DTYPE_NP[p.param_dtype]) for p in pl.params]
    for o, p in zip(out, pl.params):
        _check(o, p.param_dtype, p.numel, "full parameter")
    keep = [_i64([p.numel for p in pl.params]), _i64(pl.chunk),
            _i32([p.param_dtype for p in pl.params]), _i32(pl.group_of),
            _i64(pl.group_elem_off), _i64(pl.group_byte_off)]
    _load().oracle_allgather_copy_out(
        pl.W, len(pl.params), *(a.ctypes.data for a in keep), pl.S_ag,
        ag_out.ctypes.data, _ptrs(out))
    return out


_CODE = {"f32": F32, "bf16": BF16}


def params_from_specs(specs):
    """Oracle parameter descriptors from workload specs (dtype strings)."""
    return [Param(s.numel, _CODE[s.grad_dtype], _CODE[s.reduce_dtype],
                  _CODE[s.shard_dtype], _CODE[s.param_dtype]) for s in specs]


def reduce_scatter_copy_out(pl: Plan, rows, out=None):
    """This rank's reduced bucket rows (S_b elements each) -> per-parameter
    sharded gradients (c_p elements of the shard dtype)."""
    _check_plan(pl)
    rows = [np.ascontiguousarray(r).reshape(-1) for r in rows]
    for b, (dt, S) in enumerate(zip(pl.bucket_dtype, pl.bucket_S)):
        _check(rows[b], dt, S, "reduced row")
    if out is None:
        out = [np.empty(c, DTYPE_NP[p.shard_dtype]) for p, c in zip(pl.params, pl.chunk)]
    for o, p, c in zip(out, pl.params, pl.chunk):
        _check(o, p.shard_dtype, c, "sharded gradient")
    keep = [_i64(pl.chunk), _i32(pl.bucket_of), _i64(pl.bucket_off), _i32(pl.bucket_dtype),
            _i32([p.shard_dtype for p in pl.params])]
    _load().oracle_reduce_scatter_copy_out(len(pl.params), *(a.ctypes.data for a in keep), _ptrs(rows), _ptrs(out))
    return out


def emulated_reduce_scatter(pl: Plan, packed):
    """packed[q] = rank q's bucket buffers (as from pack_reduce_scatter).
    Returns, per bucket, the [W * S_b] elementwise sum over ranks in rank
    order; row r is rank r's reduce-scatter output."""
    out = []
    for b, (dt, S) in enumerate(zip(pl.bucket_dtype, pl.bucket_S)):
        ins = [np.ascontiguousarray(packed[q][b]).reshape(-1) for q in range(len(packed))]
        for x in ins:
            _check(x, dt, pl.W * S, "packed buffer")
        res = np.empty(pl.W * S, DTYPE_NP[dt])
        if ins:
            _load().oracle_emulated_reduce_scatter(res.size, dt, len(ins), _ptrs(ins), res.ctypes.data)
        out.append(res)
    return out


# ---------------------------------------------------------------------------
# One run at a time (the same loops, entered per segment): lets the CPU
# baseline time bounded samples of a workload.
# ---------------------------------------------------------------------------
def _bind_segments(lib):
    P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.oracle_pack_segment.argtypes = [I32, I64, I32, I64, I64, I32, I64, P, P]
    lib.oracle_allgather_copy_in_segment.argtypes = [I64, I32, I32, I64, I64, P, P]
    lib.oracle_allgather_copy_out_segment.argtypes = [I32, I64, I64, I32, I64, I64, I64, P, P]
    for n in ("oracle_pack_segment", "oracle_allgather_copy_in_segment", "oracle_allgather_copy_out_segment"):
        getattr(lib, n).restype = None
    return lib


def pack_segment(pl: Plan, grads, bufs, r: int, p: int) -> None:
    """Row r's slots of parameter p in its bucket buffer (bufs as from pack_reduce_scatter)."""
    lib = _bind_segments(_load())
    b = pl.bucket_of[p]
    lib.oracle_pack_segment(r, pl.params[p].numel, pl.params[p].grad_dtype, pl.chunk[p], pl.bucket_off[p],
                            pl.bucket_dtype[b], pl.bucket_S[b], grads[p].ctypes.data, bufs[b].ctypes.data)


def allgather_copy_in_clear(pl: Plan, ag_in: np.ndarray) -> None:
    """The zero bytes of one rank's all-gather input (gaps and tail included)."""
    ag_in[:] = 0


def allgather_copy_in_segment(pl: Plan, shards, ag_in: np.ndarray, p: int) -> None:
    lib = _bind_segments(_load())
    g = pl.group_of[p]
    lib.oracle_allgather_copy_in_segment(pl.chunk[p], pl.params[p].shard_dtype, pl.params[p].param_dtype,
                                         pl.group_elem_off[p], pl.group_byte_off[g], shards[p].ctypes.data,
                                         ag_in.ctypes.data)


def allgather_copy_out_segment(pl: Plan, ag_out: np.ndarray, params, p: int, r: int) -> None:
    lib = _bind_segments(_load())
    g = pl.group_of[p]
    lib.oracle_allgather_copy_out_segment(r, pl.params[p].numel, pl.chunk[p], pl.params[p].param_dtype,
                                          pl.group_elem_off[p], pl.group_byte_off[g], pl.S_ag,
                                          ag_out.ctypes.data, params[p].ctypes.data)
