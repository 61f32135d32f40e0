"""Thin ctypes binding of the C ABI in include/fsdp_pack.h.

Each function here has the name of the C entry point it calls and only
marshals arguments: tensors become device pointers (``data_ptr()``), the
stream becomes a ``cudaStream_t`` handle, and a non-OK status becomes an
``FsdpError``.  Because the C functions read as many pointers as the layout
has slots, the binding first checks the pointer counts, and the size, dtype,
contiguity and device of any torch tensor it is given (``ValueError``).  All
packing work runs in the library's CUDA kernels; there is no fallback path.  Importing this module fails if the library has not been
built (``__graft_entry__.build()`` or ``python -m
fsdp2_gradient_packing_gb300._build``).
"""
from __future__ import annotations

import ctypes
import os

from . import _build

if not os.path.exists(_build.LIB):
    raise ImportError(
        f"{_build.LIB} is missing: build the CUDA library first "
        "(python -c 'import __graft_entry__ as g; g.build()')")

_lib = ctypes.CDLL(_build.LIB)

FSDP_DTYPE_F32 = 0
FSDP_DTYPE_BF16 = 1
DTYPE_CODES = {"f32": FSDP_DTYPE_F32, "bf16": FSDP_DTYPE_BF16}
DTYPE_BYTES = {FSDP_DTYPE_F32: 4, FSDP_DTYPE_BF16: 2}

FSDP_OK, FSDP_EINVAL, FSDP_ENOMEM, FSDP_ECUDA, FSDP_EUNSUPPORTED, FSDP_ETIMEOUT = range(6)
FSDP_MAX_PARAMS = 4000
FSDP_PLAN_HOST_ONLY = 1
FSDP_SCHEDULE_DEFAULT, FSDP_SCHEDULE_FIXED, FSDP_SCHEDULE_SHARED, FSDP_SCHEDULE_MIXED = range(4)


class fsdp_param_desc_t(ctypes.Structure):
    _fields_ = [("numel", ctypes.c_int64), ("grad_dtype", ctypes.c_int32),
                ("reduce_dtype", ctypes.c_int32), ("shard_dtype", ctypes.c_int32),
                ("param_dtype", ctypes.c_int32)]


class fsdp_layout_info_t(ctypes.Structure):
    _fields_ = [("world_size", ctypes.c_int32), ("n_params", ctypes.c_int32),
                ("n_buckets", ctypes.c_int32), ("n_groups", ctypes.c_int32),
                ("ag_bytes", ctypes.c_int64), ("total_numel", ctypes.c_int64),
                ("device", ctypes.c_int32), ("has_device_table", ctypes.c_int32),
                ("pack_items", ctypes.c_int64), ("copy_in_items", ctypes.c_int64),
                ("copy_out_items", ctypes.c_int64), ("rs_copy_out_items", ctypes.c_int64)]


class fsdp_param_info_t(ctypes.Structure):
    _fields_ = [("chunk", ctypes.c_int64), ("bucket", ctypes.c_int32), ("group", ctypes.c_int32),
                ("bucket_offset", ctypes.c_int64), ("group_offset", ctypes.c_int64),
                ("ag_byte_offset", ctypes.c_int64)]


class fsdp_bucket_info_t(ctypes.Structure):
    _fields_ = [("reduce_dtype", ctypes.c_int32), ("n_params", ctypes.c_int32),
                ("row_elems", ctypes.c_int64), ("bytes", ctypes.c_int64)]


class fsdp_group_info_t(ctypes.Structure):
    _fields_ = [("shard_dtype", ctypes.c_int32), ("param_dtype", ctypes.c_int32),
                ("n_params", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("byte_offset", ctypes.c_int64), ("elems", ctypes.c_int64),
                ("bytes", ctypes.c_int64)]


_P = ctypes.c_void_p
_ST = ctypes.c_int
_LAYOUT = ctypes.c_void_p
_SIGNATURES = {
    "fsdp_plan_layout": (_ST, [ctypes.POINTER(fsdp_param_desc_t), ctypes.c_int32, ctypes.c_int32,
                               ctypes.POINTER(_LAYOUT)]),
    "fsdp_plan_layout_host": (_ST, [ctypes.POINTER(fsdp_param_desc_t), ctypes.c_int32, ctypes.c_int32,
                                    ctypes.POINTER(_LAYOUT)]),
    "fsdp_plan_layout_ex": (_ST, [ctypes.POINTER(fsdp_param_desc_t), ctypes.POINTER(ctypes.c_int64), ctypes.c_int32,
                                  ctypes.c_int32, ctypes.c_uint32, ctypes.POINTER(_LAYOUT)]),
    "fsdp_layout_query": (_ST, [_LAYOUT, ctypes.POINTER(fsdp_layout_info_t)]),
    "fsdp_layout_param": (_ST, [_LAYOUT, ctypes.c_int32, ctypes.POINTER(fsdp_param_info_t)]),
    "fsdp_layout_bucket": (_ST, [_LAYOUT, ctypes.c_int32, ctypes.POINTER(fsdp_bucket_info_t)]),
    "fsdp_layout_group": (_ST, [_LAYOUT, ctypes.c_int32, ctypes.POINTER(fsdp_group_info_t)]),
    "fsdp_pack_reduce_scatter": (_ST, [_LAYOUT, ctypes.POINTER(_P), ctypes.POINTER(_P), _P]),
    "fsdp_allgather_copy_in": (_ST, [_LAYOUT, ctypes.POINTER(_P), _P, _P]),
    "fsdp_allgather_copy_out": (_ST, [_LAYOUT, _P, ctypes.POINTER(_P), _P]),
    "fsdp_reduce_scatter_copy_out": (_ST, [_LAYOUT, ctypes.POINTER(_P), ctypes.POINTER(_P), _P]),
    "fsdp_emulated_reduce_scatter": (_ST, [_LAYOUT, ctypes.POINTER(_P), ctypes.POINTER(_P), _P]),
    "fsdp_reduce_scatter_copy_out_batched": (_ST, [ctypes.POINTER(_LAYOUT), ctypes.c_int32, ctypes.POINTER(_P),
                                                   ctypes.POINTER(_P), _P]),
    "fsdp_pack_reduce_scatter_batched": (_ST, [ctypes.POINTER(_LAYOUT), ctypes.c_int32, ctypes.POINTER(_P),
                                               ctypes.POINTER(_P), _P]),
    "fsdp_allgather_copy_in_batched": (_ST, [ctypes.POINTER(_LAYOUT), ctypes.c_int32, ctypes.POINTER(_P),
                                             ctypes.POINTER(_P), _P]),
    "fsdp_allgather_copy_out_batched": (_ST, [ctypes.POINTER(_LAYOUT), ctypes.c_int32, ctypes.POINTER(_P),
                                              ctypes.POINTER(_P), _P]),
    "fsdp_pack_reduce_scatter_noalloc": (_ST, [_LAYOUT, ctypes.POINTER(_P), ctypes.POINTER(_P), _P]),
    "fsdp_sync_status": (_ST, [_LAYOUT, _P]),
    "fsdp_debug_set_wait_fault": (None, [ctypes.c_int32, ctypes.c_int64]),
    "fsdp_debug_set_upload_fault": (None, [ctypes.c_int32]),
    "fsdp_debug_set_schedule": (_ST, [ctypes.c_int32]),
    "fsdp_debug_set_grid_cap": (_ST, [ctypes.c_int32]),
    "fsdp_debug_stream_widen": (_ST, [_P, ctypes.c_int64, _P, _P]),
    "fsdp_layout_destroy": (None, [_LAYOUT]),
    "fsdp_status_string": (ctypes.c_char_p, [_ST]),
    "fsdp_last_error": (ctypes.c_char_p, []),
}
for _name, (_res, _args) in _SIGNATURES.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


class FsdpError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib.fsdp_last_error().decode()
        super().__init__(f"{where}: {fsdp_status_string(status)}" + (f" ({msg})" if msg else ""))


def _check(status: int, where: str) -> None:
    if status != FSDP_OK:
        raise FsdpError(status, where)


def fsdp_status_string(status: int) -> str:
    return _lib.fsdp_status_string(status).decode()


def fsdp_last_error() -> str:
    return _lib.fsdp_last_error().decode()


class Layout:
    """Owner of an ``fsdp_layout_t *``; destroyed on ``close()`` or collection.
    Keeps the parameter descriptors it was planned from, so that the entry
    points can check the buffers they are given against it."""

    def __init__(self, handle: int, n_params: int, descs=None):
        self.handle = handle
        self.n_params = n_params
        self.descs = [(d.numel, d.grad_dtype, d.reduce_dtype, d.shard_dtype, d.param_dtype)
                      for d in (descs or [])][:n_params]
        self._slots = None

    def close(self) -> None:
        if self.handle:
            _lib.fsdp_layout_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


def _descs(params):
    """Descriptors from fsdp_param_desc_t, (numel, g, rho, sigma, pi) tuples, or specs
    with numel and dtype-string attributes (workloads.ParamSpec)."""
    arr = (fsdp_param_desc_t * max(1, len(params)))()
    for k, p in enumerate(params):
        if isinstance(p, fsdp_param_desc_t):
            arr[k] = p
        elif isinstance(p, tuple):
            arr[k] = fsdp_param_desc_t(*p)
        else:
            arr[k] = fsdp_param_desc_t(p.numel, DTYPE_CODES[p.grad_dtype], DTYPE_CODES[p.reduce_dtype],
                                       DTYPE_CODES[p.shard_dtype], DTYPE_CODES[p.param_dtype])
    return arr


def fsdp_plan_layout(params, world_size: int) -> Layout:
    arr = _descs(params)
    out = _LAYOUT()
    _check(_lib.fsdp_plan_layout(arr, len(params), world_size, ctypes.byref(out)), "fsdp_plan_layout")
    return Layout(out.value, len(params), arr)


def fsdp_plan_layout_host(params, world_size: int) -> Layout:
    arr = _descs(params)
    out = _LAYOUT()
    _check(_lib.fsdp_plan_layout_host(arr, len(params), world_size, ctypes.byref(out)),
           "fsdp_plan_layout_host")
    return Layout(out.value, len(params), arr)


def fsdp_plan_layout_ex(params, world_size: int, row_elems=None, flags: int = 0) -> Layout:
    """row_elems: per-parameter elements per dim-0 row (0 = flattened), or None."""
    arr = _descs(params)
    rows = None
    if row_elems is not None:
        rows = (ctypes.c_int64 * max(1, len(row_elems)))(*row_elems)
    out = _LAYOUT()
    _check(_lib.fsdp_plan_layout_ex(arr, rows, len(params), world_size, flags, ctypes.byref(out)),
           "fsdp_plan_layout_ex")
    return Layout(out.value, len(params), arr)


def row_elems_of(specs):
    """Elements per dim-0 row of each spec's shape (1 for 1-D parameters)."""
    out = []
    for s in specs:
        r = 1
        for d in s.shape[1:]:
            r *= d
        out.append(r)
    return out


def fsdp_layout_query(layout: Layout) -> fsdp_layout_info_t:
    info = fsdp_layout_info_t()
    _check(_lib.fsdp_layout_query(layout.handle, ctypes.byref(info)), "fsdp_layout_query")
    return info


def fsdp_layout_param(layout: Layout, p: int) -> fsdp_param_info_t:
    info = fsdp_param_info_t()
    _check(_lib.fsdp_layout_param(layout.handle, p, ctypes.byref(info)), "fsdp_layout_param")
    return info


def fsdp_layout_bucket(layout: Layout, b: int) -> fsdp_bucket_info_t:
    info = fsdp_bucket_info_t()
    _check(_lib.fsdp_layout_bucket(layout.handle, b, ctypes.byref(info)), "fsdp_layout_bucket")
    return info


def fsdp_layout_group(layout: Layout, g: int) -> fsdp_group_info_t:
    info = fsdp_group_info_t()
    _check(_lib.fsdp_layout_group(layout.handle, g, ctypes.byref(info)), "fsdp_layout_group")
    return info


# ---------------------------------------------------------------------------
# Argument checks.  The C ABI takes bare pointers and reads as many as the
# layout has slots, so the binding checks what it can before the call: the
# number of pointers always, and for torch tensors their size, dtype,
# contiguity and device.  Integers and prebuilt pointer arrays are passed
# through unchecked beyond their count.
# ---------------------------------------------------------------------------
def _layout_slots(layout: Layout) -> dict:
    """Per slot list of one operation: (bytes, dtype code or None) of each slot."""
    if layout._slots is None:
        info = fsdp_layout_query(layout)
        W, d = info.world_size, layout.descs
        prm = [fsdp_layout_param(layout, p) for p in range(info.n_params)]
        bkt = [fsdp_layout_bucket(layout, b) for b in range(info.n_buckets)]
        sz = DTYPE_BYTES
        layout._slots = {
            "grads": [(n * sz[g], g) for n, g, _, _, _ in d],
            "buckets": [(b.bytes, b.reduce_dtype) for b in bkt],
            "shards": [(q.chunk * sz[x[3]], x[3]) for q, x in zip(prm, d)],
            "ag_input": [(info.ag_bytes, None)],
            "ag_output": [(W * info.ag_bytes, None)],
            "full": [(x[0] * sz[x[4]], x[4]) for x in d],
            "rows": [(b.row_elems * sz[b.reduce_dtype], b.reduce_dtype) for b in bkt],
            "sharded": [(q.chunk * sz[x[3]], x[3]) for q, x in zip(prm, d)],
            "packed": [(b.bytes, b.reduce_dtype) for b in bkt for _ in range(W)],
            "reduced": [(b.bytes, b.reduce_dtype) for b in bkt],
            "device": info.device if info.has_device_table else None,
        }
    return layout._slots


_FLOAT_CODES = None
_TENSOR_TYPE = [None]


def _float_codes() -> dict:
    """torch float dtype -> FSDP dtype code (built on first use, with the
    tensor type the checks recognise)."""
    global _FLOAT_CODES
    if _FLOAT_CODES is None:
        import torch
        _TENSOR_TYPE[0] = torch.Tensor
        _FLOAT_CODES = {torch.float32: FSDP_DTYPE_F32, torch.bfloat16: FSDP_DTYPE_BF16}
    return _FLOAT_CODES


def _dtype_name(dt: int) -> str:
    return "f32" if dt == FSDP_DTYPE_F32 else "bf16"


def _slot_name(what: str, k: int, single: bool) -> str:
    return what if single else f"{what}[{k}]"


def _scan_args(where: str, what: str, ts, slots, device):
    """Check ``ts`` (a list, a tensor or int for a single slot, or a prebuilt
    pointer array) against ``slots`` in one pass, gathering its pointers as it
    goes.  Returns (error, placement error, value for the C call): the first
    count, size, dtype or contiguity error and the first device error, each a
    message or None, and the pointer array or pointer to pass."""
    if ts is None or isinstance(ts, int):
        return None, None, ts
    if isinstance(ts, ctypes.Array):
        if len(slots) > len(ts):
            return f"{where}: {what} holds {len(ts)} pointers, the layout needs {len(slots)}", None, None
        return None, None, ts
    single = not isinstance(ts, (list, tuple))
    items = (ts,) if single else ts
    if len(items) != len(slots):
        return f"{where}: {len(items)} {what} given, the layout has {len(slots)}", None, None
    codes, tensor_type = _float_codes(), _TENSOR_TYPE[0]
    placement = None
    ptrs = []
    for k, t in enumerate(items):
        if not isinstance(t, tensor_type):
            ptrs.append(t)  # an int or None; anything else is refused by ctypes
            continue
        need, dt = slots[k]
        if not t.is_contiguous():
            return f"{where}: {_slot_name(what, k, single)} is not contiguous", None, None
        have = t.nbytes
        if have < need:
            return f"{where}: {_slot_name(what, k, single)} holds {have} bytes, the layout needs {need}", None, None
        if dt is not None:
            tdt = t.dtype
            code = codes.get(tdt)
            if code != dt and (code is not None or tdt.is_floating_point):
                return (f"{where}: {_slot_name(what, k, single)} is {tdt}, the layout's dtype is "
                        f"{_dtype_name(dt)} (pass raw bits as an integer tensor)"), None, None
        if placement is None and need:
            index = t.get_device()  # -1 off the GPU
            if index < 0:
                placement = f"{where}: {_slot_name(what, k, single)} is not a CUDA tensor"
            elif device is not None and index != device:
                placement = (f"{where}: {_slot_name(what, k, single)} is on cuda:{index}, "
                             f"the layout on cuda:{device}")
        ptrs.append(t.data_ptr())
    if single:
        return None, placement, ptrs[0]
    return None, placement, (_P * max(1, len(ptrs)))(*ptrs)


def _check_lists(where: str, slots: dict, lists: dict) -> list:
    """Raise ValueError for the first count, size, dtype or contiguity error
    of any list (in list order); only if there is none, for the first device
    error.  Returns the lists' values for the C call, in order."""
    device = slots["device"]
    placement = None
    values = []
    for what, ts in lists.items():
        err, perr, value = _scan_args(where, what, ts, slots.get(what, []), device)
        if err is not None:
            raise ValueError(err)
        if placement is None:
            placement = perr
        values.append(value)
    if placement is not None:
        raise ValueError(placement)
    return values


def _as_list(ts):
    """A per-layout argument of a batched call as a list (a lone tensor or
    pointer stands for a batch of one)."""
    return ts if isinstance(ts, (list, tuple, ctypes.Array)) else [ts]


def _marshal(ts):
    """The value for the C call without checks: a prebuilt array as is, a
    list as a pointer array, a single tensor or int as its pointer."""
    if isinstance(ts, ctypes.Array):
        return ts
    if isinstance(ts, (list, tuple)):
        return pointer_array(ts)
    return _ptr(ts)


def _layout_args(where: str, layout: Layout, **lists) -> list:
    """Check the lists against one layout and return them marshalled."""
    if not isinstance(layout, Layout) or not layout.handle:
        return [_marshal(ts) for ts in lists.values()]  # the C call reports a null or closed layout
    return _check_lists(where, _layout_slots(layout), lists)


def _batched_args(where: str, la: "LayoutArray", **lists) -> list:
    """Check the concatenated lists against a layout array and return them marshalled."""
    if not all(isinstance(L, Layout) and L.handle for L in la.layouts):
        return [_marshal(ts) for ts in lists.values()]  # the C call reports a null or closed layout
    if la.slots is None:  # the layouts' slot lists concatenated, once per array
        per = [_layout_slots(L) for L in la.layouts]
        devices = {s["device"] for s in per}
        la.slots = {k: [x for s in per for x in s[k]] for k in per[0] if k != "device"} if per else {}
        la.slots["device"] = devices.pop() if len(devices) == 1 else None
    return _check_lists(where, la.slots, lists)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def pointer_array(ts):
    """A C array of device pointers (tensors, ints or None); pass it in place
    of a list to skip re-marshalling on every call."""
    if isinstance(ts, ctypes.Array):
        return ts
    if not ts:
        return (_P * 1)()
    return (_P * len(ts))(*[t if t is None or isinstance(t, int) else t.data_ptr() for t in ts])


_current_stream_fn = None


def _current_stream() -> int:
    """torch's current CUDA stream on the current device, as a handle.  The
    first call takes it through torch.cuda (which initialises CUDA); later
    calls read the raw handle directly when this torch build exposes it and
    it agreed with torch.cuda on that first call."""
    global _current_stream_fn
    if _current_stream_fn is None:
        import torch
        public = torch.cuda.current_stream().cuda_stream
        raw, dev = getattr(torch._C, "_cuda_getCurrentRawStream", None), getattr(torch._C, "_cuda_getDevice", None)
        if raw is not None and dev is not None and raw(dev()) == public:
            _current_stream_fn = lambda: raw(dev())  # noqa: E731
        else:
            _current_stream_fn = lambda: torch.cuda.current_stream().cuda_stream  # noqa: E731
        return public
    return _current_stream_fn()


def _stream(stream) -> int | None:
    if stream is None:
        return _current_stream()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def fsdp_pack_reduce_scatter(layout: Layout, grads, bucket_bufs, stream=None) -> None:
    g, b = _layout_args("fsdp_pack_reduce_scatter", layout, grads=grads, buckets=bucket_bufs)
    _check(_lib.fsdp_pack_reduce_scatter(layout.handle, g, b, _stream(stream)), "fsdp_pack_reduce_scatter")


def fsdp_allgather_copy_in(layout: Layout, local_shards, ag_input, stream=None) -> None:
    sh, a = _layout_args("fsdp_allgather_copy_in", layout, shards=local_shards, ag_input=ag_input)
    _check(_lib.fsdp_allgather_copy_in(layout.handle, sh, a, _stream(stream)), "fsdp_allgather_copy_in")


def fsdp_allgather_copy_out(layout: Layout, ag_output, full_params, stream=None) -> None:
    a, f = _layout_args("fsdp_allgather_copy_out", layout, ag_output=ag_output, full=full_params)
    _check(_lib.fsdp_allgather_copy_out(layout.handle, a, f, _stream(stream)), "fsdp_allgather_copy_out")


def fsdp_reduce_scatter_copy_out(layout: Layout, reduced_rows, sharded_grads, stream=None) -> None:
    r, sg = _layout_args("fsdp_reduce_scatter_copy_out", layout, rows=reduced_rows, sharded=sharded_grads)
    _check(_lib.fsdp_reduce_scatter_copy_out(layout.handle, r, sg, _stream(stream)), "fsdp_reduce_scatter_copy_out")


def fsdp_emulated_reduce_scatter(layout: Layout, packed, reduced, stream=None) -> None:
    """packed: n_buckets * W pointers, bucket-major (packed[b*W + q] = rank q's
    bucket b); reduced: one [W, S_b] buffer per bucket."""
    pk, rd = _layout_args("fsdp_emulated_reduce_scatter", layout, packed=packed, reduced=reduced)
    _check(_lib.fsdp_emulated_reduce_scatter(layout.handle, pk, rd, _stream(stream)), "fsdp_emulated_reduce_scatter")


class LayoutArray:
    """A C array of layout handles plus its length; pass it in place of a
    list of layouts to skip re-marshalling on every batched call."""

    def __init__(self, layouts):
        self.n = len(layouts)
        self.layouts = list(layouts)
        self.slots = None
        self.arr = (_LAYOUT * max(1, self.n))()
        for k, L in enumerate(layouts):
            self.arr[k] = L.handle


def layout_array(layouts) -> LayoutArray:
    return layouts if isinstance(layouts, LayoutArray) else LayoutArray(layouts)


def fsdp_pack_reduce_scatter_batched(layouts, grads, bucket_bufs, stream=None) -> None:
    """grads / bucket_bufs: the per-layout lists concatenated in layout order."""
    la = layout_array(layouts)
    g, b = _batched_args("fsdp_pack_reduce_scatter_batched", la, grads=grads, buckets=bucket_bufs)
    _check(_lib.fsdp_pack_reduce_scatter_batched(la.arr, la.n, g, b, _stream(stream)),
           "fsdp_pack_reduce_scatter_batched")


def fsdp_allgather_copy_in_batched(layouts, local_shards, ag_inputs, stream=None) -> None:
    """local_shards concatenated in layout order; one ag_input per layout."""
    la = layout_array(layouts)
    sh, a = _batched_args("fsdp_allgather_copy_in_batched", la, shards=local_shards, ag_input=_as_list(ag_inputs))
    _check(_lib.fsdp_allgather_copy_in_batched(la.arr, la.n, sh, a, _stream(stream)),
           "fsdp_allgather_copy_in_batched")


def fsdp_allgather_copy_out_batched(layouts, ag_outputs, full_params, stream=None) -> None:
    """One ag_output per layout; full_params concatenated in layout order."""
    la = layout_array(layouts)
    a, f = _batched_args("fsdp_allgather_copy_out_batched", la, ag_output=_as_list(ag_outputs), full=full_params)
    _check(_lib.fsdp_allgather_copy_out_batched(la.arr, la.n, a, f, _stream(stream)),
           "fsdp_allgather_copy_out_batched")


def fsdp_reduce_scatter_copy_out_batched(layouts, reduced_rows, sharded_grads, stream=None) -> None:
    """reduced_rows / sharded_grads: the per-layout lists concatenated in layout order."""
    la = layout_array(layouts)
    r, sg = _batched_args("fsdp_reduce_scatter_copy_out_batched", la, rows=reduced_rows, sharded=sharded_grads)
    _check(_lib.fsdp_reduce_scatter_copy_out_batched(la.arr, la.n, r, sg, _stream(stream)),
           "fsdp_reduce_scatter_copy_out_batched")


def fsdp_pack_reduce_scatter_noalloc(layout: Layout, grads, bucket_bufs, stream=None) -> None:
    """The pack with its scratch in the library's static array (no allocation)."""
    g, b = _layout_args("fsdp_pack_reduce_scatter_noalloc", layout, grads=grads, buckets=bucket_bufs)
    _check(_lib.fsdp_pack_reduce_scatter_noalloc(layout.handle, g, b, _stream(stream)),
           "fsdp_pack_reduce_scatter_noalloc")


def fsdp_sync_status(layout: Layout, stream=None) -> None:
    _check(_lib.fsdp_sync_status(layout.handle, _stream(stream)), "fsdp_sync_status")


def fsdp_debug_set_wait_fault(fault: int, wait_limit_ns: int) -> None:
    _lib.fsdp_debug_set_wait_fault(fault, wait_limit_ns)


def fsdp_debug_set_upload_fault(fail_upload: bool) -> None:
    _lib.fsdp_debug_set_upload_fault(1 if fail_upload else 0)


def fsdp_debug_set_schedule(mode: int) -> None:
    _check(_lib.fsdp_debug_set_schedule(mode), "fsdp_debug_set_schedule")


def fsdp_debug_set_grid_cap(max_blocks: int) -> None:
    """Run every table-driven launch on at most max_blocks blocks (0: the
    planned grid); a test hook."""
    _check(_lib.fsdp_debug_set_grid_cap(max_blocks), "fsdp_debug_set_grid_cap")


def fsdp_debug_stream_widen(src, n: int, dst, stream=None) -> None:
    """Plain BF16 -> FP32 streaming widen of n elements (a measurement
    utility: the pack's 1 : 2 byte mix without its layout)."""
    _check(_lib.fsdp_debug_stream_widen(_ptr(src), n, _ptr(dst), _stream(stream)), "fsdp_debug_stream_widen")


def fsdp_layout_destroy(layout: Layout) -> None:
    layout.close()
