"""The C-ABI library without a GPU: it builds, loads, exports every symbol
that include/*.h declares, plans layouts on the host exactly as the oracle
does, and rejects bad arguments with the documented status codes."""
import ctypes
import glob
import os
import re

import pytest

import oracle
from fsdp2_gradient_packing_gb300 import _build
from fsdp2_gradient_packing_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def fp():
    _build.build()
    from fsdp2_gradient_packing_gb300 import fsdp_pack
    return fsdp_pack


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w \t\*]*?\b(fsdp_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol(fp):
    names = declared_functions()
    assert "fsdp_pack_reduce_scatter" in names and len(names) >= 10
    lib = ctypes.CDLL(_build.LIB)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_has_a_function_per_entry_point(fp):
    for n in declared_functions():
        assert callable(getattr(fp, n)), n


def _compare_with_oracle(fp, specs, W, rows=False):
    row_elems = fp.row_elems_of(specs) if rows else None
    pl = oracle.plan(oracle.params_from_specs(specs), W, row_elems=row_elems)
    plan = (lambda: fp.fsdp_plan_layout_ex(specs, W, row_elems, fp.FSDP_PLAN_HOST_ONLY)) if rows else \
        (lambda: fp.fsdp_plan_layout_host(specs, W))
    with plan() as L:
        info = fp.fsdp_layout_query(L)
        assert info.world_size == W and info.n_params == len(specs)
        assert info.n_buckets == len(pl.bucket_dtype) and info.n_groups == len(pl.group_pair)
        assert info.ag_bytes == pl.S_ag and info.has_device_table == 0 and info.device == -1
        assert info.total_numel == sum(s.numel for s in specs)
        for p in range(len(specs)):
            pi = fp.fsdp_layout_param(L, p)
            assert pi.chunk == pl.chunk[p]
            assert (pi.bucket, pi.bucket_offset) == (pl.bucket_of[p], pl.bucket_off[p])
            assert (pi.group, pi.group_offset) == (pl.group_of[p], pl.group_elem_off[p])
            g = pl.group_of[p]
            assert pi.ag_byte_offset == pl.group_byte_off[g] + pl.group_elem_off[p] * oracle.DTYPE_SIZE[pl.group_pair[g][1]]
        for b in range(info.n_buckets):
            bi = fp.fsdp_layout_bucket(L, b)
            assert bi.reduce_dtype == pl.bucket_dtype[b] and bi.row_elems == pl.bucket_S[b]
            assert bi.bytes == W * pl.bucket_S[b] * oracle.DTYPE_SIZE[pl.bucket_dtype[b]]
            assert bi.n_params == pl.bucket_of.count(b)
        for g in range(info.n_groups):
            gi = fp.fsdp_layout_group(L, g)
            assert (gi.shard_dtype, gi.param_dtype) == pl.group_pair[g]
            assert gi.byte_offset == pl.group_byte_off[g] and gi.elems == pl.group_elems[g]


@pytest.mark.parametrize("make", [
    lambda: wl.tiny_two_blocks(grouping="linear"), lambda: wl.tiny_two_blocks(grouping="block"),
    lambda: wl.tiny_two_blocks(grouping="model"), lambda: wl.transformer_500(),
    lambda: wl.mixed_50m(), lambda: wl.kda_block(W=8, reduce="grad"),
    lambda: wl.kda_block(W=64, reduce="f32"), lambda: wl.kda_block(W=64, reduce="bf16"),
])
def test_host_plan_matches_oracle_on_workloads(fp, make):
    work = make()
    for g in work.groups:
        _compare_with_oracle(fp, g, work.W)


def test_host_plan_matches_oracle_on_random_layouts(fp):
    for seed in range(400):
        work = wl.random_layout(seed)
        _compare_with_oracle(fp, work.groups[0], work.W)


def test_row_mode_host_plan_matches_oracle(fp):
    for seed in range(300):
        work = wl.random_layout_2d(seed)
        _compare_with_oracle(fp, work.groups[0], work.W, rows=True)
    for make in (lambda: wl.transformer_500(W=7, layers=2), lambda: wl.kda_block(W=64, d=512, ffn=1536)):
        work = make()
        for g in work.groups:
            _compare_with_oracle(fp, g, work.W, rows=True)


def test_row_mode_rejects_bad_rows_and_flags(fp):
    specs = [wl.ParamSpec("w", (6, 6))]
    for rows, flags in (([-1], 1), ([7], 1), ([6], 1 | 2)):
        with pytest.raises(fp.FsdpError) as e:
            fp.fsdp_plan_layout_ex(specs, 4, rows, flags)
        assert e.value.status == fp.FSDP_EINVAL
    with fp.fsdp_plan_layout_ex(specs, 4, [6], fp.FSDP_PLAN_HOST_ONLY) as L:
        assert fp.fsdp_layout_param(L, 0).chunk == 12
    with fp.fsdp_plan_layout_ex(specs, 4, [0], fp.FSDP_PLAN_HOST_ONLY) as L:
        assert fp.fsdp_layout_param(L, 0).chunk == 9


def test_empty_layout(fp):
    with fp.fsdp_plan_layout_host([], 4) as L:
        info = fp.fsdp_layout_query(L)
        assert (info.n_params, info.n_buckets, info.n_groups, info.ag_bytes) == (0, 0, 0, 0)
        assert (info.pack_items, info.copy_in_items, info.copy_out_items) == (0, 0, 0)


def test_work_items_cover_the_buffers(fp):
    # Pack items are (rank, parameter) runs cut to at most 16 KiB of
    # destination and 16 KiB of source: the counts follow from the run lengths.
    work = wl.mixed_50m()
    with fp.fsdp_plan_layout_host(work.groups[0], 8) as L:
        info = fp.fsdp_layout_query(L)
        # 8 ranks x (24 BF16 matrices of 131072 or 524288 elements per rank, cut
        # at 4096 elements) + 8 ranks x 8 norms of 128 elements
        runs_bf16 = 8 * 4 * (4 * 131072 + 2 * 524288) // 4096
        assert info.pack_items == runs_bf16 + 8 * 8


@pytest.mark.parametrize("bad,status", [
    (dict(W=0), "FSDP_EINVAL"),
    (dict(numel=-1), "FSDP_EINVAL"),
    (dict(dtype=7), "FSDP_EINVAL"),
    (dict(n=4001), "FSDP_EUNSUPPORTED"),
])
def test_plan_rejects_bad_arguments(fp, bad, status):
    W = bad.get("W", 4)
    n = bad.get("n", 3)
    descs = [fp.fsdp_param_desc_t(bad.get("numel", 10), bad.get("dtype", 0), 0, 0, 0) for _ in range(n)]
    with pytest.raises(fp.FsdpError) as e:
        fp.fsdp_plan_layout_host(descs, W)
    assert fp.fsdp_status_string(e.value.status) == status
    assert fp.fsdp_last_error()


def test_entry_points_reject_host_only_layout_without_launching(fp):
    with fp.fsdp_plan_layout_host(wl.tiny_two_blocks().groups[0], 4) as L:
        with pytest.raises(fp.FsdpError) as e:
            fp.fsdp_pack_reduce_scatter(L, [0x1000], [0x2000], stream=0)
        assert e.value.status == fp.FSDP_EINVAL
        with pytest.raises(fp.FsdpError):
            fp.fsdp_allgather_copy_in(L, [0x1000], 0x2000, stream=0)
        with pytest.raises(fp.FsdpError):
            fp.fsdp_allgather_copy_out(L, 0x2000, [0x1000], stream=0)


def test_batched_calls_check_their_arguments_without_launching(fp):
    specs = wl.tiny_two_blocks(grouping="model").groups[0]
    layouts = [fp.fsdp_plan_layout_host(specs, 4) for _ in range(65)]
    try:
        with pytest.raises(fp.FsdpError) as e:
            fp.fsdp_pack_reduce_scatter_batched(layouts, [0x1000] * (4 * 65), [0x2000] * 65, stream=0)
        assert e.value.status == fp.FSDP_EUNSUPPORTED          # more than 64 layouts
        for call, args in ((fp.fsdp_pack_reduce_scatter_batched, ([0x1000] * 8, [0x2000] * 2)),
                           (fp.fsdp_allgather_copy_in_batched, ([0x1000] * 8, [0x2000] * 2)),
                           (fp.fsdp_allgather_copy_out_batched, ([0x2000] * 2, [0x1000] * 8))):
            with pytest.raises(fp.FsdpError) as e:
                call(layouts[:2], *args, stream=0)
            assert e.value.status == fp.FSDP_EINVAL             # host-only layouts
    finally:
        for L in layouts:
            L.close()


def test_binding_checks_pointer_counts_and_tensors_before_calling(fp):
    """The C entry points read as many pointers as the layout has slots, so
    the binding refuses short lists (and short prebuilt arrays) of any kind,
    and checks torch tensors against the layout: size, floating dtype,
    contiguity, device.  All of it happens before the C call."""
    import torch
    specs = wl.tiny_two_blocks(grouping="block").groups[1]       # BF16 grads, FP32 bucket
    W = 4
    with fp.fsdp_plan_layout_host(specs, W) as L:
        b = fp.fsdp_layout_bucket(L, 0)
        grads = [torch.zeros(s.numel, dtype=torch.bfloat16) for s in specs]
        bucket = torch.zeros(b.bytes // 4, dtype=torch.float32)
        cases = [
            (([grads[0]], [bucket]), "1 grads given, the layout has 2"),
            (([0x1000], [0x2000]), "1 grads given, the layout has 2"),
            ((fp.pointer_array([0x1000]), [bucket]), "holds 1 pointers, the layout needs 2"),
            (([grads[0], grads[1][:-1]], [bucket]), "grads[1] holds 70 bytes, the layout needs 72"),
            (([grads[0], grads[1].float()], [bucket]), "grads[1] is torch.float32, the layout's dtype is bf16"),
            ((grads, [bucket[:-1]]), f"buckets[0] holds {b.bytes - 4} bytes, the layout needs {b.bytes}"),
            ((grads, [torch.zeros(b.bytes // 2, dtype=torch.bfloat16)]),
             "buckets[0] is torch.bfloat16, the layout's dtype is f32"),
            ((grads, [torch.zeros(2 * (b.bytes // 4), dtype=torch.float32)[::2]]), "buckets[0] is not contiguous"),
            ((grads, [bucket]), "grads[0] is not a CUDA tensor"),
            (([g.view(torch.int16) for g in grads], [bucket.view(torch.uint8)]), "grads[0] is not a CUDA tensor"),
        ]
        for args, msg in cases:
            with pytest.raises(ValueError, match=re.escape(msg)):
                fp.fsdp_pack_reduce_scatter(L, *args, stream=0)
        c = [fp.fsdp_layout_param(L, p).chunk for p in range(2)]
        S_ag = fp.fsdp_layout_query(L).ag_bytes
        with pytest.raises(ValueError, match="ag_input holds 8 bytes"):
            fp.fsdp_allgather_copy_in(L, [torch.zeros(ci) for ci in c], torch.zeros(2), stream=0)
        with pytest.raises(ValueError, match=re.escape(f"ag_output holds {W * S_ag - 1} bytes")):
            fp.fsdp_allgather_copy_out(L, torch.zeros(W * S_ag - 1, dtype=torch.uint8), [0x1000, 0x2000], stream=0)
        with pytest.raises(ValueError, match="full\\[1\\] is torch.float32, the layout's dtype is bf16"):
            fp.fsdp_allgather_copy_out(L, 0x1000, [torch.zeros(36, dtype=torch.bfloat16), torch.zeros(36)], stream=0)
        with pytest.raises(ValueError, match="3 rows given, the layout has 1"):
            fp.fsdp_reduce_scatter_copy_out(L, [0x1000] * 3, [0x2000] * 2, stream=0)
        with pytest.raises(ValueError, match=f"{W - 1} packed given, the layout has {W}"):
            fp.fsdp_emulated_reduce_scatter(L, [0x1000] * (W - 1), [0x2000], stream=0)
        with pytest.raises(ValueError, match="1 grads given, the layout has 2"):
            fp.fsdp_pack_reduce_scatter_noalloc(L, [0x1000], [0x2000], stream=0)
        # Batched: the lists are the layouts' lists concatenated.
        with pytest.raises(ValueError, match="3 grads given, the layout has 4"):
            fp.fsdp_pack_reduce_scatter_batched([L, L], [0x1000] * 3, [0x2000] * 2, stream=0)
        with pytest.raises(ValueError, match="grads\\[3\\] holds 70 bytes"):
            fp.fsdp_pack_reduce_scatter_batched(fp.layout_array([L, L]), grads + [grads[0], grads[1][:-1]],
                                                [bucket, bucket], stream=0)
        # Right counts of plain integers reach the library, which refuses a host-only layout.
        with pytest.raises(fp.FsdpError):
            fp.fsdp_pack_reduce_scatter(L, [0x1000, 0x2000], [0x3000], stream=0)


def test_query_index_out_of_range(fp):
    with fp.fsdp_plan_layout_host(wl.tiny_two_blocks().groups[0], 4) as L:
        for fn in (fp.fsdp_layout_param, fp.fsdp_layout_bucket, fp.fsdp_layout_group):
            with pytest.raises(fp.FsdpError):
                fn(L, 99)
            with pytest.raises(fp.FsdpError):
                fn(L, -1)


def test_status_strings(fp):
    names = [fp.fsdp_status_string(s) for s in range(6)]
    assert names == ["FSDP_OK", "FSDP_EINVAL", "FSDP_ENOMEM", "FSDP_ECUDA", "FSDP_EUNSUPPORTED", "FSDP_ETIMEOUT"]
    assert fp.fsdp_status_string(99) == "FSDP_UNKNOWN_STATUS"


def test_plan_without_gpu_reports_cuda_error(fp):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is visible")
    with pytest.raises(fp.FsdpError) as e:
        fp.fsdp_plan_layout(wl.tiny_two_blocks().groups[0], 4)
    assert e.value.status == fp.FSDP_ECUDA


def test_schedule_hook_accepts_its_modes_and_refuses_others(fp):
    for mode in (fp.FSDP_SCHEDULE_FIXED, fp.FSDP_SCHEDULE_SHARED, fp.FSDP_SCHEDULE_MIXED,
                 fp.FSDP_SCHEDULE_DEFAULT):
        fp.fsdp_debug_set_schedule(mode)
    for bad in (-1, 4, 1 << 20):
        with pytest.raises(fp.FsdpError) as e:
            fp.fsdp_debug_set_schedule(bad)
        assert e.value.status == fp.FSDP_EINVAL and "unknown schedule mode" in str(e.value)


def test_stream_widen_checks_its_arguments_without_launching(fp):
    fp.fsdp_debug_stream_widen(0, 0, 0, stream=0)  # n = 0: nothing to do, no CUDA call
    for src, n, dst, why in ((0x1000, 12, 0x100000, "multiple of 8"), (0x1000, -8, 0x100000, "multiple of 8"),
                             (0x1008, 16, 0x100000, "16-byte aligned"), (0x1000, 16, 0x100004, "16-byte aligned"),
                             (0, 16, 0x100000, "NULL"), (0x1000, 64, 0x1040, "overlap")):
        with pytest.raises(fp.FsdpError) as e:
            fp.fsdp_debug_stream_widen(src, n, dst, stream=0)
        assert e.value.status == fp.FSDP_EINVAL and why in str(e.value), (src, n, dst)



def test_grid_cap_hook_accepts_counts_and_refuses_negative(fp):
    for cap in (1, 7, 456, 1 << 30, 0):
        fp.fsdp_debug_set_grid_cap(cap)
    for bad in (-1, -(1 << 20)):
        with pytest.raises(fp.FsdpError) as e:
            fp.fsdp_debug_set_grid_cap(bad)
        assert e.value.status == fp.FSDP_EINVAL and "grid cap" in str(e.value)
    fp.fsdp_debug_set_grid_cap(0)
