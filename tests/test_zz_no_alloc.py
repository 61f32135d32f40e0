"""The allocation-free pack entry point, through the C ABI, against the
regular one.

fsdp_pack_reduce_scatter_noalloc serves callers that cannot allocate device
memory when they pack (a device memory budget owned by another component,
allocator callbacks, runtimes that forbid allocation after start-up): its
kernel keeps its work table and status word in a fixed array inside the
library.  Two calls in a row, on two different layouts planned without any
CUDA call, must each give exactly the regular entry point's result.  The
first layout has the longer work table, so the second call runs with the
first call's items still in the array past its own; and the second call
must leave free device memory unchanged.  This file is named to be collected
last.
"""
import numpy as np
import pytest
import torch

from fsdp2_gradient_packing_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _inputs(work, specs):
    return [torch.from_numpy(wl.grad_values(work, 0, i, specials=0.02).view(
        np.int16 if s.grad_dtype == "bf16" else np.int32).copy()).cuda() for i, s in enumerate(specs)]


def _buckets(fp, L, fill):
    info = fp.fsdp_layout_query(L)
    return [torch.full((fp.fsdp_layout_bucket(L, b).bytes,), fill, dtype=torch.uint8, device="cuda")
            for b in range(info.n_buckets)]


def test_noalloc_pack_matches_regular_pack_on_two_calls_in_a_row():
    from fsdp2_gradient_packing_gb300 import _build
    _build.build()
    from fsdp2_gradient_packing_gb300 import fsdp_pack as fp

    cases = [wl.transformer_500(W=8, layers=1), wl.kda_block(W=64, reduce="grad", d=512, ffn=1536)]
    host_layouts, grads, want, got = [], [], [], []
    try:
        for work in cases:
            specs = work.groups[0]
            g = _inputs(work, specs)
            with fp.fsdp_plan_layout(specs, work.W) as L_regular:
                w = _buckets(fp, L_regular, 0xA5)
                fp.fsdp_pack_reduce_scatter(L_regular, g, w)
                fp.fsdp_sync_status(L_regular)
            L_host = fp.fsdp_plan_layout_host(specs, work.W)
            host_layouts.append(L_host)
            grads.append(g)
            want.append(w)
            got.append(_buckets(fp, L_host, 0x5A))
        items = [fp.fsdp_layout_query(L).pack_items for L in host_layouts]
        assert items[0] > items[1], "the first call must leave items past the second call's table"

        torch.cuda.synchronize()
        fp.fsdp_pack_reduce_scatter_noalloc(host_layouts[0], grads[0], got[0])
        torch.cuda.synchronize()
        free_before, _ = torch.cuda.mem_get_info()  # the first call on a device may load the library's module
        fp.fsdp_pack_reduce_scatter_noalloc(host_layouts[1], grads[1], got[1])
        torch.cuda.synchronize()
        free_after, _ = torch.cuda.mem_get_info()

        for n in range(2):
            for b, (x, y) in enumerate(zip(got[n], want[n])):
                assert torch.equal(x, y), f"call {n}, bucket {b} differs from the regular pack"
        assert free_after == free_before, "the no-alloc pack changed free device memory"
    finally:
        for L in host_layouts:
            L.close()


def test_noalloc_rejects_a_table_beyond_its_scratch():
    from fsdp2_gradient_packing_gb300 import fsdp_pack as fp
    # At least 131,065 items of at most 4096 BF16 elements: more than the
    # array holds (131,064).
    specs = [wl.ParamSpec("big", (131_065 * 4096,), "bf16", "f32")]
    with fp.fsdp_plan_layout_host(specs, 1) as L:
        assert fp.fsdp_layout_query(L).pack_items > 131_064
        with pytest.raises(fp.FsdpError) as e:
            fp.fsdp_pack_reduce_scatter_noalloc(L, [0x1000], [0x2000])
        assert e.value.status == fp.FSDP_EUNSUPPORTED
