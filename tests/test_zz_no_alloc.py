"""The allocation-free pack entry point, through the C ABI, against the
oracle.

fsdp_pack_reduce_scatter_noalloc serves callers that cannot allocate device
memory when they pack (a device memory budget owned by another component,
allocator callbacks, runtimes that forbid allocation after start-up): its
kernel keeps its work table and status word in a fixed array inside the
library.  The cases:
  * two calls in a row, on two different layouts planned without any CUDA
    call, each equal to the oracle's pack (and to the regular entry point's);
    the first layout has the longer work table, so the second call runs with
    the first call's items still in the array past its own, and the second
    call must leave free device memory unchanged;
  * a call queued on the same stream right behind a regular pack launch,
    with no synchronisation between them;
  * a layout of exactly as many work items as the array holds, with a ragged
    last item;
  * a layout one item too large, refused before anything is launched;
  * calls on grids cut short by the test hook, so that every block walks
    many of the array's items.
This file is named to be collected last.
"""
import numpy as np
import pytest
import torch

import oracle
from fsdp2_gradient_packing_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

NP = {"f32": np.uint32, "bf16": np.uint16}
CAPACITY = 131_064  # work items the library's scratch array holds


@pytest.fixture(scope="module")
def fp():
    from fsdp2_gradient_packing_gb300 import _build
    _build.build()
    from fsdp2_gradient_packing_gb300 import fsdp_pack
    return fsdp_pack


def _inputs(work, specs):
    host = [wl.grad_values(work, 0, i, specials=0.02) for i in range(len(specs))]
    dev = [torch.from_numpy(h.view(np.int16 if s.grad_dtype == "bf16" else np.int32).copy()).cuda()
           for h, s in zip(host, specs)]
    return host, dev


def _buckets(fp, L, fill):
    info = fp.fsdp_layout_query(L)
    return [torch.full((fp.fsdp_layout_bucket(L, b).bytes,), fill, dtype=torch.uint8, device="cuda")
            for b in range(info.n_buckets)]


def _expected(specs, W, host_grads):
    pl = oracle.plan(oracle.params_from_specs(specs), W)
    return pl, oracle.pack_reduce_scatter(pl, host_grads)


def _assert_equal_to_oracle(got, want, what):
    for b, (x, y) in enumerate(zip(got, want)):
        g = x.cpu().numpy().view(y.dtype)
        assert np.array_equal(g, y), f"{what}, bucket {b}: {int(np.count_nonzero(g != y))} elements differ"


def test_noalloc_pack_matches_oracle_on_two_calls_in_a_row(fp):
    cases = [wl.transformer_500(W=8, layers=1), wl.kda_block(W=64, reduce="grad", d=512, ffn=1536)]
    host_layouts, grads, want, regular, got = [], [], [], [], []
    try:
        for work in cases:
            specs = work.groups[0]
            h, g = _inputs(work, specs)
            _, w = _expected(specs, work.W, h)
            with fp.fsdp_plan_layout(specs, work.W) as L_regular:
                r = _buckets(fp, L_regular, 0xA5)
                fp.fsdp_pack_reduce_scatter(L_regular, g, r)
                fp.fsdp_sync_status(L_regular)
            L_host = fp.fsdp_plan_layout_host(specs, work.W)
            host_layouts.append(L_host)
            grads.append(g)
            want.append(w)
            regular.append(r)
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
            _assert_equal_to_oracle(got[n], want[n], f"no-alloc call {n}")
            for b, (x, y) in enumerate(zip(got[n], regular[n])):
                assert torch.equal(x, y), f"call {n}, bucket {b} differs from the regular pack"
        assert free_after == free_before, "the no-alloc pack changed free device memory"
    finally:
        for L in host_layouts:
            L.close()


def test_noalloc_pack_right_behind_a_regular_pack_on_one_stream(fp):
    """A regular pack (its kernel walks the layout's own table) and then a
    no-alloc pack of another layout, queued back to back on one side stream
    with nothing between them; both outputs must equal the oracle's."""
    w1 = wl.transformer_500(W=8, layers=1)
    w2 = wl.mixed_50m(W=8, layers=1)
    s1, s2 = w1.groups[0], w2.groups[0]
    h1, g1 = _inputs(w1, s1)
    h2, g2 = _inputs(w2, s2)
    _, want1 = _expected(s1, w1.W, h1)
    _, want2 = _expected(s2, w2.W, h2)
    stream = torch.cuda.Stream()
    with fp.fsdp_plan_layout(s1, w1.W) as L1, fp.fsdp_plan_layout_host(s2, w2.W) as L2:
        out1, out2 = _buckets(fp, L1, 0xA5), _buckets(fp, L2, 0x5A)
        torch.cuda.synchronize()
        for _ in range(3):
            fp.fsdp_pack_reduce_scatter(L1, g1, out1, stream)
            fp.fsdp_pack_reduce_scatter_noalloc(L2, g2, out2, stream)
        stream.synchronize()
        fp.fsdp_sync_status(L1, stream)
        _assert_equal_to_oracle(out1, want1, "regular pack")
        _assert_equal_to_oracle(out2, want2, "no-alloc pack after a regular pack")


def test_noalloc_pack_at_full_capacity(fp):
    """One BF16 gradient of 536,838,143 elements reduced in FP32 at W = 1: its
    pack table has exactly the array's capacity of work items (4,096
    elements each, the last one ragged)."""
    n = CAPACITY * 4096 - 1
    specs = [wl.ParamSpec("big", (n,), "bf16", "f32")]
    g = wl.device_normal_bits(n, "bf16", 1.0, 1005, 0, 0, 1)
    with fp.fsdp_plan_layout_host(specs, 1) as L:
        assert fp.fsdp_layout_query(L).pack_items == CAPACITY
        out = _buckets(fp, L, 0x5A)
        fp.fsdp_pack_reduce_scatter_noalloc(L, [g], out)
        torch.cuda.synchronize()
        host = g.cpu().numpy().view(np.uint16)
        del g
        got = out[0].cpu().numpy().view(np.uint32)
        del out
    pl = oracle.plan(oracle.params_from_specs(specs), 1)
    want = oracle.pack_reduce_scatter(pl, [host])[0]
    assert got.shape == want.shape
    assert np.array_equal(got, want), f"{int(np.count_nonzero(got != want))} elements differ"


def test_noalloc_rejects_a_table_beyond_its_scratch(fp):
    # At least 131,065 items of at most 4096 BF16 elements: more than the
    # array holds (131,064).
    specs = [wl.ParamSpec("big", (CAPACITY * 4096 + 1,), "bf16", "f32")]
    with fp.fsdp_plan_layout_host(specs, 1) as L:
        assert fp.fsdp_layout_query(L).pack_items > CAPACITY
        with pytest.raises(fp.FsdpError) as e:
            fp.fsdp_pack_reduce_scatter_noalloc(L, [0x1000], [0x2000])
        assert e.value.status == fp.FSDP_EUNSUPPORTED


@pytest.mark.parametrize("blocks", [1, 5, 40])
def test_noalloc_pack_on_few_blocks(fp, blocks):
    """One layer of the ~500-parameter layout (913 pack items) on 1, 5 and
    40 blocks: every block walks many of the array's items in the fixed
    order."""
    work = wl.transformer_500(W=8, layers=1)
    specs = work.groups[0]
    h, g = _inputs(work, specs)
    _, want = _expected(specs, work.W, h)
    fp.fsdp_debug_set_grid_cap(blocks)
    try:
        with fp.fsdp_plan_layout_host(specs, work.W) as L:
            out = _buckets(fp, L, 0x5A)
            fp.fsdp_pack_reduce_scatter_noalloc(L, g, out)
            torch.cuda.synchronize()
    finally:
        fp.fsdp_debug_set_grid_cap(0)
    _assert_equal_to_oracle(out, want, f"no-alloc pack on {blocks} blocks")
