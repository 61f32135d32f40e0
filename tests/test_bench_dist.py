"""bench.py's multi-rank plumbing on CPU: two gloo ranks, a barrier and the
max over ranks that the timing uses (the path itself is replicas only)."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    assert bench.dist_env() == (rank, world, rank)
    assert bench.init_dist("gloo") == world
    bench.barrier()
    out[rank] = bench.max_over_ranks(10.0 + 5 * rank)
    import torch.distributed as dist
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_max_over_ranks_with_gloo(world):
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert [out[r] for r in range(world)] == [10.0 + 5 * (world - 1)] * world


def test_single_process_max_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5


def test_reference_arm_prints_one_line(capsys):
    sys.path.insert(0, ROOT)
    import json

    import bench
    bench.main(["--impl", "reference", "--steps", "40", "--warmup", "2"])
    lines = [l for l in capsys.readouterr().out.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["metric"] == bench.METRIC and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1


def test_reference_arm_runs_on_rank_0_only(capsys, monkeypatch):
    """Under torchrun with N > 1 the reference arm (the CPU oracle) runs and
    prints on rank 0 alone; any other rank returns at once, printing nothing."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    bench.main(["--impl", "reference", "--gpus", "2", "--steps", "40", "--warmup", "2"])
    assert capsys.readouterr().out.strip() == ""


def test_reference_arm_config_equals_our_arms(capsys):
    """Both arms print the same `config` for the same flags.  The reference arm
    takes the pack's bytes from the oracle's plan; ours takes them from the C
    planner's layout (planned here on the host), so this also checks that the
    two agree on the bytes the metric is computed from."""
    sys.path.insert(0, ROOT)
    import json

    import bench
    from fsdp2_gradient_packing_gb300 import _build
    _build.build()
    from fsdp2_gradient_packing_gb300 import fsdp_pack as fp
    bench.main(["--impl", "reference", "--steps", "10", "--warmup", "1"])
    d = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    args = bench.parse_args([])
    factory, description = bench.WORKLOADS[args.workload]
    work = factory()
    specs = work.groups[0]
    with fp.fsdp_plan_layout_host(specs, work.W) as L:
        info = fp.fsdp_layout_query(L)
        bucket_bytes = [fp.fsdp_layout_bucket(L, b).bytes for b in range(info.n_buckets)]
        pack = bench.op_bytes(specs, work.W, bucket_bytes, info.ag_bytes)["pack"]
    assert pack == 302_055_424
    assert d["config"] == bench.make_config(args, work, description, 1, 1, pack, 1)
