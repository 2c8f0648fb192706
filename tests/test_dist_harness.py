"""The multi-process side of bench.py on CPU ranks (gloo, world size 2): the
timed region's barrier, the max over ranks and the whole-job aggregate, and the
reference arm's rank behaviour.  The data path itself has no collective: each
rank runs its own replica (rows and sequences shard with no exchange)."""
import os
import socket

import pytest

import bench

torch = pytest.importorskip("torch")


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    d = bench.dist_init(world, "gloo")
    t = bench.max_over_ranks(1.0 + rank, d)      # rank r took 1 + r seconds
    bench.barrier(d)
    q.put((rank, t, bench.aggregate_value(world, 8192, 10, t)))
    dist.destroy_process_group()


def test_two_ranks_report_the_slowest_rank_and_the_whole_job():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[1] for o in out] == [2.0, 2.0]
    assert all(o[2] == pytest.approx(2 * 8192 * 10 / 2.0) for o in out)


def test_reference_arm_prints_only_on_rank_zero(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"]) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_line_carries_the_contract_keys(monkeypatch, capsys):
    """Rank 0's reference line, on the tiny head so that it runs in a second: the
    oracle timed on the host cores, reported with its cpu_baseline and an e2e
    entry that moves no bytes, on the same metric, unit and workload names as the
    GB300 arm."""
    import json

    import workloads as wl
    tiny = wl.CONFIGS["tiny"]

    def tiny_workload(seed=0, tokens=None):
        h, W = wl.draw_head(tiny, seed=seed)
        off = wl.draw_segments(tiny, seed=seed)
        return tiny, h, W, wl.draw_targets(tiny, tiny.N, seed=seed), off, wl.draw_mask(tiny, off, seed=seed)

    monkeypatch.setattr(bench, "make_workload", tiny_workload)
    monkeypatch.setenv("TIM_BENCH_ORACLE_SECONDS", "0.2")
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.main(["--impl", "reference", "--steps", "2", "--warmup", "3"]) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert (line["metric"], line["unit"], line["higher_is_better"]) == (bench.METRIC, bench.UNIT, True)
    assert (line["n_gpus"], line["steps"], line["warmup"]) == (1, 2, 3)
    assert line["value"] > 0 and line["ms_per_step"] == pytest.approx(tiny.N / line["value"] * 1e3)
    assert line["config"]["workload"] == "%s_head+mismatch" % tiny.name
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["value"] == line["value"] and cpu["cores"] >= 1 and cpu["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"],
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_single_process_needs_no_process_group():
    assert bench.dist_init(1, "gloo") is None
    assert bench.max_over_ranks(3.5, None) == 3.5
    assert bench.aggregate_value(1, 8192, 30, 0.2) == pytest.approx(8192 * 30 / 0.2)


def _gather_worker(rank, world, port, q):
    import torch.distributed as dist
    from rollout_logprob_mismatch_gb300 import sharded
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    bench.dist_init(world, "gloo")
    sizes = [3, 0, 5][:world]
    # rank r's part: records whose first word is its global sequence index
    first = sum(sizes[:rank])
    local = torch.arange(first, first + sizes[rank], dtype=torch.int32).repeat_interleave(16).view(-1, 16)
    local[:, 1] = rank
    got = sharded.gather_seq_records(local)   # the default group
    q.put((rank, got.tolist()))
    dist.destroy_process_group()


def test_sharded_records_are_gathered_in_the_batch_order():
    """The sharded batch record's one exchange: every rank gets all ranks'
    sequence records in rank order (parts of 3, 0 and 5 sequences), which is
    the batch's sequence order the fold needs."""
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    world = 3
    procs = [ctx.Process(target=_gather_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    owner = [0, 0, 0, 2, 2, 2, 2, 2]
    for _, rows in out:
        assert [r[0] for r in rows] == list(range(8))
        assert [r[1] for r in rows] == owner
        assert all(len(r) == 16 for r in rows)
