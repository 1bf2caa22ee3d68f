"""The benchmark's multi-rank host logic on CPU: world_size 2 over gloo.

Ranks run independent batches against replicated weights (tokens are
independent, so the path shards by batch with no data-path collective); the
timed region is bracketed by barriers and the slowest rank's time is the one
reported.  No GPU is used."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from sparse_mixture_experts_58_b300 import inputs


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    try:
        r, w, local = bench.dist_env()
        assert (r, w, local) == (rank, world, rank)
        bench.dist_init(w, "gloo")
        # each rank's batch differs, the weights are shared
        seed = bench.rank_token_seed(0, r)
        x, _ = inputs.draw_tokens(inputs.generator(seed, "cpu"), 8, 64, "bf16", "cpu")
        layer = inputs.draw_weights(inputs.generator(1000, "cpu"), 64, 64, 4, "bf16", "cpu")
        bench.barrier(w)
        # the slowest rank's time is the job's time
        t = bench.reduce_max(1.0 + rank, w, "cpu")
        digests = [None] * w
        dist.all_gather_object(digests, (float(x.float().sum()), float(layer.W1.float().sum())))
        q.put((rank, t, digests))
        dist.destroy_process_group()
    except Exception as e:  # report to the parent instead of hanging it
        q.put((rank, "error", repr(e)))


def test_two_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=240) for _ in range(2)]
    for p in procs:
        p.join(timeout=60)
    for rank, t, digests in results:
        assert t != "error", digests
        assert t == 2.0                          # max over ranks
        (x0, w0), (x1, w1) = digests
        assert x0 != x1                          # different batches per rank
        assert w0 == w1                          # replicated weights
    assert all(p.exitcode == 0 for p in procs)


def test_single_rank_helpers_are_identities():
    assert bench.reduce_max(3.5, 1, "cpu") == 3.5
    bench.barrier(1)
    assert bench.rank_token_seed(0, 0) == 0 and bench.rank_token_seed(0, 1) != 0


def test_bench_main_two_ranks_dry_run(capfd):
    """bench.main with --gpus 2 outside torchrun relaunches itself with two
    ranks (gloo in the dry run, no GPU work); rank 0 prints one line for
    the job: n_gpus 2, each rank its own batch, the weights shared."""
    import json
    assert "WORLD_SIZE" not in os.environ
    rc = bench.main(["--gpus", "2", "--dry-run", "--steps", "3", "--warmup", "3"])
    assert rc == 0
    lines = [ln for ln in capfd.readouterr().out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["dry_run"] is True and rec["n_gpus"] == 2
    assert [r["rank"] for r in rec["ranks"]] == [0, 1]
    assert rec["ranks"][0]["tokens_sum"] != rec["ranks"][1]["tokens_sum"]
    assert rec["ranks"][0]["w1_sum"] == rec["ranks"][1]["w1_sum"]


def test_bench_refuses_a_world_that_differs_from_gpus(monkeypatch):
    """A launch whose world size is not --gpus fails loudly."""
    monkeypatch.setenv("WORLD_SIZE", "1")
    monkeypatch.setenv("RANK", "0")
    with pytest.raises(SystemExit):
        bench.main(["--gpus", "2", "--dry-run", "--steps", "1"])
