"""The N > 1 bookkeeping of bench.py on CPU: two gloo ranks.

Rows of the block are independent, so `bench.py --gpus N` runs N replicas,
each on its own synthetic batch, with no data-path collective; what the ranks
share is the barrier around the timed region, the max over ranks of the step
time, the whole-job value (tokens of all ranks / slowest rank's time), and, for
the reference arm, rank 0 alone running and printing.  These run here as two
processes on the gloo backend (no GPU).
"""
import contextlib
import io
import json
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, outdir):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import bench
    import moe_inputs as mi
    args = bench.parse(["--impl", "reference", "--config", "tiny", "--gpus", str(world),
                        "--steps", "1", "--warmup", "0", "--ref-step-seconds", "0.2"])
    w, r, _ = bench.dist_setup(args)
    res = {"world": w, "rank": r}
    try:
        bench.barrier(w)
        res["max"] = bench.max_over_ranks(1.5 + r, w, "cpu")
        cfg = mi.CONFIGS["tiny"]
        res["seed"] = bench.replica_seed(cfg, r)
        res["x_sum"] = float(mi.make_inputs(cfg, "cpu", seed=res["seed"])["x"].float().sum())
        buf = io.StringIO()
        with contextlib.redirect_stdout(buf):
            bench.run_reference(args, w, r)
        res["printed"] = buf.getvalue()
        bench.barrier(w)
    finally:
        import torch.distributed as dist
        dist.destroy_process_group()
    with open(os.path.join(outdir, f"rank{rank}.json"), "w") as f:
        json.dump(res, f)


@pytest.fixture(scope="module")
def two_ranks(tmp_path_factory):
    import oracle
    oracle.build()  # once, before the ranks start
    out = tmp_path_factory.mktemp("ranks")
    mp.spawn(_rank_main, args=(2, _free_port(), str(out)), nprocs=2, join=True)
    return [json.load(open(out / f"rank{r}.json")) for r in range(2)]


def test_ranks_see_the_world(two_ranks):
    assert [d["rank"] for d in two_ranks] == [0, 1]
    assert all(d["world"] == 2 for d in two_ranks)


def test_step_time_is_the_max_over_ranks(two_ranks):
    assert all(d["max"] == 2.5 for d in two_ranks)


def test_replicas_draw_their_own_batches(two_ranks):
    assert two_ranks[0]["seed"] != two_ranks[1]["seed"]
    assert two_ranks[0]["x_sum"] != two_ranks[1]["x_sum"]


def test_reference_arm_prints_on_rank0_only(two_ranks):
    line = json.loads(two_ranks[0]["printed"].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert two_ranks[1]["printed"] == ""


def test_whole_job_value_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    # 4096 tokens per rank, 2 ranks, slowest rank 0.5 ms per step
    assert bench.aggregate_value(4096, 2, 0.5) == pytest.approx(4096 * 2 / 0.5e-3)
    assert bench.aggregate_value(4096, 1, 0.5) == pytest.approx(4096 / 0.5e-3)


# ---- token-sharded aux: the one exchange a sharded forward would need ----------

def _shard_main(rank, world, port, outdir):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import numpy as np
    import torch.distributed as dist
    import moe_inputs as mi
    import oracle
    dist.init_process_group("gloo")
    try:
        cfg = mi.MoEConfig("shard", 96, 256, 16, 4, 128, True, seed=13)
        b = {k: mi.bits(v) for k, v in mi.make_inputs(cfg, "cpu").items()}
        lo, hi = rank * cfg.T // world, (rank + 1) * cfg.T // world
        logits = oracle.router_logits(b["x"][lo:hi], b["W_router"])
        idx, _ = oracle.route_from_logits(logits, cfg.K, cfg.norm)
        counts = np.bincount(idx.ravel(), minlength=cfg.E).astype(np.float64)
        psum = oracle.softmax(logits).sum(axis=0)
        # all-gather both vectors, then add them in rank order (deterministic)
        mine = torch.from_numpy(np.concatenate([counts, psum]))
        parts = [torch.empty_like(mine) for _ in range(world)]
        dist.all_gather(parts, mine)
        tot = parts[0].clone()
        for p in parts[1:]:
            tot += p
        c_g, p_g = tot[:cfg.E].numpy(), tot[cfg.E:].numpy()
        aux = cfg.E * float(np.sum((c_g / (cfg.T * cfg.K)) * (p_g / cfg.T)))
    finally:
        dist.destroy_process_group()
    with open(os.path.join(outdir, f"shard{rank}.json"), "w") as f:
        json.dump({"aux": aux}, f)


def test_token_sharded_aux_equals_unsharded(tmp_path):
    import numpy as np
    import moe_inputs as mi
    import oracle
    oracle.build()
    mp.spawn(_shard_main, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    got = [json.load(open(tmp_path / f"shard{r}.json"))["aux"] for r in range(2)]
    cfg = mi.MoEConfig("shard", 96, 256, 16, 4, 128, True, seed=13)
    b = {k: mi.bits(v) for k, v in mi.make_inputs(cfg, "cpu").items()}
    logits = oracle.router_logits(b["x"], b["W_router"])
    idx, _ = oracle.route_from_logits(logits, cfg.K, cfg.norm)
    want = oracle.aux(oracle.softmax(logits), np.bincount(idx.ravel(), minlength=cfg.E)
                      .astype(np.int32), cfg.K)
    assert got[0] == got[1]
    assert abs(got[0] - want) <= 1e-12 * max(1.0, want)
