"""The N > 1 path of the bench on CPU: two gloo ranks.

The layer shards by tokens across replicas (each GPU runs its own batch and
no collective touches the data path), so the multi-rank logic is the host's:
every rank draws distinct tokens, the job's time is the slowest rank's
(max over ranks after a barrier), the whole-job value counts every rank's
tokens, and the oracle arm runs on rank 0 alone."""

import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    from nvfp4_mixture_experts_counting_gb300 import workloads as W
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        assert bench.dist_env() == (ws, rank, rank)
        # each rank "timed" a different duration; the job takes the slowest
        ms = 10.0 + 5.0 * rank
        bench._barrier_and_sync(ws)
        ms_max = bench._max_over_ranks(ws, ms)
        value = bench.whole_job_tokens_per_s(ws, 16, 100, ms_max)
        # the tokens this rank draws for its first steps
        wl = W.WORKLOADS["tiny"]
        xs = [W.hidden(wl, wl.tokens[0], step=bench.replica_step_seed(rank, s)) for s in range(3)]
        gathered = [None] * ws
        dist.all_gather_object(gathered, [x.float().sum().item() for x in xs])
        q.put((rank, ms_max, value, gathered))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_time_max_and_distinct_inputs():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(ws)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    for rank, ms_max, value, gathered in res:
        assert ms_max == 15.0  # the slowest rank's time on every rank
        assert value == pytest.approx(2 * 16 * 100 / 0.015)
        # every rank's inputs differ from every other rank's
        flat = [v for per_rank in gathered for v in per_rank]
        assert len(set(flat)) == len(flat)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")

    class Args:
        workload, T, steps, warmup = "decode", 16, 3, 3

    bench.run_reference(Args())
    assert capsys.readouterr().out == ""


def test_single_rank_helpers_need_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench._max_over_ranks(1, 3.5) == 3.5
    assert bench.whole_job_tokens_per_s(1, 16, 1000, 156.0) == pytest.approx(16 * 1000 / 0.156)
    assert bench.replica_step_seed(0, 7) == 7 and bench.replica_step_seed(1, 7) != 7


def _window_rank_main(rank, ws, port, q):
    """One rank of the intermediate-axis split on CPU: its window's oracle
    partial of the tiny layer, the partials exchanged with gloo, summed in
    rank order."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import numpy as np
    import bench
    from nvfp4_mixture_experts_counting_gb300 import workloads as W
    from oracle import moe
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        wl = W.WORKLOADS["tiny"]
        x = W.hidden(wl, 4).float().numpy()
        rw = W.router_weight(wl).numpy()
        sgu, sdn, sg = [t.float().numpy() for t in W.shared_weights(wl)]
        banks = {}

        def get(e):
            if e not in banks:
                g, d = W.expert_masters(wl, e)
                banks[e] = moe.quantize_expert(g.numpy(), d.numpy())
            return banks[e]

        i0, I_loc = bench.window_of_rank(rank, ws, wl.I)
        part = moe.moe_layer(x, rw, None, get, sgu, sdn, sg, I=wl.I, I_s=wl.I_s, top_k=wl.top_k,
                             i0=i0, I_loc=I_loc, out_dtype="fp32").out64
        gathered = [torch.empty(part.shape, dtype=torch.float64) for _ in range(ws)]
        dist.all_gather(gathered, torch.from_numpy(part))
        total = gathered[0].clone()
        for r in range(1, ws):
            total += gathered[r]
        full = moe.moe_layer(x, rw, None, get, sgu, sdn, sg, I=wl.I, I_s=wl.I_s, top_k=wl.top_k,
                             out_dtype="fp32").out64
        q.put((rank, (i0, I_loc), float(np.max(np.abs(total.numpy() - full)) / np.max(np.abs(full)))))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("ws", [2, 4])
def test_window_split_partials_sum_to_the_full_layer(ws):
    """The pages' split across processes: rank r holds window r of every
    expert and of the shared expert, with the router replicated; the SUM of
    the ranks' partials is the whole layer (exact up to fp64 rounding: the
    windows share no term)."""
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_window_rank_main, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in range(ws))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    windows = [w for _, w, _ in res]
    assert windows == [(r * 64 // ws, 64 // ws) for r in range(ws)]
    for _, _, err in res:
        assert err <= 1e-12


def test_window_of_rank_covers_I_once():
    sys.path.insert(0, ROOT)
    import bench
    for I, ws in ((640, 1), (640, 2), (640, 4), (2048, 2), (2048, 8)):
        w = [bench.window_of_rank(r, ws, I) for r in range(ws)]
        assert w[0][0] == 0 and sum(l for _, l in w) == I
        assert all(a + l == b for (a, l), (b, _) in zip(w, w[1:]))
    for ws in (3, 16):   # 640 / 3 is not whole; 640 / 16 = 40 is off the 16-block grid
        with pytest.raises(ValueError):
            bench.window_of_rank(0, ws, 640)
