"""The intermediate-axis split across processes, on the one GPU this run has:
two ranks (gloo process group, host exchange) each load and run their own
window of the layer with ftmoe_forward, exchange their fp32 partials, and
sum them in rank order with ftmoe_reduce_partials.  No kernel of one rank
waits for the other's: each rank's kernels finish before the exchange.  The
result must equal a single process's full-window forward up to fp32
reordering, and the oracle to the parity bar."""

import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, name, T, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import bench
    from gpu_helpers import GpuBank, make_layer
    from nvfp4_mixture_experts_counting_gb300 import ftmoe, workloads as W
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        torch.cuda.set_device(0)
        wl = W.WORKLOADS[name]
        bank = GpuBank(wl)
        i0, I_loc = bench.window_of_rank(rank, ws, wl.I)
        layer = make_layer(wl, max_tokens=T)
        layer.load_bank(0, bank.desc(), i0=i0, I_loc=I_loc)
        x = W.hidden(wl, T, step=31, device="cuda")
        part = torch.empty((T, wl.H), dtype=torch.float32, device="cuda")
        layer.forward(0, x, part, out_flags=ftmoe.OUT_FP32, i0=i0, I_loc=I_loc)
        torch.cuda.synchronize()
        assert layer.check_status() == 0
        gathered = [torch.empty((T, wl.H), dtype=torch.float32) for _ in range(ws)]
        dist.all_gather(gathered, part.cpu())
        parts = torch.stack(gathered).cuda()
        out = torch.empty((T, wl.H), dtype=torch.bfloat16, device="cuda")
        out32 = torch.empty((T, wl.H), dtype=torch.float32, device="cuda")
        ftmoe.ftmoe_reduce_partials(parts, ws, T * wl.H, out, ftmoe.OUT_BF16)
        ftmoe.ftmoe_reduce_partials(parts, ws, T * wl.H, out32, ftmoe.OUT_FP32)
        torch.cuda.synchronize()
        layer.close()
        if rank == 0:
            q.put((out.float().cpu().numpy(), out32.cpu().numpy(), parts.cpu().numpy()))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("name,T", [("decode", 16), ("prefill", 1024)])
def test_two_processes_window_split_equals_full_layer(name, T):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from nvfp4_mixture_experts_counting_gb300 import build
    build.build()
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, ws, port, name, T, q)) for r in range(ws)]
    for p in procs:
        p.start()
    out, out32, parts = q.get(timeout=600)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    # the fixed-order sum of the partials
    assert np.array_equal(out32, parts[0] + parts[1])
    # against one process running the whole window, and the oracle
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from gpu_helpers import GpuBank, check_output, make_layer, rel_l2
    from nvfp4_mixture_experts_counting_gb300 import ftmoe, workloads as W
    wl = W.WORKLOADS[name]
    bank = GpuBank(wl)
    layer = make_layer(wl, max_tokens=T)
    layer.load_bank(0, bank.desc())
    x = W.hidden(wl, T, step=31, device="cuda")
    full = torch.empty((T, wl.H), dtype=torch.float32, device="cuda")
    layer.forward(0, x, full, out_flags=ftmoe.OUT_FP32)
    torch.cuda.synchronize()
    assert rel_l2(out32, full.cpu().numpy()) <= 1e-6
    rows = np.arange(0, T, max(1, T // 64))
    ref = bank.oracle_layer(x, tokens=rows)
    check_output(torch.from_numpy(out), ref.out, rows=rows)
    layer.close()
