#!/usr/bin/env python
"""Throughput of the routed NVFP4 MoE layer on GB300, through libftmoe.so.

python bench.py --gpus N --steps K --warmup W [--impl reference]

A step is one forward of one MoE layer (router, top-k, counting sort,
activation quantisation, gate_up + SwiGLU, down, shared expert, combine) over
a batch of T tokens.  The default workload is the decode-shaped layer
(H=2560, I=I_s=640, E=256, top_k=8, T=16, the whole of I).  Each step uses the
next of 8 independently seeded layers, so the banks the steps read (8 x 712
MB) are far larger than L2.  All inputs are synthetic and seeded.

Under torchrun each rank runs the same workload on its own tokens (weak
scaling, no collective on the data path); the printed value is the sum over
ranks divided by the slowest rank's time.

--impl reference times the CPU oracle (the fp64 numpy restatement used by the
tests) on the host cores, on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
FALLBACK_HBM_GBS = 6800.0

KERNEL_SOURCES = {
    "k_dec_route": ("decode_route.cu", "decode_common.cuh", "tma.cuh"),
    "k_dec_gate_up": ("decode_gate_up.cu", "decode_common.cuh", "tma.cuh"),
    "k_dec_down": ("decode_down.cu", "decode_common.cuh", "tma.cuh"),
    "k_dtc_gate_up": ("decode_tc.cu", "decode_common.cuh", "tc_common.cuh", "tma.cuh"),
    "k_dtc_down": ("decode_tc.cu", "decode_common.cuh", "tc_common.cuh", "tma.cuh"),
    "k_pf_gate_up": ("prefill.cu", "tc_common.cuh", "tma.cuh"), "k_pf_down": ("prefill.cu", "tc_common.cuh", "tma.cuh"),
    "k_pf_prep": ("prefill.cu",),
    "k_gate_up": ("experts.cu",), "k_down": ("experts.cu",), "k_shared_gate_up": ("experts.cu",),
    "k_shared_down": ("experts.cu",), "k_combine": ("experts.cu",), "k_router_logits": ("route.cu",),
    "k_topk": ("route.cu",), "k_sort": ("route.cu",), "k_xquant_sigma": ("route.cu",),
}


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="decode")
    p.add_argument("--T", type=int, default=16)
    p.add_argument("--layers", type=int, default=0,
                   help="independently seeded layers rotated per step (default: 8 for decode, 2 for prefill)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-prefill", action="store_true",
                   help="decode workload: leave out the prefill half of the metric (T=16384 and 4096)")
    p.add_argument("--slots-frac", type=float, default=0.37,
                   help="offload workload: HBM slots as a fraction of the experts (byte budget of full windows)")
    p.add_argument("--iloc", type=int, default=0, help="load and run the window [0, iloc) (0: all of I)")
    p.add_argument("--compare", choices=["none", "ep"], default="none",
                   help="ep: time each rank's compute of the intermediate split against expert "
                        "parallelism, on this one GPU (a comparison, not the benchmark line)")
    p.add_argument("--ranks", type=int, default=2, help="--compare ep: ranks to emulate")
    p.add_argument("--split", choices=["replicas", "window"], default="replicas",
                   help="N>1: replicas run their own tokens with no collective (default); window splits "
                        "the intermediate axis over the ranks, which exchange their fp32 partials "
                        "(NCCL all-gather) and sum them in rank order")
    return p.parse_args()


# ------------------------------------------------------------------ small helpers

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# fp32 FMA peak of the CUDA cores: 152 SMs x 128 fp32 lanes x 2 flops x 2070 MHz
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.070e9 / 1e12
FP32_ALU_SOURCE = "derived: 152 SMs x 128 fp32 lanes x 2 flops x 2070 MHz (nominal)"
FP4_PER_BF16 = 13.5 / 2.25  # nominal dense NVFP4 / BF16 tensor rates


def load_bf16_peak():
    """Dense bf16 tensor peak: the measured cuBLAS bf16 burst rate, else the
    1.9 PFLOP/s fallback."""
    try:
        with open(PEAKS_FILE) as f:
            pk = json.load(f)
        return float(pk["bf16_tflops"]), "measured cuBLAS bf16 burst (MEASURED_PEAKS.json bf16_tflops)"
    except Exception:
        return 1900.0, "fallback bf16 1.9 PFLOP/s"


def load_fp4_peak():
    """Dense NVFP4 peak: the measured cuBLAS bf16 burst rate x the nominal
    FP4/BF16 ratio (6), else the 1.9 PFLOP/s bf16 fallback x 6."""
    try:
        with open(PEAKS_FILE) as f:
            pk = json.load(f)
        return float(pk["bf16_tflops"]) * FP4_PER_BF16, "measured cuBLAS bf16 burst x nominal NVFP4/BF16 ratio 6"
    except Exception:
        return 1900.0 * FP4_PER_BF16, "fallback bf16 1.9 PFLOP/s x nominal NVFP4/BF16 ratio 6"


def source_digest(kernel: str) -> str:
    """Digest of the sources a kernel is compiled from (its files + common.cuh)."""
    csrc = os.path.join(ROOT, "nvfp4_mixture_experts_counting_gb300", "csrc")
    h = hashlib.sha256()
    for name in (*KERNEL_SOURCES.get(kernel, ()), "common.cuh"):
        path = os.path.join(csrc, name)
        if os.path.exists(path):
            h.update(open(path, "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload_key: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current source of that kernel (else None)."""
    try:
        with open(TRAFFIC_FILE) as f:
            tab = json.load(f)
        ent = tab[kernel][workload_key]
        if ent.get("source_digest") != source_digest(kernel):
            return None
        return float(ent["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi samples (every 100 ms) while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        note = "samples inside the timed region"
        if not inside:
            # the timed region was shorter than the sampling period: take the
            # samples nearest to it
            near = sorted(self.samples, key=lambda s: abs(s[0] - (t0 + t1) / 2))[:3]
            inside = [p for (_, p) in near]
            note = "timed region shorter than the 100 ms sampling period; nearest samples"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        smax = [num(p[2]) for p in inside if num(p[2]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for p in inside:
            for n, v in zip(names, p[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(inside), "note": note}


# ------------------------------------------------------------------ oracle timing (CPU)

def _oracle_steps(workload: str, T: int, tokens_per_step: int, max_steps: int, budget_s: float,
                  threads: int):
    """Runs in a spawned process.  Each step times the oracle layer on the
    next tokens_per_step tokens of a seeded batch of T tokens; the experts
    those tokens route to are quantised by the oracle beforehand (untimed,
    as bank loading is on the GPU side).  Stops after max_steps steps or
    once budget_s seconds of timed work are spent.  Returns the step times."""
    os.environ["OMP_NUM_THREADS"] = str(threads)
    os.environ["OPENBLAS_NUM_THREADS"] = str(threads)
    import numpy as np
    from nvfp4_mixture_experts_counting_gb300 import workloads as W
    from oracle import moe
    wl = W.WORKLOADS[workload]
    x = W.hidden(wl, T).float().numpy()
    rw = W.router_weight(wl).numpy()
    b = W.router_bias(wl)
    b = None if b is None else b.numpy()
    sgu, sdn, sg = [t.float().numpy() for t in W.shared_weights(wl)]
    idx, _ = moe.select_topk(moe.router_logits(x, rw, b), wl.top_k)
    banks = {}
    times = []
    spent = 0.0
    s = 0
    while s < max_steps and spent < budget_s:
        toks = np.array([(s * tokens_per_step + j) % T for j in range(tokens_per_step)])
        for e in sorted(set(idx[toks].reshape(-1).tolist())):
            if e not in banks:
                g, d = W.expert_masters(wl, e)
                banks[e] = moe.quantize_expert(g.numpy(), d.numpy())
        t0 = time.perf_counter()
        moe.moe_layer(x, rw, b, lambda e: banks[e], sgu, sdn, sg, I=wl.I, I_s=wl.I_s,
                      top_k=wl.top_k, tokens=toks)
        dt = time.perf_counter() - t0
        times.append(dt)
        spent += dt
        s += 1
    return times


def oracle_times(workload: str, T: int, tokens_per_step: int, max_steps: int, budget_s: float,
                 threads: int):
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    with ctx.Pool(1) as pool:
        return pool.apply(_oracle_steps, (workload, T, tokens_per_step, max_steps, budget_s, threads))


def cpu_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ------------------------------------------------------------------ GPU arm

def build_layers(wl, n_layers, max_tokens, dev, hbm_slot_bytes=0, I_loc=0, i0=0):
    import torch
    from nvfp4_mixture_experts_counting_gb300 import ftmoe, workloads as W
    cfg = ftmoe.make_config(H=wl.H, I=wl.I, E=wl.E, top_k=wl.top_k, I_shared=wl.I_s,
                            num_layers=n_layers, max_tokens=max_tokens,
                            norm_topk_prob=wl.norm_topk_prob, has_router_bias=wl.router_bias,
                            hbm_slot_bytes=hbm_slot_bytes)
    layer = ftmoe.Layer(cfg, torch.cuda.current_device())
    E, I, H = wl.E, wl.I, wl.H
    for l in range(n_layers):
        gu = torch.empty((E, 2 * I, H), dtype=torch.float32, device=dev)
        dn = torch.empty((E, H, I), dtype=torch.float32, device=dev)
        for e in range(E):
            g, d = W.expert_masters(wl, e, l, device=dev)
            gu[e].copy_(g)
            dn[e].copy_(d)
        q = {
            "gu_codes": torch.empty((E, 2 * I, H // 2), dtype=torch.uint8, device=dev),
            "gu_scales": torch.empty((E, 2 * I, H // 16), dtype=torch.uint8, device=dev),
            "gu_global": torch.empty((E, 2 * I), dtype=torch.float32, device=dev),
            "dn_codes": torch.empty((E, H, I // 2), dtype=torch.uint8, device=dev),
            "dn_scales": torch.empty((E, H, I // 16), dtype=torch.uint8, device=dev),
            "dn_global": torch.empty((E, H), dtype=torch.float32, device=dev),
        }
        ftmoe.ftmoe_quantize_weights(gu, E * 2 * I, H, q["gu_codes"], q["gu_scales"], q["gu_global"])
        ftmoe.ftmoe_quantize_weights(dn, E * H, I, q["dn_codes"], q["dn_scales"], q["dn_global"])
        del gu, dn
        rw = W.router_weight(wl, l, device=dev)
        rb = W.router_bias(wl, l, device=dev)
        sgu, sdn, sg = W.shared_weights(wl, l, device=dev)
        desc = ftmoe.bank_desc(rw, rb, q["gu_codes"], q["gu_scales"], q["gu_global"], q["dn_codes"],
                               q["dn_scales"], q["dn_global"], sgu, sdn, sg, on_device=True)
        layer.load_bank(l, desc, i0, I_loc or None)
        del q
        torch.cuda.synchronize()
    return layer


def _barrier_and_sync(ws):
    import torch
    import torch.distributed as dist
    if ws > 1:
        dist.barrier()
    if torch.cuda.is_available():
        torch.cuda.synchronize()


def _max_over_ranks(ws, v: float) -> float:
    """The largest of the ranks' values (the job's time is its slowest rank's)."""
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cpu" if dist.get_backend() == "gloo" else "cuda"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_step_seed(rank: int, step: int) -> int:
    """Input step index of a replica: every rank draws its own tokens."""
    return step + 100000 * rank


def whole_job_tokens_per_s(ws: int, T: int, steps: int, ms_max: float) -> float:
    """Tokens all ranks processed / the slowest rank's time."""
    return ws * T * steps / (ms_max / 1e3)


def window_of_rank(rank: int, ws: int, I: int):
    """(i0, I_loc) of rank `rank` when the intermediate axis is split over
    `ws` ranks: contiguous equal windows in rank order, each a multiple of 16
    (the NVFP4 block), as the pages' TP patch splits I."""
    if I % ws or (I // ws) % 16:
        raise ValueError(f"I={I} does not split into {ws} windows of a multiple of 16")
    w = I // ws
    return rank * w, w


def window_tokens_per_s(T: int, steps: int, ms_max: float) -> float:
    """Window split: every rank works on the same T tokens, so the job's
    tokens are T per step whatever the number of ranks."""
    return T * steps / (ms_max / 1e3)


def kernel_roofline(kernel: str, launches: int, kernel_ms: float, steps: int, unit_bytes_info, unit_flops_info,
                    pairs: int, T: int, touched_per_step: float, hbm_peak, fp4_peak):
    """The dominant kernel's achieved rate against its roofline: algorithmic
    bytes (or flops) per launch over the mean launch time.  `steps` steps
    made `launches` launches taking `kernel_ms` in all; a step's work is
    spread over that kernel's launches in a step (an offloaded forward
    launches the expert kernels once per batch of slots)."""
    avg_s = kernel_ms / launches / 1e3
    per = steps / launches
    unit_bytes, unit, fixed = unit_bytes_info
    unit_flops, funit, path = unit_flops_info
    if unit_flops is not None:
        units = (pairs if funit == "pair" else T) * per
        achieved = unit_flops * units / avg_s / 1e12
        if path.startswith("nvfp4"):
            (pk, pk_src), bound = fp4_peak, "tensor"
        elif path.startswith("bf16"):
            (pk, pk_src), bound = load_bf16_peak(), "tensor"
        else:
            pk, pk_src, bound = FP32_ALU_TFLOPS, FP32_ALU_SOURCE, "alu"
        return {"bound": bound, "kernel": kernel, "achieved": round(achieved, 1), "peak": round(pk, 1),
                "unit": "TFLOP/s", "frac": round(achieved / pk, 4), "traffic": None,
                "algorithmic_flops_per_launch": int(unit_flops * units), "unit_flops": unit_flops,
                "units_per_launch": round(units, 2), "units": funit, "datapath": path,
                "avg_launch_us": round(avg_s * 1e6, 2), "peak_source": pk_src}
    if unit_bytes is None:
        return None  # no algorithmic accounting for this kernel
    peak, peak_kind = hbm_peak
    units = (touched_per_step if unit.startswith("touched") else 1.0) * per
    alg = unit_bytes * units + fixed * per
    achieved = alg / avg_s / 1e9
    return {"bound": "hbm", "kernel": kernel, "achieved": round(achieved, 1), "peak": peak,
            "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": None,
            "algorithmic_bytes_per_launch": int(alg), "unit_bytes": unit_bytes,
            "units_per_launch": round(units, 2), "units": unit,
            "avg_launch_us": round(avg_s * 1e6, 2),
            "peak_source": f"{peak_kind} HBM copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"}


def prefill_leg(T, K, Wm, rank, ws, local, cpu_baseline: bool):
    """The prefill-shaped layer (Zipf-biased routing) timed the same way as
    the headline: K steps after Wm warm-up steps, CUDA events on the launch
    stream around the steps alone, two independently seeded layers rotated
    (1.4 GB of banks, far larger than L2).  Returns the sub-report: tokens/s,
    the routed GEMM's roofline against the NVFP4 peak, the layer's fraction
    of the NVFP4 peak and of its combined roofline, kernel shares, clocks and
    the oracle's rate on a token sample."""
    import torch
    from nvfp4_mixture_experts_counting_gb300 import accounting as A
    from nvfp4_mixture_experts_counting_gb300 import ftmoe, workloads as W
    wl = W.WORKLOADS["prefill"]
    L = 2
    layer = build_layers(wl, L, T, "cuda")
    xs = [W.hidden(wl, T, step=replica_step_seed(rank, s), device="cuda") for s in range(2)]
    out = torch.empty((T, wl.H), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()

    def step(i):
        layer.forward(i % L, xs[i % 2], out, stream=stream)

    for i in range(Wm):
        step(i)
    torch.cuda.synchronize()
    rerank0 = layer.stats(0).reranked_tokens
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    _barrier_and_sync(ws)
    t_wall0 = time.time()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(K):
        step(Wm + i)
    ev1.record(stream)
    _barrier_and_sync(ws)
    t_wall1 = time.time()
    time.sleep(0.25)
    clocks.stop()
    reranked = layer.stats(0).reranked_tokens - rerank0
    ms_max = _max_over_ranks(ws, ev0.elapsed_time(ev1))
    value = whole_job_tokens_per_s(ws, T, K, ms_max)
    t_step = ms_max / K / 1e3

    KP = min(K, 10)
    ftmoe.ftmoe_profile_enable(layer.handle, True)
    ftmoe.ftmoe_profile_read(layer.handle)
    for i in range(KP):
        step(i)
    torch.cuda.synchronize()
    ktimes = ftmoe.ftmoe_profile_read(layer.handle)
    ftmoe.ftmoe_profile_enable(layer.handle, False)

    offs = torch.empty((wl.E + 1,), dtype=torch.int32, device="cuda")
    aux = ftmoe.Aux(None, None, offs.data_ptr(), None, None)
    touched = []
    for li in range(L):
        layer.forward(li, xs[li % 2], out, aux=aux, stream=stream)
        o = offs.cpu()
        touched.append(int(((o[1:] - o[:-1]) > 0).sum()))
    mean_touched = sum(touched) / len(touched)

    hbm, hbm_kind = load_peaks()
    fp4, fp4_kind = load_fp4_peak()
    bf16, _ = load_bf16_peak()
    pairs = T * wl.top_k
    total_k = sum(v[1] for v in ktimes.values()) or 1.0
    roof = {}
    for kname in ("k_pf_gate_up", "k_pf_down"):
        if kname in ktimes:
            launches, kms = ktimes[kname]
            r = kernel_roofline(kname, launches, kms, KP, A.kernel_unit_bytes(kname, wl.H, wl.I, wl.I_s, wl.E),
                                A.kernel_unit_flops(kname, wl.H, wl.I, wl.I_s, wl.E), pairs, T, mean_touched,
                                (hbm, hbm_kind), (fp4, fp4_kind))
            r["traffic"] = ncu_traffic(kname, f"prefill_T{T}")
            roof[kname] = r
    comb = A.combined_ideal_seconds(wl.H, wl.E, wl.I, wl.I_s, T, pairs, mean_touched, fp4, bf16, hbm)
    routed = A.routed_flops(wl.H, wl.I, pairs)
    cpu = None
    if cpu_baseline and rank == 0:
        th = cpu_threads()
        n_tok = 4
        try:
            secs = sum(oracle_times("prefill", T, n_tok, 1, 1e9, th))
            cpu = {"value": round(n_tok / secs, 4), "unit": "tokens/s", "cores": th, "kind": "oracle",
                   "sample": f"{n_tok} tokens of one seeded T={T} batch of the prefill layer (their experts' "
                             f"banks quantised beforehand, untimed); numpy fp64, BLAS threads={th}"}
        except Exception as ex:
            cpu = {"value": None, "unit": "tokens/s", "cores": th, "kind": "oracle", "sample": f"failed: {ex}"}
    res = {
        "workload": f"prefill layer: H={wl.H} I={wl.I} I_s={wl.I_s} E={wl.E} top_k={wl.top_k}, T={T}, "
                    f"full I window, Zipf(1.1) router bias",
        "value": round(value, 1), "unit": "tokens/s", "steps": K, "warmup": Wm,
        "ms_per_step": round(ms_max / K, 4),
        "l2": f"inputs larger than L2: {L} independently seeded layers rotated per step "
              f"({L} x {A.expert_window_bytes(wl.H, wl.I) * wl.E / 1e6:.0f} MB of banks)",
        "touched_experts_per_step": round(mean_touched, 2),
        "reranked_tokens_per_step": round(reranked / K, 2),
        "routed_fp4_tflops": round(routed / t_step / 1e12, 1),
        "routed_frac_of_fp4_peak": round(routed / t_step / 1e12 / fp4, 4),
        "fp4_peak_tflops": round(fp4, 1), "fp4_peak_source": fp4_kind,
        "combined_roofline": {"frac": round(comb["bound_s"] / t_step, 4), "bound": comb["bound"],
                              "ideal_us": round(comb["bound_s"] * 1e6, 2),
                              "tensor_us": round(comb["tensor_s"] * 1e6, 2),
                              "hbm_us": round(comb["hbm_s"] * 1e6, 2),
                              "note": "routed FP4 flops at the NVFP4 peak + shared-expert flops at the bf16 "
                                      "peak + 3 x router flops (three exact bf16 parts) at the bf16 peak, "
                                      "against touched bytes at the HBM peak; frac = ideal / measured step"},
        "roofline": roof.get("k_pf_gate_up"),
        "roofline_down": roof.get("k_pf_down"),
        "kernel_shares": {k: {"launches": v[0], "ms": round(v[1], 3), "share": round(v[1] / total_k, 4)}
                          for k, v in ktimes.items()},
        "gpu_launches": int(round(sum(v[0] for v in ktimes.values()) * K / KP)),
        "clocks": clocks.summary(t_wall0, t_wall1),
        "cpu_baseline": cpu,
    }
    layer.close()
    del xs, out
    torch.cuda.empty_cache()
    return res


def run_gpu(args):
    import torch
    import torch.distributed as dist
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group("nccl")
    from nvfp4_mixture_experts_counting_gb300 import build as B
    if rank == 0:
        B.build()
    if ws > 1:
        dist.barrier()
    from nvfp4_mixture_experts_counting_gb300 import accounting as A
    from nvfp4_mixture_experts_counting_gb300 import ftmoe, workloads as W

    wl = W.WORKLOADS[args.workload]
    T, K, Wm = args.T, args.steps, max(args.warmup, 3)
    offload = args.workload == "offload"
    L = args.layers or (1 if offload else (8 if T <= 32 else 2))
    dev = "cuda"
    split = args.split == "window"
    if split:
        if offload or args.iloc:
            raise SystemExit("--split window runs the resident layer over its whole I")
        i0, I_loc = window_of_rank(rank, ws, wl.I)
    else:
        i0, I_loc = 0, args.iloc or wl.I
    sI_loc = I_loc * wl.I_s // wl.I
    # offload: the slot budget is a fraction of the experts at full-window
    # bytes; a narrower window keeps the byte budget (more, smaller slots)
    slot_bytes = int(round(args.slots_frac * wl.E)) * A.expert_window_bytes(wl.H, wl.I) if offload else 0
    layer = build_layers(wl, L, T, dev, hbm_slot_bytes=slot_bytes, I_loc=I_loc, i0=i0)
    # offload: a fresh input every step (the slot cache must not see repeats);
    # otherwise 8 inputs in turn
    NX = (K + Wm) if offload else 8
    # replicas draw their own tokens; the ranks of a window split share them
    xs = [W.hidden(wl, T, step=replica_step_seed(0 if split else rank, s), device=dev) for s in range(NX)]
    out = torch.empty((T, wl.H), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    part = torch.empty((T, wl.H), dtype=torch.float32, device=dev) if split else None
    parts = torch.empty((ws, T, wl.H), dtype=torch.float32, device=dev) if split and ws > 1 else part

    def step(i, o=out, x=None):
        xi = xs[i % NX] if x is None else x
        if not split:
            layer.forward(i % L, xi, o, i0=i0, I_loc=I_loc, stream=stream)
            return
        # this rank's window partial, every rank's partial gathered, summed in
        # rank order and rounded once
        layer.forward(i % L, xi, part, out_flags=ftmoe.OUT_FP32, i0=i0, I_loc=I_loc, stream=stream)
        if ws > 1:
            dist.all_gather_into_tensor(parts, part)
        ftmoe.ftmoe_reduce_partials(parts, ws, T * wl.H, o, ftmoe.OUT_BF16, stream=stream)

    for i in range(Wm):
        step(i)
    torch.cuda.synchronize()

    # ---- timed region: the steps alone (per-kernel events would sit between
    # the kernels and stop programmatic dependent launch from overlapping them)
    st_before = layer.stats(0)
    rerank0 = st_before.reranked_tokens
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    _barrier_and_sync(ws)
    t_wall0 = time.time()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(K):
        step(Wm + i)
    ev1.record(stream)
    _barrier_and_sync(ws)
    t_wall1 = time.time()
    time.sleep(0.25)
    clocks.stop()
    ms = ev0.elapsed_time(ev1)
    st_after = layer.stats(0)
    reranked = st_after.reranked_tokens - rerank0
    ms_max = _max_over_ranks(ws, ms)
    value = window_tokens_per_s(T, K, ms_max) if split else whole_job_tokens_per_s(ws, T, K, ms_max)

    # ---- per-kernel durations: a second pass of the same steps with CUDA
    # events around every kernel on the launch stream
    KP = min(K, 500)
    ftmoe.ftmoe_profile_enable(layer.handle, True)
    ftmoe.ftmoe_profile_read(layer.handle)          # drop older records
    for i in range(KP):
        step(i)
    torch.cuda.synchronize()
    ktimes = ftmoe.ftmoe_profile_read(layer.handle)
    ftmoe.ftmoe_profile_enable(layer.handle, False)

    # ---- untimed: touched experts of every (layer, x) combination used above
    offs = torch.empty((wl.E + 1,), dtype=torch.int32, device=dev)
    aux = ftmoe.Aux(None, None, offs.data_ptr(), None, None)
    touched = {}
    for li in range(L):
        for xi in range(NX):
            layer.forward(li, xs[xi], out, i0=i0, I_loc=I_loc, aux=aux, stream=stream)
            o = offs.cpu()
            touched[(li, xi)] = int(((o[1:] - o[:-1]) > 0).sum())
    per_step_touched = [touched[((Wm + i) % L, (Wm + i) % NX)] for i in range(K)]
    mean_touched = sum(per_step_touched) / K
    bytes_step = sum(A.layer_touched_bytes(wl.H, wl.E, I_loc, sI_loc, T, tt) for tt in per_step_touched) / K
    routed_bytes_step = mean_touched * A.expert_window_bytes(wl.H, I_loc)

    # ---- dominant kernel roofline
    peak, peak_kind = load_peaks()
    fp4_peak, fp4_kind = load_fp4_peak()
    pairs = T * wl.top_k
    total_k = sum(v[1] for v in ktimes.values()) or 1.0
    dom = max(ktimes.items(), key=lambda kv: kv[1][1])[0] if ktimes else None
    roof = None
    if dom:
        launches, kms = ktimes[dom]
        roof = kernel_roofline(dom, launches, kms, KP, A.kernel_unit_bytes(dom, wl.H, I_loc, sI_loc, wl.E),
                               A.kernel_unit_flops(dom, wl.H, I_loc, sI_loc, wl.E), pairs, T, mean_touched,
                               (peak, peak_kind), (fp4_peak, fp4_kind))
        if roof:
            roof["traffic"] = ncu_traffic(dom, f"{args.workload}_T{T}")
    shares = {k: {"launches": v[0], "ms": round(v[1], 3), "share": round(v[1] / total_k, 4)}
              for k, v in ktimes.items()}

    # ---- end to end through the C ABI with host buffers: every step copies
    # its tokens in from pinned host memory and its output back, on a copy
    # stream with two buffers each way, so step i+1's input lands while step
    # i computes and step i's output leaves while step i+1 computes
    xh = [x.cpu().pin_memory() for x in xs]
    oh = [torch.empty((T, wl.H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    xd = [torch.empty_like(xs[0]) for _ in range(2)]
    od = [torch.empty_like(out) for _ in range(2)]
    cs = torch.cuda.Stream()
    ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]

    def copy_in(i):
        b = i % 2
        with torch.cuda.stream(cs):
            if i >= 2:
                cs.wait_event(done[b])  # step i-2 has finished with xd[b]
            xd[b].copy_(xh[i % NX], non_blocking=True)
            ready[b].record(cs)

    def run_e2e(n):
        copy_in(0)
        for i in range(n):
            b = i % 2
            if i + 1 < n:
                copy_in(i + 1)
            stream.wait_event(ready[b])
            step(i, od[b], xd[b])
            done[b].record(stream)
            with torch.cuda.stream(cs):
                cs.wait_event(done[b])
                oh[b].copy_(od[b], non_blocking=True)
        stream.wait_stream(cs)

    run_e2e(Wm)
    _barrier_and_sync(ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run_e2e(K)
    e1.record(stream)
    _barrier_and_sync(ws)
    e2e_ms = _max_over_ranks(ws, e0.elapsed_time(e1))
    e2e_value = window_tokens_per_s(T, K, e2e_ms) if split else whole_job_tokens_per_s(ws, T, K, e2e_ms)

    # ---- GPU launch count inside the timed region (the profiled pass counts
    # the launches of KP steps)
    launches_total = int(round(sum(v[0] for v in ktimes.values()) * K / KP))

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        n_tok = 4
        th = cpu_threads()
        try:
            secs = sum(oracle_times(args.workload, T, n_tok, 1, 1e9, th))
            cpu = {"value": round(n_tok / secs, 4), "unit": "tokens/s", "cores": th, "kind": "oracle",
                   "sample": f"{n_tok} tokens of one seeded T={T} batch of the {args.workload} layer "
                             f"(their experts' banks quantised beforehand, untimed); numpy fp64, "
                             f"BLAS threads={th}"}
        except Exception as ex:  # the baseline is reported, never required
            cpu = {"value": None, "unit": "tokens/s", "cores": th, "kind": "oracle", "sample": f"failed: {ex}"}

    # the prefill half of the metric, on the default decode run
    prefill = None
    if args.workload == "decode" and not args.no_prefill and not split:
        layer.close()
        torch.cuda.empty_cache()
        prefill = {f"T{Tp}": prefill_leg(Tp, Kp, 3, rank, ws, local, not args.no_cpu_baseline)
                   for Tp, Kp in ((16384, 20), (4096, 40))}

    if rank == 0:
        cl = clocks.summary(t_wall0, t_wall1)
        line = {
            "metric": "MoE-layer tokens/s at 1 GB300; % of HBM peak (decode) / NVFP4 tensor peak (prefill)",
            "value": round(value, 2), "unit": "tokens/s", "n_gpus": ws, "steps": K, "warmup": Wm,
            "ms_per_step": round(ms_max / K, 5), "higher_is_better": True,
            "scaling": "strong" if split else "weak",
            "vs_baseline": None, "dtype": "nvfp4 (e2m1 x e2m1, fp32 accumulate); bf16 shared expert",
            "data": "synthetic, seeded",
            "config": {"workload": f"{args.workload} layer: H={wl.H} I={wl.I} I_s={wl.I_s} E={wl.E} "
                                   f"top_k={wl.top_k}, T={T}, "
                                   + (f"window [{i0}, {i0 + I_loc}) per rank" if split else
                                      f"window [0, {I_loc})" if I_loc != wl.I else "full I window")
                                   + (", Zipf(1.1) router bias" if wl.router_bias else "")
                                   + (f", offloaded banks, HBM slots for {args.slots_frac:.0%} of the experts"
                                      if offload else ""),
                       "global_batch": T if split else T * ws, "layers_rotated": L,
                       "l2": f"inputs larger than L2: {L} independently seeded layers rotated per step "
                             f"({L} x {A.expert_window_bytes(wl.H, I_loc) * wl.E / 1e6:.0f} MB of banks)",
                       "parallelism": (f"intermediate axis split over {ws} ranks: fp32 partials, NCCL "
                                       f"all-gather, fixed rank-order sum" if split else
                                       f"replicas x{ws} (token-parallel, no collective)")},
            "touched_experts_per_step": round(mean_touched, 2),
            **({"offload": {"slots": st_after.resident_slots, "residency": round(st_after.residency, 4),
                            "hit_rate": round((st_after.hits - st_before.hits) /
                                              max(1, st_after.hits - st_before.hits + st_after.misses
                                                  - st_before.misses), 4),
                            "h2d_gbs": round((st_after.h2d_bytes - st_before.h2d_bytes) / (ms_max / 1e3) / 1e9, 1),
                            "h2d_bytes_per_step": int((st_after.h2d_bytes - st_before.h2d_bytes) / K)}}
               if offload else {}),
            "reranked_tokens_per_step": round(reranked / K, 4),
            "touched_bytes_per_step": int(bytes_step),
            "layer_hbm_frac": round(bytes_step / (ms_max / K / 1e3) / 1e9 / peak, 4),
            "layer_hbm_gbs": round(bytes_step / (ms_max / K / 1e3) / 1e9, 1),
            "routed_only_gbs": round(routed_bytes_step / (ms_max / K / 1e3) / 1e9, 1),
            "roofline": roof,
            "routed_fp4_tflops": round(A.routed_flops(wl.H, I_loc, pairs) / (ms_max / K / 1e3) / 1e12, 2),
            "routed_frac_of_fp4_peak": round(A.routed_flops(wl.H, I_loc, pairs) / (ms_max / K / 1e3) / 1e12
                                             / fp4_peak, 4),
            "kernel_shares": shares,
            "kernel_shares_note": f"CUDA events around each kernel over {KP} separate steps (events between "
                                  f"kernels disable their programmatic dependent launch overlap)",
            "gpu_launches": launches_total,
            "e2e": {"value": round(e2e_value, 2), "unit": "tokens/s", "h2d_bytes_per_step": T * wl.H * 2,
                    "d2h_bytes_per_step": T * wl.H * 2},
            "clocks": cl,
            "cpu_baseline": cpu,
            **({"prefill": prefill} if prefill else {}),
        }
        print(json.dumps(line), flush=True)
    layer.close()
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    from nvfp4_mixture_experts_counting_gb300 import workloads as W
    wl = W.WORKLOADS[args.workload]
    th = cpu_threads()
    K, Wm = args.steps, args.warmup
    # one token of the batch per step; stop running steps once the budget is
    # spent so the whole run stays within a few minutes
    budget_s = 120.0
    times = oracle_times(args.workload, args.T, 1, K, budget_s, th)
    n = max(len(times), 1)
    tot = sum(times)
    value = n / tot
    line = {
        "impl": "reference",
        "metric": "MoE-layer tokens/s at 1 GB300; % of HBM peak (decode) / NVFP4 tensor peak (prefill)",
        "value": round(value, 4), "unit": "tokens/s", "n_gpus": ws, "steps": K, "warmup": Wm,
        "ms_per_step": round(1e3 * tot / n, 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic, seeded",
        "config": {"workload": f"{args.workload} layer: H={wl.H} I={wl.I} I_s={wl.I_s} E={wl.E} "
                               f"top_k={wl.top_k}, T={args.T}, full I window"},
        "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": th, "kind": "oracle",
                         "sample": f"one token of a seeded T={args.T} batch per step; {n} of {K} steps "
                                   f"run within a {budget_s:.0f} s budget"},
        "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_stack(args):
    """The layer stack (every layer's own seeded weights, RMS renorm between
    layers), one CUDA graph per step replayed K times."""
    import torch
    import torch.distributed as dist
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group("nccl")
    from nvfp4_mixture_experts_counting_gb300 import build as B
    if rank == 0:
        B.build()
    if ws > 1:
        dist.barrier()
    from nvfp4_mixture_experts_counting_gb300 import accounting as A
    from nvfp4_mixture_experts_counting_gb300 import ftmoe, workloads as W

    wl = W.WORKLOADS[args.workload]
    T, K, Wm, NL = args.T, args.steps, max(args.warmup, 3), wl.layers
    dev = "cuda"
    layer = build_layers(wl, NL, T, dev)
    x = W.hidden(wl, T, step=replica_step_seed(rank, 0), device=dev)
    out = torch.empty((T, wl.H), dtype=torch.bfloat16, device=dev)
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cs):
        for _ in range(Wm):
            layer.forward_stack(x, out, stream=cs)
    cs.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cs):
        layer.forward_stack(x, out, stream=cs)
    for _ in range(Wm):
        graph.replay()
    torch.cuda.synchronize()

    st0 = layer.stats(0)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    _barrier_and_sync(ws)
    t_wall0 = time.time()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    for _ in range(K):
        graph.replay()
    ev1.record()
    _barrier_and_sync(ws)
    t_wall1 = time.time()
    time.sleep(0.25)
    clocks.stop()
    st1 = layer.stats(0)
    ms_max = _max_over_ranks(ws, ev0.elapsed_time(ev1))
    value = whole_job_tokens_per_s(ws, T, K, ms_max)
    touched_per_layer = (st1.touched_total - st0.touched_total) / (K * NL)
    reranked = (st1.reranked_tokens - st0.reranked_tokens) / K
    bytes_step = NL * A.layer_touched_bytes(wl.H, wl.E, wl.I, wl.I_s, T, touched_per_layer)
    peak, peak_kind = load_peaks()

    # per-kernel durations: separate steps without the graph, events around kernels
    KP = min(K, 20)
    ftmoe.ftmoe_profile_enable(layer.handle, True)
    ftmoe.ftmoe_profile_read(layer.handle)
    for _ in range(KP):
        layer.forward_stack(x, out)
    torch.cuda.synchronize()
    ktimes = ftmoe.ftmoe_profile_read(layer.handle)
    ftmoe.ftmoe_profile_enable(layer.handle, False)
    total_k = sum(v[1] for v in ktimes.values()) or 1.0
    dom = max(ktimes.items(), key=lambda kv: kv[1][1])[0] if ktimes else None
    roof = None
    if dom and A.kernel_unit_bytes(dom, wl.H, wl.I, wl.I_s, wl.E)[0] is not None:
        launches, kms = ktimes[dom]
        # one launch per layer: a "step" of the helper is one layer
        roof = kernel_roofline(dom, launches, kms, launches, A.kernel_unit_bytes(dom, wl.H, wl.I, wl.I_s, wl.E),
                               (None, None, None), T * wl.top_k, T, touched_per_layer, (peak, peak_kind), (None, None))
        roof["traffic"] = ncu_traffic(dom, f"{args.workload}_T{T}")
    shares = {k: {"launches": v[0], "ms": round(v[1], 3), "share": round(v[1] / total_k, 4)}
              for k, v in ktimes.items()}

    # end to end: the input in from pinned host memory and the output back,
    # around every graph replay
    xh = x.cpu().pin_memory()
    oh = torch.empty((T, wl.H), dtype=torch.bfloat16).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(K):
        x.copy_(xh, non_blocking=True)
        graph.replay()
        oh.copy_(out, non_blocking=True)
    e1.record()
    _barrier_and_sync(ws)
    e2e_ms = _max_over_ranks(ws, e0.elapsed_time(e1))
    launches_total = int(round(sum(v[0] for v in ktimes.values()) * K / KP))

    if rank == 0:
        line = {
            "metric": "MoE-layer tokens/s at 1 GB300; % of HBM peak (decode) / NVFP4 tensor peak (prefill)",
            "value": round(value, 2), "unit": "tokens/s", "n_gpus": ws, "steps": K, "warmup": Wm,
            "ms_per_step": round(ms_max / K, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "nvfp4 (e2m1 x e2m1, fp32 accumulate); bf16 shared expert",
            "data": "synthetic, seeded",
            "config": {"workload": f"{NL}-layer stack of the decode layer (H={wl.H} I={wl.I} I_s={wl.I_s} "
                                   f"E={wl.E} top_k={wl.top_k}), independent seeded weights per layer, RMS "
                                   f"renorm between layers, T={T}, one CUDA graph per step",
                       "global_batch": T * ws,
                       "l2": f"inputs larger than L2: {NL} layers x "
                             f"{A.expert_window_bytes(wl.H, wl.I) * wl.E / 1e6:.0f} MB of banks per step",
                       "parallelism": f"replicas x{ws} (token-parallel, no collective)"},
            "moe_ms_per_step": round(ms_max / K, 4),
            "touched_experts_per_layer": round(touched_per_layer, 2),
            "touched_bytes_per_step": int(bytes_step),
            "reranked_tokens_per_step": round(reranked, 4),
            "stack_hbm_frac": round(bytes_step / (ms_max / K / 1e3) / 1e9 / peak, 4),
            "stack_hbm_gbs": round(bytes_step / (ms_max / K / 1e3) / 1e9, 1),
            "roofline": roof,
            "kernel_shares": shares,
            "kernel_shares_note": f"CUDA events around each kernel over {KP} steps run without the graph",
            "gpu_launches": launches_total,
            "e2e": {"value": round(whole_job_tokens_per_s(ws, T, K, e2e_ms), 2), "unit": "tokens/s",
                    "h2d_bytes_per_step": T * wl.H * 2, "d2h_bytes_per_step": T * wl.H * 2},
            "clocks": clocks.summary(t_wall0, t_wall1),
            "cpu_baseline": None,
        }
        print(json.dumps(line), flush=True)
    layer.close()
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()


def _kernel_ms_per_step(layer, fn, K):
    """Summed CUDA-event times of the library's kernels per call of fn()."""
    import torch
    from nvfp4_mixture_experts_counting_gb300 import ftmoe
    ftmoe.ftmoe_profile_enable(layer.handle, True)
    ftmoe.ftmoe_profile_read(layer.handle)
    for _ in range(K):
        fn()
    torch.cuda.synchronize()
    kt = ftmoe.ftmoe_profile_read(layer.handle)
    ftmoe.ftmoe_profile_enable(layer.handle, False)
    return sum(v[1] for v in kt.values()) / K


def run_compare(args):
    """The two ways to put one MoE layer on G GPUs, each rank's compute timed
    on this one GPU: the pages' intermediate split (rank r runs window r of
    every expert: balanced by construction, one all-reduce of [T, H]) and
    expert parallelism (rank r owns the experts e % G == r: its load follows
    the routing, two all-to-alls of the dispatched rows, padded to T * top_k
    rows for static shapes).  A step of either takes its slowest rank's time;
    the collectives are reported as the bytes each rank sends, not timed
    (this run has one GPU)."""
    import numpy as np
    import torch
    from nvfp4_mixture_experts_counting_gb300 import build as B
    B.build()
    from nvfp4_mixture_experts_counting_gb300 import ftmoe, workloads as W
    G, K = args.ranks, max(args.steps, 5)
    out_lines = {}
    for wname, T in (("decode", 16), ("prefill", 4096)):
        wl = W.WORKLOADS[wname]
        layer = build_layers(wl, 1, T, "cuda")
        x = W.hidden(wl, T, step=7, device="cuda")
        out = torch.empty((T, wl.H), dtype=torch.bfloat16, device="cuda")
        aux_idx = torch.empty((T, wl.top_k), dtype=torch.int32, device="cuda")
        layer.forward(0, x, out, aux=ftmoe.Aux(aux_idx.data_ptr(), None, None, None, None))
        torch.cuda.synchronize()
        idx = aux_idx.cpu().numpy()
        full_ms = _kernel_ms_per_step(layer, lambda: layer.forward(0, x, out), K)
        win, ep, pairs = [], [], []
        for r in range(G):
            i0, I_loc = window_of_rank(r, G, wl.I)
            win.append(_kernel_ms_per_step(layer, lambda: layer.forward(0, x, out, i0=i0, I_loc=I_loc), K))
            mask = (np.arange(wl.E) % G == r).astype(np.uint8)
            si0, sI = window_of_rank(r, G, wl.I_s)
            ep.append(_kernel_ms_per_step(
                layer, lambda: ftmoe.ftmoe_forward_experts(layer.handle, 0, x, T, out, ftmoe.OUT_BF16, mask,
                                                           si0, sI), K))
            pairs.append(int(np.isin(idx, np.nonzero(mask)[0]).sum()))
        layer.close()
        torch.cuda.empty_cache()
        mean_pairs = T * wl.top_k / G
        out_lines[f"{wname}_T{T}"] = {
            "workload": f"{wname} layer: H={wl.H} I={wl.I} E={wl.E} top_k={wl.top_k}, T={T}"
                        + (", Zipf(1.1) router bias" if wl.router_bias else ""),
            "ranks": G,
            "full_layer_kernel_ms": round(full_ms, 4),
            "window_split": {"rank_kernel_ms": [round(v, 4) for v in win], "step_ms": round(max(win), 4),
                             "allreduce_bytes_per_rank": T * wl.H * 2,
                             "note": "rank r: window [r*I/G, (r+1)*I/G) of every expert and of the shared "
                                     "expert, router and shared gate replicated"},
            "expert_parallel": {"rank_kernel_ms": [round(v, 4) for v in ep], "step_ms": round(max(ep), 4),
                                "rank_pairs": pairs, "pair_imbalance_max_over_mean": round(max(pairs) / mean_pairs, 3),
                                "alltoall_bytes_per_rank_padded": 2 * T * wl.top_k * wl.H * 2,
                                "note": "rank r: the routed slots of experts e % G == r (routing replicated) "
                                        "and window r of the shared expert"},
            "speedup_window_over_expert": round(max(ep) / max(win), 3),
        }
    line = {"mode": "window split vs expert parallel, per-rank kernel time on one GB300",
            "unit": "ms", "steps": K, "comparison": out_lines,
            "note": "kernel times are CUDA-event sums over the library's kernels per call; collectives not timed"}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.compare == "ep":
        run_compare(args)
    elif args.workload == "stack48":
        run_stack(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
