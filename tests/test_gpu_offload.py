"""Offload mode: banks in pinned host memory, a few HBM slots filled
least-recently-used first.  Outputs must equal the resident handle's
(bitwise where the arithmetic is the same; within fp32 reordering where a
decode forward runs its experts in several batches), and the hit / miss
counts must equal a host simulation of the stated replacement rule."""

import numpy as np
import pytest
import torch

from nvfp4_mixture_experts_counting_gb300 import ftmoe, accounting as A, workloads as W
from oracle import moe

from gpu_helpers import AuxBufs, GpuBank, make_layer, rel_l2

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from nvfp4_mixture_experts_counting_gb300 import build
    build.build()


def simulate_lru(n_slots, steps):
    """Hits and misses of the replacement rule: a forward's touched experts,
    those already resident first (each group in expert order), go in
    batches of n_slots; per batch, refresh the hits, then give each miss the
    lowest empty slot, else the least recently used slot the batch does not
    use."""
    slot_of, owner, stamp = {}, [None] * n_slots, [0] * n_slots
    clock = hits = misses = 0
    for touched in steps:
        touched = [e for e in touched if e in slot_of] + [e for e in touched if e not in slot_of]
        for b0 in range(0, len(touched), n_slots):
            batch = sorted(touched[b0:b0 + n_slots])  # the kernels' order within a batch
            start = clock + 1
            for e in batch:
                if e in slot_of:
                    clock += 1
                    stamp[slot_of[e]] = clock
                    hits += 1
            for e in batch:
                if e in slot_of and stamp[slot_of[e]] >= start:
                    continue
                empty = [s for s in range(n_slots) if owner[s] is None]
                if empty:
                    v = empty[0]
                else:
                    v = min((s for s in range(n_slots) if stamp[s] < start), key=lambda s: stamp[s])
                    del slot_of[owner[v]]
                owner[v] = e
                slot_of[e] = v
                clock += 1
                stamp[v] = clock
                misses += 1
    return hits, misses


def test_offload_matches_resident_and_lru():
    wl = W.WORKLOADS["mid"]
    bank = GpuBank(wl)
    res = make_layer(wl, max_tokens=128)
    res.load_bank(0, bank.desc())
    n_slots = 6
    cfg = ftmoe.make_config(H=wl.H, I=wl.I, E=wl.E, top_k=wl.top_k, I_shared=wl.I_s, max_tokens=128,
                            hbm_slot_bytes=n_slots * A.expert_window_bytes(wl.H, wl.I) + 100)
    off = ftmoe.Layer(cfg)
    off.load_bank(0, bank.desc())
    st = off.stats(0)
    assert st.resident_slots == n_slots
    assert abs(st.residency - n_slots / wl.E) < 1e-12
    steps = []
    for i, T in enumerate([1, 2, 5, 16, 40, 3, 100, 1, 24, 64]):
        x = W.hidden(wl, T, step=50 + i, device=DEV)
        ya = torch.empty((T, wl.H), dtype=torch.float32, device=DEV)
        yb = torch.empty_like(ya)
        aux = AuxBufs(T, wl.top_k, wl.E)
        res.forward(0, x, ya, out_flags=ftmoe.OUT_FP32)
        off.forward(0, x, yb, out_flags=ftmoe.OUT_FP32, aux=aux.c)
        torch.cuda.synchronize()
        assert off.check_status() == 0
        offs = aux.offsets.cpu().numpy()
        touched = [e for e in range(wl.E) if offs[e + 1] > offs[e]]
        steps.append(touched)
        if T > 32 or len(touched) <= n_slots:
            assert torch.equal(ya.view(torch.int32), yb.view(torch.int32)), f"T={T}"
        else:
            assert rel_l2(yb.cpu().numpy(), ya.cpu().numpy()) <= 1e-6, f"T={T}"
    st = off.stats(0)
    hits, misses = simulate_lru(n_slots, steps)
    assert (st.hits, st.misses) == (hits, misses)
    assert st.h2d_bytes % max(misses, 1) == 0 and st.h2d_bytes // misses >= A.expert_window_bytes(wl.H, wl.I)


def test_offload_bf16_output_matches_oracle():
    wl = W.WORKLOADS["mid"]
    bank = GpuBank(wl)
    cfg = ftmoe.make_config(H=wl.H, I=wl.I, E=wl.E, top_k=wl.top_k, I_shared=wl.I_s, max_tokens=64,
                            hbm_slot_bytes=4 * A.expert_window_bytes(wl.H, wl.I))
    off = ftmoe.Layer(cfg)
    off.load_bank(0, bank.desc())
    from gpu_helpers import check_output, check_routing
    for T in (16, 48):
        x = W.hidden(wl, T, step=70 + T, device=DEV)
        out = torch.empty((T, wl.H), dtype=torch.bfloat16, device=DEV)
        aux = AuxBufs(T, wl.top_k, wl.E)
        off.forward(0, x, out, aux=aux.c)
        torch.cuda.synchronize()
        ref = bank.oracle_layer(x)
        check_routing(aux, ref)
        check_output(out, ref.out)


def test_offload_full_size_decode_matches_resident_and_lru():
    """The offload workload's own sizes (H=4096, I=2048, E=256, 95 slots =
    37% of the experts): a run of single-token and small decode steps, each
    with fresh tokens, must give the resident handle's output and exactly
    the hits and misses of the replacement rule (a touched list read back
    stale would show up as too many hits)."""
    wl = W.WORKLOADS["offload"]
    bank = GpuBank(wl)
    res = make_layer(wl, max_tokens=32)
    res.load_bank(0, bank.desc())
    n_slots = int(round(0.37 * wl.E))
    cfg = ftmoe.make_config(H=wl.H, I=wl.I, E=wl.E, top_k=wl.top_k, I_shared=wl.I_s, max_tokens=32,
                            hbm_slot_bytes=n_slots * A.expert_window_bytes(wl.H, wl.I))
    off = ftmoe.Layer(cfg)
    off.load_bank(0, bank.desc())
    assert off.stats(0).resident_slots == n_slots
    steps = []
    for i, T in enumerate([1, 1, 1, 1, 16, 1, 1, 32, 1, 1, 8, 1]):
        x = W.hidden(wl, T, step=300 + i, device=DEV)
        ya = torch.empty((T, wl.H), dtype=torch.float32, device=DEV)
        yb = torch.empty_like(ya)
        aux = AuxBufs(T, wl.top_k, wl.E)
        res.forward(0, x, ya, out_flags=ftmoe.OUT_FP32)
        off.forward(0, x, yb, out_flags=ftmoe.OUT_FP32, aux=aux.c)
        torch.cuda.synchronize()
        assert off.check_status() == 0
        offs = aux.offsets.cpu().numpy()
        touched = [e for e in range(wl.E) if offs[e + 1] > offs[e]]
        steps.append(touched)
        if len(touched) <= n_slots:
            assert torch.equal(ya.view(torch.int32), yb.view(torch.int32)), f"step {i} T={T}"
        else:
            assert rel_l2(yb.cpu().numpy(), ya.cpu().numpy()) <= 1e-6, f"step {i} T={T}"
    st = off.stats(0)
    hits, misses = simulate_lru(n_slots, steps)
    assert (st.hits, st.misses) == (hits, misses)
    assert st.h2d_bytes == misses * (st.h2d_bytes // max(misses, 1))
