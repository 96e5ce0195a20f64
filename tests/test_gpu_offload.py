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

from gpu_helpers import AuxBufs, GpuBank, check_output, make_layer, rel_l2

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


@pytest.fixture(scope="module")
def offload_bank():
    wl = W.WORKLOADS["offload"]
    return wl, GpuBank(wl)


def test_offload_full_size_decode_matches_resident_and_lru(offload_bank):
    """The offload workload's own sizes (H=4096, I=2048, E=256, 95 slots =
    37% of the experts): a run of single-token and small decode steps, each
    with fresh tokens, must give the resident handle's output and exactly
    the hits and misses of the replacement rule (a touched list read back
    stale would show up as too many hits)."""
    wl, bank = offload_bank
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


def _offload_run(wl, res, off, steps_T, n_slots, step0, i0=0, I_loc=None):
    """Forward the same fresh tokens through the resident and the offloaded
    handle; outputs must agree bitwise where one batch of slots holds every
    touched expert (and on every prefill-sized step, which keeps each pair's
    output and combines once), else within fp32 reordering.  Returns the
    touched lists and the last step's tokens and offloaded output."""
    touched_steps = []
    x = yb = None
    for i, T in enumerate(steps_T):
        x = W.hidden(wl, T, step=step0 + i, device=DEV)
        ya = torch.empty((T, wl.H), dtype=torch.float32, device=DEV)
        yb = torch.empty_like(ya)
        aux = AuxBufs(T, wl.top_k, wl.E)
        res.forward(0, x, ya, out_flags=ftmoe.OUT_FP32, i0=i0, I_loc=I_loc)
        off.forward(0, x, yb, out_flags=ftmoe.OUT_FP32, i0=i0, I_loc=I_loc, aux=aux.c)
        torch.cuda.synchronize()
        assert off.check_status() == 0
        offs = aux.offsets.cpu().numpy()
        touched = [e for e in range(wl.E) if offs[e + 1] > offs[e]]
        touched_steps.append(touched)
        # the step's touched experts, counted on the host even when they
        # needed several batches of slots
        assert off.stats(0).touched_experts == len(touched), f"step {i} T={T}"
        if T > 32 or len(touched) <= n_slots:
            assert torch.equal(ya.view(torch.int32), yb.view(torch.int32)), f"step {i} T={T}"
        else:
            assert rel_l2(yb.cpu().numpy(), ya.cpu().numpy()) <= 1e-6, f"step {i} T={T}"
    return touched_steps, x, yb


def test_offload_prefill_T2048_matches_resident_oracle_and_lru(offload_bank):
    """T = 2048 on the offload workload: every expert is touched, so each
    step runs three batches of the 95 slots (37% of the experts); its output
    equals the resident handle's bitwise, the hits and misses equal the
    replacement rule's, and a token sample matches the oracle."""
    wl, bank = offload_bank
    res = make_layer(wl, max_tokens=2048)
    res.load_bank(0, bank.desc())
    n_slots = int(round(0.37 * wl.E))
    cfg = ftmoe.make_config(H=wl.H, I=wl.I, E=wl.E, top_k=wl.top_k, I_shared=wl.I_s, max_tokens=2048,
                            hbm_slot_bytes=n_slots * A.expert_window_bytes(wl.H, wl.I))
    off = ftmoe.Layer(cfg)
    off.load_bank(0, bank.desc())
    assert off.stats(0).resident_slots == n_slots
    steps, x, yb = _offload_run(wl, res, off, [2048, 16, 2048, 1, 2048], n_slots, step0=500)
    assert len(steps[0]) == wl.E  # every expert touched: batches of the slot count
    st = off.stats(0)
    hits, misses = simulate_lru(n_slots, steps)
    assert (st.hits, st.misses) == (hits, misses)
    rows = np.array([0, 1, 777, 1500, 2046, 2047])
    bank.prefetch_oracle_experts(np.unique(_topk_of(res, wl, x)[rows]))
    ref = bank.oracle_layer(x, out_dtype="fp32", tokens=rows)
    check_output(yb, ref.out64, rows=rows)
    res.close()
    off.close()


def _topk_of(layer, wl, x, **window):
    aux = AuxBufs(x.shape[0], wl.top_k, wl.E)
    out = torch.empty((x.shape[0], wl.H), dtype=torch.bfloat16, device=DEV)
    layer.forward(0, x, out, aux=aux.c, **window)
    torch.cuda.synchronize()
    return aux.topk_idx.cpu().numpy()


def test_offload_half_windows_keep_the_byte_budget(offload_bank):
    """Windows of I_loc = 1024 halve a slot, so the byte budget of 95 full
    slots holds 189 half slots (73.8% of the experts).  Each half, loaded on
    its own offloaded handle, equals a resident handle holding the same
    window (bitwise at T = 2048 and for a single batch), its hits and misses
    equal the replacement rule's, a token sample of each half matches the
    oracle's partial, and the two halves add up to the full layer."""
    wl, bank = offload_bank
    budget = int(round(0.37 * wl.E)) * A.expert_window_bytes(wl.H, wl.I)
    half = wl.I // 2
    n_slots = budget // A.expert_window_bytes(wl.H, half)
    assert n_slots == 189
    full = make_layer(wl, max_tokens=2048)
    full.load_bank(0, bank.desc())
    acc = None
    last_x = None
    for i0 in (0, half):
        res = make_layer(wl, max_tokens=2048)
        res.load_bank(0, bank.desc(), i0=i0, I_loc=half)
        cfg = ftmoe.make_config(H=wl.H, I=wl.I, E=wl.E, top_k=wl.top_k, I_shared=wl.I_s, max_tokens=2048,
                                hbm_slot_bytes=budget)
        off = ftmoe.Layer(cfg)
        off.load_bank(0, bank.desc(), i0=i0, I_loc=half)
        st = off.stats(0)
        assert st.resident_slots == n_slots
        assert abs(st.residency - n_slots / wl.E) < 1e-12
        steps, x, yb = _offload_run(wl, res, off, [2048, 16, 1, 2048], n_slots, step0=600, i0=i0, I_loc=half)
        st = off.stats(0)
        hits, misses = simulate_lru(n_slots, steps)
        assert (st.hits, st.misses) == (hits, misses)
        rows = np.array([3, 1024, 2040])
        bank.prefetch_oracle_experts(np.unique(_topk_of(res, wl, x, i0=i0, I_loc=half)[rows]))
        ref = bank.oracle_layer(x, i0=i0, I_loc=half, out_dtype="fp32", tokens=rows)
        check_output(yb, ref.out64, rows=rows)
        acc = yb.clone() if acc is None else acc + yb
        last_x = x
        res.close()
        off.close()
    y_full = torch.empty_like(acc)
    full.forward(0, last_x, y_full, out_flags=ftmoe.OUT_FP32)
    torch.cuda.synchronize()
    # the same sums in another order: each half's down product adds 1024
    # fp32 terms per output, the full run 2048, so the two differ by fp32
    # reordering of about sqrt(2048) * 2^-24 ~ 3e-6 relative at most
    assert rel_l2(acc.cpu().numpy(), y_full.cpu().numpy()) <= 4e-6
    full.close()
