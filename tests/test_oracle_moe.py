"""Pins of the oracle's layer against things other than itself: brute-force
top-k, torch's stable argsort and bincount, a textbook dense SwiGLU MLP in
torch fp64 for the one-expert case, degenerate inputs, the slice identity
over every 16-aligned partition, and the byte and residency figures the pages
print (tests/golden/paper_figures.json)."""

import itertools
import json
import os

import numpy as np
import pytest
import torch

from oracle import moe, nvfp4
from nvfp4_mixture_experts_counting_gb300 import workloads as wl_mod

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "paper_figures.json")


# ---------------------------------------------------------------- top-k

def _brute_topk(l, k):
    """The unique k-subset whose members all precede every non-member in the
    order (logit desc, index asc), found by trying every subset."""
    E = len(l)

    def before(a, b):
        return l[a] > l[b] or (l[a] == l[b] and a < b)

    found = []
    for S in itertools.combinations(range(E), k):
        rest = [e for e in range(E) if e not in S]
        if all(before(a, b) for a in S for b in rest):
            found.append(S)
    assert len(found) == 1
    S = list(found[0])
    # order inside the subset by the same relation
    S.sort(key=lambda e: (-l[e], e))
    return S


@pytest.mark.parametrize("k", [1, 2, 3, 8])
def test_topk_brute_force_with_ties(k):
    rng = np.random.default_rng(10 + k)
    for trial in range(60):
        l = rng.integers(-3, 4, size=8).astype(np.float64)  # many exact ties
        if trial % 3 == 0:
            l = rng.standard_normal(8)
        idx, w = moe.select_topk(l[None, :], k)
        assert idx[0].tolist() == _brute_topk(l, k)
        assert abs(w.sum() - 1.0) < 1e-15


def test_topk_equals_stable_torch_sort():
    rng = np.random.default_rng(11)
    l = np.round(rng.standard_normal((64, 256)), 1)
    idx, _ = moe.select_topk(l, 8)
    ref = torch.sort(torch.from_numpy(l), dim=1, descending=True, stable=True).indices[:, :8]
    assert np.array_equal(idx, ref.numpy())


def test_topk_weights_softmax_forms():
    rng = np.random.default_rng(12)
    l = rng.standard_normal((5, 16)) * 3
    idx, w = moe.select_topk(l, 4, norm_topk_prob=True)
    full = torch.softmax(torch.from_numpy(l), dim=1).numpy()
    chosen = np.take_along_axis(full, idx.astype(np.int64), 1)
    assert np.allclose(w, chosen / chosen.sum(1, keepdims=True), rtol=1e-13, atol=0)
    idx2, w2 = moe.select_topk(l, 4, norm_topk_prob=False)
    assert np.array_equal(idx, idx2)
    assert np.allclose(w2, chosen, rtol=1e-13, atol=0)


def test_duplicate_router_rows_choose_lower_index():
    rng = np.random.default_rng(13)
    H, E = 32, 8
    W = rng.standard_normal((E, H)).astype(np.float32)
    W[5] = W[2]                                 # experts 2 and 5 always tie
    W[2] *= 10.0
    W[5] = W[2]
    x = np.abs(rng.standard_normal((6, H))).astype(np.float32)
    x = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    l = moe.router_logits(x, W)
    idx, _ = moe.select_topk(l, 2)
    for t in range(6):
        s = set(idx[t].tolist())
        if 5 in s:
            assert 2 in s
        if 2 in s and 5 in s:
            assert idx[t].tolist().index(2) < idx[t].tolist().index(5)


def test_router_products_exact():
    # bf16 x fp32 products are exact in fp64; compare with a Fraction sum
    from fractions import Fraction
    rng = np.random.default_rng(14)
    x = torch.from_numpy(rng.standard_normal((2, 16)).astype(np.float32)).to(torch.bfloat16).float().numpy()
    W = rng.standard_normal((3, 16)).astype(np.float32)
    l = moe.router_logits(x, W, np.float32([0.5, -0.25, 0.0]))
    for t in range(2):
        for e in range(3):
            exact = sum(Fraction(float(x[t, h])) * Fraction(float(W[e, h])) for h in range(16))
            exact += Fraction([0.5, -0.25, 0.0][e])
            assert abs(float(exact) - l[t, e]) <= 4e-16 * max(1.0, abs(float(exact)))


# ---------------------------------------------------------------- counting sort

def test_counting_sort_matches_torch():
    rng = np.random.default_rng(15)
    for T, k, E in [(4, 2, 8), (37, 8, 256), (1, 8, 256), (300, 3, 5)]:
        idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
        offsets, perm, inv = moe.counting_sort(idx, E)
        flat = torch.from_numpy(idx.reshape(-1).astype(np.int64))
        assert np.array_equal(perm, torch.argsort(flat, stable=True).numpy())
        cnt = torch.bincount(flat, minlength=E).numpy()
        assert offsets[0] == 0 and np.array_equal(np.diff(offsets), cnt)
        assert np.array_equal(perm[inv], np.arange(T * k))


def test_counting_sort_empty():
    offsets, perm, inv = moe.counting_sort(np.zeros((0, 2), dtype=np.int32), 8)
    assert offsets.tolist() == [0] * 9 and perm.size == 0 and inv.size == 0


# ---------------------------------------------------------------- layer helpers

def _tiny_inputs(wl, T=4, seed_step=0):
    x = wl_mod.hidden(wl, T, seed_step).float().numpy()
    rw = wl_mod.router_weight(wl).numpy()
    banks = {}

    def get(e):
        if e not in banks:
            gu, dn = wl_mod.expert_masters(wl, e)
            banks[e] = moe.quantize_expert(gu.numpy(), dn.numpy())
        return banks[e]

    sgu, sdn, sg = wl_mod.shared_weights(wl)
    return x, rw, get, sgu.float().numpy(), sdn.float().numpy(), sg.float().numpy()


def test_window_rows_cover_once():
    I = 640
    for i0, n in [(0, 320), (320, 320)]:
        rows = moe.slice_window_rows(I, i0, n)
        assert len(set(rows.tolist())) == 2 * n
        gate, up = rows[:n], rows[n:]
        assert gate.min() == i0 and gate.max() == i0 + n - 1
        assert up.min() == I + i0 and up.max() == I + i0 + n - 1
    both = np.concatenate([moe.slice_window_rows(I, 0, 320), moe.slice_window_rows(I, 320, 320)])
    assert sorted(both.tolist()) == list(range(2 * I))
    with pytest.raises(ValueError):
        moe.check_window(640, 8, 320)
    with pytest.raises(ValueError):
        moe.check_window(640, 0, 328)
    with pytest.raises(ValueError):
        moe.check_window(640, 320, 336)


def test_one_expert_reduces_to_dense_swiglu_mlp():
    """E=1, k=1, zero shared expert: the layer is a dense SwiGLU MLP on the
    dequantised operands (torch fp64 matmuls and silu)."""
    rng = np.random.default_rng(16)
    H, I = 64, 32
    x = torch.from_numpy(rng.standard_normal((3, H)).astype(np.float32)).to(torch.bfloat16).float()
    gu = (rng.standard_normal((2 * I, H)) * 0.1).astype(np.float32)
    dn = (rng.standard_normal((H, I)) * 0.1).astype(np.float32)
    bank = moe.quantize_expert(gu, dn)
    res = moe.moe_layer(x.numpy(), np.ones((1, H), np.float32), None, lambda e: bank,
                        np.zeros((2 * I, H)), np.zeros((H, I)), np.zeros(H),
                        I=I, I_s=I, top_k=1, out_dtype="fp32")
    # reference, step by step with torch
    xc, xs = nvfp4.quantize_activation_rows(x.numpy())
    xq = torch.from_numpy(nvfp4.dequantize_rows(xc, xs))
    Wgu = torch.from_numpy(nvfp4.dequantize_rows(bank.gu_codes, bank.gu_scales, bank.gu_global))
    Wdn = torch.from_numpy(nvfp4.dequantize_rows(bank.dn_codes, bank.dn_scales, bank.dn_global))
    G = torch.nn.functional.linear(xq, Wgu)
    h = (torch.nn.functional.silu(G[:, :I]) * G[:, I:]).float()
    hc, hs = nvfp4.quantize_activation_rows(h.numpy())
    hq = torch.from_numpy(nvfp4.dequantize_rows(hc, hs))
    y = torch.nn.functional.linear(hq, Wdn)
    assert np.allclose(res.out64, y.numpy(), rtol=1e-12, atol=1e-14)
    assert np.all(res.topk_w == 1.0)


def test_pair_intermediate_is_the_dense_mlps_quantised_h():
    """expert_pair_intermediate against the same torch step by step as the
    dense SwiGLU pin above (torch fp64 matmul and silu, then the oracle's
    quantiser), on a window of a wider expert: the rows it takes are the
    window's gate and up rows."""
    rng = np.random.default_rng(17)
    H, I, i0, I_loc = 64, 64, 16, 32
    x = torch.from_numpy(rng.standard_normal((5, H)).astype(np.float32)).to(torch.bfloat16).float()
    gu = (rng.standard_normal((2 * I, H)) * 0.1).astype(np.float32)
    dn = (rng.standard_normal((H, I)) * 0.1).astype(np.float32)
    bank = moe.quantize_expert(gu, dn)
    xc, xs = nvfp4.quantize_activation_rows(x.numpy())
    xq = nvfp4.dequantize_rows(xc, xs)
    hc, hs = moe.expert_pair_intermediate(bank, xq, I, i0, I_loc)
    Wgu = torch.from_numpy(nvfp4.dequantize_rows(bank.gu_codes, bank.gu_scales, bank.gu_global))
    G = torch.nn.functional.linear(torch.from_numpy(xq), Wgu)  # all 2I rows
    h = (torch.nn.functional.silu(G[:, i0:i0 + I_loc]) * G[:, I + i0:I + i0 + I_loc]).float()
    rc, rs = nvfp4.quantize_activation_rows(h.numpy())
    assert np.array_equal(hc, rc) and np.array_equal(hs, rs)


def test_one_expert_bf16_activations_reduce_to_weight_only_mlp():
    """The bf16-activation (W4A16) mode, E=1, k=1, zero shared expert: a
    dense SwiGLU MLP on the dequantised weights with x unquantised and the
    intermediate rounded to bf16 (torch fp64 matmuls, silu and bf16 cast)."""
    rng = np.random.default_rng(26)
    H, I = 64, 32
    x = torch.from_numpy(rng.standard_normal((3, H)).astype(np.float32)).to(torch.bfloat16).float()
    gu = (rng.standard_normal((2 * I, H)) * 0.1).astype(np.float32)
    dn = (rng.standard_normal((H, I)) * 0.1).astype(np.float32)
    bank = moe.quantize_expert(gu, dn)
    res = moe.moe_layer(x.numpy(), np.ones((1, H), np.float32), None, lambda e: bank,
                        np.zeros((2 * I, H)), np.zeros((H, I)), np.zeros(H),
                        I=I, I_s=I, top_k=1, out_dtype="fp32", activations="bf16")
    Wgu = torch.from_numpy(nvfp4.dequantize_rows(bank.gu_codes, bank.gu_scales, bank.gu_global))
    Wdn = torch.from_numpy(nvfp4.dequantize_rows(bank.dn_codes, bank.dn_scales, bank.dn_global))
    G = torch.nn.functional.linear(x.double(), Wgu)
    h = (torch.nn.functional.silu(G[:, :I]) * G[:, I:]).to(torch.bfloat16).double()
    y = torch.nn.functional.linear(h, Wdn)
    assert np.allclose(res.out64, y.numpy(), rtol=1e-12, atol=1e-14)
    # and it differs from the W4A4 layer (the activations are not quantised)
    res4 = moe.moe_layer(x.numpy(), np.ones((1, H), np.float32), None, lambda e: bank,
                         np.zeros((2 * I, H)), np.zeros((H, I)), np.zeros(H),
                         I=I, I_s=I, top_k=1, out_dtype="fp32")
    assert not np.allclose(res4.out64, res.out64, rtol=1e-3)


def test_expert_subsets_add_up_to_the_layer():
    """The routed parts over a partition of the experts (rank r owning the
    experts e with e % G == r), plus the gated shared expert once, are the
    whole layer; a subset's part has no term of another subset's expert."""
    from nvfp4_mixture_experts_counting_gb300 import workloads as W
    wl = W.WORKLOADS["tiny"]
    x = W.hidden(wl, 6, step=4).float().numpy()
    rw = W.router_weight(wl).numpy()
    sgu, sdn, sg = [t.float().numpy() for t in W.shared_weights(wl)]
    banks = {e: moe.quantize_expert(*[m.numpy() for m in W.expert_masters(wl, e)]) for e in range(wl.E)}
    kw = dict(I=wl.I, I_s=wl.I_s, top_k=wl.top_k, out_dtype="fp32")
    full = moe.moe_layer(x, rw, None, banks.__getitem__, sgu, sdn, sg, **kw)
    shared_only = moe.moe_layer(x, rw, None, banks.__getitem__, sgu, sdn, sg,
                                expert_mask=np.zeros(wl.E, bool), **kw).out64
    for G in (2, 4):
        parts = [moe.moe_layer(x, rw, None, banks.__getitem__, sgu, sdn, sg, include_shared=False,
                               expert_mask=(np.arange(wl.E) % G == r), **kw).out64 for r in range(G)]
        assert np.allclose(sum(parts) + shared_only, full.out64, rtol=1e-12, atol=1e-14)
    # a token whose k experts all sit outside the subset gets exactly zero
    mask = np.zeros(wl.E, bool)
    mask[full.topk_idx[0]] = True
    none = ~mask
    part = moe.moe_layer(x, rw, None, banks.__getitem__, sgu, sdn, sg, include_shared=False,
                         expert_mask=none, **kw).out64
    assert np.all(part[0] == 0.0)


def test_shared_expert_alone_matches_torch():
    rng = np.random.default_rng(17)
    H, I = 64, 32
    x = torch.from_numpy(rng.standard_normal((3, H)).astype(np.float32)).to(torch.bfloat16).float()
    zero_bank = moe.quantize_expert(np.zeros((2 * I, H), np.float32), np.zeros((H, I), np.float32))
    sgu = torch.from_numpy((rng.standard_normal((2 * I, H)) * 0.1).astype(np.float32)).to(torch.bfloat16).double()
    sdn = torch.from_numpy((rng.standard_normal((H, I)) * 0.1).astype(np.float32)).to(torch.bfloat16).double()
    sg = torch.from_numpy((rng.standard_normal(H) * 0.1).astype(np.float32)).to(torch.bfloat16).double()
    res = moe.moe_layer(x.numpy(), np.ones((1, H), np.float32), None, lambda e: zero_bank,
                        sgu.numpy(), sdn.numpy(), sg.numpy(), I=I, I_s=I, top_k=1, out_dtype="fp32")
    xd = x.double()
    Gs = torch.nn.functional.linear(xd, sgu)
    hs = (torch.nn.functional.silu(Gs[:, :I]) * Gs[:, I:])
    hs = torch.from_numpy(nvfp4.bf16_round(hs.numpy()))
    S = torch.nn.functional.linear(hs, sdn)
    ref = torch.sigmoid(xd @ sg)[:, None] * S
    assert np.allclose(res.out64, ref.numpy(), rtol=1e-12, atol=1e-14)


def test_zero_input_gives_zero_output():
    wl = wl_mod.WORKLOADS["tiny"]
    x, rw, get, sgu, sdn, sg = _tiny_inputs(wl)
    res = moe.moe_layer(np.zeros_like(x), rw, None, get, sgu, sdn, sg,
                        I=wl.I, I_s=wl.I_s, top_k=wl.top_k)
    assert np.all(res.out == 0.0)


def test_dominant_router_row_selects_one_expert():
    wl = wl_mod.WORKLOADS["tiny"]
    x, rw, get, sgu, sdn, sg = _tiny_inputs(wl)
    rw = rw.copy()
    rw[6] = np.sign(x[0]) * 50.0               # token 0's logit for expert 6 is huge
    res = moe.moe_layer(x, rw, None, get, sgu, sdn, sg, I=wl.I, I_s=wl.I_s, top_k=2, out_dtype="fp32")
    assert res.topk_idx[0, 0] == 6 and res.topk_w[0, 1] == 0.0
    xc, xs = nvfp4.quantize_activation_rows(x[:1])
    y6 = moe.expert_pair_outputs(get(6), nvfp4.dequantize_rows(xc, xs), wl.I, 0, wl.I)
    S, sigma = moe.shared_expert(x[:1], sgu, sdn, sg, wl.I_s, 0, wl.I_s)
    assert np.allclose(res.out64[0], y6[0] + sigma[0] * S[0], rtol=1e-13, atol=1e-15)


def test_slice_identity_every_partition():
    """Windows that cover I exactly once sum to the unsliced output
    (exact in exact arithmetic; fp64 rounding only)."""
    wl = wl_mod.WORKLOADS["tiny"]
    x, rw, get, sgu, sdn, sg = _tiny_inputs(wl)
    full = moe.moe_layer(x, rw, None, get, sgu, sdn, sg, I=wl.I, I_s=wl.I_s, top_k=wl.top_k)
    nblk = wl.I // 16

    def compositions(n):
        if n == 0:
            yield []
            return
        for first in range(1, n + 1):
            for rest in compositions(n - first):
                yield [first] + rest

    count = 0
    for comp in compositions(nblk):
        i0 = 0
        acc = np.zeros_like(full.out64)
        for nb in comp:
            part = moe.moe_layer(x, rw, None, get, sgu, sdn, sg, I=wl.I, I_s=wl.I_s,
                                 top_k=wl.top_k, i0=i0, I_loc=nb * 16)
            assert np.array_equal(part.topk_idx, full.topk_idx)
            acc += part.out64
            i0 += nb * 16
        assert np.allclose(acc, full.out64, rtol=1e-12, atol=1e-13)
        count += 1
    assert count == 2 ** (nblk - 1)


def test_tokens_subset_matches_full():
    wl = wl_mod.WORKLOADS["tiny"]
    x, rw, get, sgu, sdn, sg = _tiny_inputs(wl)
    full = moe.moe_layer(x, rw, None, get, sgu, sdn, sg, I=wl.I, I_s=wl.I_s, top_k=wl.top_k)
    sub = moe.moe_layer(x, rw, None, get, sgu, sdn, sg, I=wl.I, I_s=wl.I_s, top_k=wl.top_k,
                        tokens=np.array([2, 0]))
    assert np.array_equal(sub.out[[0, 2]], full.out[[0, 2]])
    assert np.all(np.isnan(sub.out[[1, 3]]))


# ---------------------------------------------------------------- figures on the pages

def test_slot_bytes_match_pages():
    g = json.load(open(GOLDEN))
    f = g["slot_bytes_half_slice"]
    b = moe.expert_slice_bytes(f["H"], f["I_loc"])
    assert b == 1395200
    assert round(moe.bytes_per_mib(b), 2) == f["value_mib"]
    # two half slices plus one extra set of down globals make a whole expert
    assert moe.expert_slice_bytes(f["H"], f["I"]) + f["H"] * 4 == 2 * b
    s = g["slots_times_slot_bytes"]
    gib = s["slots"] * b / float(1 << 30)
    assert abs(gib - s["value_gib"]) / s["value_gib"] < s["rel_tol"]


def test_residency_arithmetic_matches_pages():
    g = json.load(open(GOLDEN))
    f = g["expert_layer_slices"]
    assert f["experts"] * f["layers"] == f["value"]
    for key in ("residency_tp1", "residency_tp2"):
        r = g[key]
        pct = 100 * moe.residency_fraction(r["slots"], f["experts"], f["layers"])
        assert round(pct) == r["percent"]


def test_allreduce_bytes_match_pages():
    g = json.load(open(GOLDEN))
    for key in ("allreduce_bs1_H4096", "allreduce_decode_2560"):
        f = g[key]
        assert moe.allreduce_bytes(f["bs"], f["H"]) == f["bytes"]


def test_rms_renorm_hand_worked_rows():
    """Rows worked out by hand from x = bf16(y / sqrt(mean(y^2) + 1e-6)).

    * four values of 1e-3: mean square 1e-6 equals eps, so x = 1e-3 /
      sqrt(2e-6) = 0.70710678..., whose nearest bf16 is 362/512 = 0.70703125
      (eps = 1e-5 would give 0.3015...);
    * (3, -4, 0, 0): mean square 25/4, x = (1.2, -1.6, 0, 0) up to 8e-8, i.e.
      bf16 154/128 and -205/128 (a sum over H - 1 = 3 would give 1.039...);
    * (1e-4, 0, 0, 0): eps dominates, x0 = 1e-4 / sqrt(1.0025e-6) =
      0.09987..., bf16 205/2048 (eps = 1e-5 would give 0.0316...);
    * zeros stay zero (no 0/0)."""
    y = np.array([[1e-3] * 4, [3.0, -4.0, 0.0, 0.0], [1e-4, 0.0, 0.0, 0.0], [0.0] * 4])
    want = np.array([[362 / 512] * 4, [154 / 128, -205 / 128, 0.0, 0.0], [205 / 2048, 0.0, 0.0, 0.0],
                     [0.0] * 4])
    assert np.array_equal(moe.rms_renorm(y), want)


def test_rms_renorm_matches_torch():
    rng = np.random.default_rng(18)
    y = rng.standard_normal((3, 256)) * 5
    r = moe.rms_renorm(y)
    ref = torch.from_numpy(y).float()
    ref = (ref / torch.sqrt((ref.double() ** 2).mean(1, keepdim=True) + 1e-6).float()).to(torch.bfloat16)
    assert np.max(np.abs(r - ref.double().numpy())) <= 2 ** -7 * np.max(np.abs(r))
