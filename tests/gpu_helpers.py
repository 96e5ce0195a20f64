"""Test-side helpers: build a library handle from the seeded workload on the
GPU, and give the oracle the same inputs (the fp32 masters are drawn on the
GPU per expert seed and copied to the host for the oracle, which quantises
them with its own encoder)."""

from __future__ import annotations

import numpy as np
import torch

from nvfp4_mixture_experts_counting_gb300 import ftmoe, workloads as W
from oracle import moe

# acceptance bar for bf16 outputs
MAX_ABS = 2e-2
REL_L2 = 5e-3


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


class GpuBank:
    """One layer's weights on the device: fp32 masters quantised by the
    library's own quantiser, plus the bf16/fp32 dense tensors."""

    def __init__(self, wl: W.Workload, layer: int = 0, dev="cuda"):
        self.wl, self.layer = wl, layer
        E, I, H = wl.E, wl.I, wl.H
        gu = torch.empty((E, 2 * I, H), dtype=torch.float32, device=dev)
        dn = torch.empty((E, H, I), dtype=torch.float32, device=dev)
        for e in range(E):
            g, d = W.expert_masters(wl, e, layer, device=dev)
            gu[e].copy_(g)
            dn[e].copy_(d)
        self.gu_codes = torch.empty((E, 2 * I, H // 2), dtype=torch.uint8, device=dev)
        self.gu_scales = torch.empty((E, 2 * I, H // 16), dtype=torch.uint8, device=dev)
        self.gu_global = torch.empty((E, 2 * I), dtype=torch.float32, device=dev)
        self.dn_codes = torch.empty((E, H, I // 2), dtype=torch.uint8, device=dev)
        self.dn_scales = torch.empty((E, H, I // 16), dtype=torch.uint8, device=dev)
        self.dn_global = torch.empty((E, H), dtype=torch.float32, device=dev)
        ftmoe.ftmoe_quantize_weights(gu, E * 2 * I, H, self.gu_codes, self.gu_scales, self.gu_global)
        ftmoe.ftmoe_quantize_weights(dn, E * H, I, self.dn_codes, self.dn_scales, self.dn_global)
        torch.cuda.synchronize()
        del gu, dn
        self.router_w = W.router_weight(wl, layer, device=dev)
        b = W.router_bias(wl, layer)
        self.router_bias = b.to(dev) if b is not None else None
        sgu, sdn, sg = W.shared_weights(wl, layer, device=dev)
        self.sh_gate_up, self.sh_down, self.sh_gate = sgu, sdn, sg
        self._oracle_cache = {}

    def desc(self) -> ftmoe.BankDesc:
        return ftmoe.bank_desc(self.router_w, self.router_bias, self.gu_codes, self.gu_scales,
                               self.gu_global, self.dn_codes, self.dn_scales, self.dn_global,
                               self.sh_gate_up, self.sh_down, self.sh_gate, on_device=True)

    # ---- oracle side
    def oracle_expert(self, e: int) -> moe.ExpertBank:
        if e not in self._oracle_cache:
            g, d = W.expert_masters(self.wl, e, self.layer, device="cuda")
            self._oracle_cache[e] = moe.quantize_expert(g.cpu().numpy(), d.cpu().numpy())
        return self._oracle_cache[e]

    def prefetch_oracle_experts(self, experts, threads: int = 16):
        """Quantise many experts with the oracle's encoder at once: the
        masters are drawn on the GPU first (in this thread), the numpy
        encoding then runs on a thread pool (numpy releases the GIL inside
        its array loops)."""
        from concurrent.futures import ThreadPoolExecutor
        todo = [int(e) for e in experts if int(e) not in self._oracle_cache]
        if not todo:
            return
        masters = {}
        for e in todo:
            g, d = W.expert_masters(self.wl, e, self.layer, device="cuda")
            masters[e] = (g.cpu().numpy(), d.cpu().numpy())
        with ThreadPoolExecutor(max_workers=threads) as ex:
            banks = list(ex.map(lambda e: moe.quantize_expert(*masters[e]), todo))
        for e, b in zip(todo, banks):
            self._oracle_cache[e] = b

    def oracle_layer(self, x_bf16: torch.Tensor, i0=0, I_loc=None, out_dtype="bf16", tokens=None):
        wl = self.wl
        return moe.moe_layer(
            x_bf16.float().cpu().numpy(), self.router_w.cpu().numpy(),
            None if self.router_bias is None else self.router_bias.cpu().numpy(),
            self.oracle_expert, self.sh_gate_up.float().cpu().numpy(),
            self.sh_down.float().cpu().numpy(), self.sh_gate.float().cpu().numpy(),
            I=wl.I, I_s=wl.I_s, top_k=wl.top_k, i0=i0, I_loc=I_loc,
            norm_topk_prob=wl.norm_topk_prob, out_dtype=out_dtype, tokens=tokens)


def make_layer(wl: W.Workload, max_tokens: int, num_layers: int = 1) -> ftmoe.Layer:
    cfg = ftmoe.make_config(H=wl.H, I=wl.I, E=wl.E, top_k=wl.top_k, I_shared=wl.I_s,
                            num_layers=num_layers, max_tokens=max_tokens,
                            norm_topk_prob=wl.norm_topk_prob, has_router_bias=wl.router_bias)
    return ftmoe.Layer(cfg)


class AuxBufs:
    def __init__(self, T, k, E, dev="cuda"):
        P = T * k
        self.topk_idx = torch.full((T, k), -1, dtype=torch.int32, device=dev)
        self.topk_w = torch.zeros((T, k), dtype=torch.float32, device=dev)
        self.offsets = torch.full((E + 1,), -1, dtype=torch.int32, device=dev)
        self.perm = torch.full((P,), -1, dtype=torch.int32, device=dev)
        self.inv = torch.full((P,), -1, dtype=torch.int32, device=dev)
        self.c = ftmoe.Aux(self.topk_idx.data_ptr(), self.topk_w.data_ptr(), self.offsets.data_ptr(),
                           self.perm.data_ptr(), self.inv.data_ptr())

    def numpy(self):
        return {k: getattr(self, k).cpu().numpy() for k in ("topk_idx", "topk_w", "offsets", "perm", "inv")}


def check_routing(aux: AuxBufs, ref: moe.LayerResult):
    got = aux.numpy()
    assert np.array_equal(got["topk_idx"], ref.topk_idx), "top-k indices differ"
    assert np.array_equal(got["offsets"], ref.offsets), "offsets differ"
    assert np.array_equal(got["perm"], ref.perm), "perm differs"
    assert np.array_equal(got["inv"], ref.inv), "inv differs"
    # the weights are fp32 softmaxes of fp32 logits; the tensor-core router's
    # logits carry up to ~2^-19 * ||x|| * ||w|| (~1e-4) of error, which moves a
    # renormalised weight by at most twice that, relatively
    assert np.allclose(got["topk_w"], ref.topk_w, rtol=5e-4, atol=1e-6), "routing weights differ"


def stratified_tokens(topk_idx: np.ndarray, n: int, seed: int, hot: int = 8, per_hot: int = 32) -> np.ndarray:
    """A seeded sample of n tokens that holds, for each of the `hot` most
    loaded experts, up to `per_hot` of the tokens routed to it (the experts
    whose many full 128-row tiles a uniform sample would rarely reach), the
    first and last token, and uniform draws for the rest."""
    T = topk_idx.shape[0]
    if n >= T:
        return np.arange(T)
    g = np.random.default_rng(seed)
    load = np.bincount(topk_idx.reshape(-1), minlength=int(topk_idx.max()) + 1)
    chosen = {0, T - 1}
    for e in np.argsort(-load, kind="stable")[:hot]:
        toks = np.nonzero((topk_idx == e).any(axis=1))[0]
        if toks.size:
            chosen.update(g.choice(toks, size=min(per_hot, toks.size), replace=False).tolist())
    rest = np.setdiff1d(np.arange(T), np.fromiter(chosen, dtype=np.int64))
    chosen.update(g.choice(rest, size=max(0, n - len(chosen)), replace=False).tolist())
    return np.sort(np.fromiter(chosen, dtype=np.int64))


def check_output(out: torch.Tensor, ref_out: np.ndarray, rows=None):
    got = out.float().cpu().numpy().astype(np.float64)
    ref = np.asarray(ref_out, dtype=np.float64)
    if rows is not None:
        got, ref = got[rows], ref[rows]
    mae = float(np.max(np.abs(got - ref)))
    rl2 = rel_l2(got, ref)
    assert mae <= MAX_ABS and rl2 <= REL_L2, f"max-abs {mae:.3e}, rel-L2 {rl2:.3e}"
    return mae, rl2
