"""Plain fp64 oracle of the routed NVFP4 MoE layer (TEST INFRASTRUCTURE ONLY).

Each function states the passage it follows.  Pages, by title:

* [PR385] "feat(qwen4_exp): tensor parallelism for Qwen3.8-Flash-Next
  (offload backend)".
* [I62] "Offloaded MoE ignores tensor parallelism: TP=2 is a regression, and
  the fix is not expert parallelism".

The layer, for tokens x [T, H] (bf16 values) and the intermediate window
[i0, i0 + I_loc):

1. router logits l = x . W_r^T (+ b), fp64 with exact products;
2. top-k by (logit descending, expert ascending), weights renormalised over
   the chosen k (norm_topk_prob) or the full softmax otherwise;
3. counting sort of the pairs p = t*k + j by expert -> offsets, perm, inv;
4. per pair: G = W_gu[window rows] . xq_t, h = silu(G_gate) * G_up, rounded to
   fp32 and NVFP4-quantised, Y_p = W_dn[:, window] . hq;
5. shared expert on the bf16 x: Gs = Ws_gu[window rows] . x,
   hs = bf16(silu(Gs_gate) * Gs_up), S_t = Ws_dn[:, window] . hs,
   sigma_t = 1 / (1 + exp(-g . x_t));
6. out_t = sum_j w_tj * Y_{p(t,j)} + sigma_t * S_t in fp64, rounded once.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, Optional

import numpy as np

from . import nvfp4


# --------------------------------------------------------------------------
# 1-2. router and top-k
# --------------------------------------------------------------------------

def router_logits(x, router_w, router_bias=None) -> np.ndarray:
    """Router logits [T, E] in fp64.

    The router is replicated and runs on the unquantised hidden state
    ([PR385] "What this adds", first bullet: the router stays replicated).
    ``x`` holds bf16 values and ``router_w`` fp32 values, so every product is
    exact in fp64; the sum is an fp64 sum.  The optional per-expert bias is
    added after the sum."""
    x64 = np.asarray(x, dtype=np.float64)
    w64 = np.asarray(router_w, dtype=np.float64)
    logits = x64 @ w64.T
    if router_bias is not None:
        logits = logits + np.asarray(router_bias, dtype=np.float64)[None, :]
    return logits


def select_topk(logits, k: int, norm_topk_prob: bool = True):
    """Top-k experts per token and their routing weights.

    Softmax then top-k, renormalised over the chosen experts when
    norm_topk_prob is set ([I62], first comment, "And the parts you predicted
    would be free were free": norm_topk_prob defaults to True).  The pages fix
    no tie-break; the reading taken is a total order by logit descending, then
    expert index ascending, and the slots are listed in that order.

    Returns (idx int32 [T, k], w fp64 [T, k])."""
    l = np.asarray(logits, dtype=np.float64)
    T, E = l.shape
    if not 1 <= k <= E:
        raise ValueError("k must be in [1, E]")
    # a stable sort of -l keeps the lower expert index first among equal logits
    order = np.argsort(-l, axis=1, kind="stable")
    idx = order[:, :k].astype(np.int32)
    chosen = np.take_along_axis(l, order[:, :k], axis=1)
    lmax = l.max(axis=1, keepdims=True)
    if norm_topk_prob:
        ex = np.exp(chosen - lmax)
        w = ex / ex.sum(axis=1, keepdims=True)
    else:
        full = np.exp(l - lmax)
        w = np.take_along_axis(full / full.sum(axis=1, keepdims=True), order[:, :k], axis=1)
    return idx, w


# --------------------------------------------------------------------------
# 3. counting sort
# --------------------------------------------------------------------------

def counting_sort(idx, num_experts: int):
    """Token->expert permutation by counting sort.

    Pairs are numbered p = t*k + j.  A histogram over experts, its exclusive
    scan, then a scatter of the pairs in increasing p gives, per expert, its
    pairs in increasing p.  ``perm[s]`` is the pair at sorted position s,
    ``inv[p]`` the sorted position of pair p, and ``offsets[e]`` the first
    sorted position of expert e (offsets[E] = T*k).  The pages' expert kernels
    are "dense-in/dense-out" ([I62], first comment); the sort is how the
    grouped contraction gathers each expert's rows."""
    flat = np.asarray(idx, dtype=np.int64).reshape(-1)
    P = flat.size
    counts = np.zeros(num_experts, dtype=np.int64)
    for e in flat:
        counts[e] += 1
    offsets = np.zeros(num_experts + 1, dtype=np.int64)
    for e in range(num_experts):
        offsets[e + 1] = offsets[e] + counts[e]
    cursor = offsets[:-1].copy()
    perm = np.empty(P, dtype=np.int64)
    inv = np.empty(P, dtype=np.int64)
    for p in range(P):
        e = flat[p]
        perm[cursor[e]] = p
        inv[p] = cursor[e]
        cursor[e] += 1
    return offsets.astype(np.int32), perm.astype(np.int32), inv.astype(np.int32)


# --------------------------------------------------------------------------
# 4-6. the layer
# --------------------------------------------------------------------------

def silu(z):
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


@dataclass
class ExpertBank:
    """One expert's NVFP4 bank, unsliced.

    gate_up: codes [2I, H/2], scales [2I, H/16], globals [2I]; gate rows are
    [0, I) and up rows [I, 2I).  down: codes [H, I/2], scales [H, I/16],
    globals [H]  ([I62] "What it touches")."""
    gu_codes: np.ndarray
    gu_scales: np.ndarray
    gu_global: np.ndarray
    dn_codes: np.ndarray
    dn_scales: np.ndarray
    dn_global: np.ndarray


def quantize_expert(gate_up_f32, down_f32) -> ExpertBank:
    """Quantise one expert's fp32 masters with the oracle's own encoder."""
    c, s, g = nvfp4.quantize_weight_rows(gate_up_f32)
    dc, ds, dg = nvfp4.quantize_weight_rows(down_f32)
    return ExpertBank(c, s, g, dc, ds, dg)


def slice_window_rows(I: int, i0: int, I_loc: int) -> np.ndarray:
    """Row indices of gate_up that an intermediate window [i0, i0+I_loc)
    keeps: two disjoint row ranges, gate [i0, i0+I_loc) and up
    [I+i0, I+i0+I_loc)  ([I62] "What it touches")."""
    check_window(I, i0, I_loc)
    return np.concatenate([np.arange(i0, i0 + I_loc), np.arange(I + i0, I + i0 + I_loc)])


def check_window(I: int, i0: int, I_loc: int) -> None:
    """I_loc (and i0) must be multiples of the 16-wide NVFP4 block
    ([I62] "What it touches", the divisibility guard)."""
    if I_loc <= 0 or i0 < 0 or i0 + I_loc > I:
        raise ValueError("window [i0, i0+I_loc) must lie inside [0, I)")
    if I_loc % nvfp4.BLOCK or i0 % nvfp4.BLOCK:
        raise ValueError("i0 and I_loc must be multiples of 16")


def expert_pair_intermediate(bank: ExpertBank, xq_rows: np.ndarray, I: int, i0: int, I_loc: int):
    """The W4A4 intermediate of one expert's m pairs: G = W_gu[window rows] .
    xq in fp64, h = silu(G_gate) * G_up, rounded to fp32 and quantised per
    16-block along the window with global 1.0.  Returns (codes uint8
    [m, I_loc/2], scales uint8 [m, I_loc/16]); the same steps as
    expert_pair_outputs' "nvfp4" mode."""
    rows = slice_window_rows(I, i0, I_loc)
    w_gu = nvfp4.dequantize_rows(bank.gu_codes[rows], bank.gu_scales[rows], bank.gu_global[rows])
    G = xq_rows @ w_gu.T                                   # [m, 2*I_loc]
    h = silu(G[:, :I_loc]) * G[:, I_loc:]
    return nvfp4.quantize_activation_rows(h.astype(np.float32))


def expert_pair_outputs(bank: ExpertBank, xq_rows: np.ndarray, I: int, i0: int, I_loc: int,
                        activations: str = "nvfp4"):
    """Y rows [m, H] (fp64) of one expert for the activations of its m pairs
    (``xq_rows`` [m, H] fp64: dequantised NVFP4 values, or the bf16 values
    themselves in the bf16-activation mode).

    G = W_gu[window rows] . xq in fp64; h = silu(G_gate) * G_up; then
    * activations "nvfp4" (W4A4, the layer's reading): h rounded to fp32 and
      quantised per 16-block along the window with global 1.0;
    * activations "bf16" (W4A16, the weight-only 4-bit kernel the pages'
      review thread selects for this backend, PR #385 mirror, kernel-selection
      fix): h rounded to bf16, as the shared expert's intermediate;
    Y = W_dn[:, window] . h  (gate/up rows and down columns per [I62]
    "What it touches"; SwiGLU on the gate/up pair)."""
    rows = slice_window_rows(I, i0, I_loc)
    w_gu = nvfp4.dequantize_rows(bank.gu_codes[rows], bank.gu_scales[rows], bank.gu_global[rows])
    G = xq_rows @ w_gu.T                                   # [m, 2*I_loc]
    h = silu(G[:, :I_loc]) * G[:, I_loc:]
    if activations == "bf16":
        hq = nvfp4.bf16_round(h)
    elif activations == "nvfp4":
        h32 = h.astype(np.float32)
        hc, hs = nvfp4.quantize_activation_rows(h32)
        hq = nvfp4.dequantize_rows(hc, hs)                 # [m, I_loc]
    else:
        raise ValueError("activations must be 'nvfp4' or 'bf16'")
    c0, c1 = i0 // 2, (i0 + I_loc) // 2
    b0, b1 = i0 // nvfp4.BLOCK, (i0 + I_loc) // nvfp4.BLOCK
    w_dn = nvfp4.dequantize_rows(bank.dn_codes[:, c0:c1], bank.dn_scales[:, b0:b1], bank.dn_global)
    return hq @ w_dn.T                                     # [m, H]


def shared_expert(x, sh_gate_up, sh_down, sh_gate, I_s: int, i0: int, I_loc: int):
    """Shared expert and its sigmoid gate on the bf16 hidden state.

    Gs = Ws_gu[window rows] . x (fp64), hs = bf16(silu(Gs_gate) * Gs_up),
    S_t = Ws_dn[:, window] . hs, sigma_t = 1 / (1 + exp(-g . x_t)).
    The shared gate_up is sharded per part and down is row-parallel
    ([PR385] "What this adds", first bullet).  Returns (S [T, H], sigma [T])."""
    x64 = np.asarray(x, dtype=np.float64)
    rows = slice_window_rows(I_s, i0, I_loc)
    wgu = np.asarray(sh_gate_up, dtype=np.float64)[rows]
    Gs = x64 @ wgu.T
    hs = nvfp4.bf16_round(silu(Gs[:, :I_loc]) * Gs[:, I_loc:])
    wdn = np.asarray(sh_down, dtype=np.float64)[:, i0:i0 + I_loc]
    S = hs @ wdn.T
    z = x64 @ np.asarray(sh_gate, dtype=np.float64)
    sigma = 1.0 / (1.0 + np.exp(-z))
    return S, sigma


@dataclass
class LayerResult:
    out64: np.ndarray          # [T, H] fp64 before the final rounding
    out: np.ndarray            # [T, H] rounded once to the output type (fp64 holder)
    topk_idx: np.ndarray
    topk_w: np.ndarray
    offsets: np.ndarray
    perm: np.ndarray
    inv: np.ndarray
    logits: np.ndarray
    x_codes: np.ndarray
    x_scales: np.ndarray


def moe_layer(x, router_w, router_bias, get_expert: Callable[[int], ExpertBank],
              sh_gate_up, sh_down, sh_gate, *, I: int, I_s: int, top_k: int,
              i0: int = 0, I_loc: Optional[int] = None, norm_topk_prob: bool = True,
              out_dtype: str = "bf16", tokens: Optional[np.ndarray] = None,
              activations: str = "nvfp4", expert_mask: Optional[np.ndarray] = None,
              include_shared: bool = True) -> LayerResult:
    """The whole layer for the window [i0, i0+I_loc) (default: all of I).

    ``x`` [T, H] holds bf16 values (any float dtype).  ``get_expert(e)``
    returns expert e's bank.  Routing always runs over the full replicated
    router.  The combine is routed + sigmoid(gate) * shared formed before any
    reduction ([PR385] "What this adds", third bullet) in fp64 and rounded
    once.  With a window, the result is the partial sum whose sum over a
    partition of I is the full layer ([I62] "The fix that fits").

    ``tokens`` restricts the per-token outputs to a subset (routing and the
    permutation are still computed for all T); rows outside it are NaN.

    ``activations`` selects the expert contractions' activation format:
    "nvfp4" (x and the intermediate NVFP4-quantised, the layer's reading) or
    "bf16" (x as given and the intermediate rounded to bf16: weight-only
    4-bit, see ``expert_pair_outputs``).

    ``expert_mask`` (bool [E]) keeps only the slots whose expert is in it, and
    ``include_shared`` drops the gated shared expert when False: with both,
    the result is what one rank of an expert-parallel layer contributes when
    it owns those experts ([I62] "Why not expert parallelism proper")."""
    if I_loc is None:
        I_loc = I - i0
    check_window(I, i0, I_loc)
    if I_s != I:
        # the shared window follows the routed one scaled by I_s / I
        si0, sil = i0 * I_s // I, I_loc * I_s // I
        check_window(I_s, si0, sil)
    else:
        si0, sil = i0, I_loc
    x32 = np.asarray(x, dtype=np.float32)
    T, H = x32.shape
    logits = router_logits(x32, router_w, router_bias)
    idx, w = select_topk(logits, top_k, norm_topk_prob)
    E = np.asarray(router_w).shape[0]
    offsets, perm, inv = counting_sort(idx, E)
    xc, xs = nvfp4.quantize_activation_rows(x32)
    xq = nvfp4.dequantize_rows(xc, xs) if activations == "nvfp4" else x32.astype(np.float64)

    sel = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    want = np.zeros(T, dtype=bool)
    want[sel] = True
    Y = {}
    keep = np.ones(E, dtype=bool) if expert_mask is None else np.asarray(expert_mask, dtype=bool)
    for e in range(E):
        if not keep[e]:
            continue
        pairs = perm[offsets[e]:offsets[e + 1]]
        pairs = [int(p) for p in pairs if want[int(p) // top_k]]
        if not pairs:
            continue
        toks = np.array([p // top_k for p in pairs])
        ye = expert_pair_outputs(get_expert(e), xq[toks], I, i0, I_loc, activations)
        for r, p in enumerate(pairs):
            Y[p] = ye[r]
    S, sigma = shared_expert(x32[sel], sh_gate_up, sh_down, sh_gate, I_s, si0, sil)
    out64 = np.full((T, H), np.nan)
    for r, t in enumerate(sel):
        acc = np.zeros(H)
        for j in range(top_k):
            if keep[idx[t, j]]:
                acc = acc + w[t, j] * Y[int(t) * top_k + j]
        out64[t] = acc + sigma[r] * S[r] if include_shared else acc
    if out_dtype == "bf16":
        out = nvfp4.bf16_round(out64)
    elif out_dtype == "fp32":
        out = out64.astype(np.float32).astype(np.float64)
    else:
        raise ValueError("out_dtype must be 'bf16' or 'fp32'")
    return LayerResult(out64, out, idx, w, offsets, perm, inv, logits, xc, xs)


def rms_renorm(y, eps: float = 1e-6) -> np.ndarray:
    """Hidden state passed between the layers of a stack: y / sqrt(mean(y^2)
    + eps) per token, rounded to bf16; no residual and no learned weight (the
    stack workload's "renormalised by RMS between layers, with no
    attention")."""
    y64 = np.asarray(y, dtype=np.float64)
    r = np.sqrt(np.mean(y64 * y64, axis=1, keepdims=True) + eps)
    return nvfp4.bf16_round(y64 / r)


# --------------------------------------------------------------------------
# byte accounting of a bank slice (pinned against the slot size on the pages)
# --------------------------------------------------------------------------

def expert_slice_bytes(H: int, I_loc: int) -> int:
    """Bytes of one expert's bank restricted to an I_loc-wide window.

    gate/up rows: 2*I_loc rows of H/2 code bytes, H/16 scale bytes and one
    fp32 global; down: H rows of I_loc/2 code bytes and I_loc/16 scale bytes,
    and all H fp32 row globals, since a per-row global of a down row cannot
    be split by a column slice ([PR385] "What this adds", second bullet)."""
    gu = 2 * I_loc * (H // 2 + H // 16 + 4)
    dn = H * (I_loc // 2 + I_loc // 16) + H * 4
    return gu + dn


def bytes_per_mib(n: int) -> float:
    return n / float(1 << 20)


def allreduce_bytes(bs: int, H: int, elem_bytes: int = 2) -> int:
    """Size of the one reduce per MoE layer: bs * H elements
    ([I62] "The fix that fits", "No new collectives")."""
    return bs * H * elem_bytes


def residency_fraction(slots: int, experts: int, layers: int) -> float:
    """Share of a rank's expert-layer slices that an offload cache of
    ``slots`` holds.  A rank needs one slice (whole or its intermediate-axis
    part) of every expert in every MoE layer, and a slot holds one such
    slice ([I62] comment "Your extrapolation holds at a residency point
    neither of your boxes sits at")."""
    return slots / float(experts * layers)


__all__ = [
    "router_logits", "select_topk", "counting_sort", "silu", "ExpertBank",
    "quantize_expert", "slice_window_rows", "check_window", "expert_pair_outputs",
    "shared_expert", "LayerResult", "moe_layer", "rms_renorm", "expert_slice_bytes",
    "bytes_per_mib", "allreduce_bytes", "residency_fraction",
]
