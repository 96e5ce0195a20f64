"""Algorithmic byte and flop counts of the MoE layer, for roofline reporting.

Byte counts are those of the bank format itself (packed E2M1 codes, one E4M3
scale per 16 elements, one fp32 global per row), restricted to the
intermediate window a forward uses, with no padding.
"""

from __future__ import annotations


def gate_up_window_bytes(H: int, I_loc: int) -> int:
    """gate_up rows of one expert in a window: 2*I_loc rows of H/2 code bytes,
    H/16 scale bytes and a 4-byte global."""
    return 2 * I_loc * (H // 2 + H // 16 + 4)


def down_window_bytes(H: int, I_loc: int) -> int:
    """down of one expert in a window: H rows of I_loc/2 code bytes and
    I_loc/16 scale bytes, plus all H row globals."""
    return H * (I_loc // 2 + I_loc // 16 + 4)


def expert_window_bytes(H: int, I_loc: int) -> int:
    return gate_up_window_bytes(H, I_loc) + down_window_bytes(H, I_loc)


def shared_window_bytes(H: int, sI_loc: int) -> int:
    """bf16 shared expert: gate and up rows (2*sI_loc x H) and down columns
    (H x sI_loc), plus the bf16 gate vector."""
    return 2 * sI_loc * H * 2 + H * sI_loc * 2 + H * 2


def layer_touched_bytes(H: int, E: int, I_loc: int, sI_loc: int, T: int, touched: int,
                        out_bytes_per_elem: int = 2) -> int:
    """HBM bytes one forward must move at least: the touched experts' window
    bytes, the shared expert, the fp32 router, x in and out."""
    return (touched * expert_window_bytes(H, I_loc) + shared_window_bytes(H, sI_loc)
            + E * H * 4 + T * H * 2 + T * H * out_bytes_per_elem)


def routed_flops(H: int, I_loc: int, pairs: int) -> int:
    """Multiply-adds x 2 of the routed experts: gate_up (2*I_loc x H) and down
    (H x I_loc) per token-expert pair."""
    return pairs * (2 * H * 2 * I_loc + 2 * I_loc * H)


def shared_flops(H: int, sI_loc: int, tokens: int) -> int:
    """Multiply-adds x 2 of the bf16 shared expert: gate_up (2*sI_loc x H)
    and down (H x sI_loc) per token."""
    return tokens * (2 * H * 2 * sI_loc + 2 * sI_loc * H)


def router_flops(H: int, E: int, tokens: int) -> int:
    """Multiply-adds x 2 of the router logits, [T, H] x [H, E]."""
    return tokens * 2 * H * E


def combined_ideal_seconds(H: int, E: int, I_loc: int, sI_loc: int, T: int, pairs: int, touched: float,
                           fp4_tflops: float, bf16_tflops: float, hbm_gbs: float,
                           router_bf16_parts: int = 3) -> dict:
    """The layer's time at its combined roofline: the routed FP4 flops at the
    NVFP4 peak, plus the shared expert's flops at the bf16 peak, plus the
    router's flops at the bf16 peak times the bf16 parts it is computed in
    (an fp32 router row is three exact bf16 parts), against the touched
    bytes at the HBM peak; the larger of the two is the bound."""
    t_tensor = (routed_flops(H, I_loc, pairs) / (fp4_tflops * 1e12)
                + shared_flops(H, sI_loc, T) / (bf16_tflops * 1e12)
                + router_bf16_parts * router_flops(H, E, T) / (bf16_tflops * 1e12))
    t_hbm = layer_touched_bytes(H, E, I_loc, sI_loc, T, int(round(touched))) / (hbm_gbs * 1e9)
    return {"tensor_s": t_tensor, "hbm_s": t_hbm, "bound_s": max(t_tensor, t_hbm),
            "bound": "tensor" if t_tensor >= t_hbm else "hbm"}


def kernel_unit_bytes(kernel: str, H: int, I_loc: int, sI_loc: int, E: int = 0):
    """(bytes per unit, unit name, fixed bytes per launch) of a kernel's
    algorithmic HBM traffic; units are touched experts where named so."""
    if kernel in ("k_gate_up", "k_dec_gate_up"):
        return gate_up_window_bytes(H, I_loc), "touched expert (gate_up window)", 0
    if kernel == "k_down":
        return down_window_bytes(H, I_loc), "touched expert (down window)", 0
    if kernel == "k_dec_down":
        # routed down rows of every touched expert, plus the shared expert's
        # bf16 down columns (one launch streams both)
        return down_window_bytes(H, I_loc), "touched expert (down window), + shared down", H * sI_loc * 2
    if kernel == "k_dtc_gate_up":
        # routed gate_up rows of every touched expert, plus the shared expert's
        # bf16 gate_up rows (one launch streams both)
        return gate_up_window_bytes(H, I_loc), "touched expert (gate_up window), + shared gate_up", 2 * sI_loc * H * 2
    if kernel == "k_dtc_down":
        return down_window_bytes(H, I_loc), "touched expert (down window), + shared down", H * sI_loc * 2
    if kernel == "k_dec_route":
        # fp32 router and the shared expert's bf16 gate_up rows
        return 0, "launch (router + shared gate_up)", E * H * 4 + 2 * sI_loc * H * 2
    if kernel == "k_shared_gate_up":
        return 0, "launch (shared gate_up rows)", 2 * sI_loc * H * 2
    if kernel == "k_shared_down":
        return 0, "launch (shared down columns)", H * sI_loc * 2
    return None, None, None


def kernel_unit_flops(kernel: str, H: int, I_loc: int, sI_loc: int, E: int = 0):
    """(flops per unit, unit name, datapath) of a contraction kernel, or
    (None, None, None).  Units are token-expert pairs for the routed GEMMs
    and tokens for the shared expert and the router; flops = 2 x
    multiply-adds of the contraction as defined, no padding counted."""
    if kernel == "k_pf_gate_up":
        return 2 * H * 2 * I_loc, "pair", "nvfp4 tensor"
    if kernel == "k_pf_down":
        return 2 * I_loc * H, "pair", "nvfp4 tensor"
    if kernel == "k_pf_shared_gate_up":
        return 2 * H * 2 * sI_loc, "token", "bf16 tensor"
    if kernel == "k_pf_shared_down":
        return 2 * sI_loc * H, "token", "bf16 tensor"
    if kernel == "k_pf_router":
        # x times the three exact bf16 parts of every fp32 router row
        return 3 * 2 * H * E, "token", "bf16 tensor"
    if kernel == "k_shared_gate_up":
        return 2 * H * 2 * sI_loc, "token", "fp32 CUDA cores"
    if kernel == "k_shared_down":
        return 2 * sI_loc * H, "token", "fp32 CUDA cores"
    if kernel == "k_router_logits":
        return 2 * H * E, "token", "fp32 CUDA cores"
    return None, None, None
