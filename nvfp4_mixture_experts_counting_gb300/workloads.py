"""Seeded synthetic inputs for the routed NVFP4 MoE layer.

This module only draws numbers: it holds none of the layer's arithmetic (no
quantisation, routing or contraction).  The tests feed what it draws both to
the CUDA library and to the CPU oracle; the benchmark feeds it to the library.

Workloads (all synthetic; no dataset or trained weights exist for this path):

* ``tiny``      T=4, H=256, E=8, top_k=2, I=I_s=64.
* ``mid``       H=512, I=I_s=256, E=16, top_k=4, T in {33, 100, 600}: the
                smallest layer whose shapes take the tensor-core path, small
                enough for the oracle to check every token.
* ``decode``    H=2560, I=I_s=640, E=256, top_k=8, T in {1, 8, 16}.
* ``stack48``   the decode layer as 48 layers of independent weights.
* ``prefill``   the decode layer's sizes, T in {1024, 4096, 16384}, with a
                per-expert router bias b[pi[r-1]] = -1.1 * ln(r) over a random
                expert order pi (a Zipf(s=1.1) prior), so routing is skewed.
* ``offload``   H=4096, I=I_s=2048, E=256, top_k=8, T in {1, 16, 2048}.

Distributions: hidden bf16 from N(0, 1); router weights fp32 N(0, 0.02);
expert fp32 masters N(0, 0.02) (quantised to NVFP4 by each side on its own);
shared expert weights and the shared gate vector bf16, drawn in fp32 from
N(0, 0.02) and rounded to bf16.  Every tensor has its own seed derived from
(workload, layer, tensor name, expert), so any one expert can be drawn again
on its own.
"""

from __future__ import annotations

import math
import zlib
from dataclasses import dataclass, field
from typing import Optional, Tuple

import torch

STD_W = 0.02


@dataclass(frozen=True)
class Workload:
    name: str
    H: int
    I: int
    E: int
    top_k: int
    I_s: int
    tokens: Tuple[int, ...]
    layers: int = 1
    router_bias: bool = False
    norm_topk_prob: bool = True
    slices: Tuple[Tuple[int, int], ...] = field(default_factory=tuple)


WORKLOADS = {
    "tiny": Workload("tiny", H=256, I=64, E=8, top_k=2, I_s=64, tokens=(4,),
                     slices=((0, 16), (16, 48))),
    "mid": Workload("mid", H=512, I=256, E=16, top_k=4, I_s=256, tokens=(33, 100, 600)),
    "decode": Workload("decode", H=2560, I=640, E=256, top_k=8, I_s=640, tokens=(1, 8, 16),
                       slices=((0, 320), (320, 320))),
    "stack48": Workload("stack48", H=2560, I=640, E=256, top_k=8, I_s=640, tokens=(1, 8, 16),
                        layers=48),
    "prefill": Workload("prefill", H=2560, I=640, E=256, top_k=8, I_s=640,
                        tokens=(1024, 4096, 16384), router_bias=True),
    "offload": Workload("offload", H=4096, I=2048, E=256, top_k=8, I_s=2048,
                        tokens=(1, 16, 2048), slices=((0, 1024), (1024, 1024))),
}


def seed_of(*parts) -> int:
    """Deterministic 31-bit seed of a tuple of names and numbers."""
    return zlib.crc32("/".join(str(p) for p in parts).encode()) & 0x7FFFFFFF


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    """fp32 N(0, std^2) draw of ``shape`` from a generator seeded with ``seed``."""
    t = torch.randn(shape, generator=_gen(seed, device), device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t


def hidden(wl: Workload, T: int, step: int = 0, device="cpu", layer: int = 0) -> torch.Tensor:
    """Hidden state x [T, H] bf16, N(0, 1); seed 1000 + T + step."""
    s = 1000 + T + step if layer == 0 else seed_of(wl.name, layer, "x", T, step)
    return normal((T, wl.H), 1.0, s, device).to(torch.bfloat16)


def router_weight(wl: Workload, layer: int = 0, device="cpu") -> torch.Tensor:
    return normal((wl.E, wl.H), STD_W, seed_of(wl.name, layer, "router_w"), device)


def router_bias(wl: Workload, layer: int = 0, device="cpu") -> Optional[torch.Tensor]:
    """Zipf(s=1.1) prior over a random expert order: b[pi[r-1]] = -1.1 ln r."""
    if not wl.router_bias:
        return None
    g = _gen(seed_of(wl.name, layer, "router_bias"), "cpu")
    pi = torch.randperm(wl.E, generator=g)
    b = torch.empty(wl.E, dtype=torch.float32)
    for r in range(1, wl.E + 1):
        b[pi[r - 1]] = -1.1 * math.log(r)
    return b.to(device)


def expert_masters(wl: Workload, e: int, layer: int = 0, device="cpu"):
    """fp32 masters of expert e: gate_up [2I, H] (gate rows first) and down [H, I]."""
    gu = normal((2 * wl.I, wl.H), STD_W, seed_of(wl.name, layer, "gate_up", e), device)
    dn = normal((wl.H, wl.I), STD_W, seed_of(wl.name, layer, "down", e), device)
    return gu, dn


def shared_weights(wl: Workload, layer: int = 0, device="cpu"):
    """Shared expert bf16 gate_up [2I_s, H], down [H, I_s] and gate vector [H]."""
    gu = normal((2 * wl.I_s, wl.H), STD_W, seed_of(wl.name, layer, "sh_gate_up"), device)
    dn = normal((wl.H, wl.I_s), STD_W, seed_of(wl.name, layer, "sh_down"), device)
    g = normal((wl.H,), STD_W, seed_of(wl.name, layer, "sh_gate"), device)
    return gu.to(torch.bfloat16), dn.to(torch.bfloat16), g.to(torch.bfloat16)


def format_matrix(fmt: str, N: int, K: int, seed: int) -> dict:
    """Random bytes of a matrix [N, K] stored in one of the bank formats that
    the loader slices (any byte pattern is a matrix of the format; NaN codes
    are avoided), as numpy arrays named like the format's tensors:

    * ``nvfp4``     codes [N, K/2], E4M3 scales [N, K/16], fp32 globals [N]
    * ``fp8_block`` E4M3 q [N, K], fp32 scale [ceil(N/128), ceil(K/128)]
    * ``q4_0``      blocks [N, K/32, 18] (fp16 scale, then 16 code bytes)
    * ``mxfp4``     blocks_t [K/2, N], UE8M0 scales_t [K/32, N]"""
    import numpy as np
    rng = np.random.default_rng(seed)
    if fmt == "nvfp4":
        return {"codes": rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8),
                "scales": rng.integers(0, 0x7F, size=(N, K // 16), dtype=np.uint8),
                "globals": rng.random(N).astype(np.float32)}
    if fmt == "fp8_block":
        q = rng.integers(0, 256, size=(N, K), dtype=np.uint8)
        q[(q & 0x7F) == 0x7F] = 0
        return {"q": q, "scale": rng.random(((N + 127) // 128, (K + 127) // 128)).astype(np.float32)}
    if fmt == "q4_0":
        blocks = rng.integers(0, 256, size=(N, K // 32, 18), dtype=np.uint8)
        d = (rng.random((N, K // 32)) * 0.01).astype(np.float16)
        blocks[:, :, 0:2] = d.view(np.uint8).reshape(N, K // 32, 2)
        return {"blocks": blocks}
    if fmt == "mxfp4":
        return {"blocks_t": rng.integers(0, 256, size=(K // 2, N), dtype=np.uint8),
                "scales_t": rng.integers(100, 140, size=(K // 32, N), dtype=np.uint8)}
    raise ValueError(fmt)


def bf16_bits(t: torch.Tensor) -> torch.Tensor:
    """The raw 16-bit patterns of a bf16 tensor (as int16)."""
    return t.contiguous().view(torch.int16)
