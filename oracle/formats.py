"""Other expert-bank formats and their intermediate-axis slicing, for the
oracle (TEST INFRASTRUCTURE ONLY).

Issue #62 "Offloaded MoE ignores tensor parallelism: TP=2 is a regression,
and the fix is not expert parallelism", section "What it touches", asks for
per-format bank slicing at load: gate_up [2I, H] keeps two disjoint row
ranges (gate rows [i0, i0+I_loc) and up rows [I+i0, I+i0+I_loc)), down
[H, I] keeps a column range, the slice width must stay a multiple of each
format's block size (128 for fp8_block, 32 for the fp4 scale blocks, 32 for
q4_0), and mxfp4 is stored transposed (blocks_t [K//2, N]), so its slice runs
along N and its scales slice differently again.  Section "Suggested
staging" orders the formats (bf16, then the row-major fp4 formats, then
fp8_block and q4_0, mxfp4 last).

The pages name the formats without spelling out their bytes.  The readings
taken here are the formats' published definitions:

* fp8_block: a matrix W [N, K] of E4M3 ("fn") values, one fp32 scale per
  128 x 128 tile, scales [ceil(N/128), ceil(K/128)]; W[n, k] = e4m3(q[n, k])
  * scale[n // 128, k // 128].
* q4_0: each row of K values in blocks of 32, a block being 18 bytes: an
  IEEE fp16 scale d (little endian) and 16 bytes of 4-bit codes, byte j
  holding element j in its low nibble and element j + 16 in its high nibble;
  value = d * (code - 8).  Stored [N, K/32, 18].
* mxfp4 (OCP microscaling, FP4 elements): E2M1 codes in blocks of 32 along K
  with one UE8M0 scale per block (value 2^(s - 127); 0xFF is NaN), stored
  transposed: blocks_t [K/2, N] with byte [j, n] holding element (n, 2j) in
  its low nibble and (n, 2j+1) in its high nibble, scales_t [K/32, N].
* nvfp4 (the library's own bank): codes [N, K/2], E4M3 scales [N, K/16],
  fp32 row globals [N] (see ``nvfp4``); its slice keeps whole rows and every
  down-row global.

Every slice below is written as plain indexing of the stored arrays, so that
a reader can check it against the layout above; the tests pin it by the
identity dequantise(slice(W)) == slice(dequantise(W)).
"""

from __future__ import annotations

import numpy as np

from . import nvfp4

#: block size along the intermediate axis that a window must respect
BLOCK = {"nvfp4": 16, "fp8_block": 128, "q4_0": 32, "mxfp4": 32}


def check_format_window(fmt: str, I: int, i0: int, I_loc: int) -> None:
    """The divisibility guard of "What it touches": the window (and, for the
    up rows of a row-blocked format, I itself) on the format's block grid."""
    b = BLOCK[fmt]
    if I_loc <= 0 or i0 < 0 or i0 + I_loc > I:
        raise ValueError("window [i0, i0+I_loc) must lie inside [0, I)")
    if i0 % b or I_loc % b or I % b:
        raise ValueError(f"{fmt}: I, i0 and I_loc must be multiples of {b}")


# --------------------------------------------------------------------------
# decoders (value of every element, fp64)
# --------------------------------------------------------------------------

def fp8_block_dequant(q: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """W [N, K] from E4M3 bytes q [N, K] and fp32 tile scales [ceil(N/128), ceil(K/128)]."""
    N, K = q.shape
    v = nvfp4.e4m3_decode(q)
    s = np.asarray(scale, dtype=np.float64)
    return v * s[np.arange(N)[:, None] // 128, np.arange(K)[None, :] // 128]


def q4_0_dequant(blocks: np.ndarray) -> np.ndarray:
    """W [N, K] from q4_0 blocks [N, K/32, 18]."""
    blocks = np.asarray(blocks, dtype=np.uint8)
    N, nb, _ = blocks.shape
    d = blocks[:, :, 0:2].copy().view("<f2")[:, :, 0].astype(np.float64)     # [N, nb]
    qs = blocks[:, :, 2:18]
    lo = (qs & 0xF).astype(np.float64) - 8.0
    hi = (qs >> 4).astype(np.float64) - 8.0
    vals = np.concatenate([lo, hi], axis=2) * d[:, :, None]                 # [N, nb, 32]
    return vals.reshape(N, nb * 32)


def ue8m0_decode(s: np.ndarray) -> np.ndarray:
    s = np.asarray(s, dtype=np.uint8).astype(np.int64)
    return np.where(s == 0xFF, np.nan, np.exp2((s - 127).astype(np.float64)))


def mxfp4_dequant(blocks_t: np.ndarray, scales_t: np.ndarray) -> np.ndarray:
    """W [N, K] from the transposed mxfp4 arrays blocks_t [K/2, N] and
    scales_t [K/32, N]."""
    blocks_t = np.asarray(blocks_t, dtype=np.uint8)
    K2, N = blocks_t.shape
    codes = np.empty((2 * K2, N), dtype=np.uint8)          # [K, N]
    codes[0::2] = blocks_t & 0xF
    codes[1::2] = blocks_t >> 4
    v = nvfp4.e2m1_decode(codes) * np.repeat(ue8m0_decode(scales_t), 32, axis=0)
    return v.T


def nvfp4_dequant(codes, scales, globals_) -> np.ndarray:
    return nvfp4.dequantize_rows(codes, scales, globals_)


def dequant(fmt: str, t: dict) -> np.ndarray:
    """Values [N, K] of one matrix held as the arrays of its format."""
    if fmt == "nvfp4":
        return nvfp4_dequant(t["codes"], t["scales"], t["globals"])
    if fmt == "fp8_block":
        return fp8_block_dequant(t["q"], t["scale"])
    if fmt == "q4_0":
        return q4_0_dequant(t["blocks"])
    if fmt == "mxfp4":
        return mxfp4_dequant(t["blocks_t"], t["scales_t"])
    raise ValueError(fmt)


# --------------------------------------------------------------------------
# slices of one expert's gate_up [2I, H] and down [H, I]
# --------------------------------------------------------------------------

def _gate_up_rows(I: int, i0: int, I_loc: int) -> np.ndarray:
    return np.concatenate([np.arange(i0, i0 + I_loc), np.arange(I + i0, I + i0 + I_loc)])


def slice_gate_up(fmt: str, t: dict, I: int, i0: int, I_loc: int) -> dict:
    """The gate rows [i0, i0+I_loc) and the up rows [I+i0, I+i0+I_loc) of
    gate_up [2I, H], in the format's own arrays."""
    check_format_window(fmt, I, i0, I_loc)
    rows = _gate_up_rows(I, i0, I_loc)
    if fmt == "nvfp4":
        return {"codes": t["codes"][rows], "scales": t["scales"][rows], "globals": t["globals"][rows]}
    if fmt == "fp8_block":
        # whole 128-row tiles: the tile rows of the gate part, then the up part
        trows = np.concatenate([np.arange(i0 // 128, (i0 + I_loc) // 128),
                                np.arange((I + i0) // 128, (I + i0 + I_loc) // 128)])
        return {"q": t["q"][rows], "scale": t["scale"][trows]}
    if fmt == "q4_0":
        return {"blocks": t["blocks"][rows]}
    if fmt == "mxfp4":
        # transposed: output rows are columns of blocks_t and scales_t
        return {"blocks_t": t["blocks_t"][:, rows], "scales_t": t["scales_t"][:, rows]}
    raise ValueError(fmt)


def slice_down(fmt: str, t: dict, I: int, i0: int, I_loc: int) -> dict:
    """The columns [i0, i0+I_loc) of down [H, I], in the format's own arrays;
    the nvfp4 row globals stay whole (a column slice cannot split them)."""
    check_format_window(fmt, I, i0, I_loc)
    if fmt == "nvfp4":
        return {"codes": t["codes"][:, i0 // 2:(i0 + I_loc) // 2],
                "scales": t["scales"][:, i0 // 16:(i0 + I_loc) // 16], "globals": t["globals"]}
    if fmt == "fp8_block":
        return {"q": t["q"][:, i0:i0 + I_loc], "scale": t["scale"][:, i0 // 128:(i0 + I_loc) // 128]}
    if fmt == "q4_0":
        return {"blocks": t["blocks"][:, i0 // 32:(i0 + I_loc) // 32]}
    if fmt == "mxfp4":
        # transposed: K runs down the rows of blocks_t (two per byte) and scales_t
        return {"blocks_t": t["blocks_t"][i0 // 2:(i0 + I_loc) // 2],
                "scales_t": t["scales_t"][i0 // 32:(i0 + I_loc) // 32]}
    raise ValueError(fmt)


__all__ = ["BLOCK", "check_format_window", "fp8_block_dequant", "q4_0_dequant", "ue8m0_decode", "mxfp4_dequant",
           "nvfp4_dequant", "dequant", "slice_gate_up", "slice_down"]
