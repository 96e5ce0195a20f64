"""NVFP4 encoding and decoding for the oracle (TEST INFRASTRUCTURE ONLY).

The bank format is the one PR #385 "feat(qwen4_exp): tensor parallelism for
Qwen3.8-Flash-Next (offload backend)", section "What this adds", names for the
expert banks: packed E2M1 codes, 16-wide scale blocks and per-row globals.
The pages do not spell the arithmetic out; the readings taken here are:

* E2M1 (4 bits: sign, 2 exponent bits, 1 mantissa bit) encodes the
  magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}.  Encoding rounds to nearest with
  ties to the even code, saturates at 6, and gives a zero magnitude the sign
  bit 0.
* Scales are E4M3 "fn" (bias 7, no infinities, 0x7F/0xFF are NaN, largest
  finite 448, subnormals m * 2**-9).  Encoding rounds to nearest with ties to
  the even code and saturates at 448.  Scales are never negative.
* Two codes share a byte: element 2j sits in the low nibble of byte j.
* Weight rows: g = fp32(row_amax / 2688) with 2688 = 448 * 6; per 16-block,
  s = E4M3(fp32(fp32(block_amax / 6) / g)); each element is encoded as
  E2M1(fp32(w / fp32(dec(s) * g))).  A zero row (g = 0), a zero scale, or a
  zero denominator encodes every code of the block as 0.
* Activations (token rows of x and pair rows of the SwiGLU output) use the
  same block steps with the global fixed at 1.0.  The pages say nothing about
  activation quantisation; it is the design reading that makes the layer a
  W4A4 NVFP4 contraction (parity unpinned by the pages).
* Dequantisation is dec(code) * dec(scale) * g, formed in fp64.

All fp32 steps use IEEE single precision with correctly rounded division, in
exactly the order written above.
"""

from __future__ import annotations

import numpy as np

BLOCK = 16
E2M1_MAX = 6.0
E4M3_MAX = 448.0
WEIGHT_GLOBAL_DIVISOR = np.float32(E4M3_MAX * E2M1_MAX)  # 2688

#: E2M1 magnitudes indexed by the low three bits of a code.
E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)


def e2m1_decode(codes) -> np.ndarray:
    """Value of each 4-bit E2M1 code (0..15), as fp64."""
    c = np.asarray(codes, dtype=np.uint8) & 0xF
    mag = E2M1_MAGNITUDES[c & 0x7]
    return np.where(c & 0x8, -mag, mag)


def e4m3_decode(codes) -> np.ndarray:
    """Value of each E4M3 "fn" byte, as fp64 (NaN for 0x7F and 0xFF)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    sub = m * 2.0 ** -9
    val = np.where(e == 0, sub, normal)
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return sign * val


def _nearest_even(table: np.ndarray, u: np.ndarray) -> np.ndarray:
    """Index of the entry of ``table`` (ascending, index parity = code parity)
    nearest to each ``u`` >= 0, ties to the even index; beyond the last entry
    the last index (saturation)."""
    mids = (table[:-1] + table[1:]) / 2.0  # exact: the table is dyadic
    u64 = np.asarray(u, dtype=np.float64)
    j = np.searchsorted(mids, u64, side="left")  # number of midpoints < u
    jc = np.minimum(j, len(mids) - 1)
    tie = (j < len(mids)) & (u64 == mids[jc])
    # at a tie u sits between entries j and j+1: take the even one
    j = np.where(tie & (j % 2 == 1), j + 1, j)
    return j.astype(np.uint8)


_E4M3_FINITE = e4m3_decode(np.arange(127, dtype=np.uint8))  # codes 0..126, ascending


def e4m3_encode(u) -> np.ndarray:
    """E4M3 "fn" code of each non-negative fp32 value: round to nearest, ties
    to even, saturate at 448."""
    u = np.asarray(u, dtype=np.float32)
    if np.any(u < 0) or np.any(np.isnan(u)):
        raise ValueError("scales are encoded from non-negative finite values")
    return _nearest_even(_E4M3_FINITE, u)


def e2m1_encode(v) -> np.ndarray:
    """E2M1 code of each fp32 value: magnitude rounded to nearest with ties to
    the even code, saturating at 6; the sign bit is set only for a negative
    value whose magnitude code is not zero."""
    v = np.asarray(v, dtype=np.float32)
    mag = _nearest_even(E2M1_MAGNITUDES, np.abs(v))
    neg = (v < 0) & (mag != 0)
    return (mag | np.where(neg, 0x8, 0)).astype(np.uint8)


def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """Pack 4-bit codes [..., K] into bytes [..., K/2]; element 2j -> low nibble."""
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)


def unpack_nibbles(packed: np.ndarray) -> np.ndarray:
    """Inverse of :func:`pack_nibbles`."""
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = packed & 0xF
    out[..., 1::2] = packed >> 4
    return out


def _quantize_blocks(w: np.ndarray, g: np.ndarray):
    """Block steps shared by weights and activations.

    ``w`` fp32 [R, K], ``g`` fp32 [R] (the row global; 1.0 for activations).
    Returns codes uint8 [R, K] (unpacked) and scales uint8 [R, K/16]."""
    R, K = w.shape
    blocks = w.reshape(R, K // BLOCK, BLOCK)
    bamax = np.max(np.abs(blocks), axis=2)                       # fp32, exact
    t = (bamax / np.float32(E2M1_MAX)).astype(np.float32)         # fp32(bamax / 6)
    gz = (g == 0)
    g_safe = np.where(gz, np.float32(1.0), g).astype(np.float32)
    u = (t / g_safe[:, None]).astype(np.float32)                  # fp32(t / g)
    s = e4m3_encode(u)
    s = np.where(gz[:, None], np.uint8(0), s).astype(np.uint8)
    denom = (e4m3_decode(s).astype(np.float32) * g[:, None]).astype(np.float32)  # fp32(dec(s) * g)
    live = denom != 0
    denom_safe = np.where(live, denom, np.float32(1.0)).astype(np.float32)
    v = (blocks / denom_safe[:, :, None]).astype(np.float32)      # fp32(w / denom)
    q = e2m1_encode(v)
    q = np.where(live[:, :, None], q, np.uint8(0)).astype(np.uint8)
    return q.reshape(R, K), s


def quantize_weight_rows(w) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Quantise fp32 weight rows [R, K] (K a multiple of 16) to NVFP4.

    Returns (codes uint8 [R, K/2], scales uint8 [R, K/16], globals fp32 [R])."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    R, K = w.shape
    if K % BLOCK:
        raise ValueError("row length must be a multiple of 16")
    ramax = np.max(np.abs(w), axis=1).astype(np.float32)
    g = (ramax / WEIGHT_GLOBAL_DIVISOR).astype(np.float32)        # fp32(ramax / 2688)
    q, s = _quantize_blocks(w, g)
    return pack_nibbles(q), s, g


def quantize_activation_rows(a) -> tuple[np.ndarray, np.ndarray]:
    """Quantise fp32 activation rows [R, K] to NVFP4 with the global fixed at
    1.0.  Returns (codes uint8 [R, K/2], scales uint8 [R, K/16])."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    R, K = a.shape
    if K % BLOCK:
        raise ValueError("row length must be a multiple of 16")
    q, s = _quantize_blocks(a, np.ones(R, dtype=np.float32))
    return pack_nibbles(q), s


def dequantize_rows(codes, scales, globals_=None) -> np.ndarray:
    """fp64 values of NVFP4 rows: dec(code) * dec(scale) * global."""
    q = e2m1_decode(unpack_nibbles(codes))
    R, K = q.shape
    s = e4m3_decode(scales)
    val = q.reshape(R, K // BLOCK, BLOCK) * s[:, :, None]
    if globals_ is not None:
        val = val * np.asarray(globals_, dtype=np.float64)[:, None, None]
    return val.reshape(R, K)


def bf16_round(v) -> np.ndarray:
    """Round fp64 values to the nearest bfloat16 (8 significant bits), ties to
    even, returned as fp64.  Used once per output element and for the shared
    expert's intermediate."""
    v = np.asarray(v, dtype=np.float64)
    m, e = np.frexp(v)  # v = m * 2**e, 0.5 <= |m| < 1
    # bfloat16 keeps 8 significant bits in its normal range (exponent >= -125
    # in frexp terms); below that the spacing is fixed at 2**-133.
    bits = np.where(e >= -125, 8, 8 - (-125 - e))
    bits = np.maximum(bits, 0)
    scaled = np.ldexp(m, bits)
    r = np.rint(scaled)  # round half to even
    return np.ldexp(r, e - bits)
