"""Pins of the oracle's NVFP4 encoder/decoder against things other than
itself: closed forms, torch's float8_e4m3fn and bfloat16 casts (library
routines), brute-force nearest-value search, and exact round trips."""

import numpy as np
import pytest
import torch

from oracle import nvfp4


def test_e2m1_decode_closed_form():
    # E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; exponent 0 is subnormal
    for c in range(16):
        s, e, m = c >> 3, (c >> 1) & 3, c & 1
        val = (m * 0.5) if e == 0 else (2.0 ** (e - 1)) * (1 + m / 2)
        val = -val if s else val
        got = nvfp4.e2m1_decode(np.array([c], dtype=np.uint8))[0]
        assert got == val, (c, got, val)


def test_e4m3_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = nvfp4.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def _sweep_e4m3():
    vals = nvfp4.e4m3_decode(np.arange(127, dtype=np.uint8))
    mids = (vals[:-1] + vals[1:]) / 2
    pts = np.concatenate([vals, mids]).astype(np.float32)
    up = np.nextafter(pts, np.float32(np.inf))
    dn = np.nextafter(pts, np.float32(0))
    rng = np.random.default_rng(1)
    rnd = (rng.random(20000) * 448).astype(np.float32)
    tiny = (rng.random(2000) * 0.02).astype(np.float32)
    allv = np.concatenate([pts, up, dn, rnd, tiny, np.float32([0.0])])
    return allv[allv <= 448.0]


def test_e4m3_encode_matches_torch_in_range():
    u = _sweep_e4m3()
    ours = nvfp4.e4m3_encode(u)
    ref = torch.from_numpy(u).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, (u[bad[:5]], ours[bad[:5]], ref[bad[:5]])


def test_e4m3_encode_saturates():
    u = np.float32([448.0, 448.5, 463.9, 464.0, 480.0, 1e6, 3.0e38])
    assert np.all(nvfp4.e4m3_encode(u) == 0x7E)
    with pytest.raises(ValueError):
        nvfp4.e4m3_encode(np.float32([-1.0]))


def _brute_e2m1(v: float) -> int:
    """Nearest E2M1 magnitude by exhaustive search, ties to the even code."""
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    a = abs(float(v))
    d = [abs(a - m) for m in mags]
    best = min(d)
    cands = [i for i in range(8) if d[i] == best]
    code = cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0]
    if v < 0 and code != 0:
        code |= 8
    return code


def test_e2m1_encode_brute_force():
    rng = np.random.default_rng(2)
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    mids = (mags[:-1] + mags[1:]) / 2
    base = np.concatenate([mags, mids, [6.5, 7.0, 100.0]]).astype(np.float32)
    pts = np.concatenate([base, np.nextafter(base, np.float32(np.inf)),
                          np.nextafter(base, np.float32(0)),
                          (rng.random(3000) * 8).astype(np.float32)])
    pts = np.concatenate([pts, -pts])
    ours = nvfp4.e2m1_encode(pts)
    for v, c in zip(pts, ours):
        assert c == _brute_e2m1(v), (v, c)


def test_e2m1_ties_listed():
    # ties go to the even code
    cases = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0, 9.0: 6.0}
    for v, want in cases.items():
        c = nvfp4.e2m1_encode(np.float32([v]))[0]
        assert nvfp4.e2m1_decode([c])[0] == want
        cn = nvfp4.e2m1_encode(np.float32([-v]))[0]
        assert nvfp4.e2m1_decode([cn])[0] == -want
    # a zero magnitude carries sign bit 0
    assert nvfp4.e2m1_encode(np.float32([-0.2]))[0] == 0
    assert nvfp4.e2m1_encode(np.float32([-0.0]))[0] == 0


def test_pack_nibble_order():
    codes = np.array([[1, 2, 3, 4]], dtype=np.uint8)
    packed = nvfp4.pack_nibbles(codes)
    assert packed.tolist() == [[0x21, 0x43]]
    assert np.array_equal(nvfp4.unpack_nibbles(packed), codes)


def _exact_rows(rng, R, K, g_pow):
    """Rows that NVFP4 represents exactly: every 16-block holds a +-6 code and
    a power-of-two or any E4M3 scale; one block per row has scale 448, so the
    row global is exactly 2**g_pow."""
    nb = K // 16
    codes = rng.integers(0, 16, size=(R, K)).astype(np.uint8)
    codes[codes == 8] = 0                      # no negative zero
    pos = rng.integers(0, 16, size=(R, nb))
    for r in range(R):
        for b in range(nb):
            codes[r, b * 16 + pos[r, b]] = 7 | (8 if rng.random() < 0.5 else 0)
    scales = rng.integers(0x20, 0x7E, size=(R, nb)).astype(np.uint8)  # normal E4M3
    scales[:, 0] = 0x7E                        # 448 in the first block of every row
    g = np.float32(2.0 ** g_pow)
    w = nvfp4.e2m1_decode(codes).reshape(R, nb, 16) * nvfp4.e4m3_decode(scales)[:, :, None] * float(g)
    return codes, scales, g, w.reshape(R, K).astype(np.float32)


def test_weight_quantiser_round_trip_exact():
    rng = np.random.default_rng(3)
    codes, scales, g, w = _exact_rows(rng, 24, 256, -14)
    qc, qs, qg = nvfp4.quantize_weight_rows(w)
    assert np.all(qg == g)
    assert np.array_equal(qs, scales)
    assert np.array_equal(nvfp4.unpack_nibbles(qc), codes)
    assert np.array_equal(nvfp4.dequantize_rows(qc, qs, qg), w.astype(np.float64))


def test_activation_quantiser_round_trip_exact():
    rng = np.random.default_rng(4)
    codes, scales, _, w = _exact_rows(rng, 8, 128, 0)
    # with the global fixed at 1 the scales are the block maxima / 6 exactly
    qc, qs = nvfp4.quantize_activation_rows(w)
    assert np.array_equal(qs, scales)
    assert np.array_equal(nvfp4.unpack_nibbles(qc), codes)


def test_quantiser_error_bound_and_zero_rows():
    rng = np.random.default_rng(5)
    w = (rng.standard_normal((64, 512)) * 0.02).astype(np.float32)
    w[3] = 0.0                                  # a zero row
    w[5, 32:48] = 0.0                           # a zero block
    c, s, g = nvfp4.quantize_weight_rows(w)
    assert g[3] == 0 and np.all(s[3] == 0) and np.all(c[3] == 0)
    assert np.all(s[5, 2] == 0) and np.all(c[5, 16:24] == 0)
    deq = nvfp4.dequantize_rows(c, s, g)
    assert np.all(np.isfinite(deq))
    # |w - w_hat| <= half an E2M1 step (at most 1.0 for |v| in (4, 6]) times
    # the block's dequantised scale, plus the saturation gap for the block max
    blk_scale = (nvfp4.e4m3_decode(s) * g[:, None].astype(np.float64))
    v = np.abs(w.astype(np.float64)).reshape(64, 32, 16)
    step = np.where(v <= 2 * blk_scale[:, :, None], 0.25, np.where(v <= 4 * blk_scale[:, :, None], 0.5, 1.0))
    err = np.abs(deq - w).reshape(64, 32, 16)
    # the block max maps to at most 6 * scale; scale rounding is relative 2**-4
    bound = step * blk_scale[:, :, None] + v * 2.0 ** -3
    assert np.all(err <= bound + 1e-12)
    rel = np.linalg.norm(deq - w) / np.linalg.norm(w)
    assert rel < 0.12


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(6)
    v = np.concatenate([rng.standard_normal(50000) * 10 ** rng.uniform(-6, 6, 50000),
                        [0.0, -0.0, 1.0, 1.00390625, 1.01171875]]).astype(np.float32)
    ours = nvfp4.bf16_round(v.astype(np.float64))
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ours, ref)
