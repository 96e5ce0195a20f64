"""Pins of the oracle's other bank formats and their window slices against
things other than the oracle itself: torch's float8_e4m3fn and float16 casts
(library routines), blocks built by hand from the formats' definitions, an
element-by-element loop, and the identity dequantise(slice) == slice of the
dequantised matrix, which a dropped row range, a wrong scale row or a
transposed slice would break."""

import numpy as np
import pytest
import torch

from nvfp4_mixture_experts_counting_gb300 import workloads as W
from oracle import formats as F

FORMATS = ("nvfp4", "fp8_block", "q4_0", "mxfp4")


def test_fp8_block_matches_torch_cast_tile_by_tile():
    m = W.format_matrix("fp8_block", 200, 300, seed=1)
    got = F.fp8_block_dequant(m["q"], m["scale"])
    vals = torch.from_numpy(m["q"]).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for n in (0, 127, 128, 199):
        for k in (0, 127, 128, 255, 256, 299):
            assert got[n, k] == vals[n, k] * np.float64(m["scale"][n // 128, k // 128])


def test_q4_0_hand_built_block():
    # d = 0.5 (fp16 0x3800); byte j holds code j (low) and 15 - j (high):
    # element j = 0.5 * (j - 8), element j + 16 = 0.5 * (7 - j)
    blk = np.zeros((1, 1, 18), dtype=np.uint8)
    blk[0, 0, 0:2] = np.frombuffer(np.float16(0.5).tobytes(), dtype=np.uint8)
    assert blk[0, 0, 0] == 0x00 and blk[0, 0, 1] == 0x38
    for j in range(16):
        blk[0, 0, 2 + j] = j | ((15 - j) << 4)
    got = F.q4_0_dequant(blk)[0]
    want = [0.5 * (j - 8) for j in range(16)] + [0.5 * (7 - j) for j in range(16)]
    assert np.array_equal(got, np.array(want))


def test_q4_0_scale_is_ieee_half():
    m = W.format_matrix("q4_0", 3, 64, seed=2)
    d = torch.from_numpy(m["blocks"][:, :, 0:2].copy()).view(torch.float16).to(torch.float64).numpy()[..., 0]
    got = F.q4_0_dequant(m["blocks"])
    for n in range(3):
        for b in range(2):
            code = m["blocks"][n, b, 2] & 0xF
            assert got[n, 32 * b] == d[n, b] * (int(code) - 8)


def test_ue8m0_closed_form():
    got = F.ue8m0_decode(np.array([0, 126, 127, 128, 254, 255], dtype=np.uint8))
    assert np.array_equal(got[:5], [2.0 ** -127, 0.5, 1.0, 2.0, 2.0 ** 127])
    assert np.isnan(got[5])


def test_mxfp4_transposed_layout_by_loop():
    m = W.format_matrix("mxfp4", 5, 64, seed=3)
    got = F.mxfp4_dequant(m["blocks_t"], m["scales_t"])
    e2m1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for n in range(5):
        for k in range(64):
            byte = int(m["blocks_t"][k // 2, n])
            c = (byte >> 4) if k % 2 else (byte & 0xF)
            v = (-1.0 if c & 8 else 1.0) * e2m1[c & 7] * 2.0 ** (int(m["scales_t"][k // 32, n]) - 127)
            assert got[n, k] == v, (n, k)


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("H,I,i0,I_loc", [(256, 256, 0, 128), (256, 256, 128, 128), (384, 512, 128, 256)])
def test_slice_identity(fmt, H, I, i0, I_loc):
    """gate_up keeps two row ranges, down a column range, in every format."""
    gu = W.format_matrix(fmt, 2 * I, H, seed=10 + i0)
    dn = W.format_matrix(fmt, H, I, seed=20 + i0)
    full_gu, full_dn = F.dequant(fmt, gu), F.dequant(fmt, dn)
    rows = np.r_[i0:i0 + I_loc, I + i0:I + i0 + I_loc]
    assert np.array_equal(F.dequant(fmt, F.slice_gate_up(fmt, gu, I, i0, I_loc)), full_gu[rows])
    assert np.array_equal(F.dequant(fmt, F.slice_down(fmt, dn, I, i0, I_loc)), full_dn[:, i0:i0 + I_loc])


@pytest.mark.parametrize("fmt,I,i0,I_loc", [
    ("fp8_block", 256, 64, 128), ("fp8_block", 256, 0, 64), ("fp8_block", 320, 0, 160),
    ("q4_0", 256, 16, 32), ("q4_0", 256, 0, 48), ("mxfp4", 256, 16, 64), ("mxfp4", 256, 0, 80),
    ("nvfp4", 64, 8, 16), ("nvfp4", 64, 48, 32),
])
def test_slice_guards(fmt, I, i0, I_loc):
    """Windows off the format's block grid (or outside I) are refused."""
    with pytest.raises(ValueError):
        F.check_format_window(fmt, I, i0, I_loc)


def test_block_sizes_match_the_pages():
    # "I/tp must stay a multiple of each format's block size -- 128 for
    # fp8_block, 32 for the fp4 scale blocks, 32 for q4_0"
    assert F.BLOCK["fp8_block"] == 128 and F.BLOCK["q4_0"] == 32 and F.BLOCK["mxfp4"] == 32
