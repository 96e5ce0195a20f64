"""The device slicer of the other bank formats (ftmoe_slice_format) against
the oracle's slices, byte for byte, at the decode and offload layers' sizes:
gate_up keeps the gate and up row ranges of the window, down its columns,
mxfp4 (stored transposed) along its columns and rows respectively; windows
off a format's block grid are refused."""

import numpy as np
import pytest
import torch

from nvfp4_mixture_experts_counting_gb300 import ftmoe, workloads as W
from oracle import formats as F

pytestmark = pytest.mark.gpu

DEV = "cuda"
ARRAYS = {"nvfp4": ("codes", "scales", "globals"), "fp8_block": ("q", "scale"), "q4_0": ("blocks",),
          "mxfp4": ("blocks_t", "scales_t")}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from nvfp4_mixture_experts_counting_gb300 import build
    build.build()


def _experts(fmt, E, N, K, seed):
    return [W.format_matrix(fmt, N, K, seed=seed + e) for e in range(E)]


def _stack_to_device(mats, fmt):
    return [torch.from_numpy(np.ascontiguousarray(np.stack([m[k] for m in mats]))).to(DEV) for k in ARRAYS[fmt]]


@pytest.mark.parametrize("fmt", ["nvfp4", "fp8_block", "q4_0", "mxfp4"])
@pytest.mark.parametrize("H,I,i0,I_loc", [(2560, 640, 0, 384), (2560, 640, 256, 384), (4096, 2048, 1024, 1024)])
def test_device_slices_equal_oracle_slices(fmt, H, I, i0, I_loc):
    b = F.BLOCK[fmt]
    if i0 % b or I_loc % b or I % b:
        pytest.skip("window off this format's grid (checked by the guard test)")
    E = 3
    for matrix, (N, K) in ((ftmoe.MAT_GATE_UP, (2 * I, H)), (ftmoe.MAT_DOWN, (H, I))):
        mats = _experts(fmt, E, N, K, seed=100 * matrix + i0)
        src = _stack_to_device(mats, fmt)
        cut = F.slice_gate_up if matrix == ftmoe.MAT_GATE_UP else F.slice_down
        want = [cut(fmt, m, I, i0, I_loc) for m in mats]
        # outputs start as a sentinel byte pattern, so a byte the slicer misses shows up
        dst = [torch.full((E,) + want[0][k].shape, 0xAB if src[j].dtype == torch.uint8 else -7e30,
                          dtype=src[j].dtype, device=DEV)
               for j, k in enumerate(ARRAYS[fmt])]
        ftmoe.ftmoe_slice_format(fmt, matrix, E, H, I, i0, I_loc, src, dst)
        torch.cuda.synchronize()
        for j, k in enumerate(ARRAYS[fmt]):
            got = dst[j].cpu().numpy()
            ref = np.stack([w[k] for w in want])
            assert got.shape == ref.shape, (k, got.shape, ref.shape)
            assert np.array_equal(got.view(np.uint8), np.ascontiguousarray(ref).view(np.uint8)), (fmt, matrix, k)
        # and the values: the sliced arrays decode to the window of the matrix
        for e in range(E):
            sl = {k: dst[j][e].cpu().numpy() for j, k in enumerate(ARRAYS[fmt])}
            full = F.dequant(fmt, mats[e])
            part = full[np.r_[i0:i0 + I_loc, I + i0:I + i0 + I_loc]] if matrix == ftmoe.MAT_GATE_UP \
                else full[:, i0:i0 + I_loc]
            assert np.array_equal(F.dequant(fmt, sl), part)


@pytest.mark.parametrize("fmt,I,i0,I_loc", [("fp8_block", 640, 64, 128), ("q4_0", 640, 16, 32),
                                            ("mxfp4", 640, 0, 48), ("nvfp4", 640, 8, 16)])
def test_device_slicer_refuses_off_grid_windows(fmt, I, i0, I_loc):
    x = torch.zeros(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(ftmoe.FtmoeError) as ei:
        ftmoe.ftmoe_slice_format(fmt, ftmoe.MAT_DOWN, 1, 2560, I, i0, I_loc, [x, x, x], [x, x, x])
    assert ei.value.name == "ALIGNMENT"
