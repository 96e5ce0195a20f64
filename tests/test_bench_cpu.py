"""Host-side arithmetic of bench.py's dominant-kernel roofline (no GPU):
algorithmic bytes or flops per launch over the mean launch time, with a
step's work spread over the kernel's launches in a step."""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from nvfp4_mixture_experts_counting_gb300 import accounting as A  # noqa: E402

H, I, IS, E = 2560, 640, 640, 256
HBM = (6786.0, "measured")
FP4 = (11580.0, "measured x 6")


def test_one_launch_per_step_hbm():
    # 500 steps, one gate_up launch each, 24.8 ms in all: 49.6 us per launch
    r = bench.kernel_roofline("k_dtc_gate_up", 500, 24.8, 500, A.kernel_unit_bytes("k_dtc_gate_up", H, I, IS, E),
                              A.kernel_unit_flops("k_dtc_gate_up", H, I, IS, E), 128, 16, 102.75, HBM, FP4)
    alg = 1_848_320 * 102.75 + 2 * IS * H * 2
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["algorithmic_bytes_per_launch"] == int(alg)
    assert r["avg_launch_us"] == pytest.approx(49.6)
    assert r["achieved"] == pytest.approx(alg / 49.6e-6 / 1e9, rel=1e-4)
    assert r["frac"] == pytest.approx(r["achieved"] / HBM[0], rel=1e-3)


def test_batched_launches_split_the_step():
    # an offloaded forward: two gate_up launches per step, each half the work
    one = bench.kernel_roofline("k_dtc_gate_up", 100, 5.0, 100, A.kernel_unit_bytes("k_dtc_gate_up", H, I, IS, E),
                                (None, None, None), 128, 16, 100.0, HBM, FP4)
    two = bench.kernel_roofline("k_dtc_gate_up", 200, 5.0, 100, A.kernel_unit_bytes("k_dtc_gate_up", H, I, IS, E),
                                (None, None, None), 128, 16, 100.0, HBM, FP4)
    assert two["units_per_launch"] == pytest.approx(one["units_per_launch"] / 2)
    assert two["algorithmic_bytes_per_launch"] == pytest.approx(one["algorithmic_bytes_per_launch"] / 2, abs=1)
    # half the bytes in half the time per launch: the same rate
    assert two["achieved"] == pytest.approx(one["achieved"], rel=1e-4)


def test_tensor_bound_flops_per_pair():
    pairs = 4096 * 8
    r = bench.kernel_roofline("k_pf_gate_up", 6, 6 * 0.157, 6, A.kernel_unit_bytes("k_pf_gate_up", H, I, IS, E),
                              A.kernel_unit_flops("k_pf_gate_up", H, I, IS, E), pairs, 4096, 171.0, HBM, FP4)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["algorithmic_flops_per_launch"] == 2 * H * 2 * I * pairs
    assert r["achieved"] == pytest.approx(2 * H * 2 * I * pairs / 157e-6 / 1e12, rel=1e-3)
    assert r["peak"] == pytest.approx(FP4[0])


def test_kernel_without_accounting_has_no_roofline():
    assert bench.kernel_roofline("k_sort", 10, 1.0, 10, A.kernel_unit_bytes("k_sort", H, I, IS, E),
                                 A.kernel_unit_flops("k_sort", H, I, IS, E), 128, 16, 100.0, HBM, FP4) is None


# ---- the algorithmic byte and flop counts, against hand-worked figures of
# the bank format (E2M1 codes at 1/2 byte, one E4M3 scale per 16 elements,
# one fp32 global per row; the down globals cover all H rows in any window)

@pytest.mark.parametrize("H,I,full", [(256, 64, 29_184), (2560, 640, 2_780_160), (4096, 2048, 14_188_544)])
def test_expert_bytes_full_bank(H, I, full):
    assert A.expert_window_bytes(H, I) == full


def test_expert_bytes_half_window_keeps_every_down_global():
    # gate_up: 2 * 320 rows * (1280 + 160 + 4); down: 2560 rows * (160 + 20 + 4)
    assert A.gate_up_window_bytes(2560, 320) == 924_160
    assert A.down_window_bytes(2560, 320) == 471_040
    assert A.expert_window_bytes(2560, 320) == 1_395_200


def test_shared_expert_and_routed_flops():
    # bf16 gate/up rows and down columns (9,830,400 B) plus the bf16 gate vector
    assert A.shared_window_bytes(2560, 640) == 9_830_400 + 2560 * 2
    # 2 flops per multiply-add: gate_up 2*H*2I and down 2*I*H per pair, 8 pairs a token
    assert A.routed_flops(2560, 640, 8) == 78_643_200


def test_prefill_kernel_flops_per_unit():
    # per pair: gate_up 2*2560*1280, down 2*640*2560; per token: the shared
    # expert's gate_up 2*2560*1280 and down 2*640*2560, the router x times
    # three bf16 parts of 256 rows of 2560
    f = lambda k: A.kernel_unit_flops(k, 2560, 640, 640, 256)[:2]
    assert f("k_pf_gate_up") == (6_553_600, "pair")
    assert f("k_pf_down") == (3_276_800, "pair")
    assert f("k_pf_shared_gate_up") == (6_553_600, "token")
    assert f("k_pf_shared_down") == (3_276_800, "token")
    assert f("k_pf_router") == (3_932_160, "token")


@pytest.mark.parametrize("T,touched,mb", [(1, 8, 34.7), (16, 102, 296.2)])
def test_decode_layer_bytes(T, touched, mb):
    # touched experts + shared expert + fp32 router + x in and bf16 out
    assert A.layer_touched_bytes(2560, 256, 640, 640, T, touched) / 1e6 == pytest.approx(mb, abs=0.05)
