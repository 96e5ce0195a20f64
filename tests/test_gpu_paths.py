"""The CUDA-core kernels and the device-side failure path, on the GPU.

* With FTMOE_NO_TC=1 set before a handle is created, the handle runs the
  CUDA-core kernels (decode GEMVs for T <= 32, the any-T kernels above)
  instead of the tensor-core ones; at the decode and mid shapes they must
  match the oracle to the same bar, and the per-kernel record shows which
  kernels ran.
* A bounded wait made to run out (one CTA of the tensor-core down kernel
  withholds a pipeline stage) must end in FTMOE_ERR_TIMEOUT from
  ftmoe_check_status, with no GPU fault, and the next forward of the same
  handle must be right again.
* The RMS renorm kernel on the rows worked out by hand for the oracle."""

import numpy as np
import pytest
import torch

from nvfp4_mixture_experts_counting_gb300 import ftmoe, workloads as W

from gpu_helpers import AuxBufs, GpuBank, check_output, check_routing, make_layer

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from nvfp4_mixture_experts_counting_gb300 import build
    build.build()


def _kernels_run(layer, fn):
    ftmoe.ftmoe_profile_enable(layer.handle, True)
    ftmoe.ftmoe_profile_read(layer.handle)
    fn()
    torch.cuda.synchronize()
    names = set(ftmoe.ftmoe_profile_read(layer.handle))
    ftmoe.ftmoe_profile_enable(layer.handle, False)
    return names


@pytest.mark.parametrize("name,Ts", [("mid", (1, 16, 32, 40, 100)), ("decode", (1, 16, 40))])
def test_cuda_core_kernels_match_oracle(monkeypatch, name, Ts):
    wl = W.WORKLOADS[name]
    bank = GpuBank(wl)
    monkeypatch.setenv("FTMOE_NO_TC", "1")
    layer = make_layer(wl, max_tokens=128)   # the variable is read when the handle is created
    monkeypatch.delenv("FTMOE_NO_TC")
    layer.load_bank(0, bank.desc())
    for T in Ts:
        x = W.hidden(wl, T, step=40, device=DEV)
        aux = AuxBufs(T, wl.top_k, wl.E)
        out = torch.empty((T, wl.H), dtype=torch.bfloat16, device=DEV)
        names = _kernels_run(layer, lambda: layer.forward(0, x, out, aux=aux.c))
        assert not any(n.startswith(("k_dtc", "k_pf")) for n in names), names
        want = "k_dec_gate_up" if T <= 32 else "k_gate_up"
        assert want in names, names
        assert layer.check_status() == 0
        ref = bank.oracle_layer(x)
        check_routing(aux, ref)
        check_output(out, ref.out)
    layer.close()


def test_expired_wait_reports_timeout_and_the_handle_recovers():
    wl = W.WORKLOADS["decode"]
    bank = GpuBank(wl)
    layer = make_layer(wl, max_tokens=32)
    layer.load_bank(0, bank.desc())
    T = 16
    x = W.hidden(wl, T, step=77, device=DEV)
    good = torch.empty((T, wl.H), dtype=torch.float32, device=DEV)
    layer.forward(0, x, good, out_flags=ftmoe.OUT_FP32)
    torch.cuda.synchronize()
    assert layer.check_status() == 0
    # one CTA of the down kernel withholds its first stage: its waits give up
    # after 2 ms, it marks the status word and leaves its tile unwritten
    ftmoe.ftmoe_test_withhold_stage(layer.handle, True, 2_000_000)
    bad = torch.zeros_like(good)
    layer.forward(0, x, bad, out_flags=ftmoe.OUT_FP32)
    rc = layer.check_status()
    ftmoe.ftmoe_test_withhold_stage(layer.handle, False)
    assert rc == -7, ftmoe.STATUS.get(rc, rc)  # FTMOE_ERR_TIMEOUT
    assert layer.stats(0).device_status & 2
    # the tiles of the other CTAs were written as usual
    assert torch.equal(bad[:, 128:].view(torch.int32), good[:, 128:].view(torch.int32))
    # the same handle, next forwards: the same bits as before, no status
    for _ in range(2):
        again = torch.empty_like(good)
        layer.forward(0, x, again, out_flags=ftmoe.OUT_FP32)
        torch.cuda.synchronize()
        assert layer.check_status() == 0
        assert torch.equal(again.view(torch.int32), good.view(torch.int32))
    ref = bank.oracle_layer(x, out_dtype="fp32")
    check_output(again, ref.out64)
    layer.close()


def test_rms_renorm_kernel_hand_worked_rows():
    """The rows of the oracle's hand-worked pin: mean square equal to eps,
    (3, -4, 0, 0), eps dominating, and zeros."""
    y = torch.tensor([[1e-3] * 4, [3.0, -4.0, 0.0, 0.0], [1e-4, 0.0, 0.0, 0.0], [0.0] * 4],
                     dtype=torch.float32, device=DEV)
    x = torch.empty((4, 4), dtype=torch.bfloat16, device=DEV)
    ftmoe.ftmoe_rms_renorm(y, x, 4, 4)
    torch.cuda.synchronize()
    want = np.array([[362 / 512] * 4, [154 / 128, -205 / 128, 0.0, 0.0], [205 / 2048, 0.0, 0.0, 0.0],
                     [0.0] * 4])
    assert np.array_equal(x.double().cpu().numpy(), want)
