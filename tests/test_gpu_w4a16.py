"""The W4A16 numerics mode (FTMOE_ACT_BF16) on the GPU against the oracle's
bf16-activation mode: routing bit-exact, outputs to the same bar as the
W4A4 layer, windows adding up to the full layer; and the distance between
the two numerics modes, which is the accuracy cost of quantising the
activations, measured on both sides."""

import numpy as np
import pytest
import torch

from nvfp4_mixture_experts_counting_gb300 import ftmoe, workloads as W

from gpu_helpers import AuxBufs, GpuBank, check_output, check_routing, make_layer, rel_l2

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from nvfp4_mixture_experts_counting_gb300 import build
    build.build()


def _oracle(bank, x, **kw):
    from oracle import moe
    wl = bank.wl
    return moe.moe_layer(
        x.float().cpu().numpy(), bank.router_w.cpu().numpy(),
        None if bank.router_bias is None else bank.router_bias.cpu().numpy(),
        bank.oracle_expert, bank.sh_gate_up.float().cpu().numpy(), bank.sh_down.float().cpu().numpy(),
        bank.sh_gate.float().cpu().numpy(), I=wl.I, I_s=wl.I_s, top_k=wl.top_k,
        norm_topk_prob=wl.norm_topk_prob, **kw)


@pytest.fixture(scope="module")
def decode():
    wl = W.WORKLOADS["decode"]
    bank = GpuBank(wl)
    layer = make_layer(wl, max_tokens=64)
    layer.load_bank(0, bank.desc())
    return wl, bank, layer


@pytest.mark.parametrize("T", [1, 8, 16, 32])
def test_w4a16_decode_matches_oracle(decode, T):
    wl, bank, layer = decode
    x = W.hidden(wl, T, step=21, device=DEV)
    aux = AuxBufs(T, wl.top_k, wl.E)
    out = torch.empty((T, wl.H), dtype=torch.bfloat16, device=DEV)
    layer.forward(0, x, out, out_flags=ftmoe.OUT_BF16 | ftmoe.ACT_BF16, aux=aux.c)
    torch.cuda.synchronize()
    assert layer.check_status() == 0
    ref = _oracle(bank, x, activations="bf16")
    check_routing(aux, ref)
    check_output(out, ref.out)


def test_w4a16_halves_add_up(decode):
    wl, bank, layer = decode
    T = 16
    x = W.hidden(wl, T, step=22, device=DEV)
    full = torch.empty((T, wl.H), dtype=torch.float32, device=DEV)
    layer.forward(0, x, full, out_flags=ftmoe.OUT_FP32 | ftmoe.ACT_BF16)
    acc = torch.zeros_like(full)
    for i0 in (0, 320):
        layer.forward(0, x, acc, out_flags=ftmoe.OUT_FP32 | ftmoe.OUT_ACCUMULATE | ftmoe.ACT_BF16, i0=i0, I_loc=320)
    torch.cuda.synchronize()
    assert rel_l2(acc.cpu().numpy(), full.cpu().numpy()) <= 1e-6
    check_output(full, _oracle(bank, x, activations="bf16", out_dtype="fp32").out64)


def test_w4a16_mid_any_T():
    wl = W.WORKLOADS["mid"]
    bank = GpuBank(wl)
    layer = make_layer(wl, max_tokens=128)
    layer.load_bank(0, bank.desc())
    for T in (5, 40, 128):
        x = W.hidden(wl, T, step=23, device=DEV)
        aux = AuxBufs(T, wl.top_k, wl.E)
        out = torch.empty((T, wl.H), dtype=torch.bfloat16, device=DEV)
        layer.forward(0, x, out, out_flags=ftmoe.ACT_BF16, aux=aux.c)
        torch.cuda.synchronize()
        ref = _oracle(bank, x, activations="bf16")
        check_routing(aux, ref)
        check_output(out, ref.out)
    layer.close()


def test_cost_of_quantised_activations(decode, capsys):
    """rel-L2 between the W4A4 and the W4A16 layer on the same tokens: the
    GPU's figure equals the oracle's (both modes match their oracle), and it
    is far above the parity tolerance, so the two modes are told apart."""
    wl, bank, layer = decode
    T = 16
    x = W.hidden(wl, T, step=24, device=DEV)
    a4 = torch.empty((T, wl.H), dtype=torch.float32, device=DEV)
    a16 = torch.empty_like(a4)
    layer.forward(0, x, a4, out_flags=ftmoe.OUT_FP32)
    layer.forward(0, x, a16, out_flags=ftmoe.OUT_FP32 | ftmoe.ACT_BF16)
    torch.cuda.synchronize()
    gpu_cost = rel_l2(a4.cpu().numpy(), a16.cpu().numpy())
    o4 = _oracle(bank, x, out_dtype="fp32").out64
    o16 = _oracle(bank, x, out_dtype="fp32", activations="bf16").out64
    oracle_cost = rel_l2(o4, o16)
    with capsys.disabled():
        print(f"\nW4A4 vs W4A16 rel-L2 (decode layer, T={T}): GPU {gpu_cost:.4e}, oracle {oracle_cost:.4e}")
    assert abs(gpu_cost - oracle_cost) <= 0.05 * oracle_cost
    assert oracle_cost > 10 * 5e-3
