"""One rank's share of an expert-parallel layer (ftmoe_forward_experts): the
routed slots of the experts it owns (e % G == r), no shared expert.  Each
share matches the oracle's, and the shares of a partition of the experts add
up to the routed part of the whole layer, at decode and prefill sizes."""

import numpy as np
import pytest
import torch

from nvfp4_mixture_experts_counting_gb300 import ftmoe, workloads as W

from gpu_helpers import GpuBank, check_output, make_layer, rel_l2

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


@pytest.mark.parametrize("name,T,G", [("decode", 16, 2), ("decode", 1, 4), ("prefill", 1024, 2)])
def test_expert_shares_match_oracle_and_add_up(name, T, G):
    wl = W.WORKLOADS[name]
    bank = GpuBank(wl)
    layer = make_layer(wl, max_tokens=max(T, 64))
    layer.load_bank(0, bank.desc())
    x = W.hidden(wl, T, step=41, device=DEV)
    rows = np.arange(T) if T <= 64 else np.unique(np.r_[0:T:16, T - 1])
    if T > 64:
        bank.prefetch_oracle_experts(range(wl.E))
    total = torch.zeros((T, wl.H), dtype=torch.float32, device=DEV)
    with_shared = torch.zeros_like(total)
    for r in range(G):
        mask = (np.arange(wl.E) % G == r)
        share = torch.empty((T, wl.H), dtype=torch.float32, device=DEV)
        ftmoe.ftmoe_forward_experts(layer.handle, 0, x, T, share, ftmoe.OUT_FP32, mask.astype(np.uint8))
        bf = torch.empty((T, wl.H), dtype=torch.bfloat16, device=DEV)
        ftmoe.ftmoe_forward_experts(layer.handle, 0, x, T, bf, ftmoe.OUT_BF16, mask.astype(np.uint8))
        # the same share with window r of the shared expert (a whole rank's
        # work), where the window fits the tensor-core tiles (64-wide)
        si0, sI = r * wl.I_s // G, wl.I_s // G
        rank = torch.zeros((T, wl.H), dtype=torch.float32, device=DEV)
        if sI % 64 == 0:
            ftmoe.ftmoe_forward_experts(layer.handle, 0, x, T, rank, ftmoe.OUT_FP32, mask.astype(np.uint8), si0, sI)
        torch.cuda.synchronize()
        assert layer.check_status() == 0
        ref = _oracle(bank, x, expert_mask=mask, include_shared=False, out_dtype="fp32", tokens=rows)
        check_output(share, ref.out64, rows=rows)
        refb = _oracle(bank, x, expert_mask=mask, include_shared=False, tokens=rows)
        check_output(bf, refb.out, rows=rows)
        total += share
        with_shared += rank
    routed = _oracle(bank, x, include_shared=False, out_dtype="fp32", tokens=rows)
    check_output(total, routed.out64, rows=rows)
    if (wl.I_s // G) % 64:
        layer.close()
        return
    # the ranks' shares, shared windows included, add up to the whole layer
    full = torch.empty((T, wl.H), dtype=torch.float32, device=DEV)
    layer.forward(0, x, full, out_flags=ftmoe.OUT_FP32)
    torch.cuda.synchronize()
    assert rel_l2(with_shared.cpu().numpy()[rows], full.cpu().numpy()[rows]) <= 1e-5
    check_output(with_shared, _oracle(bank, x, out_dtype="fp32", tokens=rows).out64, rows=rows)
    layer.close()
