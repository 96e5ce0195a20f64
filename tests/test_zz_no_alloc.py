"""The allocation-free routing entry point, ftmoe_route_static.

Callers that cannot allocate device memory when they route (a serving
runtime whose free memory is all pre-assigned to KV-cache and graph pools, a
plugin host that forbids allocations, code running during CUDA-graph
capture) call this entry point with buffers they already own; its scratch is
a fixed array inside the library.  The test calls it through the C ABI twice
in a row and checks each result against the routing outputs of
ftmoe_forward on the same inputs.  This file is collected last on purpose,
and it builds everything it needs itself, so it also passes alone in a
fresh process."""

import ctypes as C

import numpy as np
import pytest
import torch

from nvfp4_mixture_experts_counting_gb300 import ftmoe, workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def routed_layer():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from nvfp4_mixture_experts_counting_gb300 import build
    build.build()
    from gpu_helpers import GpuBank, make_layer
    wl = W.WORKLOADS["decode"]
    bank = GpuBank(wl)
    layer = make_layer(wl, max_tokens=64)
    layer.load_bank(0, bank.desc())
    return wl, bank, layer


def _forward_routing(layer, wl, x):
    from gpu_helpers import AuxBufs
    T = x.shape[0]
    aux = AuxBufs(T, wl.top_k, wl.E)
    out = torch.empty((T, wl.H), dtype=torch.bfloat16, device=DEV)
    layer.forward(0, x, out, aux=aux.c)
    torch.cuda.synchronize()
    return aux.numpy()


def _static_routing(bank, wl, x):
    T = x.shape[0]
    P = T * wl.top_k
    idx = torch.full((T, wl.top_k), -1, dtype=torch.int32, device=DEV)
    w = torch.zeros((T, wl.top_k), dtype=torch.float32, device=DEV)
    offs = torch.full((wl.E + 1,), -1, dtype=torch.int32, device=DEV)
    perm = torch.full((P,), -1, dtype=torch.int32, device=DEV)
    inv = torch.full((P,), -1, dtype=torch.int32, device=DEV)
    ftmoe.ftmoe_route_static(x, T, wl.H, bank.router_w, bank.router_bias, wl.E, wl.top_k,
                             wl.norm_topk_prob, idx, w, offs, perm, inv)
    return dict(topk_idx=idx, topk_w=w, offsets=offs, perm=perm, inv=inv)


def test_route_static_matches_forward_two_calls(routed_layer):
    wl, bank, layer = routed_layer
    xa = W.hidden(wl, 16, step=11, device=DEV)
    xb = W.hidden(wl, 5, step=12, device=DEV)
    # two calls in a row, the second overwriting the shared scratch
    got_a = _static_routing(bank, wl, xa)
    got_b = _static_routing(bank, wl, xb)
    torch.cuda.synchronize()
    for x, got in ((xa, got_a), (xb, got_b)):
        ref = _forward_routing(layer, wl, x)
        for k in ("topk_idx", "offsets", "perm", "inv"):
            assert np.array_equal(got[k].cpu().numpy(), ref[k]), k
        assert np.allclose(got["topk_w"].cpu().numpy(), ref["topk_w"], rtol=1e-5, atol=1e-6)


def _oracle_routing(x, rw, rb, top_k):
    from oracle import moe
    logits = moe.router_logits(x.float().cpu().numpy(), rw.cpu().numpy(), None if rb is None else rb.cpu().numpy())
    idx, w = moe.select_topk(logits, top_k)
    offs, perm, inv = moe.counting_sort(idx, rw.shape[0])
    return dict(topk_idx=idx, topk_w=w, offsets=offs, perm=perm, inv=inv)


@pytest.mark.parametrize("T,H,E,top_k,bias", [
    (16, 2560, 256, 8, False),    # the decode layer
    (16, 2560, 1024, 8, True),    # T * E at the scratch's limit, Zipf-biased router
    (32, 8192, 256, 8, True),     # T * H and H at the limit
    (1024, 256, 16, 4, True),     # T and T * E at the limit
])
def test_route_static_matches_oracle_at_the_limits(routed_layer, T, H, E, top_k, bias):
    """Against the oracle directly: indices, offsets, perm and inv bit-exact,
    weights within the tolerance of the fp32 softmax, at sizes up to the
    fixed scratch's limits, with and without a router bias; the status
    reader reports no failed check."""
    wl = W.Workload("route_static", H=H, I=64, E=E, top_k=top_k, I_s=64, tokens=(T,), router_bias=bias)
    x = W.hidden(wl, T, step=5, device=DEV)
    rw = W.router_weight(wl, device=DEV)
    rb = W.router_bias(wl, device=DEV)
    got = _static_routing_raw(x, rw, rb, wl)
    assert ftmoe.ftmoe_route_static_status() == 0
    ref = _oracle_routing(x, rw, rb, top_k)
    for k in ("topk_idx", "offsets", "perm", "inv"):
        assert np.array_equal(got[k].cpu().numpy(), ref[k]), k
    assert np.allclose(got["topk_w"].cpu().numpy(), ref["topk_w"], rtol=5e-4, atol=1e-6)


def _static_routing_raw(x, rw, rb, wl):
    T = x.shape[0]
    P = T * wl.top_k
    idx = torch.full((T, wl.top_k), -1, dtype=torch.int32, device=DEV)
    w = torch.zeros((T, wl.top_k), dtype=torch.float32, device=DEV)
    offs = torch.full((wl.E + 1,), -1, dtype=torch.int32, device=DEV)
    perm = torch.full((P,), -1, dtype=torch.int32, device=DEV)
    inv = torch.full((P,), -1, dtype=torch.int32, device=DEV)
    ftmoe.ftmoe_route_static(x, T, wl.H, rw, rb, wl.E, wl.top_k, wl.norm_topk_prob, idx, w, offs, perm, inv)
    torch.cuda.synchronize()
    return dict(topk_idx=idx, topk_w=w, offsets=offs, perm=perm, inv=inv)


def test_route_static_rejects_oversized(routed_layer):
    wl, bank, _ = routed_layer
    lib = ftmoe.lib()
    # T*E beyond the fixed scratch: refused before any device work
    rc = lib.ftmoe_route_static(None, 65, wl.H, None, None, wl.E, wl.top_k, 1,
                                None, None, None, None, None, None)
    assert rc == -11
    rc = lib.ftmoe_route_static(None, 4, 8192 + 16, None, None, 8, 2, 1, None, None, None, None, None, None)
    assert rc == -11
    assert lib.ftmoe_route_static(None, 0, wl.H, None, None, wl.E, wl.top_k, 1,
                                  None, None, None, None, None, None) == 0
