"""GPU parity of the CUDA path against the CPU oracle, through the C ABI.

Bar: routing indices, offsets, perm and inv bit-exact; NVFP4 codes, scales
and globals byte-exact; bf16 outputs within max-abs 2e-2 and rel-L2 5e-3;
windows that cover I once add up to the full layer."""

import numpy as np
import pytest
import torch

from nvfp4_mixture_experts_counting_gb300 import ftmoe, workloads as W
from oracle import moe, nvfp4

from gpu_helpers import (AuxBufs, GpuBank, check_output, check_routing, make_layer, rel_l2)

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from nvfp4_mixture_experts_counting_gb300 import build
    build.build()


# ------------------------------------------------------------------ quantisers

@pytest.mark.parametrize("rows,K,std", [(37, 256, 0.02), (64, 2560, 0.02), (5, 640, 3.0), (3, 16, 1e-3)])
def test_weight_quantiser_bytes_match_oracle(rows, K, std):
    g = torch.Generator(device=DEV).manual_seed(rows * K)
    w = torch.randn((rows, K), generator=g, device=DEV) * std
    w[0] = 0.0                      # zero row
    if rows > 2:
        w[2, :16] = 0.0             # zero block
        w[1, 5] = 1e4 * std         # an outlier that saturates scales of small blocks
    codes = torch.empty((rows, K // 2), dtype=torch.uint8, device=DEV)
    scales = torch.empty((rows, K // 16), dtype=torch.uint8, device=DEV)
    glob = torch.empty((rows,), dtype=torch.float32, device=DEV)
    ftmoe.ftmoe_quantize_weights(w, rows, K, codes, scales, glob)
    torch.cuda.synchronize()
    oc, os_, og = nvfp4.quantize_weight_rows(w.cpu().numpy())
    assert np.array_equal(glob.cpu().numpy(), og)
    assert np.array_equal(scales.cpu().numpy(), os_)
    assert np.array_equal(codes.cpu().numpy(), oc)


def test_activation_quantiser_bytes_match_oracle():
    g = torch.Generator(device=DEV).manual_seed(7)
    a = (torch.randn((33, 2560), generator=g, device=DEV) * 2).to(torch.bfloat16)
    a[3] = 0
    a[4, :16] = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, -0.25, -0.75,
                             -1.25, -1.75, -2.5, -3.5, -5.0, -6.0], dtype=torch.bfloat16)
    codes = torch.empty((33, 1280), dtype=torch.uint8, device=DEV)
    scales = torch.empty((33, 160), dtype=torch.uint8, device=DEV)
    ftmoe.ftmoe_quantize_activations(a, 33, 2560, codes, scales)
    torch.cuda.synchronize()
    oc, os_ = nvfp4.quantize_activation_rows(a.float().cpu().numpy())
    assert np.array_equal(scales.cpu().numpy(), os_)
    assert np.array_equal(codes.cpu().numpy(), oc)


# ------------------------------------------------------------------ tiny layer

@pytest.fixture(scope="module")
def tiny():
    wl = W.WORKLOADS["tiny"]
    bank = GpuBank(wl)
    layer = make_layer(wl, max_tokens=64)
    layer.load_bank(0, bank.desc())
    return wl, bank, layer


@pytest.mark.parametrize("T", [4, 1, 3, 32, 33, 37, 64])
def test_tiny_layer_matches_oracle(tiny, T):
    wl, bank, layer = tiny
    x = W.hidden(wl, T, device=DEV)
    aux = AuxBufs(T, wl.top_k, wl.E)
    out = torch.empty((T, wl.H), dtype=torch.bfloat16, device=DEV)
    layer.forward(0, x, out, aux=aux.c)
    torch.cuda.synchronize()
    ref = bank.oracle_layer(x)
    check_routing(aux, ref)
    check_output(out, ref.out)


def test_tiny_bank_bytes_match_oracle(tiny):
    wl, bank, _ = tiny
    for e in range(wl.E):
        ob = bank.oracle_expert(e)
        assert np.array_equal(bank.gu_codes[e].cpu().numpy(), ob.gu_codes)
        assert np.array_equal(bank.gu_scales[e].cpu().numpy(), ob.gu_scales)
        assert np.array_equal(bank.gu_global[e].cpu().numpy(), ob.gu_global)
        assert np.array_equal(bank.dn_codes[e].cpu().numpy(), ob.dn_codes)
        assert np.array_equal(bank.dn_scales[e].cpu().numpy(), ob.dn_scales)
        assert np.array_equal(bank.dn_global[e].cpu().numpy(), ob.dn_global)


def _compositions(n):
    if n == 0:
        yield []
        return
    for first in range(1, n + 1):
        for rest in _compositions(n - first):
            yield [first] + rest


def test_tiny_every_partition_adds_up(tiny):
    """Windows of every 16-aligned partition of I, accumulated in order into
    one fp32 buffer, equal the full fp32 output (and the oracle)."""
    wl, bank, layer = tiny
    T = 4
    x = W.hidden(wl, T, device=DEV)
    full = torch.empty((T, wl.H), dtype=torch.float32, device=DEV)
    layer.forward(0, x, full, out_flags=ftmoe.OUT_FP32)
    ref = bank.oracle_layer(x, out_dtype="fp32")
    for comp in _compositions(wl.I // 16):
        acc = torch.zeros((T, wl.H), dtype=torch.float32, device=DEV)
        i0 = 0
        for nb in comp:
            layer.forward(0, x, acc, out_flags=ftmoe.OUT_FP32 | ftmoe.OUT_ACCUMULATE, i0=i0, I_loc=nb * 16)
            i0 += nb * 16
        torch.cuda.synchronize()
        assert rel_l2(acc.cpu().numpy(), full.cpu().numpy()) <= 1e-6
        check_output(acc, ref.out64)


def test_tiny_sliced_load_matches_window(tiny):
    """A bank loaded with only a window computes the same partial as the full
    bank run on that window."""
    wl, bank, layer = tiny
    x = W.hidden(wl, 4, device=DEV)
    part_full = torch.empty((4, wl.H), dtype=torch.float32, device=DEV)
    layer.forward(0, x, part_full, out_flags=ftmoe.OUT_FP32, i0=16, I_loc=32)
    sl = make_layer(wl, max_tokens=8)
    sl.load_bank(0, bank.desc(), i0=16, I_loc=32)
    part_sl = torch.empty_like(part_full)
    sl.forward(0, x, part_sl, out_flags=ftmoe.OUT_FP32, i0=16, I_loc=32)
    torch.cuda.synchronize()
    assert torch.equal(part_full, part_sl)
    ref = bank.oracle_layer(x, i0=16, I_loc=32, out_dtype="fp32")
    check_output(part_sl, ref.out64)
    with pytest.raises(ftmoe.FtmoeError) as ei:
        sl.forward(0, x, part_sl, out_flags=ftmoe.OUT_FP32, i0=0, I_loc=32)
    assert ei.value.name == "SLICE_OUT_OF_RANGE"


def test_tiny_edge_cases(tiny):
    wl, bank, layer = tiny
    x = W.hidden(wl, 4, device=DEV)
    out = torch.empty((4, wl.H), dtype=torch.bfloat16, device=DEV)
    layer.forward(0, x[:0], out[:0])                      # T = 0
    for kw, name in [(dict(i0=8, I_loc=16), "ALIGNMENT"), (dict(i0=0, I_loc=24), "ALIGNMENT"),
                     (dict(i0=48, I_loc=32), "SLICE_OUT_OF_RANGE"),
                     (dict(out_flags=ftmoe.OUT_BF16 | ftmoe.OUT_ACCUMULATE), "INVALID_ARG")]:
        with pytest.raises(ftmoe.FtmoeError) as ei:
            layer.forward(0, x, out, **kw)
        assert ei.value.name == name
    with pytest.raises(ftmoe.FtmoeError) as ei:
        big = W.hidden(wl, 65, device=DEV)
        layer.forward(0, big, torch.empty((65, wl.H), dtype=torch.bfloat16, device=DEV))
    assert ei.value.name == "INVALID_ARG"
    with pytest.raises(ftmoe.FtmoeError) as ei:
        layer.forward(0, x, x)
    assert ei.value.name == "INVALID_ARG"
    assert layer.check_status() == 0


def test_tiny_zero_input(tiny):
    wl, bank, layer = tiny
    x = torch.zeros((4, wl.H), dtype=torch.bfloat16, device=DEV)
    out = torch.full((4, wl.H), 7.0, dtype=torch.bfloat16, device=DEV)
    aux = AuxBufs(4, wl.top_k, wl.E)
    layer.forward(0, x, out, aux=aux.c)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0
    # all logits tie at 0: experts 0 and 1 in that order for every token
    assert np.array_equal(aux.topk_idx.cpu().numpy(), np.tile([0, 1], (4, 1)))


def test_tied_router_rows_choose_lower_index():
    wl = W.WORKLOADS["tiny"]
    bank = GpuBank(wl)
    bank.router_w[5] = bank.router_w[2]
    bank.router_w[6] = bank.router_w[1]
    layer = make_layer(wl, max_tokens=64)
    layer.load_bank(0, bank.desc())
    T = 64
    x = W.hidden(wl, T, step=3, device=DEV)
    aux = AuxBufs(T, wl.top_k, wl.E)
    out = torch.empty((T, wl.H), dtype=torch.bfloat16, device=DEV)
    layer.forward(0, x, out, aux=aux.c)
    torch.cuda.synchronize()
    ref = bank.oracle_layer(x)
    check_routing(aux, ref)
    check_output(out, ref.out)


def test_deterministic_repeat(tiny):
    wl, bank, layer = tiny
    x = W.hidden(wl, 37, device=DEV)
    outs = []
    for _ in range(5):
        o = torch.empty((37, wl.H), dtype=torch.float32, device=DEV)
        layer.forward(0, x, o, out_flags=ftmoe.OUT_FP32)
        outs.append(o)
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int32), outs[0].view(torch.int32))


# ------------------------------------------------------------------ decode layer

@pytest.fixture(scope="module")
def decode():
    wl = W.WORKLOADS["decode"]
    bank = GpuBank(wl)
    layer = make_layer(wl, max_tokens=64)
    layer.load_bank(0, bank.desc())
    return wl, bank, layer


@pytest.mark.parametrize("T", [1, 8, 16, 24, 32, 40])
def test_decode_layer_matches_oracle(decode, T):
    wl, bank, layer = decode
    x = W.hidden(wl, T, device=DEV)
    aux = AuxBufs(T, wl.top_k, wl.E)
    out = torch.empty((T, wl.H), dtype=torch.bfloat16, device=DEV)
    layer.forward(0, x, out, aux=aux.c)
    torch.cuda.synchronize()
    ref = bank.oracle_layer(x)
    check_routing(aux, ref)
    check_output(out, ref.out)


def test_decode_router_logit_error_within_bound(decode):
    """The decode router's logits (tensor cores over the exact three-way bf16
    split of the fp32 router, 256-product chunks added in fp32) stay within
    the bound its top-k certificate assumes, 2^-20 * ||x|| * ||w|| (plus the
    rigorous term of the chunk additions), by a margin of 16: the bound is
    empirical, and this test is its measurement."""
    wl, bank, layer = decode
    rw = bank.router_w.cpu().numpy().astype(np.float64)
    wn = np.linalg.norm(rw, axis=1)
    worst = 0.0
    for step in range(3):
        T = 32
        x = W.hidden(wl, T, step=300 + step, device=DEV)
        logits = torch.empty((T, wl.E), dtype=torch.float32, device=DEV)
        aux = AuxBufs(T, wl.top_k, wl.E)
        aux.c.logits = logits.data_ptr()
        out = torch.empty((T, wl.H), dtype=torch.bfloat16, device=DEV)
        layer.forward(0, x, out, aux=aux.c)
        torch.cuda.synchronize()
        x64 = x.float().cpu().numpy().astype(np.float64)
        exact = moe.router_logits(x64, rw, None)
        rel = np.abs(logits.cpu().numpy() - exact) / (np.linalg.norm(x64, axis=1)[:, None] * wn[None, :])
        worst = max(worst, float(rel.max()))
        idx, _ = moe.select_topk(exact, wl.top_k)
        assert np.array_equal(aux.topk_idx.cpu().numpy(), idx)
    assert worst <= 2.0 ** -20 / 16, f"largest relative logit error {worst:.3e}"


def test_decode_bank_bytes_sampled(decode):
    wl, bank, _ = decode
    for e in (0, 77, 255):
        ob = bank.oracle_expert(e)
        assert np.array_equal(bank.gu_codes[e].cpu().numpy(), ob.gu_codes)
        assert np.array_equal(bank.gu_scales[e].cpu().numpy(), ob.gu_scales)
        assert np.array_equal(bank.dn_codes[e].cpu().numpy(), ob.dn_codes)
        assert np.array_equal(bank.dn_global[e].cpu().numpy(), ob.dn_global)


@pytest.mark.parametrize("T", [1, 16])
def test_decode_two_halves_sum_to_full(decode, T):
    wl, bank, layer = decode
    x = W.hidden(wl, T, step=1, device=DEV)
    full = torch.empty((T, wl.H), dtype=torch.float32, device=DEV)
    layer.forward(0, x, full, out_flags=ftmoe.OUT_FP32)
    acc = torch.zeros_like(full)
    halves = []
    for i0 in (0, 320):
        part = torch.empty_like(full)
        layer.forward(0, x, part, out_flags=ftmoe.OUT_FP32, i0=i0, I_loc=320)
        layer.forward(0, x, acc, out_flags=ftmoe.OUT_FP32 | ftmoe.OUT_ACCUMULATE, i0=i0, I_loc=320)
        halves.append(part)
    torch.cuda.synchronize()
    assert rel_l2(acc.cpu().numpy(), full.cpu().numpy()) <= 1e-6
    ref = bank.oracle_layer(x, out_dtype="fp32")
    check_output(acc, ref.out64)
    for i0, part in zip((0, 320), halves):
        refp = bank.oracle_layer(x, i0=i0, I_loc=320, out_dtype="fp32")
        check_output(part, refp.out64)


def test_decode_stats(decode):
    wl, bank, layer = decode
    x = W.hidden(wl, 16, device=DEV)
    aux = AuxBufs(16, wl.top_k, wl.E)
    out = torch.empty((16, wl.H), dtype=torch.bfloat16, device=DEV)
    layer.forward(0, x, out, aux=aux.c)
    st = layer.stats(0)
    offs = aux.offsets.cpu().numpy()
    touched = int(np.count_nonzero(np.diff(offs)))
    assert st.touched_experts == touched
    assert st.touched_bytes == touched * moe.expert_slice_bytes(wl.H, wl.I)
