"""ctypes binding of libftmoe.so (argument marshalling only).

The functions carry the C names of ``include/ftmoe.h``.  Torch supplies device
memory and streams; every step of the layer runs in the library's CUDA
kernels.  If the library is missing or fails to load, every call raises:
there is no fallback path.

``Layer`` is a small convenience wrapper that owns one handle.
"""

from __future__ import annotations

import ctypes as C
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libftmoe.so")

ABI_VERSION = 3
OUT_BF16, OUT_FP32, OUT_ACCUMULATE, ACT_BF16 = 0, 1, 0x100, 0x200

STATUS = {
    0: "OK", -1: "INVALID_ARG", -2: "ALIGNMENT", -3: "NOT_LOADED", -4: "SLICE_OUT_OF_RANGE",
    -5: "OOM", -6: "CUDA", -7: "TIMEOUT", -8: "FAULT_INJECTED", -9: "DEVICE", -10: "DEVICE_CHECK",
    -11: "TOO_LARGE",
}


class FtmoeError(RuntimeError):
    def __init__(self, code: int, where: str, detail: str = ""):
        self.code = code
        self.name = STATUS.get(code, str(code))
        super().__init__(f"{where}: {self.name} ({code}) {detail}".rstrip())


class Config(C.Structure):
    _fields_ = [("abi_version", C.c_int32), ("H", C.c_int32), ("I", C.c_int32), ("E", C.c_int32),
                ("top_k", C.c_int32), ("I_shared", C.c_int32), ("num_layers", C.c_int32),
                ("max_tokens", C.c_int32), ("norm_topk_prob", C.c_int32),
                ("has_router_bias", C.c_int32), ("hbm_slot_bytes", C.c_int64)]


class BankDesc(C.Structure):
    _fields_ = [("router_w", C.c_void_p), ("router_bias", C.c_void_p), ("gu_codes", C.c_void_p),
                ("gu_scales", C.c_void_p), ("gu_global", C.c_void_p), ("dn_codes", C.c_void_p),
                ("dn_scales", C.c_void_p), ("dn_global", C.c_void_p), ("sh_gate_up", C.c_void_p),
                ("sh_down", C.c_void_p), ("sh_gate", C.c_void_p), ("on_device", C.c_int32)]


class Aux(C.Structure):
    _fields_ = [("topk_idx", C.c_void_p), ("topk_w", C.c_void_p), ("offsets", C.c_void_p),
                ("perm", C.c_void_p), ("inv", C.c_void_p), ("logits", C.c_void_p),
                ("h_codes", C.c_void_p), ("h_scales", C.c_void_p)]


class Stats(C.Structure):
    _fields_ = [("touched_experts", C.c_int32), ("resident_slots", C.c_int32),
                ("touched_bytes", C.c_int64), ("hits", C.c_int64), ("misses", C.c_int64),
                ("h2d_bytes", C.c_int64), ("residency", C.c_double), ("device_status", C.c_int32),
                ("reranked_tokens", C.c_int64), ("touched_total", C.c_int64)]


class KernelTime(C.Structure):
    _fields_ = [("name", C.c_char * 48), ("launches", C.c_int64), ("total_ms", C.c_double)]


_lib = None

#: every symbol the header declares, with its argument and result types
SIGNATURES = {
    "ftmoe_create": ([C.POINTER(Config), C.c_int, C.POINTER(C.c_void_p)], C.c_int),
    "ftmoe_load_bank": ([C.c_void_p, C.c_int, C.POINTER(BankDesc), C.c_int, C.c_int, C.c_void_p], C.c_int),
    "ftmoe_forward": ([C.c_void_p, C.c_int, C.c_void_p, C.c_int, C.c_void_p, C.c_int, C.c_int, C.c_int,
                       C.POINTER(Aux), C.c_void_p], C.c_int),
    "ftmoe_forward_stack": ([C.c_void_p, C.c_void_p, C.c_int, C.c_void_p, C.c_void_p], C.c_int),
    "ftmoe_rms_renorm": ([C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_void_p], C.c_int),
    "ftmoe_destroy": ([C.c_void_p], C.c_int),
    "ftmoe_error_string": ([C.c_int], C.c_char_p),
    "ftmoe_last_cuda_error": ([], C.c_char_p),
    "ftmoe_get_stats": ([C.c_void_p, C.c_int, C.POINTER(Stats)], C.c_int),
    "ftmoe_check_status": ([C.c_void_p, C.c_void_p], C.c_int),
    "ftmoe_profile_enable": ([C.c_void_p, C.c_int], C.c_int),
    "ftmoe_profile_read": ([C.c_void_p, C.POINTER(KernelTime), C.c_int, C.POINTER(C.c_int)], C.c_int),
    "ftmoe_route_static": ([C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int,
                            C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p], C.c_int),
    "ftmoe_route_static_status": ([C.c_void_p], C.c_int),
    "ftmoe_forward_experts": ([C.c_void_p, C.c_int, C.c_void_p, C.c_int, C.c_void_p, C.c_int, C.c_void_p,
                               C.c_int, C.c_int, C.POINTER(Aux), C.c_void_p], C.c_int),
    "ftmoe_reduce_partials": ([C.c_void_p, C.c_int, C.c_int64, C.c_void_p, C.c_int, C.c_void_p], C.c_int),
    "ftmoe_test_withhold_stage": ([C.c_void_p, C.c_int, C.c_int64], C.c_int),
    "ftmoe_slice_format": ([C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int,
                            C.POINTER(C.c_void_p), C.POINTER(C.c_void_p), C.c_void_p], C.c_int),
    "ftmoe_quantize_weights": ([C.c_void_p, C.c_int64, C.c_int, C.c_void_p, C.c_void_p, C.c_void_p,
                                C.c_void_p], C.c_int),
    "ftmoe_quantize_activations": ([C.c_void_p, C.c_int64, C.c_int, C.c_void_p, C.c_void_p, C.c_void_p],
                                   C.c_int),
}


def lib():
    """The loaded libftmoe.so (raises if it is missing: no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libftmoe.so is not built ({LIB_PATH}); run build.build() first")
        L = C.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def _check(rc: int, where: str):
    if rc != 0:
        detail = ""
        if rc == -6:
            detail = lib().ftmoe_last_cuda_error().decode()
        raise FtmoeError(rc, where, detail)


def _ptr(t) -> Optional[int]:
    """Raw address of a torch tensor or numpy array (None stays None)."""
    if t is None:
        return None
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    return t.ctypes.data


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream
    return int(stream)


# ----------------------------------------------------------------- C-named calls

def ftmoe_create(config: Config, device: int = 0) -> int:
    h = C.c_void_p()
    _check(lib().ftmoe_create(C.byref(config), device, C.byref(h)), "ftmoe_create")
    return h.value


def ftmoe_load_bank(h: int, layer: int, desc: BankDesc, i0: int, I_loc: int, stream=None):
    _check(lib().ftmoe_load_bank(h, layer, C.byref(desc), i0, I_loc, _stream(stream)), "ftmoe_load_bank")


def ftmoe_forward(h: int, layer: int, x, T: int, out, out_flags: int, i0: int, I_loc: int,
                  aux: Optional[Aux] = None, stream=None):
    _check(lib().ftmoe_forward(h, layer, _ptr(x), T, _ptr(out), out_flags, i0, I_loc,
                               C.byref(aux) if aux is not None else None, _stream(stream)),
           "ftmoe_forward")


def ftmoe_forward_stack(h: int, x, T: int, out, stream=None):
    _check(lib().ftmoe_forward_stack(h, _ptr(x), T, _ptr(out), _stream(stream)), "ftmoe_forward_stack")


def ftmoe_rms_renorm(y, x, T: int, H: int, stream=None):
    _check(lib().ftmoe_rms_renorm(_ptr(y), _ptr(x), T, H, _stream(stream)), "ftmoe_rms_renorm")


def ftmoe_destroy(h: int):
    _check(lib().ftmoe_destroy(h), "ftmoe_destroy")


def ftmoe_error_string(code: int) -> str:
    return lib().ftmoe_error_string(code).decode()


def ftmoe_last_cuda_error() -> str:
    return lib().ftmoe_last_cuda_error().decode()


def ftmoe_get_stats(h: int, layer: int) -> Stats:
    s = Stats()
    _check(lib().ftmoe_get_stats(h, layer, C.byref(s)), "ftmoe_get_stats")
    return s


def ftmoe_check_status(h: int, stream=None) -> int:
    return lib().ftmoe_check_status(h, _stream(stream))


def ftmoe_profile_enable(h: int, enable: bool):
    _check(lib().ftmoe_profile_enable(h, int(enable)), "ftmoe_profile_enable")


def ftmoe_profile_read(h: int, max_entries: int = 64) -> dict:
    """{kernel name: (launches, total ms)} recorded since the last read."""
    arr = (KernelTime * max_entries)()
    n = C.c_int()
    _check(lib().ftmoe_profile_read(h, arr, max_entries, C.byref(n)), "ftmoe_profile_read")
    return {arr[i].name.decode(): (arr[i].launches, arr[i].total_ms) for i in range(n.value)}


def ftmoe_route_static(x, T: int, H: int, router_w, router_bias, E: int, top_k: int, norm_topk_prob: bool,
                       topk_idx, topk_w, offsets, perm, inv, stream=None):
    """Routing with no device allocation (scratch in a fixed device array)."""
    _check(lib().ftmoe_route_static(_ptr(x), T, H, _ptr(router_w), _ptr(router_bias), E, top_k,
                                    int(norm_topk_prob), _ptr(topk_idx), _ptr(topk_w), _ptr(offsets),
                                    _ptr(perm), _ptr(inv), _stream(stream)), "ftmoe_route_static")


def ftmoe_forward_experts(h: int, layer: int, x, T: int, out, out_flags: int, expert_mask,
                          shared_i0: int = 0, shared_I_loc: int = 0, aux: Optional[Aux] = None, stream=None):
    """One expert-parallel rank's share: the routed slots of the experts whose
    mask byte (host numpy uint8 [E]) is set, plus the shared expert's window
    [shared_i0, shared_i0 + shared_I_loc) (none when shared_I_loc is 0)."""
    import numpy as np
    m = np.ascontiguousarray(expert_mask, dtype=np.uint8)
    _check(lib().ftmoe_forward_experts(h, layer, _ptr(x), T, _ptr(out), out_flags, m.ctypes.data, shared_i0,
                                       shared_I_loc, C.byref(aux) if aux is not None else None, _stream(stream)),
           "ftmoe_forward_experts")


def ftmoe_reduce_partials(parts, n_parts: int, n: int, out, out_flags: int = OUT_BF16, stream=None):
    """out <- sum over ranks of fp32 partials [n_parts][n], in rank order."""
    _check(lib().ftmoe_reduce_partials(_ptr(parts), n_parts, n, _ptr(out), out_flags, _stream(stream)),
           "ftmoe_reduce_partials")


def ftmoe_route_static_status(stream=None) -> int:
    """Status of the latest ftmoe_route_static call (0, DEVICE_CHECK or TIMEOUT)."""
    return lib().ftmoe_route_static_status(_stream(stream))


def ftmoe_test_withhold_stage(h: int, enable: bool, wait_limit_ns: int = 0):
    _check(lib().ftmoe_test_withhold_stage(h, int(enable), wait_limit_ns), "ftmoe_test_withhold_stage")


FMT = {"nvfp4": 0, "fp8_block": 1, "q4_0": 2, "mxfp4": 3}
MAT_GATE_UP, MAT_DOWN = 0, 1


def ftmoe_slice_format(fmt: str, matrix: int, E: int, H: int, I: int, i0: int, I_loc: int, src, dst, stream=None):
    """Slice E experts' matrix in bank format `fmt` to a window; src / dst
    are lists of device tensors (the format's arrays, in the header's order)."""
    S = (C.c_void_p * 3)(*[_ptr(t) for t in src] + [None] * (3 - len(src)))
    D = (C.c_void_p * 3)(*[_ptr(t) for t in dst] + [None] * (3 - len(dst)))
    _check(lib().ftmoe_slice_format(FMT[fmt], matrix, E, H, I, i0, I_loc, S, D, _stream(stream)),
           "ftmoe_slice_format")


def ftmoe_quantize_weights(w, rows: int, K: int, codes, scales, globals_, stream=None):
    _check(lib().ftmoe_quantize_weights(_ptr(w), rows, K, _ptr(codes), _ptr(scales), _ptr(globals_),
                                        _stream(stream)), "ftmoe_quantize_weights")


def ftmoe_quantize_activations(a, rows: int, K: int, codes, scales, stream=None):
    _check(lib().ftmoe_quantize_activations(_ptr(a), rows, K, _ptr(codes), _ptr(scales), _stream(stream)),
           "ftmoe_quantize_activations")


# ----------------------------------------------------------------- convenience

def make_config(H, I, E, top_k, I_shared, num_layers=1, max_tokens=16, norm_topk_prob=True,
                has_router_bias=False, hbm_slot_bytes=0) -> Config:
    return Config(ABI_VERSION, H, I, E, top_k, I_shared, num_layers, max_tokens, int(norm_topk_prob),
                  int(has_router_bias), hbm_slot_bytes)


def bank_desc(router_w, router_bias, gu_codes, gu_scales, gu_global, dn_codes, dn_scales, dn_global,
              sh_gate_up, sh_down, sh_gate, on_device: bool) -> BankDesc:
    return BankDesc(_ptr(router_w), _ptr(router_bias), _ptr(gu_codes), _ptr(gu_scales), _ptr(gu_global),
                    _ptr(dn_codes), _ptr(dn_scales), _ptr(dn_global), _ptr(sh_gate_up), _ptr(sh_down),
                    _ptr(sh_gate), int(on_device))


class Layer:
    """Owns one ftmoe handle (all layers of one shape)."""

    def __init__(self, config: Config, device: int = 0):
        self.config = config
        self.handle = ftmoe_create(config, device)

    def close(self):
        if self.handle:
            ftmoe_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def load_bank(self, layer: int, desc: BankDesc, i0: int = 0, I_loc: Optional[int] = None, stream=None):
        I_loc = self.config.I - i0 if I_loc is None else I_loc
        ftmoe_load_bank(self.handle, layer, desc, i0, I_loc, stream)

    def forward(self, layer: int, x, out, out_flags: int = OUT_BF16, i0: int = 0,
                I_loc: Optional[int] = None, aux: Optional[Aux] = None, stream=None):
        I_loc = self.config.I - i0 if I_loc is None else I_loc
        ftmoe_forward(self.handle, layer, x, x.shape[0], out, out_flags, i0, I_loc, aux, stream)
        return out

    def forward_stack(self, x, out, stream=None):
        ftmoe_forward_stack(self.handle, x, x.shape[0], out, stream)
        return out

    def stats(self, layer: int) -> Stats:
        return ftmoe_get_stats(self.handle, layer)

    def check_status(self, stream=None) -> int:
        return ftmoe_check_status(self.handle, stream)
