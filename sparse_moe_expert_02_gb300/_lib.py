"""ctypes binding of libmoe (include/moe.h): argument marshalling only.

Every function here has the name of the C entry point it calls and turns
torch tensors into device pointers and the current torch stream into the
cudaStream_t the library expects.  All arithmetic happens in the library's
CUDA kernels; if the library cannot be loaded the import fails loudly --
there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

_lock = threading.Lock()
_lib = None

# moe_status
MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE = 0, 1, 2, 3
MOE_ERR_CUDA, MOE_ERR_DEVICE_TIMEOUT, MOE_ERR_BOUNDS, MOE_ERR_NONFINITE = 4, 5, 6, 7
# moe_dtype
MOE_F32, MOE_BF16, MOE_FP8_E4M3_B128 = 0, 1, 2
MOE_FLAG_FORCE_SIMT = 0x1
MOE_FLAG_PAIR_CTA_OFF = 0x2
MOE_FLAG_PAIR_CTA_ON = 0x4
MOE_FLAG_DOWN_HILO = 0x8
MOE_FLAG_MCAST_ON = 0x10
MOE_FLAG_MCAST_OFF = 0x20
MOE_FLAG_NARROW_TAILS_ON = 0x40
MOE_FLAG_NARROW_TAILS_OFF = 0x80
MOE_FLAG_TOPK_HIST_OFF = 0x100
MOE_FLAG_FUSED_COMBINE = 0x200
MOE_FLAG_SPLIT_GEMM_OFF = 0x400

DTYPE_CODE = {"f32": MOE_F32, "bf16": MOE_BF16, "fp8": MOE_FP8_E4M3_B128}

# Every symbol include/moe.h declares (tests check the library exports them).
SYMBOLS = (
    "moe_plan_create", "moe_plan_destroy", "moe_plan_config", "moe_workspace_layout", "moe_workspace_size",
    "moe_workspace_init", "moe_quantize_weights", "moe_forward", "moe_route", "moe_topk", "moe_permute",
    "moe_gemm_gateup", "moe_gemm_down", "moe_unpermute", "moe_check", "moe_selftest_wait_timeout",
    "moe_status_str", "moe_last_error_detail", "moe_build_info", "moe_launch_count",
    "moe_permute_index_noalloc", "moe_pack_routing_words", "moe_convert_down_weights", "moe_pointer_kind",
)


class moe_config(ctypes.Structure):
    _fields_ = [("T_max", ctypes.c_int32), ("D", ctypes.c_int32), ("E", ctypes.c_int32), ("I", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("dtype", ctypes.c_int32), ("out_dtype", ctypes.c_int32),
                ("has_router_bias", ctypes.c_int32), ("flags", ctypes.c_uint32), ("spin_limit_ns", ctypes.c_int64)]


class moe_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("w_router", "b_router", "w_gate", "w_up", "w_down", "s_gate", "s_up", "s_down", "w_down_f16")]


class moe_ws_layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("total", "err", "logits", "blob", "counts", "offsets", "tiles", "inv", "src_tok", "hist", "xq",
                 "xq_scale", "xp", "xp_scale", "h", "h_scale", "y", "logits_part", "tiles2", "pairs")]


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        L = lib()
        msg = L.moe_status_str(status).decode()
        detail = L.moe_last_error_detail().decode()
        super().__init__(f"{where}: {msg} ({detail})")


def lib_path() -> str:
    return _build.LIB


def lib():
    """Load libmoe (building it first if the sources changed)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            L = ctypes.CDLL(path)
            P, I32, I64, S = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
            st = ctypes.c_int
            sig = {
                "moe_plan_create": (st, [ctypes.POINTER(moe_config), ctypes.c_int, ctypes.POINTER(P)]),
                "moe_plan_destroy": (None, [P]),
                "moe_plan_config": (ctypes.POINTER(moe_config), [P]),
                "moe_workspace_layout": (st, [P, I32, ctypes.POINTER(moe_ws_layout)]),
                "moe_workspace_size": (st, [P, I32, ctypes.POINTER(S)]),
                "moe_workspace_init": (st, [P, P, S, P]),
                "moe_quantize_weights": (st, [P, P, I64, I32, I32, P, P, P]),
                "moe_forward": (st, [P, ctypes.POINTER(moe_weights), P, I32, P, P, P, P, S, P]),
                "moe_route": (st, [P, ctypes.POINTER(moe_weights), P, I32, P, S, P]),
                "moe_topk": (st, [P, I32, P, S, P]),
                "moe_permute": (st, [P, P, I32, P, S, P]),
                "moe_gemm_gateup": (st, [P, ctypes.POINTER(moe_weights), P, I32, P, S, P]),
                "moe_gemm_down": (st, [P, ctypes.POINTER(moe_weights), I32, P, S, P]),
                "moe_unpermute": (st, [P, I32, P, P, S, P]),
                "moe_check": (st, [P, P, P]),
                "moe_selftest_wait_timeout": (st, [P, P, S, I64, P]),
                "moe_status_str": (ctypes.c_char_p, [st]),
                "moe_last_error_detail": (ctypes.c_char_p, []),
                "moe_build_info": (ctypes.c_char_p, []),
                "moe_launch_count": (ctypes.c_uint64, []),
                "moe_permute_index_noalloc": (st, [P, I32, I32, I32, P, P, P, P, P, P]),
                "moe_pack_routing_words": (st, [P, I32, P, S, P, P]),
                "moe_convert_down_weights": (st, [P, P, P, P, S, P]),
                "moe_pointer_kind": (st, [P, ctypes.POINTER(ctypes.c_int32)]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _ptr(t, host_mapped_ok: bool = False):
    """Address of a contiguous device tensor; with host_mapped_ok also of a
    page-locked host tensor that the device addresses at the same place
    (moe_pointer_kind == host_mapped), which kernels then read or write
    directly."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("libmoe takes contiguous tensors")
    if not t.is_cuda:
        if not (host_mapped_ok and t.is_pinned() and moe_pointer_kind(t) == "host_mapped"):
            raise ValueError("libmoe takes device tensors (or, for out, mapped page-locked host tensors)")
    return t.data_ptr()


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _ok(status: int, where: str):
    if status != MOE_OK:
        raise MoEError(status, where)


# ------------------------------------------------------------ entry points

def moe_plan_create(T_max: int, D: int, E: int, I: int, top_k: int, dtype: str, out_dtype: str = "f32",
                    has_router_bias: bool = False, flags: int = 0, spin_limit_ns: int = 0, device: int = 0):
    cfg = moe_config(T_max, D, E, I, top_k, DTYPE_CODE[dtype], DTYPE_CODE[out_dtype], int(has_router_bias), flags,
                     spin_limit_ns)
    plan = ctypes.c_void_p()
    _ok(lib().moe_plan_create(ctypes.byref(cfg), device, ctypes.byref(plan)), "moe_plan_create")
    return plan


def moe_plan_destroy(plan):
    lib().moe_plan_destroy(plan)


def moe_workspace_layout(plan, T: int) -> moe_ws_layout:
    L = moe_ws_layout()
    _ok(lib().moe_workspace_layout(plan, T, ctypes.byref(L)), "moe_workspace_layout")
    return L


def moe_workspace_size(plan, T: int) -> int:
    n = ctypes.c_size_t()
    _ok(lib().moe_workspace_size(plan, T, ctypes.byref(n)), "moe_workspace_size")
    return n.value


def moe_workspace_init(plan, ws, stream=None):
    _ok(lib().moe_workspace_init(plan, _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
        "moe_workspace_init")


def moe_quantize_weights(plan, w, q, s, stream=None):
    G, R, C = w.shape
    _ok(lib().moe_quantize_weights(plan, _ptr(w), G, R, C, _ptr(q), _ptr(s), _stream(stream)),
        "moe_quantize_weights")


POINTER_KINDS = {0: "host", 1: "host_mapped", 2: "device", 3: "managed"}


def moe_pointer_kind(t) -> str:
    k = ctypes.c_int32(0)
    p = t if isinstance(t, int) else t.data_ptr()
    _ok(lib().moe_pointer_kind(p, ctypes.byref(k)), "moe_pointer_kind")
    return POINTER_KINDS.get(k.value, "host")


def moe_convert_down_weights(plan, w_down, w_down_f16, ws, stream=None):
    _ok(lib().moe_convert_down_weights(plan, _ptr(w_down), _ptr(w_down_f16), _ptr(ws), _wsb(ws), _stream(stream)),
        "moe_convert_down_weights")


def make_weights(w: dict) -> moe_weights:
    return moe_weights(*[_ptr(w.get(n)) for n in
                         ("w_router", "b_router", "w_gate", "w_up", "w_down", "s_gate", "s_up", "s_down", "w_down_f16")])


def _wsb(ws):
    return ws.numel() * ws.element_size()


def moe_forward(plan, weights: moe_weights, x, T, out, blob_out, logits_out, ws, stream=None):
    _ok(lib().moe_forward(plan, ctypes.byref(weights), _ptr(x), T, _ptr(out, host_mapped_ok=True), _ptr(blob_out),
                          _ptr(logits_out),
                          _ptr(ws), _wsb(ws), _stream(stream)), "moe_forward")


def moe_route(plan, weights, x, T, ws, stream=None):
    _ok(lib().moe_route(plan, ctypes.byref(weights), _ptr(x), T, _ptr(ws), _wsb(ws), _stream(stream)), "moe_route")


def moe_topk(plan, T, ws, stream=None):
    _ok(lib().moe_topk(plan, T, _ptr(ws), _wsb(ws), _stream(stream)), "moe_topk")


def moe_permute(plan, x, T, ws, stream=None):
    _ok(lib().moe_permute(plan, _ptr(x), T, _ptr(ws), _wsb(ws), _stream(stream)), "moe_permute")


def moe_gemm_gateup(plan, weights, x, T, ws, stream=None):
    _ok(lib().moe_gemm_gateup(plan, ctypes.byref(weights), _ptr(x), T, _ptr(ws), _wsb(ws), _stream(stream)),
        "moe_gemm_gateup")


def moe_gemm_down(plan, weights, T, ws, stream=None):
    _ok(lib().moe_gemm_down(plan, ctypes.byref(weights), T, _ptr(ws), _wsb(ws), _stream(stream)), "moe_gemm_down")


def moe_unpermute(plan, T, out, ws, stream=None):
    _ok(lib().moe_unpermute(plan, T, _ptr(out), _ptr(ws), _wsb(ws), _stream(stream)), "moe_unpermute")


def moe_check(plan, ws, stream=None):
    _ok(lib().moe_check(plan, _ptr(ws), _stream(stream)), "moe_check")


def moe_check_status(plan, ws, stream=None) -> int:
    return lib().moe_check(plan, _ptr(ws), _stream(stream))


def moe_selftest_wait_timeout(plan, ws, limit_ns: int, stream=None):
    _ok(lib().moe_selftest_wait_timeout(plan, _ptr(ws), _wsb(ws), limit_ns, _stream(stream)),
        "moe_selftest_wait_timeout")


def moe_permute_index_noalloc(idx, T, E, top_k, counts, offsets, tiles, inv, src_tok, stream=None) -> int:
    """Allocation-free permutation index build; returns the moe_status."""
    return lib().moe_permute_index_noalloc(_ptr(idx), T, E, top_k, _ptr(counts), _ptr(offsets), _ptr(tiles),
                                           _ptr(inv), _ptr(src_tok), _stream(stream))


def moe_pack_routing_words(plan, T, ws, words, stream=None):
    _ok(lib().moe_pack_routing_words(plan, T, _ptr(ws), _wsb(ws), _ptr(words), _stream(stream)),
        "moe_pack_routing_words")


def moe_launch_count() -> int:
    return lib().moe_launch_count()


def moe_build_info() -> str:
    return lib().moe_build_info().decode()
