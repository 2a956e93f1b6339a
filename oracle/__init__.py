"""fp64 CPU oracle of the routed-MoE FFN layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
leg of ``bench.py`` may import this package.  The CUDA path of
``sparse_moe_expert_02_gb300`` never imports or calls it, and the two share no
code: the arithmetic lives in ``oracle.c`` (plain C, fp64, OpenMP over
tokens), which this module compiles with gcc and calls through ctypes.

Parity status per function (what pins each one, see ``oracle.c`` header):
  codecs (bf16, E4M3)      pinned: exhaustive tables, torch casts
  orc_topk                 pinned: brute-force stable sort, planted ties,
                           sum-to-one, top_k = E dense-softmax closed form
  orc_permute              pinned: counts/offsets/bijection invariants,
                           identity-expert round trip, brute-force sort
  orc_moe_tokens / layer   pinned by closed forms: E=1,k=1 vs a numpy
                           dense SwiGLU; top_k = E and (all other experts
                           biased to zero softmax mass) top_k < E vs the
                           dense softmax mixture in numpy/scipy; identity
                           experts, equivariances.  The pages print no
                           worked value of the layer.
  orc_quant_blocks         pinned: block-amax definition on planted blocks,
                           codes vs torch.float8_e4m3fn.
  quant_row_128            pinned: per-row, per-128-column amax/448 against
  (orc_quant_rows_128)     torch.float8_e4m3fn, group amaxes over four
                           decades, an all-zero group, exact E4M3 ties; and
                           in place in the FP8 layer (E = 1, k = 1 against a
                           numpy pipeline over the same torch quantiser).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

MODE = {"f32": 0, "bf16": 1, "fp8": 2}
DT_F32, DT_BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile oracle.c into _build/liboracle.so (gcc, -O2, OpenMP)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fvisibility=hidden", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
            L.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
            L.orc_bf16_to_f64.restype = ctypes.c_double
            L.orc_f32_to_bf16.argtypes = [ctypes.c_float]
            L.orc_f32_to_bf16.restype = ctypes.c_uint16
            L.orc_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            L.orc_e4m3_to_f64.restype = ctypes.c_double
            L.orc_f32_to_e4m3.argtypes = [ctypes.c_float]
            L.orc_f32_to_e4m3.restype = ctypes.c_uint8
            L.orc_e4m3_encode_array.argtypes = [I64, P, P]
            L.orc_bf16_encode_array.argtypes = [I64, P, P]
            L.orc_quant_blocks.argtypes = [I64, I64, I64, I64, P, P, P]
            L.orc_quant_rows_128.argtypes = [I64, I64, P, P]
            L.orc_logits.argtypes = [I64, I32, I32, I32, P, I32, P, P, P]
            L.orc_topk.argtypes = [I64, I32, I32, P, P, P]
            L.orc_permute.argtypes = [I64, I32, I32, P, P, P, P, P]
            L.orc_moe_tokens.argtypes = [I64, I32, I32, I32, I32, I32, P, P, P, P, P, P, P, P, P, P, P]
            L.orc_moe_layer.argtypes = [I64, I32, I32, I32, I32, I32, P, P, P, P, P, P, P, P, P, P, P, P]
            L.orc_pack_blob.argtypes = [I64, I32, P, P, P]
            L.orc_pack_words.argtypes = [I64, I32, P, P, P]
            L.orc_unpermute.argtypes = [I64, I32, I32, P, P, P, P]
            _lib = L
    return _lib


# ------------------------------------------------------------------ helpers

def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def as_bits(t) -> tuple[np.ndarray, int]:
    """A torch CPU tensor (fp32 or bf16) as (contiguous numpy array, dtype code)."""
    import torch
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.float32:
        return t.numpy(), DT_F32
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16), DT_BF16
    if t.dtype == torch.uint8:
        return t.numpy(), 2
    raise TypeError(f"oracle takes fp32, bf16 or uint8 tensors, got {t.dtype}")


# ---------------------------------------------------------------- functions

def bf16_encode(a: np.ndarray) -> np.ndarray:
    a = _c(a, np.float32)
    out = np.empty(a.shape, np.uint16)
    lib().orc_bf16_encode_array(a.size, _p(a), _p(out))
    return out


def e4m3_encode(a: np.ndarray) -> np.ndarray:
    a = _c(a, np.float32)
    out = np.empty(a.shape, np.uint8)
    lib().orc_e4m3_encode_array(a.size, _p(a), _p(out))
    return out


def e4m3_decode(q: np.ndarray) -> np.ndarray:
    L = lib()
    table = np.array([L.orc_e4m3_to_f64(i) for i in range(256)], np.float64)
    return table[np.asarray(q, np.uint8)]


def quant_blocks(w: np.ndarray, br: int, bc: int):
    """Block E4M3 quantisation of a row-major fp32 matrix (last two dims)."""
    w = _c(w, np.float32)
    rows, cols = w.shape[-2], w.shape[-1]
    lead = int(np.prod(w.shape[:-2])) if w.ndim > 2 else 1
    q = np.empty(w.shape, np.uint8)
    s = np.empty(w.shape[:-2] + (rows // br, cols // bc), np.float32)
    w2 = w.reshape(lead * rows, cols)
    # blocks never straddle two leading slices because rows % br == 0
    lib().orc_quant_blocks(lead * rows, cols, br, bc, _p(w2), _p(q), _p(s))
    return q, s


def quant_rows_128(v: np.ndarray) -> np.ndarray:
    """The FP8 layer's activation quantiser (per row, per 128 columns) as
    the doubles its codes stand for (code * scale)."""
    v = _c(v, np.float32)
    rows, cols = v.shape
    deq = np.empty((rows, cols), np.float64)
    lib().orc_quant_rows_128(rows, cols, _p(v), _p(deq))
    return deq


def logits(x, w_r, bias=None) -> np.ndarray:
    xb, xdt = as_bits(x)
    wb, wdt = as_bits(w_r)
    T, D = xb.shape
    E = wb.shape[0]
    b = None if bias is None else _c(bias.detach().cpu().numpy() if hasattr(bias, "detach") else bias, np.float32)
    z = np.empty((T, E), np.float64)
    lib().orc_logits(T, D, E, xdt, _p(xb), wdt, _p(wb), _p(b), _p(z))
    return z


def topk(z: np.ndarray, k: int):
    z = _c(z, np.float64)
    T, E = z.shape
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    lib().orc_topk(T, E, k, _p(z), _p(idx), _p(w))
    return idx, w


def permute(idx: np.ndarray, E: int):
    idx = _c(idx, np.int32)
    T, k = idx.shape
    counts = np.empty(E + 1, np.int32)
    offsets = np.empty(E + 2, np.int32)
    inv = np.empty(T * k, np.int32)
    src = np.empty(T * k + T, np.int32)
    lib().orc_permute(T, E, k, _p(idx), _p(counts), _p(offsets), _p(inv), _p(src))
    return counts, offsets, inv, src


def pack_blob(idx: np.ndarray, w: np.ndarray) -> np.ndarray:
    idx = _c(idx, np.int32)
    w32 = _c(w, np.float32)
    T, k = idx.shape
    blob = np.empty((2, T, k), np.int32)
    lib().orc_pack_blob(T, k, _p(idx), _p(w32), _p(blob))
    return blob


def pack_words(idx: np.ndarray, w: np.ndarray) -> np.ndarray:
    """One int32 per slot: index in bits 0..15, bf16 weight in bits 16..31."""
    idx = _c(idx, np.int32)
    w32 = _c(w, np.float32)
    T, k = idx.shape
    out = np.empty((T, k), np.int32)
    lib().orc_pack_words(T, k, _p(idx), _p(w32), _p(out))
    return out


def unpermute(y: np.ndarray, w: np.ndarray, inv: np.ndarray, T: int, k: int) -> np.ndarray:
    y = _c(y, np.float64)
    w = _c(w, np.float64)
    inv = _c(inv, np.int32)
    D = y.shape[1]
    out = np.empty((T, D), np.float64)
    lib().orc_unpermute(T, D, k, _p(y), _p(w), _p(inv), _p(out))
    return out


class Experts:
    """Expert weights in the form the oracle reads: (E+1) groups, the last one
    being the shared expert; mode 'f32' / 'bf16' take the tensors as stored,
    mode 'fp8' takes E4M3 codes plus [G, rows/128, cols/128] fp32 scales."""

    def __init__(self, mode: str, wg, wu, wd, sg=None, su=None, sd=None):
        self.mode = mode
        conv = (lambda a: _c(a, np.uint8)) if mode == "fp8" else (lambda a: as_bits(a)[0])
        self.wg, self.wu, self.wd = conv(wg), conv(wu), conv(wd)
        self.sg = None if sg is None else _c(sg, np.float32)
        self.su = None if su is None else _c(su, np.float32)
        self.sd = None if sd is None else _c(sd, np.float32)
        self.G, self.I, self.D = self.wg.shape

    @classmethod
    def quantised(cls, wg_f32, wu_f32, wd_f32):
        """Quantise fp32 weights with the oracle's own 128x128 block codec."""
        f = lambda t: t.detach().cpu().float().numpy() if hasattr(t, "detach") else t
        qg, sg = quant_blocks(f(wg_f32), 128, 128)
        qu, su = quant_blocks(f(wu_f32), 128, 128)
        qd, sd = quant_blocks(f(wd_f32), 128, 128)
        return cls("fp8", qg, qu, qd, sg, su, sd)


def moe_tokens(x, idx: np.ndarray, w: np.ndarray, ex: Experts, want_y: bool = False):
    """Layer output for the given tokens with the given routing (fp64)."""
    xb, _ = as_bits(x)
    n, D = xb.shape
    idx = _c(idx, np.int32)
    w = _c(w, np.float64)
    k = idx.shape[1]
    E = ex.G - 1
    out = np.empty((n, D), np.float64)
    y = np.empty((n, k + 1, D), np.float64) if want_y else None
    lib().orc_moe_tokens(n, D, E, ex.I, k, MODE[ex.mode], _p(xb), _p(idx), _p(w), _p(ex.wg),
                         _p(ex.wu), _p(ex.wd), _p(ex.sg), _p(ex.su), _p(ex.sd), _p(out), _p(y))
    return (out, y) if want_y else out


def moe_layer(x, w_r, bias, ex: Experts, k: int):
    """The whole layer from x (fp64 logits, own routing)."""
    xb, _ = as_bits(x)
    wb, _ = as_bits(w_r)
    T, D = xb.shape
    E = wb.shape[0]
    b = None if bias is None else _c(bias.detach().cpu().numpy() if hasattr(bias, "detach") else bias, np.float32)
    out = np.empty((T, D), np.float64)
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    lib().orc_moe_layer(T, D, E, ex.I, k, MODE[ex.mode], _p(xb), _p(wb), _p(b), _p(ex.wg), _p(ex.wu),
                        _p(ex.wd), _p(ex.sg), _p(ex.su), _p(ex.sd), _p(out), _p(idx), _p(w))
    return out, idx, w
