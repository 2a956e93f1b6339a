"""MoELayer: one routed-MoE FFN layer held on the GPU, driven through libmoe.

Holds the plan, the device weights (E4M3 codes and block scales for the FP8
layer, quantised by the library's own kernel), and a workspace sized for
T_max tokens.  forward() is one moe_forward call.
"""
from __future__ import annotations

import torch

from . import _lib as L

_TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16}


class MoELayer:
    def __init__(self, D: int, E: int, I: int, top_k: int, dtype: str, weights: dict, T_max: int,
                 out_dtype: str = "f32", has_router_bias: bool = False, flags: int = 0, device: int = 0,
                 spin_limit_ns: int = 0, keep_fp32: bool = False):
        self.D, self.E, self.I, self.top_k, self.dtype = D, E, I, top_k, dtype
        self.out_dtype, self.T_max, self.device = out_dtype, T_max, device
        self.plan = L.moe_plan_create(T_max, D, E, I, top_k, dtype, out_dtype, has_router_bias, flags,
                                      spin_limit_ns, device)
        dev = torch.device("cuda", device)
        w = {n: weights[n] for n in ("w_router", "b_router") if weights.get(n) is not None}
        if not has_router_bias:
            w.pop("b_router", None)
        if dtype == "fp8":
            for n, sn in (("w_gate", "s_gate"), ("w_up", "s_up"), ("w_down", "s_down")):
                src = weights[n]
                if src.dtype == torch.uint8:          # already quantised
                    w[n], w[sn] = src, weights[sn]
                    continue
                G, R, C = src.shape
                q = torch.empty((G, R, C), dtype=torch.uint8, device=dev)
                s = torch.empty((G, R // 128, C // 128), dtype=torch.float32, device=dev)
                L.moe_quantize_weights(self.plan, src.contiguous(), q, s)
                w[n], w[sn] = q, s
                if keep_fp32:
                    w[n + "_f32"] = src
        else:
            for n in ("w_gate", "w_up", "w_down"):
                w[n] = weights.get(n)
        self.ws = torch.empty(L.moe_workspace_size(self.plan, T_max), dtype=torch.uint8, device=dev)
        L.moe_workspace_init(self.plan, self.ws)
        self.hilo = dtype == "bf16" and bool(flags & L.MOE_FLAG_DOWN_HILO)
        if dtype == "bf16" and not self.hilo:
            if weights.get("w_down_f16") is not None:
                w["w_down_f16"] = weights["w_down_f16"]  # w_down may then be absent
            elif w.get("w_down") is not None:
                wd = w["w_down"].contiguous()
                w["w_down"] = wd
                w["w_down_f16"] = torch.empty(wd.shape, dtype=torch.float16, device=dev)
                L.moe_convert_down_weights(self.plan, wd, w["w_down_f16"], self.ws)
                L.moe_check(self.plan, self.ws)
        self.w = w
        self.cw = L.make_weights(w)

    @classmethod
    def from_shape(cls, shape, inputs: dict, T_max: int = None, **kw):
        return cls(shape.D, shape.E, shape.I, shape.top_k, shape.dtype, inputs, T_max or shape.T,
                   has_router_bias=shape.has_bias, **kw)

    def __del__(self):
        try:
            L.moe_plan_destroy(self.plan)
        except Exception:
            pass

    # ------------------------------------------------------------- calls

    def new_out(self, T: int) -> torch.Tensor:
        return torch.empty((T, self.D), dtype=_TORCH_DT[self.out_dtype], device=self.ws.device)

    def forward(self, x: torch.Tensor, out: torch.Tensor = None, blob_out=None, logits_out=None) -> torch.Tensor:
        T = x.shape[0]
        if out is None:
            out = self.new_out(T)
        L.moe_forward(self.plan, self.cw, x, T, out, blob_out, logits_out, self.ws)
        return out

    def route(self, x):
        L.moe_route(self.plan, self.cw, x, x.shape[0], self.ws)

    def topk(self, T):
        L.moe_topk(self.plan, T, self.ws)

    def permute(self, x):
        L.moe_permute(self.plan, x, x.shape[0], self.ws)

    def gemm_gateup(self, x):
        L.moe_gemm_gateup(self.plan, self.cw, x, x.shape[0], self.ws)

    def gemm_down(self, T):
        L.moe_gemm_down(self.plan, self.cw, T, self.ws)

    def unpermute(self, T, out=None):
        if out is None:
            out = self.new_out(T)
        L.moe_unpermute(self.plan, T, out, self.ws)
        return out

    def check(self):
        L.moe_check(self.plan, self.ws)

    def init_ws(self):
        L.moe_workspace_init(self.plan, self.ws)

    # ----------------------------------------------------- workspace views

    def ws_view(self, T: int, part: str, dtype: torch.dtype, shape) -> torch.Tensor:
        """A view of one workspace part for T tokens (see moe_ws_layout)."""
        lay = L.moe_workspace_layout(self.plan, T)
        off = getattr(lay, part)
        n = 1
        for s in shape:
            n *= s
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        return self.ws[off:off + nbytes].view(dtype).view(*shape)

    def views(self, T: int) -> dict:
        k, E, D, I = self.top_k, self.E, self.D, self.I
        TK, R = T * k, T * k + T
        act = {"f32": torch.float32, "bf16": torch.bfloat16, "fp8": torch.uint8}[self.dtype]
        f16_down = self.dtype == "bf16" and not self.hilo
        ydt = torch.bfloat16 if self.dtype == "fp8" else torch.float16 if f16_down else torch.float32
        hcols = 2 * I if self.hilo else I
        hdt = torch.float16 if f16_down else act
        v = {
            "err": self.ws_view(T, "err", torch.int32, (4,)),
            "logits": self.ws_view(T, "logits", torch.float32, (T, E)),
            "blob": self.ws_view(T, "blob", torch.int32, (2, T, k)),
            "counts": self.ws_view(T, "counts", torch.int32, (E + 1,)),
            "offsets": self.ws_view(T, "offsets", torch.int32, (E + 2,)),
            "tiles": self.ws_view(T, "tiles", torch.int32, (E + 2,)),
            "inv": self.ws_view(T, "inv", torch.int32, (TK,)),
            "src_tok": self.ws_view(T, "src_tok", torch.int32, (R,)),
            "xp": self.ws_view(T, "xp", act, (TK, D)),
            "h": self.ws_view(T, "h", hdt, (R, hcols)),
            "y": self.ws_view(T, "y", ydt, (R, D)),
        }
        if self.dtype == "fp8":
            v["xq"] = self.ws_view(T, "xq", torch.uint8, (T, D))
            v["xq_scale"] = self.ws_view(T, "xq_scale", torch.float32, (T, D // 128))
            v["xp_scale"] = self.ws_view(T, "xp_scale", torch.float32, (TK, D // 128))
            v["h_scale"] = self.ws_view(T, "h_scale", torch.float32, (R, I // 128))
        return v
