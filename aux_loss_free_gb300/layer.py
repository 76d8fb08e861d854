"""Device-side layer state: weights uploaded once, packed by the library's kernels.

PyTorch provides the device memory; packing (gate/up interleave, int4 quantisation)
runs in the library (moe_pack_gate_up, moe_quantize_int4).  `LayerOnDevice.forward`
is one moe_layer_fwd call.
"""
from __future__ import annotations

import numpy as np
import torch

from . import _lib as L


def to_device_bf16(bits: np.ndarray, device) -> torch.Tensor:
    """Upload bf16 bit patterns (uint16 numpy) as a torch.bfloat16 tensor."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def to_device_tokens(x: np.ndarray, device) -> torch.Tensor:
    if x.dtype == np.uint16:
        return to_device_bf16(x, device)
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device)


def pack_gate_up(w_gate: torch.Tensor, w_up: torch.Tensor) -> torch.Tensor:
    """[G][width][d] gate and up (bf16, device) -> interleaved [G][2*width][d]."""
    G, width, d = w_gate.shape
    out = torch.empty((G, 2 * width, d), dtype=torch.bfloat16, device=w_gate.device)
    L.moe_pack_gate_up(G, width, d, w_gate, w_up, out)
    return out


def quantize_int4(w: torch.Tensor):
    """bf16 [..., K] (device) -> (uint8 codes [..., K/2], fp16-bit scales int16 [..., K/32])."""
    K = w.shape[-1]
    rows = w.numel() // K
    q = torch.empty(w.shape[:-1] + (K // 2,), dtype=torch.uint8, device=w.device)
    s = torch.empty(w.shape[:-1] + (K // 32,), dtype=torch.int16, device=w.device)
    L.moe_quantize_int4(rows, K, w, q, s)
    return q, s


class LayerOnDevice:
    """One MoE layer's parameters on the GPU, in the layouts the library expects."""

    def __init__(self, shape, host: dict, device="cuda", x_dtype=None):
        self.spec = shape
        dev = torch.device(device)
        self.device = dev
        x_dt = x_dtype if x_dtype is not None else shape.x_dtype
        self.shape = L.make_shape(shape.T, shape.d, shape.E, shape.f, shape.F, shape.k,
                                  renorm=shape.renorm,
                                  x_dtype=L.MOE_X_F32 if x_dt == "f32" else L.MOE_X_BF16,
                                  w_format=L.MOE_W_INT4_G32 if shape.w_format == "int4" else L.MOE_W_BF16)
        self.w_router = torch.from_numpy(host["w_router"]).to(dev)
        self.bias = torch.from_numpy(host["bias"].copy()).to(dev)
        lo = host.get("logit_offset")
        self.logit_offset = None if lo is None else torch.from_numpy(lo).to(dev)
        self.gamma = float(host["gamma"])
        wg = to_device_bf16(host["w_gate"], dev)
        wu = to_device_bf16(host["w_up"], dev)
        self.w_gate_up = pack_gate_up(wg, wu)
        del wg, wu
        self.w_down = to_device_bf16(host["w_down"], dev)
        self.scale_gate_up = self.scale_down = None
        if shape.w_format == "int4":
            self.w_gate_up, self.scale_gate_up = quantize_int4(self.w_gate_up)
            self.w_down, self.scale_down = quantize_int4(self.w_down)
        self.shared_gate_up = self.shared_down = None
        if shape.F:
            sg = to_device_bf16(host["s_gate"], dev)[None]
            su = to_device_bf16(host["s_up"], dev)[None]
            self.shared_gate_up = pack_gate_up(sg, su)[0]
            self.shared_down = to_device_bf16(host["s_down"], dev)
        self.weights = L.make_weights(self.w_gate_up, self.w_down, self.shared_gate_up,
                                      self.shared_down, self.scale_gate_up, self.scale_down)
        self.ws_bytes = L.moe_layer_workspace_size(self.shape)
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)

    def forward(self, x: torch.Tensor, out: torch.Tensor, update_bias: bool = True,
                residual: torch.Tensor | None = None, debug=None, stream=None):
        L.moe_layer_fwd(self.shape, x, self.w_router, self.logit_offset, self.bias, self.gamma,
                        update_bias, self.weights, residual, out, self.workspace, debug=debug,
                        stream=stream)
        return out


class SavedForward:
    """The forward's routing state that moe_layer_bwd needs (device tensors)."""

    def __init__(self, T: int, E: int, k: int, device):
        dev = torch.device(device)
        self.scores = torch.empty((T, E), dtype=torch.float32, device=dev)
        self.idx = torch.empty((T, k), dtype=torch.int32, device=dev)
        self.gate = torch.empty((T, k), dtype=torch.float32, device=dev)
        self.load = torch.empty(E, dtype=torch.int32, device=dev)
        self.offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
        self.perm_tok = torch.empty(T * k, dtype=torch.int32, device=dev)
        self.inv_pos = torch.empty((T, k), dtype=torch.int32, device=dev)
        self.debug = L.make_debug(self.scores, self.idx, self.gate, self.load, self.offsets,
                                  self.perm_tok, self.inv_pos)


class LayerGrads:
    """Gradient buffers of one layer: bf16 dx, fp32 weight gradients."""

    def __init__(self, layer: "LayerOnDevice", want_dgate: bool = False):
        s, dev = layer.spec, layer.device
        self.dx = torch.empty((s.T, s.d), dtype=torch.bfloat16, device=dev)
        self.dw_router = torch.empty((s.E, s.d), dtype=torch.float32, device=dev)
        self.dw_gate_up = torch.empty((s.E, 2 * s.f, s.d), dtype=torch.float32, device=dev)
        self.dw_down = torch.empty((s.E, s.d, s.f), dtype=torch.float32, device=dev)
        self.ds_gate_up = self.ds_down = None
        if s.F:
            self.ds_gate_up = torch.empty((2 * s.F, s.d), dtype=torch.float32, device=dev)
            self.ds_down = torch.empty((s.d, s.F), dtype=torch.float32, device=dev)
        self.dgate = torch.empty((s.T, s.k), dtype=torch.float32, device=dev) if want_dgate else None
        self.struct = L.make_grads(self.dx, self.dw_router, self.dw_gate_up, self.dw_down,
                                   self.ds_gate_up, self.ds_down, self.dgate)


def attach_backward(layer: "LayerOnDevice"):
    """Allocate the backward workspace of a bf16 layer (once)."""
    if getattr(layer, "bwd_workspace", None) is None:
        n = L.moe_layer_bwd_workspace_size(layer.shape)
        if n == 0:
            raise L.MoEError("moe_layer_bwd_workspace_size", 2)
        layer.bwd_workspace = torch.empty(n, dtype=torch.uint8, device=layer.device)
    return layer


def layer_backward(layer: "LayerOnDevice", x: torch.Tensor, saved: SavedForward, dout: torch.Tensor,
                   grads: LayerGrads, residual: bool = False, stream=None):
    """One moe_layer_bwd call with the state a forward wrote into `saved`."""
    attach_backward(layer)
    L.moe_layer_bwd(layer.shape, x, layer.w_router, layer.weights, saved.debug, dout, residual,
                    grads.struct, layer.bwd_workspace, stream=stream)
    return grads


class ExpertCache:
    """GPU-side residency cache of a serving layer's int4 routed experts.

    The layer's int4 codes and scales are copied once to pinned host memory (the
    streaming source); the GPU keeps `slots` experts in HBM and fills them per step
    inside moe_layer_fwd_cached."""

    def __init__(self, layer: "LayerOnDevice", slots: int):
        if layer.spec.w_format != "int4":
            raise ValueError("the expert cache serves int4 layers")
        self.layer, self.slots = layer, slots
        self.host = {}
        for name in ("w_gate_up", "scale_gate_up", "w_down", "scale_down"):
            t = getattr(layer, name)
            h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
            h.copy_(t)
            self.host[name] = h
        self.host_weights = L.make_weights(self.host["w_gate_up"], self.host["w_down"], layer.shared_gate_up,
                                           layer.shared_down, self.host["scale_gate_up"], self.host["scale_down"])
        n = L.moe_expert_cache_bytes(layer.shape, slots)
        if n == 0:
            raise L.MoEError("moe_expert_cache_bytes", 2)
        self.mem = torch.empty(n, dtype=torch.uint8, device=layer.device)
        self.reset()

    def reset(self, stream=None):
        L.moe_expert_cache_init(self.layer.shape, self.slots, self.mem, stream=stream)

    def forward(self, x, out, update_bias=False, residual=None, debug=None, stream=None):
        ly = self.layer
        L.moe_layer_fwd_cached(ly.shape, x, ly.w_router, ly.logit_offset, ly.bias, ly.gamma, update_bias,
                               self.host_weights, self.slots, self.mem, residual, out, ly.workspace,
                               debug=debug, stream=stream)
        return out

    def read(self, stream=None):
        return L.moe_expert_cache_read(self.layer.shape, self.slots, self.mem, stream=stream)
