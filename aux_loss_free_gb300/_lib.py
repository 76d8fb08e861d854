"""ctypes binding of libmoe_gb300.so: argument marshalling only.

Every function here has the name of a C entry point in include/moe_gb300.h, takes
torch tensors that already live on the GPU (PyTorch supplies device memory and the
stream) and passes their pointers through.  All computation happens in the library's
CUDA kernels; there is no other code path.  If the library has not been built the
first call raises, it never falls back to anything else.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmoe_gb300.so")

MOE_X_BF16, MOE_X_F32 = 0, 1
MOE_W_BF16, MOE_W_INT4_G32 = 0, 1

STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
                3: "MOE_ERR_WORKSPACE", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT",
                6: "MOE_ERR_DEVICE"}

# Every symbol the header declares, with (restype, argtypes).
_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_F = ctypes.c_float


class MoEShape(ctypes.Structure):
    _fields_ = [("T", _I32), ("d", _I32), ("E", _I32), ("f", _I32), ("F", _I32), ("k", _I32),
                ("renorm", _I32), ("x_dtype", _I32), ("w_format", _I32)]


class MoEWeights(ctypes.Structure):
    _fields_ = [("w_gate_up", _P), ("w_down", _P), ("scale_gate_up", _P), ("scale_down", _P),
                ("shared_gate_up", _P), ("shared_down", _P)]


class MoEDebug(ctypes.Structure):
    _fields_ = [("scores", _P), ("idx", _P), ("gate", _P), ("load", _P), ("offsets", _P),
                ("perm_tok", _P), ("inv_pos", _P), ("balance", _P)]


# moe_balance_t: int64 pairs, int32 max_load, min_load, dead_experts, float
# max_over_mean, min_over_mean, dead_fraction (32 bytes).
BALANCE_BYTES = 32
MOE_TK_FROM_LOAD = -1


class MoEGrads(ctypes.Structure):
    _fields_ = [("dx", _P), ("dw_router", _P), ("dw_gate_up", _P), ("dw_down", _P),
                ("ds_gate_up", _P), ("ds_down", _P), ("dgate", _P)]


class MoEAttnShape(ctypes.Structure):
    _fields_ = [("batch", _I32), ("seq", _I32), ("d", _I32), ("n_head", _I32), ("n_kv_head", _I32),
                ("head_dim", _I32), ("eps", _F)]


class MoECacheStats(ctypes.Structure):
    _fields_ = [("steps", _I64), ("hits", _I64), ("misses", _I64), ("evictions", _I64), ("bytes", _I64),
                ("overflow", _I64)]


_SHAPE_P = ctypes.POINTER(MoEShape)
SIGNATURES = {
    "moe_abi_version": (_I32, []),
    "moe_status_string": (ctypes.c_char_p, [_I32]),
    "moe_gate_up_block": (_I32, [_I32]),
    "moe_route_workspace_size": (_SZ, [_SHAPE_P]),
    "moe_route": (_I32, [_SHAPE_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_permute_workspace_size": (_SZ, [_SHAPE_P]),
    "moe_permute": (_I32, [_SHAPE_P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_permute_noalloc": (_I32, [_SHAPE_P, _P, _P, _P, _P, _P]),
    "moe_expert_ffn_workspace_size": (_SZ, [_SHAPE_P]),
    "moe_expert_ffn": (_I32, [_SHAPE_P, _P, _P, _P, ctypes.POINTER(MoEWeights), _P, _P, _P, _SZ,
                              _P]),
    "moe_combine": (_I32, [_SHAPE_P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_gather_rows": (_I32, [_I64, _I32, _P, _P, _P, _P]),
    "moe_ep_regroup": (_I32, [_I32, _I32, _P, _P, _P, _P, _P]),
    "moe_bias_update": (_I32, [_I32, _I64, _P, _F, _P, _P]),
    "moe_load_balance": (_I32, [_I32, _P, _P, _P]),
    "moe_layer_workspace_size": (_SZ, [_SHAPE_P]),
    "moe_layer_fwd": (_I32, [_SHAPE_P, _P, _P, _P, _P, _F, _I32, ctypes.POINTER(MoEWeights), _P,
                             _P, ctypes.POINTER(MoEDebug), _P, _SZ, _P]),
    "moe_layer_bwd_workspace_size": (_SZ, [_SHAPE_P]),
    "moe_layer_bwd": (_I32, [_SHAPE_P, _P, _P, ctypes.POINTER(MoEWeights), ctypes.POINTER(MoEDebug),
                             _P, _I32, ctypes.POINTER(MoEGrads), _P, _SZ, _P]),
    "moe_expert_cache_bytes": (_SZ, [_SHAPE_P, _I32]),
    "moe_expert_cache_init": (_I32, [_SHAPE_P, _I32, _P, _SZ, _P]),
    "moe_expert_cache_read": (_I32, [_SHAPE_P, _I32, _P, ctypes.POINTER(MoECacheStats), _P, _P, _P, _P]),
    "moe_layer_fwd_cached": (_I32, [_SHAPE_P, _P, _P, _P, _P, _F, _I32, ctypes.POINTER(MoEWeights), _I32, _P,
                                    _SZ, _P, _P, ctypes.POINTER(MoEDebug), _P, _SZ, _P]),
    "moe_attention_workspace_size": (_SZ, [ctypes.POINTER(MoEAttnShape)]),
    "moe_attention_fwd": (_I32, [ctypes.POINTER(MoEAttnShape), _P, _P, _P, _I32, _P, _P, _SZ, _P]),
    "moe_attention_core": (_I32, [ctypes.POINTER(MoEAttnShape), _P, _P, _P]),
    "moe_pack_gate_up": (_I32, [_I32, _I32, _I32, _P, _P, _P, _P]),
    "moe_quantize_int4": (_I32, [_I64, _I32, _P, _P, _P, _P]),
    "moe_device_status": (_I32, [_P, ctypes.POINTER(_I32)]),
    "moe_selftest_bounded_wait": (_I32, [_I64, ctypes.POINTER(_I32), _P]),
    "moe_last_device_status": (_I32, [_P]),
    "moe_workspace_size": (_SZ, [_SHAPE_P]),
    "moe_profile_stage_count": (_I32, []),
    "moe_profile_stage_name": (ctypes.c_char_p, [_I32]),
    "moe_profile_stage_calls": (_I32, [_I32]),
    "moe_profile_start": (_I32, [_I32, _I32]),
    "moe_profile_stop": (_I32, [ctypes.POINTER(_F), ctypes.POINTER(_I32)]),
}

_lib = None


class MoEError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(code, code)}")
        self.code = code


def load_library(path: str = LIB_PATH):
    """Load the shared library once and declare every entry point's signature."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m aux_loss_free_gb300.build`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(name: str, code: int):
    if code != 0:
        raise MoEError(name, code)


def make_shape(T, d, E, f, F, k, renorm=True, x_dtype=MOE_X_BF16, w_format=MOE_W_BF16) -> MoEShape:
    return MoEShape(T, d, E, f, F, k, int(bool(renorm)), x_dtype, w_format)


def make_weights(w_gate_up, w_down, shared_gate_up=None, shared_down=None, scale_gate_up=None,
                 scale_down=None) -> MoEWeights:
    return MoEWeights(_ptr(w_gate_up), _ptr(w_down), _ptr(scale_gate_up), _ptr(scale_down),
                      _ptr(shared_gate_up), _ptr(shared_down))


def moe_abi_version() -> int:
    return load_library().moe_abi_version()


def moe_gate_up_block(width: int) -> int:
    return load_library().moe_gate_up_block(width)


def moe_route_workspace_size(shape) -> int:
    return load_library().moe_route_workspace_size(ctypes.byref(shape))


def moe_route(shape, x, w_router, logit_offset, bias, scores, idx, gate, load, workspace=None,
              stream=None):
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("moe_route", load_library().moe_route(
        ctypes.byref(shape), _ptr(x), _ptr(w_router), _ptr(logit_offset), _ptr(bias), _ptr(scores),
        _ptr(idx), _ptr(gate), _ptr(load), _ptr(workspace), nbytes, _stream(stream)))


def moe_permute_workspace_size(shape) -> int:
    return load_library().moe_permute_workspace_size(ctypes.byref(shape))


def moe_permute(shape, idx, offsets, perm_tok, inv_pos, workspace, stream=None):
    _check("moe_permute", load_library().moe_permute(
        ctypes.byref(shape), _ptr(idx), _ptr(offsets), _ptr(perm_tok), _ptr(inv_pos),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_permute_noalloc(shape, idx, offsets, perm_tok, inv_pos, stream=None):
    """moe_permute with the library's fixed static scratch instead of a workspace."""
    _check("moe_permute_noalloc", load_library().moe_permute_noalloc(
        ctypes.byref(shape), _ptr(idx), _ptr(offsets), _ptr(perm_tok), _ptr(inv_pos),
        _stream(stream)))


def moe_expert_ffn_workspace_size(shape) -> int:
    return load_library().moe_expert_ffn_workspace_size(ctypes.byref(shape))


def moe_expert_ffn(shape, x, offsets, perm_tok, weights: MoEWeights, y_perm, shared_out, workspace,
                   stream=None):
    _check("moe_expert_ffn", load_library().moe_expert_ffn(
        ctypes.byref(shape), _ptr(x), _ptr(offsets), _ptr(perm_tok), ctypes.byref(weights),
        _ptr(y_perm), _ptr(shared_out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_combine(shape, y_perm, shared_out, inv_pos, gate, residual, out, stream=None):
    _check("moe_combine", load_library().moe_combine(
        ctypes.byref(shape), _ptr(y_perm), _ptr(shared_out), _ptr(inv_pos), _ptr(gate),
        _ptr(residual), _ptr(out), _stream(stream)))


def moe_gather_rows(rows, d, src, index, dst, stream=None):
    _check("moe_gather_rows", load_library().moe_gather_rows(
        rows, d, _ptr(src), _ptr(index), _ptr(dst), _stream(stream)))


def moe_ep_regroup(world, experts_local, counts, perm, inv, offsets, stream=None):
    _check("moe_ep_regroup", load_library().moe_ep_regroup(
        world, experts_local, _ptr(counts), _ptr(perm), _ptr(inv), _ptr(offsets), _stream(stream)))


def moe_bias_update(E, tokens_times_k, load, gamma, bias, stream=None):
    _check("moe_bias_update", load_library().moe_bias_update(
        E, tokens_times_k, _ptr(load), gamma, _ptr(bias), _stream(stream)))


def moe_load_balance(E, load, balance, stream=None):
    """balance: a device buffer of at least BALANCE_BYTES bytes (see balance_from_bytes)."""
    _check("moe_load_balance", load_library().moe_load_balance(E, _ptr(load), _ptr(balance), _stream(stream)))


def balance_from_bytes(raw) -> dict:
    """Decode one moe_balance_t from its 32 bytes (a uint8 tensor or bytes on the host)."""
    import numpy as np
    b = np.frombuffer(bytes(raw.cpu().numpy().tobytes() if hasattr(raw, "cpu") else raw)[:BALANCE_BYTES],
                      dtype=np.uint8)
    return {"pairs": int(b[0:8].view(np.int64)[0]),
            "max_load": int(b[8:12].view(np.int32)[0]),
            "min_load": int(b[12:16].view(np.int32)[0]),
            "dead_experts": int(b[16:20].view(np.int32)[0]),
            "max_over_mean": b[20:24].view(np.float32)[0],
            "min_over_mean": b[24:28].view(np.float32)[0],
            "dead_fraction": b[28:32].view(np.float32)[0]}


def moe_layer_workspace_size(shape) -> int:
    return load_library().moe_layer_workspace_size(ctypes.byref(shape))


def moe_layer_fwd(shape, x, w_router, logit_offset, bias, gamma, update_bias, weights: MoEWeights,
                  residual, out, workspace, debug: MoEDebug | None = None, stream=None):
    _check("moe_layer_fwd", load_library().moe_layer_fwd(
        ctypes.byref(shape), _ptr(x), _ptr(w_router), _ptr(logit_offset), _ptr(bias), gamma,
        int(update_bias), ctypes.byref(weights), _ptr(residual), _ptr(out),
        ctypes.byref(debug) if debug is not None else None, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def make_debug(scores=None, idx=None, gate=None, load=None, offsets=None, perm_tok=None,
               inv_pos=None, balance=None) -> MoEDebug:
    return MoEDebug(_ptr(scores), _ptr(idx), _ptr(gate), _ptr(load), _ptr(offsets), _ptr(perm_tok),
                    _ptr(inv_pos), _ptr(balance))


def moe_layer_bwd_workspace_size(shape) -> int:
    return load_library().moe_layer_bwd_workspace_size(ctypes.byref(shape))


def make_grads(dx, dw_router, dw_gate_up, dw_down, ds_gate_up=None, ds_down=None,
               dgate=None) -> MoEGrads:
    return MoEGrads(_ptr(dx), _ptr(dw_router), _ptr(dw_gate_up), _ptr(dw_down), _ptr(ds_gate_up),
                    _ptr(ds_down), _ptr(dgate))


def moe_layer_bwd(shape, x, w_router, weights: MoEWeights, saved: MoEDebug, dout, residual,
                  grads: MoEGrads, workspace, stream=None):
    _check("moe_layer_bwd", load_library().moe_layer_bwd(
        ctypes.byref(shape), _ptr(x), _ptr(w_router), ctypes.byref(weights), ctypes.byref(saved),
        _ptr(dout), int(residual), ctypes.byref(grads), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_expert_cache_bytes(shape, slots) -> int:
    return load_library().moe_expert_cache_bytes(ctypes.byref(shape), slots)


def moe_expert_cache_init(shape, slots, cache, stream=None):
    _check("moe_expert_cache_init", load_library().moe_expert_cache_init(
        ctypes.byref(shape), slots, _ptr(cache), cache.numel() * cache.element_size(), _stream(stream)))


def moe_expert_cache_read(shape, slots, cache, stream=None):
    """-> (stats dict, slot_expert, expert_slot, stamp) as numpy int32 arrays (synchronises)."""
    import numpy as np
    st = MoECacheStats()
    se = np.empty(slots, np.int32)
    es = np.empty(shape.E, np.int32)
    sp = np.empty(slots, np.int32)
    _check("moe_expert_cache_read", load_library().moe_expert_cache_read(
        ctypes.byref(shape), slots, _ptr(cache), ctypes.byref(st), se.ctypes.data_as(_P),
        es.ctypes.data_as(_P), sp.ctypes.data_as(_P), _stream(stream)))
    return {n: getattr(st, n) for n, _ in MoECacheStats._fields_}, se, es, sp


def moe_layer_fwd_cached(shape, x, w_router, logit_offset, bias, gamma, update_bias, host_weights: MoEWeights,
                         slots, cache, residual, out, workspace, debug: MoEDebug | None = None, stream=None):
    _check("moe_layer_fwd_cached", load_library().moe_layer_fwd_cached(
        ctypes.byref(shape), _ptr(x), _ptr(w_router), _ptr(logit_offset), _ptr(bias), gamma, int(update_bias),
        ctypes.byref(host_weights), slots, _ptr(cache), cache.numel() * cache.element_size(), _ptr(residual),
        _ptr(out), ctypes.byref(debug) if debug is not None else None, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def make_attn_shape(batch, seq, d, n_head, n_kv_head, head_dim=128, eps=1e-6) -> MoEAttnShape:
    return MoEAttnShape(batch, seq, d, n_head, n_kv_head, head_dim, eps)


def moe_attention_workspace_size(shape) -> int:
    return load_library().moe_attention_workspace_size(ctypes.byref(shape))


def moe_attention_fwd(shape, x, w_qkv, w_o, residual, out, workspace, stream=None):
    _check("moe_attention_fwd", load_library().moe_attention_fwd(
        ctypes.byref(shape), _ptr(x), _ptr(w_qkv), _ptr(w_o), int(residual), _ptr(out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_attention_core(shape, qkv, o, stream=None):
    _check("moe_attention_core", load_library().moe_attention_core(
        ctypes.byref(shape), _ptr(qkv), _ptr(o), _stream(stream)))


def moe_pack_gate_up(G, width, d, w_gate, w_up, w_gate_up, stream=None):
    _check("moe_pack_gate_up", load_library().moe_pack_gate_up(
        G, width, d, _ptr(w_gate), _ptr(w_up), _ptr(w_gate_up), _stream(stream)))


def moe_quantize_int4(rows, K, w, q, scale, stream=None):
    _check("moe_quantize_int4", load_library().moe_quantize_int4(
        rows, K, _ptr(w), _ptr(q), _ptr(scale), _stream(stream)))


def moe_device_status(stream=None) -> int:
    out = _I32(0)
    _check("moe_device_status", load_library().moe_device_status(_stream(stream), ctypes.byref(out)))
    return out.value


def moe_selftest_bounded_wait(limit_ns: int, stream=None) -> int:
    """Make one bounded device wait run out (see the header); returns 1 if it gave up."""
    out = _I32(-1)
    _check("moe_selftest_bounded_wait", load_library().moe_selftest_bounded_wait(
        limit_ns, ctypes.byref(out), _stream(stream)))
    return out.value


def moe_profile_start(max_calls: int, period: int = 1):
    _check("moe_profile_start", load_library().moe_profile_start(max_calls, period))


def moe_profile_stop(per_stage_calls: bool = False):
    """-> ({stage name: summed ms}, recorded calls); with per_stage_calls, the second
    item is {stage name: recorded calls that had the stage}."""
    lib = load_library()
    n = lib.moe_profile_stage_count()
    ms = (_F * n)()
    calls = _I32(0)
    _check("moe_profile_stop", lib.moe_profile_stop(ms, ctypes.byref(calls)))
    names = [lib.moe_profile_stage_name(i).decode() for i in range(n)]
    sums = {nm: float(v) for nm, v in zip(names, ms) if nm}
    if per_stage_calls:
        return sums, {nm: int(lib.moe_profile_stage_calls(i)) for i, nm in enumerate(names) if nm}
    return sums, calls.value
