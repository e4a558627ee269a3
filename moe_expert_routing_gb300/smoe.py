"""Thin Python binding of libsmoe (C ABI in include/smoe.h), same function names.

Argument marshalling only: torch tensors in, device pointers and the current CUDA stream
out to the library; every step of the MoE block runs in libsmoe's kernels.  There is no
fallback: if ``libsmoe.so`` is missing or fails to load, the first call raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, field
from typing import Dict, Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libsmoe.so")

SMOE_OK, SMOE_ERR_INVALID_ARG, SMOE_ERR_UNSUPPORTED, SMOE_ERR_WORKSPACE, SMOE_ERR_CUDA, SMOE_ERR_DEVICE_FAULT = range(6)
SMOE_LAYOUT_SEPARATE, SMOE_LAYOUT_FUSED_GATE_UP = 0, 1
SMOE_FAULT_EXPERT_INDEX, SMOE_FAULT_FP16_RANGE, SMOE_FAULT_TIMEOUT, SMOE_FAULT_TOKEN_INDEX = 1, 2, 4, 8
SMOE_FAULT_SLOT_POOL = 0x10

EXPORTED = ("smoe_workspace_bytes", "smoe_route", "smoe_route_ranked", "smoe_expert_union", "smoe_moe_ffn_batch",
            "smoe_moe_ffn_batch_norm", "smoe_moe_layer", "smoe_shared_expert_ffn", "smoe_rmsnorm_bf16",
            "smoe_clear_device_status", "smoe_read_device_status", "smoe_status_string", "smoe_route_noalloc",
            "smoe_stream_state_bytes", "smoe_stream_init", "smoe_stream_plan", "smoe_stream_copy")


class SmoeError(RuntimeError):
    def __init__(self, status: int, what: str, bits: int = 0):
        self.status, self.bits = status, bits
        super().__init__(f"{what}: {_status_string(status)} (status {status}, device bits {bits:#x})")


class LayerDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("d_model", "num_experts", "top_k", "ffn_dim", "group_size", "norm_topk_prob", "layout")]


class ExpertWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("w_up", "s_up", "b_up", "w_gate", "s_gate", "b_gate",
                 "w_gate_up", "s_gate_up", "b_gate_up", "w_down", "s_down", "b_down")]


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libsmoe.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"libsmoe.so not found at {path}: build it with moe_expert_routing_gb300/build.py "
                               "(or __graft_entry__.build())")
        L = ctypes.CDLL(path)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        L.smoe_workspace_bytes.restype = sz
        L.smoe_workspace_bytes.argtypes = [vp, i32]
        L.smoe_route.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, sz, vp]
        L.smoe_route_ranked.argtypes = [vp, vp, vp, vp, i32, i32, vp, vp, vp, vp, vp, sz, vp]
        L.smoe_expert_union.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, vp, sz, vp]
        L.smoe_moe_ffn_batch.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.smoe_moe_ffn_batch_norm.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, i32, vp,
                                              vp, sz, vp]
        L.smoe_moe_layer.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, sz, vp]
        L.smoe_shared_expert_ffn.argtypes = [vp, vp, vp, i32, vp, vp, sz, vp]
        L.smoe_rmsnorm_bf16.argtypes = [vp, ctypes.c_float, i32, i32, i32, vp, vp]
        L.smoe_route_noalloc.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp]
        L.smoe_route_noalloc.restype = ctypes.c_int
        L.smoe_stream_state_bytes.restype = sz
        L.smoe_stream_state_bytes.argtypes = [i32, i32]
        L.smoe_stream_init.argtypes = [vp, i32, i32, vp]
        L.smoe_stream_plan.argtypes = [vp, i32, i32, vp, vp, vp, i32, i32, vp, vp, vp, sz, vp]
        L.smoe_stream_copy.argtypes = [vp, vp, vp, i32, vp, vp, sz, vp]
        L.smoe_clear_device_status.argtypes = [vp, vp]
        L.smoe_read_device_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
        L.smoe_status_string.restype = ctypes.c_char_p
        L.smoe_status_string.argtypes = [ctypes.c_int]
        for name in ("smoe_route", "smoe_route_ranked", "smoe_expert_union", "smoe_moe_ffn_batch",
                     "smoe_moe_ffn_batch_norm", "smoe_moe_layer",
                     "smoe_shared_expert_ffn", "smoe_rmsnorm_bf16", "smoe_clear_device_status",
                     "smoe_read_device_status", "smoe_stream_init", "smoe_stream_plan", "smoe_stream_copy"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def _status_string(status: int) -> str:
    try:
        return load_library().smoe_status_string(status).decode()
    except Exception:  # pragma: no cover
        return "?"


def _check(status: int, what: str):
    if status != SMOE_OK:
        raise SmoeError(status, what)


def _p(t: Optional[torch.Tensor]):
    """Device pointer of a contiguous CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libsmoe takes CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("libsmoe takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def make_desc(d_model: int, num_experts: int, top_k: int, ffn_dim: int, layout: str = "separate",
              norm_topk_prob: int = 1, group_size: int = 64) -> LayerDesc:
    return LayerDesc(d_model, num_experts, top_k, ffn_dim, group_size, norm_topk_prob,
                     SMOE_LAYOUT_SEPARATE if layout == "separate" else SMOE_LAYOUT_FUSED_GATE_UP)


def _hp(t: torch.Tensor):
    """Host address of a contiguous pinned CPU tensor (the streamed-expert copy reads it)."""
    if t.is_cuda or not t.is_pinned():
        raise ValueError("host expert tensors must be pinned CPU tensors")
    if not t.is_contiguous():
        raise ValueError("libsmoe takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


@dataclass
class Weights:
    """Expert weight tensors of one layer (CUDA); names as in smoe_expert_weights."""
    tensors: Dict[str, torch.Tensor]
    struct: ExpertWeights = field(init=False)

    def __post_init__(self):
        self.struct = ExpertWeights()
        for name, _ in ExpertWeights._fields_:
            t = self.tensors.get(name)
            if t is not None:
                setattr(self.struct, name, self._ptr(t).value)

    @staticmethod
    def _ptr(t):
        return _p(t)


class HostWeights(Weights):
    """Expert weight tensors of one layer in pinned host memory (smoe_stream_copy's source)."""

    @staticmethod
    def _ptr(t):
        return _hp(t)


def pin_weights(tensors: Dict[str, torch.Tensor]) -> HostWeights:
    """Pinned host copies of a layer's expert tensors."""
    return HostWeights({k: v.cpu().pin_memory() for k, v in tensors.items()})


def pool_tensors(tensors: Dict[str, torch.Tensor], n_slots: int, device="cuda") -> Dict[str, torch.Tensor]:
    """Empty device tensors shaped like a layer's expert tensors with n_slots experts."""
    return {k: torch.empty((n_slots,) + tuple(v.shape[1:]), dtype=v.dtype, device=device)
            for k, v in tensors.items()}


# ------------------------------------------------------------------------------ C ABI calls
def smoe_workspace_bytes(desc: LayerDesc, max_tokens: int) -> int:
    return int(load_library().smoe_workspace_bytes(ctypes.byref(desc), max_tokens))


def alloc_workspace(desc: LayerDesc, max_tokens: int, device="cuda") -> torch.Tensor:
    """A zeroed workspace tensor (the torch caching allocator returns 512-byte aligned blocks)."""
    n = smoe_workspace_bytes(desc, max_tokens)
    if n == 0:
        raise SmoeError(SMOE_ERR_INVALID_ARG, "smoe_workspace_bytes")
    ws = torch.zeros(n, dtype=torch.uint8, device=device)
    assert ws.data_ptr() % 256 == 0
    return ws


def smoe_route(desc, x, gate_w, gate_bias, topk_idx, topk_w, ws, stream=None):
    _check(load_library().smoe_route(ctypes.byref(desc), _p(x), _p(gate_w), _p(gate_bias), x.shape[0],
                                     _p(topk_idx), _p(topk_w), _p(ws), ws.numel(), _stream(stream)), "smoe_route")


def smoe_route_ranked(desc, x, gate_w, gate_bias, topk_idx, topk_w, spec_idx, spec_p, ws, stream=None):
    """smoe_route plus ranks top_k .. top_k + n_spec - 1 (n_spec = spec_idx.shape[1]); spec_p may be None."""
    n_spec = 0 if spec_idx is None else spec_idx.shape[1]
    _check(load_library().smoe_route_ranked(ctypes.byref(desc), _p(x), _p(gate_w), _p(gate_bias), x.shape[0], n_spec,
                                            _p(topk_idx), _p(topk_w), _p(spec_idx), _p(spec_p), _p(ws), ws.numel(),
                                            _stream(stream)), "smoe_route_ranked")


def smoe_route_noalloc(desc, x, gate_w, gate_bias, topk_idx, topk_w, stream=None):
    """smoe_route without a workspace (a fixed 4 MiB scratch array inside the library; see smoe.h)."""
    _check(load_library().smoe_route_noalloc(ctypes.byref(desc), _p(x), _p(gate_w), _p(gate_bias), x.shape[0],
                                             _p(topk_idx), _p(topk_w), _stream(stream)), "smoe_route_noalloc")


def smoe_expert_union(desc, topk_idx, union_ids, n_union, offsets, token_list, slot_list, ws, stream=None):
    _check(load_library().smoe_expert_union(ctypes.byref(desc), _p(topk_idx), topk_idx.shape[0], _p(union_ids),
                                            _p(n_union), _p(offsets), _p(token_list), _p(slot_list), _p(ws),
                                            ws.numel(), _stream(stream)), "smoe_expert_union")


def smoe_moe_ffn_batch(desc, weights: Weights, x, union_ids, n_union, offsets, token_list, slot_list, topk_w,
                       residual, ws, stream=None):
    _check(load_library().smoe_moe_ffn_batch(ctypes.byref(desc), ctypes.byref(weights.struct), _p(x), x.shape[0],
                                             _p(union_ids), _p(n_union), _p(offsets), _p(token_list),
                                             _p(slot_list), _p(topk_w), _p(residual), _p(ws), ws.numel(),
                                             _stream(stream)), "smoe_moe_ffn_batch")


def smoe_moe_ffn_batch_norm(desc, weights: Weights, x, union_ids, n_union, offsets, token_list, slot_list, topk_w,
                            residual, x_next, ws, eps: float = 1e-6, center: int = 0, stream=None):
    """smoe_moe_ffn_batch, then x_next = bf16(norm(residual)) (the next block's input; may be x)."""
    _check(load_library().smoe_moe_ffn_batch_norm(ctypes.byref(desc), ctypes.byref(weights.struct), _p(x),
                                                  x.shape[0], _p(union_ids), _p(n_union), _p(offsets),
                                                  _p(token_list), _p(slot_list), _p(topk_w), _p(residual),
                                                  ctypes.c_float(eps), int(center), _p(x_next), _p(ws), ws.numel(),
                                                  _stream(stream)), "smoe_moe_ffn_batch_norm")


def smoe_moe_layer(desc, weights: Weights, x, gate_w, gate_bias, residual, ws, topk_idx=None, topk_w=None,
                   stream=None):
    _check(load_library().smoe_moe_layer(ctypes.byref(desc), ctypes.byref(weights.struct), _p(x), _p(gate_w),
                                         _p(gate_bias), x.shape[0], _p(residual), _p(topk_idx), _p(topk_w), _p(ws),
                                         ws.numel(), _stream(stream)), "smoe_moe_layer")


def smoe_shared_expert_ffn(desc, weights: Weights, x, residual, ws, stream=None):
    """residual += shared expert(x) for every row of x (weights as P column slices, see smoe.h)."""
    _check(load_library().smoe_shared_expert_ffn(ctypes.byref(desc), ctypes.byref(weights.struct), _p(x), x.shape[0],
                                                 _p(residual), _p(ws), ws.numel(), _stream(stream)),
           "smoe_shared_expert_ffn")


def smoe_rmsnorm_bf16(h, x_out, eps: float = 1e-6, center: int = 0, stream=None):
    _check(load_library().smoe_rmsnorm_bf16(_p(h), ctypes.c_float(eps), int(center), h.shape[0], h.shape[1],
                                            _p(x_out), _stream(stream)), "smoe_rmsnorm_bf16")


def smoe_stream_state_bytes(n_keys: int, n_slots: int) -> int:
    return int(load_library().smoe_stream_state_bytes(n_keys, n_slots))


def alloc_stream_state(n_keys: int, n_slots: int, device="cuda", stream=None) -> torch.Tensor:
    """A device state buffer for n_keys (layer, expert) keys and n_slots pool slots, initialised
    to an empty pool."""
    n = smoe_stream_state_bytes(n_keys, n_slots)
    if n == 0:
        raise SmoeError(SMOE_ERR_INVALID_ARG, "smoe_stream_state_bytes")
    st = torch.empty(n // 4, dtype=torch.int32, device=device)
    smoe_stream_init(st, n_keys, n_slots, stream)
    return st


def smoe_stream_init(state, n_keys: int, n_slots: int, stream=None):
    _check(load_library().smoe_stream_init(_p(state), n_keys, n_slots, _stream(stream)), "smoe_stream_init")


def smoe_stream_plan(desc, B: int, key_base: int, union_ids, n_union, state, n_keys: int, n_slots: int, slot_ids,
                     copy_list, ws, stream=None):
    _check(load_library().smoe_stream_plan(ctypes.byref(desc), B, key_base, _p(union_ids), _p(n_union), _p(state),
                                           n_keys, n_slots, _p(slot_ids), _p(copy_list), _p(ws), ws.numel(),
                                           _stream(stream)), "smoe_stream_plan")


def smoe_stream_copy(desc, host_weights: Weights, pool_weights: Weights, n_slots: int, copy_list, ws, stream=None):
    _check(load_library().smoe_stream_copy(ctypes.byref(desc), ctypes.byref(host_weights.struct),
                                           ctypes.byref(pool_weights.struct), n_slots, _p(copy_list), _p(ws),
                                           ws.numel(), _stream(stream)), "smoe_stream_copy")


def smoe_clear_device_status(ws, stream=None):
    _check(load_library().smoe_clear_device_status(_p(ws), _stream(stream)), "smoe_clear_device_status")


def smoe_read_device_status(ws, stream=None) -> int:
    """Synchronises the stream; returns the device status bits (0 = no fault)."""
    bits = ctypes.c_uint32(0)
    st = load_library().smoe_read_device_status(_p(ws), _stream(stream), ctypes.byref(bits))
    if st not in (SMOE_OK, SMOE_ERR_DEVICE_FAULT):
        raise SmoeError(st, "smoe_read_device_status")
    return int(bits.value)


def smoe_status_string(status: int) -> str:
    return _status_string(status)


# ------------------------------------------------------------------------------ conveniences
def bf16_bits(t: torch.Tensor) -> torch.Tensor:
    """A bf16 tensor viewed as its uint16 bit patterns (int16 storage)."""
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t
