"""CPU oracle for the per-layer MoE block (double precision) -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference
leg use this package.  It wraps ``oracle/smoe_oracle.cpp`` (plain C++, built by
``oracle/build.py``) through ctypes and shares nothing with the CUDA library.

Each function cites the passage it follows (page title and section):

* ``dequant``      -- "SSD Streaming Expert Layers", "Quantized Layout"
* ``logits``/``topk``/``route`` -- "Layer-Major Batched Prefill", "Choreography Per Chunk"
  step 5 (real router gate on the true hidden state, norm_topk_prob re-normalisation);
  "Surface Scout", "The Model Config" (``norm_topk_prob`` field)
* ``route_ranked`` -- "Data Flow", "Serial Step Trace" (ranked top-(8 + spec), the ranks
  beyond 8 as next-token bets)
* ``expert_union`` -- "Layer-Major Batched Prefill", "The Inversion" (dedupe into the
  expert UNION, each union expert applied to every routed token)
* ``expert_ffn``   -- "SSD Streaming Expert Layers", "Math Contract" (down(silu(gate(x)) * up(x)))
* ``moe_layer``    -- "Data Flow", "Serial Step Trace" FFN block (gather outputs x routing
  weights into the residual); token-major vs layer-major: "Layer-Major Batched Prefill",
  "The Inversion" and "Measured Result" (identical outputs)
* ``rmsnorm_bf16`` -- "Data Flow", "Serial Step Trace" (RMS norm before the FFN block)
* ``shared_dense_layer`` / ``shared_expert_ffn`` -- "Data Flow", "Serial Step Trace" (the
  shared expert FFN on every token, residual += shared_out + routed_out); "Surface Scout",
  "The Model Config" (shared_expert_ffn_dim)
* ``SlotPool``     -- "Data Flow", "Ring Buffer State Machine" (slots keyed by (layer, expert)
  retained as cache entries; EMPTY slots first, else the least-recently-used idle slot is
  evicted; freshly loaded slots carry the new tick) and "Handling Misses"; "Layer-Major
  Batched Prefill", "Retention, never replay" (keep what was read, never wipe per token)
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libsmoe_oracle.so")
_lib = None


class _Desc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("d_model", "num_experts", "top_k", "ffn_dim", "group_size", "norm_topk_prob", "layout")]


class _Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("w_up", "s_up", "b_up", "w_gate", "s_gate", "b_gate",
                 "w_gate_up", "s_gate_up", "b_gate_up", "w_down", "s_down", "b_down")]


def lib():
    """The loaded oracle library (built on first use if missing), signatures installed."""
    global _lib
    if _lib is None:
        from . import build as _b
        _b.build()
        L = ctypes.CDLL(_LIB_PATH)
        _setup_signatures(L)
        _lib = L
    return _lib


def _np(a, dtype):
    """Contiguous numpy view of a torch tensor or array with the given dtype (bit view)."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().contiguous()
            if a.dtype == torch.bfloat16:
                a = a.view(torch.int16)
            a = a.numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        if a.dtype.itemsize == np.dtype(dtype).itemsize and a.dtype.kind in "iu" and np.dtype(dtype).kind in "iu":
            a = a.view(dtype)
        else:
            a = a.astype(dtype)
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def hardware_threads() -> int:
    return int(lib().oracle_hardware_threads())


def dequant(words, scales, biases, group_size: int = 64) -> np.ndarray:
    """fp32 weights [rows, in] of one projection: w = scale * q + bias per 64-group."""
    q = _np(words, np.uint32)
    s = _np(scales, np.uint16)
    b = _np(biases, np.uint16)
    rows = q.shape[-2] if q.ndim >= 2 else 1
    lead = int(np.prod(q.shape[:-1]))
    inn = q.shape[-1] * 8
    out = np.empty((lead, inn), np.float32)
    rc = lib().oracle_dequant(_ptr(q), _ptr(s), _ptr(b), ctypes.c_int64(lead), ctypes.c_int64(inn),
                              ctypes.c_int32(group_size), _ptr(out))
    if rc:
        raise ValueError(f"oracle_dequant rc={rc}")
    return out.reshape(q.shape[:-1] + (inn,)) if rows else out


def logits(x_bf16, gate_w, gate_bias=None) -> np.ndarray:
    """Router logits in double [B, E]."""
    x = _np(x_bf16, np.uint16)
    W = _np(gate_w, np.float32)
    bias = None if gate_bias is None else _np(gate_bias, np.float32)
    B, d = x.shape
    E = W.shape[0]
    out = np.empty((B, E), np.float64)
    rc = lib().oracle_logits(_ptr(x), _ptr(W), _ptr(bias), B, d, E, _ptr(out))
    if rc:
        raise ValueError(f"oracle_logits rc={rc}")
    return out


def topk(lg: np.ndarray, K: int, norm_topk_prob: int = 1):
    """(idx int32 [B,K], w64 [B,K], w32 [B,K]) from double logits."""
    lg = np.ascontiguousarray(lg, np.float64)
    B, E = lg.shape
    idx = np.empty((B, K), np.int32)
    w64 = np.empty((B, K), np.float64)
    w32 = np.empty((B, K), np.float32)
    rc = lib().oracle_topk(_ptr(lg), B, E, K, norm_topk_prob, _ptr(idx), _ptr(w64), _ptr(w32))
    if rc:
        raise ValueError(f"oracle_topk rc={rc}")
    return idx, w64, w32


def route(x_bf16, gate_w, gate_bias, K: int, norm_topk_prob: int = 1):
    """Exact routing: (idx, w64, w32, logits)."""
    lg = logits(x_bf16, gate_w, gate_bias)
    idx, w64, w32 = topk(lg, K, norm_topk_prob)
    return idx, w64, w32, lg


def route_ranked(x_bf16, gate_w, gate_bias, K: int, n_spec: int, norm_topk_prob: int = 1):
    """Exact routing with the ranking continued: (idx, w64, spec_idx, spec_p64, logits).

    Page "Data Flow", "Serial Step Trace": the exact gate matvec produces a ranked
    top-(8 + spec); ranks 8 and beyond are the next token's prefetch bets.  idx / w64 are
    the routing of ``route``; spec_idx holds ranks K .. K + n_spec - 1 of the same order
    (descending logit, ties -> lower id) and spec_p64 their probabilities under the
    softmax over all experts (not renormalised).
    """
    lg = logits(x_bf16, gate_w, gate_bias)
    idx, w64, _ = topk(lg, K, norm_topk_prob)
    full, p64, _ = topk(lg, K + n_spec, 0)
    return idx, w64, full[:, K:].copy(), p64[:, K:].copy(), lg


def expert_union(idx, E: int):
    """(union_ids [n_union], offsets [n_union+1], token_list, slot_list)."""
    idx = _np(idx, np.int32)
    B, K = idx.shape
    uid = np.zeros(E, np.int32)
    nu = np.zeros(1, np.int32)
    off = np.zeros(E + 1, np.int32)
    tl = np.zeros(max(1, B * K), np.int32)
    sl = np.zeros(max(1, B * K), np.int32)
    rc = lib().oracle_union(_ptr(idx), B, K, E, _ptr(uid), _ptr(nu), _ptr(off), _ptr(tl), _ptr(sl))
    if rc:
        raise ValueError(f"oracle_union rc={rc}")
    n = int(nu[0])
    return uid[:n].copy(), off[:n + 1].copy(), tl[:B * K].copy(), sl[:B * K].copy()


class SlotPool:
    """Residency of (layer, expert) keys in a pool of n_slots weight slots (plain Python).

    One ``plan`` per layer call, in the order the pages give: the tick advances; every key of
    the call's union that a slot already holds is a hit (its slot is re-stamped with the tick);
    the misses, in union order, take the idle slots (slots holding no key of this union) in
    order of (stamp, slot id) -- empty slots carry stamp -1, so they come first, then the least
    recently used; equal stamps (slots loaded by the same call) go lowest slot id first.  A
    taken slot's previous key stops being resident; the slot now holds the missed key with the
    new tick.  Returns (slot of each union position, [(key, slot)] copies in miss order).
    """

    def __init__(self, n_keys: int, n_slots: int):
        self.n_keys, self.n_slots = n_keys, n_slots
        self.tick = 0
        self.slot_of = [-1] * n_keys
        self.owner = [-1] * n_slots
        self.stamp = [-1] * n_slots

    def plan(self, keys: Sequence[int]):
        keys = [int(k) for k in keys]
        if len(set(keys)) != len(keys) or any(not 0 <= k < self.n_keys for k in keys):
            raise ValueError("a union holds distinct keys in range")
        self.tick += 1
        slots = [-1] * len(keys)
        in_use = set()
        for u, k in enumerate(keys):
            if self.slot_of[k] >= 0:
                slots[u] = self.slot_of[k]
                in_use.add(slots[u])
        idle = sorted((self.stamp[s], s) for s in range(self.n_slots) if s not in in_use)
        misses = [u for u in range(len(keys)) if slots[u] < 0]
        if len(misses) > len(idle):
            raise ValueError("more misses than idle slots")
        copies = []
        for m, u in enumerate(misses):
            s = idle[m][1]
            old = self.owner[s]
            if old >= 0:
                self.slot_of[old] = -1
            self.owner[s] = keys[u]
            self.slot_of[keys[u]] = s
            slots[u] = s
            copies.append((keys[u], s))
        for s in slots:
            self.stamp[s] = self.tick
        return slots, copies


class Layer:
    """One layer's descriptor + weights (numpy copies kept alive for the C calls)."""

    def __init__(self, d_model, num_experts, top_k, ffn_dim, weights: Dict, layout="separate",
                 norm_topk_prob=1, group_size=64):
        self.desc = _Desc(d_model, num_experts, top_k, ffn_dim, group_size, norm_topk_prob,
                          0 if layout == "separate" else 1)
        self._arrs = {}
        wts = _Weights()
        for name in _Weights._fields_:
            n = name[0]
            if n in weights and weights[n] is not None:
                a = _np(weights[n], np.uint32 if n.startswith("w_") else np.uint16)
                self._arrs[n] = a
                setattr(wts, n, a.ctypes.data)
        self.weights = wts

    @classmethod
    def from_workload(cls, w, weights: Dict, layout=None):
        return cls(w.d_model, w.num_experts, w.top_k, w.ffn_dim, weights, layout or w.layout,
                   w.norm_topk_prob, w.group_size)


def expert_ffn(layer: Layer, expert: int, x_bf16, tokens: Sequence[int]) -> np.ndarray:
    """y [n, d] (double) of one expert for the listed token rows of x."""
    x = _np(x_bf16, np.uint16)
    t = np.ascontiguousarray(np.asarray(tokens, np.int32))
    y = np.empty((len(t), layer.desc.d_model), np.float64)
    rc = lib().oracle_expert_ffn(ctypes.byref(layer.desc), ctypes.byref(layer.weights), expert, _ptr(x),
                                 _ptr(t), len(t), _ptr(y))
    if rc:
        raise ValueError(f"oracle_expert_ffn rc={rc}")
    return y


def moe_layer(layer: Layer, x_bf16, idx, w64, residual, mode: str = "layer", threads: int = 0,
              rows: Optional[Sequence[int]] = None, want_slots: bool = False):
    """out = residual + sum_k w[t,k] * y_{idx[t,k]}(x[t]) for the given routing.

    Returns (out fp32 [B,d], out64 [B,d], y_slots [B,K,d] or None).  Only ``rows`` are
    computed when given (the other rows of the outputs are left zero).
    """
    x = _np(x_bf16, np.uint16)
    idx = _np(idx, np.int32)
    w64 = np.ascontiguousarray(w64, np.float64)
    res = _np(residual, np.float32)
    B, d = x.shape
    K = layer.desc.top_k
    out = np.zeros((B, d), np.float32)
    out64 = np.zeros((B, d), np.float64)
    ys = np.zeros((B, K, d), np.float64) if want_slots else None
    r = None if rows is None else np.ascontiguousarray(np.asarray(rows, np.int32))
    if threads <= 0:
        threads = hardware_threads()
    rc = lib().oracle_moe_combine(ctypes.byref(layer.desc), ctypes.byref(layer.weights), _ptr(x), B, _ptr(idx),
                                  _ptr(w64), _ptr(res), _ptr(out), _ptr(out64), 0 if mode == "layer" else 1,
                                  threads, _ptr(ys), _ptr(r), 0 if r is None else len(r))
    if rc:
        raise ValueError(f"oracle_moe_combine rc={rc}")
    return out, out64, ys


def shared_dense_layer(slices: Dict, d_model: int, P: int, F: int, layout: str = "separate") -> Layer:
    """The shared expert as ONE dense expert of ffn width P * F, reassembled from its P
    column slices (slice p = FFN columns pF .. pF + F - 1): gate / up rows of the slices
    stacked in slice order, down input columns (packed words, scale and bias groups)
    concatenated in slice order.  Returned in the separate layout."""
    a = {k: _np(v, np.uint32 if k.startswith("w_") else np.uint16) for k, v in slices.items()}
    if layout == "fused":
        gu = {k[0]: a[f"{k}_gate_up"] for k in ("w", "s", "b")}
        gate = {c: np.ascontiguousarray(gu[c][:, :F]) for c in gu}
        up = {c: np.ascontiguousarray(gu[c][:, F:]) for c in gu}
    else:
        gate = {c: a[f"{c}_gate"] for c in ("w", "s", "b")}
        up = {c: a[f"{c}_up"] for c in ("w", "s", "b")}
    dense = {}
    for c in ("w", "s", "b"):
        dense[f"{c}_gate"] = np.ascontiguousarray(gate[c].reshape(1, P * F, -1))
        dense[f"{c}_up"] = np.ascontiguousarray(up[c].reshape(1, P * F, -1))
        dense[f"{c}_down"] = np.ascontiguousarray(np.concatenate(list(a[f"{c}_down"]), axis=-1)[None])
    assert dense["w_down"].shape == (1, d_model, P * F // 8)
    return Layer(d_model, 1, 1, P * F, dense, "separate", 1)


def shared_expert_ffn(dense: Layer, x_bf16) -> np.ndarray:
    """y [B, d] (double): the shared expert applied to every row of x."""
    B = _np(x_bf16, np.uint16).shape[0]
    return expert_ffn(dense, 0, x_bf16, list(range(B)))


def rmsnorm_bf16(h, eps: float = 1e-6, center: bool = False) -> np.ndarray:
    """bf16 bits (uint16) of (h - c) / sqrt(mean((h - c)^2) + eps), c = row mean if center else 0,
    computed in double."""
    h = _np(h, np.float32)
    B, d = h.shape
    out = np.empty((B, d), np.uint16)
    rc = lib().oracle_rmsnorm_bf16(_ptr(h), B, d, ctypes.c_double(eps), int(bool(center)), _ptr(out))
    if rc:
        raise ValueError(f"oracle_rmsnorm_bf16 rc={rc}")
    return out


def to_bf16(v) -> np.ndarray:
    """Round doubles to bf16 bits (nearest, ties to even)."""
    v = np.ascontiguousarray(v, np.float64)
    out = np.empty(v.shape, np.uint16)
    rc = lib().oracle_to_bf16(_ptr(v), ctypes.c_int64(v.size), _ptr(out))
    if rc:
        raise ValueError("oracle_to_bf16")
    return out


def _setup_signatures(L):
    L.oracle_dequant.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                                                          ctypes.c_void_p]
    L.oracle_logits.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int32] * 3 + [ctypes.c_void_p]
    L.oracle_topk.argtypes = [ctypes.c_void_p] + [ctypes.c_int32] * 4 + [ctypes.c_void_p] * 3
    L.oracle_union.argtypes = [ctypes.c_void_p] + [ctypes.c_int32] * 3 + [ctypes.c_void_p] * 5
    L.oracle_expert_ffn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                    ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p]
    L.oracle_moe_combine.argtypes = ([ctypes.c_void_p] * 3 + [ctypes.c_int32] + [ctypes.c_void_p] * 5 +
                                     [ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_int32])
    L.oracle_rmsnorm_bf16.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_double,
                                      ctypes.c_int32, ctypes.c_void_p]
    L.oracle_to_bf16.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]

