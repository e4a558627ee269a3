"""Seeded synthetic inputs for the MoE layer block (shared by the oracle and the CUDA path).

This module only draws numbers: it holds none of the layer's arithmetic (no
dequantisation, routing, union, FFN or combine).  Every value comes from a
counter-based hash of (seed, layer, tensor, expert, attempt, element index), so any
slice -- one expert of one layer, one token row -- can be regenerated on its own, on
the CPU or on a CUDA device, with integer-exact operations.

Hash: Chris Wellons' "lowbias32" 32-bit integer mixer (hash-prospector), evaluated in
int64 with 16-bit limbs so nothing overflows on either device.  Floating point values:

* uniforms  u = (h >> 8) / 2^24, in [0, 1)
* normals   Box-Muller in float64 from two independent hashes, rounded to fp32
* bf16      round-to-nearest-even of the fp32 value (torch's conversion)

Value distributions follow the workloads the layer is measured on ("Qwen3-235B"- and
"Qwen3.5-MoE"-shaped layers with 4-bit affine, group-64 expert weights; page "SSD
Streaming Expert Layers", section "Quantized Layout"):

* hidden x ~ N(0, 1) -> bf16
* router gate W fp32 [E, d] ~ N(0, sigma_gate)
* packed weights: every nibble q uniform on 0..15 (one 32-bit hash = one u32 word)
* scale ~ U[0.005, 0.02) -> bf16;  bias = bf16(-8 * scale + N(0, 1e-3))
* optional per-expert Zipf(s) logit bias: -s * ln(rank_e) * sigma_logit, rank_e a
  seeded permutation of 1..E per layer
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch

MASK32 = 0xFFFFFFFF

# tensor ids mixed into the stream key
T_X, T_GATE_W, T_ZIPF, T_X_SEQ = 1, 2, 3, 4
T_WORDS, T_SCALE, T_BIASN = 10, 11, 12
PROJ_ID = {"up": 0, "gate": 1, "down": 2}


# --------------------------------------------------------------------------- hashing
def _mul32_const(a: torch.Tensor, c: int) -> torch.Tensor:
    lo, hi = c & 0xFFFF, c >> 16
    return (a * lo + (((a * hi) & 0xFFFF) << 16)) & MASK32


def hash32(x: torch.Tensor) -> torch.Tensor:
    """lowbias32 on an int64 tensor holding values in [0, 2^32)."""
    x = x ^ (x >> 16)
    x = _mul32_const(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32_const(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


def hash32_int(x: int) -> int:
    x &= MASK32
    x ^= x >> 16
    x = (x * 0x7FEB352D) & MASK32
    x ^= x >> 15
    x = (x * 0x846CA68B) & MASK32
    x ^= x >> 16
    return x


def stream_key(seed: int, layer: int, tensor: int, expert: int = 0, attempt: int = 0) -> int:
    h = hash32_int(seed * 0x9E3779B1 + 0x632BE5AB)
    for v in (layer, tensor, expert, attempt):
        h = hash32_int(h ^ hash32_int(v + 0x85EBCA6B))
    return h


def stream_bits(key: int, index: torch.Tensor) -> torch.Tensor:
    """32 random bits per element index (int64 tensor) for one stream."""
    h = hash32((index + key) & MASK32)
    return hash32(h ^ hash32_int(key ^ 0x27D4EB2F))


def _indices(n: int, device) -> torch.Tensor:
    return torch.arange(n, dtype=torch.int64, device=device)


def uniform(key: int, n: int, device="cpu") -> torch.Tensor:
    return (stream_bits(key, _indices(n, device)) >> 8).to(torch.float64) * (1.0 / 16777216.0)


def normal(key: int, n: int, device="cpu") -> torch.Tensor:
    idx = _indices(n, device)
    u1 = ((stream_bits(key, 2 * idx) >> 8).to(torch.float64) + 0.5) * (1.0 / 16777216.0)
    u2 = (stream_bits(key, 2 * idx + 1) >> 8).to(torch.float64) * (1.0 / 16777216.0)
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)


# --------------------------------------------------------------------------- workloads
@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    d_model: int
    num_experts: int
    top_k: int
    ffn_dim: int
    tokens: int
    layers: int
    layout: str                  # "separate" | "fused"
    gate_sigma: float
    zipf_s: float = 0.0          # 0 = no logit bias
    norm_topk_prob: int = 1
    group_size: int = 64
    chained: bool = False        # RMSNorm chaining between layers
    chain_center: bool = True    # the chaining norm removes the row mean first
    seed: int = 0
    spec: int = 0                # ranks beyond top_k exported by the router (next-token bets)
    shared_ffn_dim: int = 0      # shared expert ffn width, 0 = none
    shared_slices: int = 0       # the shared expert is stored as this many column slices
    stream_slots: int = 0        # > 0: experts in pinned host memory, a pool of this many HBM slots
    seq_rho: float = 0.0         # streamed decode: AR(1) correlation of consecutive tokens

    @property
    def shared_bytes(self) -> int:
        """Bytes of the shared expert's packed weights, scales and biases (0 without one)."""
        if not self.shared_ffn_dim:
            return 0
        d, f, g = self.d_model, self.shared_ffn_dim, self.group_size
        return 3 * (f * d // 2 + f * (d // g) * 4)

    @property
    def expert_bytes(self) -> int:
        d, f, g = self.d_model, self.ffn_dim, self.group_size
        up_gate = 2 * (f * d // 2 + f * (d // g) * 4)
        down = d * f // 2 + d * (f // g) * 4
        return up_gate + down


WORKLOADS: Dict[str, Workload] = {
    # toy single MoE layer
    "toy": Workload("toy_d512_e16_k4_f256_b16", 512, 16, 4, 256, 16, 1, "separate", 0.05, seed=0),
    # Qwen3-235B-shaped decode layer, B=1 and B=8
    "decode_b1": Workload("qwen3_235b_decode_b1", 4096, 128, 8, 1536, 1, 1, "separate", 0.02, seed=1),
    "decode_b8": Workload("qwen3_235b_decode_b8", 4096, 128, 8, 1536, 8, 1, "separate", 0.02, seed=1),
    # Qwen3-235B-shaped layer-major prefill chunk: B=64, 8 chained layers
    "prefill64": Workload("qwen3_235b_prefill_b64_l8", 4096, 128, 8, 1536, 64, 8, "separate", 0.02,
                          chained=True, seed=2),
    # Qwen3.5-MoE-shaped prefill: fused gate_up, 40 chained layers
    "q35_prefill64": Workload("qwen35_moe_prefill_b64_l40", 2048, 256, 8, 512, 64, 40, "fused", 0.02,
                              chained=True, seed=3),
    # Qwen3-235B-shaped decode chain: one token through all 94 MoE layers, the router also
    # ranking 8 more experts per layer (the next token's prefetch bets)
    "decode_b1_l94": Workload("qwen3_235b_decode_b1_l94", 4096, 128, 8, 1536, 1, 94, "separate", 0.02,
                              chained=True, seed=5, spec=8),
    # Qwen2-MoE-shaped prefill chunk (57B-A14B layer shape): 64 experts, top-8 without
    # norm_topk_prob, and a shared expert of ffn 20480 stored as 8 slices of 2560
    "qwen2_prefill64": Workload("qwen2_57b_a14b_prefill_b64_l8", 3584, 64, 8, 2560, 64, 8, "separate", 0.02,
                                norm_topk_prob=0, chained=True, seed=6, shared_ffn_dim=20480, shared_slices=8),
    # the decode chain with its experts in pinned host memory (Grace memory on GB300, read over
    # NVLink-C2C): 8 chained layers, one token per step from a correlated sequence, one pool of
    # 256 HBM slots shared by the layers
    "stream_b1_l8": Workload("qwen3_235b_stream_decode_b1_l8", 4096, 128, 8, 1536, 1, 8, "separate", 0.02,
                             chained=True, seed=7, stream_slots=256, seq_rho=0.9),
    # long skewed prompt: 4096 tokens, Zipf(1.1) logit bias, 4 chained layers
    "long4096": Workload("qwen3_235b_zipf_b4096_l4", 4096, 128, 8, 1536, 4096, 4, "separate", 0.02,
                         zipf_s=1.1, chained=True, seed=4),
}


def scaled(w: Workload, **kw) -> Workload:
    """A copy with some fields replaced (smaller parity cases of a workload)."""
    return dataclasses.replace(w, **kw)


# --------------------------------------------------------------------------- generators
def _bf16_bits(v64: torch.Tensor) -> torch.Tensor:
    """float64 -> fp32 (RNE) -> bf16 (RNE); returned as the bf16 tensor."""
    return v64.to(torch.float32).to(torch.bfloat16)


def gen_x(w: Workload, layer: int, tokens: int, attempts: Optional[torch.Tensor] = None,
          device="cpu", token_offset: int = 0) -> torch.Tensor:
    """Hidden rows x[t] ~ N(0,1) as bf16 [tokens, d].  attempts[t] > 0 re-draws row t from
    another stream (used to pick rows whose router logits are well separated)."""
    d = w.d_model
    if attempts is None:
        attempts = torch.zeros(tokens, dtype=torch.int64)
    keys = [stream_key(w.seed, layer, T_X, 0, int(a)) for a in attempts.tolist()]
    k = torch.tensor(keys, dtype=torch.int64, device=device).unsqueeze(1)
    k2 = torch.tensor([hash32_int(q ^ 0x27D4EB2F) for q in keys], dtype=torch.int64, device=device).unsqueeze(1)
    idx = (_indices(tokens, device).unsqueeze(1) + token_offset) * d + _indices(d, device).unsqueeze(0)
    h1 = hash32(hash32(((2 * idx) + k) & MASK32) ^ k2)
    h2 = hash32(hash32(((2 * idx + 1) + k) & MASK32) ^ k2)
    u1 = ((h1 >> 8).to(torch.float64) + 0.5) * (1.0 / 16777216.0)
    u2 = (h2 >> 8).to(torch.float64) * (1.0 / 16777216.0)
    z = torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)
    return _bf16_bits(z)


def gen_x_sequence(w: Workload, layer: int, tokens: int, rho: float, device="cpu") -> torch.Tensor:
    """A correlated decode sequence of hidden rows, bf16 [tokens, d]: x_0 = z_0,
    x_t = rho x_{t-1} + sqrt(1 - rho^2) z_t (z ~ N(0, 1) per element, so every x_t ~ N(0, 1)),
    in float64 before the rounding.  rho = 0 gives independent tokens."""
    d = w.d_model
    z = normal(stream_key(w.seed, layer, T_X_SEQ), tokens * d, device).reshape(tokens, d)
    x = torch.empty_like(z)
    c = math.sqrt(max(0.0, 1.0 - rho * rho))
    x[0] = z[0]
    for t in range(1, tokens):
        x[t] = rho * x[t - 1] + c * z[t]
    return _bf16_bits(x)


def gen_gate(w: Workload, layer: int, device="cpu") -> torch.Tensor:
    """Router gate weights fp32 [E, d] ~ N(0, gate_sigma)."""
    z = normal(stream_key(w.seed, layer, T_GATE_W), w.num_experts * w.d_model, device)
    return (w.gate_sigma * z).to(torch.float32).reshape(w.num_experts, w.d_model)


def gen_gate_bias(w: Workload, layer: int, device="cpu") -> Optional[torch.Tensor]:
    """Per-expert Zipf(s) logit bias fp32 [E] (None when the workload has none)."""
    if w.zipf_s <= 0.0:
        return None
    E = w.num_experts
    h = stream_bits(stream_key(w.seed, layer, T_ZIPF), _indices(E, "cpu"))
    # seeded permutation of ranks 1..E: rank of each expert = position in hash order
    order = torch.argsort(h * E + _indices(E, "cpu"))
    rank = torch.empty(E, dtype=torch.int64)
    rank[order] = torch.arange(1, E + 1, dtype=torch.int64)
    sigma_logit = w.gate_sigma * math.sqrt(w.d_model)
    bias = [-w.zipf_s * math.log(float(r)) * sigma_logit for r in rank.tolist()]
    return torch.tensor(bias, dtype=torch.float64).to(torch.float32).to(device)


def _stream_bits_multi(keys, n: int, device) -> torch.Tensor:
    """stream_bits for several streams at once: [len(keys), n]."""
    k = torch.tensor(keys, dtype=torch.int64, device=device).unsqueeze(1)
    k2 = torch.tensor([hash32_int(q ^ 0x27D4EB2F) for q in keys], dtype=torch.int64,
                      device=device).unsqueeze(1)
    h = hash32((_indices(n, device).unsqueeze(0) + k) & MASK32)
    return hash32(h ^ k2)


def gen_proj(w: Workload, layer: int, proj: str, experts=None, device="cpu"):
    """One projection of the selected experts (all by default).

    Returns (words int32 [n, out, in/8] holding u32 bits, scales bf16 [n, out, in/64],
    biases bf16 [n, out, in/64]).  Shapes: up/gate out=F in=d; down out=d in=F.
    """
    d, f, g = w.d_model, w.ffn_dim, w.group_size
    out, inn = (f, d) if proj in ("up", "gate") else (d, f)
    if experts is None:
        experts = range(w.num_experts)
    experts = list(experts)
    n = len(experts)
    pid = PROJ_ID[proj]
    nw, ng = out * inn // 8, out * inn // g
    bits = _stream_bits_multi([stream_key(w.seed, layer, T_WORDS + 16 * pid, e) for e in experts], nw, device)
    words = torch.where(bits >= 2 ** 31, bits - 2 ** 32, bits).to(torch.int32)
    del bits
    ub = _stream_bits_multi([stream_key(w.seed, layer, T_SCALE + 16 * pid, e) for e in experts], ng, device)
    s = _bf16_bits(0.005 + 0.015 * ((ub >> 8).to(torch.float64) * (1.0 / 16777216.0)))
    bk = [stream_key(w.seed, layer, T_BIASN + 16 * pid, e) for e in experts]
    idx2 = _indices(ng, device)
    k = torch.tensor(bk, dtype=torch.int64, device=device).unsqueeze(1)
    k2 = torch.tensor([hash32_int(q ^ 0x27D4EB2F) for q in bk], dtype=torch.int64, device=device).unsqueeze(1)
    h1 = hash32(hash32(((2 * idx2).unsqueeze(0) + k) & MASK32) ^ k2)
    h2 = hash32(hash32(((2 * idx2 + 1).unsqueeze(0) + k) & MASK32) ^ k2)
    u1 = ((h1 >> 8).to(torch.float64) + 0.5) * (1.0 / 16777216.0)
    u2 = (h2 >> 8).to(torch.float64) * (1.0 / 16777216.0)
    z = torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)
    b = _bf16_bits(-8.0 * s.to(torch.float64) + 1e-3 * z)
    return (words.reshape(n, out, inn // 8), s.reshape(n, out, inn // g), b.reshape(n, out, inn // g))


def shared_workload(w: Workload) -> Workload:
    """The shared expert's slices as a workload of their own: shared_slices experts of ffn
    width shared_ffn_dim / shared_slices, drawn from streams of their own (seed offset)."""
    P = w.shared_slices
    return dataclasses.replace(w, num_experts=P, top_k=P, ffn_dim=w.shared_ffn_dim // P, seed=w.seed + 0x10000,
                               shared_ffn_dim=0, shared_slices=0, spec=0)


def gen_shared_weights(w: Workload, layer: int, device="cpu", layout=None) -> Dict[str, torch.Tensor]:
    """The shared expert of one layer as its column slices (tensors [P, ...], layout of w)."""
    return gen_layer_weights(shared_workload(w), layer, device=device, layout=layout)


def gen_layer_weights(w: Workload, layer: int, experts=None, device="cpu", layout=None) -> Dict[str, torch.Tensor]:
    """All expert weights of one layer in the requested layout.

    separate: w_up/s_up/b_up, w_gate/s_gate/b_gate, w_down/s_down/b_down.
    fused:    w_gate_up/s_gate_up/b_gate_up (per expert: gate rows on top, up rows below,
              the same values as the separate gate and up projections) plus the down tensors.
    """
    layout = layout or w.layout
    up = gen_proj(w, layer, "up", experts, device)
    gate = gen_proj(w, layer, "gate", experts, device)
    down = gen_proj(w, layer, "down", experts, device)
    out = {"w_down": down[0], "s_down": down[1], "b_down": down[2]}
    if layout == "separate":
        out.update(w_up=up[0], s_up=up[1], b_up=up[2], w_gate=gate[0], s_gate=gate[1], b_gate=gate[2])
    elif layout == "fused":
        out.update(w_gate_up=torch.cat([gate[0], up[0]], 1).contiguous(),
                   s_gate_up=torch.cat([gate[1], up[1]], 1).contiguous(),
                   b_gate_up=torch.cat([gate[2], up[2]], 1).contiguous())
    else:
        raise ValueError(layout)
    return out
