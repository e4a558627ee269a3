"""Shared test helpers: seeded cases for the oracle and the CUDA path (no layer arithmetic).

The only arithmetic here is bookkeeping on oracle outputs (logit gaps, error norms).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from moe_expert_routing_gb300 import workload as W


def logit_gaps(lg: np.ndarray, K: int) -> np.ndarray:
    """Per token, the smallest gap between adjacent sorted logits among ranks 1..K+1."""
    s = -np.sort(-lg, axis=1)
    kk = min(K + 1, lg.shape[1])
    return (s[:, :kk - 1] - s[:, 1:kk]).min(axis=1) if kk > 1 else np.full(lg.shape[0], np.inf)


def resampled_x(w: W.Workload, layer: int, B: int, gate_w, gate_bias=None, delta: float = 1e-3, max_rounds=64):
    """Layer-0 inputs with every adjacent oracle logit gap among ranks 1..K+1 >= delta:
    rows that fail are redrawn from the next stream (attempt counter) until all pass."""
    attempts = torch.zeros(B, dtype=torch.int64)
    x = W.gen_x(w, layer, B, attempts)
    bad = logit_gaps(oracle.logits(x, gate_w, gate_bias), w.top_k) < delta
    for _ in range(max_rounds):
        if not bad.any():
            return x, attempts
        rows = np.nonzero(bad)[0]
        attempts[rows] += 1
        x[rows] = W.gen_x(w, layer, B, attempts)[rows] if B <= 64 else torch.stack(
            [W.gen_x(w, layer, 1, attempts[r:r + 1], token_offset=int(r))[0] for r in rows])
        bad[rows] = logit_gaps(oracle.logits(x[rows], gate_w, gate_bias), w.top_k) < delta
    raise RuntimeError("could not draw well-separated router logits")


def bf16_to_f64(bits) -> np.ndarray:
    return (np.asarray(bits, np.uint32).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rmsnorm_glue_close(gpu_bits, oracle_bits, abs_tol: float = 1e-4):
    """The fp32 RMSNorm glue against the double-precision one: each value within one bf16 ulp
    of the oracle's plus an absolute slack for the fp32 rounding of near-zero values (the row
    mean is removed in fp32); returns the fraction of values that differ at all."""
    g = bf16_to_f64(np.asarray(gpu_bits).astype(np.int64) & 0xFFFF)
    o = bf16_to_f64(np.asarray(oracle_bits).astype(np.int64) & 0xFFFF)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(o), 1e-30))) - 7)
    assert np.all(np.abs(g - o) <= ulp + abs_tol), float(np.max(np.abs(g - o) - ulp))
    return float((g != o).mean())


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def max_abs(a, b) -> float:
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64)))) if np.size(a) else 0.0


# Output tolerance of the MoE block: relative L2 <= 5e-3 on the layer delta and on the output,
# max-abs <= 2e-2 (absolute).  The GPU path computes with fp16 operands (exact dequantised
# integers, bf16->fp16 exact activations, fp16-rounded SwiGLU activations) and fp32
# accumulation; the oracle in double.
REL_L2_TOL = 5e-3
MAX_ABS_TOL = 2e-2
# Routing weights: fp32 softmax (expf) vs double.
W_RTOL = 1e-5
