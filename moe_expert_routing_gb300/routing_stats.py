"""Routing statistics of a token sequence: how much of the next token's routing the current
token already knows.  Instrumentation over the device's routing outputs (not a step of the
MoE block).

Page "Data Flow" (the measured fact the design rests on: adjacent tokens reuse 46.4% of each
other's experts; the current token's top-16 gate ranking covers 63.7% of the next token's
top-8) and "Why There Is No Routing Predictor" (the coverage table: share of the next
token's true top-8 found in a predictor's set).

    python -m moe_expert_routing_gb300.routing_stats [--rho R ...] [--tokens T]

routes a seeded correlated decode sequence (workload.gen_x_sequence) through one
Qwen3-235B-shaped router with smoe_route_ranked (top-8 plus 8 ranked bets) on the GPU and
prints one JSON line per rho.
"""
from __future__ import annotations

import argparse
import json

import numpy as np


def next_token_coverage(pred, true_idx) -> float:
    """Mean over t of |pred[t] & true_idx[t + 1]| / K: the share of token t+1's routed
    experts (true_idx [T, K]) already in token t's predicted set (pred [T, R], R >= 1)."""
    pred = np.asarray(pred)
    true_idx = np.asarray(true_idx)
    T, K = true_idx.shape
    if T < 2:
        return float("nan")
    hits = [len(set(pred[t].tolist()) & set(true_idx[t + 1].tolist())) for t in range(T - 1)]
    return float(np.mean(hits) / K)


def adjacent_reuse(idx) -> float:
    """Mean over t of |idx[t] & idx[t + 1]| / K (each token's routed experts against the next)."""
    return next_token_coverage(idx, idx)


def sequence_stats(topk_idx, spec_idx) -> dict:
    """Reuse of the previous token's top-K and coverage by its top-(K + spec) ranking."""
    ranked = np.concatenate([np.asarray(topk_idx), np.asarray(spec_idx)], axis=1)
    return {"adjacent_reuse": adjacent_reuse(topk_idx), "ranked_coverage": next_token_coverage(ranked, topk_idx),
            "ranks": int(ranked.shape[1])}


def main():
    import torch

    from . import smoe
    from . import workload as W

    ap = argparse.ArgumentParser()
    ap.add_argument("--rho", type=float, nargs="+", default=[0.0, 0.5, 0.9, 0.97, 0.99])
    ap.add_argument("--tokens", type=int, default=512)
    ap.add_argument("--spec", type=int, default=8)
    args = ap.parse_args()
    w = W.WORKLOADS["decode_b1"]
    dev = torch.device("cuda")
    desc = smoe.make_desc(w.d_model, w.num_experts, w.top_k, w.ffn_dim, w.layout, w.norm_topk_prob)
    gate = W.gen_gate(w, 0, device=dev).contiguous()
    T = args.tokens
    ws = smoe.alloc_workspace(desc, T, dev)
    idx = torch.empty(T, w.top_k, dtype=torch.int32, device=dev)
    wt = torch.empty(T, w.top_k, dtype=torch.float32, device=dev)
    sidx = torch.empty(T, args.spec, dtype=torch.int32, device=dev)
    for rho in args.rho:
        x = W.gen_x_sequence(w, 0, T, rho).to(dev).view(torch.int16).contiguous()
        smoe.smoe_route_ranked(desc, x, gate, None, idx, wt, sidx, None, ws)
        st = sequence_stats(idx.cpu().numpy(), sidx.cpu().numpy())
        print(json.dumps({"rho": rho, "tokens": T, "router": w.name, **st}), flush=True)


if __name__ == "__main__":
    main()
