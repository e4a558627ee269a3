"""Routing statistics (next-token coverage, adjacent reuse) and the correlated decode
sequence they are measured on: host-side checks against brute force and closed forms."""
import numpy as np

import oracle
from moe_expert_routing_gb300 import routing_stats as RS
from moe_expert_routing_gb300 import workload as W


def _coverage_loop(pred, true_idx):
    """Brute force: count, element by element, the next token's experts found in pred."""
    T, K = true_idx.shape
    total = 0
    for t in range(T - 1):
        for e in true_idx[t + 1]:
            found = False
            for p in pred[t]:
                if p == e:
                    found = True
            total += found
    return total / (K * (T - 1))


def test_coverage_matches_bruteforce():
    rng = np.random.default_rng(31)
    for E, K, R in [(16, 4, 4), (128, 8, 16), (9, 3, 7)]:
        idx = np.stack([rng.choice(E, R, replace=False) for _ in range(40)])
        top = idx[:, :K]
        assert RS.next_token_coverage(idx, top) == _coverage_loop(idx, top)
        assert RS.adjacent_reuse(top) == _coverage_loop(top, top)


def test_coverage_closed_forms():
    same = np.tile(np.array([[3, 1, 4, 7]]), (10, 1))
    assert RS.adjacent_reuse(same) == 1.0
    disjoint = np.array([[0, 1], [2, 3], [0, 1], [2, 3]])
    assert RS.adjacent_reuse(disjoint) == 0.0
    half = np.array([[0, 1], [1, 2], [2, 3]])
    assert RS.adjacent_reuse(half) == 0.5
    # a ranking that contains the top-K never covers less than the top-K alone
    rng = np.random.default_rng(32)
    ranked = np.stack([rng.choice(64, 12, replace=False) for _ in range(30)])
    assert RS.next_token_coverage(ranked, ranked[:, :6]) >= RS.adjacent_reuse(ranked[:, :6])


def test_sequence_is_ar1_with_unit_variance():
    w = W.scaled(W.WORKLOADS["toy"], d_model=512)
    for rho in (0.0, 0.9):
        x = W.gen_x_sequence(w, 0, 400, rho).float().numpy().astype(np.float64)
        assert abs(x.var() - 1.0) < 0.05
        lag1 = np.mean(np.sum(x[1:] * x[:-1], axis=1) / np.sqrt(np.sum(x[1:] ** 2, 1) * np.sum(x[:-1] ** 2, 1)))
        assert abs(lag1 - rho) < 0.02


def test_oracle_routing_reuse_grows_with_correlation():
    """On the oracle's exact routing of a toy router: independent tokens reuse about K/E of
    each other's experts, strongly correlated ones nearly all; a wider ranking covers more."""
    w = W.WORKLOADS["toy"]
    gate = W.gen_gate(w, 0)
    stats = []
    for rho in (0.0, 0.9, 0.999):
        x = W.gen_x_sequence(w, 0, 200, rho)
        idx, _, sidx, _, _ = oracle.route_ranked(x, gate, None, w.top_k, 4, 1)
        stats.append(RS.sequence_stats(idx, sidx))
    reuse = [s["adjacent_reuse"] for s in stats]
    assert abs(reuse[0] - w.top_k / w.num_experts) < 0.1
    assert reuse[0] < reuse[1] < reuse[2] and reuse[2] > 0.9
    assert all(s["ranked_coverage"] >= s["adjacent_reuse"] for s in stats)
