"""Pins for the CPU oracle: each test ties it to something other than itself.

The pages print no worked example with numbers, so the oracle is pinned by hand-packed
fixtures, closed forms, library routines on special cases, brute force on tiny inputs and
the invariants the pages state (layer-major == token-major; fused gate_up == separate).
Several tests also plant a mistake in the oracle's inputs to show that the pin notices it.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import expit, softmax

import oracle
from moe_expert_routing_gb300 import workload as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_bits(v):
    """bf16 bits of values that are exactly representable (test fixtures only)."""
    a = np.asarray(v, np.float32)
    return (a.view(np.uint32) >> 16).astype(np.uint16)


def _pack_rows(q):
    """Pack nibbles q[..., in] low nibble first into u32 words (fixture builder)."""
    q = np.asarray(q, np.uint32)
    sh = q.reshape(q.shape[:-1] + (q.shape[-1] // 8, 8)) << (4 * np.arange(8, dtype=np.uint32))
    return np.bitwise_or.reduce(sh, axis=-1).astype(np.uint32)


# ------------------------------------------------------------------ dequantisation
def test_dequant_handpacked_fixture():
    """Quantized Layout: hand-packed words, exact expected weights for every nibble position."""
    fx = json.load(open(os.path.join(GOLDEN, "dequant_handpacked.json")))
    for row in fx["rows"]:
        words = np.array([int(w, 16) for w in row["words"]], np.uint32)[None]
        s = np.array([int(v, 16) for v in row["scales"]], np.uint16)[None]
        b = np.array([int(v, 16) for v in row["biases"]], np.uint16)[None]
        got = oracle.dequant(words, s, b)[0]
        assert got.tolist() == row["expected"]


def test_dequant_handpacked_detects_nibble_order():
    """Planted mistake: high-nibble-first words no longer reproduce the fixture."""
    row = json.load(open(os.path.join(GOLDEN, "dequant_handpacked.json")))["rows"][0]
    words = np.array([int(w, 16) for w in row["words"]], np.uint32)
    rev = np.zeros_like(words)
    for i in range(8):
        rev |= ((words >> (4 * i)) & 15) << (4 * (7 - i))
    s = np.array([int(v, 16) for v in row["scales"]], np.uint16)[None]
    b = np.array([int(v, 16) for v in row["biases"]], np.uint16)[None]
    assert oracle.dequant(rev[None], s, b)[0].tolist() != row["expected"]


def test_dequant_random_words_match_bit_arithmetic():
    """Every nibble of random words, via numpy bit slicing, times exact scales plus biases."""
    rng = np.random.default_rng(5)
    q = rng.integers(0, 16, size=(3, 128))
    s = np.array([[2.0 ** -6, 2.0 ** -5], [0.25, 1.0], [2.0 ** -9, 0.5]])
    b = np.array([[-0.125, 0.0], [1.0, -2.0], [0.5, -0.25]])
    got = oracle.dequant(_pack_rows(q), _bf16_bits(s), _bf16_bits(b))
    want = np.repeat(s, 64, axis=1) * q + np.repeat(b, 64, axis=1)
    assert np.array_equal(got, want.astype(np.float32))


def test_bf16_rounding_fixture():
    fx = json.load(open(os.path.join(GOLDEN, "bf16_rounding.json")))
    vals = np.array([c["value"] for c in fx["cases"]])
    got = oracle.to_bf16(vals)
    assert [int(g) for g in got] == [int(c["bits"], 16) for c in fx["cases"]]


# ------------------------------------------------------------------ routing
def _one_hot_x(d, val=1.0):
    x = np.zeros((1, d), np.float32)
    x[0, 0] = val
    return _bf16_bits(x)


def test_route_closed_form_norm_topk():
    """Logits [3,1,2,0], K=2, norm_topk_prob: ids [0,2], weights e/(1+e) and 1/(1+e)."""
    d, E = 64, 4
    Wg = np.zeros((E, d), np.float32)
    Wg[:, 0] = [3.0, 1.0, 2.0, 0.0]
    idx, w64, w32, lg = oracle.route(_one_hot_x(d), Wg, None, 2, 1)
    assert lg.tolist() == [[3.0, 1.0, 2.0, 0.0]]
    assert idx.tolist() == [[0, 2]]
    e = math.e
    assert w64[0] == pytest.approx([e / (1 + e), 1 / (1 + e)], rel=1e-15)


def test_route_closed_form_no_norm():
    """norm_topk_prob = 0 keeps the full-softmax probabilities of the selected experts."""
    d, E = 64, 4
    Wg = np.zeros((E, d), np.float32)
    Wg[:, 0] = [3.0, 1.0, 2.0, 0.0]
    idx, w64, _, _ = oracle.route(_one_hot_x(d), Wg, None, 2, 0)
    e = math.e
    S = e ** 3 + e + e ** 2 + 1
    assert idx.tolist() == [[0, 2]]
    assert w64[0] == pytest.approx([e ** 3 / S, e ** 2 / S], rel=1e-14)


def test_route_bias_shifts_logits():
    d, E = 64, 4
    Wg = np.zeros((E, d), np.float32)
    Wg[:, 0] = [3.0, 1.0, 2.0, 0.0]
    bias = np.array([-5.0, 0.0, 0.0, 4.0], np.float32)
    idx, _, _, lg = oracle.route(_one_hot_x(d), Wg, bias, 2, 1)
    assert lg.tolist() == [[-2.0, 1.0, 2.0, 4.0]]
    assert idx.tolist() == [[3, 2]]


def test_route_tie_break_lower_id():
    d, E = 64, 5
    Wg = np.zeros((E, d), np.float32)
    Wg[:, 0] = [1.0, 2.0, 2.0, 0.5, 2.0]
    idx, w64, _, _ = oracle.route(_one_hot_x(d), Wg, None, 3, 1)
    assert idx.tolist() == [[1, 2, 4]]
    assert w64[0] == pytest.approx([1 / 3] * 3, rel=1e-15)


def test_route_full_k_equals_softmax_and_argsort():
    """K = E: weights are scipy's softmax and the order is a full stable argsort."""
    rng = np.random.default_rng(1)
    lg = rng.normal(size=(7, 16)) * 2
    idx, w64, _ = oracle.topk(lg, 16, 1)
    for t in range(7):
        order = np.argsort(-lg[t], kind="stable")
        assert idx[t].tolist() == order.tolist()
        assert np.allclose(w64[t], softmax(lg[t])[order], rtol=1e-13, atol=0)


def test_route_ranked_closed_form():
    """Logits [3,1,2,0], K=1, three more ranks: ids [0] then [2,1,3] with the full-softmax
    probabilities e^2/S, e/S, 1/S (S = e^3 + e + e^2 + 1); the routing itself is route's."""
    d, E = 64, 4
    Wg = np.zeros((E, d), np.float32)
    Wg[:, 0] = [3.0, 1.0, 2.0, 0.0]
    idx, w64, sidx, sp, lg = oracle.route_ranked(_one_hot_x(d), Wg, None, 1, 3, 1)
    e = math.e
    S = e ** 3 + e + e ** 2 + 1
    assert idx.tolist() == [[0]] and w64[0].tolist() == [1.0]
    assert sidx.tolist() == [[2, 1, 3]]
    assert sp[0] == pytest.approx([e ** 2 / S, e / S, 1 / S], rel=1e-14)


def test_route_ranked_continues_the_stable_argsort():
    """K + n_spec = E: routing ids followed by the ranked ids are the full stable argsort of
    the logits (ties -> lower id), and the probabilities of all ranks sum to 1."""
    rng = np.random.default_rng(5)
    d, E, K = 64, 12, 3
    Wg = rng.integers(-3, 4, size=(E, d)).astype(np.float32)   # integer logits: ties occur
    x = _bf16_bits(rng.integers(-2, 3, size=(6, d)).astype(np.float32))
    idx, w64, sidx, sp, lg = oracle.route_ranked(x, Wg, None, K, E - K, 0)
    for t in range(6):
        order = np.argsort(-lg[t], kind="stable")
        assert idx[t].tolist() + sidx[t].tolist() == order.tolist()
        assert np.allclose(np.concatenate([w64[t], sp[t]]), softmax(lg[t])[order], rtol=1e-13, atol=0)
        assert abs(w64[t].sum() + sp[t].sum() - 1.0) < 1e-12
    assert any(len(set(r)) < E for r in lg.tolist())   # the case really has ties


def test_route_bruteforce_subsets():
    """Tiny E: the chosen set maximises the summed probability over all K-subsets."""
    rng = np.random.default_rng(2)
    E, K = 7, 3
    lg = rng.normal(size=(20, E))
    idx, w64, _ = oracle.topk(lg, K, 1)
    for t in range(20):
        best = max(itertools.combinations(range(E), K), key=lambda c: sum(math.exp(lg[t, e]) for e in c))
        assert sorted(idx[t].tolist()) == sorted(best)
        assert all(lg[t, idx[t, k]] >= lg[t, idx[t, k + 1]] for k in range(K - 1))
        assert abs(w64[t].sum() - 1.0) <= 1e-12


def test_logits_integer_case_exact():
    """Small-integer gate and hidden values: every logit is an exact integer dot product."""
    rng = np.random.default_rng(3)
    d, E, B = 128, 8, 5
    x = rng.integers(-4, 5, size=(B, d)).astype(np.float32)
    Wg = rng.integers(-3, 4, size=(E, d)).astype(np.float32)
    lg = oracle.logits(_bf16_bits(x), Wg)
    assert np.array_equal(lg, (x.astype(np.int64) @ Wg.astype(np.int64).T).astype(np.float64))


def test_route_weights_sum_to_one_generated():
    w = W.WORKLOADS["toy"]
    x = W.gen_x(w, 0, 16)
    idx, w64, w32, _ = oracle.route(x, W.gen_gate(w, 0), None, w.top_k, 1)
    assert np.all(np.abs(w64.sum(1) - 1.0) <= 1e-12)
    assert np.all(np.diff(w64, axis=1) <= 0)
    assert all(len(set(r)) == w.top_k for r in idx.tolist())


# ------------------------------------------------------------------ union
def test_union_bruteforce():
    rng = np.random.default_rng(4)
    for B, K, E in [(1, 8, 128), (16, 4, 16), (64, 8, 128), (37, 3, 9)]:
        idx = np.stack([rng.choice(E, K, replace=False) for _ in range(B)]).astype(np.int32)
        uid, off, tl, sl = oracle.expert_union(idx, E)
        expect = sorted(set(idx.ravel().tolist()))
        assert uid.tolist() == expect
        for u, e in enumerate(expect):
            pairs = [(t, k) for t in range(B) for k in range(K) if idx[t, k] == e]
            assert list(zip(tl[off[u]:off[u + 1]].tolist(), sl[off[u]:off[u + 1]].tolist())) == pairs
        assert off[-1] == B * K


def test_union_rejects_bad_index():
    idx = np.array([[0, 1], [2, 16]], np.int32)
    with pytest.raises(ValueError):
        oracle.expert_union(idx, 16)


# ------------------------------------------------------------------ expert FFN
def _const_weights(F, d, s_gate, s_up, s_down, nexp=1, layout="separate"):
    """Every nibble 9, bias -8*s: each weight equals its scale exactly."""
    def proj(out, inn, s):
        q = np.full((nexp, out, inn), 9)
        return (_pack_rows(q), _bf16_bits(np.full((nexp, out, inn // 64), s)),
                _bf16_bits(np.full((nexp, out, inn // 64), -8 * s)))
    g, u, dn = proj(F, d, s_gate), proj(F, d, s_up), proj(d, F, s_down)
    wts = {"w_down": dn[0], "s_down": dn[1], "b_down": dn[2]}
    if layout == "separate":
        wts.update(w_gate=g[0], s_gate=g[1], b_gate=g[2], w_up=u[0], s_up=u[1], b_up=u[2])
    else:
        wts.update(w_gate_up=np.concatenate([g[0], u[0]], 1), s_gate_up=np.concatenate([g[1], u[1]], 1),
                   b_gate_up=np.concatenate([g[2], u[2]], 1))
    return wts


@pytest.mark.parametrize("layout", ["separate", "fused"])
def test_ffn_closed_form(layout):
    """Constant weights: g = s_g*sum(x), v = s_u*sum(x), y_j = s_d * F * silu(g) * v."""
    d, F = 128, 64
    s_g, s_u, s_d = 2.0 ** -6, 2.0 ** -7, 2.0 ** -5
    layer = oracle.Layer(d, 1, 1, F, _const_weights(F, d, s_g, s_u, s_d, layout=layout), layout)
    rng = np.random.default_rng(6)
    x = _bf16_bits(rng.integers(-8, 9, size=(3, d)) / 8.0)
    y = oracle.expert_ffn(layer, 0, x, [0, 1, 2])
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    S = xf.sum(1)
    g, v = s_g * S, s_u * S
    h = g * expit(g) * v
    want = np.repeat((s_d * F * h)[:, None], d, axis=1)
    assert np.allclose(y, want, rtol=1e-12, atol=1e-12)


def test_ffn_closed_form_detects_gate_up_swap():
    """Planted mistake: gate and up exchanged changes the closed-form output."""
    d, F = 128, 64
    s_g, s_u, s_d = 2.0 ** -6, 2.0 ** -7, 2.0 ** -5
    good = oracle.Layer(d, 1, 1, F, _const_weights(F, d, s_g, s_u, s_d))
    bad = oracle.Layer(d, 1, 1, F, _const_weights(F, d, s_u, s_g, s_d))
    x = _bf16_bits(np.linspace(0.5, 2.0, d)[None])
    assert not np.allclose(oracle.expert_ffn(good, 0, x, [0]), oracle.expert_ffn(bad, 0, x, [0]), rtol=1e-3)


def test_silu_matches_library_on_random_weights():
    """One expert, numpy dense fp64 evaluation (dequant via bit slicing) on a tiny case."""
    rng = np.random.default_rng(7)
    d, F = 64, 128
    qg, qu, qd = rng.integers(0, 16, (F, d)), rng.integers(0, 16, (F, d)), rng.integers(0, 16, (d, F))
    sg, su, sd = (rng.integers(1, 64, (F, 1)) / 1024.0, rng.integers(1, 64, (F, 1)) / 1024.0,
                  rng.integers(1, 64, (d, F // 64)) / 1024.0)
    bg, bu, bd = -8 * sg, -8 * su, -8 * sd + 1.0 / 512
    wts = {"w_gate": _pack_rows(qg)[None], "s_gate": _bf16_bits(sg)[None], "b_gate": _bf16_bits(bg)[None],
           "w_up": _pack_rows(qu)[None], "s_up": _bf16_bits(su)[None], "b_up": _bf16_bits(bu)[None],
           "w_down": _pack_rows(qd)[None], "s_down": _bf16_bits(sd)[None], "b_down": _bf16_bits(bd)[None]}
    layer = oracle.Layer(d, 1, 1, F, wts)
    x = _bf16_bits(rng.normal(size=(2, d)).astype(np.float32).round(2))
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    Wg = sg * qg + bg
    Wu = su * qu + bu
    Wd = np.repeat(sd, 64, axis=1) * qd + np.repeat(bd, 64, axis=1)
    g, v = xf @ Wg.T, xf @ Wu.T
    want = (g * expit(g) * v) @ Wd.T
    got = oracle.expert_ffn(layer, 0, x, [0, 1])
    assert np.allclose(got, want, rtol=1e-11, atol=1e-11)


# ------------------------------------------------------------------ shared expert (column slices)
def _random_slices(P, F, d, seed, layout="separate"):
    """P random column slices of a shared expert (distinct nibbles, exact bf16 scales) and
    the dense fp64 matrices they stand for, built here by plain numpy stacking."""
    rng = np.random.default_rng(seed)
    qg, qu = rng.integers(0, 16, (P, F, d)), rng.integers(0, 16, (P, F, d))
    qd = rng.integers(0, 16, (P, d, F))
    sg, su = rng.integers(1, 64, (P, F, d // 64)) / 1024.0, rng.integers(1, 64, (P, F, d // 64)) / 1024.0
    sd = rng.integers(1, 64, (P, d, F // 64)) / 1024.0
    bg, bu, bd = -8 * sg + 1.0 / 256, -8 * su - 1.0 / 512, -8 * sd + 1.0 / 512
    w = {"w_down": np.stack([_pack_rows(q) for q in qd]), "s_down": _bf16_bits(sd), "b_down": _bf16_bits(bd)}
    g = (np.stack([_pack_rows(q) for q in qg]), _bf16_bits(sg), _bf16_bits(bg))
    u = (np.stack([_pack_rows(q) for q in qu]), _bf16_bits(su), _bf16_bits(bu))
    if layout == "separate":
        w.update(w_gate=g[0], s_gate=g[1], b_gate=g[2], w_up=u[0], s_up=u[1], b_up=u[2])
    else:
        w.update(w_gate_up=np.concatenate([g[0], u[0]], 1), s_gate_up=np.concatenate([g[1], u[1]], 1),
                 b_gate_up=np.concatenate([g[2], u[2]], 1))
    deq = lambda q, s, b: np.repeat(s, 64, axis=-1) * q + np.repeat(b, 64, axis=-1)
    Wg = np.concatenate(list(deq(qg, sg, bg)), axis=0)      # [P F, d]: slice p = rows pF..
    Wu = np.concatenate(list(deq(qu, su, bu)), axis=0)
    Wd = np.concatenate(list(deq(qd, sd, bd)), axis=1)      # [d, P F]: slice p = columns pF..
    return w, (Wg, Wu, Wd)


@pytest.mark.parametrize("layout", ["separate", "fused"])
def test_shared_dense_matches_numpy(layout):
    """The reassembled shared expert equals a numpy dense SwiGLU of the stacked slices."""
    P, F, d = 3, 64, 128
    w, (Wg, Wu, Wd) = _random_slices(P, F, d, 21, layout)
    dense = oracle.shared_dense_layer(w, d, P, F, layout)
    rng = np.random.default_rng(22)
    x = _bf16_bits(rng.normal(size=(4, d)).astype(np.float32).round(2))
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    g, v = xf @ Wg.T, xf @ Wu.T
    want = (g * expit(g) * v) @ Wd.T
    assert np.allclose(oracle.shared_expert_ffn(dense, x), want, rtol=1e-11, atol=1e-11)


def test_shared_equals_weight_one_route_over_slices():
    """SwiGLU acts column by column: the sum of the slices' outputs (each slice an expert of
    the sliced layer, every token routed to all P with weight 1) is the dense expert."""
    P, F, d = 4, 64, 128
    w, _ = _random_slices(P, F, d, 23)
    dense = oracle.shared_dense_layer(w, d, P, F)
    sliced = oracle.Layer(d, P, P, F, w, "separate", 0)
    rng = np.random.default_rng(24)
    x = _bf16_bits(rng.normal(size=(5, d)).astype(np.float32).round(2))
    res = rng.normal(size=(5, d)).astype(np.float32)
    idx = np.tile(np.arange(P, dtype=np.int32), (5, 1))
    _, out64, _ = oracle.moe_layer(sliced, x, idx, np.ones((5, P)), res)
    assert np.allclose(out64 - res, oracle.shared_expert_ffn(dense, x), rtol=1e-11, atol=1e-11)
    # a planted mistake: slices stacked in the wrong order give another expert
    swapped = {k: (v[::-1].copy() if k.endswith("_down") else v) for k, v in w.items()}
    bad = oracle.shared_dense_layer(swapped, d, P, F)
    assert not np.allclose(oracle.shared_expert_ffn(bad, x), oracle.shared_expert_ffn(dense, x), rtol=1e-3)


# ------------------------------------------------------------------ whole layer
def _toy_case(w=None, layout=None, tokens=None):
    w = w or W.WORKLOADS["toy"]
    B = tokens or w.tokens
    x = W.gen_x(w, 0, B)
    wts = W.gen_layer_weights(w, 0, layout=layout)
    layer = oracle.Layer.from_workload(w, wts, layout)
    idx, w64, w32, _ = oracle.route(x, W.gen_gate(w, 0), None, w.top_k, w.norm_topk_prob)
    res = x.float()
    return w, x, layer, idx, w64, res


def test_token_major_equals_layer_major():
    """Layer-Major Batched Prefill, 'Measured Result': both evaluation orders agree exactly."""
    w, x, layer, idx, w64, res = _toy_case()
    a, a64, ya = oracle.moe_layer(layer, x, idx, w64, res, "layer", want_slots=True)
    b, b64, yb = oracle.moe_layer(layer, x, idx, w64, res, "token", want_slots=True)
    assert np.array_equal(a64, b64) and np.array_equal(ya, yb) and np.array_equal(a, b)


def test_layer_major_equals_bruteforce_dense_numpy():
    """Tiny layer: a dense numpy fp64 evaluation (every token x every routed expert)."""
    w = W.scaled(W.WORKLOADS["toy"], d_model=128, num_experts=6, top_k=2, ffn_dim=64, tokens=5)
    x = W.gen_x(w, 0, 5)
    wts = W.gen_layer_weights(w, 0)
    layer = oracle.Layer.from_workload(w, wts)
    idx, w64, _, _ = oracle.route(x, W.gen_gate(w, 0), None, 2, 1)
    res = np.random.default_rng(8).normal(size=(5, 128)).astype(np.float32)
    out, out64, _ = oracle.moe_layer(layer, x, idx, w64, res, "layer")

    def deq(name, e):
        q = wts["w_" + name][e].numpy().view(np.uint32)
        nib = (q[..., None] >> (4 * np.arange(8, dtype=np.uint32))) & 15
        nib = nib.reshape(q.shape[0], -1).astype(np.float64)
        s = wts["s_" + name][e].float().numpy().astype(np.float64)
        b = wts["b_" + name][e].float().numpy().astype(np.float64)
        return np.repeat(s, 64, 1) * nib + np.repeat(b, 64, 1)

    xf = x.float().numpy().astype(np.float64)
    want = res.astype(np.float64).copy()
    for t in range(5):
        for k in range(2):
            e = idx[t, k]
            g, v = deq("gate", e) @ xf[t], deq("up", e) @ xf[t]
            want[t] += w64[t, k] * (deq("down", e) @ (g * expit(g) * v))
    assert np.allclose(out64, want, rtol=1e-12, atol=1e-10)


def test_fused_layout_equals_separate():
    """Math Contract: gate rows on top, up rows below gives the identical result."""
    w, x, lsep, idx, w64, res = _toy_case(layout="separate")
    lfus = oracle.Layer.from_workload(w, W.gen_layer_weights(w, 0, layout="fused"), "fused")
    a = oracle.moe_layer(lsep, x, idx, w64, res)[1]
    b = oracle.moe_layer(lfus, x, idx, w64, res)[1]
    assert np.array_equal(a, b)


def test_swapped_gate_up_is_far_off():
    """Negative control from 'Math Contract': a gate/up reorder moves the result by ~100% rel-L2."""
    w, x, lsep, idx, w64, res = _toy_case(layout="separate")
    wf = W.gen_layer_weights(w, 0, layout="fused")
    F = w.ffn_dim
    swapped = {k: (torch.cat([v[:, F:], v[:, :F]], 1) if k.endswith("gate_up") else v) for k, v in wf.items()}
    lbad = oracle.Layer.from_workload(w, swapped, "fused")
    good = oracle.moe_layer(lsep, x, idx, w64, res)[1] - res.numpy()
    bad = oracle.moe_layer(lbad, x, idx, w64, res)[1] - res.numpy()
    rel = np.linalg.norm(bad - good) / np.linalg.norm(good)
    assert rel > 0.5


def test_k1_output_is_residual_plus_top_expert():
    w = W.scaled(W.WORKLOADS["toy"], top_k=1)
    x = W.gen_x(w, 0, 4)
    layer = oracle.Layer.from_workload(w, W.gen_layer_weights(w, 0))
    idx, w64, _, _ = oracle.route(x, W.gen_gate(w, 0), None, 1, 1)
    assert np.all(w64 == 1.0)
    res = x.float()
    out, out64, _ = oracle.moe_layer(layer, x, idx, w64, res)
    for t in range(4):
        y = oracle.expert_ffn(layer, int(idx[t, 0]), x, [t])[0]
        assert np.array_equal(out64[t], res[t].numpy().astype(np.float64) + y)


def test_identical_tokens_union_is_k_experts():
    w = W.WORKLOADS["toy"]
    x = W.gen_x(w, 0, 1).repeat(6, 1)
    idx, w64, _, _ = oracle.route(x, W.gen_gate(w, 0), None, w.top_k, 1)
    uid, off, tl, sl = oracle.expert_union(idx, w.num_experts)
    assert len(uid) == w.top_k and np.all(np.diff(off) == 6)
    layer = oracle.Layer.from_workload(w, W.gen_layer_weights(w, 0))
    out = oracle.moe_layer(layer, x, idx, w64, x.float())[1]
    assert np.all(out == out[0])


def test_unrouted_expert_never_in_union():
    idx = np.array([[0, 3], [3, 5]], np.int32)
    uid, off, _, _ = oracle.expert_union(idx, 8)
    assert uid.tolist() == [0, 3, 5] and off.tolist() == [0, 1, 3, 4]


def test_rmsnorm_closed_forms():
    h = np.array([[3.0, -3.0, 3.0, -3.0], [2.0, 0.0, 0.0, 0.0], [1e-3, 1e-3, 1e-3, 1e-3]], np.float32)
    x = oracle.rmsnorm_bf16(h, 1e-6)
    assert x[0].tolist() == [0x3F80, 0xBF80, 0x3F80, 0xBF80]        # +-1
    assert x[1].tolist() == [0x4000, 0, 0, 0]                        # 2.0
    # eps matters at small scale: 1e-3 / sqrt(1e-6 + 1e-6) = 1/sqrt(2) -> bf16 0x3F35
    assert x[2].tolist() == [0x3F35] * 4


def test_centred_rmsnorm_closed_form():
    """Centring removes the row mean first: [5,3,5,3] -> [1,-1,1,-1]; [2,2,2,10] -> mean 4,
    deviations [-2,-2,-2,6], RMS sqrt(12): -1/sqrt(3) = -0.57735 lies between the bf16 values
    -0.57421875 (0xBF13) and -0.578125 (0xBF14), nearer the latter; sqrt(3) = 1.73205 between
    1.7265625 (0x3FDD) and 1.734375 (0x3FDE), nearer the latter."""
    h = np.array([[5.0, 3.0, 5.0, 3.0], [2.0, 2.0, 2.0, 10.0]], np.float32)
    x = oracle.rmsnorm_bf16(h, 1e-9, center=True)
    assert x[0].tolist() == [0x3F80, 0xBF80, 0x3F80, 0xBF80]
    assert x[1].tolist() == [0xBF14, 0xBF14, 0xBF14, 0x3FDE]
    # without centring the same rows keep their offset
    assert oracle.rmsnorm_bf16(h, 1e-9)[0].tolist() != x[0].tolist()


def test_oracle_row_subset_matches_full():
    w, x, layer, idx, w64, res = _toy_case()
    full = oracle.moe_layer(layer, x, idx, w64, res)[1]
    part = oracle.moe_layer(layer, x, idx, w64, res, rows=[3, 7, 11])[1]
    assert np.array_equal(part[[3, 7, 11]], full[[3, 7, 11]])


# ----------------------------------------------------------------------------- slot pool
def _slot_pool_case():
    fx = json.load(open(os.path.join(GOLDEN, "slot_pool_handworked.json")))
    return fx["n_keys"], fx["n_slots"], [(c["keys"], c["slots"], [tuple(p) for p in c["copies"]]) for c in fx["calls"]]


def test_slot_pool_hand_worked():
    n_keys, n_slots, calls = _slot_pool_case()
    pool = oracle.SlotPool(n_keys=n_keys, n_slots=n_slots)
    for keys, slots, copies in calls:
        got_s, got_c = pool.plan(keys)
        assert got_s == slots and got_c == copies, (keys, got_s, got_c)


def test_slot_pool_keys_of_different_layers_are_distinct():
    E = 4
    pool = oracle.SlotPool(n_keys=2 * E, n_slots=2)
    assert pool.plan([1]) == ([0], [(1, 0)])              # layer 0, expert 1
    assert pool.plan([E + 1]) == ([1], [(E + 1, 1)])      # layer 1, expert 1: its own slot
    assert pool.plan([1, 2]) == ([0, 1], [(2, 1)])        # layer 0 again: hit, and 2 evicts (1, 1)


def test_slot_pool_planted_mru_eviction_fails_the_pin():
    class MostRecent(oracle.SlotPool):   # a plausible mistake: evict the newest idle slot
        def plan(self, keys):
            saved = self.stamp
            self.stamp = [-s if s >= 0 else -(10 ** 9) for s in saved]
            try:
                return super().plan(keys)
            finally:
                fresh = self.stamp
                self.stamp = [self.tick if f == self.tick else saved[i] for i, f in enumerate(fresh)]

    n_keys, n_slots, calls = _slot_pool_case()
    pool = MostRecent(n_keys=n_keys, n_slots=n_slots)
    results = [pool.plan(keys) for keys, _, _ in calls]
    assert results != [(s, c) for _, s, c in calls]


def test_slot_pool_retains_a_cycle_that_fits():
    # unions over 6 distinct keys, pool of 6: after the first pass nothing is copied again
    cycle = [[0, 2, 4], [1, 2, 3], [4, 5], [0, 5]]
    pool = oracle.SlotPool(n_keys=16, n_slots=6)
    first = sum(len(pool.plan(u)[1]) for u in cycle)
    assert first == 6
    for _ in range(3):
        assert sum(len(pool.plan(u)[1]) for u in cycle) == 0


def test_slot_pool_invariants_random():
    rng = np.random.default_rng(11)
    n_keys, n_slots = 40, 12
    pool = oracle.SlotPool(n_keys, n_slots)
    for step in range(300):
        keys = sorted(rng.choice(n_keys, size=int(rng.integers(1, 9)), replace=False).tolist())
        before_owner, before_stamp = list(pool.owner), list(pool.stamp)
        resident_before = {k for k in before_owner if k >= 0}
        slots, copies = pool.plan(keys)
        # every key of the union is resident in the slot returned for it
        assert all(pool.owner[s] == k and pool.slot_of[k] == s for k, s in zip(keys, slots))
        assert len(set(slots)) == len(slots)
        # copies are exactly the keys not resident before, in union order
        assert [k for k, _ in copies] == [k for k in keys if k not in resident_before]
        # the slots taken are the (stamp, id)-smallest of the slots no hit used
        hit_slots = {before_owner.index(k) for k in keys if k in resident_before}
        idle = sorted((before_stamp[s], s) for s in range(n_slots) if s not in hit_slots)
        assert [s for _, s in copies] == [s for _, s in idle[:len(copies)]]
        # residency table and slot owners agree
        assert sum(1 for k in range(n_keys) if pool.slot_of[k] >= 0) == sum(1 for o in pool.owner if o >= 0)
        assert all(pool.stamp[s] == pool.tick for s in slots)
