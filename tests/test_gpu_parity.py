"""Parity of the CUDA path (through the C ABI) with the CPU oracle, on seeded workloads.

Routing indices, the union and the token lists must match bit-exactly (layer-0 inputs are
drawn with a logit gap >= 1e-3 between adjacent ranks 1..K+1); routing weights to 1e-5
relative; layer outputs to relative L2 <= 5e-3 (on the layer delta and on the output) and
max-abs <= 2e-2 (absolute, at every layer).  Chained stacks are checked layer by layer,
teacher-forced (the oracle's layer l consumes the GPU's own hidden state h_l), and end to end
(each side runs its own chain; tokens whose routing flips at some layer are counted).  In the
teacher-forced check, tokens whose oracle gap between ranks K and K+1 is below 1e-4 are exempt
from the index comparison, and so are tokens with the same expert set whose ranks swapped on
oracle logits that tie within 1e-4; both together must stay under 0.1% of the token-layers.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import MAX_ABS_TOL, REL_L2_TOL, W_RTOL, logit_gaps, max_abs, rel_l2, resampled_x, rmsnorm_glue_close
from moe_expert_routing_gb300 import smoe
from moe_expert_routing_gb300 import workload as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


class Case:
    """One layer of a workload: inputs on the host (oracle) and on the device (CUDA path)."""

    def __init__(self, w: W.Workload, layer: int = 0, B: int = None, gap: bool = True, x=None, gen_device=None):
        _need_gpu()
        self.w, self.layer = w, layer
        self.B = B if B is not None else w.tokens
        self.gate = W.gen_gate(w, layer)
        self.bias = W.gen_gate_bias(w, layer)
        if x is not None:
            self.x = x
        elif gap:
            self.x, _ = resampled_x(w, layer, self.B, self.gate, self.bias)
        else:
            self.x = W.gen_x(w, layer, self.B)
        big = w.num_experts * w.expert_bytes > (256 << 20)
        gdev = gen_device or (DEV if big else "cpu")
        wts = W.gen_layer_weights(w, layer, device=gdev)
        self.wts_cpu = {k: v.cpu() for k, v in wts.items()}
        self.wts_gpu = {k: v.to(DEV) for k, v in wts.items()}
        self.weights = smoe.Weights(self.wts_gpu)
        self.desc = smoe.make_desc(w.d_model, w.num_experts, w.top_k, w.ffn_dim, w.layout, w.norm_topk_prob)
        self.layer_o = oracle.Layer.from_workload(w, self.wts_cpu)
        self.ws = smoe.alloc_workspace(self.desc, max(self.B, 1))
        self.gate_d = self.gate.to(DEV)
        self.bias_d = None if self.bias is None else self.bias.to(DEV)

    def x_dev(self):
        return self.x.to(DEV).view(torch.int16)

    def run_layer(self, residual=None):
        """Full smoe_moe_layer on the device: (out fp32 [B,d], idx, w)."""
        B, K = self.B, self.w.top_k
        res = (self.x.float() if residual is None else residual).to(DEV).contiguous()
        idx = torch.empty(B, K, dtype=torch.int32, device=DEV)
        wt = torch.empty(B, K, dtype=torch.float32, device=DEV)
        smoe.smoe_clear_device_status(self.ws)
        smoe.smoe_moe_layer(self.desc, self.weights, self.x_dev(), self.gate_d, self.bias_d, res, self.ws, idx, wt)
        bits = smoe.smoe_read_device_status(self.ws)
        assert bits == 0, f"device status {bits:#x}"
        return res.cpu(), idx.cpu(), wt.cpu()

    def oracle_layer(self, residual=None, rows=None):
        idx, w64, w32, lg = oracle.route(self.x, self.gate, self.bias, self.w.top_k, self.w.norm_topk_prob)
        res = self.x.float() if residual is None else residual
        out, out64, _ = oracle.moe_layer(self.layer_o, self.x, idx, w64, res, rows=rows)
        return out64, idx, w64, lg


def check_outputs(gpu_out, oracle_out64, residual, rows=None):
    """rel-L2 <= 5e-3 on the delta and the output; max-abs <= 2e-2 (absolute)."""
    g = np.asarray(gpu_out, np.float64)
    o = np.asarray(oracle_out64, np.float64)
    r = np.asarray(residual, np.float64)
    if rows is not None:
        g, o, r = g[rows], o[rows], r[rows]
    assert np.all(np.isfinite(g))
    d_rel = rel_l2(g - r, o - r)
    o_rel = rel_l2(g, o)
    mab = max_abs(g, o)
    assert d_rel <= REL_L2_TOL, f"delta rel-L2 {d_rel:.3e}"
    assert o_rel <= REL_L2_TOL, f"output rel-L2 {o_rel:.3e}"
    assert mab <= MAX_ABS_TOL, f"max-abs {mab:.3e}"
    return d_rel, mab


# ----------------------------------------------------------------------------- routing
ROUTE_CASES = [
    ("toy", None), ("decode_b1", None), ("decode_b8", None), ("prefill64", None), ("q35_prefill64", None),
    ("long4096", 1024),
]


@pytest.mark.parametrize("name,B", ROUTE_CASES)
def test_route_parity(name, B):
    _need_gpu()
    w = W.WORKLOADS[name]
    B = B or w.tokens
    gate = W.gen_gate(w, 0)
    bias = W.gen_gate_bias(w, 0)
    x, _ = resampled_x(w, 0, B, gate, bias)
    desc = smoe.make_desc(w.d_model, w.num_experts, w.top_k, w.ffn_dim, w.layout, w.norm_topk_prob)
    ws = smoe.alloc_workspace(desc, B)
    idx = torch.empty(B, w.top_k, dtype=torch.int32, device=DEV)
    wt = torch.empty(B, w.top_k, dtype=torch.float32, device=DEV)
    smoe.smoe_route(desc, x.to(DEV).view(torch.int16), gate.to(DEV), None if bias is None else bias.to(DEV), idx, wt, ws)
    torch.cuda.synchronize()
    oi, ow64, _, _ = oracle.route(x, gate, bias, w.top_k, w.norm_topk_prob)
    assert np.array_equal(idx.cpu().numpy(), oi)
    np.testing.assert_allclose(wt.cpu().numpy(), ow64, rtol=W_RTOL, atol=1e-7)


def test_route_norm_topk_prob_off_and_k_equals_e():
    _need_gpu()
    w = W.scaled(W.WORKLOADS["toy"], norm_topk_prob=0)
    for K in (4, 16):
        wk = W.scaled(w, top_k=K)
        gate = W.gen_gate(wk, 0)
        x, _ = resampled_x(wk, 0, 16, gate, None)
        desc = smoe.make_desc(wk.d_model, wk.num_experts, K, wk.ffn_dim, "separate", 0)
        ws = smoe.alloc_workspace(desc, 16)
        idx = torch.empty(16, K, dtype=torch.int32, device=DEV)
        wt = torch.empty(16, K, dtype=torch.float32, device=DEV)
        smoe.smoe_route(desc, x.to(DEV).view(torch.int16), gate.to(DEV), None, idx, wt, ws)
        oi, ow64, _, _ = oracle.route(x, gate, None, K, 0)
        assert np.array_equal(idx.cpu().numpy(), oi)
        np.testing.assert_allclose(wt.cpu().numpy(), ow64, rtol=W_RTOL, atol=1e-7)


@pytest.mark.parametrize("name,B,n_spec,norm", [("decode_b1", 1, 8, 1), ("decode_b8", 8, 8, 1),
                                                 ("prefill64", 64, 24, 1), ("toy", 16, 12, 0), ("long4096", 512, 8, 1)])
def test_route_ranked_parity(name, B, n_spec, norm):
    """Ranked continuation: the routing equals smoe_route's bit for bit; the ranks K..K+N-1
    match the oracle exactly (inputs drawn with separated logits over ranks 1..K+N+1) and
    their full-softmax probabilities to 1e-5."""
    _need_gpu()
    w = W.scaled(W.WORKLOADS[name], norm_topk_prob=norm)
    K = w.top_k
    gate = W.gen_gate(w, 0)
    bias = W.gen_gate_bias(w, 0)
    x, _ = resampled_x(W.scaled(w, top_k=K + n_spec), 0, B, gate, bias)
    desc = smoe.make_desc(w.d_model, w.num_experts, K, w.ffn_dim, w.layout, norm)
    ws = smoe.alloc_workspace(desc, B)
    xd, gd, bd = x.to(DEV).view(torch.int16), gate.to(DEV), None if bias is None else bias.to(DEV)
    idx0 = torch.empty(B, K, dtype=torch.int32, device=DEV)
    wt0 = torch.empty(B, K, dtype=torch.float32, device=DEV)
    smoe.smoe_route(desc, xd, gd, bd, idx0, wt0, ws)
    idx = torch.empty(B, K, dtype=torch.int32, device=DEV)
    wt = torch.empty(B, K, dtype=torch.float32, device=DEV)
    sidx = torch.empty(B, n_spec, dtype=torch.int32, device=DEV)
    sp = torch.empty(B, n_spec, dtype=torch.float32, device=DEV)
    smoe.smoe_route_ranked(desc, xd, gd, bd, idx, wt, sidx, sp, ws)
    sidx2 = torch.empty(B, n_spec, dtype=torch.int32, device=DEV)
    smoe.smoe_route_ranked(desc, xd, gd, bd, idx, wt, sidx2, None, ws)   # probabilities not wanted
    torch.cuda.synchronize()
    assert torch.equal(idx, idx0) and torch.equal(wt, wt0)
    assert torch.equal(sidx, sidx2)
    oi, ow64, osi, osp, _ = oracle.route_ranked(x, gate, bias, K, n_spec, norm)
    assert np.array_equal(idx.cpu().numpy(), oi)
    np.testing.assert_allclose(wt.cpu().numpy(), ow64, rtol=W_RTOL, atol=1e-7)
    assert np.array_equal(sidx.cpu().numpy(), osi)
    np.testing.assert_allclose(sp.cpu().numpy(), osp, rtol=W_RTOL, atol=1e-9)


def test_routing_stats_of_a_correlated_sequence():
    """Next-token coverage on a correlated decode sequence routed by the GPU equals the same
    statistics of the oracle's routing (Qwen3-235B-shaped router, top-8 plus 8 ranks)."""
    _need_gpu()
    from moe_expert_routing_gb300 import routing_stats as RS
    w = W.WORKLOADS["decode_b1"]
    T, N = 128, 8
    gate = W.gen_gate(w, 0)
    x = W.gen_x_sequence(w, 0, T, 0.9)
    desc = smoe.make_desc(w.d_model, w.num_experts, w.top_k, w.ffn_dim, w.layout, w.norm_topk_prob)
    ws = smoe.alloc_workspace(desc, T)
    idx = torch.empty(T, w.top_k, dtype=torch.int32, device=DEV)
    wt = torch.empty(T, w.top_k, dtype=torch.float32, device=DEV)
    sidx = torch.empty(T, N, dtype=torch.int32, device=DEV)
    smoe.smoe_route_ranked(desc, x.to(DEV).view(torch.int16), gate.to(DEV), None, idx, wt, sidx, None, ws)
    oi, _, osi, _, lg = oracle.route_ranked(x, gate, None, w.top_k, N, w.norm_topk_prob)
    sure = logit_gaps(lg, w.top_k + N) >= 1e-4          # no near-tie among ranks 1..K+N+1
    assert sure.mean() > 0.9
    gi, gs = idx.cpu().numpy(), sidx.cpu().numpy()
    assert np.array_equal(gi[sure], oi[sure]) and np.array_equal(gs[sure], osi[sure])
    if sure.all():
        assert RS.sequence_stats(gi, gs) == RS.sequence_stats(oi, osi)
    st = RS.sequence_stats(gi, gs)
    assert 0.0 < st["adjacent_reuse"] <= st["ranked_coverage"] <= 1.0


# ----------------------------------------------------------------------------- union
@pytest.mark.parametrize("B,K,E", [(1, 8, 128), (16, 4, 16), (64, 8, 128), (64, 8, 256), (37, 3, 9), (4096, 8, 128),
                                   (200, 16, 16), (1, 1, 1), (3, 5, 200), (8, 8, 256), (16, 8, 128), (33, 4, 256)])
def test_union_parity(B, K, E):
    _need_gpu()
    rng = np.random.default_rng(B * 1000 + K * 10 + E)
    # skewed: a few hot experts plus uniform picks
    p = rng.zipf(1.3, size=E).astype(np.float64)
    p /= p.sum()
    idx = np.stack([rng.choice(E, K, replace=False, p=p) for _ in range(B)]).astype(np.int32)
    d = max(256, 256)
    desc = smoe.make_desc(d, E, K, 256)
    ws = smoe.alloc_workspace(desc, B)
    uid = torch.full((E,), -7, dtype=torch.int32, device=DEV)
    nu = torch.zeros(1, dtype=torch.int32, device=DEV)
    off = torch.full((E + 1,), -7, dtype=torch.int32, device=DEV)
    tl = torch.full((B * K,), -7, dtype=torch.int32, device=DEV)
    sl = torch.full((B * K,), -7, dtype=torch.int32, device=DEV)
    smoe.smoe_expert_union(desc, torch.from_numpy(idx).to(DEV), uid, nu, off, tl, sl, ws)
    ou, oo, otl, osl = oracle.expert_union(idx, E)
    n = int(nu.item())
    assert n == len(ou)
    assert np.array_equal(uid.cpu().numpy()[:n], ou)
    assert np.array_equal(off.cpu().numpy()[:n + 1], oo)
    assert np.array_equal(tl.cpu().numpy(), otl)
    assert np.array_equal(sl.cpu().numpy(), osl)


def test_union_bad_index_sets_fault_and_leaves_residual():
    _need_gpu()
    c = Case(W.WORKLOADS["toy"], gap=False)
    B, K = c.B, c.w.top_k
    idx = np.tile(np.arange(K, dtype=np.int32), (B, 1))
    idx[3, 1] = c.w.num_experts + 5
    idx_d = torch.from_numpy(idx).to(DEV)
    E = c.w.num_experts
    uid = torch.zeros(E, dtype=torch.int32, device=DEV)
    nu = torch.zeros(1, dtype=torch.int32, device=DEV)
    off = torch.zeros(E + 1, dtype=torch.int32, device=DEV)
    tl = torch.zeros(B * K, dtype=torch.int32, device=DEV)
    sl = torch.zeros(B * K, dtype=torch.int32, device=DEV)
    smoe.smoe_clear_device_status(c.ws)
    smoe.smoe_expert_union(c.desc, idx_d, uid, nu, off, tl, sl, c.ws)
    res = c.x.float().to(DEV)
    before = res.clone()
    wt = torch.full((B, K), 0.25, device=DEV)
    smoe.smoe_moe_ffn_batch(c.desc, c.weights, c.x_dev(), uid, nu, off, tl, sl, wt, res, c.ws)
    bits = smoe.smoe_read_device_status(c.ws)
    assert bits & smoe.SMOE_FAULT_EXPERT_INDEX
    assert int(nu.item()) == 0
    assert torch.equal(res, before)
    smoe.smoe_clear_device_status(c.ws)
    assert smoe.smoe_read_device_status(c.ws) == 0


def _routed_lists(c, x_dev):
    """Route and build the union of case c for the given device input; returns the buffers."""
    B, K, E = c.B, c.w.top_k, c.w.num_experts
    idx = torch.empty(B, K, dtype=torch.int32, device=DEV)
    wt = torch.empty(B, K, dtype=torch.float32, device=DEV)
    smoe.smoe_route(c.desc, x_dev, c.gate_d, c.bias_d, idx, wt, c.ws)
    uid = torch.zeros(E, dtype=torch.int32, device=DEV)
    nu = torch.zeros(1, dtype=torch.int32, device=DEV)
    off = torch.zeros(E + 1, dtype=torch.int32, device=DEV)
    tl = torch.zeros(B * K, dtype=torch.int32, device=DEV)
    sl = torch.zeros(B * K, dtype=torch.int32, device=DEV)
    smoe.smoe_expert_union(c.desc, idx, uid, nu, off, tl, sl, c.ws)
    return wt, uid, nu, off, tl, sl


@pytest.mark.parametrize("value", [-600.0, 70000.0])
def test_fp16_range_fault_bit(value):
    """Hidden states far outside the workloads' N(0, 1) scale, made on the host: at x = -600
    the SwiGLU activations reach ~1e6 (the synthetic weights have mean -0.5 scale, so gate
    and up both grow like 3 |x| per row) and do not fit fp16; x = 70000 does not fit fp16
    itself.  The FFN sets SMOE_FAULT_FP16_RANGE and returns; nothing hangs."""
    c = Case(W.WORKLOADS["toy"], gap=False)
    x = torch.full((c.B, c.w.d_model), value, dtype=torch.bfloat16)
    xd = x.to(DEV).view(torch.int16)
    smoe.smoe_clear_device_status(c.ws)
    wt, uid, nu, off, tl, sl = _routed_lists(c, xd)
    res = x.float().to(DEV)
    smoe.smoe_moe_ffn_batch(c.desc, c.weights, xd, uid, nu, off, tl, sl, wt, res, c.ws)
    bits = smoe.smoe_read_device_status(c.ws)
    assert bits & smoe.SMOE_FAULT_FP16_RANGE, f"status {bits:#x}"
    assert not bits & smoe.SMOE_FAULT_TIMEOUT
    smoe.smoe_clear_device_status(c.ws)
    assert smoe.smoe_read_device_status(c.ws) == 0


@pytest.mark.parametrize("which", ["token", "slot"])
def test_token_index_fault_bit(which):
    """A caller-built list with a token entry outside [0, B) or a slot entry outside [0, K):
    the FFN sets SMOE_FAULT_TOKEN_INDEX, drops that entry's output (reading row 0 in place of
    a bad token) and returns; nothing hangs."""
    c = Case(W.WORKLOADS["toy"], gap=False)
    xd = c.x_dev()
    smoe.smoe_clear_device_status(c.ws)
    wt, uid, nu, off, tl, sl = _routed_lists(c, xd)
    if which == "token":
        tl[5] = c.B + 3
    else:
        sl[5] = c.w.top_k
    res = c.x.float().to(DEV)
    smoe.smoe_moe_ffn_batch(c.desc, c.weights, xd, uid, nu, off, tl, sl, wt, res, c.ws)
    bits = smoe.smoe_read_device_status(c.ws)
    assert bits & smoe.SMOE_FAULT_TOKEN_INDEX, f"status {bits:#x}"
    assert not bits & smoe.SMOE_FAULT_TIMEOUT


# ----------------------------------------------------------------------------- whole layer
LAYER_CASES = [
    ("toy", None), ("decode_b1", None), ("decode_b8", None), ("prefill64", None), ("q35_prefill64", None),
    ("prefill64", 37), ("toy", 1), ("q35_prefill64", 5),
]


@pytest.mark.parametrize("name,B", LAYER_CASES)
def test_layer_parity(name, B):
    c = Case(W.WORKLOADS[name], B=B)
    out, idx, wt = c.run_layer()
    o64, oidx, ow64, _ = c.oracle_layer()
    assert np.array_equal(idx.numpy(), oidx)
    np.testing.assert_allclose(wt.numpy(), ow64, rtol=W_RTOL, atol=1e-7)
    check_outputs(out.numpy(), o64, c.x.float().numpy())


def test_ffn_batch_step_by_step_matches_layer():
    """route -> union -> ffn_batch through the separate entry points equals smoe_moe_layer."""
    c = Case(W.WORKLOADS["decode_b8"])
    B, K, E = c.B, c.w.top_k, c.w.num_experts
    idx = torch.empty(B, K, dtype=torch.int32, device=DEV)
    wt = torch.empty(B, K, dtype=torch.float32, device=DEV)
    smoe.smoe_route(c.desc, c.x_dev(), c.gate_d, None, idx, wt, c.ws)
    uid = torch.zeros(E, dtype=torch.int32, device=DEV)
    nu = torch.zeros(1, dtype=torch.int32, device=DEV)
    off = torch.zeros(E + 1, dtype=torch.int32, device=DEV)
    tl = torch.zeros(B * K, dtype=torch.int32, device=DEV)
    sl = torch.zeros(B * K, dtype=torch.int32, device=DEV)
    smoe.smoe_expert_union(c.desc, idx, uid, nu, off, tl, sl, c.ws)
    res = c.x.float().to(DEV)
    smoe.smoe_moe_ffn_batch(c.desc, c.weights, c.x_dev(), uid, nu, off, tl, sl, wt, res, c.ws)
    out_layer, _, _ = c.run_layer()
    assert torch.equal(res.cpu(), out_layer)


@pytest.mark.parametrize("name,B,d,center,alias", [("toy", 16, None, 1, False), ("prefill64", 64, None, 1, True),
                                                   ("q35_prefill64", 37, None, 0, True), ("toy", 5, 8192, 1, False),
                                                   ("toy512", 512, None, 1, True), ("toy512", 384, None, 0, False)])
def test_ffn_batch_norm_equals_ffn_then_norm(name, B, d, center, alias):
    """smoe_moe_ffn_batch_norm gives smoe_moe_ffn_batch's residual and smoe_rmsnorm_bf16's
    next-block input bit for bit (the combine + norm kernel for d_model <= 4096, the standalone
    norm after the combine beyond; also with hot experts on the tensor-core path at B >= 256),
    also when x_next is the input buffer x itself."""
    if name == "toy512":   # d, ffn_dim multiples of 512: hot experts on the tensor-core path
        w = W.scaled(W.WORKLOADS["toy"], ffn_dim=512, tokens=B, num_experts=32, zipf_s=1.1)
    else:
        w = W.WORKLOADS[name] if d is None else W.scaled(W.WORKLOADS[name], d_model=d)
    c = Case(w, B=B)
    xd = c.x_dev()
    wt, uid, nu, off, tl, sl = _routed_lists(c, xd)
    smoe.smoe_clear_device_status(c.ws)
    res_a = c.x.float().to(DEV) * 3.0
    res_b = res_a.clone()
    smoe.smoe_moe_ffn_batch(c.desc, c.weights, xd, uid, nu, off, tl, sl, wt, res_a, c.ws)
    xn_a = torch.empty_like(xd)
    smoe.smoe_rmsnorm_bf16(res_a, xn_a, 1e-6, center=center)
    x_in = xd.clone()
    xn_b = x_in if alias else torch.full_like(xd, -1)
    smoe.smoe_moe_ffn_batch_norm(c.desc, c.weights, x_in, uid, nu, off, tl, sl, wt, res_b, xn_b, c.ws, 1e-6, center)
    assert smoe.smoe_read_device_status(c.ws) == 0
    assert torch.equal(res_a, res_b)
    assert torch.equal(xn_a, xn_b)


@pytest.mark.parametrize("B,same", [(12, [(0, 8), (8, 12)]), (16, [(0, 16)]), (64, [(0, 64)])])
def test_hot_experts_many_tokens_per_expert(B, same):
    """B identical tokens: K experts with B tokens each, so every expert runs several token
    chunks: at B = 12 and 16 (B K <= 4 E) the down pass takes chunks of 8 (8 + 4 and 8 + 8), at
    B = 64 chunks of 16 (gate/up always takes chunks of 16).  Tokens that share a chunk shape
    get the same output bit for bit; a down chunk of at most 4 tokens packs the hi and lo terms
    of h into one n-tile, which sums them in another order, so at B = 12 tokens 8-11 agree with
    the oracle as closely as tokens 0-7 but not bit for bit with them."""
    w = W.WORKLOADS["toy"]
    x1 = W.gen_x(w, 0, 1)
    c = Case(w, B=B, x=x1.repeat(B, 1))
    out, idx, _ = c.run_layer()
    o64, oidx, _, _ = c.oracle_layer()
    assert np.array_equal(idx.numpy(), oidx)
    check_outputs(out.numpy(), o64, c.x.float().numpy())
    for a, b in same:
        assert torch.all(out[a:b] == out[a])


@pytest.mark.parametrize("layout,d", [("separate", 512), ("fused", 512), ("separate", 256)])
def test_wide_gate_up_tiles(layout, d):
    """ffn_dim 1536 (a multiple of 192) over 64 experts with 64 tokens: 8 gate/up tiles of 192 h
    columns per expert and more than two waves of them, so the gate/up pass runs with 12
    consumer warps; both weight layouts (separate tensors, fused gate_up with gate rows on top),
    and d_model 256, whose 4-group scale rows travel as the packed [rows / 2, 8] tables."""
    w = W.scaled(W.WORKLOADS["toy"], d_model=d, num_experts=64, top_k=8, ffn_dim=1536, tokens=64, layout=layout)
    c = Case(w)
    out, idx, _ = c.run_layer()
    o64, oidx, _, _ = c.oracle_layer()
    assert np.array_equal(idx.numpy(), oidx)
    check_outputs(out.numpy(), o64, c.x.float().numpy())


@pytest.mark.parametrize("layout", ["separate", "fused"])
def test_tensor_core_path_many_tokens_per_expert(layout):
    """512 tokens over 16 experts (top-4): every expert has ~128 entries (>= 32) and runs on
    the tcgen05 path (d and ffn_dim multiples of 512, B >= 256)."""
    w = W.scaled(W.WORKLOADS["toy"], ffn_dim=512, tokens=512, layout=layout)
    c = Case(w)
    out, idx, _ = c.run_layer()
    o64, oidx, _, _ = c.oracle_layer()
    assert np.array_equal(idx.numpy(), oidx)
    counts = np.bincount(oidx.ravel(), minlength=w.num_experts)
    assert counts.min() >= 64
    check_outputs(out.numpy(), o64, c.x.float().numpy())


def test_tensor_core_and_small_paths_mixed():
    """Skewed routing: a few hot experts on the tcgen05 path, the rest on the mma.sync path."""
    w = W.scaled(W.WORKLOADS["toy"], ffn_dim=512, tokens=384, num_experts=32, zipf_s=1.1)
    c = Case(w)
    out, idx, _ = c.run_layer()
    o64, oidx, _, _ = c.oracle_layer()
    assert np.array_equal(idx.numpy(), oidx)
    counts = np.bincount(oidx.ravel(), minlength=w.num_experts)
    assert counts.max() >= 32 and (counts[counts > 0] < 32).any()
    check_outputs(out.numpy(), o64, c.x.float().numpy())


def _reshape_scales(c: "Case"):
    """Weight rows outside the sampled scale range, in every projection of every expert:
    rows 7j whose group scales (and biases) fall by 2^-(g mod 16) along the row (a 2^15
    spread), rows 11j + 3 that are constant (s = 0, b = +-0.01) and rows 13j + 5 with
    scales and biases times 4.  The oracle and the device get the same tensors."""
    for name in list(c.wts_cpu):
        if not name.startswith("s_"):
            continue
        s = c.wts_cpu[name].to(torch.float64).clone()
        b = c.wts_cpu["b_" + name[2:]].to(torch.float64).clone()
        _, out, G = s.shape
        f = torch.pow(2.0, -(torch.arange(G, dtype=torch.float64) % 16))
        s[:, 0::7, :] *= f
        b[:, 0::7, :] *= f
        s[:, 3::11, :] = 0.0
        b[:, 3::11, :] = 0.01 * torch.where(torch.arange(G) % 2 == 0, 1.0, -1.0).to(torch.float64)
        s[:, 5::13, :] *= 4.0
        b[:, 5::13, :] *= 4.0
        c.wts_cpu[name] = W._bf16_bits(s)
        c.wts_cpu["b_" + name[2:]] = W._bf16_bits(b)
    c.wts_gpu = {k: v.to(DEV) for k, v in c.wts_cpu.items()}
    c.weights = smoe.Weights(c.wts_gpu)
    c.layer_o = oracle.Layer.from_workload(c.w, c.wts_cpu)


@pytest.mark.parametrize("layout,zipf", [("separate", 0.0), ("fused", 0.0), ("separate", 1.1)])
def test_tensor_core_path_rows_outside_the_sampled_scale_range(layout, zipf):
    """Weights outside the sampled scale range on the tcgen05 path: groups whose scale is 2^-15
    of the row's largest (s (q - 8) among the fp16 subnormals), constant rows whose whole
    weight is the per-group term b + 8 s, and rows with four times the scales; with zipf = 1.1
    the cold experts take the mma.sync path over the same tensors."""
    w = W.scaled(W.WORKLOADS["toy"], ffn_dim=512, tokens=512 if zipf == 0.0 else 384,
                 num_experts=16 if zipf == 0.0 else 32, layout=layout, zipf_s=zipf)
    c = Case(w)
    _reshape_scales(c)
    out, idx, _ = c.run_layer()
    o64, oidx, _, _ = c.oracle_layer()
    assert np.array_equal(idx.numpy(), oidx)
    counts = np.bincount(oidx.ravel(), minlength=w.num_experts)
    assert counts.max() >= 32
    check_outputs(out.numpy(), o64, c.x.float().numpy())


# ----------------------------------------------------------------------------- shared expert
@pytest.mark.parametrize("layout,B,F", [("separate", 16, 256), ("fused", 37, 256), ("separate", 512, 512)])
def test_shared_expert_parity(layout, B, F):
    """residual += shared expert (3 column slices) on every token: few-token path, fused
    layout with a ragged batch, and the tcgen05 path (every slice holds B >= 256 entries)."""
    _need_gpu()
    P = 3
    w = W.scaled(W.WORKLOADS["toy"], shared_ffn_dim=P * F, shared_slices=P, layout=layout, tokens=B)
    x = W.gen_x(w, 0, B)
    sl = W.gen_shared_weights(w, 0)
    desc = smoe.make_desc(w.d_model, P, P, F, layout, 1)
    ws = smoe.alloc_workspace(desc, B)
    weights = smoe.Weights({k: v.to(DEV) for k, v in sl.items()})
    res = x.float().to(DEV)
    smoe.smoe_clear_device_status(ws)
    smoe.smoe_shared_expert_ffn(desc, weights, x.to(DEV).view(torch.int16), res, ws)
    assert smoe.smoe_read_device_status(ws) == 0
    dense = oracle.shared_dense_layer(sl, w.d_model, P, F, layout)
    r0 = x.float().numpy().astype(np.float64)
    check_outputs(res.cpu().numpy(), r0 + oracle.shared_expert_ffn(dense, x), r0)


def test_qwen2_layer_with_shared_expert():
    """Qwen2-MoE-shaped layer: top-8 of 64 without norm_topk_prob, then the 20480-wide shared
    expert (8 slices): residual + routed + shared against the oracle on sampled rows."""
    w = W.WORKLOADS["qwen2_prefill64"]
    c = Case(w, B=64)
    P, F = w.shared_slices, w.shared_ffn_dim // w.shared_slices
    sl = W.gen_shared_weights(w, 0, device=DEV)
    sdesc = smoe.make_desc(w.d_model, P, P, F, w.layout, 1)
    sws = smoe.alloc_workspace(sdesc, 64)
    res = c.x.float().to(DEV)
    idx = torch.empty(64, w.top_k, dtype=torch.int32, device=DEV)
    wt = torch.empty(64, w.top_k, dtype=torch.float32, device=DEV)
    smoe.smoe_clear_device_status(c.ws)
    smoe.smoe_clear_device_status(sws)
    smoe.smoe_moe_layer(c.desc, c.weights, c.x_dev(), c.gate_d, None, res, c.ws, idx, wt)
    smoe.smoe_shared_expert_ffn(sdesc, smoe.Weights(sl), c.x_dev(), res, sws)
    assert smoe.smoe_read_device_status(c.ws) == 0 and smoe.smoe_read_device_status(sws) == 0
    rows = list(range(0, 64, 4))
    o64, oidx, ow64, _ = c.oracle_layer(rows=rows)
    assert np.array_equal(idx.cpu().numpy(), oidx)
    np.testing.assert_allclose(wt.cpu().numpy(), ow64, rtol=W_RTOL, atol=1e-7)
    sliced = oracle.Layer(w.d_model, P, P, F, {k: v.cpu() for k, v in sl.items()}, w.layout, 1)
    shared = np.zeros((64, w.d_model))
    for p in range(P):
        shared[rows] += oracle.expert_ffn(sliced, p, c.x, rows)
    check_outputs(res.cpu().numpy(), o64 + shared, c.x.float().numpy(), rows=rows)


@pytest.mark.parametrize("B,K,E,d,F", [
    (64, 16, 256, 512, 256),    # the largest top_k and expert count; 1024 entries: one-CTA union
    (129, 8, 64, 512, 256),     # 1032 entries: the chunked union just past the one-CTA limit
    (24, 4, 16, 256, 256),      # d_model = ffn_dim = 256: 8-byte scale rows in both passes
])
def test_layer_parity_at_the_limits(B, K, E, d, F):
    w = W.scaled(W.WORKLOADS["toy"], top_k=K, num_experts=E, d_model=d, ffn_dim=F, tokens=B)
    c = Case(w)
    out, idx, wt = c.run_layer()
    o64, oidx, ow64, _ = c.oracle_layer()
    assert np.array_equal(idx.numpy(), oidx)
    np.testing.assert_allclose(wt.numpy(), ow64, rtol=W_RTOL, atol=1e-7)
    check_outputs(out.numpy(), o64, c.x.float().numpy())


def test_top1_routing():
    w = W.scaled(W.WORKLOADS["toy"], top_k=1)
    c = Case(w)
    out, idx, wt = c.run_layer()
    o64, oidx, _, _ = c.oracle_layer()
    assert np.array_equal(idx.numpy(), oidx) and torch.all(wt == 1.0)
    check_outputs(out.numpy(), o64, c.x.float().numpy())


def test_zero_tokens_is_noop():
    c = Case(W.WORKLOADS["toy"], gap=False)
    empty = torch.empty(0, c.w.d_model, dtype=torch.int16, device=DEV)
    res = torch.empty(0, c.w.d_model, dtype=torch.float32, device=DEV)
    smoe.smoe_moe_layer(c.desc, c.weights, empty, c.gate_d, None, res, c.ws)
    torch.cuda.synchronize()


def test_layer_is_deterministic():
    c = Case(W.WORKLOADS["prefill64"], B=64)
    a, _, _ = c.run_layer()
    b, _, _ = c.run_layer()
    assert torch.equal(a, b)


def test_tensor_core_layer_is_deterministic():
    """Hot experts on the tensor-core path, cold ones on the few-token queue: repeated calls
    agree bit for bit."""
    w = W.scaled(W.WORKLOADS["toy"], ffn_dim=512, tokens=384, num_experts=32, zipf_s=1.1)
    c = Case(w)
    outs = [c.run_layer()[0] for _ in range(3)]
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


def test_graph_replay_equals_direct():
    c = Case(W.WORKLOADS["decode_b8"])
    direct, _, _ = c.run_layer()
    res0 = c.x.float().to(DEV)
    res = res0.clone()
    xd = c.x_dev()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        smoe.smoe_moe_layer(c.desc, c.weights, xd, c.gate_d, None, res, c.ws)
    res.copy_(res0)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(res.cpu(), direct)


# ----------------------------------------------------------------------------- chained stacks
# Per-layer figures of the chained tests (layer, max-abs, delta rel-L2, delta RMS), printed at
# the end of each test so that a run with -s records them.
CHAIN_RECORD = {}


def tile_covering_rows(idx: np.ndarray, E: int, extra: int = 512, tile: int = 192, tc_min: int = 32,
                       hottest: int = 2) -> list:
    """Token rows that exercise every output column of the tensor-core tiles.

    From the (oracle) routing idx [B, K]: an expert's token list is its tokens in ascending
    order, and list position p sits in tile p // tile at column p % tile.  The rows chosen hit
    every column residue 0..tile-1 of the `hottest` experts with the longest lists (residue r
    taken in tile r % tiles, so the residues spread over the tiles), the first and the last
    position of every tile of every expert with at least tc_min entries (so each one's last
    short tile is hit), and evenly spaced rows up to `extra` more."""
    B = idx.shape[0]
    lists = [np.nonzero((idx == e).any(axis=1))[0] for e in range(E)]
    counts = np.array([len(t) for t in lists])
    rows = set()
    for e in np.argsort(-counts, kind="stable")[:hottest]:
        n = counts[e]
        tiles = (n + tile - 1) // tile
        for r in range(min(tile, n)):
            p = (r % tiles) * tile + r
            rows.add(int(lists[e][p if p < n else r]))
    for e in np.nonzero(counts >= tc_min)[0]:
        n = counts[e]
        for t0 in range(0, n, tile):
            rows.add(int(lists[e][t0]))
            rows.add(int(lists[e][min(n, t0 + tile) - 1]))
    step = max(1, B // extra)
    rows.update(range(0, B, step))
    return sorted(rows)


def _chain(name, layers, B=None, sample_rows=None, cover_tiles=False):
    """Teacher-forced check of a chained stack, layer by layer: the oracle's layer l consumes
    the GPU's own x_l and h_l.  Routing indices must match exactly; a token whose oracle gap
    between ranks K and K+1 is below 1e-4 is exempt, and so is a token whose expert set
    matches but two ranks swapped where their oracle logits tie within 1e-4 (fp32 against
    fp64 logits on a near-tie); exempt and swapped tokens together stay within 0.1% of the
    token-layers.  Outputs within the literal tolerances (rel-L2 5e-3, max-abs 2e-2) on
    `sample_rows` (all rows if None), or on rows chosen per layer by tile_covering_rows."""
    w = W.WORKLOADS[name]
    B = B or w.tokens
    first = Case(w, 0, B)
    h = first.x.float().to(DEV)
    xb = torch.empty(B, w.d_model, dtype=torch.int16, device=DEV)
    exempt, swapped, total, worst = 0, 0, 0, 0.0
    record = []
    for l in range(layers):
        c = first if l == 0 else Case(w, l, B, x=first.x)
        smoe.smoe_rmsnorm_bf16(h, xb, 1e-6, center=int(w.chain_center))
        x_l = xb.cpu().view(torch.bfloat16)
        h_in = h.cpu().clone()
        # the rmsnorm glue itself: at most one bf16 ulp from the double-precision oracle
        ox = oracle.rmsnorm_bf16(h_in.numpy(), 1e-6, center=w.chain_center)
        assert rmsnorm_glue_close(x_l.view(torch.int16).numpy(), ox) < 1e-2
        idx = torch.empty(B, w.top_k, dtype=torch.int32, device=DEV)
        wt = torch.empty(B, w.top_k, dtype=torch.float32, device=DEV)
        smoe.smoe_clear_device_status(c.ws)
        smoe.smoe_moe_layer(c.desc, c.weights, xb, c.gate_d, c.bias_d, h, c.ws, idx, wt)
        assert smoe.smoe_read_device_status(c.ws) == 0
        # teacher-forced oracle on the GPU's own layer input
        c.x = x_l
        oi, ow64, _, lg = oracle.route(x_l, c.gate, c.bias, w.top_k, w.norm_topk_prob)
        s = -np.sort(-lg, axis=1)
        near = (s[:, w.top_k - 1] - s[:, w.top_k]) < 1e-4
        gi = idx.cpu().numpy()
        swap = np.zeros(B, bool)
        for t in np.nonzero(np.any(gi != oi, axis=1) & ~near)[0]:
            # same expert set; ranks may only swap where the oracle logits tie within 1e-4
            assert set(gi[t].tolist()) == set(oi[t].tolist()), f"layer {l} token {t}: expert set differs"
            diff = gi[t] != oi[t]
            assert np.all(np.abs(lg[t, gi[t][diff]] - lg[t, oi[t][diff]]) < 1e-4), \
                f"layer {l} token {t}: rank order differs on separated logits"
            swap[t] = True
        exempt += int(near.sum())
        swapped += int(swap.sum())
        total += B
        if cover_tiles:
            rows = tile_covering_rows(oi, w.num_experts)
        else:
            rows = sample_rows if sample_rows is not None else list(range(B))
        rows = [r for r in rows if not near[r] and not swap[r]]
        _, o64, _ = oracle.moe_layer(c.layer_o, x_l, oi, ow64, h_in, rows=rows)
        d_rel, mab = check_outputs(h.cpu().numpy(), o64, h_in.numpy(), rows=rows)
        delta = o64[rows] - h_in.numpy()[rows]
        record.append((l, len(rows), mab, d_rel, float(np.sqrt(np.mean(delta ** 2)))))
        worst = max(worst, d_rel)
    CHAIN_RECORD[name] = record
    for l, n, mab, d_rel, rms in record:
        print(f"[chain {name}] layer {l}: rows {n}, max-abs {mab:.3e}, delta rel-L2 {d_rel:.3e}, delta RMS {rms:.3g}")
    print(f"[chain {name}] near-tie tokens {exempt}, swapped ranks {swapped}, of {total} token-layers")
    assert exempt + swapped <= max(1, 0.001 * total), f"{exempt} near-tie + {swapped} swapped token-layers"
    return worst


def _chain_free(name, layers, rows=None):
    """The stack run end to end on each side, with no teacher forcing: the GPU's chain (glue
    norm and smoe_moe_layer per layer, all B tokens) against the oracle's own chain over the
    sampled rows (tokens are independent through the stack, so the oracle runs the rows alone).

    The two chains round their layer inputs to bf16 independently (fp32 against fp64 norms),
    so from layer 1 on their inputs differ in a few elements by one bf16 ulp, and the
    difference grows through the stack.  A token whose routing differs from the oracle's at
    some layer has flipped: its later layers use other experts, so it is counted and left out
    of the output comparison.  Every flip must be explained by the inputs: the oracle's
    smallest adjacent logit gap among ranks 1..K+1 on its own input is below twice the
    largest change of any logit between the two inputs (both evaluated by the oracle), plus
    the 1e-4 near-tie margin of the GPU's fp32 logits.  The tokens that never flip match the
    oracle's output and the stack's total update (output - input) to rel-L2 5e-3."""
    w = W.WORKLOADS[name]
    B = w.tokens
    rows = list(range(B)) if rows is None else list(rows)
    first = Case(w, 0, B)
    h = first.x.float().to(DEV)
    xb = torch.empty(B, w.d_model, dtype=torch.int16, device=DEV)
    h_o = first.x.float().numpy()[rows]
    h0 = h_o.astype(np.float64)
    flipped = np.zeros(len(rows), bool)
    for l in range(layers):
        c = first if l == 0 else Case(w, l, B, x=first.x)
        smoe.smoe_rmsnorm_bf16(h, xb, 1e-6, center=int(w.chain_center))
        idx = torch.empty(B, w.top_k, dtype=torch.int32, device=DEV)
        wt = torch.empty(B, w.top_k, dtype=torch.float32, device=DEV)
        smoe.smoe_clear_device_status(c.ws)
        smoe.smoe_moe_layer(c.desc, c.weights, xb, c.gate_d, c.bias_d, h, c.ws, idx, wt)
        assert smoe.smoe_read_device_status(c.ws) == 0
        xo = torch.from_numpy(oracle.rmsnorm_bf16(h_o.astype(np.float32), 1e-6, center=w.chain_center)
                              .view(np.int16)).view(torch.bfloat16)
        xg = xb.cpu()[rows].view(torch.bfloat16)
        oi, ow64, _, lg_o = oracle.route(xo, c.gate, c.bias, w.top_k, w.norm_topk_prob)
        lg_g = oracle.logits(xg, c.gate, c.bias)
        new = np.any(idx.cpu().numpy()[rows] != oi, axis=1) & ~flipped
        pert = np.max(np.abs(lg_g - lg_o), axis=1)
        gap = logit_gaps(lg_o, w.top_k)
        for t in np.nonzero(new)[0]:
            assert gap[t] < 2 * pert[t] + 1e-4, \
                f"layer {l} row {rows[t]}: routing flipped at logit gap {gap[t]:.3e} > 2 x input change {pert[t]:.3e}"
        flipped |= new
        out, _, _ = oracle.moe_layer(c.layer_o, xo, oi, ow64, h_o.astype(np.float32))
        h_o = out.astype(np.float64)
        keep = ~flipped
        g = h.cpu().numpy()[rows].astype(np.float64)
        print(f"[chain-free {name}] layer {l}: flipped {int(flipped.sum())} of {len(rows)}, output rel-L2 "
              f"{rel_l2(g[keep], h_o[keep]):.3e}, max logit change {pert.max():.2e}")
    g = h.cpu().numpy()[rows].astype(np.float64)
    keep = ~flipped
    o_rel = rel_l2(g[keep], h_o[keep])
    d_rel = rel_l2(g[keep] - h0[keep], h_o[keep] - h0[keep])
    mab = max_abs(g[keep], h_o[keep])
    print(f"[chain-free {name}] {layers} layers, {len(rows)} tokens: flipped {int(flipped.sum())}, output rel-L2 "
          f"{o_rel:.3e}, update rel-L2 {d_rel:.3e}, max-abs {mab:.3e}, output RMS {np.sqrt(np.mean(h_o ** 2)):.3g}")
    assert keep.sum() >= len(rows) // 4, "too few tokens kept their routing to compare outputs"
    assert o_rel <= REL_L2_TOL and d_rel <= REL_L2_TOL, (o_rel, d_rel)
    return flipped.sum(), o_rel, mab


@pytest.mark.parametrize("center", [0, 1])
def test_rmsnorm_glue_parity(center):
    _need_gpu()
    rng = np.random.default_rng(11 + center)
    for B, d in [(1, 512), (64, 4096), (37, 2048)]:
        h = (rng.normal(size=(B, d)) * rng.uniform(0.1, 100.0, size=(B, 1)) + rng.normal(size=(B, 1)) * 50)
        h = torch.from_numpy(h.astype(np.float32))
        xb = torch.empty(B, d, dtype=torch.int16, device=DEV)
        smoe.smoe_rmsnorm_bf16(h.to(DEV), xb, 1e-6, center=center)
        ox = oracle.rmsnorm_bf16(h.numpy(), 1e-6, center=bool(center))
        assert rmsnorm_glue_close(xb.cpu().numpy(), ox) < 1e-2


def test_chain_prefill64_teacher_forced():
    _chain("prefill64", 2)


def test_chain_qwen35_fused_teacher_forced():
    _chain("q35_prefill64", 3)


def test_chain_decode_b1_teacher_forced():
    """One token through the first 4 layers of the 94-layer decode chain."""
    _chain("decode_b1_l94", 4)


def test_chain_long_skewed_tile_covering_rows():
    """4096 tokens with the Zipf logit bias, layers 0 and 1 at full size: rows chosen from the
    oracle's token lists to hit every tile column of the hottest experts and every
    tensor-core expert's last short tile (hot experts far above the 32-entry threshold)."""
    _chain("long4096", 2, cover_tiles=True)


def test_chain_free_prefill64_all_layers():
    """The 8-layer B=64 stack end to end, GPU chain against oracle chain."""
    _chain_free("prefill64", 8)


def test_chain_free_long4096_sampled_rows():
    """The 4-layer 4096-token Zipf stack end to end on 256 sampled tokens."""
    _chain_free("long4096", 4, rows=range(0, 4096, 16))
