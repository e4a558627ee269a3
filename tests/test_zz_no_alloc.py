"""smoe_route_noalloc: routing for callers that cannot allocate device memory.

Such callers (a plugin inside an application that owns the whole device-memory budget, or a
latency-critical loop that cannot risk cudaMalloc's synchronisation) get their split-K scratch
from a fixed array inside the library.  The test calls the no-allocation entry point through
the C ABI twice in a row and checks both results against smoe_route (the workspace-based entry
point), with the routing tolerance the other tests use: indices bit-exact, weights to 1e-5
relative.  It sits in a file of its own, collected last.
"""
import numpy as np
import pytest
import torch

from helpers import W_RTOL, resampled_x
from moe_expert_routing_gb300 import smoe
from moe_expert_routing_gb300 import workload as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("name,B", [("toy", 16), ("decode_b8", 8), ("prefill64", 64), ("q35_prefill64", 64),
                                    ("long4096", 256)])
def test_route_noalloc_matches_route(name, B):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = W.WORKLOADS[name]
    gate = W.gen_gate(w, 0)
    bias = W.gen_gate_bias(w, 0)
    x, _ = resampled_x(w, 0, B, gate, bias)
    desc = smoe.make_desc(w.d_model, w.num_experts, w.top_k, w.ffn_dim, w.layout, w.norm_topk_prob)
    xd = x.to(DEV).view(torch.int16)
    gd = gate.to(DEV)
    bd = None if bias is None else bias.to(DEV)
    ws = smoe.alloc_workspace(desc, B)
    ref_idx = torch.empty(B, w.top_k, dtype=torch.int32, device=DEV)
    ref_w = torch.empty(B, w.top_k, dtype=torch.float32, device=DEV)
    smoe.smoe_route(desc, xd, gd, bd, ref_idx, ref_w, ws)
    for _ in range(2):   # two calls in a row share (and overwrite) the fixed scratch
        idx = torch.full((B, w.top_k), -1, dtype=torch.int32, device=DEV)
        wt = torch.full((B, w.top_k), -1.0, dtype=torch.float32, device=DEV)
        smoe.smoe_route_noalloc(desc, xd, gd, bd, idx, wt)
        torch.cuda.synchronize()
        assert np.array_equal(idx.cpu().numpy(), ref_idx.cpu().numpy())
        np.testing.assert_allclose(wt.cpu().numpy(), ref_w.cpu().numpy(), rtol=W_RTOL, atol=1e-7)


def test_route_noalloc_large_batch_matches_oracle():
    """Beyond 256 tokens fewer split-K partials fit the fixed scratch; the routing still
    agrees with the oracle like smoe_route's does (indices exact, weights to 1e-5)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import oracle
    w = W.WORKLOADS["long4096"]
    B = 1024
    gate = W.gen_gate(w, 0)
    bias = W.gen_gate_bias(w, 0)
    x, _ = resampled_x(w, 0, B, gate, bias)
    desc = smoe.make_desc(w.d_model, w.num_experts, w.top_k, w.ffn_dim)
    idx = torch.empty(B, w.top_k, dtype=torch.int32, device=DEV)
    wt = torch.empty(B, w.top_k, dtype=torch.float32, device=DEV)
    smoe.smoe_route_noalloc(desc, x.to(DEV).view(torch.int16), gate.to(DEV), bias.to(DEV), idx, wt)
    oi, ow64, _, _ = oracle.route(x, gate, bias, w.top_k, 1)
    assert np.array_equal(idx.cpu().numpy(), oi)
    np.testing.assert_allclose(wt.cpu().numpy(), ow64, rtol=W_RTOL, atol=1e-7)


@pytest.mark.parametrize("B", [8192])
def test_route_noalloc_whole_scratch_matches_oracle(B):
    """The largest batch the fixed scratch takes at 128 experts: 8192 x 128 = 2^20 partial
    logits, one split-K partial, the whole array used; indices exact, weights to 1e-5."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import oracle
    w = W.WORKLOADS["long4096"]
    gate = W.gen_gate(w, 0)
    bias = W.gen_gate_bias(w, 0)
    x, _ = resampled_x(w, 0, B, gate, bias)
    desc = smoe.make_desc(w.d_model, w.num_experts, w.top_k, w.ffn_dim)
    idx = torch.empty(B, w.top_k, dtype=torch.int32, device=DEV)
    wt = torch.empty(B, w.top_k, dtype=torch.float32, device=DEV)
    smoe.smoe_route_noalloc(desc, x.to(DEV).view(torch.int16), gate.to(DEV), bias.to(DEV), idx, wt)
    oi, ow64, _, _ = oracle.route(x, gate, bias, w.top_k, 1)
    assert np.array_equal(idx.cpu().numpy(), oi)
    np.testing.assert_allclose(wt.cpu().numpy(), ow64, rtol=W_RTOL, atol=1e-7)


@pytest.mark.parametrize("B", [8193, 16384])
def test_route_noalloc_rejects_oversize_batch(B):
    """One token past the scratch (8193 x 128 > 2^20 floats even with one split) is refused
    with SMOE_ERR_UNSUPPORTED before anything is launched."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = W.WORKLOADS["prefill64"]
    desc = smoe.make_desc(w.d_model, w.num_experts, w.top_k, w.ffn_dim)
    x = torch.zeros(B, w.d_model, dtype=torch.int16, device=DEV)
    gate = torch.zeros(w.num_experts, w.d_model, dtype=torch.float32, device=DEV)
    idx = torch.full((B, w.top_k), -1, dtype=torch.int32, device=DEV)
    wt = torch.empty(B, w.top_k, dtype=torch.float32, device=DEV)
    with pytest.raises(smoe.SmoeError) as ei:
        smoe.smoe_route_noalloc(desc, x, gate, None, idx, wt)
    assert ei.value.status == smoe.SMOE_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(idx == -1)   # nothing was launched
