"""Experts streamed from pinned host memory into an HBM slot pool, through the C ABI.

The residency plan (smoe_stream_plan) must equal the oracle's SlotPool call by call, bit for
bit (slots, copy lists and the final state); a slot must hold exactly the bytes of the host
expert copied into it (smoe_stream_copy); and a layer run over the pool must equal the
resident layer bit for bit (same kernels, same bytes, same order) and the oracle within the
layer tolerances.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import resampled_x
from moe_expert_routing_gb300 import smoe
from moe_expert_routing_gb300 import workload as W
from test_gpu_parity import Case, check_outputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _union(desc, idx, ws):
    B, K = idx.shape
    E = desc.num_experts
    uid = torch.zeros(E, dtype=torch.int32, device=DEV)
    nu = torch.zeros(1, dtype=torch.int32, device=DEV)
    off = torch.zeros(E + 1, dtype=torch.int32, device=DEV)
    tl = torch.zeros(B * K, dtype=torch.int32, device=DEV)
    sl = torch.zeros(B * K, dtype=torch.int32, device=DEV)
    smoe.smoe_expert_union(desc, idx, uid, nu, off, tl, sl, ws)
    return uid, nu, off, tl, sl


def _state_arrays(state, n_keys, S):
    s = state.cpu().numpy()
    return int(s[0]), s[4:4 + n_keys].tolist(), s[4 + n_keys:4 + n_keys + S].tolist(), \
        s[4 + n_keys + S:4 + n_keys + 2 * S].tolist()


def test_stream_plan_matches_oracle_pool():
    _need_gpu()
    E, K, B, layers, S = 16, 4, 3, 3, 14
    n_keys = layers * E
    desc = smoe.make_desc(512, E, K, 256)
    ws = smoe.alloc_workspace(desc, B)
    rng = np.random.default_rng(21)
    p = rng.zipf(1.5, size=E).astype(np.float64)
    p /= p.sum()
    pool = oracle.SlotPool(n_keys, S)
    state = smoe.alloc_stream_state(n_keys, S)
    slot_ids = torch.full((E,), -7, dtype=torch.int32, device=DEV)
    copy_list = torch.full((1 + 2 * E,), -7, dtype=torch.int32, device=DEV)
    smoe.smoe_clear_device_status(ws)
    n_hits = n_copies = 0
    for call in range(60):
        layer = call % layers
        idx = np.stack([rng.choice(E, K, replace=False, p=p) for _ in range(B)]).astype(np.int32)
        uid, nu, *_ = _union(desc, torch.from_numpy(idx).to(DEV), ws)
        smoe.smoe_stream_plan(desc, B, layer * E, uid, nu, state, n_keys, S, slot_ids, copy_list, ws)
        n = int(nu.item())
        ou = oracle.expert_union(idx, E)[0]
        slots, copies = pool.plan([layer * E + int(e) for e in ou])
        assert slot_ids[:n].cpu().tolist() == slots
        cl = copy_list.cpu().tolist()
        assert cl[0] == len(copies)
        assert [(cl[1 + 2 * m], cl[2 + 2 * m]) for m in range(cl[0])] == [(k - layer * E, s) for k, s in copies]
        n_hits += n - len(copies)
        n_copies += len(copies)
    assert smoe.smoe_read_device_status(ws) == 0
    tick, slot_of, owner, stamp = _state_arrays(state, n_keys, S)
    assert (tick, slot_of, owner, stamp) == (pool.tick, pool.slot_of, pool.owner, pool.stamp)
    assert n_hits > 0 and n_copies > S   # the sequence exercised hits, fills and evictions


def test_stream_plan_bad_union_id_sets_fault():
    _need_gpu()
    E, K, B, S = 16, 4, 2, 8
    desc = smoe.make_desc(512, E, K, 256)
    ws = smoe.alloc_workspace(desc, B)
    state = smoe.alloc_stream_state(E, S)
    idx = torch.tensor([[0, 1, 2, 3], [1, 2, 3, 4]], dtype=torch.int32, device=DEV)
    uid, nu, *_ = _union(desc, idx, ws)
    uid[2] = E + 3   # an id the plan must reject
    slot_ids = torch.zeros(E, dtype=torch.int32, device=DEV)
    copy_list = torch.full((1 + 2 * E,), 5, dtype=torch.int32, device=DEV)
    smoe.smoe_clear_device_status(ws)
    smoe.smoe_stream_plan(desc, B, 0, uid, nu, state, E, S, slot_ids, copy_list, ws)
    bits = smoe.smoe_read_device_status(ws)
    assert bits & smoe.SMOE_FAULT_SLOT_POOL
    assert int(copy_list[0].item()) == 0
    assert (slot_ids[:int(nu.item())] == -1).all()
    tick, slot_of, owner, _ = _state_arrays(state, E, S)
    assert tick == 0 and all(v == -1 for v in slot_of) and all(v == -1 for v in owner)   # nothing changed
    smoe.smoe_clear_device_status(ws)


STREAM_CASES = [("toy", None, 24), ("decode_b8", None, 72), ("q35_prefill64", 8, 128), ("long4096", 512, 128)]


@pytest.mark.parametrize("name,B,S", STREAM_CASES)
def test_streamed_layer_equals_resident_layer(name, B, S):
    _need_gpu()
    w = W.WORKLOADS[name]
    c = Case(w, B=B)
    B, K, E, d = c.B, w.top_k, w.num_experts, w.d_model
    host = smoe.pin_weights(c.wts_cpu)
    pool_t = smoe.pool_tensors(c.wts_cpu, S)
    pool = smoe.Weights(pool_t)
    pdesc = smoe.make_desc(d, S, K, w.ffn_dim, w.layout, w.norm_topk_prob)
    pws = smoe.alloc_workspace(pdesc, B)
    state = smoe.alloc_stream_state(E, S)
    slot_ids = torch.zeros(E, dtype=torch.int32, device=DEV)
    copy_list = torch.zeros(1 + 2 * E, dtype=torch.int32, device=DEV)
    # three calls: a fresh pool (all misses), new tokens (hits and misses), the first tokens again
    x1 = c.x
    x2, _ = resampled_x(w, 1, B, c.gate, c.bias)
    smoe.smoe_clear_device_status(c.ws)
    smoe.smoe_clear_device_status(pws)
    for call, x in enumerate([x1, x2, x1]):
        xd = x.to(DEV).view(torch.int16)
        idx = torch.empty(B, K, dtype=torch.int32, device=DEV)
        wt = torch.empty(B, K, dtype=torch.float32, device=DEV)
        smoe.smoe_route(c.desc, xd, c.gate_d, c.bias_d, idx, wt, c.ws)
        uid, nu, off, tl, sl = _union(c.desc, idx, c.ws)
        res_r = x.float().to(DEV)
        smoe.smoe_moe_ffn_batch(c.desc, c.weights, xd, uid, nu, off, tl, sl, wt, res_r, c.ws)
        smoe.smoe_stream_plan(c.desc, B, 0, uid, nu, state, E, S, slot_ids, copy_list, c.ws)
        smoe.smoe_stream_copy(c.desc, host, pool, S, copy_list, c.ws)
        res_s = x.float().to(DEV)
        smoe.smoe_moe_ffn_batch(pdesc, pool, xd, slot_ids, nu, off, tl, sl, wt, res_s, pws)
        assert smoe.smoe_read_device_status(c.ws) == 0 and smoe.smoe_read_device_status(pws) == 0
        assert torch.equal(res_s, res_r), f"call {call}"
        n = int(nu.item())
        copies = int(copy_list[0].item())
        if call == 0:
            assert copies == n
        if call == 2:
            assert copies < n   # retention: the first tokens' experts are hits unless evicted
        # every union expert's slot holds that expert's bytes
        for u, s in zip(uid[:n].cpu().tolist(), slot_ids[:n].cpu().tolist()):
            for k, v in c.wts_cpu.items():
                assert torch.equal(pool_t[k][s].cpu(), v[u]), (k, u, s)
        if call == 0:
            out64 = c.oracle_layer()[0]
            check_outputs(res_s.cpu().numpy(), out64, x.float().numpy())
