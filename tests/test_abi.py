"""Host-side checks of the C ABI (no GPU): the library builds and loads, exports every entry
point include/smoe.h declares, and rejects bad arguments before launching anything."""
import ctypes
import os
import re

import pytest

from moe_expert_routing_gb300 import build as smoe_build
from moe_expert_routing_gb300 import smoe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    smoe_build.build()
    return smoe.load_library()


def _declared():
    src = open(os.path.join(ROOT, "include", "smoe.h")).read()
    return sorted(set(re.findall(r"SMOE_API\s+[\w\s\*]*?\b(smoe_\w+)\s*\(", src)))


def test_header_declares_the_entry_points():
    assert _declared() == sorted(smoe.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_only_the_c_abi_is_exported(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", smoe.LIB_PATH], capture_output=True, text=True).stdout
    names = {ln.split()[-1] for ln in out.splitlines() if ln.strip()}
    assert {n for n in names if n.startswith("smoe_")} == set(_declared())
    assert not [n for n in names if "smoe" in n and not n.startswith("smoe_")]


def _desc(**kw):
    base = dict(d_model=4096, num_experts=128, top_k=8, ffn_dim=1536)
    base.update(kw)
    layout = base.pop("layout", "separate")
    g = base.pop("group_size", 64)
    norm = base.pop("norm_topk_prob", 1)
    return smoe.make_desc(base["d_model"], base["num_experts"], base["top_k"], base["ffn_dim"], layout, norm, g)


def test_workspace_size_monotone_and_invalid(lib):
    d = _desc()
    sizes = [smoe.smoe_workspace_bytes(d, b) for b in (1, 8, 64, 512, 4096)]
    assert all(s > 0 and s % 256 == 0 for s in sizes)
    assert sizes == sorted(sizes)
    # B=64: the FFN scratch dominates: 512 rows x (d fp16 + d fp32 + F fp16) plus group sums
    assert sizes[2] >= 512 * (4096 * 2 + 4096 * 4 + 1536 * 2)
    assert smoe.smoe_workspace_bytes(_desc(group_size=32), 8) == 0
    assert smoe.smoe_workspace_bytes(_desc(top_k=200), 8) == 0
    assert smoe.smoe_workspace_bytes(_desc(d_model=4000), 8) == 0
    # scale rows must be 8 bytes (256 inputs) or a multiple of 16 bytes (512 inputs)
    assert smoe.smoe_workspace_bytes(_desc(d_model=768), 8) == 0
    assert smoe.smoe_workspace_bytes(_desc(ffn_dim=1280), 8) == 0
    assert smoe.smoe_workspace_bytes(_desc(d_model=256, ffn_dim=256), 8) > 0
    assert smoe.smoe_workspace_bytes(_desc(num_experts=512), 8) == 0


def _call_route(lib, desc, x=1024, w=1024, idx=1024, wt=1024, B=4, ws=4096, wsb=1 << 30):
    vp = ctypes.c_void_p
    return lib.smoe_route(ctypes.byref(desc), vp(x), vp(w), None, B, vp(idx), vp(wt), vp(ws), wsb, None)


def test_route_argument_errors(lib):
    d = _desc()
    assert _call_route(lib, d, x=0) == smoe.SMOE_ERR_INVALID_ARG
    assert _call_route(lib, d, idx=0) == smoe.SMOE_ERR_INVALID_ARG
    assert _call_route(lib, d, B=-1) == smoe.SMOE_ERR_INVALID_ARG
    assert _call_route(lib, d, x=1032) == smoe.SMOE_ERR_UNSUPPORTED        # 8-byte aligned only
    assert _call_route(lib, d, ws=0) == smoe.SMOE_ERR_WORKSPACE
    assert _call_route(lib, d, ws=4096 + 128) == smoe.SMOE_ERR_WORKSPACE   # not 256-aligned
    assert _call_route(lib, d, wsb=1024) == smoe.SMOE_ERR_WORKSPACE        # too small
    assert _call_route(lib, _desc(group_size=128)) == smoe.SMOE_ERR_UNSUPPORTED
    assert _call_route(lib, _desc(top_k=0)) == smoe.SMOE_ERR_INVALID_ARG
    assert _call_route(lib, _desc(top_k=129)) == smoe.SMOE_ERR_INVALID_ARG
    assert _call_route(lib, _desc(norm_topk_prob=2)) == smoe.SMOE_ERR_INVALID_ARG
    assert _call_route(lib, d, B=0, x=0, idx=0) == smoe.SMOE_OK            # B == 0: no-op
    assert lib.smoe_route(None, None, None, None, 1, None, None, None, 0, None) == smoe.SMOE_ERR_INVALID_ARG


def test_route_noalloc_argument_errors(lib):
    """The no-allocation router validates like smoe_route (same descriptor check) and refuses
    batches whose partial logits do not fit its fixed 2^20-float scratch, all before touching
    CUDA."""
    d = _desc()   # 128 experts
    vp = ctypes.c_void_p

    def call(desc=d, B=4, x=1024, w=1024, idx=1024, wt=1024):
        return lib.smoe_route_noalloc(None if desc is None else ctypes.byref(desc), vp(x), vp(w), None, B, vp(idx),
                                      vp(wt), None)

    assert call(desc=None) == smoe.SMOE_ERR_INVALID_ARG
    assert call(desc=_desc(top_k=0)) == smoe.SMOE_ERR_INVALID_ARG
    assert call(desc=_desc(norm_topk_prob=3)) == smoe.SMOE_ERR_INVALID_ARG
    assert call(desc=_desc(group_size=32)) == smoe.SMOE_ERR_UNSUPPORTED
    assert call(desc=_desc(num_experts=300)) == smoe.SMOE_ERR_UNSUPPORTED
    assert call(B=-1) == smoe.SMOE_ERR_INVALID_ARG
    assert call(B=0, x=0, idx=0) == smoe.SMOE_OK          # B == 0: no-op
    assert call(x=0) == smoe.SMOE_ERR_INVALID_ARG
    assert call(w=0) == smoe.SMOE_ERR_INVALID_ARG
    assert call(idx=0) == smoe.SMOE_ERR_INVALID_ARG
    assert call(wt=0) == smoe.SMOE_ERR_INVALID_ARG
    assert call(x=1032) == smoe.SMOE_ERR_UNSUPPORTED      # 8-byte aligned only
    assert call(w=1028) == smoe.SMOE_ERR_UNSUPPORTED
    assert call(B=8193) == smoe.SMOE_ERR_UNSUPPORTED      # 8193 x 128 > 2^20 partial logits
    assert call(B=4097, desc=_desc(num_experts=256)) == smoe.SMOE_ERR_UNSUPPORTED


def test_route_ranked_argument_errors(lib):
    d = _desc()   # top_k 8, 128 experts: at most 24 further ranks
    vp = ctypes.c_void_p

    def call(n_spec, spec=1024, B=4, x=1024):
        return lib.smoe_route_ranked(ctypes.byref(d), vp(x), vp(1024), None, B, n_spec, vp(1024), vp(1024),
                                     vp(spec), None, vp(4096), 1 << 30, None)

    assert call(-1) == smoe.SMOE_ERR_INVALID_ARG
    assert call(25) == smoe.SMOE_ERR_INVALID_ARG                 # top_k + n_spec > 32
    assert call(8, spec=0) == smoe.SMOE_ERR_INVALID_ARG          # no spec_idx buffer
    assert call(8, B=0, x=0) == smoe.SMOE_OK                     # B == 0: no-op
    assert call(8, x=1032) == smoe.SMOE_ERR_UNSUPPORTED
    small = _desc(num_experts=10, top_k=4)
    assert lib.smoe_route_ranked(ctypes.byref(small), vp(1024), vp(1024), None, 4, 7, vp(1024), vp(1024), vp(1024),
                                 None, vp(4096), 1 << 30, None) == smoe.SMOE_ERR_INVALID_ARG   # 11 ranks > 10


def test_layer_and_ffn_argument_errors(lib):
    d = _desc()
    vp = ctypes.c_void_p
    w = smoe.ExpertWeights()
    # down weights missing
    rc = lib.smoe_moe_layer(ctypes.byref(d), ctypes.byref(w), vp(1024), vp(1024), None, 4, vp(1024), None, None,
                            vp(4096), 1 << 30, None)
    assert rc == smoe.SMOE_ERR_INVALID_ARG
    rc = lib.smoe_moe_layer(ctypes.byref(d), None, vp(1024), vp(1024), None, 4, vp(1024), None, None, vp(4096),
                            1 << 30, None)
    assert rc == smoe.SMOE_ERR_INVALID_ARG
    # fused layout without gate_up tensors
    w.w_down = w.s_down = w.b_down = 1024
    w.w_up = w.s_up = w.b_up = w.w_gate = w.s_gate = w.b_gate = 2048
    fd = _desc(layout="fused")
    rc = lib.smoe_moe_layer(ctypes.byref(fd), ctypes.byref(w), vp(1024), vp(1024), None, 4, vp(1024), None, None,
                            vp(4096), 1 << 30, None)
    assert rc == smoe.SMOE_ERR_INVALID_ARG
    # misaligned down scales
    w.s_down = 1032
    rc = lib.smoe_moe_layer(ctypes.byref(d), ctypes.byref(w), vp(1024), vp(1024), None, 4, vp(1024), None, None,
                            vp(4096), 1 << 30, None)
    assert rc == smoe.SMOE_ERR_UNSUPPORTED
    rc = lib.smoe_moe_ffn_batch(ctypes.byref(d), ctypes.byref(w), vp(1024), 4, None, vp(1), vp(1), vp(1), vp(1),
                                vp(1), vp(1024), vp(4096), 1 << 30, None)
    assert rc == smoe.SMOE_ERR_INVALID_ARG


def test_ffn_batch_norm_argument_errors(lib):
    d = _desc()
    vp, f = ctypes.c_void_p, ctypes.c_float
    w = smoe.ExpertWeights()
    for name, _ in smoe.ExpertWeights._fields_:
        setattr(w, name, 4096)

    def call(x_next=2048, eps=1e-6, center=1, B=4, weights=w):
        return lib.smoe_moe_ffn_batch_norm(ctypes.byref(d), ctypes.byref(weights), vp(1024), B, vp(1), vp(1), vp(1),
                                           vp(1), vp(1), vp(1), vp(1024), f(eps), center, vp(x_next), vp(4096),
                                           1 << 30, None)

    assert call(x_next=0) == smoe.SMOE_ERR_INVALID_ARG
    assert call(eps=-1.0) == smoe.SMOE_ERR_INVALID_ARG
    assert call(center=2) == smoe.SMOE_ERR_INVALID_ARG
    assert call(B=-1) == smoe.SMOE_ERR_INVALID_ARG
    assert call(B=0, x_next=0) == smoe.SMOE_OK                     # B == 0: no-op
    assert call(x_next=2052) == smoe.SMOE_ERR_UNSUPPORTED          # 4-byte aligned only
    assert call(weights=smoe.ExpertWeights()) == smoe.SMOE_ERR_INVALID_ARG


def test_union_and_norm_argument_errors(lib):
    d = _desc()
    vp = ctypes.c_void_p
    rc = lib.smoe_expert_union(ctypes.byref(d), None, 4, vp(1), vp(1), vp(1), vp(1), vp(1), vp(4096), 1 << 30, None)
    assert rc == smoe.SMOE_ERR_INVALID_ARG
    rc = lib.smoe_expert_union(ctypes.byref(d), vp(1), 4, vp(1), vp(1), vp(1), vp(1), vp(1), vp(4097), 1 << 30, None)
    assert rc == smoe.SMOE_ERR_WORKSPACE
    f = ctypes.c_float
    assert lib.smoe_rmsnorm_bf16(None, f(1e-6), 0, 4, 4096, vp(1024), None) == smoe.SMOE_ERR_INVALID_ARG
    assert lib.smoe_rmsnorm_bf16(vp(1024), f(-1.0), 0, 4, 4096, vp(1024), None) == smoe.SMOE_ERR_INVALID_ARG
    assert lib.smoe_rmsnorm_bf16(vp(1024), f(1e-6), 2, 4, 4096, vp(1024), None) == smoe.SMOE_ERR_INVALID_ARG
    assert lib.smoe_rmsnorm_bf16(vp(1024), f(1e-6), 1, 4, 4094, vp(1024), None) == smoe.SMOE_ERR_UNSUPPORTED
    assert lib.smoe_rmsnorm_bf16(None, f(1e-6), 1, 0, 4096, None, None) == smoe.SMOE_OK
    assert lib.smoe_clear_device_status(vp(4097), None) == smoe.SMOE_ERR_WORKSPACE
    assert lib.smoe_read_device_status(None, None, None) == smoe.SMOE_ERR_WORKSPACE


def test_status_strings(lib):
    for s in range(6):
        assert smoe.smoe_status_string(s) not in ("", "unknown status")
    assert smoe.smoe_status_string(99) == "unknown status"


def test_binding_refuses_cpu_tensors(lib):
    import torch
    d = _desc(d_model=512, num_experts=16, top_k=4, ffn_dim=256)
    with pytest.raises(ValueError):
        smoe.smoe_rmsnorm_bf16(torch.zeros(2, 512), torch.zeros(2, 512, dtype=torch.int16))
    del d


def test_stream_argument_errors(lib):
    vp = ctypes.c_void_p
    d = _desc()   # 128 experts, top-8
    E, K = d.num_experts, d.top_k
    assert lib.smoe_stream_state_bytes(0, 8) == 0
    assert lib.smoe_stream_state_bytes(10, 0) == 0
    assert lib.smoe_stream_state_bytes(10, 257) == 0
    assert lib.smoe_stream_state_bytes(10, 8) == 4 * (4 + 10 + 2 * 8)
    assert lib.smoe_stream_init(None, 10, 8, None) == smoe.SMOE_ERR_INVALID_ARG
    assert lib.smoe_stream_init(vp(1026), 10, 8, None) == smoe.SMOE_ERR_INVALID_ARG
    assert lib.smoe_stream_init(vp(1024), 10, 257, None) == smoe.SMOE_ERR_UNSUPPORTED

    def plan(B=4, key_base=0, n_keys=2 * E, n_slots=64, uid=vp(1), ws=vp(4096)):
        return lib.smoe_stream_plan(ctypes.byref(d), B, key_base, uid, vp(1), vp(1024), n_keys, n_slots, vp(1),
                                    vp(1), ws, 1 << 30, None)
    assert plan(key_base=E + 1) == smoe.SMOE_ERR_INVALID_ARG          # keys of the layer beyond n_keys
    assert plan(key_base=-1) == smoe.SMOE_ERR_INVALID_ARG
    assert plan(B=4, n_slots=4 * K - 1) == smoe.SMOE_ERR_INVALID_ARG  # a union of 32 experts cannot fit
    assert plan(B=64, n_slots=E - 1) == smoe.SMOE_ERR_INVALID_ARG     # min(B K, E) = E
    assert plan(n_slots=257) == smoe.SMOE_ERR_UNSUPPORTED
    assert plan(B=0, uid=None) == smoe.SMOE_OK                         # empty batch: nothing to plan
    assert plan(uid=None) == smoe.SMOE_ERR_INVALID_ARG
    assert plan(ws=vp(4097)) == smoe.SMOE_ERR_WORKSPACE

    W = smoe.ExpertWeights()
    assert lib.smoe_stream_copy(ctypes.byref(d), None, ctypes.byref(W), 64, vp(1), vp(4096), 1 << 30,
                                None) == smoe.SMOE_ERR_INVALID_ARG
    assert lib.smoe_stream_copy(ctypes.byref(d), ctypes.byref(W), ctypes.byref(W), 64, vp(1), vp(4096), 1 << 30,
                                None) == smoe.SMOE_ERR_INVALID_ARG      # separate layout, NULL tensors
    H = smoe.ExpertWeights()
    for name, _ in smoe.ExpertWeights._fields_:
        setattr(H, name, 4096)
    H.w_down = 4096 + 8                                                  # misaligned
    assert lib.smoe_stream_copy(ctypes.byref(d), ctypes.byref(H), ctypes.byref(H), 64, vp(1), vp(4096), 1 << 30,
                                None) == smoe.SMOE_ERR_UNSUPPORTED
    assert lib.smoe_stream_copy(ctypes.byref(d), ctypes.byref(H), ctypes.byref(H), 300, vp(1), vp(4096), 1 << 30,
                                None) == smoe.SMOE_ERR_UNSUPPORTED


def test_host_weights_must_be_pinned(lib):
    import torch
    with pytest.raises(ValueError):
        smoe.HostWeights({"w_down": torch.zeros(4, 8, dtype=torch.int32)})   # pageable CPU memory
    with pytest.raises(ValueError):
        smoe.HostWeights({"w_down": torch.zeros(4, 8, dtype=torch.int32)[:, ::2]})
