"""The C ABI's host-side argument validation under AddressSanitizer and UndefinedBehaviorSanitizer.

`csrc/api.cu` and `csrc/noalloc.cu` (every entry point's validation) are recompiled with the
sanitizers and linked with the library's other objects; a child interpreter with the sanitizer
runtimes preloaded drives the argument-error paths of every call through plain ctypes.  These paths return before any CUDA
call, so no GPU is needed; an out-of-bounds access or undefined behaviour in them aborts the child.
"""
import glob
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import ctypes
L = ctypes.CDLL(LIB)
vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
OK, INVALID, UNSUPPORTED, WORKSPACE = 0, 1, 2, 3


class Desc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("d_model", "num_experts", "top_k", "ffn_dim", "group_size", "norm_topk_prob", "layout")]


class W(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("w_up", "s_up", "b_up", "w_gate", "s_gate", "b_gate",
                 "w_gate_up", "s_gate_up", "b_gate_up", "w_down", "s_down", "b_down")]


L.smoe_workspace_bytes.restype = sz
L.smoe_workspace_bytes.argtypes = [vp, i32]
L.smoe_stream_state_bytes.restype = sz
L.smoe_stream_state_bytes.argtypes = [i32, i32]
L.smoe_status_string.restype = ctypes.c_char_p
d = Desc(4096, 128, 8, 1536, 64, 1, 0)
bad = [Desc(4096, 128, 8, 1536, 32, 1, 0), Desc(4096, 4, 8, 1536, 64, 1, 0), Desc(4000, 128, 8, 1536, 64, 1, 0),
       Desc(4096, 300, 8, 1536, 64, 1, 0), Desc(4096, 128, 8, 1536, 64, 2, 0), Desc(4096, 128, 8, 1536, 64, 1, 7)]
r = ctypes.byref
assert L.smoe_workspace_bytes(r(d), 64) > 0
for b in bad:
    assert L.smoe_workspace_bytes(r(b), 64) == 0
    assert L.smoe_route(r(b), vp(1024), vp(1024), None, 4, vp(1024), vp(1024), vp(4096), sz(1 << 30), None) != OK
assert L.smoe_route(None, vp(1024), vp(1024), None, 4, vp(1024), vp(1024), vp(4096), sz(1 << 30), None) == INVALID
assert L.smoe_route(r(d), vp(1024), vp(1024), None, 4, vp(1024), vp(1024), vp(4097), sz(1 << 30), None) == WORKSPACE
assert L.smoe_route(r(d), vp(1026), vp(1024), None, 4, vp(1024), vp(1024), vp(4096), sz(1 << 30), None) == UNSUPPORTED
assert L.smoe_route_ranked(r(d), vp(1024), vp(1024), None, 4, 40, vp(1024), vp(1024), vp(1024), None, vp(4096),
                           sz(1 << 30), None) == INVALID
assert L.smoe_expert_union(r(d), None, 4, vp(1), vp(1), vp(1), vp(1), vp(1), vp(4096), sz(1 << 30), None) == INVALID
w = W()
assert L.smoe_moe_ffn_batch(r(d), r(w), vp(1024), 4, vp(1), vp(1), vp(1), vp(1), vp(1), vp(1), vp(1024), vp(4096),
                            sz(1 << 30), None) == INVALID
assert L.smoe_moe_layer(r(d), None, vp(1024), vp(1024), None, 4, vp(1024), None, None, vp(4096), sz(1 << 30),
                        None) == INVALID
assert L.smoe_shared_expert_ffn(r(d), r(w), vp(1024), 4, vp(1024), vp(4096), sz(1 << 30), None) == INVALID
assert L.smoe_rmsnorm_bf16(None, ctypes.c_float(1e-6), 0, 4, 4096, vp(1024), None) == INVALID
assert L.smoe_stream_state_bytes(0, 8) == 0 and L.smoe_stream_state_bytes(10, 8) == 4 * (4 + 10 + 16)
assert L.smoe_stream_init(None, 10, 8, None) == INVALID
assert L.smoe_stream_plan(r(d), 4, 129, vp(1), vp(1), vp(1024), 256, 64, vp(1), vp(1), vp(4096), sz(1 << 30),
                          None) == INVALID
assert L.smoe_stream_plan(r(d), 4, 0, vp(1), vp(1), vp(1024), 256, 31, vp(1), vp(1), vp(4096), sz(1 << 30),
                          None) == INVALID
h = W()
for name, _ in W._fields_:
    setattr(h, name, 4096)
h.w_down = 4096 + 8
assert L.smoe_stream_copy(r(d), r(h), r(h), 64, vp(1), vp(4096), sz(1 << 30), None) == UNSUPPORTED
assert L.smoe_stream_copy(r(d), r(w), r(w), 64, vp(1), vp(4096), sz(1 << 30), None) == INVALID
assert L.smoe_route_noalloc(None, vp(1024), vp(1024), None, 4, vp(1024), vp(1024), None) == INVALID
assert L.smoe_route_noalloc(r(bad[0]), vp(1024), vp(1024), None, 4, vp(1024), vp(1024), None) == UNSUPPORTED
assert L.smoe_route_noalloc(r(d), vp(1024), vp(1024), None, -1, vp(1024), vp(1024), None) == INVALID
assert L.smoe_route_noalloc(r(d), None, None, None, 0, None, None, None) == OK
assert L.smoe_route_noalloc(r(d), vp(1024), vp(1024), None, 4, None, vp(1024), None) == INVALID
assert L.smoe_route_noalloc(r(d), vp(1032), vp(1024), None, 4, vp(1024), vp(1024), None) == UNSUPPORTED
assert L.smoe_route_noalloc(r(d), vp(1024), vp(1024), None, 8193, vp(1024), vp(1024), None) == UNSUPPORTED
for s in range(7):
    assert L.smoe_status_string(s)
print("sanitized abi ok")
"""


def _runtime(name):
    p = subprocess.run(["gcc", f"-print-file-name={name}"], capture_output=True, text=True).stdout.strip()
    return p if os.path.isabs(p) and os.path.exists(p) else None


def test_abi_validation_under_asan_and_ubsan(tmp_path):
    sys.path.insert(0, ROOT)
    from moe_expert_routing_gb300 import build as B
    asan, ubsan = _runtime("libasan.so"), _runtime("libubsan.so")
    if not asan or not ubsan or not os.path.exists(B.NVCC):
        pytest.skip("nvcc or the gcc sanitizer runtimes are not installed")
    B.build()   # the library's objects
    san = ("api", "noalloc")
    san_objs = []
    for name in san:
        o = str(tmp_path / f"{name}_san.o")
        # (nvcc splits -Xcompiler values at commas: one flag per sanitizer)
        cmd = [B.NVCC, *B.ARCH, *B.FLAGS, "-Xcompiler", "-fsanitize=address", "-Xcompiler", "-fsanitize=undefined",
               "-Xcompiler", "-fno-omit-frame-pointer", "-c", os.path.join(B.CSRC, name + ".cu"), "-o", o]
        subprocess.run(cmd, check=True, capture_output=True)
        san_objs.append(o)
    objs = [o for o in glob.glob(os.path.join(B.OUT_DIR, "*.o")) if os.path.basename(o)[:-2] not in san]
    lib = str(tmp_path / "libsmoe_san.so")
    subprocess.run([B.NVCC, *B.ARCH, "-shared", "-cudart", "shared", "-o", lib, *san_objs, *objs], check=True,
                   capture_output=True)
    undef = subprocess.run(["nm", "-D", "--undefined-only", lib], capture_output=True, text=True).stdout
    assert "__asan_" in undef and "__ubsan_" in undef   # the validation code is instrumented
    env = dict(os.environ, LD_PRELOAD=f"{asan}:{ubsan}",
               ASAN_OPTIONS="detect_leaks=0:abort_on_error=1:protect_shadow_gap=0",
               UBSAN_OPTIONS="halt_on_error=1:print_stacktrace=1")
    r = subprocess.run([sys.executable, "-c", f"LIB = {lib!r}\n" + CHILD], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and "sanitized abi ok" in r.stdout, (r.stdout[-2000:], r.stderr[-4000:])
