"""The oracle's C++ under AddressSanitizer and UndefinedBehaviorSanitizer (host only).

Every entry point of the oracle library runs once on small inputs (separate and fused layouts,
layer-major and token-major, ranked routing, union, dequant, RMSNorm) in a child interpreter
with the ASan runtime preloaded; any out-of-bounds access, use after free or undefined
behaviour aborts the child.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
sys.modules["torch"] = None          # numpy inputs only
sys.path.insert(0, ROOT)
import numpy as np
import oracle
oracle._LIB_PATH = SAN
rng = np.random.default_rng(0)
d, E, K, F, B = 256, 8, 2, 256, 5


def bf16(v):
    return (np.asarray(v, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def proj(rows, inn):
    w = rng.integers(0, 2 ** 32, size=(E, rows, inn // 8), dtype=np.uint64).astype(np.uint32)
    s = bf16(rng.uniform(0.005, 0.02, size=(E, rows, inn // 64)))
    b = bf16(-8 * rng.uniform(0.005, 0.02, size=(E, rows, inn // 64)))
    return w, s, b


wg, sg, bg = proj(F, d)
wu, su, bu = proj(F, d)
wd, sd, bd = proj(d, F)
sep = dict(w_gate=wg, s_gate=sg, b_gate=bg, w_up=wu, s_up=su, b_up=bu, w_down=wd, s_down=sd, b_down=bd)
fused = dict(w_gate_up=np.concatenate([wg, wu], 1), s_gate_up=np.concatenate([sg, su], 1),
             b_gate_up=np.concatenate([bg, bu], 1), w_down=wd, s_down=sd, b_down=bd)
x = bf16(rng.standard_normal((B, d)))
gate = (0.05 * rng.standard_normal((E, d))).astype(np.float32)
bias = (0.1 * rng.standard_normal(E)).astype(np.float32)
idx, w64, w32, lg = oracle.route(x, gate, bias, K, 1)
oracle.route_ranked(x, gate, None, K, 3, 0)
oracle.expert_union(idx, E)
res = rng.standard_normal((B, d)).astype(np.float32)
for layout, wts in (("separate", sep), ("fused", fused)):
    layer = oracle.Layer(d, E, K, F, wts, layout)
    a = oracle.moe_layer(layer, x, idx, w64, res, want_slots=True)[1]
    b = oracle.moe_layer(layer, x, idx, w64, res, mode="token", threads=2)[1]
    assert np.array_equal(a, b)
    oracle.moe_layer(layer, x, idx, w64, res, rows=[1, 3])
    oracle.expert_ffn(layer, int(idx[0, 0]), x, [0, 2])
oracle.dequant(wd[1], sd[1], bd[1])
oracle.rmsnorm_bf16(res, 1e-6, True)
oracle.to_bf16(rng.standard_normal(17))
print("sanitized oracle ok")
"""


def _runtime(name):
    p = subprocess.run(["gcc", f"-print-file-name={name}"], capture_output=True, text=True).stdout.strip()
    return p if os.path.isabs(p) and os.path.exists(p) else None


def test_oracle_under_asan_and_ubsan():
    from oracle import build as ob
    asan, ubsan = _runtime("libasan.so"), _runtime("libubsan.so")
    if not asan or not ubsan:
        pytest.skip("gcc sanitizer runtimes not installed")
    san = ob.build(sanitize=True)
    env = dict(os.environ, LD_PRELOAD=f"{asan}:{ubsan}",
               ASAN_OPTIONS="detect_leaks=0:abort_on_error=1",
               UBSAN_OPTIONS="halt_on_error=1:print_stacktrace=1")
    script = f"ROOT = {ROOT!r}\nSAN = {san!r}\n" + CHILD
    r = subprocess.run([sys.executable, "-c", script], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "sanitized oracle ok" in r.stdout, (r.stdout[-2000:], r.stderr[-4000:])


def test_sanitizer_catches_a_planted_overread():
    # a planted mistake on the host: the oracle's RMSNorm told the input has 4 rows, given 3
    from oracle import build as ob
    asan, ubsan = _runtime("libasan.so"), _runtime("libubsan.so")
    if not asan or not ubsan:
        pytest.skip("gcc sanitizer runtimes not installed")
    san = ob.build(sanitize=True)
    env = dict(os.environ, LD_PRELOAD=f"{asan}:{ubsan}", ASAN_OPTIONS="detect_leaks=0")
    script = f"""
import sys, ctypes
sys.modules["torch"] = None
sys.path.insert(0, {ROOT!r})
import numpy as np
import oracle
oracle._LIB_PATH = {san!r}
h = np.ones((3, 256), np.float32)
out = np.empty((4, 256), np.uint16)
oracle.lib().oracle_rmsnorm_bf16(oracle._ptr(h), 4, 256, ctypes.c_double(1e-6), 0, oracle._ptr(out))
print("not caught")
"""
    r = subprocess.run([sys.executable, "-c", script], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0 and "AddressSanitizer" in r.stderr and "not caught" not in r.stdout
