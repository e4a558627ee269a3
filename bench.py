"""Benchmark of the per-layer MoE block (route -> union -> 4-bit SwiGLU experts -> combine).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl gb300|reference]

A step is one pass of the whole hot path over one batch: for every layer of the workload's
stack, RMSNorm glue (chained stacks), exact routing, the expert union, the expert FFN and
the weighted combine, all through libsmoe's C ABI.  Inputs are seeded and synthetic (the
workload generator), resident in HBM when the timed region starts.  A step of a stack reads
far more expert weights than L2 holds; a step that reads less than ~1 GB (one decode layer) is
timed on its own after a write that evicts L2.

The JSON line reports MoE-layer tokens/s (token-layers per second) for the whole job, the
union-expert bytes/s, the roofline of the expert FFN step, the end-to-end figure through
host buffers, and the CPU oracle timed on a bounded sample (`cpu_baseline`).
`--impl reference` times the oracle alone on the host cores (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s and union-expert GB/s at 1 GB300; % of roofline"
UNIT = "token-layers/s"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def max_over_ranks(value: float, world: int, device="cpu") -> float:
    """The largest of every rank's value (the slowest rank's time); the value itself at N = 1."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class NvmlClocks:
    """SM clock and clock-event reasons sampled through NVML (ctypes, read-only queries) every
    5 ms from a thread, while the timed region runs."""

    SM = 1   # NVML_CLOCK_SM
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch_device):
        import ctypes
        import threading
        import torch
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        props = torch.cuda.get_device_properties(torch_device)
        bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0".encode()
        if self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(self.h)) != 0:
            raise RuntimeError("no NVML handle for " + bus.decode())
        self.get_reasons = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.ct = ctypes
        mx = ctypes.c_uint()
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.SM, ctypes.byref(mx))
        self.max_mhz = float(mx.value)
        self.sm, self.reasons, self.stop_flag = [], set(), False
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def _run(self):
        ct = self.ct
        clk, r = ct.c_uint(), ct.c_ulonglong()
        while not self.stop_flag:
            if self.lib.nvmlDeviceGetClockInfo(self.h, self.SM, ct.byref(clk)) == 0:
                self.sm.append(float(clk.value))
            if self.get_reasons(self.h, ct.byref(r)) == 0:
                self.reasons.update(n for bit, n in self.REASONS.items() if r.value & bit)
            time.sleep(0.005)

    def stop(self):
        self.stop_flag = True
        self.thread.join()
        if not self.sm:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["no samples"], "source": "nvml"}
        s = sorted(self.sm)
        return {"sm_mhz": s[len(s) // 2], "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                "samples": len(s), "source": "nvml, 5 ms"}


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region (fallback
    when NVML cannot be loaded)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.idx = gpu_index
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(gpu_index), "-lms", "200"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in out.splitlines():
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(smax), "reasons": sorted(reasons), "samples": len(sm),
                "source": "nvidia-smi, 200 ms"}


def start_clocks(torch_device, gpu_index: int):
    try:
        return NvmlClocks(torch_device)
    except Exception:
        return Clocks(gpu_index)


def _host_link_gbs(torch, dev) -> float:
    """Pinned host -> device copy bandwidth (GB/s), best of 3 copies of 1 GiB: the denominator
    of the streamed-expert copy."""
    n = 1 << 30
    hbuf = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    dbuf = torch.empty(n, dtype=torch.uint8, device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = float("inf")
    for _ in range(3):
        e0.record()
        dbuf.copy_(hbuf, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    del hbuf, dbuf
    return n / (best * 1e-3) / 1e9


def _traffic_from_profile(workload: str):
    """(DRAM bytes per FFN-step launch, union size of that launch) from the JSON record written
    beside the committed ncu summary of this workload, if every kernel source it names is
    unchanged since the capture (sha256 match); else None."""
    path = os.path.join(ROOT, "profiles", f"expert_ffn_{workload}.traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    try:
        for src, sha in rec["sources_sha256"].items():
            with open(os.path.join(ROOT, src), "rb") as f:
                if hashlib.sha256(f.read()).hexdigest() != sha:
                    return None
        return int(rec["dram_bytes_per_ffn_call"]), int(rec["union_experts"])
    except (OSError, KeyError, TypeError, ValueError):
        return None


# ------------------------------------------------------------------------------ oracle timing
def oracle_layers(w, x_rows, layer_source, budget_s: float, threads: int = 0):
    """Time the oracle (layer-major, all host cores) on the given token rows through the
    workload's stack, layer after layer (glue norm for chained stacks, routing, routed
    experts, shared expert), passing over the stack again while less than budget_s seconds
    of CPU work are done: returns (token-layers timed, seconds, cores).  layer_source(l)
    gives layer l's host tensors (copied outside the timed region): (weights, gate, bias,
    shared slices or None)."""
    import numpy as np
    import oracle
    cores = threads if threads > 0 else oracle.hardware_threads()
    B = x_rows.shape[0]
    x0 = x_rows.contiguous()
    P = w.shared_slices
    spent, n_layers = 0.0, 0
    for step in range(10 ** 6):
        if spent >= budget_s:
            break
        if step % w.layers == 0:   # a new pass starts from the stack's input
            h = x0.float().numpy()
        l = step % w.layers
        wts, gate, bias, shared = layer_source(l)
        lay = oracle.Layer.from_workload(w, wts)
        sl = oracle.Layer(w.d_model, P, P, w.shared_ffn_dim // P, shared, w.layout, 0) if P else None
        all_slices = np.tile(np.arange(P, dtype=np.int32), (B, 1)) if P else None
        t0 = time.perf_counter()
        xl = oracle.rmsnorm_bf16(h, 1e-6, center=w.chain_center) if w.chained else x0
        idx, w64, _, _ = oracle.route(xl, gate, bias, w.top_k, w.norm_topk_prob)
        out, _, _ = oracle.moe_layer(lay, xl, idx, w64, h, threads=threads)
        if P:
            out, _, _ = oracle.moe_layer(sl, xl, all_slices, np.ones((B, P)), out, threads=threads)
        h = out
        spent += time.perf_counter() - t0
        n_layers += 1
    return B * n_layers, spent, cores


def _sample_rows(w, budget_s: float = 6.0):
    """Token rows whose first layer the oracle finishes in about budget_s on the host."""
    macs_per_token = 3 * w.d_model * (w.ffn_dim * w.top_k + w.shared_ffn_dim)
    return max(1, min(w.tokens, int(budget_s * 2.0e9 / macs_per_token)))


def run_reference(args, w):
    import torch
    from moe_expert_routing_gb300 import workload as W

    gdev = "cuda" if torch.cuda.is_available() else "cpu"
    per_step = max(0.5, args.ref_seconds / max(1, args.steps + args.warmup))
    n = _sample_rows(w, budget_s=per_step / 2)
    x = W.gen_x(w, 0, n)
    cache = {}

    def layer_source(l):
        if l not in cache:
            wts = {k: v.cpu() for k, v in W.gen_layer_weights(w, l, device=gdev).items()}
            sh = ({k: v.cpu() for k, v in W.gen_shared_weights(w, l, device=gdev).items()}
                  if w.shared_slices else None)
            cache[l] = (wts, W.gen_gate(w, l), W.gen_gate_bias(w, l), sh)
        return cache[l]

    for _ in range(args.warmup):
        oracle_layers(w, x, layer_source, per_step)
    rates, cores, units, spent = [], 0, 0, 0.0
    for _ in range(args.steps):
        units, spent, cores = oracle_layers(w, x, layer_source, per_step)
        rates.append(units / spent)
    value = sum(rates) / len(rates)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": spent * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "tokens": w.tokens, "layers": w.layers, "sample_tokens": n,
                   "sample_token_layers": units},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"first {n} of {w.tokens} tokens, {units // n} layer passes over the "
                                   f"{w.layers}-layer stack, layer-major fp64 oracle, {spent:.1f} s per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------ GPU arm
def run_gpu(args, w, world, rank, local):
    import torch
    import torch.distributed as dist
    from moe_expert_routing_gb300 import smoe
    from moe_expert_routing_gb300 import workload as W

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    smoe.load_library()
    B, L, K, E, d, F = w.tokens, w.layers, w.top_k, w.num_experts, w.d_model, w.ffn_dim
    desc = smoe.make_desc(d, E, K, F, w.layout, w.norm_topk_prob)

    # streamed experts: every layer's experts in pinned host memory, one pool of S HBM slots
    # shared by the layers (keys layer * E + expert)
    S = w.stream_slots
    streamed = S > 0
    # shared expert (if the workload has one): column slices, its own descriptor and workspace
    P = w.shared_slices
    sdesc = smoe.make_desc(d, P, P, w.shared_ffn_dim // P, w.layout, 1) if P else None
    sws = smoe.alloc_workspace(sdesc, B, dev) if P else None
    def pinned_copy(v):
        hv = torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
        hv.copy_(v)
        return hv

    layers = []
    for l in range(L):
        wts = W.gen_layer_weights(w, l, device=dev)
        host = None
        if streamed:   # the layer's experts live in host memory only
            wts = {k: pinned_copy(v) for k, v in wts.items()}
            host = smoe.HostWeights(wts)
        bias = W.gen_gate_bias(w, l)
        layers.append({
            "shared": smoe.Weights(W.gen_shared_weights(w, l, device=dev)) if P else None,
            "weights": None if streamed else smoe.Weights(wts), "host": host, "wts": wts,
            "gate": W.gen_gate(w, l, device=dev).contiguous(),
            "cl": torch.zeros(1 + 2 * E, dtype=torch.int32, device=dev),
            "bias": None if bias is None else bias.to(dev),
            "uid": torch.zeros(E, dtype=torch.int32, device=dev), "nu": torch.zeros(1, dtype=torch.int32, device=dev),
            "off": torch.zeros(E + 1, dtype=torch.int32, device=dev),
            "tl": torch.zeros(B * K, dtype=torch.int32, device=dev),
            "sl": torch.zeros(B * K, dtype=torch.int32, device=dev),
        })
    if streamed:
        pool_t = smoe.pool_tensors(layers[0]["wts"], S, dev)
        pool = smoe.Weights(pool_t)
        pdesc = smoe.make_desc(d, S, K, F, w.layout, w.norm_topk_prob)
        pws = smoe.alloc_workspace(pdesc, B, dev)
        n_keys = L * E
        sstate = smoe.alloc_stream_state(n_keys, S, dev)
        slot_ids = torch.zeros(E, dtype=torch.int32, device=dev)
        # one token per step from a correlated sequence: warm-up, 3 graph warm-ups, timed, e2e
        T = max(3, args.warmup) + 3 + args.steps + 16
        x_seq = W.gen_x_sequence(w, 0, T, w.seq_rho).to(dev).view(torch.int16).contiguous()
        x_in = x_seq[0:1]
    else:
        x_in = W.gen_x(w, 0, B, device=dev).view(torch.int16).contiguous()

    def x_of(i):
        return x_seq[i % T:i % T + 1] if streamed else x_in

    ws = smoe.alloc_workspace(desc, B, dev)
    h = torch.empty(B, d, dtype=torch.float32, device=dev)
    xb = torch.empty(B, d, dtype=torch.int16, device=dev)
    idx = torch.empty(B, K, dtype=torch.int32, device=dev)
    wt = torch.empty(B, K, dtype=torch.float32, device=dev)
    # workloads with a ranked router: ranks K..K+spec-1 (ids and probabilities) every layer
    spec_idx = torch.empty(B, w.spec, dtype=torch.int32, device=dev) if w.spec else None
    spec_p = torch.empty(B, w.spec, dtype=torch.float32, device=dev) if w.spec else None
    stream = torch.cuda.current_stream()
    # kernels per layer: router (2), union (1, or 3 above 1024 entries), FFN (gather, two passes
    # or the both-pass + two tensor-core passes, combine), shared expert (slice routing + FFN),
    # glue norm where it is not fused into the combine, slot plan + copy for streamed experts
    def ffn_kernels(b, dd, ff):
        tc = dd % 512 == 0 and ff % 512 == 0 and dd <= 4096 and ff <= 4096 and b >= 256
        return 5 if tc else 4
    # chained stacks without a shared expert: the norm that feeds layer l+1 runs in layer l's
    # combine kernel (smoe_moe_ffn_batch_norm); with a shared expert it follows the shared expert
    fused_norm = w.chained and not P
    launches_per_layer = (2 + (1 if B * K <= 1024 else 3) + ffn_kernels(B, d, F) +
                          (1 + ffn_kernels(B, d, w.shared_ffn_dim // P) if P else 0) + (2 if streamed else 0) +
                          (1 if w.chained and not fused_norm else 0))
    launches_per_step = launches_per_layer * L + (1 if fused_norm else 0)

    def step(x_dev, ev=None, rec=None):
        # rec: per layer (n_union, copy list) buffers of this step (streamed), kept for the stats
        cur = torch.cuda.current_stream()   # the capture stream while a graph is captured
        h.copy_(x_dev.view(torch.bfloat16))
        if fused_norm:
            smoe.smoe_rmsnorm_bf16(h, xb, 1e-6, center=int(w.chain_center))
        for l, ly in enumerate(layers):
            if w.chained:
                if not fused_norm:
                    smoe.smoe_rmsnorm_bf16(h, xb, 1e-6, center=int(w.chain_center))
                xl = xb
            else:
                xl = x_dev
            if w.spec:
                smoe.smoe_route_ranked(desc, xl, ly["gate"], ly["bias"], idx, wt, spec_idx, spec_p, ws)
            else:
                smoe.smoe_route(desc, xl, ly["gate"], ly["bias"], idx, wt, ws)
            nu = rec[l][0] if rec is not None else ly["nu"]
            smoe.smoe_expert_union(desc, idx, ly["uid"], nu, ly["off"], ly["tl"], ly["sl"], ws)
            if streamed:
                cl = rec[l][1] if rec is not None else ly["cl"]
                smoe.smoe_stream_plan(desc, B, l * E, ly["uid"], nu, sstate, n_keys, S, slot_ids, cl, ws)
                if ev is not None:
                    ev[l][2].record(cur)
                smoe.smoe_stream_copy(desc, ly["host"], pool, S, cl, ws)
                if ev is not None:
                    ev[l][3].record(cur)
            if ev is not None:
                ev[l][0].record(cur)
            wdesc, wts_l, uids, wsl = (pdesc, pool, slot_ids, pws) if streamed else (desc, ly["weights"], ly["uid"], ws)
            if fused_norm and l + 1 < L:   # this layer's combine also writes layer l+1's input
                smoe.smoe_moe_ffn_batch_norm(wdesc, wts_l, xl, uids, nu, ly["off"], ly["tl"], ly["sl"], wt, h, xb,
                                             wsl, 1e-6, int(w.chain_center))
            else:
                smoe.smoe_moe_ffn_batch(wdesc, wts_l, xl, uids, nu, ly["off"], ly["tl"], ly["sl"], wt, h, wsl)
            if P:
                smoe.smoe_shared_expert_ffn(sdesc, ly["shared"], xl, h, sws)
            if ev is not None:
                ev[l][1].record(cur)

    smoe.smoe_clear_device_status(ws)
    if streamed:
        smoe.smoe_clear_device_status(pws)
    n_warm = max(3, args.warmup)
    for i in range(n_warm):
        step(x_of(i))
    bits = smoe.smoe_read_device_status(ws) | (smoe.smoe_read_device_status(pws) if streamed else 0)
    if bits:
        raise RuntimeError(f"device status {bits:#x} during warm-up")
    c2c_peak = _host_link_gbs(torch, dev) if streamed else None

    # ---- timed region: inputs resident in HBM
    def ffn_event():
        # recorded inside a captured graph: an external event record node keeps it timeable
        return torch.cuda.Event(enable_timing=True, external=not args.eager)

    # streamed: 3 extra graphs replayed as warm-up (each graph is one token of the sequence, so
    # the timed graphs must not be replayed before the timed region)
    n_graphs = args.steps + (3 if streamed else 0)
    evs = [[[ffn_event() for _ in range(4 if streamed else 2)] for _ in range(L)] for _ in range(n_graphs)]
    recs = [[(torch.zeros(1, dtype=torch.int32, device=dev), torch.zeros(1 + 2 * E, dtype=torch.int32, device=dev))
             for _ in range(L)] for _ in range(n_graphs)] if streamed else [None] * n_graphs
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # A step that reads less than ~1 GB (every routed expert distinct, plus the gate matrices)
    # could find the previous step's experts in the 129 MB L2: such steps are timed one by one,
    # with a 256 MiB write between them (outside their events) that evicts L2.
    eb = w.expert_bytes
    step_bytes_max = L * (min(B * K, E) * eb + w.shared_bytes + E * d * 4)
    flush = step_bytes_max < 1e9
    flush_buf = torch.empty(256 * 2**20 // 4, dtype=torch.int32, device=dev) if flush else None
    step_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(args.steps)] if flush else None
    graphs = []
    if not args.eager:
        # one CUDA graph per timed step (each with its own FFN events), captured from the
        # same library calls; replaying them removes the host launch gaps between kernels
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        for s in range(n_graphs):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                step(x_of(n_warm + s), evs[s], recs[s])
            graphs.append(g)
        stream.wait_stream(cap)
        for g in graphs[:3]:   # upload / warm the graphs
            g.replay()
        if streamed:   # the warm-up tokens; the timed graphs follow them in the sequence
            graphs, evs, recs = graphs[3:], evs[3:], recs[3:]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = start_clocks(dev, local) if rank == 0 else None
    time.sleep(0.3 if clocks else 0.0)
    t_start.record(stream)
    for s in range(args.steps):
        if flush:
            flush_buf.fill_(s)
            step_evs[s][0].record(stream)
        if graphs:
            graphs[s].replay()
        else:
            step(x_of(n_warm + s), evs[s], recs[s])
        if flush:
            step_evs[s][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop() if clocks else None
    if world > 1:
        dist.barrier()
    ms_total = (sum(a.elapsed_time(b) for a, b in step_evs) if flush else t_start.elapsed_time(t_end))
    ffn_ms = [evs[s][l][0].elapsed_time(evs[s][l][1]) for s in range(args.steps) for l in range(L)]
    ms_total = max_over_ranks(ms_total, world, dev)
    ms_step = ms_total / args.steps
    bits = smoe.smoe_read_device_status(ws) | (smoe.smoe_read_device_status(pws) if streamed else 0)
    if bits:
        raise RuntimeError(f"device status {bits:#x} in the timed region")

    # ---- algorithmic work (measured union sizes)
    if streamed:
        U = [int(recs[-1][l][0].item()) for l in range(L)]
        n_copied = sum(int(recs[s][l][1][0].item()) for s in range(args.steps) for l in range(L))
        n_routed = sum(int(recs[s][l][0].item()) for s in range(args.steps) for l in range(L))
        copy_ms = sum(evs[s][l][2].elapsed_time(evs[s][l][3]) for s in range(args.steps) for l in range(L))
    else:
        U = [int(ly["nu"].item()) for ly in layers]
    hbm, tf_burst, tf_sus, peak_kind = _peaks()
    # (+ the next layer's input, bf16, where the combine also writes it)
    ffn_bytes = [u * eb + w.shared_bytes + B * d * 2 + 2 * B * d * 4 + (B * d * 2 if fused_norm and l + 1 < L else 0)
                 for l, u in enumerate(U)]
    layer_bytes = [fb + E * d * 4 for fb in ffn_bytes]
    layer_flops = 6 * B * K * d * F + 6 * B * d * w.shared_ffn_dim + 2 * B * d * E
    t_roof_step = sum(max(bb / (hbm * 1e9), layer_flops / (tf_sus * 1e12)) for bb in layer_bytes)
    ffn_ms_mean = sum(ffn_ms) / len(ffn_ms)
    ffn_bytes_mean = sum(ffn_bytes) / len(ffn_bytes)
    ffn_flops = 6 * B * K * d * F + 6 * B * d * w.shared_ffn_dim
    # the FFN step's binding roof: union expert bytes at HBM bandwidth, or its flops at the
    # sustained tensor rate (fp16 and bf16 run at the same nominal rate)
    tensor_bound = ffn_flops / (tf_sus * 1e12) > ffn_bytes_mean / (hbm * 1e9)
    if tensor_bound:
        achieved = ffn_flops / (ffn_ms_mean * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": tf_sus, "unit": "TFLOP/s",
                "frac": achieved / tf_sus, "traffic": None, "peak_kind": f"{peak_kind} sustained bf16 dense"}
    else:
        achieved = ffn_bytes_mean / (ffn_ms_mean * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "traffic": None, "peak_kind": f"{peak_kind} copy bandwidth"}
    value = world * B * L / (ms_step * 1e-3)
    union_gbs = world * sum(U) * eb / (ms_step * 1e-3) / 1e9

    # ---- end to end through host buffers: pinned H2D of x, D2H of the final hidden state
    # (streamed: the tokens after the timed ones, one per step)
    tok0 = n_warm + 3 + args.steps
    x_host = (x_seq.cpu() if streamed else x_in.cpu()).pin_memory()

    def x_host_of(i):
        return x_host[i % T:i % T + 1] if streamed else x_host

    out_host = torch.empty(B, d, dtype=torch.float32).pin_memory()
    x_dev2 = torch.empty_like(x_in)
    e_s, e_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(2):
        x_dev2.copy_(x_host_of(tok0 + i), non_blocking=True)
        step(x_dev2)
        out_host.copy_(h, non_blocking=True)
    torch.cuda.synchronize()
    e2e_steps = max(3, min(args.steps, 10))
    e2e_total = 0.0
    e_s.record(stream)
    for i in range(e2e_steps):
        if flush:
            flush_buf.fill_(1)
            e_s.record(stream)
        x_dev2.copy_(x_host_of(tok0 + 2 + i), non_blocking=True)
        step(x_dev2)
        out_host.copy_(h, non_blocking=True)
        if flush:
            e_e.record(stream)
        torch.cuda.current_stream().synchronize()
        if flush:
            e2e_total += e_s.elapsed_time(e_e)
    if not flush:
        e_e.record(stream)
        torch.cuda.synchronize()
        e2e_total = e_s.elapsed_time(e_e)
    e2e_ms = e2e_total / e2e_steps
    e2e_value = world * B * L / (e2e_ms * 1e-3)

    if rank != 0:
        return
    # ---- CPU oracle on a bounded sample of the same workload (host cores, rank 0, N=1 only)
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        n = _sample_rows(w)
        host = {}

        def layer_source(l):
            if l not in host:
                ly = layers[l]
                host[l] = ({k: v.cpu() for k, v in ly["wts"].items()}, ly["gate"].cpu(),
                           None if ly["bias"] is None else ly["bias"].cpu(),
                           {k: v.cpu() for k, v in ly["shared"].tensors.items()} if ly["shared"] is not None
                           else None)
            return host[l]

        units, dt, cores = oracle_layers(w, x_in.view(torch.bfloat16)[:n].cpu(), layer_source, 12.0)
        del host
        cpu = {"value": units / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"first {n} of {B} tokens, {units // n} layer passes over the {L}-layer stack "
                         f"({units} token-layers), layer-major fp64 oracle, {dt:.1f} s"}
    rec = _traffic_from_profile(args.workload)
    traffic = None
    if rec is not None:
        # the capture is of one layer; scale to the timed layers' mean union by algorithmic bytes
        cap_bytes, cap_u = rec
        traffic = cap_bytes * ffn_bytes_mean / (cap_u * eb + w.shared_bytes + B * d * 2 + 2 * B * d * 4)
    ffn_roof = dict(roof, traffic=traffic if not tensor_bound else None,
                    kernel="expert FFN step (smoe_moe_ffn_batch: gather, gate/up+SwiGLU, down, combine"
                           + (", and smoe_shared_expert_ffn)" if P else ")"))
    stream_info = None
    if streamed:
        # the dominant kernel of a streamed step is the slot copy: host-link bound
        c2c = n_copied * eb / (copy_ms * 1e-3) / 1e9 if copy_ms > 0 else 0.0
        stream_info = {"slots": S, "keys": n_keys, "seq_rho": w.seq_rho,
                       "hit_rate": 1.0 - n_copied / max(1, n_routed),
                       "experts_copied_per_step": n_copied / args.steps,
                       "host_bytes_per_step": n_copied * eb / args.steps,
                       "ffn_roofline": ffn_roof}
        roof_line = {"bound": "c2c", "achieved": c2c, "peak": c2c_peak, "unit": "GB/s",
                     "frac": c2c / c2c_peak if c2c_peak else None, "traffic": None,
                     "peak_kind": "measured in this run: pinned host -> device cudaMemcpyAsync, 1 GiB, best of 3",
                     "kernel": "smoe_stream_copy (missed experts, pinned host memory -> HBM slots)"}
    else:
        roof_line = ffn_roof
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp16", "data": "synthetic",
        "config": {"workload": w.name, "tokens": B, "layers": L, "d_model": d, "experts": E, "top_k": K,
                   "spec_ranks": w.spec, "shared_ffn_dim": w.shared_ffn_dim, "stream_slots": S,
                   "norm_topk_prob": w.norm_topk_prob,
                   "ffn_dim": F, "layout": w.layout, "weights": "4-bit affine g64, bf16 scales/biases",
                   "l2": (f"L2 flushed between timed steps (256 MiB write outside the step events): a step "
                          f"reads at most {step_bytes_max / 1e6:.0f} MB" if flush else
                          f"inputs larger than L2: {sum(U) * eb / 1e9:.1f} GB of union expert weights per step"),
                   "parallelism": f"replicas x{world}",
                   "launch": "eager" if args.eager else "one CUDA graph per step, replayed"},
        "union_expert_gbs": union_gbs,
        "union_sizes": U,
        # streamed: the step cannot beat its bytes over the host link either
        "step_roofline_frac": max(t_roof_step, (n_copied * eb / args.steps / (c2c_peak * 1e9)) if streamed else 0.0)
                              / (ms_step * 1e-3),
        "roofline": roof_line,
        "stream": stream_info,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": B * d * 2, "d2h_bytes_per_step": B * d * 4},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="prefill64")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-seconds", type=float, default=60.0,
                    help="reference arm: seconds of oracle work over all its steps (warm-up included)")
    ap.add_argument("--eager", action="store_true", help="launch the timed steps directly instead of replaying "
                                                         "one captured CUDA graph per step")
    ap.add_argument("--layers", type=int, default=0, help="profiling only: run the first N layers of the stack")
    args = ap.parse_args()
    from moe_expert_routing_gb300 import workload as W
    w = W.WORKLOADS[args.workload]
    if args.layers:
        w = W.scaled(w, layers=args.layers)
    world, rank, local = _dist()
    if args.impl == "reference":
        if rank == 0:
            run_reference(args, w)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    try:
        run_gpu(args, w, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
