#!/usr/bin/env python3
"""MoE-layer throughput on B300: tokens/s through sparse MoE FFN layers of the
Flint shape, with the achieved HBM GB/s or bf16 TFLOP/s of the layer and of its
dominant kernel against the measured peaks.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Headline workload (default): the 47-layer MoE stack of the Flint decoder
(d = 2048, 256 routed experts + 1 shared, expert FFN 512, top-6), T = 2048
tokens, router bias drawn so expert load follows Zipf(1.1), residual add
between layers, layers chained (layer l + 1 reads layer l's output).  One
step = one pass of all 47 layers (router, top-k, grouping, expert gate/up +
SwiGLU, down + gated combine + shared expert + residual); value = tokens x
layers / time.  The other configurations (decode T = 1, 8, 32, 64; prefill
T = 4096 and 16384; NVFP4 decode T = 32) are measured in the same run and
reported under "sweep", each against its binding roof.  Weights and
activations are seeded synthetic draws made on the device.

With --gpus N (N > 1) the script starts N ranks itself under
torch.distributed.run; every rank runs an independent replica on its own GPU
(the layer has no cross-GPU step); value = units of all ranks / slowest rank's
time.
"""
import argparse
import hashlib
import json
import math
import os
import socket
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# name: (layer kind, tokens, layers in the rotation, chained)
WORKLOADS = {
    "stack47": ("stack", 2048, 47, True),
    "decode1": ("bf16", 1, 16, False),
    "decode8": ("bf16", 8, 16, False),
    "decode32": ("bf16", 32, 16, False),
    "decode64": ("bf16", 64, 16, False),
    "prefill4096": ("bf16", 4096, 8, False),
    "prefill16384": ("bf16", 16384, 4, False),   # ~384 tokens per expert: past the ridge, tensor peak binds
    "nvfp4_32": ("nvfp4", 32, 32, False),
}
DEFAULT = "stack47"
SWEEP = ["decode1", "decode8", "decode32", "decode64", "prefill4096", "prefill16384", "nvfp4_32"]
# measured on the headline's resident 47-layer stack: the persistent decode kernel
STACK_DECODE = {"stack47_decode1": 1, "stack47_decode8": 8}
# the 4-bit output layer (vocabulary 146,432 x d 2048, NVFP4), four copies in rotation
HEAD = {"lmhead1": 1, "lmhead8": 8}
HEAD_COPIES = 4
# sliding-window attention at decode: B sequences at position 4096 (full 513-token window), 8 layers in rotation
ATTN = {"attn1": 1, "attn8": 8}
ATTN_LAYERS = 8
ATTN_POS = 4096
D, E_ROUTED, F_EXP, TOPK = 2048, 256, 512, 6
B_EXP_BF16 = 3 * D * F_EXP * 2                       # bytes of one expert's three bf16 matrices
B_EXP_NVFP4 = 3 * (D * F_EXP // 2 + D * F_EXP // 16 + 4)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        m = json.load(open(p))
        return {"hbm_gbs": m["hbm_gbs"], "bf16_tflops": m["bf16_tflops"],
                "bf16_tflops_sustained": m.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ helpers
def csrc_sha():
    """Hash of every kernel source: a traffic figure is kept only while the code it was taken on is unchanged."""
    d = os.path.join(ROOT, "sparse_moe_transformer_02_b300", "csrc")
    h = hashlib.sha256()
    for f in sorted(f for f in os.listdir(d) if f.endswith((".cu", ".cuh"))):
        h.update(open(os.path.join(d, f), "rb").read())
    return h.hexdigest()[:16]


def dram_traffic(kernel, workload):
    """Per-launch DRAM bytes from the committed ncu summary, if taken on the current source."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(f"{kernel}|{workload}")
    if not rec or rec.get("src_sha") != csrc_sha():
        return None
    return rec.get("bytes_per_launch")


def max_over_ranks(v, device):
    """The largest of the ranks' values, on every rank (v itself without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return v
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, t_max_s, world):
    """Whole-job rate of independent replicas: the units all ranks processed over the slowest rank's time."""
    return world * units_per_rank / t_max_s


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def launcher_command(argv, n):
    """The torch.distributed.run command that starts n ranks of this script with the same arguments."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
            "--master-addr", "127.0.0.1", "--master-port", str(free_port()), os.path.abspath(__file__)] + list(argv)


def layer_bytes_flops(kind, T, U_mean):
    """Algorithmic bytes and flops of one layer: the touched experts' weights
    (realised routing) + the shared expert + router + x in and y out; bf16
    tensor flops of the k + 1 expert passes + the fp32 router's."""
    b_exp = B_EXP_NVFP4 if kind == "nvfp4" else B_EXP_BF16
    byt = (U_mean + 1) * b_exp + 4 * D * E_ROUTED + 4 * E_ROUTED + T * D * 2 * 2
    flops = 2 * T * (TOPK + 1) * 3 * D * F_EXP + 2 * T * D * E_ROUTED
    return byt, flops


def kernel_bytes_flops(kname, kind, T, U_mean):
    """Algorithmic bytes and tensor flops of one launch of a kernel of the layer."""
    if kname == "fused":                       # the persistent kernel does the whole layer
        return layer_bytes_flops(kind, T, U_mean)
    b_exp = B_EXP_NVFP4 if kind == "nvfp4" else B_EXP_BF16
    byt = {"route": 4 * D * E_ROUTED + 4 * E_ROUTED + T * D * 2,
           "gemv_gateup": (U_mean + 1) * b_exp * 2 / 3 + T * D * 2,
           "gemv_down": (U_mean + 1) * b_exp / 3 + T * D * 2,
           "tc_gateup": (U_mean + 1) * b_exp * 2 / 3 + T * D * 2,
           "tc_down": (U_mean + 1) * b_exp / 3,
           "tc_gather": 2 * T * TOPK * D * 2,
           "tc_finalize": T * D * (4 + 2)}.get(kname, 0)
    flops = {"tc_gateup": 2 * T * (TOPK + 1) * 2 * D * F_EXP,
             "tc_down": 2 * T * (TOPK + 1) * D * F_EXP,
             "gemv_gateup": 2 * T * (TOPK + 1) * 2 * D * F_EXP,
             "gemv_down": 2 * T * (TOPK + 1) * D * F_EXP,
             "route": 2 * T * D * E_ROUTED}.get(kname, 0)
    return byt, flops


def binding(byt, flops, t_s, pk):
    """The binding roof of work that moves byt bytes and does flops bf16 flops in t_s seconds."""
    t_mem = byt / (pk["hbm_gbs"] * 1e9)
    t_tc = flops / (pk["bf16_tflops"] * 1e12)
    if t_tc > t_mem:
        ach = flops / t_s / 1e12
        return {"bound": "tensor", "achieved": round(ach, 2), "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(ach / pk["bf16_tflops"], 4), "t_lb_us": round(t_tc * 1e6, 2)}
    ach = byt / t_s / 1e9
    return {"bound": "hbm", "achieved": round(ach, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": round(ach / pk["hbm_gbs"], 4), "t_lb_us": round(t_mem * 1e6, 2)}


# ------------------------------------------------------------------ layer sets on the device
def make_layer_set(kind, n_layers, device, seed):
    """n_layers independent Flint-shaped layers on the device.  bf16 and stack
    layers are drawn there; NVFP4 layers share one host-quantised expert set,
    copied to distinct buffers per layer (so every layer still reads HBM)."""
    from sparse_moe_transformer_02_b300 import binding as B
    from sparse_moe_transformer_02_b300 import inputs as I
    spec = {"bf16": I.FLINT_BF16, "nvfp4": I.FLINT_NVFP4, "stack": I.FLINT_STACK_ZIPF}[kind]
    if kind == "nvfp4":
        base = B.upload_layer(I.make_layer(spec, seed=seed), device)
        layers = []
        for li in range(n_layers):
            w = {k: (t.clone() if k not in ("router_w", "router_b") else t) for k, t in base.items()}
            layers.append(w)
        return spec, layers
    return spec, [I.make_layer_torch(spec, seed=seed, layer=li, device=device) for li in range(n_layers)]


def measure(args, name, spec, kind, wts, T, chain, device, stream, rank, world, steps, sample_clocks,
            want_e2e):
    """Time one workload on an existing layer set; returns the result dict."""
    import torch
    import torch.distributed as dist
    from sparse_moe_transformer_02_b300 import binding as B
    from sparse_moe_transformer_02_b300 import inputs as I

    handles = []
    with torch.cuda.stream(stream):
        for w in wts:
            handles.append(B.layer_from_spec(spec, w, max_tokens=max(T, 64), stream=stream,
                                             path={"auto": 0, "gemv": 1, "tc": 2}[args.path],
                                             deterministic=args.deterministic))
    x = I.make_tokens_torch(spec, seed=args.seed + 77 + rank + T, T=T, device=device)
    ys = [torch.empty_like(x) for _ in handles]
    ins = [x] + ys[:-1] if chain else [x] * len(handles)
    torch.cuda.synchronize()

    def step():
        for h, xi, y in zip(handles, ins, ys):
            h.forward(xi, y, stream=stream)

    step()
    stream.synchronize()
    for h in handles:
        st = h.check(stream)
        if st != B.MOE_OK:
            raise RuntimeError(f"{name}: device error {B.moe_status_string(st)}")
    # realised routing: distinct experts per layer (on each layer's actual input)
    U = []
    for h, xi in zip(handles, ins):
        _, _, cnt = h.route(xi, stream=stream)
        stream.synchronize()
        U.append(int((cnt > 0).sum().item()))
    Umean = sum(U) / len(U)

    for _ in range(max(args.warmup, 1)):
        step()
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    # at least ~0.4 s of timed work so that the clock samples mean something
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        graph.replay()
        ev1.record(stream)
    ev1.synchronize()
    one = ev0.elapsed_time(ev1)
    n_steps = steps if steps else max(10, int(math.ceil(400.0 / max(one, 1e-3))))

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device()) if (rank == 0 and sample_clocks) else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(n_steps):
            graph.replay()
        ev1.record(stream)
    ev1.synchronize()
    torch.cuda.synchronize()
    t_ms = ev0.elapsed_time(ev1)
    clocks = sampler.stop() if sampler else None
    t_ms = max_over_ranks(t_ms, device)
    if world > 1:
        dist.barrier()
    del graph

    n_layers = len(handles)
    ms_step = t_ms / n_steps
    value = job_throughput(T * n_layers * n_steps, t_ms / 1e3, world)
    pk = peaks()

    # per-kernel timing: a separate eager pass with event pairs around each launch
    for h in handles:
        B._ok(B.moe_profile_enable(h.h, 1, 64), "moe_profile_enable")
    prof_steps = 3
    for _ in range(prof_steps):
        step()
    tot = {}
    for h in handles:
        st, r = B.moe_profile_read(h.h)
        B._ok(st, "moe_profile_read")
        for kname, (ms, n) in r.items():
            a = tot.setdefault(kname, [0.0, 0])
            a[0] += ms
            a[1] += n
        B.moe_profile_enable(h.h, 0, 0)
    launches_per_fwd = sum(v[1] for v in tot.values()) / (prof_steps * n_layers)
    dom = max(tot, key=lambda kk: tot[kk][0])
    dom_ms = tot[dom][0] / max(tot[dom][1], 1)
    kb, kf = kernel_bytes_flops(dom, kind, T, Umean)
    roof = binding(kb, kf, dom_ms * 1e-3, pk)
    roof.update({"kernel": dom, "kernel_ms": round(dom_ms, 5), "traffic": dram_traffic(dom, name),
                 "algorithmic_bytes": int(kb), "flops": int(kf), "peak_source": pk["source"],
                 "per_kernel_ms": {kk: round(v[0] / max(v[1], 1), 5) for kk, v in tot.items() if v[1]}})

    lb, lf = layer_bytes_flops(kind, T, Umean)
    t_layer = ms_step / 1e3 / n_layers
    lay = binding(lb, lf, t_layer, pk)
    layer = {"us_per_layer": round(t_layer * 1e6, 2), "distinct_experts_mean": round(Umean, 2),
             "algorithmic_bytes": int(lb), "flops": int(lf), "bound": lay["bound"],
             "roof_frac": lay["frac"], "t_lb_us": lay["t_lb_us"],
             "hbm_gbs": round(lb / t_layer / 1e9, 1),
             "hbm_frac_of_measured": round(lb / t_layer / 1e9 / pk["hbm_gbs"], 4),
             "hbm_frac_of_8tbs": round(lb / t_layer / 1e9 / 8000.0, 4),
             "tflops": round(lf / t_layer / 1e12, 2),
             "tensor_frac_of_measured": round(lf / t_layer / 1e12 / pk["bf16_tflops"], 4)}

    e2e = None
    if want_e2e:
        # end to end with host buffers, host<->device copies inside the timed
        # region: independent layers go through moe_forward_host (copy in,
        # forward, copy out); the chained stack copies its input in and its
        # output out around the chain
        xh = x.cpu().pin_memory()
        yh = torch.empty_like(xh).pin_memory()
        for h in handles[:2]:
            h.forward_host(xh, yh, stream=stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e_steps = max(1, min(n_steps, 10))
        t0 = time.perf_counter()
        for _ in range(e_steps):
            if chain:
                with torch.cuda.stream(stream):
                    x.copy_(xh, non_blocking=True)
                    step()
                    yh.copy_(ys[-1], non_blocking=True)
                stream.synchronize()
            else:
                for h in handles:
                    h.forward_host(xh, yh, stream=stream)
        e_s = max_over_ranks(time.perf_counter() - t0, device)
        io_layers = 1 if chain else n_layers
        e2e = {"value": round(job_throughput(T * n_layers * e_steps, e_s, world), 1), "unit": "tokens/s",
               "h2d_bytes_per_step": T * spec.d * 2 * io_layers, "d2h_bytes_per_step": T * spec.d * 2 * io_layers}

    for h in handles:
        h.close()
    del ys, ins, x
    return {"name": name, "value": value, "tokens_per_s": round(value, 1), "T": T, "layers": n_layers,
            "steps": n_steps, "ms_per_step": round(ms_step, 5), "layer": layer, "roofline": roof,
            "clocks": clocks, "e2e": e2e, "launches_per_forward": launches_per_fwd,
            "gpu_launches": int(round(n_steps * n_layers * launches_per_fwd))}


def measure_stack_decode(args, name, spec, wts, T, device, stream):
    """The persistent kernel over the whole stack (one launch per pass), T tokens."""
    import torch
    from sparse_moe_transformer_02_b300 import binding as B
    from sparse_moe_transformer_02_b300 import inputs as I
    st = B.MoeStack(spec, wts, max_tokens=max(T, 8), stream=stream)
    if not st.persistent(T):
        st.close()
        return {"skipped": "the persistent kernel does not serve this shape"}
    x = I.make_tokens_torch(spec, seed=args.seed + 500 + T, T=T, device=device)
    y = torch.empty_like(x)
    with torch.cuda.stream(stream):
        _, _, it, _ = st.forward(x, trace=True, stream=stream)
    stream.synchronize()
    if st.check(stream) != B.MOE_OK:
        raise RuntimeError(f"{name}: device error")
    U = [len(set(it[l].flatten().tolist())) for l in range(st.L)]
    Umean = sum(U) / len(U)
    for _ in range(args.warmup):
        st.forward(x, y, stream=stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        st.forward(x, y, stream=stream)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = 50
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.3)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(n):
            graph.replay()
        ev1.record(stream)
    ev1.synchronize()
    clocks = sampler.stop()
    t = ev0.elapsed_time(ev1) / 1e3 / n
    del graph
    st.close()
    pk = peaks()
    lb, lf = layer_bytes_flops("stack", T, Umean)
    t_layer = t / len(wts)
    lay = binding(lb, lf, t_layer, pk)
    roof = binding(lb * len(wts), lf * len(wts), t, pk)
    roof.update({"kernel": "stack_decode_kernel", "kernel_ms": round(t * 1e3, 5), "traffic": dram_traffic("stack_decode", name),
                 "algorithmic_bytes": int(lb * len(wts)), "flops": int(lf * len(wts)), "peak_source": pk["source"]})
    return {"name": name, "tokens_per_s": round(T / t, 1), "layer_tokens_per_s": round(T * len(wts) / t, 1), "T": T,
            "layers": len(wts), "steps": n, "ms_per_step": round(t * 1e3, 5),
            "layer": {"us_per_layer": round(t_layer * 1e6, 2), "distinct_experts_mean": round(Umean, 2),
                      "algorithmic_bytes": int(lb), "bound": lay["bound"], "roof_frac": lay["frac"],
                      "t_lb_us": lay["t_lb_us"], "hbm_gbs": round(lb / t_layer / 1e9, 1),
                      "hbm_frac_of_measured": round(lb / t_layer / 1e9 / pk["hbm_gbs"], 4),
                      "hbm_frac_of_8tbs": round(lb / t_layer / 1e9 / 8000.0, 4)},
            "roofline": roof, "clocks": clocks, "launches_per_forward": 1, "gpu_launches": n}


def measure_head(args, name, T, device, stream):
    """The 4-bit output layer at T tokens, HEAD_COPIES copies of the head in rotation."""
    import torch
    from sparse_moe_transformer_02_b300 import binding as B
    from sparse_moe_transformer_02_b300 import inputs as I
    h = I.make_head(seed=args.seed)
    base = [torch.from_numpy(h["packed"]).to(device), torch.from_numpy(h["scales"]).to(device),
            torch.from_numpy(h["tscale"]).to(device)]
    heads = [B.LmHead(*(t.clone() for t in base), max_tokens=8) for _ in range(HEAD_COPIES)]
    V, d = h["packed"].shape[0], h["packed"].shape[1] * 2
    x = I.make_tokens_torch(I.FLINT_BF16, seed=args.seed + 900 + T, T=T, device=device)
    outs = [torch.empty((T, V), dtype=torch.float32, device=device) for _ in heads]

    def step():
        for hd, o in zip(heads, outs):
            hd.forward(x, o, stream=stream)
    step()
    stream.synchronize()
    for hd in heads:
        if hd.check(stream) != B.MOE_OK:
            raise RuntimeError(f"{name}: device error")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = 100
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.3)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(n):
            graph.replay()
        ev1.record(stream)
    ev1.synchronize()
    clocks = sampler.stop()
    t = ev0.elapsed_time(ev1) / 1e3 / n / len(heads)
    del graph
    for hd in heads:
        hd.close()
    pk = peaks()
    byt = V * d // 2 + V * d // 16 + 4 + T * d * 2 + T * V * 4
    flops = 2 * T * V * d
    roof = binding(byt, 0, t, pk)
    roof.update({"kernel": "lm_head_kernel", "kernel_ms": round(t * 1e3, 5), "traffic": dram_traffic("lm_head", name),
                 "algorithmic_bytes": int(byt), "flops": int(flops), "peak_source": pk["source"]})
    return {"name": name, "tokens_per_s": round(T / t, 1), "T": T, "vocab": V, "d": d, "us_per_call": round(t * 1e6, 2),
            "roofline": roof, "clocks": clocks, "launches_per_forward": 1, "gpu_launches": n * len(heads)}


def measure_attn(args, name, Bn, device, stream):
    """Sliding-window GQA attention at decode, Bn sequences, ATTN_LAYERS layers' weights and caches in rotation."""
    import numpy as np
    import torch
    from sparse_moe_transformer_02_b300 import binding as B
    from sparse_moe_transformer_02_b300 import inputs as I
    A = I.FLINT_ATTN

    def dev(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
        return torch.from_numpy(a).to(device)
    base = {k: dev(v) for k, v in I.make_attention(seed=args.seed).items()}
    kc0, vc0 = (dev(t) for t in I.make_kv_cache(args.seed, Bn, A["window"]))
    layers = []
    for _ in range(ATTN_LAYERS):
        w = {k: t.clone() for k, t in base.items()}
        layers.append((B.MoeAttn(w, A["d"], A["n_q"], A["n_kv"], A["window"], max_batch=8), kc0.clone(),
                       vc0.clone()))
    x = I.make_tokens_torch(I.FLINT_BF16, seed=args.seed + 41, T=Bn, device=device)
    pos = torch.full((Bn,), ATTN_POS, dtype=torch.int32, device=device)
    ys = [torch.empty_like(x) for _ in layers]

    def step():
        for (at, kc, vc), y in zip(layers, ys):
            at.decode(x, pos, kc, vc, y, stream=stream)
    step()
    stream.synchronize()
    for at, _, _ in layers:
        if at.check(stream) != B.MOE_OK:
            raise RuntimeError(f"{name}: device error")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = 100
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.3)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(n):
            graph.replay()
        ev1.record(stream)
    ev1.synchronize()
    clocks = sampler.stop()
    t = ev0.elapsed_time(ev1) / 1e3 / n / len(layers)
    del graph
    for at, _, _ in layers:
        at.close()
    pk = peaks()
    d, qd, kvd, W = A["d"], A["n_q"] * A["hd"], A["n_kv"] * A["hd"], A["window"]
    byt = (qd + 2 * kvd) * d * 2 + d * qd * 2 + Bn * (W * kvd * 2 * 2 + 2 * d * 2 + kvd * 2 * 2) + 4 * Bn
    flops = 2 * Bn * ((qd + 2 * kvd) * d + d * qd + 2 * W * qd)
    roof = binding(byt, 0, t, pk)
    roof.update({"kernel": "attn_decode_kernel", "kernel_ms": round(t * 1e3, 5), "traffic": dram_traffic("attn", name),
                 "algorithmic_bytes": int(byt), "flops": int(flops), "peak_source": pk["source"]})
    return {"name": name, "tokens_per_s": round(Bn / t, 1), "B": Bn, "position": ATTN_POS,
            "us_per_layer": round(t * 1e6, 2), "roofline": roof, "clocks": clocks, "launches_per_forward": 1,
            "gpu_launches": n * len(layers)}


# ------------------------------------------------------------------ the CPU oracle as a baseline
def oracle_rates(kind, T, seed, budget_s, steps=1, procs=1):
    """The float64 oracle on bounded samples of the workload, in a fresh
    interpreter that never touches CUDA: one layer of the workload's kind,
    tokens split over `procs` worker processes (one BLAS thread each).
    Returns ([tokens/s per step], description)."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-sample", kind, str(T), str(seed), str(budget_s),
           str(steps), str(procs)]
    res = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=1800)
    if res.returncode != 0:
        raise RuntimeError("oracle sample failed: " + res.stderr[-2000:])
    r = json.loads(res.stdout.strip().splitlines()[-1])
    return r["rates"], r["sample"]


def _oracle_worker(args):
    x, k, residual = args
    W = _ORACLE_STATE["W"]
    import oracle
    t0 = time.perf_counter()
    oracle.moe_forward(x, W, k, residual=residual)
    return time.perf_counter() - t0


_ORACLE_STATE = {}


def oracle_sample_main(kind, T, seed, budget_s, steps, procs):
    """Child side of oracle_rates: prints {"rates", "sample"}.  The layer is
    made once; worker processes are forked from this CUDA-free interpreter
    after that, so they share it."""
    import multiprocessing as mp
    import oracle
    from sparse_moe_transformer_02_b300 import inputs as I
    spec = {"bf16": I.FLINT_BF16, "nvfp4": I.FLINT_NVFP4, "stack": I.FLINT_STACK_ZIPF}[kind]
    L = I.make_layer(spec, seed=seed)
    _ORACLE_STATE["W"] = oracle.LayerWeights(L)
    x = I.make_tokens(spec, seed=seed, T=max(T, 1))
    chunk = min(T, 4)
    pool = mp.get_context("fork").Pool(procs) if procs > 1 else None
    rates, total_tok, total_t = [], 0, 0.0
    pos = 0
    for _ in range(steps):
        done, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < budget_s:
            jobs = []
            for _ in range(procs):
                jobs.append((x[pos:pos + chunk], spec.top_k, spec.add_residual))
                pos = (pos + chunk) % max(T - chunk + 1, 1)
            if pool:
                pool.map(_oracle_worker, jobs)
            else:
                _oracle_worker(jobs[0])
            done += chunk * len(jobs)
        dt = time.perf_counter() - t0
        rates.append(done / dt)
        total_tok += done
        total_t += dt
    if pool:
        pool.close()
        pool.join()
    print(json.dumps({"rates": rates,
                      "sample": f"{total_tok} tokens of the workload's {T} ({chunk} per call) through one layer "
                                f"({kind} weights), float64 numpy oracle, {procs} process(es) x 1 BLAS thread, "
                                f"{total_t:.1f} s"}))


def cpu_baseline(kind, T, seed):
    """The oracle single-threaded and on all host cores (token-parallel processes)."""
    cores = os.cpu_count() or 1
    out = {"kind": "oracle", "unit": "tokens/s", "host_cores": cores}
    r1, s1 = oracle_rates(kind, T, seed, budget_s=10.0)
    out["single_thread"] = {"value": round(r1[0], 3), "cores": 1, "sample": s1}
    rn, sn = oracle_rates(kind, T, seed, budget_s=10.0, procs=cores)
    out.update({"value": round(rn[0], 3), "cores": cores, "sample": sn})
    return out


# ------------------------------------------------------------------ our arm
def run_ours(args, rank, world, local_rank):
    import torch
    from sparse_moe_transformer_02_b300 import build

    build.build()
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    stream = torch.cuda.Stream(device)

    kind, T, n_layers, chain = WORKLOADS[args.workload]
    if args.layers:
        n_layers = args.layers
    spec, wts = make_layer_set(kind, n_layers, device, seed=args.seed + rank)
    head = measure(args, args.workload, spec, kind, wts, T, chain, device, stream, rank, world, args.steps,
                   sample_clocks=True, want_e2e=True)
    sweep = {}
    if args.sweep and world == 1 and kind == "stack" and len(wts) == WORKLOADS["stack47"][2]:
        for wname, Tn in STACK_DECODE.items():
            sweep[wname] = measure_stack_decode(args, wname, spec, wts, Tn, device, stream)
    del wts
    torch.cuda.empty_cache()

    if args.sweep and world == 1:
        sets = {}
        for wname in SWEEP:
            if wname == args.workload:
                continue
            k2, T2, n2, ch2 = WORKLOADS[wname]
            key = (k2, n2)
            if key not in sets:
                sets.clear()
                torch.cuda.empty_cache()
                sets[key] = make_layer_set(k2, n2, device, seed=args.seed + 1)
            sp2, w2 = sets[key]
            r = measure(args, wname, sp2, k2, w2, T2, ch2, device, stream, rank, world, 0, sample_clocks=True,
                        want_e2e=False)
            r.pop("e2e", None)
            r.pop("value", None)
            sweep[wname] = r
        sets.clear()
        torch.cuda.empty_cache()
        for wname, Tn in HEAD.items():
            sweep[wname] = measure_head(args, wname, Tn, device, stream)
        for wname, Bn in ATTN.items():
            sweep[wname] = measure_attn(args, wname, Bn, device, stream)
        torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        try:
            cpu = cpu_baseline(kind, T, seed=args.seed)
        except Exception as exc:          # the GPU numbers stand without it
            cpu = {"kind": "oracle", "value": None, "error": str(exc)[-300:]}

    if rank == 0:
        out = {"metric": "MoE-layer tokens/s", "value": round(head["value"], 1), "unit": "tokens/s",
               "n_gpus": world, "steps": head["steps"], "warmup": args.warmup,
               "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
               "vs_baseline": None, "dtype": "nvfp4" if kind == "nvfp4" else "bf16",
               "data": "synthetic (seeded N(0,0.02) weights and N(0,1) activations drawn on the device)",
               "config": {"workload": f"flint_moe_{args.workload}", "tokens": T, "d": spec.d,
                          "experts": spec.num_experts, "shared_experts": 1, "top_k": spec.top_k,
                          "expert_ffn": spec.ffn, "weights": kind, "layers_per_step": head["layers"],
                          "chained": chain, "router_bias": spec.bias, "residual": bool(spec.add_residual),
                          "l2": f"inputs larger than L2: {head['layers']} distinct layers' weights per step",
                          "parallelism": f"replicas{world}", "path": args.path, "deterministic": bool(args.deterministic)},
               "layer": head["layer"], "roofline": head["roofline"], "cpu_baseline": cpu, "e2e": head["e2e"],
               "gpu_launches": head["gpu_launches"], "clocks": head["clocks"]}
        if sweep:
            out["sweep"] = sweep
        print(json.dumps(out), flush=True)


def run_only(args):
    """One sweep entry alone (for profiling): prints its result as a JSON line."""
    import torch
    from sparse_moe_transformer_02_b300 import build
    build.build()
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    stream = torch.cuda.Stream(device)
    if args.only in STACK_DECODE:
        spec, wts = make_layer_set("stack", args.layers or WORKLOADS["stack47"][2], device, seed=args.seed)
        r = measure_stack_decode(args, args.only, spec, wts, STACK_DECODE[args.only], device, stream)
    elif args.only in HEAD:
        r = measure_head(args, args.only, HEAD[args.only], device, stream)
    elif args.only in ATTN:
        r = measure_attn(args, args.only, ATTN[args.only], device, stream)
    else:
        kind, T, n, chain = WORKLOADS[args.only]
        spec, wts = make_layer_set(kind, args.layers or n, device, seed=args.seed)
        r = measure(args, args.only, spec, kind, wts, T, chain, device, stream, 0, 1, 0, True, False)
    print(json.dumps(r), flush=True)


# ------------------------------------------------------------------ reference arm (the CPU oracle)
def run_reference(args, rank):
    if rank != 0:
        return
    kind, T, _, chain = WORKLOADS[args.workload]
    cores = os.cpu_count() or 1
    t0 = time.perf_counter()
    rates, sample = oracle_rates(kind, T, args.seed, budget_s=2.0, steps=args.warmup + args.steps, procs=cores)
    total = time.perf_counter() - t0
    timed = rates[args.warmup:]
    v = statistics.median(timed)
    out = {"impl": "reference", "metric": "MoE-layer tokens/s", "value": round(v, 3), "unit": "tokens/s",
           "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(1e3 * total / max(args.steps + args.warmup, 1), 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": f"flint_moe_{args.workload}", "tokens": T, "weights": kind, "chained": chain},
           "cpu_baseline": {"kind": "oracle", "cores": cores, "sample": sample, "value": round(v, 3),
                            "unit": "tokens/s"},
           "e2e": {"value": round(v, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


# ------------------------------------------------------------------ rank plumbing self-test (CPU)
def run_rank_selftest(rank, world):
    """Exercises the multi-rank plumbing without a GPU: gloo ranks, each
    'times' a fixed amount of host work, max over ranks, job throughput."""
    import torch
    import torch.distributed as dist
    dev = torch.device("cpu")
    t = 0.25 * (rank + 1)
    t_max = max_over_ranks(t, dev)
    if rank == 0:
        print(json.dumps({"metric": "selftest units/s", "value": job_throughput(100, t_max, world),
                          "n_gpus": world, "t_max": t_max}), flush=True)


def main():
    if len(sys.argv) > 1 and sys.argv[1] == "--oracle-sample":
        a = sys.argv[2:]
        oracle_sample_main(a[0], int(a[1]), int(a[2]), float(a[3]), int(a[4]), int(a[5]))
        return
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT, choices=sorted(WORKLOADS))
    ap.add_argument("--layers", type=int, default=0)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-sweep", dest="sweep", action="store_false")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--path", default="auto", choices=["auto", "gemv", "tc"])
    ap.add_argument("--deterministic", action="store_true",
                    help="the tcgen05 paths' fixed-order combine (moe_config.deterministic)")
    ap.add_argument("--only", default=None,
                    choices=sorted(list(WORKLOADS) + list(STACK_DECODE) + list(HEAD) + list(ATTN)),
                    help="run one sweep entry alone and print its result (profiling)")
    ap.add_argument("--rank-selftest", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # start the ranks ourselves, one per GPU, and pass their exit status on
        sys.exit(subprocess.call(launcher_command(sys.argv[1:], args.gpus)))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if args.only:
        run_only(args)
        return
    import torch.distributed as dist
    if args.rank_selftest:
        if world > 1:
            dist.init_process_group("gloo")
        try:
            run_rank_selftest(rank, world)
        finally:
            if world > 1:
                dist.destroy_process_group()
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
