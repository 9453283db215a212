#!/usr/bin/env python3
"""MoE-layer throughput on B300: tokens/s through one sparse MoE FFN layer,
with the achieved HBM GB/s (decode) or bf16 TFLOP/s (prefill) of the
dominant kernel against the measured peak.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one forward pass of the whole layer (router, top-k, grouping,
expert gate/up + SwiGLU, down + gated combine + shared expert) through L
distinct layers' weights, so the weights streamed per step are far larger
than L2 and every layer reads HBM.  Inputs are seeded synthetic tensors with
the Flint-shaped layer's sizes (d=2048, 256 routed experts + 1 shared,
expert FFN 512, top-6); weights are drawn on the device.

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the layer has no cross-GPU step); value = tokens of all ranks / max time.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOADS = {
    # name: (layer spec name, tokens, layers in the rotation)
    "decode64": ("bf16", 64, 16),
    "decode32": ("bf16", 32, 16),
    "decode8": ("bf16", 8, 16),
    "decode1": ("bf16", 1, 16),
    "prefill4096": ("bf16", 4096, 8),
    "prefill16384": ("bf16", 16384, 4),   # ~384 tokens per expert: past the ridge, tensor peak binds
    "nvfp4_32": ("nvfp4", 32, 32),
    "stack47": ("stack", 2048, 47),      # 47 chained layers, residual adds, Zipf(1.1) load
}
DEFAULT = "decode64"
SWEEP = ["decode1", "decode8", "decode32"]
B_EXP_BF16 = 3 * 2048 * 512 * 2                    # bytes of one expert's three matrices
B_EXP_NVFP4 = 3 * (2048 * 512 // 2 + 2048 * 512 // 16 + 4)


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
def src_sha(*files):
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, "sparse_moe_transformer_02_b300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def csrc_sha():
    """Hash of every kernel source: a traffic figure is kept only while the code it was taken on is unchanged."""
    d = os.path.join(ROOT, "sparse_moe_transformer_02_b300", "csrc")
    return src_sha(*sorted(f for f in os.listdir(d) if f.endswith((".cu", ".cuh"))))


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


def make_device_layers(kind, n_layers, device, seed):
    """n_layers independent Flint-shaped layers drawn on the device (bf16), or NVFP4
    layers that share one host-quantised expert set copied to distinct buffers."""
    import torch
    from sparse_moe_transformer_02_b300 import binding as B
    from sparse_moe_transformer_02_b300 import inputs as I
    spec = {"bf16": I.FLINT_BF16, "nvfp4": I.FLINT_NVFP4, "stack": I.FLINT_STACK_ZIPF}[kind]
    E, d, F, Fs = spec.num_experts, spec.d, spec.ffn, spec.shared_ffn
    g = torch.Generator(device=device)
    layers = []
    base = None
    if kind == "nvfp4":
        base = B.upload_layer(I.make_layer(spec, seed=seed), device)
    for li in range(n_layers):
        g.manual_seed(seed * 1000 + li)
        w = {"router_w": torch.randn(E, d, generator=g, device=device) * spec.sigma_router,
             "router_b": torch.zeros(E, device=device)}
        if spec.bias == "zipf":
            w["router_b"] = torch.from_numpy(I.zipf_bias(seed, li, E)).to(device)
        if kind in ("bf16", "stack"):
            for name, shape in (("w_gate", (E, F, d)), ("w_up", (E, F, d)), ("w_down", (E, d, F)),
                                ("ws_gate", (Fs, d)), ("ws_up", (Fs, d)), ("ws_down", (d, Fs))):
                w[name] = (torch.randn(*shape, generator=g, device=device) * spec.sigma_w).to(torch.bfloat16)
        else:
            for name, t in base.items():
                if name not in ("router_w", "router_b"):
                    w[name] = t.clone()
        layers.append(w)
    return spec, layers


def oracle_tokens_per_s(kind, T, seed, budget_s=20.0):
    """The CPU oracle (float64 numpy) on a bounded sample of the workload, timed in a
    fresh interpreter whose BLAS is limited to one thread."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-sample", kind, str(T), str(seed), str(budget_s)]
    # (the stack's oracle sample is one layer of the stack)
    res = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=600)
    if res.returncode != 0:
        raise RuntimeError("oracle sample failed: " + res.stderr[-2000:])
    r = json.loads(res.stdout.strip().splitlines()[-1])
    return r["tokens_per_s"], {"kind": "oracle", "cores": 1, "sample": r["sample"]}


def oracle_sample_main(kind, T, seed, budget_s):
    """Child side of oracle_tokens_per_s: prints {"tokens_per_s", "sample"}."""
    import oracle
    from sparse_moe_transformer_02_b300 import inputs as I
    spec = {"bf16": I.FLINT_BF16, "nvfp4": I.FLINT_NVFP4, "stack": I.FLINT_STACK_ZIPF}[kind]
    L = I.make_layer(spec, seed=seed)
    W = oracle.LayerWeights(L)
    x = I.make_tokens(spec, seed=seed, T=max(T, 1))
    done, t_used = 0, 0.0
    n = min(T, 8)
    while t_used < budget_s and done < T:
        t0 = time.perf_counter()
        oracle.moe_forward(x[done:done + n], W, spec.top_k, residual=spec.add_residual)
        t_used += time.perf_counter() - t0
        done += n
    print(json.dumps({"tokens_per_s": done / t_used,
                      "sample": f"{done} of the workload's {T} tokens through one layer ({kind} weights), "
                                f"float64 numpy oracle, 1 BLAS thread, {t_used:.1f} s"}))


# ------------------------------------------------------------------ our arm
def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    from sparse_moe_transformer_02_b300 import binding as B
    from sparse_moe_transformer_02_b300 import build

    build.build()
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    kind, T, n_layers = WORKLOADS[args.workload]
    if args.layers:
        n_layers = args.layers
    spec, wts = make_device_layers(kind, n_layers, device, seed=args.seed + rank)
    stream = torch.cuda.Stream(device)
    handles = []
    with torch.cuda.stream(stream):
        for w in wts:
            handles.append(B.layer_from_spec(spec, w, max_tokens=max(T, 64), stream=stream,
                                             path={"auto": 0, "gemv": 1, "tc": 2}[args.path]))
    g = torch.Generator(device=device)
    g.manual_seed(args.seed + 77 + rank)
    x = (torch.randn(T, spec.d, generator=g, device=device) * spec.sigma_x).to(torch.bfloat16)
    ys = [torch.empty_like(x) for _ in handles]
    chain = kind == "stack"          # layer l + 1 reads layer l's output
    ins = [x] + ys[:-1] if chain else [x] * len(handles)
    torch.cuda.synchronize()

    def step():
        for h, xi, y in zip(handles, ins, ys):
            h.forward(xi, y, stream=stream)

    # realised routing: distinct experts per layer (on each layer's actual input)
    step()
    stream.synchronize()
    U = []
    for h, xi in zip(handles, ins):
        _, _, cnt = h.route(xi, stream=stream)
        stream.synchronize()
        U.append(int((cnt > 0).sum().item()))
    # kernels one forward launches: router, slot placement / activation copy,
    # gate/up, down, finalise on the tensor-core path; router, (NVFP4: f16
    # activation copy,) gate/up, down-and-combine on the GEMV path
    tc_path = args.path != "gemv"
    kernels_per_fwd = 5 if tc_path else (4 if kind == "nvfp4" else 3)

    for _ in range(max(args.warmup, 1)):
        step()
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        ev1.record(stream)
    ev1.synchronize()
    torch.cuda.synchronize()
    t_ms = ev0.elapsed_time(ev1)
    clocks = sampler.stop() if sampler else None
    t_ms = max_over_ranks(t_ms, device)
    if world > 1:
        dist.barrier()

    ms_step = t_ms / args.steps
    value = job_throughput(T * n_layers * args.steps, t_ms / 1e3, world)

    # per-kernel timing (separate, eager pass with event pairs around each launch)
    for h in handles:
        B._ok(B.moe_profile_enable(h.h, 1, 64 * kernels_per_fwd), "moe_profile_enable")
    prof_steps = 5
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
    dom = max(tot, key=lambda kk: tot[kk][0])
    dom_ms = tot[dom][0] / max(tot[dom][1], 1)
    pk = peaks()
    Umean = sum(U) / len(U)
    b_exp = B_EXP_NVFP4 if kind == "nvfp4" else B_EXP_BF16
    d, E, F = spec.d, spec.num_experts, spec.ffn
    per_kernel_bytes = {
        "route": 4 * d * E + 4 * E + T * d * 2,
        "gemv_gateup": (Umean + 1) * b_exp * 2 / 3 + T * d * 2,
        "gemv_down": (Umean + 1) * b_exp / 3 + T * d * 2,
        "tc_gateup": (Umean + 1) * b_exp * 2 / 3 + T * d * 2,
        "tc_down": (Umean + 1) * b_exp / 3,
        "tc_gather": 2 * T * spec.top_k * d * 2,
        "tc_finalize": T * d * (4 + 2),
    }
    layer_bytes = (Umean + 1) * b_exp + 4 * d * E + 4 * E + T * d * 2 * 2
    layer_flops = 2 * T * (spec.top_k + 1) * 3 * d * F + 2 * T * d * E
    # the dominant kernel's binding roof: whichever of HBM bytes / measured
    # bandwidth and tensor flops / measured bf16 peak takes longer
    per_kernel_flops = {"tc_gateup": 2 * T * (spec.top_k + 1) * 2 * d * F,
                        "tc_down": 2 * T * (spec.top_k + 1) * d * F}
    dom_bytes = per_kernel_bytes.get(dom, 0)
    dom_flops = per_kernel_flops.get(dom, 0)
    if dom_flops / (pk["bf16_tflops"] * 1e12) > dom_bytes / (pk["hbm_gbs"] * 1e9):
        bound, unit, peak = "tensor", "TFLOP/s", pk["bf16_tflops"]
        achieved = dom_flops / (dom_ms * 1e-3) / 1e12
    else:
        bound, unit, peak = "hbm", "GB/s", pk["hbm_gbs"]
        achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    traffic = dram_traffic(dom, args.workload)
    roofline = {"bound": bound, "kernel": dom, "achieved": round(achieved, 1), "peak": peak, "unit": unit,
                "frac": round(achieved / peak, 4), "traffic": traffic, "peak_source": pk["source"],
                "kernel_ms": round(dom_ms, 5),
                "per_kernel_ms": {kk: round(v[0] / max(v[1], 1), 5) for kk, v in tot.items() if v[1]}}
    layer_time_s = ms_step / 1e3 / n_layers
    layer = {"us_per_layer": round(layer_time_s * 1e6, 2), "distinct_experts_mean": round(Umean, 2),
             "algorithmic_bytes": int(layer_bytes), "hbm_gbs": round(layer_bytes / layer_time_s / 1e9, 1),
             "hbm_frac_of_measured": round(layer_bytes / layer_time_s / 1e9 / pk["hbm_gbs"], 4),
             "hbm_frac_of_8tbs": round(layer_bytes / layer_time_s / 1e9 / 8000.0, 4),
             "tflops": round(layer_flops / layer_time_s / 1e12, 2)}

    # end to end with host buffers, host<->device copies inside the timed region:
    # independent layers go through moe_forward_host (copy in, forward, copy out);
    # the chained stack copies its input in and its output out around the chain
    xh = x.cpu().pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    for h in handles[:2]:
        h.forward_host(xh, yh, stream=stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e_steps = max(1, min(args.steps, 10))
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

    sweep = {}
    if args.sweep and rank == 0 and world == 1 and args.workload.startswith("decode"):
        for wname in SWEEP:
            sweep[wname] = sweep_point(args, wname, handles, spec, device, stream)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        try:
            v, info = oracle_tokens_per_s(kind, T, seed=args.seed)
            cpu = dict(info, value=round(v, 3), unit="tokens/s")
        except Exception as exc:          # the GPU numbers stand without it
            cpu = {"kind": "oracle", "value": None, "error": str(exc)[-300:]}

    for h in handles:
        h.close()
    if rank == 0:
        out = {"metric": "MoE-layer tokens/s", "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
               "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
               "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
               "dtype": "nvfp4" if kind == "nvfp4" else "bf16",
               "data": "synthetic (seeded N(0,0.02) weights drawn on the device, N(0,1) activations)",
               "config": {"workload": f"flint_moe_layer_{args.workload}", "tokens": T, "d": spec.d,
                          "experts": spec.num_experts, "shared_experts": 1, "top_k": spec.top_k,
                          "expert_ffn": spec.ffn, "weights": kind, "layers_per_step": n_layers,
                          "l2": f"inputs larger than L2: {n_layers} distinct layers' weights per step",
                          "chained": chain, "router_bias": spec.bias,
                          "parallelism": f"replicas{world}", "path": args.path},
               "layer": layer, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
               "gpu_launches": args.steps * n_layers * kernels_per_fwd, "clocks": clocks}
        if sweep:
            out["sweep"] = sweep
        print(json.dumps(out), flush=True)


def sweep_point(args, wname, handles, spec, device, stream):
    """Tokens/s and HBM GB/s of the same layers at another decode batch size."""
    import torch
    kind, T, _ = WORKLOADS[wname]
    g = torch.Generator(device=device)
    g.manual_seed(args.seed + 1234 + T)
    x = (torch.randn(T, spec.d, generator=g, device=device) * spec.sigma_x).to(torch.bfloat16)
    ys = [torch.empty_like(x) for _ in handles]
    U = []
    for h in handles:
        _, _, cnt = h.route(x, stream=stream)
        stream.synchronize()
        U.append(int((cnt > 0).sum().item()))

    def step():
        for h, y in zip(handles, ys):
            h.forward(x, y, stream=stream)
    for _ in range(3):
        step()
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = max(args.steps, 10)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(n):
            graph.replay()
        ev1.record(stream)
    ev1.synchronize()
    t = ev0.elapsed_time(ev1) / 1e3 / n / len(handles)
    Um = sum(U) / len(U)
    byt = (Um + 1) * B_EXP_BF16 + 4 * spec.d * spec.num_experts + 4 * spec.num_experts + T * spec.d * 4
    return {"tokens_per_s": round(T / t, 1), "us_per_layer": round(t * 1e6, 2), "distinct_experts_mean": Um,
            "hbm_gbs": round(byt / t / 1e9, 1), "hbm_frac_of_measured": round(byt / t / 1e9 / peaks()["hbm_gbs"], 4)}


# ------------------------------------------------------------------ reference arm (the CPU oracle)
def run_reference(args, rank):
    if rank != 0:
        return
    kind, T, _ = WORKLOADS[args.workload]
    for _ in range(args.warmup):
        oracle_tokens_per_s(kind, T, seed=args.seed, budget_s=0.5)
    vals, infos = [], []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        v, info = oracle_tokens_per_s(kind, T, seed=args.seed, budget_s=2.0)
        vals.append(v)
        infos.append(info)
    total = time.perf_counter() - t0
    v = statistics.median(vals)
    out = {"impl": "reference", "metric": "MoE-layer tokens/s", "value": round(v, 3), "unit": "tokens/s",
           "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(1e3 * total / max(args.steps, 1), 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": f"flint_moe_layer_{args.workload}", "tokens": T},
           "cpu_baseline": dict(infos[-1], value=round(v, 3), unit="tokens/s"),
           "e2e": {"value": round(v, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    if len(sys.argv) > 1 and sys.argv[1] == "--oracle-sample":
        oracle_sample_main(sys.argv[2], int(sys.argv[3]), int(sys.argv[4]), float(sys.argv[5]))
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
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
