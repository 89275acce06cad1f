#!/usr/bin/env python3
"""Benchmark of the multi-LoRA segmented linear on GB300 (one JSON line on rank 0).

Metric: LoRA-linear tokens/s = tokens that pass through one LoRA-augmented linear per
second, summed over every linear of the step and over all ranks.

Workloads (synthetic, seeded, shaped like the multi-LoRA serving pages' 7B model):
  decode  (default)  one decode batch of 64 tokens through the q_proj (4096 x 4096, fp16) of
                     32 layers, each layer with its own base weight, its own pool of 100
                     rank-8/alpha-16 adapters and its own input; idx Zipf(1.1) over 100 slots
                     with 10 % base-only, routed once per batch (one segment build per step).
  prefill            32 requests x 512 tokens (16384, bf16) through q_proj and v_proj
                     (4096 x 4096 each, 100 rank-16/alpha-32 adapters per projection).
  mixed              one batch of --tokens tokens (1..64) through 32 layer copies of a
                     4096 x 4096 fp16 linear whose 6 adapters have ranks {8,8,16,16,64,64}
                     padded to 64.
  load               mounts one 7B-shaped rank-8 adapter (224 slots) from pinned host memory
                     (lora_pool_load_slot reads it over NVLink-C2C); ms per adapter.
A step = one lora_segment + every lora_linear_fwd of the step, captured once in a CUDA graph
and replayed.  Each step's inputs exceed the 129 MB L2 (no flush needed).

Extra legs: per-kernel CUDA-event timing (roofline of the base-GEMM kernel), end-to-end
timing with pinned host buffers and host<->device copies inside the timed region, the CPU
oracle timed on the host cores (cpu_baseline), and SM clocks sampled during the timed region.
`--impl reference` times the CPU oracle alone (the reference arm of this build).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "LoRA-linear tokens/s at 1 GB300 + % of HBM (decode) / tensor (prefill) roofline"
UNIT = "tokens/s"
DEFAULT_STEPS = {"decode": 4000, "mixed": 4000, "prefill": 400, "layer": 1000, "load": 20}


def parse_args():
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=["decode", "prefill", "mixed", "layer", "load"], default="decode")
    p.add_argument("--variant", type=int, default=0, help="0 auto, 1 fused, 2 separate, 3 CUDA-core")
    p.add_argument("--ungrouped", action="store_true",
                   help="layer and prefill workloads: one call per projection instead of grouping the projections "
                        "that read the same x (q|k|v and gate|up; q|v)")
    p.add_argument("--layers", type=int, default=None, help="layer copies per step (32; 4 for --workload layer)")
    p.add_argument("--tokens", type=int, default=64, help="batch size of the decode/mixed workloads")
    p.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU work of the cpu_baseline leg")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--prefetch-next", action="store_true",
                   help="pass the next linear's weight as the L2 prefetch hint of lora_linear_fwd_ex")
    a = p.parse_args()
    if a.steps is None:
        a.steps = DEFAULT_STEPS[a.workload]
    if a.layers is None:
        a.layers = 4 if a.workload == "layer" else 32
    a.warmup = max(3, a.warmup)
    return a


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ----------------------------------------------------------------------------------------------
# workload description (shared by both arms)
# ----------------------------------------------------------------------------------------------

def workload_cases(name, rank, layers, tokens, layer_range=None):
    """Returns (idx, [LinearCase per linear of the step], description dict)."""
    import torch

    from adapter_gemm_segment_gb300 import workloads as wl

    layer_range = range(layers) if layer_range is None else layer_range
    if name == "decode":
        seed = 1 + rank_seed_offset(rank)
        first = wl.decode_q_proj(seed=seed, n=tokens, layer=0)
        cases = [first if l == 0 else wl.decode_q_proj(seed=seed, n=tokens, layer=l) for l in layer_range]
        desc = {"workload": f"decode q_proj 4096x4096 fp16, {tokens} tokens, {layers} layers per step, "
                            "100 adapters r=8 alpha=16, Zipf(1.1) + 10% base-only",
                "tokens": tokens, "linears_per_step": layers, "h_in": 4096, "h_out": 4096, "r_max": 8,
                "n_slots": 100}
        return first.idx, cases, desc
    if name == "mixed":
        seed = 2 + rank_seed_offset(rank)
        first = wl.mixed_rank(tokens, seed=seed, layer=0)
        cases = [first if l == 0 else wl.mixed_rank(tokens, seed=seed, layer=l) for l in layer_range]
        desc = {"workload": f"mixed-rank decode 4096x4096 fp16, {tokens} tokens, {layers} layers per step, "
                            "6 adapters ranks {8,8,16,16,64,64} padded to 64, alpha=2r",
                "tokens": tokens, "linears_per_step": layers, "h_in": 4096, "h_out": 4096, "r_max": 64,
                "n_slots": 6}
        return first.idx, cases, desc
    if name == "layer":
        cases = []
        for l in layer_range:
            cases += wl.full_layer(l, seed=4 + rank_seed_offset(rank))
        desc = {"workload": f"7B-shaped decode layers: 256 tokens bf16 through q,k,v,o (4096x4096), gate/up "
                            f"(4096x11008), down (11008x4096) of {layers} layers per step, LoRA r=16 alpha=32 on "
                            "all seven, 100 adapters each, Zipf(1.1)",
                "tokens": 256, "linears_per_step": 7 * layers, "r_max": 16, "n_slots": 100}
        return (cases[0].idx if cases else _layer_idx(rank)), cases, desc
    cases = wl.prefill(seed=3 + rank_seed_offset(rank))
    desc = {"workload": "prefill 32x512 tokens bf16, q_proj + v_proj 4096x4096, 100 adapters r=16 alpha=32",
            "tokens": 16384, "linears_per_step": 2, "h_in": 4096, "h_out": 4096, "r_max": 16, "n_slots": 100}
    return cases[0].idx, cases, desc


def _layer_idx(rank):
    import numpy as np
    import torch

    from adapter_gemm_segment_gb300 import workloads as wl

    rng = np.random.default_rng([4 + rank_seed_offset(rank)])
    return torch.from_numpy(wl.draw_zipf_idx(rng, 256, 100))


def algorithmic_case(idx, h_in, h_out, R, es=2):
    """One linear's algorithmic bytes / FLOPs (W + touched adapters + x + y; base + LoRA)."""
    import numpy as np

    idx = np.asarray(idx)
    n = len(idx)
    D = len(set(idx[idx >= 0].tolist()))
    n_L = int((idx >= 0).sum())
    W = h_out * h_in * es
    A_D = D * R * h_in * es
    B_D = D * h_out * R * es
    xy = n * (h_in + h_out) * es
    return {"D": D, "n_L": n_L, "linear_bytes": W + A_D + B_D + xy, "gemm_bytes": W + B_D + xy,
            "linear_flops": 2 * n * h_in * h_out + 2 * n_L * R * (h_in + h_out),
            "gemm_flops": 2 * n * h_in * h_out + 2 * n_L * R * h_out}


# ----------------------------------------------------------------------------------------------
# multi-rank helpers (replicas: every rank runs its own batches; no data-path collective)
# ----------------------------------------------------------------------------------------------

def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The largest per-rank timing (the job is as slow as its slowest replica)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, tokens_per_step: int, steps: int, ms_max: float) -> float:
    """Whole-job throughput: the tokens all ranks processed over the slowest rank's time."""
    return world * tokens_per_step * steps / (ms_max / 1e3)


def rank_seed_offset(rank: int) -> int:
    """Each replica draws its own batches (weak scaling: fixed work per GPU)."""
    return 100 * rank


# ----------------------------------------------------------------------------------------------
# clocks
# ----------------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.samples = []
        self.proc = None
        self.err = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", gpu_id], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception as e:  # no nvidia-smi
            self.err = str(e)

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        if self.err is not None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "error": self.err}
        win = [s for t, s in self.samples if t0 <= t <= t1 + 0.15]
        if not win:  # timed region shorter than one sample period: take the closest samples
            near = sorted(self.samples, key=lambda ts: min(abs(ts[0] - t0), abs(ts[0] - t1)))[:3]
            win = [s for _, s in near]
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in win:
            f = [x.strip() for x in s.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons), "samples": len(win)}


# ----------------------------------------------------------------------------------------------
# the CPU oracle legs
# ----------------------------------------------------------------------------------------------

CPU_CHILD = r"""
import json, os, sys, time
sys.path.insert(0, {root!r})
import numpy as np
from oracle import lora_oracle as O
import bench
idx, cases, desc = bench.workload_cases({wl!r}, 0, {layers}, {tokens}, layer_range=range(1))
case = cases[0]
pool = O.pool_of_case(case)
idx_np = idx.numpy()
n = len(idx_np)
rows_all = np.arange(n)
def timed(m):
    t = time.perf_counter(); O.lora_linear(case.x, case.W, pool, idx_np, rows=rows_all[:m]); return time.perf_counter() - t
m_hi = max(1, min(n, 64))
t_lo, t_hi = timed(1), timed(m_hi)
per_row = max(0.0, (t_hi - t_lo) / max(1, m_hi - 1))  # cost model a + b m
m = n
if {step_budget} > 0:
    m = int(min(n, max(1, ({step_budget} - t_lo) / per_row + 1))) if per_row > 0 else n
tokens = 0; steps = 0
for w in range({warmup}):
    O.lora_linear(case.x, case.W, pool, idx_np, rows=rows_all[:m])
t0 = time.perf_counter()
while True:
    start = (steps * m) % n
    rows = (rows_all[start:start + m] if start + m <= n else np.concatenate([rows_all[start:], rows_all[:start + m - n]]))
    O.lora_linear(case.x, case.W, pool, idx_np, rows=rows)
    tokens += m; steps += 1
    el = time.perf_counter() - t0
    if ({fixed_steps} > 0 and steps >= {fixed_steps}) or ({fixed_steps} <= 0 and el >= {seconds}):
        break
print("RESULT " + json.dumps({{"tokens": tokens, "seconds": el, "steps": steps, "rows_per_step": m,
                              "product_library_mapped": bench.product_library_mapped()}}))
"""


def product_library_mapped():
    """Whether this process has the CUDA product library mapped (None where /proc is absent).
    The CPU-oracle legs must not: they time the oracle alone."""
    try:
        with open("/proc/self/maps") as f:
            return "liblora_gb300" in f.read()
    except OSError:
        return None


def run_cpu_oracle(workload, layers, tokens, seconds=10.0, fixed_steps=0, warmup=1, step_budget=0.0):
    cores = os.cpu_count() or 1
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = str(cores)
    env["CUDA_VISIBLE_DEVICES"] = ""
    code = CPU_CHILD.format(root=ROOT, wl=workload, layers=layers, tokens=tokens, seconds=seconds,
                            fixed_steps=fixed_steps, warmup=warmup, step_budget=step_budget)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, cwd=ROOT)
    for line in r.stdout.splitlines():
        if line.startswith("RESULT "):
            d = json.loads(line[7:])
            d["cores"] = cores
            return d
    raise RuntimeError(f"oracle timing failed: {r.stderr[-2000:]}")


# ----------------------------------------------------------------------------------------------
# reference arm: the CPU oracle as it stands
# ----------------------------------------------------------------------------------------------

def reference_arm(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    _, _, desc = workload_cases(args.workload, 0, args.layers, args.tokens, layer_range=range(1))
    budget = 120.0 / (args.steps + args.warmup)  # whole run within a few minutes
    d = run_cpu_oracle(args.workload, args.layers, args.tokens, fixed_steps=args.steps, warmup=args.warmup,
                       step_budget=budget)
    value = d["tokens"] / d["seconds"]
    sample = (f"{d['rows_per_step']} token rows of one linear of the workload per step "
              f"(float64 numpy oracle, {d['cores']} BLAS threads)")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * d["seconds"] / d["steps"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": desc,
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": d["cores"], "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "product_library_mapped": {"arm": product_library_mapped(), "oracle_child": d["product_library_mapped"]}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------------------------

def read_profile_traffic(kernel_key):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the current source."""
    import hashlib

    path = os.path.join(ROOT, "profiles", f"{kernel_key}.md")
    if not os.path.exists(path):
        return None
    src = os.path.join(ROOT, "adapter_gemm_segment_gb300", "csrc", "gemm_tc.cu")
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    fields = {}
    for line in open(path):
        if ": " in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(": ", 1)  # keys contain ':' (sha256[:16])
            fields[k.strip()] = v.strip()
    if fields.get("gemm_tc.cu sha256[:16]") != sha:
        return None
    try:
        return float(fields["dram bytes per launch (full workload)"])
    except (KeyError, ValueError):
        return None


def ours(args):
    import numpy as np
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if dist is not None:
            dist.barrier(device_ids=[local])

    import adapter_gemm_segment_gb300 as ags

    peaks = load_peaks()
    idx, cases, desc = workload_cases(args.workload, rank, args.layers, args.tokens)
    dtype = cases[0].dtype
    n = int(idx.numel())
    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)

    # ---- device-resident inputs, pools, workspaces ----
    layers = []
    x_dev = {}  # projections fed by the same input (q, k, v; gate, up) share one device copy
    for case in cases:
        ad = case.adapters
        pool = ags.LoraPool(case.h_in, case.h_out, ad.r_max, ad.n_slots, dtype, dev)
        A_all = [a.to(dev, non_blocking=True) for a in ad.A]
        B_all = [b.to(dev, non_blocking=True) for b in ad.B]
        for s in range(ad.n_slots):
            pool.load_slot(s, A_all[s], B_all[s], ad.alphas[s])
        if id(case.x) not in x_dev:
            x_dev[id(case.x)] = case.x.to(dev)
        layers.append({"pool": pool, "W": case.W.to(dev), "x": x_dev[id(case.x)],
                       "y": torch.empty(n, case.h_out, dtype=dtype, device=dev)})
        del A_all, B_all
    # prefill: q and v share x
    if args.workload == "prefill":
        layers[1]["x"] = layers[0]["x"]
    idx_dev = idx.to(dev)
    pool0 = layers[0]["pool"]
    seg_ws = pool0.segment_workspace(n, dev)
    # one workspace serves every linear of the step (sequential on one stream): size it for the largest
    lin_ws = ags._device_bytes(max(ags.lora_linear_workspace_bytes(L["pool"].handle, n) for L in layers), dev)
    torch.cuda.synchronize()

    launches_before = ags.lora_kernel_launch_count()

    # calls of one step: single linears, or (layer workload) groups of projections that read
    # the same x -- q|k|v and gate|up -- as one call over their concatenated weight
    calls = []
    grouped = args.workload in ("layer", "prefill") and not args.ungrouped
    i = 0
    while i < len(layers):
        j = i + 1
        while grouped and j < len(layers) and layers[j]["x"] is layers[i]["x"] and j - i < 4:
            j += 1
        members = layers[i:j]
        if len(members) == 1:
            calls.append({"members": members, "y": members[0]["y"]})
        else:
            handles = [L["pool"].handle for L in members]
            calls.append({"members": members, "handles": handles,
                          "W": torch.cat([L["W"] for L in members], 0), "x": members[0]["x"],
                          "y": torch.empty(n, sum(L["W"].shape[0] for L in members), dtype=dtype, device=dev)})
            lin_ws = lin_ws if lin_ws.numel() >= ags.lora_linear_group_workspace_bytes(handles, n) else \
                ags._device_bytes(ags.lora_linear_group_workspace_bytes(handles, n), dev)
            for L in members:  # the group reads the concatenated weight and writes the concatenated output
                L["W"] = L["y"] = None
        i = j
    torch.cuda.synchronize()

    prefetch = args.prefetch_next and args.workload != "prefill" and not grouped
    nxt = [calls[(i + 1) % len(calls)]["members"][0]["W"] if prefetch else None for i in range(len(calls))]

    def linear(i, c, seg):
        if "handles" in c:
            ags.lora_linear_fwd_group(c["handles"], c["W"], c["x"], c["y"], seg, lin_ws, args.variant)
        else:
            L = c["members"][0]
            ags.lora_linear_fwd_ex(L["pool"].handle, L["W"], L["x"], L["y"], seg, lin_ws, args.variant,
                                   prefetch=nxt[i])

    def step():
        seg = ags.lora_segment(idx_dev, pool0.handle, seg_ws)
        for i, c in enumerate(calls):
            linear(i, c, seg)

    # eager warm-up (also checks the status word once)
    step()
    torch.cuda.synchronize()
    seg_chk = ags.lora_segment(idx_dev, pool0.handle, seg_ws)
    seg_chk._ws = seg_ws
    assert ags.lora_segment_status(seg_chk) == 0
    kernels_per_step = None
    c0 = ags.lora_kernel_launch_count()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    kernels_per_step = ags.lora_kernel_launch_count() - c0
    torch.cuda.synchronize()

    gpu_id = str(local)
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    clocks = ClockSampler(gpu_id)
    time.sleep(0.3)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()

    # ---- timed region ----
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t_host0 = time.time()
    ev0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    t_host1 = time.time()
    ms = max_over_ranks(ev0.elapsed_time(ev1), dist, dev)
    time.sleep(0.25)
    clocks.stop()
    clk = clocks.summary(t_host0, t_host1)
    ms_per_step = ms / args.steps
    tokens_per_step = n * len(layers)
    value = job_tokens_per_s(world, tokens_per_step, args.steps, ms)

    # ---- per-kernel timing (events recorded around each kernel, graph-replayed) ----
    n_lin = len(calls)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_lin)]
    for trio in evs:
        for e in trio:
            e.record(stream)
    torch.cuda.synchronize()
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2, stream=stream):
        seg = ags.lora_segment(idx_dev, pool0.handle, seg_ws)
        for i, (c, trio) in enumerate(zip(calls, evs)):
            ags.lora_set_timing_events(*trio)
            linear(i, c, seg)
        ags.lora_set_timing_events()
    reps = max(3, min(50, args.steps // 20))
    g2.replay()
    torch.cuda.synchronize()
    t_shr = [[] for _ in range(n_lin)]
    t_gemm = [[] for _ in range(n_lin)]
    for _ in range(reps):
        g2.replay()
        torch.cuda.synchronize()
        for i, trio in enumerate(evs):
            t_shr[i].append(trio[0].elapsed_time(trio[1]))
            t_gemm[i].append(trio[1].elapsed_time(trio[2]))
    gemm_ms_i = [statistics.mean(v) for v in t_gemm]
    shrink_ms = statistics.mean(statistics.mean(v) for v in t_shr)
    gemm_ms = statistics.mean(gemm_ms_i)

    idx_np = idx.numpy()
    algs = [algorithmic_case(idx_np, c.h_in, c.h_out, c.adapters.r_max) for c in cases]
    # per-linear roofline time: the slower of bytes at HBM bandwidth and FLOPs at tensor peak
    step_roof_ms = sum(max(a_["linear_bytes"] / (peaks["hbm_gbs"] * 1e9),
                           a_["linear_flops"] / (peaks["bf16_tflops"] * 1e12)) for a_ in algs) * 1e3
    alg = {"D": algs[0]["D"], "n_L": algs[0]["n_L"]}
    if args.workload == "prefill":
        achieved = sum(a_["gemm_flops"] for a_ in algs) / (sum(gemm_ms_i) / 1e3) / 1e12
        peak = peaks["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": read_profile_traffic(f"gemm_prefill_{args.workload}"),
                "kernel": "gemm_prefill_kernel", "kernel_ms": gemm_ms,
                "algorithmic_flops_per_launch": sum(a_["gemm_flops"] for a_ in algs) / n_lin,
                "peak_source": peaks["source"] + " burst",
                "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"]}
    else:
        achieved = sum(a_["gemm_bytes"] for a_ in algs) / (sum(gemm_ms_i) / 1e3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": read_profile_traffic(f"gemm_decode_{args.workload}"),
                "kernel": ("base GEMM calls: gemm_tall_kernel (grouped q|k|v, gate|up), gemm_decode_kernel (o, down)"
                           if args.workload == "layer" and grouped else "gemm_decode_kernel"), "kernel_ms": gemm_ms,
                "algorithmic_bytes_per_launch": sum(a_["gemm_bytes"] for a_ in algs) / n_lin,
                "peak_source": peaks["source"] + " copy"}
    roof["shrink_ms"] = shrink_ms
    roof["step_roofline_ms"] = step_roof_ms
    roof["step_frac"] = step_roof_ms / ms_per_step

    # ---- end to end: pinned host buffers, copies inside the timed region ----
    # A serving loop overlaps transfers with compute: step k's inputs go in (copy stream) and
    # step k-1's outputs come out (a second copy stream) while step k-1 / k compute.  Two sets
    # of device buffers, each with its own captured graph, alternate; events order every reuse.
    e2e = None
    if not args.no_e2e:
        def x_of(c):
            return c["x"] if "handles" in c else c["members"][0]["x"]

        xs0 = {}
        for c in calls:
            xs0.setdefault(id(x_of(c)), x_of(c))
        sets = [{"idx": idx_dev, "x": xs0, "y": [c["y"] for c in calls], "graph": graph}]
        s1 = {"idx": torch.empty_like(idx_dev), "x": {k: torch.empty_like(v) for k, v in xs0.items()},
              "y": [torch.empty_like(c["y"]) for c in calls]}

        def step_on(bufs):
            seg = ags.lora_segment(bufs["idx"], pool0.handle, seg_ws)
            for i, c in enumerate(calls):
                xin, yout = bufs["x"][id(x_of(c))], bufs["y"][i]
                if "handles" in c:
                    ags.lora_linear_fwd_group(c["handles"], c["W"], xin, yout, seg, lin_ws, args.variant)
                else:
                    L = c["members"][0]
                    ags.lora_linear_fwd_ex(L["pool"].handle, L["W"], xin, yout, seg, lin_ws, args.variant,
                                           prefetch=nxt[i])

        s1["idx"].copy_(idx_dev)
        for k, v in xs0.items():
            s1["x"][k].copy_(v)
        step_on(s1)
        torch.cuda.synchronize()
        s1["graph"] = torch.cuda.CUDAGraph()
        with torch.cuda.graph(s1["graph"], stream=stream):
            step_on(s1)
        sets.append(s1)
        x_host = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True).copy_(v.cpu()) for k, v in xs0.items()}
        idx_host = torch.empty(idx.shape, dtype=torch.int32, pin_memory=True).copy_(idx)
        y_host = [[torch.empty(y.shape, dtype=dtype, pin_memory=True) for y in b["y"]] for b in sets]
        h2d = idx_host.numel() * 4 + sum(v.numel() * v.element_size() for v in x_host.values())
        d2h = sum(y.numel() * y.element_size() for y in y_host[0])
        e2e_steps = max(3, min(args.steps, 500))
        h2d_st, d2h_st = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        loaded = [torch.cuda.Event() for _ in range(2)]
        computed = [torch.cuda.Event() for _ in range(2)]
        drained = [torch.cuda.Event() for _ in range(2)]

        def e2e_step(k):
            b = sets[k % 2]
            h2d_st.wait_event(computed[k % 2])  # step k-2 no longer reads this set's inputs
            with torch.cuda.stream(h2d_st):
                b["idx"].copy_(idx_host, non_blocking=True)
                for key, v in b["x"].items():
                    v.copy_(x_host[key], non_blocking=True)
            loaded[k % 2].record(h2d_st)
            stream.wait_event(loaded[k % 2])
            stream.wait_event(drained[k % 2])  # step k-2's outputs have left this set's buffers
            b["graph"].replay()
            computed[k % 2].record(stream)
            d2h_st.wait_event(computed[k % 2])
            with torch.cuda.stream(d2h_st):
                for y, yh in zip(b["y"], y_host[k % 2]):
                    yh.copy_(y, non_blocking=True)
            drained[k % 2].record(d2h_st)

        for k in range(3):
            e2e_step(k)
        torch.cuda.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(h2d_st)
        for k in range(e2e_steps):
            e2e_step(k)
        e1.record(d2h_st)
        torch.cuda.synchronize()
        ems = max_over_ranks(e0.elapsed_time(e1), dist, dev)
        e2e = {"value": job_tokens_per_s(world, tokens_per_step, e2e_steps, ems), "unit": UNIT,
               "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": ems / e2e_steps,
               "mode": "C-ABI calls captured in CUDA graphs; every step copies its inputs in from pinned host memory "
                       "and its outputs out to pinned host memory, on two copy streams overlapping the previous and "
                       "next steps' compute (two alternating buffer sets)"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        d = run_cpu_oracle(args.workload, args.layers, args.tokens, seconds=args.cpu_seconds)
        cpu = {"value": d["tokens"] / d["seconds"], "unit": UNIT, "cores": d["cores"], "kind": "oracle",
               "sample": f"{d['steps']} passes of one linear of the workload ({d['rows_per_step']} tokens each, "
                         f"float64 numpy oracle) in {d['seconds']:.1f} s"}

    if rank == 0:
        cfg = dict(desc)
        cfg.update({"variant": {0: "auto", 1: "fused", 2: "separate", 3: "cuda-core"}[args.variant],
                    "policy_variant": ags.lora_linear_policy(pool0.handle, n),
                    "distinct_slots_touched": alg["D"], "lora_tokens": alg["n_L"],
                    "l2": "inputs larger than L2 (no flush)", "timing": "CUDA graph replay, CUDA events",
                    "l2_prefetch_next_weight": prefetch,
                    "calls_per_step": len(calls),
                    "grouped": "projections reading the same x as one call each (lora_linear_fwd_group)" if grouped else None,
                    "parallelism": f"replicas x{world} (token batches sharded across GPUs, no collective)"})
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16" if dtype == torch.bfloat16 else "f16", "data": "synthetic",
                "config": cfg, "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": int(kernels_per_step) * args.steps, "kernels_per_step": int(kernels_per_step),
                "clocks": clk}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def adapter_load(args):
    """--workload load: mount one 7B-shaped rank-8 adapter (q, k, v, o, gate, up, down of 32
    layers: 224 slots in three pools) from pinned host memory, and from device memory, with
    lora_pool_load_slot; CUDA events around the mounts.  One JSON line (ms per adapter)."""
    import torch
    import adapter_gemm_segment_gb300 as ags

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    L, r, dt = 32, 8, torch.float16
    shapes = [(4096, 4096, 4 * L), (4096, 11008, 2 * L), (11008, 4096, L)]  # (h_in, h_out, slots)
    g = torch.Generator().manual_seed(9)
    pools, host, devs = [], [], []
    for h_in, h_out, S in shapes:
        pools.append(ags.LoraPool(h_in, h_out, r, S, dt, dev))
        hA = (torch.rand(S, r, h_in, generator=g) * 0.02 - 0.01).to(dt).pin_memory()
        hB = (torch.randn(S, h_out, r, generator=g) * 0.01).to(dt).pin_memory()
        host.append((hA, hB))
        devs.append((hA.to(dev), hB.to(dev)))
    nbytes = sum(2 * (S * r * h_in + S * h_out * r) for h_in, h_out, S in shapes)
    stream = torch.cuda.Stream(dev)

    def mount(src):  # one batched call per pool
        for pool, (A, B), (_, _, S) in zip(pools, src, shapes):
            pool.load_slots(list(range(S)), [A[s] for s in range(S)], [B[s] for s in range(S)], [16.0] * S, stream)

    def unmount():
        for pool, (_, _, S) in zip(pools, shapes):
            for s in range(S):
                pool.unload_slot(s, stream)

    def timed_ms(src, reps):
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            mount(src)
            e1.record(stream)
            unmount()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    for _ in range(max(3, args.warmup // 4)):
        mount(host)
        unmount()
    torch.cuda.synchronize()
    reps = args.steps or 20
    ms_host_eager = timed_ms(host, reps)
    ms_dev_eager = timed_ms(devs, reps)

    # the mounts as a CUDA graph (no host launch gaps): each replay rewrites every slot
    def graph_ms(src):
        with torch.cuda.stream(stream):
            mount(src)
            torch.cuda.synchronize()
            gr = torch.cuda.CUDAGraph()
            unmount()
            torch.cuda.synchronize()
            with torch.cuda.graph(gr, stream=stream):
                mount(src)
            torch.cuda.synchronize()
            for _ in range(3):
                gr.replay()
            ts = []
            for _ in range(reps):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                gr.replay()
                e1.record(stream)
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1))
            unmount()
            torch.cuda.synchronize()
        return statistics.median(ts)

    ms_host = graph_ms(host)
    ms_dev = graph_ms(devs)
    # plain pinned host -> device copy of the same bytes, for the link rate
    flat = torch.empty(nbytes // 2, dtype=dt).pin_memory()
    dst = torch.empty_like(flat, device=dev)
    for _ in range(3):
        dst.copy_(flat, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        dst.copy_(flat, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    ms_copy = e0.elapsed_time(e1) / reps
    line = {"metric": "adapter mount time (7B-shaped rank-8 adapter: q,k,v,o,gate,up,down x 32 layers)",
            "value": ms_host, "unit": "ms per adapter", "higher_is_better": False, "n_gpus": 1, "steps": reps,
            "warmup": max(3, args.warmup // 4), "data": "synthetic", "dtype": "f16",
            "config": {"workload": "mount 224 slots (3 pools, r_max 8) from pinned host memory, one lora_pool_load_slots call per pool", "bytes": nbytes,
                       "slots": sum(S for _, _, S in shapes)},
            "host_GBps": nbytes / (ms_host * 1e-3) / 1e9, "from_device_ms": ms_dev,
            "device_GBps": nbytes / (ms_dev * 1e-3) / 1e9, "timing": "mount calls captured in a CUDA graph",
            "eager_ms": {"host": ms_host_eager, "device": ms_dev_eager},
            "h2d_memcpy_ms_same_bytes": ms_copy, "h2d_memcpy_GBps": nbytes / (ms_copy * 1e-3) / 1e9,
            "context": "the pages quote 30-80 ms to load a ~30 MB rank-8 adapter over PCIe 5.0 x16"}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.workload == "load":
        adapter_load(args)
    elif args.impl == "reference":
        reference_arm(args)
    else:
        ours(args)


if __name__ == "__main__":
    main()
