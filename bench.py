#!/usr/bin/env python3
"""Benchmark of the multi-LoRA segmented linear on GB300 (one JSON line on rank 0).

Metric: LoRA-linear tokens/s = tokens that pass through one LoRA-augmented linear per
second, summed over every linear of the step and over all ranks.

Workloads (synthetic, seeded, shaped like the multi-LoRA serving pages' 7B model):
  decode  (default)  one decode batch of 64 tokens through the q_proj (4096 x 4096, fp16) of
                     32 layers, each layer with its own base weight, its own pool of 100
                     rank-8/alpha-16 adapters and its own input; idx Zipf(1.1) over 100 slots
                     with 10 % base-only, routed once per batch (one segment build per step).
                     The line also carries a "prefill" leg (the workload below, measured the
                     same way), so one run reports both halves of the metric: decode against
                     the HBM roofline, prefill against the tensor roofline.
  prefill            32 requests x 512 tokens (16384, bf16) through q_proj and v_proj
                     (4096 x 4096 each, 100 rank-16/alpha-32 adapters per projection), as one
                     grouped call.
  mixed              one batch of --tokens tokens (1..64) through 32 layer copies of a
                     4096 x 4096 fp16 linear whose 6 adapters have ranks {8,8,16,16,64,64}
                     padded to 64.
  layer              256 tokens through the 7 projections of 4 7B-shaped layers (grouped
                     calls q|k|v, o, gate|up, down).
  load               mounts one 7B-shaped rank-8 adapter (224 slots) from pinned host memory
                     (lora_pool_load_slot reads it over NVLink-C2C); ms per adapter.
  concat             the segmented path against the pages' concatenated-adapter matmul
                     (cuBLAS baseline) at 1, 8 and 64 tokens.
A step = one lora_segment + every lora_linear_fwd of the step, captured once in a CUDA graph
and replayed.  Each step's inputs exceed the 129 MB L2 (no flush needed).

Extra legs: the dominant kernel's time inside the step (%globaltimer stamps of every base-GEMM
launch in the chained graph; the serialised CUDA-event figure beside it), end-to-end timing
with pinned host buffers and host<->device copies inside the timed region, the CPU oracle
timed on the host cores (cpu_baseline), SM clocks sampled during the timed region, and the
tensor-concatenation figures of the batch (concat_metrics).
`--impl reference` times the CPU oracle alone (the benchmark's reference arm: the pages hold no code to run).
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
DEFAULT_STEPS = {"decode": 4000, "mixed": 4000, "prefill": 400, "layer": 1000, "load": 20, "concat": 200}


def parse_args():
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=["decode", "prefill", "mixed", "layer", "load", "concat"], default="decode")
    p.add_argument("--variant", type=int, default=0, help="0 auto, 1 fused, 2 separate, 3 CUDA-core")
    p.add_argument("--ungrouped", action="store_true",
                   help="layer and prefill workloads: one call per projection instead of grouping the projections "
                        "that read the same x (q|k|v and gate|up; q|v)")
    p.add_argument("--layers", type=int, default=None, help="layer copies per step (32; 4 for --workload layer)")
    p.add_argument("--tokens", type=int, default=64, help="batch size of the decode/mixed workloads")
    p.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU work of the cpu_baseline leg")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-prefill-leg", action="store_true",
                   help="decode workload: skip the prefill leg (the tensor-roofline half of the metric)")
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


def concat_metrics(idx, h_in, h_out, ranks, r_max, n_slots):
    """The three figures by which the blog.lonae.com page (tensor-concatenation paragraph)
    describes a concatenated-adapter matmul, for this batch, plus the segment count:
      - elements of the concatenated matrices (all n_slots adapters' A and B at r_max): the
        memory peak of that approach;
      - its batch x seq projection: the [n, n_slots * r_max] intermediate x A_cat^T, the launch
        dimension of that approach;
      - the zero-padding share: the part of the LoRA work done at r_max that multiplies padding,
        weighted by tokens (the invalid-FLOP share of a padded path) and by the touched adapters'
        stored rows (bytes);
    and the share of the concatenated approach's LoRA FLOPs that no token needs."""
    import numpy as np

    idx = np.asarray(idx)
    lora = idx[idx >= 0]
    touched = sorted(set(lora.tolist()))
    n = int(idx.size)
    useful_padded = 2 * len(lora) * r_max * (h_in + h_out)
    concat_flops = 2 * n * n_slots * r_max * (h_in + h_out)
    tok_pad = float(sum(r_max - ranks[s] for s in lora.tolist())) / (len(lora) * r_max) if len(lora) else 0.0
    slot_pad = float(sum(r_max - ranks[s] for s in touched)) / (len(touched) * r_max) if touched else 0.0
    nseg = len(touched) + (1 if (idx < 0).any() else 0)
    return {"n_segments": nseg, "distinct_adapters": len(touched),
            "concat_elements": n_slots * r_max * (h_in + h_out), "concat_projection": [n, n_slots * r_max],
            "concat_projection_elements": n * n_slots * r_max,
            "zero_pad_flop_share": tok_pad, "zero_pad_stored_share": slot_pad,
            "concat_lora_flops_wasted_share": (1.0 - useful_padded / concat_flops) if concat_flops else 0.0}


def measure(args, wl_name, steps, warmup, world, rank, local, dist, dev, peaks):
    """Time one workload's step on this rank; returns the JSON object of the line (rank 0)."""
    import numpy as np
    import torch

    def barrier():
        if dist is not None:
            dist.barrier(device_ids=[local])

    import adapter_gemm_segment_gb300 as ags

    tokens = args.tokens if wl_name in ("decode", "mixed") else None
    n_layers = args.layers if wl_name == args.workload else (4 if wl_name == "layer" else 32)
    idx, cases, desc = workload_cases(wl_name, rank, n_layers, tokens or 64)
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
    if wl_name == "prefill":
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
    grouped = wl_name in ("layer", "prefill") and not args.ungrouped
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

    prefetch = args.prefetch_next and wl_name != "prefill" and not grouped
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
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()

    # ---- timed region ----
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t_host0 = time.time()
    ev0.record(stream)
    for _ in range(steps):
        graph.replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    t_host1 = time.time()
    ms = max_over_ranks(ev0.elapsed_time(ev1), dist, dev)
    time.sleep(0.25)
    clocks.stop()
    clk = clocks.summary(t_host0, t_host1)
    ms_per_step = ms / steps
    tokens_per_step = n * len(layers)
    value = job_tokens_per_s(world, tokens_per_step, steps, ms)

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
    reps = max(3, min(50, steps // 20))
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
    gemm_ms_ser_i = [statistics.mean(v) for v in t_gemm]
    shrink_ms = statistics.mean(statistics.mean(v) for v in t_shr)

    # ---- in-step kernel time: every base-GEMM launch stamps %globaltimer at its first CTA's
    # start and its last CTA's end, inside the same chained graph (no events between kernels,
    # so programmatic dependent launch overlaps exactly as in the timed region) ----
    stamps = torch.empty(n_lin, 2, dtype=torch.int64, device=dev)
    ags.lora_set_kernel_stamps(stamps)
    try:
        g3 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g3, stream=stream):
            step()
    finally:
        ags.lora_set_kernel_stamps()
    d_in = [[] for _ in range(n_lin)]
    step_in = []
    e3a, e3b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for r in range(reps + 1):
        stamps[:, 0].fill_(-1)  # UINT64_MAX for the kernels' atomicMin
        stamps[:, 1].fill_(0)
        e3a.record(stream)
        g3.replay()
        e3b.record(stream)
        torch.cuda.synchronize()
        if r == 0:
            continue
        st = stamps.cpu()
        step_in.append(e3a.elapsed_time(e3b))
        for i in range(n_lin):
            d_in[i].append(float(st[i, 1] - st[i, 0]) / 1e6 if int(st[i, 0]) > 0 and int(st[i, 1]) > 0 else None)
    if all(v is not None for d in d_in for v in d):
        gemm_ms_i = [statistics.mean(v) for v in d_in]
        timing_basis = "in-step (%globaltimer stamps of every base-GEMM launch inside the chained graph)"
    else:  # kernels without stamps (CUDA-core diagnostic variant): serialised events only
        gemm_ms_i = gemm_ms_ser_i
        timing_basis = "serialised (CUDA events between kernels)"
    gemm_ms = statistics.mean(gemm_ms_i)
    gemm_ms_ser = statistics.mean(gemm_ms_ser_i)

    idx_np = idx.numpy()
    algs = [algorithmic_case(idx_np, c.h_in, c.h_out, c.adapters.r_max) for c in cases]
    # per-linear roofline time: the slower of bytes at HBM bandwidth and FLOPs at tensor peak
    step_roof_ms = sum(max(a_["linear_bytes"] / (peaks["hbm_gbs"] * 1e9),
                           a_["linear_flops"] / (peaks["bf16_tflops"] * 1e12)) for a_ in algs) * 1e3
    alg = {"D": algs[0]["D"], "n_L": algs[0]["n_L"]}
    if wl_name == "prefill":
        achieved = sum(a_["gemm_flops"] for a_ in algs) / (sum(gemm_ms_i) / 1e3) / 1e12
        peak = peaks["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": read_profile_traffic(f"gemm_prefill_{wl_name}"),
                "kernel": "gemm_prefill_kernel", "kernel_ms": gemm_ms,
                "algorithmic_flops_per_launch": sum(a_["gemm_flops"] for a_ in algs) / n_lin,
                "peak_source": peaks["source"] + " burst",
                "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"]}
    else:
        achieved = sum(a_["gemm_bytes"] for a_ in algs) / (sum(gemm_ms_i) / 1e3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": read_profile_traffic(f"gemm_decode_{wl_name}"),
                "kernel": ("base GEMM calls: gemm_tall_kernel (grouped q|k|v, gate|up), gemm_decode_kernel (o, down)"
                           if wl_name == "layer" and grouped else "gemm_decode_kernel"), "kernel_ms": gemm_ms,
                "algorithmic_bytes_per_launch": sum(a_["gemm_bytes"] for a_ in algs) / n_lin,
                "peak_source": peaks["source"] + " copy"}
    alg_per_launch = sum(a_["gemm_flops" if wl_name == "prefill" else "gemm_bytes"] for a_ in algs) / n_lin
    roof["timing_basis"] = timing_basis
    roof["kernel_ms_serialised"] = gemm_ms_ser
    roof["frac_serialised"] = alg_per_launch / (gemm_ms_ser / 1e3) / (peak * (1e12 if wl_name == "prefill" else 1e9))
    roof["kernels_ms_sum_over_step_ms"] = sum(gemm_ms_i) / statistics.mean(step_in)
    roof["instrumented_step_ms"] = statistics.mean(step_in)
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
        e2e_steps = max(3, min(steps, 500))
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
        d = run_cpu_oracle(wl_name, n_layers, tokens or 64, seconds=args.cpu_seconds)
        cpu = {"value": d["tokens"] / d["seconds"], "unit": UNIT, "cores": d["cores"], "kind": "oracle",
               "sample": f"{d['steps']} passes of one linear of the workload ({d['rows_per_step']} tokens each, "
                         f"float64 numpy oracle) in {d['seconds']:.1f} s"}

    if rank == 0:
        cfg = dict(desc)
        cfg.update({"variant": {0: "auto", 1: "fused", 2: "separate", 3: "cuda-core"}[args.variant],
                    "policy_variant": ags.lora_linear_policy(pool0.handle, n),
                    "distinct_slots_touched": alg["D"], "lora_tokens": alg["n_L"],
                    "concat_metrics": concat_metrics(idx_np, cases[0].h_in, cases[0].h_out, cases[0].adapters.ranks,
                                                     cases[0].adapters.r_max, cases[0].adapters.n_slots),
                    "l2": "inputs larger than L2 (no flush)", "timing": "CUDA graph replay, CUDA events",
                    "l2_prefetch_next_weight": prefetch,
                    "calls_per_step": len(calls),
                    "grouped": "projections reading the same x as one call each (lora_linear_fwd_group)" if grouped else None,
                    "parallelism": f"replicas x{world} (token batches sharded across GPUs, no collective)"})
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
                "warmup": warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16" if dtype == torch.bfloat16 else "f16", "data": "synthetic",
                "config": cfg, "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": int(kernels_per_step) * steps, "kernels_per_step": int(kernels_per_step),
                "clocks": clk}
        return line
    return None


def ours(args):
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
    peaks = load_peaks()
    line = measure(args, args.workload, args.steps, args.warmup, world, rank, local, dist, dev, peaks)
    if args.workload == "decode" and not args.no_prefill_leg:
        # the metric has two halves: decode against the HBM roofline (the line itself) and
        # prefill against the tensor roofline (this leg, measured the same way in the same run)
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        leg = measure(args, "prefill", min(args.steps, DEFAULT_STEPS["prefill"]), args.warmup, world, rank, local,
                      dist, dev, peaks)
        if line is not None:
            line["prefill"] = {k: leg[k] for k in ("value", "unit", "ms_per_step", "steps", "warmup", "dtype",
                                                   "config", "roofline", "cpu_baseline", "e2e", "gpu_launches",
                                                   "kernels_per_step", "clocks")}
    if line is not None:
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
    line["concurrent_with_decode"] = concurrent_mount(args)
    print(json.dumps(line), flush=True)


def concurrent_mount(args):
    """Decode steps (the headline workload: 64 tokens through 32 q_proj layers) with and without
    the adapter loader mounting new adapters in the background.

    Every step: the captured decode graph runs on the compute stream and is followed by a
    release fence on the slots the batch names; meanwhile lora_loader_mount puts k new rank-8
    adapters (all 32 layers' q_proj pieces, 4 MB each, from pinned host memory) into slots the
    batch does not name, on the copy stream (one loader call per step) -- the double buffering
    of the blog.lonae.com page's adapter loader.  Returns ms per step alone and with k = 1 and
    8 mounts per step."""
    import numpy as np
    import torch

    import adapter_gemm_segment_gb300 as ags
    from adapter_gemm_segment_gb300 import workloads as wl

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    compute, copy = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    n, layers, S, R, h = 64, 32, 100, 8, 4096
    cases = [wl.decode_q_proj(seed=1, n=n, layer=l) for l in range(layers)]
    idx = cases[0].idx
    named = sorted(set(idx[idx >= 0].tolist()))
    free = [sl for sl in range(S) if sl not in set(named)]
    L = []
    with torch.cuda.stream(compute):
        for c in cases:
            pool = ags.LoraPool(h, h, R, S, c.dtype, dev)
            L.append({"pool": pool, "W": c.W.to(dev), "x": c.x.to(dev), "y": torch.empty(n, h, dtype=c.dtype, device=dev)})
        loader = ags.LoraLoader([e["pool"] for e in L], copy)
        pinned = lambda t: t.contiguous().pin_memory()  # noqa: E731
        hostA = [pinned(torch.stack(c.adapters.A)) for c in cases]  # one pinned block per layer
        hostB = [pinned(torch.stack(c.adapters.B)) for c in cases]
        loader.mount(list(range(S)), [[a[sl] for sl in range(S)] for a in hostA],
                     [[b[sl] for sl in range(S)] for b in hostB], cases[0].adapters.alphas)
        loader.acquire(list(range(S)), compute)
        idx_dev = idx.to(dev)
        seg_ws = L[0]["pool"].segment_workspace(n, dev)
        ws = ags._device_bytes(ags.lora_linear_workspace_bytes(L[0]["pool"].handle, n), dev)
    torch.cuda.synchronize()
    # the adapters that keep arriving: 16 distinct rank-8 adapters, every layer's q_proj piece
    rng = np.random.default_rng(77)
    news = []
    for k in range(16):
        ad = wl.draw_adapters(rng, h, h, [R] * layers, [16.0] * layers, torch.float16)
        Ab, Bb = pinned(torch.stack(ad.A)), pinned(torch.stack(ad.B))
        news.append(([[Ab[l]] for l in range(layers)], [[Bb[l]] for l in range(layers)]))

    def step():
        seg = ags.lora_segment(idx_dev, L[0]["pool"].handle, seg_ws, stream=compute)
        for e in L:
            ags.lora_linear_fwd(e["pool"].handle, e["W"], e["x"], e["y"], seg, ws, stream=compute)

    with torch.cuda.stream(compute):
        step()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=compute):
            step()
    steps = max(50, min(args.steps, 2000))

    def run(k_mounts):
        for _ in range(max(3, args.warmup)):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(copy)
        e0.record(compute)
        t = 0
        for i in range(steps):
            if k_mounts:  # the next k adapters land (one loader call) while this step computes
                picks = [t + j for j in range(k_mounts)]
                slots = [free[q % len(free)] for q in picks]
                As = [[news[q % len(news)][0][l][0] for q in picks] for l in range(layers)]
                Bs = [[news[q % len(news)][1][l][0] for q in picks] for l in range(layers)]
                loader.mount(slots, As, Bs, [16.0] * k_mounts)
                t += k_mounts
            with torch.cuda.stream(compute):
                g.replay()
            loader.release(named, compute)
        e1.record(compute)
        c1.record(copy)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps, c0.elapsed_time(c1), t

    alone, _, _ = run(0)
    out = {"decode_ms_per_step_alone": alone}
    for k in (1, 8):
        ms, copy_ms, mounted = run(k)
        out[f"decode_ms_per_step_with_{k}_mounts"] = ms
        out[f"mount_GBps_with_{k}_mounts"] = mounted * layers * 2 * (2 * R * h) / (copy_ms * 1e-3) / 1e9
    # the last mounted adapters are resident and exact: compare one layer's pool slot with its source
    out["mounts"] = loader.stats()["mounts"]
    out["config"] = (f"decode 64 tokens x 32 q_proj layers (4096x4096 fp16, 100 slots r=8); per step k new rank-8 "
                     f"adapters (32 layers x 128 KB each) mounted from pinned host memory on a copy stream into "
                     f"slots the batch does not name; {steps} steps")
    loader.close()
    return out


def concat_compare(args):
    """--workload concat: the segmented path against the concatenated-adapter matmul of the
    blog.lonae.com page (tensor-concatenation paragraph) on the same decode batches.

    That approach stacks every adapter of the pool (zero-padded to r_max) into A_cat
    [S*r_max, h_in] and B_cat [h_out, S*r_max], multiplies every token against all of them,
    keeps each token's own block (scaled by alpha/r) and multiplies back:
        y = x W^T + ((x A_cat^T) * M) B_cat^T,   M[t, s*r_max + j] = scale_s if idx[t] == s.
    It runs here as plain cuBLAS GEMMs (torch.matmul) captured in a CUDA graph -- a baseline
    for comparison, not part of the library.  Both sides run 32 chained decode q_proj linears
    (4096 x 4096 fp16, 100 rank-8 adapters, Zipf(1.1) + 10 % base-only) per step."""
    import numpy as np
    import torch

    import adapter_gemm_segment_gb300 as ags
    from adapter_gemm_segment_gb300 import workloads as wl

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)
    layers = args.layers
    rows = []
    for n in (1, 8, 64):
        cases = [wl.decode_q_proj(seed=1, n=n, layer=l) for l in range(layers)]
        idx = cases[0].idx
        S, R, h = 100, 8, 4096
        L = []
        for c in cases:
            ad = c.adapters
            pool = ags.LoraPool(h, h, R, S, c.dtype, dev)
            for sl in range(S):
                pool.load_slot(sl, ad.A[sl].to(dev), ad.B[sl].to(dev), ad.alphas[sl])
            L.append({"pool": pool, "W": c.W.to(dev), "x": c.x.to(dev), "y": torch.empty(n, h, dtype=c.dtype, device=dev),
                      "yc": torch.empty(n, h, dtype=c.dtype, device=dev), "ad": ad})
        torch.cuda.synchronize()
        # the concatenated matrices, from each pool's own zero-padded slabs
        a_off = 256 * ((S * 16 + 255) // 256)
        for e in L:
            mem = e["pool"].mem
            A_slab = mem[a_off:a_off + S * R * h * 2].view(torch.float16).view(S * R, h)
            b_off = (a_off + S * R * h * 2 + 255) // 256 * 256
            B_slab = mem[b_off:b_off + S * h * R * 2].view(torch.float16).view(S, h, R)
            e["A_cat"] = A_slab
            e["B_cat"] = B_slab.permute(1, 0, 2).reshape(h, S * R).contiguous()
        mask = torch.zeros(n, S * R, dtype=torch.float16)
        for t, sl in enumerate(idx.tolist()):
            if sl >= 0:
                mask[t, sl * R:(sl + 1) * R] = L[0]["ad"].alphas[sl] / L[0]["ad"].ranks[sl]
        mask = mask.to(dev)
        idx_dev = idx.to(dev)
        seg_ws = L[0]["pool"].segment_workspace(n, dev)
        ws = ags._device_bytes(ags.lora_linear_workspace_bytes(L[0]["pool"].handle, n), dev)

        def seg_step():
            seg = ags.lora_segment(idx_dev, L[0]["pool"].handle, seg_ws)
            for e in L:
                ags.lora_linear_fwd(e["pool"].handle, e["W"], e["x"], e["y"], seg, ws)

        def concat_step():
            for e in L:
                s_all = torch.matmul(e["x"], e["A_cat"].t())
                torch.add(torch.matmul(e["x"], e["W"].t()), torch.matmul(s_all * mask, e["B_cat"].t()), out=e["yc"])

        def graph_ms(fn, reps):
            fn()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn()
            for _ in range(max(3, args.warmup)):
                g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / reps

        reps = max(20, min(args.steps, 500))
        ms_seg = graph_ms(seg_step, reps)
        ms_cat = graph_ms(concat_step, reps)
        # both compute the same layer: the concatenated result must pass the float bar against ours
        y0, yc0 = L[0]["y"].double().cpu(), L[0]["yc"].double().cpu()
        agree = bool(((y0 - yc0).abs() <= 1e-2 + 1e-2 * y0.abs()).all())
        m = concat_metrics(idx.numpy(), h, h, [R] * S, R, S)
        n_L = int((idx >= 0).sum())
        rows.append({"tokens": n, "segmented_us_per_linear": 1e3 * ms_seg / layers,
                     "concat_us_per_linear": 1e3 * ms_cat / layers, "concat_over_segmented": ms_cat / ms_seg,
                     "lora_flops_segmented": 2 * n_L * R * 2 * h, "lora_flops_concat": 2 * n * S * R * 2 * h,
                     "concat_lora_flops_wasted_share": m["concat_lora_flops_wasted_share"],
                     "concat_elements": m["concat_elements"], "concat_projection": m["concat_projection"],
                     "distinct_adapters": m["distinct_adapters"], "n_segments": m["n_segments"],
                     "results_agree_within_tolerance": agree})
        del L, cases
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    line = {"metric": "decode LoRA-linear time: segmented path vs the concatenated-adapter matmul",
            "value": rows[-1]["segmented_us_per_linear"], "unit": "us per linear", "higher_is_better": False,
            "n_gpus": 1, "steps": max(20, min(args.steps, 500)), "warmup": max(3, args.warmup), "dtype": "f16",
            "data": "synthetic",
            "config": {"workload": f"decode q_proj 4096x4096 fp16, {layers} chained layers per step, 100 adapters "
                                   "r=8 alpha=16, Zipf(1.1) + 10% base-only; batches of 1, 8 and 64 tokens",
                       "concat_impl": "cuBLAS GEMMs through torch.matmul in a CUDA graph (baseline only)",
                       "timing": "CUDA graph replay, CUDA events"},
            "rows": rows}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.workload == "load":
        adapter_load(args)
    elif args.workload == "concat":
        concat_compare(args)
    elif args.impl == "reference":
        reference_arm(args)
    else:
        ours(args)


if __name__ == "__main__":
    main()
