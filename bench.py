"""Throughput of the routed-expert layer (route + forward) on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAMES] [--impl reference]

A step is one pass of the whole layer -- k3moe_route then k3moe_forward -- over one
batch of T synthetic tokens whose weights and activations are already resident in
HBM.  The 129 MB L2 is flushed between steps (a 512 MiB buffer is written outside
the timed events).  value = tokens processed by all ranks / the slowest rank's summed
step time (CUDA events on the launching stream).  e2e times the same step end to end:
torch copies x from pinned host memory to the device, the two C-ABI calls run, and out
is copied back to pinned host memory, all inside the timed events.

--workload takes a comma-separated list; the default, decode_t1,prefill_t4096, is the
headline pair (T = 1 and T = 4096 at the K3 shape).  The first workload's record is the
JSON line's top level; every other workload's complete record sits under a key named
after it.

With N > 1 (torchrun, one process per GPU) every rank runs an independent replica of
the layer: the path has no exchange step on one GPU, so there is no collective in the
data path; a barrier and a max-reduction of the timings bracket the run.

--impl reference times the CPU oracle (oracle/, fp64 C) on this host's cores on a
bounded sample of the same workloads, as the reference arm.
"""
from __future__ import annotations

import argparse
import glob
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

METRIC = "MoE-layer tokens/s at T=1 and T=4096 on 1 GB300; % of HBM/tensor roofline"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
DEFAULT_WORKLOADS = "decode_t1,prefill_t4096"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=30)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--workload", default=DEFAULT_WORKLOADS,
                   help="comma-separated workloads; the first is the line's top-level record")
    p.add_argument("--impl", default="k3moe", choices=["k3moe", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--cpu-budget-s", type=float, default=15.0)
    p.add_argument("--graph", action="store_true",
                   help="replay route + forward as one captured CUDA graph per step")
    p.add_argument("--prefill-gemm", default="default", choices=["default", "f16", "block_scaled"],
                   help="kernel of the prefill path's routed projections (k3moe_set_prefill_gemm)")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# ----------------------------------------------------------------------------- replicas (N > 1)
# The layer does not shard: N GPUs run N independent replicas of the same step.  The
# only collectives are the timing barrier and the max over ranks of the timed region.

def dist_barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def dist_max(v: float, world: int, device=None) -> float:
    """Max of v over the ranks of the initialised process group (v itself when N = 1)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world: int, tokens_per_step: int, steps: int, ms_max: float) -> float:
    """Whole-job tokens/s: each replica processes tokens_per_step per step, and the job
    takes as long as the slowest replica."""
    return world * tokens_per_step * steps / (ms_max / 1000.0)


# ----------------------------------------------------------------------------- algorithmic work

def layer_bytes_flops(w, distinct_experts: int):
    """Algorithmic bytes and FLOPs of one layer call: the distinct routed experts
    touched (packed MXFP4), the shared experts (bf16), the router (bf16), x in (bf16)
    and out (f32).  FLOPs: 2*3*f*d per (token, expert) for k routed + S shared experts,
    plus 2*E*d per token for the router."""
    if w.hidden:
        return block_bytes_flops(w, distinct_experts)
    Be = w.expert_bytes
    shared = w.S * 3 * w.f * w.d * 2
    router = w.E * w.d * 2
    act = w.T * w.d * 2 + w.T * w.d * 4
    byts = distinct_experts * Be + shared + router + act
    flops = w.T * (2 * 3 * w.f * w.d * (w.k + w.S) + 2 * w.E * w.d)
    return byts, flops


def block_bytes_flops(w, distinct_experts: int):
    """Algorithmic bytes and FLOPs of one full-width block call: the distinct routed
    experts, the full-width router [E,H], the down [d,H] and up [H,d] projections, the
    fused shared experts (3*H*S*f bf16), h in (bf16) and out (f32).  FLOPs per token:
    2*E*H (router) + 2*2*d*H (projections) + 2*3*f*d*k (routed) + 2*3*H*S*f (shared)."""
    H, SI = w.hidden, w.S * w.f
    byts = (distinct_experts * w.expert_bytes + w.E * H * 2 + 2 * w.d * H * 2 + 3 * H * SI * 2
            + w.T * H * 2 + w.T * H * 4)
    flops = w.T * (2 * w.E * H + 4 * w.d * H + 2 * 3 * w.f * w.d * w.k + 2 * 3 * H * SI)
    return byts, flops


def full_kernel_work(name: str, w, distinct_experts: int):
    """kernel_work for a full-width block: its dense projections (weights, activations in
    and out; 2*m*n*k FLOPs), else the layer's kernels as the block runs them (router on
    width H, experts on the latent without shared experts)."""
    T, H, d, SI = w.T, w.hidden, w.d, w.S * w.f
    if name == "full_down_proj":
        return d * H * 2 + T * H * 2 + T * d * 2, 2 * T * d * H
    if name == "full_up_proj":
        return H * d * 2 + T * d * 2 + T * H * 4, 2 * T * H * d
    if name == "full_shared_gateup":
        return 2 * SI * H * 2 + T * H * 2 + T * SI * 2, 2 * 2 * T * SI * H
    if name == "full_shared_down":
        return H * SI * 2 + T * SI * 2 + 2 * T * H * 4, 2 * T * H * SI
    if name in ("router_scores", "router_logits_tc", "router_wnorm"):
        return kernel_work(name, w.with_(d=H, hidden=0), distinct_experts)
    if name in ("gemv_gateup", "gemv_down", "gemm_gateup", "gemm_down", "gemm_gateup_mx", "gemm_down_mx"):
        return kernel_work(name, w.with_(S=0, hidden=0), distinct_experts)
    return block_bytes_flops(w, distinct_experts)[0], 0


def kernel_work(name: str, w, distinct_experts: int, block_scaled: bool = False):
    """Algorithmic (bytes, FLOPs) of one launch of a forward kernel: the bytes it must
    move and the multiply-adds (x2) it must do.
    router_scores: Wr and x in, sc and ch out (f32); router_logits_tc: Wr and x in, the
    logits out (f32); 2*T*E*d FLOPs each.  router_wnorm: Wr in.
    gemv_gateup / gemm_gateup: W1, W3 of the distinct routed experts (packed MXFP4,
    17/32 byte per weight) and of the shared experts (bf16), the activations in (x;
    the gathered f16 copy on the GEMM path) and h out (f16 for routed rows; on the
    mat-vec path a bf16 hi + lo pair for shared rows); 2 * rows * 2*f*d FLOPs with
    rows = T*k + S*T.  gemv_down / gemm_down: W2 likewise, h in, the output out.
    Any other kernel is charged the whole layer's bytes and no FLOPs."""
    if w.hidden:
        return full_kernel_work(name, w, distinct_experts)
    rows = w.T * w.k + w.S * w.T
    slots = w.T * w.k
    h_gemv = slots * w.f * 2 + w.S * w.T * w.f * 4
    if name == "gemm_gateup_mx":
        # routed rows only: the packed W1, W3 (codes and scales as they are), the two e4m3
        # token planes and their scale bytes in, h as two e4m3 planes and scale bytes out
        return (distinct_experts * 2 * w.f * w.d * 17 // 32 + slots * w.d * 2 + slots * w.d // 16
                + slots * w.f * 2 + slots * w.f // 16), 2 * slots * 2 * w.f * w.d
    if name == "gemm_down_mx":
        # routed rows only: the packed W2, h's two planes and scale bytes in, the output
        # (f32, accumulated in place) read and written once
        return (distinct_experts * w.d * w.f * 17 // 32 + slots * w.f * 2 + slots * w.f // 16
                + 2 * w.T * w.d * 4), 2 * slots * w.f * w.d
    if name == "gemm_gateup" and block_scaled:
        # beside the block-scaled kernels, the f16 kernel runs the shared experts alone
        return (w.S * 2 * w.f * w.d * 2 + w.T * w.d * 2 + w.S * w.T * w.f * 2), 2 * w.S * w.T * 2 * w.f * w.d
    if name == "gemm_down" and block_scaled:
        return (w.S * w.d * w.f * 2 + w.S * w.T * w.f * 2 + 2 * w.T * w.d * 4), 2 * w.S * w.T * w.f * w.d
    if name == "router_scores":
        return w.E * w.d * 2 + w.T * w.d * 2 + 2 * w.T * w.E * 4, 2 * w.T * w.E * w.d
    if name == "router_logits_tc":
        return w.E * w.d * 2 + w.T * w.d * 2 + w.T * w.E * 4, 2 * w.T * w.E * w.d
    if name == "router_wnorm":
        return w.E * w.d * 2, 2 * w.E * w.d
    if name == "gemv_gateup":
        return (distinct_experts * 2 * w.f * w.d * 17 // 32 + w.S * 2 * w.f * w.d * 2
                + w.T * w.d * 2 + h_gemv), 2 * rows * 2 * w.f * w.d
    if name == "gemv_down":
        return (distinct_experts * w.d * w.f * 17 // 32 + w.S * w.d * w.f * 2
                + h_gemv + rows * w.d * 4), 2 * rows * w.f * w.d
    if name == "gemm_gateup":
        return (distinct_experts * 2 * w.f * w.d * 17 // 32 + w.S * 2 * w.f * w.d * 2
                + slots * w.d * 2 + w.T * w.d * 2 + rows * w.f * 2), 2 * rows * 2 * w.f * w.d
    if name == "gemm_down":
        return (distinct_experts * w.d * w.f * 17 // 32 + w.S * w.d * w.f * 2
                + rows * w.f * 2 + w.T * w.d * 4), 2 * rows * w.f * w.d
    return layer_bytes_flops(w, distinct_experts)[0], 0


def workload_specs(arg: str):
    """The comma-separated workload list; a `key=value` item without a name continues the
    overrides of the workload before it (decode_t1:E=64,T=4 is one workload)."""
    specs = []
    for part in (p.strip() for p in arg.split(",")):
        if not part:
            continue
        if "=" in part and ":" not in part and specs:
            specs[-1] += "," + part
        else:
            specs.append(part)
    return specs


def workload_from(spec: str):
    """NAME or NAME:key=value,key=value (integer overrides, e.g. decode_t1:E=64)."""
    import k3moe_inputs as ki
    name, _, over = spec.partition(":")
    w = ki.WORKLOADS[name]
    if over:
        kw = {}
        for item in over.split(","):
            k, v = item.split("=")
            kw[k.strip()] = int(v)
        w = w.with_(name=spec, **kw)
    return w


def peaks():
    try:
        with open(PEAKS_FILE) as fh:
            pk = json.load(fh)
        return float(pk["hbm_gbs"]), float(pk["bf16_tflops"]), float(pk["bf16_tflops_sustained"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


# The source files that hold each timed kernel's device code (its own file, and the
# tensor-core helpers for the tcgen05 kernels).
KERNEL_SOURCES = {
    "gemv_gateup": ["k3moe_gemv.cu"], "gemv_down": ["k3moe_gemv.cu"],
    "gemm_gateup": ["k3moe_gemm.cu", "k3moe_tc.cuh"], "gemm_down": ["k3moe_gemm.cu", "k3moe_tc.cuh"],
    "gemm_gateup_mx": ["k3moe_gemm.cu", "k3moe_tc.cuh"], "gemm_down_mx": ["k3moe_gemm.cu", "k3moe_tc.cuh"],
    "router_logits_tc": ["k3moe_route_tc.cu", "k3moe_tc.cuh"],
    "full_down_proj": ["k3moe_dense.cu", "k3moe_tc.cuh"], "full_up_proj": ["k3moe_dense.cu", "k3moe_tc.cuh"],
    "full_shared_gateup": ["k3moe_dense.cu", "k3moe_tc.cuh"], "full_shared_down": ["k3moe_dense.cu", "k3moe_tc.cuh"],
}


def csrc_hash(kernel: str):
    """Hash of the files that hold a kernel's device code.  A recorded DRAM traffic figure
    is reported only while this matches the hash taken with it."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_moe_expert_k3moe_gb300", "csrc")
    for name in sorted(KERNEL_SOURCES.get(kernel, [])):
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_for(kernel: str, workload: str):
    """dram read+write bytes per launch from a committed ncu summary, or None when
    absent or taken on a different kernel source."""
    try:
        with open(TRAFFIC_FILE) as fh:
            tr = json.load(fh)
        ent = tr[workload][kernel]
        if ent.get("csrc_hash") != csrc_hash(kernel):
            return None
        return float(ent["dram_bytes_per_launch"])
    except Exception:
        return None


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if not self.rows:
            return None
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in self.rows:
            for i, n in enumerate(names):
                if r[5 + i].lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "samples": len(self.rows), "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- CPU oracle timing

def time_oracle(w, budget_s: float):
    """Route + forward of the oracle on this host's cores over a bounded sample of the
    workload: its first tokens (one batch of as many tokens as the oracle has threads, at
    most 16), cycled until budget_s seconds of oracle work, so that the routed experts
    they use are drawn once; returns (tokens/s, tokens timed, threads, seconds)."""
    import numpy as np
    import k3moe_inputs as ki
    import oracle
    c = oracle.cfg(**w.config_kwargs())
    bias = ki.make_bias(w)
    if w.hidden:
        # the full-width block: route on h, then the block's six steps
        c_route = oracle.cfg(**dict(w.config_kwargs(), d=w.hidden))
        x, Wr, full = ki.make_h(w), ki.make_full_router(w), ki.make_full(w)
        shared = {"w1": full["sh1"], "w3": full["sh3"], "w2": full["sh2"]} if w.S else None

        def run(xs, idx, wt):
            oracle.forward_full(c, w.hidden, w.latent_norm, w.rms_eps, xs, idx, wt, full["down"],
                                experts, full["gain"], full["up"], shared)
    else:
        c_route = c
        x, Wr = ki.make_x(w), ki.make_router(w)
        shared = ki.make_shared(w) if w.S else None

        def run(xs, idx, wt):
            oracle.forward(c, xs, idx, wt, experts, shared)
    batch = max(1, min(w.T, oracle.num_threads(), 16))
    xs = np.ascontiguousarray(x[:batch])
    idx, wt, _ = oracle.route(c_route, xs, Wr, bias)        # untimed draw of the needed experts
    experts = {e: ki.make_expert(w, e) for e in sorted(set(idx.ravel().tolist()))}
    done, spent = 0, 0.0
    while spent < budget_s:
        t0 = time.perf_counter()
        idx, wt, _ = oracle.route(c_route, xs, Wr, bias)
        run(xs, idx, wt)
        spent += time.perf_counter() - t0
        done += batch
    return done / spent, done, oracle.num_threads(), spent


def reference_arm(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    specs = workload_specs(args.workload)
    per_step = max(2.0, args.cpu_budget_s / max(1, args.steps))
    records = []
    for spec in specs:
        w = workload_from(spec)
        for _ in range(args.warmup):
            time_oracle(w.with_(T=1), 0.1)
        tot_tok, tot_s = 0, 0.0
        threads = oracle.num_threads()
        for _ in range(args.steps):
            tps, n, threads, s = time_oracle(w, per_step)
            tot_tok += n
            tot_s += s
        value = tot_tok / tot_s
        records.append({
            "value": value, "unit": "tokens/s", "ms_per_step": 1000.0 * tot_s / args.steps,
            "dtype": "f64",
            "config": {"workload": w.name, "T": w.T, "d": w.d, "f": w.f, "E": w.E, "top_k": w.k,
                       "n_shared": w.S},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": f"{tot_tok} tokens of {w.name} (its first tokens, cycled) over "
                                       f"{args.steps} steps (each step <= {per_step:.1f} s of oracle work)"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        })
    line = {"impl": "reference", "metric": METRIC, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "data": "synthetic", **records[0]}
    for spec, rec in zip(specs[1:], records[1:]):
        line[rec["config"]["workload"]] = rec
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU arm

ARITHMETIC = ("router: exact logits (bf16 products exact in fp32, two-sum compensated "
              "accumulation, one rounding), sigmoid from a correctly rounded float exp (fp32 double-float arithmetic); experts: "
              "MMA operands f16 (tokens x*2^-u, routed h; MXFP4 weights decoded exactly to f16) "
              "and bf16 (shared-expert weights, shared h), fp32 accumulation; on the prefill path "
              "the routed experts' projections by default on block-scaled MMAs (kind::mxf8f6f4: the "
              "E2M1 codes with their E8M0 scales as packed, the tokens and h as two e4m3 planes "
              "with E8M0 scales per 32, fp32 accumulation); output f32")


def near_tie_counts(layer, x, w):
    """From the device's exact router scores (k3moe_router_scores, every expert of every
    token): tokens whose k-th and (k+1)-th choice scores differ by less than 1e-6 without
    being equal, and tokens where they are exactly equal (decided by the lower index)."""
    import numpy as np
    if w.E <= w.k:
        return {"tokens": w.T, "gap_below_1e-6": 0, "exact_ties": 0}
    _, ch = layer.scores(x)
    top = -np.sort(-np.partition(ch.cpu().numpy(), w.E - w.k - 1, axis=1)[:, w.E - w.k - 1:], axis=1)
    gap = top[:, w.k - 1].astype(np.float64) - top[:, w.k].astype(np.float64)
    return {"tokens": w.T, "gap_below_1e-6": int(((gap > 0) & (gap < 1e-6)).sum()),
            "exact_ties": int((gap == 0).sum()),
            "from": "the device's exact scores (k3moe_router_scores)"}


def measure(w, args, rank, world, local, dev):
    """One workload: the timed steps, the per-kernel pass, e2e, the near-tie count and
    (rank 0, N = 1) the CPU baseline; returns the record (rank 0) or None."""
    import numpy as np
    import torch
    import k3moe_inputs as ki
    from k3moe_inputs.device import build_layer
    import sparse_moe_expert_k3moe_gb300 as k3

    k3.k3moe_set_prefill_gemm({"default": k3.PREFILL_GEMM_DEFAULT, "f16": k3.PREFILL_GEMM_F16,
                               "block_scaled": k3.PREFILL_GEMM_BLOCK_SCALED}[args.prefill_gemm])
    width = w.hidden or w.d                                   # token width in and out
    if w.hidden:
        from k3moe_inputs.device import build_block
        layer = build_block(w, device=dev)
        x = torch.from_numpy(ki.make_h(w).view(np.int16)).to(dev)
    else:
        layer = build_layer(w, device=dev)
        x = torch.from_numpy(ki.make_x(w).view(np.int16)).to(dev)
    out = torch.empty((w.T, width), dtype=torch.float32, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def layer_call(xin, stream):
        if w.hidden:
            layer.forward(xin, out, stream)
        else:
            layer.route(xin, stream)
            layer.forward(xin, out, stream)

    def eager_step():
        layer_call(x, stream)

    step = eager_step
    graph_launches = None
    if args.graph:
        n0 = k3.k3moe_launch_count()
        graph = layer.capture(x, out)
        graph_launches = (k3.k3moe_launch_count() - n0) // 2      # the eager call + the capture
        step = graph.replay

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    rc, code = k3.k3moe_device_status(layer.ws)
    if rc != 0:
        raise RuntimeError(f"device status {code:#x} after warm-up")
    distinct = int(torch.unique(layer.idx[: w.T]).numel())

    # ---- timed region: K steps, L2 flushed between steps outside the events
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    dist_barrier(world)
    torch.cuda.synchronize(dev)
    n0 = k3.k3moe_launch_count()
    host_s = 0.0
    for i in range(args.steps):
        flush.fill_(i & 255)
        ev[i][0].record(stream)
        h0 = time.perf_counter()
        step()
        host_s += time.perf_counter() - h0
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    dist_barrier(world)
    launches = k3.k3moe_launch_count() - n0
    if graph_launches is not None:
        launches = graph_launches * args.steps
    clk = clocks.stop()
    ms = sum(a.elapsed_time(b) for a, b in ev)
    ms = dist_max(ms, world, dev)
    value = job_value(world, w.T, args.steps, ms)

    # ---- per-kernel durations (separate pass, same work, library-side CUDA events)
    k3.k3moe_timing_reset()
    k3.k3moe_timing_enable(True)
    for i in range(args.steps):
        flush.fill_(i & 255)
        eager_step()
    torch.cuda.synchronize(dev)
    k3.k3moe_timing_enable(False)
    kt = k3.k3moe_timing_read()
    top_name, (top_n, top_ms) = max(kt.items(), key=lambda kv: kv[1][1])
    hbm, bf16, bf16_sus, src = peaks()
    per_launch_s = top_ms / top_n / 1000.0
    block_scaled = "gemm_gateup_mx" in kt
    alg_b, alg_f = kernel_work(top_name, w, distinct, block_scaled)
    # the kernel's bound: whichever of HBM and the tensor cores its algorithmic work needs
    # longer on.  The per-kernel pass times launches of at most milliseconds, so the tensor
    # peak is the burst figure (the sustained one is for seconds-long loops).  The
    # block-scaled GEMM's MMAs (kind::mxf8f6f4: e4m3 x e2m1) take the FP8 peak: the measured
    # bf16 burst figure times the nominal FP8/BF16 ratio (4.5 / 2.25 PFLOP/s).
    fp8 = top_name in ("gemm_gateup_mx", "gemm_down_mx")
    tpeak = bf16 * (2.0 if fp8 else 1.0)
    if alg_f / (tpeak * 1e12) > alg_b / (hbm * 1e9):
        roof = {"bound": "tensor", "achieved": alg_f / per_launch_s / 1e12, "peak": tpeak,
                "unit": "TFLOP/s",
                "peak_kind": ("fp8 dense, burst: the measured bf16 burst x 2 (nominal fp8/bf16); the "
                              "tokens are two e4m3 terms, so the MMAs execute twice the algorithmic "
                              "FLOPs (at most 0.5 of this peak by construction)") if fp8
                else "bf16 dense, burst (f16 runs at the same rate)"}
        roof["frac_of_sustained"] = roof["achieved"] / (bf16_sus * (2.0 if fp8 else 1.0))
        if fp8:
            roof["frac_of_bf16_burst"] = roof["achieved"] / bf16
    else:
        roof = {"bound": "hbm", "achieved": alg_b / per_launch_s / 1e9, "peak": hbm, "unit": "GB/s",
                "peak_kind": "HBM copy"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    if alg_f:
        # the algorithmic FLOPs at the bf16 dense burst peak, whatever the kernel's bound
        roof["bf16_tensor_frac"] = alg_f / per_launch_s / 1e12 / bf16
    step_bytes, step_flops = layer_bytes_flops(w, distinct)
    step_s = ms / args.steps / 1000.0
    t_roof = max(step_bytes / (hbm * 1e9), step_flops / (bf16 * 1e12))

    # ---- end to end: pinned host x -> device, the C-ABI calls, device out -> pinned host
    e2e = None
    if not args.no_e2e:
        xh = x.cpu().pin_memory()
        oh = torch.empty((w.T, width), dtype=torch.float32).pin_memory()
        xd = x if args.graph else torch.empty_like(x)
        ee = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        for i in range(args.steps + 2):
            flush.fill_(i & 255)
            if i >= 2:
                ee[i - 2][0].record(stream)
            xd.copy_(xh, non_blocking=True)
            if args.graph:
                step()
            else:
                layer_call(xd, stream)
            oh.copy_(out, non_blocking=True)
            if i >= 2:
                ee[i - 2][1].record(stream)
        torch.cuda.synchronize(dev)
        ems = dist_max(sum(a.elapsed_time(b) for a, b in ee), world, dev)
        e2e = {"value": job_value(world, w.T, args.steps, ems), "unit": "tokens/s",
               "h2d_bytes_per_step": int(xh.numel() * xh.element_size()),
               "d2h_bytes_per_step": int(oh.numel() * oh.element_size()),
               "how": "torch copies between pinned host buffers and the device around the "
                      "C-ABI calls, inside the timed events"}

    ties = None
    if rank == 0 and not w.hidden:
        ties = near_tie_counts(layer, x, w)
    del layer, flush
    torch.cuda.empty_cache()

    # ---- CPU oracle baseline (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tps, n, threads, s = time_oracle(w, args.cpu_budget_s)
        cpu = {"value": tps, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": f"{n} tokens of {w.name} (its first {min(w.T, threads, 16)} tokens, cycled), "
                         f"route + forward, {s:.1f} s of oracle work"}
    if rank != 0:
        return None
    return {
        "value": value, "unit": "tokens/s", "steps": args.steps, "warmup": max(3, args.warmup),
        "ms_per_step": ms / args.steps, "dtype": "f16",
        "config": {"workload": w.name, "T": w.T, "d": w.d, "f": w.f, "E": w.E, "top_k": w.k,
                   "n_shared": w.S, **({"hidden": w.hidden, "latent_norm": w.latent_norm}
                                       if w.hidden else {}),
                   "weights": "routed MXFP4 (E2M1 + E8M0/32), shared bf16"
                              + (", dense projections bf16" if w.hidden else ""),
                   "arithmetic": ARITHMETIC,
                   "l2": "512 MiB buffer written between timed steps",
                   "launch": "one CUDA graph replay per step" if args.graph else "eager",
                   "prefill_gemm": ("block_scaled (routed gate/up and down on kind::mxf8f6f4)" if block_scaled
                                    else ("f16 on dequantised weights" if "gemm_gateup" in kt
                                          else "not used (mat-vec path)")),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": dict(roof, kernel=top_name, peak_source=src,
                         traffic=traffic_for(top_name, w.name), alg_bytes_per_launch=alg_b,
                         alg_flops_per_launch=alg_f, launch_ms=per_launch_s * 1e3),
        "step_roofline": {"bytes": step_bytes, "flops": step_flops, "distinct_experts": distinct,
                          "hbm_frac": step_bytes / step_s / 1e9 / hbm,
                          "tensor_frac": step_flops / step_s / 1e12 / bf16,
                          "bound": "hbm" if step_bytes / (hbm * 1e9) >= step_flops / (bf16 * 1e12)
                                   else "tensor",
                          "frac": t_roof / step_s,
                          "peaks": f"HBM {hbm:.0f} GB/s, bf16 {bf16:.0f} TFLOP/s burst ({src})"},
        "kernels": {k: {"launches": v[0], "ms": v[1]} for k, v in kt.items()},
        "gpu_launches": launches,
        "host_enqueue_ms_per_step": 1000.0 * host_s / args.steps,
        "router_near_ties": ties,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "clocks": clk,
    }


def gpu_arm(args):
    import torch
    from sparse_moe_expert_k3moe_gb300 import build as kbuild

    rank, world, local = dist_env()
    kbuild.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    specs = workload_specs(args.workload)
    records = [measure(workload_from(sp), args, rank, world, local, dev) for sp in specs]
    if rank == 0:
        line = {"metric": METRIC, "n_gpus": world, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "data": "synthetic", **records[0]}
        for rec in records[1:]:
            line[rec["config"]["workload"]] = rec
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
