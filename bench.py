"""Benchmark of the gpt-oss MoE layer forward on GB300.

One step = one moe_forward (router+top-k, permutation, gate_up GEMM + GLU,
down GEMM + weighted combine) over one batch of T tokens whose activations,
router and expert weights are already resident in HBM.  The default
workload is the gpt-oss-20b layer (hidden 2880, 32 experts top-4, expert
inter 2880) at decode batch T=64 with near-uniform routing, seed 1.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--T T]

Under torchrun each rank runs an independent replica on its own GPU (the
layer is replicated, there is no collective on the data path); the timed
region is bracketed by a barrier and a device synchronisation on both
sides, and the maximum time over ranks is reported.  ``--impl reference``
times the CPU oracle (the only reference this layer has) on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "MoE-layer tokens/s; decode HBM GB/s & prefill TFLOPS as % of GB300 roofline"

# Algorithmic bytes per expert (bf16 weights and biases).
GU_BYTES = lambda H, I: 2 * I * H * 2 + 2 * I * 2          # noqa: E731
D_BYTES = lambda H, I: H * I * 2 + H * 2                    # noqa: E731
GU_BYTES_MXFP4 = lambda H, I: 2 * I * H // 2 + 2 * I * H // 32 + 2 * I * 2  # noqa: E731
D_BYTES_MXFP4 = lambda H, I: H * I // 2 + H * I // 32 + H * 2               # noqa: E731
# FP8 W8A8: one E4M3 byte per weight, the bf16 biases and one fp32 scale
GU_BYTES_FP8 = lambda H, I: 2 * I * H + 2 * I * 2 + 4                   # noqa: E731
D_BYTES_FP8 = lambda H, I: H * I + H * 2 + 4                            # noqa: E731

DESCRIPTIONS = {
    "20b_t8": "gpt-oss-20b MoE layer, T={T}, bf16, seed 0",
    "20b_decode": "gpt-oss-20b MoE layer decode, T={T}, bf16, near-uniform routing, seed 1",
    "20b_prefill_skewed": "gpt-oss-20b MoE layer prefill, T={T}, bf16, +2.0 router bias on "
                          "4 hot experts, 1% activation outliers x20, seed 2",
    "120b_shape": "gpt-oss-120b-shaped MoE layer (128 experts top-4), T={T}, bf16, "
                  "near-uniform routing, seed 3",
    "20b_mxfp4": "gpt-oss-20b MoE layer, MXFP4 expert weights, T={T}, seed 4",
    "20b_fp8": "gpt-oss-20b MoE layer, FP8 W8A8 (E4M3 weights, per-expert scales; per-token E4M3 activations), T={T}, seed 5",
    "20b_mxfp4_mxfp8": "gpt-oss-20b MoE layer, MXFP4 expert weights (those of 20b_mxfp4) with "
                       "MXFP8 activations on the block-scaled MMA, T={T}, seed 4",
}


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(
            p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def kernel_source_sha(name="grouped_gemm.cu"):
    with open(os.path.join(ROOT, "gpt_oss_moe_gb300", "csrc", name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def recorded_traffic(kernel, workload):
    """dram bytes per launch from a committed ncu summary, if still current."""
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    sha = kernel_source_sha()
    for fn in sorted(os.listdir(pdir)):
        try:
            text = open(os.path.join(pdir, fn)).read()
        except OSError:
            continue
        for m in re.finditer(r"^traffic_record: (\{.*\})\s*$", text, flags=re.M):
            try:
                rec = json.loads(m.group(1))
            except ValueError:
                continue
            if rec.get("kernel") == kernel and rec.get("workload") == workload and \
                    rec.get("source_sha256") == sha:
                return float(rec["bytes_per_launch"])
    return None


class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_id):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", device_id],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [c.strip() for c in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        inside = [s for t, s in self.samples if t0 <= t <= t1 + 0.25]
        used = inside if inside else [s for _, s in self.samples]
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"],
                    "samples": 0}
        sm = [float(s[1]) for s in used if s[1].replace(".", "").isdigit()]
        smax = [float(s[2]) for s in used if s[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in used:
            for name, v in zip(names, s[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(used),
                "window": "timed region" if inside else "whole run (timed region shorter "
                                                         "than the 200 ms sampling period)"}


def device_id_for_smi():
    try:
        u = torch.cuda.get_device_properties(torch.cuda.current_device()).uuid
        return "GPU-" + str(u)
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        return vis.split(",")[torch.cuda.current_device()] if vis else str(
            torch.cuda.current_device())


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        return world, rank, local, dist
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    return 1, 0, local, None


def barrier(dist):
    if dist is not None:
        if torch.cuda.is_available():
            dist.barrier(device_ids=[torch.cuda.current_device()])
        else:
            dist.barrier()


def max_over_ranks(dist, v):
    if dist is None:
        return v
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(dist, v):
    if dist is None:
        return v
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def base_record(args, n_gpus, workload_desc, layer):
    return {
        "metric": METRIC,
        "unit": "tokens/s",
        "n_gpus": n_gpus,
        "steps": args.steps,
        "warmup": args.warmup,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": {"bf16": "bf16", "mxfp4": "mxfp4-weights/bf16-activations",
                  "fp8": "e4m3-weights/e4m3-activations",
                  "mxfp4_mxfp8": "mxfp4-weights/mxfp8-activations"}[layer.wfmt],
        "data": "synthetic: seeded gpt-oss-shaped layer, random-init weights (no checkpoint)",
        "config": {"workload": workload_desc, "T": layer.T, "H": layer.H, "I": layer.I,
                   "E": layer.E, "top_k": layer.top_k, "weights": layer.wfmt,
                   "output": "fp32",
                   "l2": "inputs larger than L2 (touched expert weights streamed each step)",
                   "parallelism": f"replicas x{n_gpus} (no collective)"},
    }


def run_reference(args, layer, desc):
    """CPU oracle arm: each step runs the oracle on one token of the batch."""
    import oracle
    oracle.build()
    T = layer.T
    for i in range(args.warmup):
        oracle.forward(layer, tokens=[i % T])
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle.forward(layer, tokens=[i % T])
    dt = time.perf_counter() - t0
    value = args.steps / dt
    rec = base_record(args, args.gpus, desc, layer)
    rec.update({
        "impl": "reference",
        "value": value,
        "ms_per_step": dt * 1e3 / args.steps,
        "dtype": "f32",
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.max_threads(),
                         "kind": "oracle",
                         "sample": f"1 token of the T={T} batch per step, cycling through the "
                                   f"batch ({args.steps} steps)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    })
    print(json.dumps(rec), flush=True)


ALG_BYTES = {"bf16": (GU_BYTES, D_BYTES), "fp8": (GU_BYTES_FP8, D_BYTES_FP8),
             "mxfp4": (GU_BYTES_MXFP4, D_BYTES_MXFP4),
             "mxfp4_mxfp8": (GU_BYTES_MXFP4, D_BYTES_MXFP4)}


def measure(moe, layer, args, dist, workload):
    """Times K steps of one layer (inputs resident in HBM), then K more with
    a CUDA event around every kernel; returns the measurement and the
    routing and output of the last step."""
    T, H, I, E, k = layer.T, layer.H, layer.I, layer.E, layer.top_k
    dev = {}
    for name in ("x", "wr", "br", "w_gu", "b_gu", "w_d", "b_d", "s_gu", "s_d"):
        t = getattr(layer, name)
        dev[name] = None if t is None else t.to("cuda", non_blocking=True)
    torch.cuda.synchronize()
    shape = moe.layer_shape(layer)
    ws = moe.alloc_workspace(shape)
    out = torch.empty((T, H), dtype=torch.float32, device="cuda")
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def step(x=None):
        moe.moe_forward(shape, dev["x"] if x is None else x, dev["wr"], dev["br"],
                        dev["w_gu"], dev["b_gu"], dev["w_d"], dev["b_d"], out,
                        s_gu=dev["s_gu"], s_d=dev["s_d"], topk_ids_out=ids,
                        workspace=ws, stream=stream)

    clocks = ClockSampler(device_id_for_smi())
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    status = moe.moe_get_device_status(ws)
    if status:
        raise SystemExit(f"device status word {status:#x} after warm-up ({workload})")
    U = int(torch.unique(ids).numel())

    # Timed region 1: K steps, bracketed by CUDA events only (this gives
    # `value`).  Timed region 2: K more steps with a CUDA event around every
    # kernel (per-kernel durations for the roofline).  Events between kernels
    # stop dependent launches from overlapping, so region 2 runs slightly
    # slower; both step times are reported.
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize()
    wall0 = time.time()
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    elapsed_ms = ev0.elapsed_time(ev1)

    moe.moe_profile_enable(min(args.steps, 8192))
    ev2 = torch.cuda.Event(enable_timing=True)
    ev3 = torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize()
    ev2.record(stream)
    for _ in range(args.steps):
        step()
    ev3.record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    wall2 = time.time()
    profiled_ms = ev2.elapsed_time(ev3)
    kernels = moe.moe_profile_read()
    moe.moe_profile_enable(0)
    clocks.stop()
    status = moe.moe_get_device_status(ws)
    if status:
        raise SystemExit(f"device status word {status:#x} after the timed region ({workload})")

    max_ms = max_over_ranks(dist, elapsed_ms)
    tokens_all = sum_over_ranks(dist, float(T * args.steps))

    # Roofline of the dominant kernel (the gate_up GEMM: 2/3 of the bytes).
    bw, tf_burst, tf_sust, peak_kind = peaks()
    kmap = dict(kernels)
    R = T * k
    gu_b, d_b = (f(H, I) for f in ALG_BYTES[layer.wfmt])
    # activation and h bytes per element: E4M3 codes for FP8 W8A8 and MXFP8
    # (plus one scale byte per 32 for MXFP8 activations), else bf16
    ab = 1 if layer.wfmt in ("fp8", "mxfp4_mxfp8") else 2
    gu_alg = U * gu_b + R * H * ab + R * I * ab
    if layer.wfmt == "mxfp4_mxfp8":
        gu_alg += R * H // 32
    tkind = "bf16"
    if layer.wfmt in ("fp8", "mxfp4_mxfp8"):
        # an E4M3 contraction's peak: the measured bf16 rate x the nominal
        # dense fp8 / bf16 ratio (4.5 / 2.25 PFLOP/s)
        tf_burst, tf_sust = 2.0 * tf_burst, 2.0 * tf_sust
        peak_kind += ", x2 nominal fp8/bf16 ratio"
        tkind = "e4m3"
    gu_ms = kmap.get("gate_up_glu")
    flops_tok = 2 * (2 * I) * H + 2 * H * I
    gu_flops = R * 2 * (2 * I) * H
    wl_key = f"{workload}_T{T}"
    # bound: the kernel's algorithmic flops per byte against the ridge of
    # its own tensor peak (bytes per weight differ between formats)
    ridge = tf_burst * 1e12 / (bw * 1e9)
    intensity = gu_flops / max(gu_alg, 1)
    if intensity < ridge:
        roof = {"bound": "hbm", "achieved": gu_alg / (gu_ms * 1e-3) / 1e9, "peak": bw,
                "unit": "GB/s"}
        peak_kind += ", HBM copy"
    else:
        # the step lasts about a millisecond, far from the seconds-long loop
        # the sustained GEMM rate was measured on: the burst rate is the
        # denominator, the sustained one a secondary figure
        roof = {"bound": "tensor", "achieved": gu_flops / (gu_ms * 1e-3) / 1e12,
                "peak": tf_burst, "unit": "TFLOP/s"}
        roof["frac_of_sustained"] = roof["achieved"] / tf_sust
        peak_kind += f", burst {tkind} GEMM rate"
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = recorded_traffic("gate_up_glu", wl_key)
    roof["kernel"] = "gate_up_glu (tcgen05 grouped GEMM + fused bias/GLU)"
    roof["algorithmic_bytes_per_launch"] = gu_alg
    roof["algorithmic_flops_per_launch"] = gu_flops
    roof["peak_source"] = f"MEASURED_PEAKS.json ({peak_kind})"

    layer_bytes = U * (gu_b + d_b) + E * H * 2 + E * 2 + T * H * (2 + 4)
    layer_flops = T * (k * flops_tok + 2 * H * E)
    step_s = max_ms / 1e3 / args.steps
    m = {
        "value": tokens_all / (max_ms / 1e3),
        "ms_per_step": max_ms / args.steps,
        "roofline": roof,
        "layer": {"experts_touched": U, "bytes_per_step": layer_bytes,
                  "flops_per_step": layer_flops,
                  "hbm_gbs": layer_bytes / step_s / 1e9,
                  "hbm_frac": layer_bytes / step_s / 1e9 / bw,
                  "tflops": layer_flops / step_s / 1e12,
                  "tensor_frac": layer_flops / step_s / 1e12 / tf_burst,
                  "tensor_frac_of_sustained": layer_flops / step_s / 1e12 / tf_sust},
        "kernels_ms": {n: round(v, 5) for n, v in kernels},
        "kernel_timing": {"method": "CUDA events around every kernel, second timed region "
                                    "of the same K steps",
                          "ms_per_step_with_events": profiled_ms / args.steps},
        "gpu_launches": len(kernels) * args.steps,
        "clocks": clocks.summary(wall0, wall2),
    }
    return m, dev, step, out, ids


def measure_attention(moe, T=4096, reps=30):
    """The adjacent step of a gpt-oss block, attention with sinks at prefill
    (64 query / 8 KV heads, D = 64, bf16 in, fp32 out), full and 128-key
    sliding-window layers: each launch timed alone with CUDA events on the
    launching stream, an L2 flush (a 256 MB write) between launches."""
    import synth
    _, tf_burst, _, pkind = peaks()
    a = synth.make_attention(T, T, Hq=64, Hkv=8, D=64, seed=1)
    q, k, v, s = (a[n].cuda() for n in ("q", "k", "v", "sinks"))
    out = torch.empty((T, 64, 64), dtype=torch.float32, device="cuda")
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    res = {"workload": f"gpt-oss attention with sinks, prefill T={T}, 64 query / 8 KV heads, "
                       "D=64, bf16 q/k/v, fp32 out, seed 1",
           "timing": f"CUDA events per launch, mean of {reps} after 3 warm-up launches, "
                     "L2 flushed (256 MB write) before each",
           "peak": tf_burst, "unit": "TFLOP/s",
           "peak_source": f"MEASURED_PEAKS.json ({pkind}, burst bf16 GEMM rate)"}
    for name, W in (("full", 0), ("window128", 128)):
        keys = sum(min(i + 1, W) if W else i + 1 for i in range(T))
        flops = 4 * 64 * 64 * keys
        for _ in range(3):
            moe.attention_sinks(q, k, v, s, out=out, window=W, workspace=ws)
        torch.cuda.synchronize()
        tot = 0.0
        for _ in range(reps):
            flush.fill_(1)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            moe.attention_sinks(q, k, v, s, out=out, window=W, workspace=ws)
            e1.record()
            torch.cuda.synchronize()
            tot += e0.elapsed_time(e1)
        ms = tot / reps
        if moe.moe_get_device_status(ws) != 0:
            raise RuntimeError("attention device status non-zero")
        tf = flops / (ms * 1e-3) / 1e12
        res[name] = {"ms": ms, "algorithmic_flops": flops, "achieved": tf,
                     "frac": tf / tf_burst}
    del flush
    return res


def oracle_parity(layer, out, ids, n_tokens, threads=0):
    """The oracle on the first n tokens (timed) and its agreement with the
    GPU's last step on those tokens; near ties counted over all tokens."""
    import oracle
    oracle.build()
    toks = list(range(n_tokens))
    t0 = time.perf_counter()
    o_ids, _, o_out = oracle.forward(layer, tokens=toks, threads=threads)
    dt = time.perf_counter() - t0
    logits = oracle.router_logits(layer)
    srt = torch.sort(logits.double(), dim=1, descending=True).values
    k = layer.top_k
    near = (srt[:, k - 1] - srt[:, k]) < 1e-5 if k < layer.E else torch.zeros(layer.T, dtype=torch.bool)
    keep = [t for t in toks if not near[t]]
    g = out.cpu()[keep].double()
    o = o_out[[toks.index(t) for t in keep]].double()
    err = (g - o).abs().max().item() if keep else 0.0
    ref = o.abs().max().item() if keep else 0.0
    ids_equal = bool(torch.equal(ids.cpu()[keep], o_ids[[toks.index(t) for t in keep]]))
    return dt, {"tokens_compared": len(keep), "near_ties": int(near.sum()),
                "ids_bit_exact": ids_equal, "max_abs_err": err,
                "max_abs_oracle": ref, "rel_err": err / ref if ref else 0.0}


def cpu_oracle_rate(layer, budget_s, max_tokens=None, threads=0):
    """Oracle tokens/s on a bounded sample of the batch (first n tokens)."""
    import oracle
    oracle.build()
    n = 1
    max_tokens = max_tokens or layer.T
    while True:
        t0 = time.perf_counter()
        oracle.forward(layer, tokens=list(range(n)), threads=threads)
        dt = time.perf_counter() - t0
        if dt >= budget_s / 3 or n >= max_tokens:
            return n / dt, n, dt, (threads or oracle.max_threads())
        n = min(max_tokens, n * 2)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="20b_decode")
    ap.add_argument("--T", type=int, default=64)
    ap.add_argument("--prefill-workload", default="20b_prefill_skewed",
                    help="second workload timed in the same run ('none' to skip)")
    ap.add_argument("--prefill-T", type=int, default=4096)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-attention", action="store_true",
                    help="skip the attention-with-sinks figures")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle work for cpu_baseline")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")

    import synth
    world, rank, local, dist = dist_setup()
    desc = DESCRIPTIONS.get(args.workload, args.workload).format(T=args.T)

    if args.impl == "reference":
        if rank == 0:
            layer = synth.make_workload(args.workload, args.T)
            run_reference(args, layer, desc)
        if dist is not None:
            dist.destroy_process_group()
        return

    import gpt_oss_moe_gb300 as moe
    from gpt_oss_moe_gb300 import _build
    _build.build()
    moe.lib()

    layer = synth.make_workload(args.workload, args.T, pin=True)
    m, dev, step, out, ids = measure(moe, layer, args, dist, args.workload)
    T, H = layer.T, layer.H

    rec = base_record(args, world, desc, layer)
    rec.update(m)

    # End to end through the public API with host buffers.
    if not args.no_e2e:
        x_host = layer.x if layer.x.is_pinned() else layer.x.pin_memory()
        out_host = torch.empty((T, H), dtype=torch.float32, pin_memory=True)
        x_dev = torch.empty_like(dev["x"])
        n_e2e = max(3, min(args.steps, 500))
        for _ in range(3):
            x_dev.copy_(x_host, non_blocking=True)
            step(x_dev)
            out_host.copy_(out, non_blocking=True)
        torch.cuda.synchronize()
        barrier(dist)
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            x_dev.copy_(x_host, non_blocking=True)
            step(x_dev)
            out_host.copy_(out, non_blocking=True)
        torch.cuda.synchronize()
        dt = max_over_ranks(dist, time.perf_counter() - t0)
        rec["e2e"] = {"value": sum_over_ranks(dist, float(T * n_e2e)) / dt,
                      "unit": "tokens/s", "h2d_bytes_per_step": T * H * 2,
                      "d2h_bytes_per_step": T * H * 4, "steps": n_e2e,
                      "timing": "host wall clock, synchronised on both sides"}
    # the last step's routing and output, for the parity figures below
    step()
    torch.cuda.synchronize()
    out_last, ids_last = out.clone(), ids.clone()
    del dev

    # The prefill half of the metric: the same measurement on the prefill
    # workload, in the same process.
    if args.prefill_workload != "none":
        pl = synth.make_workload(args.prefill_workload, args.prefill_T, pin=True)
        pm, pdev, _, pout, pids = measure(moe, pl, args, dist, args.prefill_workload)
        pm["workload"] = DESCRIPTIONS.get(args.prefill_workload,
                                          args.prefill_workload).format(T=pl.T)
        pm["T"] = pl.T
        rec["prefill"] = pm
        rec["gpu_launches"] += pm["gpu_launches"]
        prefill_out, prefill_ids = pout.cpu(), pids.cpu()
        del pdev

    # The attention half of a gpt-oss block at prefill (outside the layer's
    # timed region and its launch count).
    if not args.no_attention:
        rec["attention"] = measure_attention(moe)

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, n, dt, cores = cpu_oracle_rate(layer, args.cpu_budget)
        # one thread on a small sample (a few seconds at most)
        rate1, n1, dt1, _ = cpu_oracle_rate(layer, min(3.0, args.cpu_budget / 4),
                                            max_tokens=8, threads=1)
        rec["cpu_baseline"] = {"value": rate, "unit": "tokens/s", "cores": cores,
                               "nproc": os.cpu_count(), "kind": "oracle",
                               "sample": f"first {n} of the {T} tokens, one oracle call "
                                         f"({dt:.1f} s)",
                               "one_thread": {"value": rate1, "unit": "tokens/s",
                                              "sample": f"first {n1} tokens ({dt1:.1f} s)"}}
        # parity of the timed runs: the headline batch in full, the prefill
        # batch on its first 64 tokens (near ties counted over all tokens)
        _, rec["parity"] = oracle_parity(layer, out_last, ids_last, T)
        if "prefill" in rec:
            _, rec["prefill"]["parity"] = oracle_parity(pl, prefill_out, prefill_ids,
                                                        min(64, pl.T))
    if rank == 0:
        print(json.dumps(rec), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
