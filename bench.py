"""Benchmark of the routed-MoE FFN layer on GB300 (one JSON line on stdout).

    python bench.py [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-cpu-baseline] [--no-extra-workloads]

A step is one pass of the whole layer (router + top-k, permutation, gate/up
GEMM with SwiGLU, down GEMM, unpermutation with the shared expert) over one
batch of T tokens of a seeded synthetic workload; the default is the
decode-shaped layer (T=128, D=4096, 512 experts of intermediate 1024, top-10,
one shared expert, bf16).  A timed step is one moe_forward call on
device-resident x and out; a second pass through the stage entry points,
with events between stages, gives the per-stage times and the dominant
kernel's roofline.  Expert weights (12.9 GB) dwarf the 129 MB L2, so no
flush is needed between steps.  The default run then times the batched
decode, prefill bf16 and FP8 prefill workloads the same way and reports
them under "workloads".

Our arm runs on one GPU: the layer shards nothing, and a launch with
WORLD_SIZE > 1 is refused before the library is loaded.

--impl reference times the fp64 CPU oracle on the host cores instead (a
bounded sample of the workload per step); it is the baseline the pages'
method is checked against, not a target.  Under torchrun (gloo) rank 0
alone runs it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_moe_expert_02_gb300 import MoELayer, synth  # noqa: E402
from sparse_moe_expert_02_gb300 import _lib as L  # noqa: E402

STAGES = ("route", "permute", "gemm_gateup", "gemm_down", "unpermute")
KERNEL_FILES = {"gemm_gateup": "gemm_tc.cu", "gemm_down": "gemm_tc.cu"}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""
    Q = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = f"/tmp/moe_clocks_{os.getpid()}.csv"
        self.gpu = gpu_index

    def mark(self, name):
        setattr(self, name, time.time())

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        import datetime
        rows, inside = [], []
        t0, t1 = getattr(self, "t_begin", 0.0), getattr(self, "t_end", 1e30)
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                r = (float(f[1]), float(f[2]), f[5], f[6], f[7], f[8])
            except ValueError:
                continue
            rows.append(r)
            if t0 - 0.25 <= ts <= t1 + 0.25:
                inside.append(r)
        rows = inside or rows[-3:]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in rows for i in range(4) if r[2 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def out_dtype(shape) -> str:
    """Layer output: fp32 for the fp32 layer, bf16 (the activations' type) for
    the bf16 and FP8 layers."""
    return "f32" if shape.dtype == "f32" else "bf16"


def algorithmic(shape, counts: np.ndarray):
    """Bytes and flops the method itself must move and compute (no padding,
    no intermediate round trips): touched routed experts + shared expert +
    router weight, x in, out, and the routing blob."""
    D, E, I, k, T = shape.D, shape.E, shape.I, shape.top_k, shape.T
    bw = {"f32": 4, "bf16": 2, "fp8": 1}[shape.dtype]
    bx = 4 if shape.dtype == "f32" else 2
    bo = 4 if out_dtype(shape) == "f32" else 2
    touched = int((counts[:E] > 0).sum())
    scale_bytes = (3 * (I // 128) * (D // 128) * 4) if shape.dtype == "fp8" else 0
    per_expert = 3 * D * I * bw + scale_bytes
    layer_bytes = (touched + 1) * per_expert + E * D * bx + T * D * bx + T * D * bo + 8 * T * k
    flops = T * (2 * D * E + (k + 1) * 6 * D * I)
    gu_bytes = (touched + 1) * (2 * I * D * bw + 2 * scale_bytes // 3) + (T * k + T) * D * bw + (T * k + T) * I * bw
    dn_bytes = (touched + 1) * (D * I * bw + scale_bytes // 3) + (T * k + T) * I * bw + (T * k + T) * D * 2
    return {"touched_experts": touched, "layer_bytes": layer_bytes, "flops": flops,
            "gemm_gateup_bytes": gu_bytes, "gemm_down_bytes": dn_bytes,
            "gemm_gateup_flops": (T * k + T) * 4 * D * I, "gemm_down_flops": (T * k + T) * 2 * D * I,
            "per_expert_bytes": per_expert}


def traffic_for(kernel: str, workload: str):
    """dram bytes of the stage (per launch; summed over its launches where a
    GEMM is split) from the committed ncu summary, if it was taken on the
    kernel sources as they stand now (else null)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        ent = d[workload][kernel]
        # a stage run as several launches (split GEMMs) lists every source
        files = ent.get("source_files") or [ent["source_file"]]
        shas = ent.get("source_shas") or [ent["source_sha"]]
        for f, want in zip(files, shas):
            src = os.path.join(ROOT, "sparse_moe_expert_02_gb300", "csrc", f)
            if hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] != want:
                return None
        return ent["dram_bytes_per_launch"]
    except Exception:
        return None


# ------------------------------------------------------------------ ours

def binding_roof(bytes_, flops, ms, shape, peaks, f32_hbm=True):
    """Roofline of a kernel or of the layer against whichever ceiling binds:
    its algorithmic bytes at the HBM copy bandwidth, or its algorithmic flops
    at the dense tensor peak of its dtype (the sustained figure: it runs
    inside a long step; FP8 = 2x bf16, the nominal dense ratio)."""
    tc_peak = (peaks["bf16_tflops_sustained"] or peaks["bf16_tflops"]) * (2.0 if shape.dtype == "fp8" else 1.0)
    t_hbm = bytes_ / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (tc_peak * 1e12)
    if (f32_hbm and shape.dtype == "f32") or t_hbm >= t_tc:
        achieved = bytes_ / (ms / 1e3) / 1e9
        return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4)}
    achieved = flops / (ms / 1e3) / 1e12
    return {"bound": "tensor", "achieved": round(achieved, 1), "peak": tc_peak, "unit": "TFLOP/s",
            "frac": round(achieved / tc_peak, 4),
            "peak_note": ("fp8 = 2 x measured bf16 sustained (nominal dense ratio)" if shape.dtype == "fp8"
                          else "measured bf16 sustained")}


def run_ours(args, shape, local, e2e=True):
    """One workload on this process's GPU: the timed moe_forward steps, the
    per-stage pass, and (e2e) the end-to-end pass through host buffers."""
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    inp = synth.make_inputs(shape, seed=args.seed, device=dev)
    layer = MoELayer.from_shape(shape, inp, device=local, flags=args.flags, out_dtype=out_dtype(shape))
    x = inp["x"]
    T = shape.T
    out = layer.new_out(T)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        layer.forward(x, out)
    layer.check()
    counts = layer.views(T)["counts"].cpu().numpy()
    alg = algorithmic(shape, counts)

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(STAGES) + 1)] for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        time.sleep(0.3)  # let nvidia-smi start sampling
        clk.mark("t_begin")
        # (1) the measured step: one moe_forward call per step (inputs resident
        # in HBM), whose shared-expert GEMMs overlap the routing on a second
        # stream
        l0 = L.moe_launch_count()
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for s in range(args.steps):
            layer.forward(x, out)
        t_end.record(stream)
        torch.cuda.synchronize(dev)
        launches = L.moe_launch_count() - l0
        # (2) the per-stage breakdown: the same layer through the stage entry
        # points, with events between the stages (stages run back to back on
        # one stream here, the shared expert inside the GEMM stages)
        for s in range(args.steps):
            e = ev[s]
            e[0].record(stream)
            layer.init_ws()
            layer.route(x)
            e[1].record(stream)
            layer.permute(x)
            e[2].record(stream)
            layer.gemm_gateup(x)
            e[3].record(stream)
            layer.gemm_down(T)
            e[4].record(stream)
            layer.unpermute(T, out)
            e[5].record(stream)
        torch.cuda.synchronize(dev)
        clk.mark("t_end")
    layer.check()
    ms = t_start.elapsed_time(t_end)
    stage_ms = {st: statistics.mean(ev[s][i].elapsed_time(ev[s][i + 1]) for s in range(args.steps))
                for i, st in enumerate(STAGES)}
    ms_per_step = ms / args.steps
    value = T * args.steps / (ms / 1e3)

    peaks = load_peaks()
    dom = max(("gemm_gateup", "gemm_down"), key=lambda s: stage_ms[s])
    roof = binding_roof(alg[dom + "_bytes"], alg[dom + "_flops"], stage_ms[dom], shape, peaks)
    roof["kernel"] = dom
    roof["traffic"] = traffic_for(dom, shape.name)
    roof["peak_source"] = peaks["source"]
    layer_roof = binding_roof(alg["layer_bytes"], alg["flops"], ms_per_step, shape, peaks)
    layer_roof.update({"alg_bytes": alg["layer_bytes"], "alg_flops": alg["flops"],
                       "tflops": round(alg["flops"] / (ms_per_step / 1e3) / 1e12, 2),
                       "gbs": round(alg["layer_bytes"] / (ms_per_step / 1e3) / 1e9, 1)})
    res = {
        "metric": "routed-MoE layer tokens/s at E=512,k=10,D=4096",
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": {"f32": "f32", "bf16": "bf16", "fp8": "e4m3"}[shape.dtype],
        "data": "synthetic (seeded; random-init weights of the layer's shape)",
        "config": {"workload": shape.name, "T": T, "D": shape.D, "E": shape.E, "I": shape.I,
                   "top_k": shape.top_k, "shared_experts": 1, "router_bias_zipf_s": shape.zipf_s,
                   "out_dtype": out_dtype(shape), "parallelism": "single GPU",
                   "l2": "inputs larger than L2 (expert weights stream from HBM every step)",
                   "touched_experts": alg["touched_experts"]},
        "roofline": roof,
        "layer_roofline": layer_roof,
        "stage_ms": {k: round(v, 4) for k, v in stage_ms.items()},
        "gpu_launches": int(launches),
        "clocks": clk.summary(),
        "impl": "ours",
        "gemm_path": "tcgen05" if "tcgen05" in L.moe_build_info() else "simt",
    }
    if e2e:
        res["e2e"] = run_e2e(args, layer, x, out, stream)
    return res, inp, layer


def run_e2e(args, layer, x, out, stream):
    """End to end through the public call, host buffers, copies inside the
    timing: x goes up by a copy from page-locked memory; the result comes back
    either written straight into mapped page-locked memory by the unpermute
    kernel or (where the host buffer is not mapped) by a copy."""
    T = x.shape[0]
    x_h = x.cpu().pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    direct_out = L.moe_pointer_kind(out_h) == "host_mapped"
    x_d = torch.empty_like(x)
    e2e_ms = []
    for i in range(args.warmup + args.steps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        x_d.copy_(x_h, non_blocking=True)
        if direct_out:
            layer.forward(x_d, out_h)
        else:
            layer.forward(x_d, out)
            out_h.copy_(out, non_blocking=True)
        b.record(stream)
        b.synchronize()
        if i >= args.warmup:
            e2e_ms.append(a.elapsed_time(b))
    layer.check()
    return {"value": round(T / (statistics.mean(e2e_ms) / 1e3), 1), "unit": "tokens/s",
            "out_path": "written by the unpermute into mapped page-locked host memory" if direct_out
            else "device buffer, then a device-to-host copy",
            "h2d_bytes_per_step": x.numel() * x.element_size(),
            "d2h_bytes_per_step": out.numel() * out.element_size()}


# The other large workloads, timed in the same process after the headline one
# (same steps and warm-up; each one's weights freed before the next).
EXTRA_BENCH = ("BATCHED_DECODE_BF16", "PREFILL_BF16", "PREFILL_FP8")
EXTRA_KEYS = ("value", "ms_per_step", "roofline", "layer_roofline", "stage_ms", "e2e", "gpu_launches", "clocks",
              "dtype", "config")


def run_extra_workloads(args, local):
    out = {}
    for name in EXTRA_BENCH:
        shape = getattr(synth, name)
        res, inp, layer = run_ours(args, shape, local)
        out[shape.name] = {k: res[k] for k in EXTRA_KEYS if k in res}
        del res, inp, layer
        torch.cuda.synchronize(local)
        torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------ oracle leg

def oracle_sample(shape, inp, n_tokens: int, seed: int = 1):
    """Time the fp64 oracle on n_tokens of the workload: its own router
    (fp64 logits, top-k) and every chosen expert plus the shared one."""
    import oracle
    g = np.random.default_rng(seed)
    rows = np.sort(g.choice(shape.T, size=min(n_tokens, shape.T), replace=False))
    x = inp["x"][torch.as_tensor(rows, device=inp["x"].device)].cpu()
    wr = inp["w_router"].cpu()
    b = inp["b_router"].cpu() if shape.has_bias else None
    t0 = time.perf_counter()
    z = oracle.logits(x, wr, b)
    idx, w = oracle.topk(z, shape.top_k)
    t_route = time.perf_counter() - t0
    used = np.unique(idx)
    groups = torch.as_tensor(np.concatenate([used, [shape.E]]), dtype=torch.long)
    remap = np.full(shape.E, -1, np.int64)
    remap[used] = np.arange(len(used))
    idx_sub = remap[idx].astype(np.int32)

    def take(n):
        t = inp[n]
        return t.index_select(0, groups.to(t.device)).cpu()

    if shape.dtype == "fp8":
        ex = oracle.Experts.quantised(take("w_gate"), take("w_up"), take("w_down"))
    else:
        ex = oracle.Experts(shape.dtype, take("w_gate"), take("w_up"), take("w_down"))
    t1 = time.perf_counter()
    oracle.moe_tokens(x, idx_sub, w, ex)
    t_exp = time.perf_counter() - t1
    return len(rows), t_route + t_exp


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def run_reference(args, shape, world, rank, local):
    """The fp64 CPU oracle, timed as it stands on the host cores."""
    if rank != 0:
        return None
    import oracle
    oracle.build()
    dev = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    inp = synth.make_inputs(shape, seed=args.seed, device=dev)
    n = args.ref_tokens
    times = []
    t_start = time.perf_counter()
    for i in range(args.warmup + args.steps):
        ntok, dt = oracle_sample(shape, inp, n, seed=100 + i)
        if i >= args.warmup:
            times.append(dt)
        # keep the whole run to a few minutes: after the first step, shrink
        # the per-step sample if the projected run would exceed ~3 min
        if i == 0 and n > 1:
            projected = (time.perf_counter() - t_start) * (args.warmup + args.steps)
            if projected > 180.0:
                n = max(1, int(n * 180.0 / projected))
    ms = sum(times) * 1e3
    value = ntok * args.steps / (ms / 1e3)
    # the oracle parallelises over tokens: it keeps at most ntok threads busy
    cores = min(ntok, int(os.environ.get("OMP_NUM_THREADS", cpu_cores())))
    sample = f"{ntok} of {shape.T} tokens per step, whole layer in fp64 (router, top-k, {shape.top_k} experts + shared)"
    return {
        "metric": "routed-MoE layer tokens/s at E=512,k=10,D=4096",
        "value": round(value, 3), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": shape.name, "T": shape.T, "D": shape.D, "E": shape.E, "I": shape.I,
                   "top_k": shape.top_k},
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=synth.DECODE_BF16.name,
                    choices=sorted(synth.WORKLOADS) + sorted(synth.EXTRA_WORKLOADS))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra-workloads", action="store_true",
                    help="time only --workload (by default the decode line also times batched decode, "
                         "prefill bf16 and FP8 prefill under its 'workloads' key)")
    ap.add_argument("--flags", type=int, default=0, help="moe_config.flags (kernel-path overrides)")
    ap.add_argument("--cpu-tokens", type=int, default=128, help="oracle sample size for cpu_baseline")
    ap.add_argument("--experts", type=int, default=0,
                    help="override E (profiling captures on a few-GB copy of the workload); not a bench line")
    ap.add_argument("--ref-tokens", type=int, default=16, help="oracle tokens per step for --impl reference")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    shape = {**synth.WORKLOADS, **synth.EXTRA_WORKLOADS}[args.workload]
    if args.experts:
        import dataclasses
        shape = dataclasses.replace(shape, E=args.experts, name=f"{shape.name}_E{args.experts}_profile")
    world, rank, local = dist_env()
    if world > 1 and args.impl == "ours":
        # The layer runs on one GPU and shards nothing; its prefill GEMMs pair
        # CTAs in 2-CTA clusters that share operand tiles through TMA
        # multicast, which is kept to single-GPU processes.  So a multi-rank
        # launch of this arm stops here, before the library is loaded.
        print(f"bench.py: --impl ours runs on one GPU only (WORLD_SIZE={world}); "
              "refused before loading libmoe", file=sys.stderr, flush=True)
        sys.exit(3)
    if world > 1:
        torch.distributed.init_process_group("gloo")
    try:
        if args.impl == "reference":
            res = run_reference(args, shape, world, rank, local)
            if res is not None:
                print(json.dumps(res), flush=True)
            return
        res, inp, layer = run_ours(args, shape, local)
        if not args.no_cpu_baseline:
            import oracle
            oracle.build()
            ntok, dt = oracle_sample(shape, inp, args.cpu_tokens)
            res["cpu_baseline"] = {"value": round(ntok / dt, 3), "unit": "tokens/s",
                                   "cores": min(ntok, int(os.environ.get("OMP_NUM_THREADS", cpu_cores()))),
                                   "kind": "oracle",
                                   "sample": f"{ntok} of {shape.T} tokens, whole layer in fp64 "
                                             f"(router, top-k, {shape.top_k} experts + shared), {dt:.1f} s"}
        if args.workload == synth.DECODE_BF16.name and not args.experts and not args.no_extra_workloads:
            del inp, layer
            torch.cuda.empty_cache()
            res["workloads"] = run_extra_workloads(args, local)
        print(json.dumps(res), flush=True)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
