#!/usr/bin/env python
"""Benchmark of the MXFP4 routed-MoE layer on GB300.

Headline (one JSON line on rank 0): MoE-layer tokens/s of the gpt-oss-20b
shaped decode step (E=32 experts, top-4, D=F=2880, MXFP4 weights, T=1), the
weight GB/s it streams, the dominant kernel's roofline fraction, the same
metric end to end through the public API with host buffers, and the CPU
oracle as a baseline. The prefill step (T=512) is measured in the same run
and reported under "prefill_t512" (bf16 grouped GEMM) and "prefill_t512_mx"
(block-scaled MXFP4 grouped GEMM).

Timing: CUDA events on the launching stream around exactly --steps steps,
captured in one CUDA graph, after --warmup eager steps; every step uses the
next of several distinct layer weight sets (more than L2 holds), so weights
always come from HBM. Under torchrun each rank runs an independent replica on
its own GPU (no collective on the data path); the time is the max over ranks.

`--impl reference` times the CPU oracle instead (the reference arm).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/s at T=1 and T=512; MXFP4 weight GB/s vs HBM peak"
E, K_TOP, D, F = 32, 4, 2880, 2880
ROW_BYTES = D // 2 + D // 32          # one MXFP4 row of 2880: 1440 nibble bytes + 90 scale bytes
MAT_BYTES = F * ROW_BYTES              # one 2880x2880 MXFP4 matrix
EXPERT_BYTES = 3 * MAT_BYTES           # gate + up + down
WORKLOAD_DECODE = "gpt-oss-20b-shaped MoE layer, decode T=1 (E=32, top-4, dim=nfe=2880, MXFP4 weights)"
WORKLOAD_PREFILL = "gpt-oss-20b-shaped MoE layer, prefill T=512 (E=32, top-4, dim=nfe=2880, MXFP4 weights)"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=8, help="distinct decode layer weight sets rotated per step")
    ap.add_argument("--prefill-steps", type=int, default=20)
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--skip-decode", action="store_true",
                    help="measure only the prefill step (profiling aid; the headline needs decode)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="minimum CPU time of the oracle sample (whole decode tokens)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# process group (replicas only: used for the barrier and the max over ranks)
# ---------------------------------------------------------------------------
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch
            import torch.distributed as dist

            backend = "nccl" if torch.cuda.is_available() else "gloo"
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            if self.pg.get_backend() == "nccl":
                import torch
                self.pg.barrier(device_ids=[torch.cuda.current_device()])
            else:
                self.pg.barrier()

    def max(self, v: float) -> float:
        if not self.pg:
            return v
        import torch

        dev = "cuda" if self.pg.get_backend() == "nccl" else "cpu"
        t = torch.tensor([float(v)], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, v: float) -> float:
        if not self.pg:
            return v
        import torch

        dev = "cuda" if self.pg.get_backend() == "nccl" else "cpu"
        t = torch.tensor([float(v)], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def whole_job_rate(units_local: float, seconds_local: float, dist: Dist):
    """Units processed by all ranks divided by the slowest rank's time."""
    units = dist.sum(units_local)
    secs = dist.max(seconds_local)
    return units / secs, secs


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                    rows.append(parts)
        except OSError:
            pass
        finally:
            try:
                os.unlink(self.path)
            except OSError:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]), "reasons": sorted(reasons),
                "samples": len(rows), "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit())
                if any(r[3].replace(".", "").isdigit() for r in rows) else None}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, 1700.0, "fallback"


def decode_config(global_batch: int, parallelism: str, l2: str, timing: str) -> dict:
    """The decode workload's config object, shared by both arms (same keys)."""
    return {"workload": WORKLOAD_DECODE, "T": 1, "E": E, "k": K_TOP, "dim": D, "nfe": F,
            "global_batch": global_batch, "parallelism": parallelism, "l2": l2, "timing": timing}


def ncu_traffic(kernel_key: str):
    """Per-launch DRAM bytes from the committed ncu summary, if the kernel source is unchanged since."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel_key)
    except (OSError, ValueError):
        return None
    if not rec:
        return None
    src = os.path.join(ROOT, "mxfp4_mixture_experts_bucket_gb300", "csrc", rec["source"])
    try:
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    return rec["bytes_per_launch"] if digest == rec["source_sha256_16"] else None


# ---------------------------------------------------------------------------
# CPU oracle baseline (bounded sample)
# ---------------------------------------------------------------------------
def host_cores():
    """Cores this process may run on (affinity / cgroup aware where the OS says), and the machine's count."""
    try:
        usable = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        usable = os.cpu_count() or 1
    return usable, os.cpu_count()


def cpu_oracle_rate(min_seconds: float = 10.0, max_tokens: int = 64):
    """Decode tokens through the float64 oracle until at least min_seconds of CPU work."""
    from oracle import moe_oracle as O
    from synthetic import make_layer, make_tokens, spec_for

    spec = spec_for(1)
    L = make_layer(spec, with_tokens=False)
    x = make_tokens(spec, T=max_tokens, seed=12345)
    t0 = time.perf_counter()
    n = 0
    while n < max_tokens and (n == 0 or time.perf_counter() - t0 < min_seconds):
        O.moe_layer(L, x[n:n + 1], spec.k)  # a fresh expert cache per token: each dequantises its experts
        n += 1
    dt = time.perf_counter() - t0
    return n / dt, dt, n


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def run_ours(args, dist: Dist):
    import torch

    import __graft_entry__ as ge

    ge.build()
    import mxfp4_mixture_experts_bucket_gb300 as moe
    from synthetic import make_layer_torch, spec_for

    torch.cuda.set_device(dist.local_rank)
    dev = torch.device("cuda", dist.local_rank)
    hbm_peak, bf16_peak, bf16_sus, peak_src = load_peaks()
    if args.skip_decode:
        stream = torch.cuda.Stream(device=dev)
        return {"prefill_t512": run_prefill(args, dist, moe, dev, stream, hbm_peak, bf16_peak, peak_src),
                "prefill_t512_mx": run_prefill(args, dist, moe, dev, stream, hbm_peak, bf16_peak, peak_src,
                                               rail=moe.MOE_RAIL_GROUPED_MX)}
    K, W, NL = args.steps, args.warmup, args.layers
    spec = spec_for(1)

    # ---- decode: NL distinct layers resident, prepacked for the block-scaled decode rail ----
    layers = [moe.MoeLayer(make_layer_torch(spec, li + 17 * dist.rank, dev), k=K_TOP, device=dev, packed=True)
              for li in range(NL)]
    g = torch.Generator(device=dev)
    g.manual_seed(4242 + dist.rank)
    xs = torch.randn((K + W, D), generator=g, device=dev)
    ys = torch.empty((K + W, D), device=dev)
    ids = torch.empty((K + W, K_TOP), dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    decode_rail = moe.MOE_RAIL_AUTO  # prepacked layer, T = 1: MOE_RAIL_DECODE_MX
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(W):  # eager warm-up steps
            layers[i % NL](xs[i:i + 1], rail=decode_rail, out=ys[i:i + 1], ids_out=ids[i:i + 1])
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    n0 = moe.moe_kernel_launches()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(K):
            j = W + i
            layers[j % NL](xs[j:j + 1], rail=decode_rail, out=ys[j:j + 1], ids_out=ids[j:j + 1])
    launches_per_step = (moe.moe_kernel_launches() - n0) / K
    with torch.cuda.stream(stream):
        graph.replay()  # first replay uploads the graph; untimed
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dist.local_rank) as clk:
        dist.barrier()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):  # replay on the stream the events are recorded on
            ev0.record(stream)
            graph.replay()
            ev1.record(stream)
        torch.cuda.synchronize()
        dist.barrier()
    secs = ev0.elapsed_time(ev1) / 1e3
    clocks = clk.summary()
    rate, secs_max = whole_job_rate(K, secs, dist)
    rc, st = moe.moe_get_status(stream)
    assert rc == 0 and st == 0, f"device status {st}"
    id_np = ids[W:].cpu().numpy()
    touched = np.mean([len(set(r.tolist())) for r in id_np])  # distinct experts per token (= k)
    step_bytes = touched * EXPERT_BYTES + K_TOP * (2 * F + D) * 4 + E * D * 4 + 2 * D * 4
    weight_bytes_step = touched * EXPERT_BYTES

    # ---- dominant kernel alone: the gate/up stage (decode_mx_kernel<0>), cold weights ----
    # Each launch runs on another layer's weights with its own workspace, prepared
    # by that token's prologue stage before the graph; the launches follow one
    # another as programmatic dependents, as inside the layer.
    Kk = min(K, 120)
    stage_ws = []
    for i in range(Kk):
        lay = layers[i % NL]
        wsb = torch.empty(lay.workspace(1, moe.MOE_RAIL_DECODE_MX).numel(), dtype=torch.uint8, device=dev)
        moe.check(moe.moe_ffn_layer_packed_stage(lay.packed_struct, xs[i:i + 1], 1, wsb, wsb.numel(),
                                                 moe.MOE_STAGE_PROLOGUE, stream=stream), "prologue")
        stage_ws.append((lay, wsb))
    torch.cuda.synchronize()
    kgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(kgraph, stream=stream):
        for lay, wsb in stage_ws:
            moe.check(moe.moe_ffn_layer_packed_stage(lay.packed_struct, None, 1, wsb, wsb.numel(),
                                                     moe.MOE_STAGE_GATEUP, stream=stream), "gateup")
    with torch.cuda.stream(stream):
        kgraph.replay()
    torch.cuda.synchronize()
    k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        k0.record(stream)
        kgraph.replay()
        k1.record(stream)
    torch.cuda.synchronize()
    kern_s = k0.elapsed_time(k1) / 1e3 / Kk
    gateup_bytes = K_TOP * 2 * MAT_BYTES + K_TOP * 2 * F * 4 + D * 4 + K_TOP * F * 4
    achieved = gateup_bytes / kern_s / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(achieved / hbm_peak, 4), "traffic": ncu_traffic("decode_mx_kernel<0>"),
                "kernel": "decode_mx_kernel<0>", "algorithmic_bytes_per_launch": gateup_bytes,
                "launch_us": round(kern_s * 1e6, 3), "peak_source": f"{peak_src} hbm_gbs (burst copy)"}
    del stage_ws

    # ---- end to end through the public API, host buffers ----
    # A serving step: MoeLayer.forward_host (one C call: the kernels read the
    # pinned x and write y into pinned host memory), then the host waits for y,
    # since the next token depends on it. Wall clock over K steps.
    x_host = torch.randn((K, D), generator=torch.Generator().manual_seed(99)).pin_memory()
    y_host = torch.empty((K, D)).pin_memory()
    with torch.cuda.stream(stream):
        for i in range(3):
            layers[i % NL].forward_host(x_host[i:i + 1], y_host[i:i + 1], stream=stream)
    torch.cuda.synchronize()
    dist.barrier()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(K):
            layers[i % NL].forward_host(x_host[i:i + 1], y_host[i:i + 1], stream=stream)
            stream.synchronize()
    e2e_secs = time.perf_counter() - t0
    dist.barrier()
    e2e_rate, _ = whole_job_rate(K, e2e_secs, dist)
    # the same calls back to back without the per-step wait (launches overlap)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(K):
            layers[i % NL].forward_host(x_host[i:i + 1], y_host[i:i + 1], stream=stream)
        e1.record(stream)
    torch.cuda.synchronize()
    pipe_rate, _ = whole_job_rate(K, e0.elapsed_time(e1) / 1e3, dist)
    rc, st = moe.moe_get_status(stream)
    assert rc == 0 and st == 0, f"device status {st}"

    # ---- the CUDA-core GEMV rail on the same layers (canonical planes), for comparison ----
    gemv_graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for i in range(3):
            layers[i % NL](xs[i:i + 1], rail=moe.MOE_RAIL_GEMV, out=ys[i:i + 1])
    torch.cuda.synchronize()
    with torch.cuda.graph(gemv_graph, stream=stream):
        for i in range(K):
            j = W + i
            layers[j % NL](xs[j:j + 1], rail=moe.MOE_RAIL_GEMV, out=ys[j:j + 1])
    with torch.cuda.stream(stream):
        gemv_graph.replay()
    torch.cuda.synchronize()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g0.record(stream)
        gemv_graph.replay()
        g1.record(stream)
    torch.cuda.synchronize()
    gemv_rate, gemv_secs = whole_job_rate(K, g0.elapsed_time(g1) / 1e3, dist)
    del gemv_graph

    result = {
        "metric": METRIC, "value": round(rate, 1), "unit": "tokens/s", "n_gpus": dist.world, "steps": K,
        "warmup": W, "ms_per_step": round(secs_max / K * 1e3, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32 accumulate; MXFP4 weights x MXFP4 activations (8 E2M1 terms per value, ~1e-7 of the block max)",
        "data": "synthetic",
        "config": decode_config(dist.world, f"replicas x{dist.world}",
                                f"inputs larger than L2: {NL} distinct layer weight sets "
                                f"({NL * E * EXPERT_BYTES / 1e9:.1f} GB) rotated every step",
                                "one CUDA graph of the timed steps, CUDA events on its stream"),
        "rail": "decode_mx (block-scaled tensor cores, prepacked weights)",
        "weight_gbs": round(weight_bytes_step * K / secs_max * dist.world / 1e9, 1),
        "layer_roofline_frac": round((step_bytes / (hbm_peak * 1e9)) / (secs_max / K), 4),
        "roofline": roofline,
        "e2e": {"value": round(e2e_rate, 1), "unit": "tokens/s", "h2d_bytes_per_step": D * 4, "d2h_bytes_per_step": D * 4,
                "path": "MoeLayer.forward_host -> moe_ffn_layer_packed_hostio, then the host waits for y every step "
                        "(wall clock); x and y move through the pinned mapping, no copy-engine transfers"},
        "e2e_pipelined": {"value": round(pipe_rate, 1), "unit": "tokens/s",
                          "path": "the same calls back to back without the per-step wait (CUDA events)"},
        "decode_t1_cuda_core": {"tokens_per_s": round(gemv_rate, 1), "ms_per_step": round(gemv_secs / K * 1e3, 5),
                                "rail": "gemv (CUDA cores, canonical planes, f16 hi/lo activations, fp32 sums)"},
        "clocks": clocks,
        "gpu_launches": int(round(launches_per_step * K)),
        "kernels_per_step": launches_per_step,
    }
    del layers
    torch.cuda.empty_cache()

    if not args.no_prefill:
        result["prefill_t512"] = run_prefill(args, dist, moe, dev, stream, hbm_peak, bf16_peak, peak_src)
        result["prefill_t512_mx"] = run_prefill(args, dist, moe, dev, stream, hbm_peak, bf16_peak, peak_src,
                                                rail=moe.MOE_RAIL_GROUPED_MX)
    return result


def run_prefill(args, dist, moe, dev, stream, hbm_peak, bf16_peak, peak_src, rail=None):
    import torch
    from synthetic import make_layer_torch, spec_for

    spec = spec_for(2)
    T, K = 512, args.prefill_steps
    if rail is None:
        rail = moe.MOE_RAIL_GROUPED_MM
    NL = 2
    layers = [moe.MoeLayer(make_layer_torch(spec, li + 31 * dist.rank, dev), k=K_TOP, device=dev) for li in range(NL)]
    g = torch.Generator(device=dev)
    g.manual_seed(777 + dist.rank)
    xs = [torch.randn((T, D), generator=g, device=dev) for _ in range(NL)]
    ys = [torch.empty((T, D), device=dev) for _ in range(NL)]
    with torch.cuda.stream(stream):
        for i in range(3):
            layers[i % NL](xs[i % NL], rail=rail, out=ys[i % NL])
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    n0 = moe.moe_kernel_launches()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(K):
            layers[i % NL](xs[i % NL], rail=rail, out=ys[i % NL])
    per_step = (moe.moe_kernel_launches() - n0) / K
    with torch.cuda.stream(stream):
        graph.replay()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    with ClockSampler(dist.local_rank) as clk:
        with torch.cuda.stream(stream):
            ev0.record(stream)
            graph.replay()
            ev1.record(stream)
        torch.cuda.synchronize()
    dist.barrier()
    secs = ev0.elapsed_time(ev1) / 1e3
    rate, secs_max = whole_job_rate(K * T, secs, dist)
    rc, st = moe.moe_get_status(stream)
    assert rc == 0 and st == 0, f"device status {st}"
    ms = secs_max / K * 1e3
    weight_bytes = E * EXPERT_BYTES
    alg_bytes = weight_bytes + 3 * E * F * 4 + E * D * 4 + 2 * T * D * 4
    flops = T * K_TOP * 3 * 2 * D * F
    t_roof = max(alg_bytes / (hbm_peak * 1e9), flops / (bf16_peak * 1e12))
    return {"tokens_per_s": round(rate, 1), "ms_per_step": round(ms, 4), "steps": K, "workload": WORKLOAD_PREFILL,
            "weight_gbs": round(weight_bytes / (ms / 1e3) / 1e9, 1),
            "dtype": ("bf16 MMA, fp32 accumulate" if rail == moe.MOE_RAIL_GROUPED_MM else
                      "MXFP4 x E4M3-term block-scaled MMA (x: 3 terms, h: 2), fp32 accumulate"),
            "rail": "grouped_mm" if rail == moe.MOE_RAIL_GROUPED_MM else "grouped_mx",
            "roofline_frac": round(t_roof / (ms / 1e3), 4),
            "roofline_bound": "hbm" if alg_bytes / (hbm_peak * 1e9) >= flops / (bf16_peak * 1e12) else "tensor",
            "algorithmic_bytes": alg_bytes, "algorithmic_flops": flops, "kernels_per_step": per_step,
            "peak_source": peak_src, "clocks": clk.summary()}


def main():
    args = parse_args()
    dist = Dist()
    if args.impl == "reference":
        if dist.rank == 0:
            rate, dt, n = cpu_oracle_rate(args.cpu_seconds)
            cores, machine_cores = host_cores()
            print(json.dumps({
                "impl": "reference", "metric": METRIC, "value": round(rate, 4), "unit": "tokens/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(dt / n * 1e3, 2), "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": decode_config(1, "float64 oracle on the host cores (rank 0)",
                                        "not applicable: host memory, every token dequantises its 4 experts",
                                        "wall clock over the sampled tokens"),
                "cpu_baseline": {"value": round(rate, 4), "unit": "tokens/s", "cores": cores,
                                 "machine_cores": machine_cores, "kind": "oracle",
                                 "sample": f"{n} decode tokens through the float64 numpy oracle "
                                           "(each dequantises its 4 experts)"},
                "e2e": {"value": round(rate, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            }), flush=True)
        dist.close()
        return
    res = run_ours(args, dist)
    if dist.rank == 0:
        if not args.no_cpu_baseline:
            rate, dt, n = cpu_oracle_rate(args.cpu_seconds)
            cores, machine_cores = host_cores()
            res["cpu_baseline"] = {"value": round(rate, 4), "unit": "tokens/s", "cores": cores,
                                   "machine_cores": machine_cores,
                                   "kind": "oracle",
                                   "sample": f"{n} decode tokens through the float64 numpy oracle "
                                             f"({dt:.1f} s; BLAS may use every core, elementwise work one)"}
        print(json.dumps(res), flush=True)
    dist.close()


if __name__ == "__main__":
    main()
