#!/usr/bin/env python
"""Benchmark of the MXFP4 routed-MoE layer on GB300.

Headline (one JSON line on rank 0): MoE-layer tokens/s of the gpt-oss-20b
shaped decode step (E=32 experts, top-4, D=F=2880, MXFP4 weights, T=1), the
weight GB/s it streams, the dominant kernel's roofline fraction, the same
metric end to end through the public API with host buffers, and the CPU
oracle as a baseline. The prefill step (T=512) is measured in the same run
and reported under "prefill_t512" (the fastest rail: grouped GEMMs on
tcgen05.mma kind::mxf4 over prepacked MXFP4 weights), with the bf16 rail
("prefill_t512_bf16") and the E4M3-term block-scaled rail ("prefill_t512_mx")
beside it; likewise the skewed T=4096 layer ("skew_t4096", ...).

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
WORKLOAD_SKEW = ("skewed-routing MoE layer, T=4096 (E=32, top-4, dim=nfe=2880; +4 router bias on 2 hot experts, "
                 "about half the assignments on them)")
WORKLOAD_STACK = ("24 distinct gpt-oss-20b-shaped MoE layers back to back, RMS-renormalised between layers; "
                  "T=1 for 128 tokens and T=512")


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
    ap.add_argument("--no-stack", action="store_true", help="skip the 24-layer stack measurement")
    ap.add_argument("--no-crossover", action="store_true", help="skip the T=1..512 rail crossover")
    ap.add_argument("--stack-steps", type=int, default=128, help="T=1 tokens through the 24-layer stack")
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


def cpu_oracle_prefill_rate(cfg: int = 2, n_tokens: int = 8):
    """A bounded sample of a prefill batch through the oracle: n_tokens of the
    batch in one call (each touched expert dequantised once for the call)."""
    from oracle import moe_oracle as O
    from synthetic import make_layer, make_tokens, spec_for

    spec = spec_for(cfg)
    L = make_layer(spec, with_tokens=False)
    x = make_tokens(spec, T=n_tokens, seed=4321)
    t0 = time.perf_counter()
    O.moe_layer(L, x, spec.k)
    dt = time.perf_counter() - t0
    return n_tokens / dt, dt


def cpu_oracle_stack_rate(n_layers: int = 2, n_stack: int = 24):
    """One token through n_layers distinct layers of the stacked workload (with
    the renormalisation between them), extrapolated to the n_stack-layer stack."""
    from oracle import moe_oracle as O
    from synthetic import make_layer, make_tokens, spec_for

    spec = spec_for(3)
    Ls = [make_layer(spec, li, with_tokens=False) for li in range(n_layers)]
    x = make_tokens(spec, T=1, seed=555)
    t0 = time.perf_counter()
    for L in Ls:
        y, _, _, _ = O.moe_layer(L, x, spec.k)
        x = O.rms_renorm(y)
    dt = time.perf_counter() - t0
    return 1.0 / (dt / n_layers * n_stack), dt


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def graph_seconds(stream, body, reps: int = 1):
    """Captures body() (a sequence of library calls on `stream`) in one CUDA
    graph, replays it once untimed, then times `reps` replays with CUDA events
    recorded on the same stream. Returns (seconds per replay, graph)."""
    import torch

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        body()
    with torch.cuda.stream(stream):
        graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3 / reps, graph


def check_status(moe, stream):
    rc, st = moe.moe_get_status(stream)
    assert rc == 0 and st == 0, f"device status {st}"


def run_ours(args, dist: Dist):
    import torch

    import __graft_entry__ as ge

    ge.build()
    import mxfp4_mixture_experts_bucket_gb300 as moe
    from synthetic import make_layer_torch, spec_for

    torch.cuda.set_device(dist.local_rank)
    dev = torch.device("cuda", dist.local_rank)
    hbm_peak, bf16_peak, bf16_sus, peak_src = load_peaks()
    stream = torch.cuda.Stream(device=dev)
    if args.skip_decode:
        return {"prefill_t512": run_prefill(args, dist, moe, dev, stream, hbm_peak, bf16_peak, peak_src,
                                            rail=moe.MOE_RAIL_GROUPED_MX4),
                "prefill_t512_bf16": run_prefill(args, dist, moe, dev, stream, hbm_peak, bf16_peak, peak_src,
                                                 rail=moe.MOE_RAIL_GROUPED_MM),
                "prefill_t512_mx": run_prefill(args, dist, moe, dev, stream, hbm_peak, bf16_peak, peak_src,
                                               rail=moe.MOE_RAIL_GROUPED_MX)}
    K, W, NL = args.steps, args.warmup, args.layers
    spec = spec_for(1)

    # ---- decode: NL distinct layers resident (canonical planes and the prepacked copy) ----
    layers = [moe.MoeLayer(make_layer_torch(spec, li + 17 * dist.rank, dev), k=K_TOP, device=dev, packed=True)
              for li in range(NL)]
    g = torch.Generator(device=dev)
    g.manual_seed(4242 + dist.rank)
    xs = torch.randn((K + W, D), generator=g, device=dev)
    ys = torch.empty((K + W, D), device=dev)
    ids = torch.empty((K + W, K_TOP), dtype=torch.int32, device=dev)
    head_rail = moe.MOE_RAIL_GEMV  # the faster decode rail at T = 1 (decode_t1_tensor_core below)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(W):  # eager warm-up steps
            layers[i % NL](xs[i:i + 1], rail=head_rail, out=ys[i:i + 1], ids_out=ids[i:i + 1])
    torch.cuda.synchronize()

    def decode_steps(rail):
        def body():
            for i in range(K):
                j = W + i
                layers[j % NL](xs[j:j + 1], rail=rail, out=ys[j:j + 1], ids_out=ids[j:j + 1])
        return body

    n0 = moe.moe_kernel_launches()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        decode_steps(head_rail)()
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
    del graph
    rate, secs_max = whole_job_rate(K, secs, dist)
    check_status(moe, stream)
    id_np = ids[W:].cpu().numpy()
    touched = np.mean([len(set(r.tolist())) for r in id_np])  # distinct experts per token (= k)
    step_bytes = touched * EXPERT_BYTES + K_TOP * (2 * F + D) * 4 + E * D * 4 + 2 * D * 4
    weight_bytes_step = touched * EXPERT_BYTES
    gateup_bytes = K_TOP * 2 * MAT_BYTES + K_TOP * 2 * F * 4 + D * 4 + K_TOP * F * 4
    Kk = min(K, 120)

    # ---- dominant kernel alone: the fused gate/up + swiglu GEMV (decode_expert_kernel<0>), cold weights ----
    routes = []
    for i in range(Kk):
        lay = layers[i % NL]
        w = lay.w
        logits = torch.empty((1, E), device=dev)
        rid = torch.empty((1, K_TOP), dtype=torch.int32, device=dev)
        rw = torch.empty((1, K_TOP), device=dev)
        x1 = xs[i:i + 1]
        moe.check(moe.moe_route_topk(x1, 1, D, w["w_router"], w["b_router"], E, K_TOP, logits, rid, rw, stream),
                  "route")
        routes.append((lay, x1, rid, torch.empty((K_TOP, F), device=dev)))
    torch.cuda.synchronize()

    def gateup_body():
        for lay, x1, rid, h in routes:
            w = lay.w
            moe.check(moe.moe_expert_gateup_swiglu(w["g_qs"], w["g_sc"], w["bg"], w["u_qs"], w["u_sc"], w["bu"],
                                                   E, F, D, 1, K_TOP, x1, rid, 1.702, 7.0, h, stream), "gateup")

    kern_s = graph_seconds(stream, gateup_body)[0] / Kk
    del routes
    achieved = gateup_bytes / kern_s / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(achieved / hbm_peak, 4), "traffic": ncu_traffic("decode_expert_kernel<0>"),
                "kernel": "decode_expert_kernel<0>", "algorithmic_bytes_per_launch": gateup_bytes,
                "launch_us": round(kern_s * 1e6, 3), "peak_source": f"{peak_src} hbm_gbs (burst copy)"}

    # ---- end to end through the public API, host buffers ----
    # A serving step: MoeLayer.forward_host (one C call: x copied in from pinned
    # host memory, the layer, y copied back), then the host waits for y, since
    # the next token depends on it. Wall clock over K steps.
    x_host = torch.randn((K, D), generator=torch.Generator().manual_seed(99)).pin_memory()
    y_host = torch.empty((K, D)).pin_memory()
    with torch.cuda.stream(stream):
        for i in range(3):
            layers[i % NL].forward_host(x_host[i:i + 1], y_host[i:i + 1], rail=head_rail, stream=stream)
    torch.cuda.synchronize()
    dist.barrier()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(K):
            layers[i % NL].forward_host(x_host[i:i + 1], y_host[i:i + 1], rail=head_rail, stream=stream)
            stream.synchronize()
    e2e_secs = time.perf_counter() - t0
    dist.barrier()
    e2e_rate, _ = whole_job_rate(K, e2e_secs, dist)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(K):
            layers[i % NL].forward_host(x_host[i:i + 1], y_host[i:i + 1], rail=head_rail, stream=stream)
        e1.record(stream)
    torch.cuda.synchronize()
    pipe_rate, _ = whole_job_rate(K, e0.elapsed_time(e1) / 1e3, dist)
    check_status(moe, stream)

    # ---- the block-scaled tensor-core decode rail on the same layers (prepacked planes) ----
    mx_secs = graph_seconds(stream, decode_steps(moe.MOE_RAIL_DECODE_MX))[0]
    check_status(moe, stream)
    stage_ws = []
    for i in range(Kk):
        lay = layers[i % NL]
        wsb = torch.empty(lay.workspace(1, moe.MOE_RAIL_DECODE_MX).numel(), dtype=torch.uint8, device=dev)
        moe.check(moe.moe_ffn_layer_packed_stage(lay.packed_struct, xs[i:i + 1], 1, wsb, wsb.numel(),
                                                 moe.MOE_STAGE_PROLOGUE, stream=stream), "prologue")
        stage_ws.append((lay, wsb))
    torch.cuda.synchronize()

    def mx_gateup_body():
        for lay, wsb in stage_ws:
            moe.check(moe.moe_ffn_layer_packed_stage(lay.packed_struct, None, 1, wsb, wsb.numel(),
                                                     moe.MOE_STAGE_GATEUP, stream=stream), "gateup")

    mx_kern_s = graph_seconds(stream, mx_gateup_body)[0] / Kk
    del stage_ws
    mx_rate, _ = whole_job_rate(K, mx_secs, dist)

    # ---- the same decode step with gate/up stored interleaved (one [2F][D] plane per expert) ----
    from synthetic import interleave_gate_up
    ilv_layers = [moe.MoeLayer(interleave_gate_up(make_layer_torch(spec, li + 17 * dist.rank, dev)), k=K_TOP,
                               device=dev) for li in range(NL)]
    with torch.cuda.stream(stream):
        for i in range(3):
            ilv_layers[i % NL](xs[i:i + 1], rail=head_rail, out=ys[i:i + 1])
    torch.cuda.synchronize()

    def ilv_body():
        for i in range(K):
            j = W + i
            ilv_layers[j % NL](xs[j:j + 1], rail=head_rail, out=ys[j:j + 1])

    ilv_secs = graph_seconds(stream, ilv_body)[0]
    check_status(moe, stream)
    ilv_rate, _ = whole_job_rate(K, ilv_secs, dist)
    del ilv_layers

    # ---- rail crossover, T = 1 .. 512 (same layers) ----
    crossover = None if args.no_crossover else run_crossover(moe, layers, stream, dev, dist)

    result = {
        "metric": METRIC, "value": round(rate, 1), "unit": "tokens/s", "n_gpus": dist.world, "steps": K,
        "warmup": W, "ms_per_step": round(secs_max / K * 1e3, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32 accumulate; MXFP4 weights, f32 activations carried as f16 hi + lo parts (~22 significant bits)",
        "data": "synthetic",
        "config": decode_config(dist.world, f"replicas x{dist.world}",
                                f"inputs larger than L2: {NL} distinct layer weight sets "
                                f"({NL * E * EXPERT_BYTES / 1e9:.1f} GB) rotated every step",
                                "one CUDA graph of the timed steps, CUDA events on its stream"),
        "rail": "gemv (router; fused gate/up + swiglu with mma.sync inner products; fused down + combine on the CUDA cores)",
        "weight_gbs": round(weight_bytes_step * K / secs_max * dist.world / 1e9, 1),
        "layer_roofline_frac": round((step_bytes / (hbm_peak * 1e9)) / (secs_max / K), 4),
        "roofline": roofline,
        "e2e": {"value": round(e2e_rate, 1), "unit": "tokens/s", "h2d_bytes_per_step": D * 4, "d2h_bytes_per_step": D * 4,
                "path": "MoeLayer.forward_host -> moe_ffn_layer_hostio (x in, layer, y out in one call), then the "
                        "host waits for y every step (wall clock)"},
        "e2e_pipelined": {"value": round(pipe_rate, 1), "unit": "tokens/s",
                          "path": "the same calls back to back without the per-step wait (CUDA events)"},
        "decode_t1_tensor_core": {
            "tokens_per_s": round(mx_rate, 1), "ms_per_step": round(mx_secs / K * 1e3, 5),
            "rail": "decode_mx (block-scaled tcgen05 MMA on prepacked MXFP4 weights, activations as 8 E2M1 terms)",
            "gateup_kernel": "decode_mx_kernel<0>", "gateup_launch_us": round(mx_kern_s * 1e6, 3),
            "gateup_frac": round(gateup_bytes / mx_kern_s / 1e9 / hbm_peak, 4)},
        "decode_t1_interleaved": {"tokens_per_s": round(ilv_rate, 1), "ms_per_step": round(ilv_secs / K * 1e3, 5),
                                  "rail": "gemv on gate/up stored interleaved (moe_ffn_layer_gu: one copy of a "
                                          "sub-task's 2x8 gate/up rows)"},
        "crossover": crossover,
        "clocks": clocks,
        "gpu_launches": int(round(launches_per_step * K)),
        "kernels_per_step": launches_per_step,
    }
    del layers
    torch.cuda.empty_cache()

    if not args.no_prefill:
        result["prefill_t512"] = run_prefill(args, dist, moe, dev, stream, hbm_peak, bf16_peak, peak_src,
                                             rail=moe.MOE_RAIL_GROUPED_MX4)
        result["prefill_t512_bf16"] = run_prefill(args, dist, moe, dev, stream, hbm_peak, bf16_peak, peak_src,
                                                  rail=moe.MOE_RAIL_GROUPED_MM)
        result["prefill_t512_mx"] = run_prefill(args, dist, moe, dev, stream, hbm_peak, bf16_peak, peak_src,
                                                rail=moe.MOE_RAIL_GROUPED_MX)
        result["skew_t4096"] = run_prefill(args, dist, moe, dev, stream, hbm_peak, bf16_peak, peak_src, cfg=4,
                                           rail=moe.MOE_RAIL_GROUPED_MX4)
        result["skew_t4096_bf16"] = run_prefill(args, dist, moe, dev, stream, hbm_peak, bf16_peak, peak_src, cfg=4,
                                                rail=moe.MOE_RAIL_GROUPED_MM)
        result["skew_t4096_mx"] = run_prefill(args, dist, moe, dev, stream, hbm_peak, bf16_peak, peak_src, cfg=4,
                                              rail=moe.MOE_RAIL_GROUPED_MX)
    if not args.no_stack:
        result["stack24"] = run_stack(args, dist, moe, dev, stream, hbm_peak)
    return result


def run_crossover(moe, layers, stream, dev, dist, Ts=(1, 2, 4, 8, 16, 32, 64, 128, 256, 512), steps=10):
    """Microseconds per layer step of each rail at T tokens (f-4: where the
    decode rails should hand over to the grouped rails)."""
    import torch

    rails = {"gemv": moe.MOE_RAIL_GEMV, "decode_mx": moe.MOE_RAIL_DECODE_MX,
             "grouped_mm": moe.MOE_RAIL_GROUPED_MM, "grouped_mx": moe.MOE_RAIL_GROUPED_MX,
             "grouped_mx4": moe.MOE_RAIL_GROUPED_MX4}
    NL = len(layers)
    out = {"unit": "us per layer step", "layers_rotated": NL, "steps": steps}
    g = torch.Generator(device=dev)
    g.manual_seed(515)
    for T in Ts:
        xs = [torch.randn((T, D), generator=g, device=dev) for _ in range(NL)]
        ys = [torch.empty((T, D), device=dev) for _ in range(NL)]
        row = {}
        for name, rail in rails.items():
            if rail in (moe.MOE_RAIL_GEMV, moe.MOE_RAIL_DECODE_MX) and T > moe.MOE_GEMV_MAX_T:
                continue
            with torch.cuda.stream(stream):
                for i in range(2):
                    layers[i % NL](xs[i % NL], rail=rail, out=ys[i % NL])
            torch.cuda.synchronize()

            def body(rail=rail):
                for i in range(steps):
                    layers[i % NL](xs[i % NL], rail=rail, out=ys[i % NL])

            sec = graph_seconds(stream, body)[0] / steps
            row[name] = round(dist.max(sec) * 1e6, 2)
        check_status(moe, stream)
        out[f"T{T}"] = row
    best = {}
    for T in Ts:
        r = out[f"T{T}"]
        best[f"T{T}"] = min(r, key=r.get)
    out["fastest"] = best
    return out


def run_prefill(args, dist, moe, dev, stream, hbm_peak, bf16_peak, peak_src, rail=None, cfg=2):
    import torch
    from synthetic import make_layer_torch, spec_for

    spec = spec_for(cfg)
    T = spec.T
    K = args.prefill_steps if cfg == 2 else max(3, args.prefill_steps // 4)
    if rail is None:
        rail = moe.MOE_RAIL_GROUPED_MM
    NL = 2
    packed = rail == moe.MOE_RAIL_GROUPED_MX4
    layers = [moe.MoeLayer(make_layer_torch(spec, li + 31 * dist.rank, dev), k=K_TOP, device=dev, packed=packed,
                           keep_canonical=not packed) for li in range(NL)]
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
    check_status(moe, stream)
    ms = secs_max / K * 1e3
    # experts touched: every expert at these sizes (near-uniform or skewed routing of T*k >= 2048 assignments)
    weight_bytes = E * EXPERT_BYTES
    alg_bytes = weight_bytes + 3 * E * F * 4 + E * D * 4 + 2 * T * D * 4
    flops = T * K_TOP * 3 * 2 * D * F
    t_roof = max(alg_bytes / (hbm_peak * 1e9), flops / (bf16_peak * 1e12))
    del graph, layers
    torch.cuda.empty_cache()
    workload = WORKLOAD_PREFILL if cfg == 2 else WORKLOAD_SKEW
    return {"tokens_per_s": round(rate, 1), "ms_per_step": round(ms, 4), "steps": K, "workload": workload,
            "weight_gbs": round(weight_bytes / (ms / 1e3) / 1e9, 1),
            "dtype": {moe.MOE_RAIL_GROUPED_MM: "bf16 MMA, fp32 accumulate",
                      moe.MOE_RAIL_GROUPED_MX: "MXFP4 x E4M3-term block-scaled MMA (x: 3 terms, h: 2), fp32 accumulate",
                      moe.MOE_RAIL_GROUPED_MX4: "MXFP4 x E2M1-term block-scaled MMA, kind::mxf4 on prepacked weights "
                                                "(x: 6 terms, h: 4), fp32 accumulate"}[rail],
            "rail": {moe.MOE_RAIL_GROUPED_MM: "grouped_mm", moe.MOE_RAIL_GROUPED_MX: "grouped_mx",
                     moe.MOE_RAIL_GROUPED_MX4: "grouped_mx4"}[rail],
            "roofline_frac": round(t_roof / (ms / 1e3), 4),
            "roofline_bound": "hbm" if alg_bytes / (hbm_peak * 1e9) >= flops / (bf16_peak * 1e12) else "tensor",
            "roofline_us": round(t_roof * 1e6, 1),
            "algorithmic_bytes": alg_bytes, "algorithmic_flops": flops, "kernels_per_step": per_step,
            "peak_source": peak_src, "clocks": clk.summary()}


def run_stack(args, dist, moe, dev, stream, hbm_peak, NLS=24):
    """The stacked workload: NLS distinct layers resident (about 10 GB of MXFP4
    weights, far beyond L2), the hidden state carried layer to layer with an RMS
    renormalisation between layers; T=1 decoded for args.stack_steps tokens, and
    T=512 for a few passes."""
    import torch
    from synthetic import make_layer_torch, spec_for

    spec = spec_for(3)
    # canonical planes (the T=1 GEMV rail) and the prepacked copy (the T=512 kind::mxf4 rail)
    layers = [moe.MoeLayer(make_layer_torch(spec, li + 101 * dist.rank, dev), k=K_TOP, device=dev, packed=True)
              for li in range(NLS)]
    res = {"workload": WORKLOAD_STACK, "layers": NLS,
           "resident_weight_gb": round(NLS * E * EXPERT_BYTES / 1e9, 2)}
    g = torch.Generator(device=dev)
    g.manual_seed(2024 + dist.rank)
    for T, steps, rail in ((1, args.stack_steps, moe.MOE_RAIL_GEMV), (512, 3, moe.MOE_RAIL_GROUPED_MX4)):
        h = [torch.randn((T, D), generator=g, device=dev), torch.empty((T, D), device=dev)]

        def one_pass():
            for li in range(NLS):
                layers[li](h[0], rail=rail, out=h[1])
                moe.check(moe.moe_rms_renorm(h[1], T, D, h[0], stream), "rms_renorm")

        with torch.cuda.stream(stream):
            one_pass()
        torch.cuda.synchronize()
        n0 = moe.moe_kernel_launches()
        sec, graph = graph_seconds(stream, lambda: [one_pass() for _ in range(steps)])
        launches = (moe.moe_kernel_launches() - n0) / steps
        del graph
        check_status(moe, stream)
        rate, secs_max = whole_job_rate(steps * T, sec, dist)
        touched = E if T > 8 else K_TOP
        per_pass = secs_max / steps
        res[f"T{T}"] = {"tokens_per_s": round(rate, 2), "ms_per_token_pass" if T == 1 else "ms_per_pass":
                        round(per_pass * 1e3, 4), "passes": steps, "rail": "gemv" if T == 1 else "grouped_mx4",
                        "us_per_layer": round(per_pass / NLS * 1e6, 2),
                        "weight_gbs": round(NLS * touched * EXPERT_BYTES / per_pass / 1e9, 1),
                        "weight_roofline_frac": round(NLS * touched * EXPERT_BYTES / per_pass / 1e9 / hbm_peak, 4),
                        "kernels_per_pass": launches}
    del layers
    torch.cuda.empty_cache()
    return res


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
            if "prefill_t512" in res:
                prate, pdt = cpu_oracle_prefill_rate(2, 8)
                res["cpu_baseline_prefill_t512"] = {
                    "value": round(prate, 4), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                    "sample": f"8 of the prefill batch's tokens in one oracle call ({pdt:.1f} s; each touched "
                              "expert dequantised once for the call)"}
            if "stack24" in res:
                srate, sdt = cpu_oracle_stack_rate(2, 24)
                res["cpu_baseline_stack24_t1"] = {
                    "value": round(srate, 5), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                    "sample": f"1 token through 2 of the 24 layers with the renormalisation ({sdt:.1f} s), "
                              "scaled to 24 layers"}
        print(json.dumps(res), flush=True)
    dist.close()


if __name__ == "__main__":
    main()
