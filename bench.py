"""Benchmark of the MXFP8 MoE hot path on GB300.

A step is one MoE FFN layer forward + backward over the MoE-FFN shapes (T=16384
tokens, top-8 of E=32 experts -> 131072 routed rows, hidden 7168, expert
intermediate 2048): weight and activation quantization (rowwise and columnwise),
permutation by expert, quantize-on-gather, the six grouped MXFP8 GEMMs (two forward,
two dgrad, two wgrad), SwiGLU fused with quantization (forward and backward), combine
back to token order and its backward.
All inputs are seeded synthetic tensors already resident in HBM (each far larger
than the 129 MB L2, so no flush is needed between steps).

value      GEMM FLOPs of the step / step time (quantize + permute time included).
roofline   the grouped-GEMM kernel (the dominant kernel): its FLOPs / its own
           CUDA-event time, against the dense FP8 peak.
quantizer  the 16384 x 7168 log-normal quantizer workload, rowwise+columnwise in
           one read, against the HBM peak.
e2e        the same metric through the public API with host buffers: per step the
           layer's inputs (activations, routing ids, gates, output gradient) are copied
           from pinned host memory and its outputs (forward output, input gradient)
           copied back, overlapped with compute on separate streams.
--impl reference  times the CPU oracle on a bounded sample of the same workload.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

CFG = dict(T=16384, E=32, k=8, hidden=7168, inter=2048)
# a reduced case of the same kernels for profiler captures (a few GB on the device)
SMALL_CFG = dict(T=4096, E=16, k=4, hidden=7168, inter=2048)
QUANT_CFG = dict(rows=16384, cols=7168)
FP8_OVER_BF16 = 2.0    # nominal dense FP8 / BF16 tensor throughput ratio (4.5 / 2.25 PFLOP/s)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
NOMINAL = {"hbm_gbs": 7900.0, "fp8_tflops": 4500.0}   # GB300 datasheet figures (dense), for context


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        out = {}
        for key in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
            v = d.get(key)
            if isinstance(v, dict):
                v = v.get("value")
            out[key] = float(v) if v is not None else FALLBACK_PEAKS[key]
        out["source"] = "measured"
        return out
    out = dict(FALLBACK_PEAKS)
    out["source"] = "fallback"
    return out


def dist_info():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(value: float, device="cpu") -> float:
    """The largest of every rank's value (the slowest replica sets the job's time)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, seconds: float) -> float:
    """Whole-job throughput of weak-scaled replicas: every rank processed units_per_rank."""
    return units_per_rank * world / seconds


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + q,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx_, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx_.append(float(parts[2]))
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx_), "reasons": sorted(reasons),
                "samples": len(sm)}


def gemm_source_hash():
    with open(os.path.join(ROOT, "mxfp8_block_scaled_rowwise_gb300", "csrc", "gemm.cu"), "rb") as f:
        return hashlib.sha1(f.read()).hexdigest()[:12]


def recorded_traffic(kernel_hash: str):
    """Average DRAM bytes per grouped-GEMM launch of the full step, from the committed ncu
    summary, if it was taken on this exact kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "grouped_gemm_ffn.md")
    if not os.path.exists(path):
        return None
    for ln in open(path):
        if ln.startswith("traffic_bytes_per_launch:"):
            parts = dict(p.split("=") for p in ln.split(":", 1)[1].split() if "=" in p)
            if parts.get("gemm_cu_sha1") == kernel_hash and parts.get("scope") == "full-step-avg":
                return float(parts["bytes"])
    return None


# ---------------------------------------------------------------------------- our arm
def fill_inputs(step, seed_base=1003):
    import torch
    from mxfp8_block_scaled_rowwise_gb300 import synth
    g = synth.generator(seed_base, step.dev)
    step.x.copy_(synth.randn_bf16(step.x.shape, g, device=step.dev))
    logits = torch.randn(step.T, step.E, generator=g, device=step.dev)
    step.ids.copy_(synth.topk_ids(logits, step.k))
    step.gate.copy_(torch.softmax(logits.gather(1, step.ids.long()), dim=1))
    step.w1.copy_(synth.randn_bf16(step.w1.shape, g, device=step.dev))
    step.w2.copy_(synth.randn_bf16(step.w2.shape, g, device=step.dev))
    g2 = synth.generator(seed_base + 1, step.dev)
    step.dout.copy_(synth.randn_bf16(step.dout.shape, g2, std=1e-2, device=step.dev))


def time_quantizer(torch, mx, dev, iters=20, warmup=5):
    from mxfp8_block_scaled_rowwise_gb300 import synth
    d = synth.quant(device=dev)
    x = d["x"]
    rows, cols = x.shape
    res = {}
    for name, mode, bpe in (("row", mx.MX_ROWWISE, 2 + 1 + 1 / 32), ("row+col", mx.MX_ROWWISE | mx.MX_COLWISE,
                                                                     2 + 2 * (1 + 1 / 32))):
        out = mx.quantize_alloc(x, mode)
        q = (out["q_row"], out["sf_row"], out["q_col"], out["sf_col"])

        def run():
            mx.mxfp8_quantize(x, rows, cols, mode, None, None, 0, out["ld_col"], *q, None)
        for _ in range(warmup):
            run()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
        for a, b in ev:
            a.record()
            run()
            b.record()
        torch.cuda.synchronize()
        ms = statistics.median(a.elapsed_time(b) for a, b in ev)
        nbytes = rows * cols * bpe
        res[name] = {"ms": ms, "GB/s": nbytes / (ms * 1e-3) / 1e9, "bytes": nbytes}
        del out, q
    del x, d
    return res


def run_ours(args):
    import torch
    import torch.distributed as dist
    from mxfp8_block_scaled_rowwise_gb300 import _build
    from mxfp8_block_scaled_rowwise_gb300 import binding as mx
    from mxfp8_block_scaled_rowwise_gb300.layer import MoEFFNStep

    rank, world, local = dist_info()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if rank == 0:
        _build.build()
    if world > 1:
        dist.barrier()
    mx.load()
    pk = peaks()
    if args.only == "gemm":
        # the GEMM1 shape alone (131072 routed rows over 32 experts, N=4096, K=7168) on seeded
        # synthetic E4M3 codes with unit scales (about 3 GB on the device), for profiler captures
        g = torch.Generator(device=dev)
        g.manual_seed(17)
        E, T_e, N, K = CFG["E"], CFG["T"] * CFG["k"] // CFG["E"], 2 * CFG["inter"], CFG["hidden"]
        R = E * T_e
        A = torch.randint(0, 256, (R, K), dtype=torch.uint8, device=dev, generator=g)
        B = torch.randint(0, 256, (E * N, K), dtype=torch.uint8, device=dev, generator=g)
        A[(A & 0x7F) == 0x7F] = 0x38
        B[(B & 0x7F) == 0x7F] = 0x38
        pb = mx.mx_padded_rows_bound(R, E)
        SFA = torch.full((mx.mx_sf_bytes(pb, K // 32),), 127, dtype=torch.uint8, device=dev)
        SFB = torch.full((mx.mx_sf_bytes_x4(E * N, K // 32),), 127, dtype=torch.uint8, device=dev)
        off = torch.arange(0, (E + 1) * T_e, T_e, dtype=torch.int32, device=dev)
        C = torch.empty(R, N, dtype=torch.bfloat16, device=dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        run = lambda: mx.grouped_gemm_mxfp8_fwd(A, SFA, B, SFB, off, off, E, R, N, K, C, err)
        for _ in range(3):
            run()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(10)]
        for a, b in ev:
            a.record()
            run()
            b.record()
        torch.cuda.synchronize()
        ms = statistics.median(a.elapsed_time(b) for a, b in ev)
        assert int(err.item()) == 0
        if rank == 0:
            print(json.dumps({"gemm": "GEMM1 shape", "ms": round(ms, 4),
                              "TFLOP/s": round(2.0 * R * N * K / (ms * 1e-3) / 1e12, 1)}), flush=True)
        return
    if args.only == "quantizer":
        # the 16384 x 7168 quantizer workload alone (about 0.8 GB on the device), for profiler captures
        q = time_quantizer(torch, mx, dev)
        if rank == 0:
            print(json.dumps({"quantizer": {k: {"GB/s": round(v["GB/s"], 1), "ms": round(v["ms"], 4),
                                                "frac": round(v["GB/s"] / pk["hbm_gbs"], 4)} for k, v in q.items()},
                              "peak_source": pk["source"]}), flush=True)
        return

    cfg = SMALL_CFG if args.shape == "small" else CFG
    step = MoEFFNStep(device=dev, **cfg)
    fill_inputs(step)
    torch.cuda.synchronize()
    flops = step.gemm_flops()
    step_flops = sum(flops.values())

    # per-launch GEMM timing with CUDA events on the launching (current) stream
    gemm_events = []

    def hook(name, fl, fn):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        gemm_events.append((name, fl, a, b))

    for _ in range(args.warmup):
        step.step()
    torch.cuda.synchronize()
    assert int(step.dev_err.item()) == 0, "device error %d" % int(step.dev_err.item())

    # timed region: K steps, barrier + synchronize on both sides
    step.gemm_hook = hook
    launches0 = step.launches
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        t_start.record()
        for _ in range(args.steps):
            step.step()
        t_end.record()
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    step.gemm_hook = None
    launches = step.launches - launches0
    ms_total = max_over_ranks(t_start.elapsed_time(t_end), dev)
    ms_step = ms_total / args.steps
    gemm_ms = sum(a.elapsed_time(b) for _, _, a, b in gemm_events)
    gemm_fl = sum(fl for _, fl, _, _ in gemm_events)
    per_kind = {}
    for name, fl, a, b in gemm_events:
        d = per_kind.setdefault(name, [0.0, 0, 0.0])
        d[0] += a.elapsed_time(b)
        d[1] += 1
        d[2] += fl
    assert int(step.dev_err.item()) == 0
    value = job_throughput(step_flops, world, ms_step * 1e-3) / 1e12

    checks = gemm_checks(torch, mx, step) if rank == 0 else None
    assert int(step.dev_err.item()) == 0

    # e2e: same step through the public API with pinned host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(torch, step, args, step_flops, world)

    quant = time_quantizer(torch, mx, dev) if (rank == 0 and args.shape == "ffn") else {}
    cpu = cpu_baseline(args) if (rank == 0 and world == 1 and not args.no_cpu_baseline) else None

    if rank == 0:
        fp8_peak = pk["bf16_tflops_sustained"] * FP8_OVER_BF16
        achieved = gemm_fl / (gemm_ms * 1e-3) / 1e12
        kh = gemm_source_hash()
        traffic = recorded_traffic(kh)
        n_launch = len(gemm_events)
        line = {
            "metric": "grouped-GEMM MXFP8 TFLOPS (% FP8 peak); quantizer GB/s (% HBM peak), 1 GB300",
            "value": round(value, 2),
            "unit": "TFLOP/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms_step, 4),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "e4m3",
            "data": "synthetic (seeded N(0,1) bf16 activations/weights, N(0,1e-2) gradients, top-8 routing of N(0,1) logits)",
            "config": {"workload": "MoE FFN fwd+bwd step: T=%d, top-%d of E=%d (R=%d), hidden %d, "
                                   "intermediate %d (GEMM1 N=%d), MXFP8 E4M3 + E8M0/32" % (
                                       cfg["T"], cfg["k"], cfg["E"], cfg["T"] * cfg["k"], cfg["hidden"],
                                       cfg["inter"], 2 * cfg["inter"]),
                       "global_batch": cfg["T"] * world, "seq_len": None, "parallelism": "replicas" if world > 1 else "single",
                       "gemm_flops_per_step": step_flops, "l2": "inputs > L2 (129 MB); no flush needed"},
            "roofline": {"bound": "tensor", "kernel": "grouped_gemm_kernel (fwd/dgrad/wgrad)",
                         "achieved": round(achieved, 1), "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
                         "frac": round(achieved / fp8_peak, 4), "traffic": traffic,
                         "frac_of_nominal": round(achieved / NOMINAL["fp8_tflops"], 4),
                         "peak_note": "dense FP8 = %s sustained bf16 cuBLAS (%.1f) x %.1f nominal FP8/BF16 ratio" % (
                             pk["source"], pk["bf16_tflops_sustained"], FP8_OVER_BF16),
                         "launches_per_step": n_launch // args.steps, "gemm_cu_sha1": kh,
                         "per_gemm": {k: {"ms": round(v[0] / v[1], 4), "TFLOP/s": round(v[2] / (v[0] * 1e-3) / 1e12, 1)}
                                      for k, v in per_kind.items()}},
            "gemm_checks": checks,
            "quantizer": {name: {"GB/s": round(v["GB/s"], 1), "ms": round(v["ms"], 4),
                                 "frac": round(v["GB/s"] / pk["hbm_gbs"], 4),
                                 "frac_of_nominal": round(v["GB/s"] / NOMINAL["hbm_gbs"], 4)} for name, v in quant.items()},
            "quantizer_note": "16384x7168 bf16 log-normal rows + 0.1%% outliers; bytes = 2 in + (1 + 1/32) per output form; "
                              "peak = %s HBM copy %.1f GB/s" % (pk["source"], pk["hbm_gbs"]),
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_e2e(torch, step, args, step_flops, world):
    """The step through the public API with host buffers.  Per step: H2D of the layer's inputs
    (x, routing ids, gates, output gradient) from pinned memory, the step, D2H of the layer's
    outputs (forward output and input gradient, token order) into pinned memory.  Copies run on their own streams and overlap the neighbouring steps' compute
    (double-buffered device inputs and outputs); the timed region spans the first H2D to the
    last D2H."""
    in_names = ["x", "ids", "gate", "dout"]
    out_names = ["out", "dx"]
    slots_in = [{n: getattr(step, n) for n in in_names},
                {n: torch.empty_like(getattr(step, n)) for n in in_names}]
    slots_out = [{n: getattr(step, n) for n in out_names},
                 {n: torch.empty_like(getattr(step, n)) for n in out_names}]
    h_in = {n: torch.empty(getattr(step, n).shape, dtype=getattr(step, n).dtype, pin_memory=True) for n in in_names}
    h_out = [{n: torch.empty(getattr(step, n).shape, dtype=getattr(step, n).dtype, pin_memory=True)
              for n in out_names} for _ in range(2)]
    for n in in_names:
        h_in[n].copy_(getattr(step, n))
    torch.cuda.synchronize()
    s_h2d, s_cmp, s_d2h = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    in_ready = [ev(), ev()]
    in_free = [ev(), ev()]
    done = [ev(), ev()]
    out_free = [ev(), ev()]
    for i in range(2):
        in_free[i].record(s_cmp)
        out_free[i].record(s_d2h)

    def run(n):
        for i in range(n):
            sl = i & 1
            with torch.cuda.stream(s_h2d):
                s_h2d.wait_event(in_free[sl])
                for nm in in_names:
                    slots_in[sl][nm].copy_(h_in[nm], non_blocking=True)
                in_ready[sl].record(s_h2d)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(in_ready[sl])
                s_cmp.wait_event(out_free[sl])
                for nm in in_names:
                    setattr(step, nm, slots_in[sl][nm])
                for nm in out_names:
                    setattr(step, nm, slots_out[sl][nm])
                step.step()
                in_free[sl].record(s_cmp)
                done[sl].record(s_cmp)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(done[sl])
                for nm in out_names:
                    h_out[sl][nm].copy_(slots_out[sl][nm], non_blocking=True)
                out_free[sl].record(s_d2h)

    run(2)
    torch.cuda.synchronize()
    n = max(4, args.steps)
    t0 = time.perf_counter()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_h2d)
    s_cmp.wait_stream(s_h2d)
    s_d2h.wait_stream(s_h2d)
    run(n)
    s_h2d.wait_stream(s_d2h)
    s_h2d.wait_stream(s_cmp)
    b.record(s_h2d)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / n
    wall_ms = (time.perf_counter() - t0) * 1e3 / n
    for nm in in_names:     # leave the step pointing at its original buffers
        setattr(step, nm, slots_in[0][nm])
    for nm in out_names:
        setattr(step, nm, slots_out[0][nm])
    return {"value": round(step_flops * world / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": int(sum(getattr(step, n).numel() * getattr(step, n).element_size() for n in in_names)),
            "d2h_bytes_per_step": int(sum(getattr(step, n).numel() * getattr(step, n).element_size() for n in out_names)),
            "ms_per_step": round(ms, 3), "host_wall_ms_per_step": round(wall_ms, 3),
            "overlap": "H2D, compute and D2H on separate streams, double-buffered device inputs/outputs"}


def gemm_checks(torch, mx, step, reps=10):
    """Target checks on the GEMM1 shape (R routed rows x N=2I x K=H): the grouped GEMM vs an
    equal-FLOP dense GEMM (same kernel, E = 1), and 2-CTA pairs vs single-CTA tiles."""
    R, H, I2, E = step.R, step.H, step.I2, step.E
    dense_off = torch.tensor([0, R], dtype=torch.int32, device=step.dev)

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a, b in ev:
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in ev)

    grouped = lambda: mx.grouped_gemm_mxfp8_fwd(step.a1_q, step.a1_sf, step.w1_q, step.w1_sf, step.off, step.poff, E,
                                                 R, I2, H, step.out1, step.dev_err)
    dense = lambda: mx.grouped_gemm_mxfp8_fwd(step.a1_q, step.a1_sf, step.w1_q, step.w1_sf, dense_off, dense_off, 1,
                                               R, I2, H, step.out1, step.dev_err)
    fl = 2.0 * R * I2 * H
    t_g = timed(grouped)
    t_d = timed(dense)
    os.environ["MXMOE_GEMM_CTAS"] = "1"
    try:
        t_1 = timed(grouped)
    finally:
        del os.environ["MXMOE_GEMM_CTAS"]
    tf = lambda ms: round(fl / (ms * 1e-3) / 1e12, 1)
    out = {"shape": "GEMM1: %d routed rows over %d experts, N=%d, K=%d" % (R, E, I2, H),
           "grouped_tflops": tf(t_g), "dense_e1_tflops": tf(t_d), "grouped_over_dense": round(t_d / t_g, 4),
           "single_cta_tflops": tf(t_1), "two_cta_speedup": round(t_1 / t_g, 4)}
    out["library_mxfp8"] = library_mxfp8(torch, step, timed, fl, tf)
    return out


def library_mxfp8(torch, step, timed, fl, tf):
    """A measured MXFP8 reference: the library block-scaled GEMM (torch._scaled_mm with E8M0
    scales, which reads the same tensor-core scale layout) on the dense GEMM1 shape, fed the
    step's own codes and scales (timing only; its output is not used by the step)."""
    R, H, I2 = step.R, step.H, step.I2
    try:
        A = step.a1_q.view(torch.float8_e4m3fn)
        B = step.w1_q[:I2].view(torch.float8_e4m3fn)                    # expert 0's W1 [2I x H]
        sa = step.a1_sf[: R * (H // 32)].view(torch.float8_e8m0fnu)      # scale rows of R padded positions
        sb = step.w1_sf.view(-1, 4, 512)[:, 0].reshape(-1)[: I2 * (H // 32)].view(torch.float8_e8m0fnu)
        out = torch.empty(R, I2, dtype=torch.bfloat16, device=step.dev)
        run = lambda: torch._scaled_mm(A, B.t(), sa, sb, out_dtype=torch.bfloat16, out=out)
        return {"tflops": tf(timed(run)), "what": "torch._scaled_mm (cuBLAS MXFP8, E8M0 1x32 scales), "
                "M=%d N=%d K=%d" % (R, I2, H)}
    except Exception as e:   # an older torch or a library without MXFP8 support
        return {"unavailable": "%s: %s" % (type(e).__name__, str(e)[:160])}


# ---------------------------------------------------------------------------- CPU oracle
def cpu_baseline(args, budget_s: float = 12.0):
    """Time the CPU oracle (as it stands, one host thread) on a bounded sample of the step's
    work and extrapolate the step time from the measured per-unit rates."""
    import numpy as np
    import torch
    import oracle
    from mxfp8_block_scaled_rowwise_gb300 import synth
    oracle.build()
    T, E, k, H, I = CFG["T"], CFG["E"], CFG["k"], CFG["hidden"], CFG["inter"]
    I2, R = 2 * I, T * k
    g = synth.generator(7)
    t0 = time.perf_counter()

    def rate(fn, units, share):
        """units per second of fn, repeated for about share x budget_s seconds"""
        n, t = 0, time.perf_counter()
        while True:
            fn()
            n += 1
            if time.perf_counter() - t > share * budget_s:
                return n * units / (time.perf_counter() - t), n

    # quantizer rates (rowwise and columnwise) on 1024 x 7168 blocks of the step's activations
    xb = synth.bf16_bits(synth.randn_bf16((1024, H), g))
    q_rate_row, n_row = rate(lambda: oracle.quantize_rowwise(xb), xb.size, 0.2)
    q_rate_col, n_col = rate(lambda: oracle.quantize_colwise_seg(xb, [0, 1024], [0, 1024], 1024), xb.size, 0.2)
    # permutation rate on the full routing of the step
    ids = synth.topk_ids(torch.randn(T, E, generator=g), k).numpy()
    p_rate, n_perm = rate(lambda: oracle.permute(ids, E), ids.size, 0.1)
    # GEMM rate: sampled rows of GEMM1 (K = 7168) against 512 weight rows
    qa, sa = oracle.quantize_rowwise(synth.bf16_bits(synth.randn_bf16((8, H), g)))
    qb, sb = oracle.quantize_rowwise(synth.bf16_bits(synth.randn_bf16((512, H), g)))
    gemm_rate, reps = rate(lambda: oracle.gemm_nt(qa, sa, qb, sb), 2 * 8 * 512 * H, 0.5)
    # extrapolated step: element counts of every quantization in the step, routed slots, GEMM FLOPs
    row_elems = E * I2 * H + E * H * I + T * H + R * I + R * H + R * I2
    col_elems = E * I2 * H + E * H * I + R * I + R * H + R * I2 + R * H
    step_flops = 3 * 2 * R * (I2 * H + H * I)
    t_step = row_elems / q_rate_row + col_elems / q_rate_col + R / p_rate + step_flops / gemm_rate
    value = step_flops / t_step / 1e12
    return {"value": value, "unit": "TFLOP/s", "cores": 1, "host_cores": os.cpu_count(), "kind": "oracle",
            "sample": "single-thread C oracle: rowwise and colwise quantize of 1024x7168 (x%d, x%d), full top-8 "
                      "permutation of 16384 tokens (x%d), fp64 GEMM of 8x512x7168 (x%d); step time extrapolated "
                      "from these rates (%.0f s measured)" % (n_row, n_col, n_perm, reps, time.perf_counter() - t0),
            "extrapolated_step_s": round(t_step, 1),
            "rates": {"quant_row_elem_per_s": round(q_rate_row), "quant_col_elem_per_s": round(q_rate_col),
                      "permute_slots_per_s": round(p_rate), "gemm_flop_per_s": round(gemm_rate)}}


def run_reference(args):
    rank, world, _ = dist_info()
    if rank != 0:
        return
    steps = []
    res = None
    for _ in range(args.warmup + args.steps):
        t = time.perf_counter()
        res = cpu_baseline(args, budget_s=4.0)
        steps.append(time.perf_counter() - t)
    value = res["value"]
    line = {
        "impl": "reference",
        "metric": "grouped-GEMM MXFP8 TFLOPS (% FP8 peak); quantizer GB/s (% HBM peak), 1 GB300",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": res["extrapolated_step_s"] * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "MoE FFN fwd+bwd step: T=16384, top-8 of E=32 (R=131072), hidden 7168, "
                               "intermediate 2048 (GEMM1 N=4096), MXFP8 E4M3 + E8M0/32"},
        "cpu_baseline": {"kind": "oracle", "cores": 1, "sample": res["sample"], "value": value},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", default=None, choices=["quantizer", "gemm"],
                    help="run only the 16384 x 7168 quantizer timing, or only the GEMM1-shape grouped GEMM "
                         "(small cases for profiler captures)")
    ap.add_argument("--shape", default="ffn", choices=["ffn", "small"],
                    help="ffn: the MoE FFN workload (default); small: a reduced case for profiler captures")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
