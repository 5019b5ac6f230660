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
import datetime
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
# the FP8 tensor pipe of one SM: 8192 multiply-adds per clock (16384 FLOP); with the SM clock
# sampled during the timed region this gives the pipe's own ceiling (5.15 PFLOP/s at 2.07 GHz)
TENSOR_PIPE_FP8_FLOP_PER_CLK_SM = 16384


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
    """nvidia-smi clock / throttle sampling during the timed region: samples every 50 ms, each
    with its timestamp; the summary keeps those taken between entering and leaving the block
    (all samples if the region was shorter than one interval, marked in "window")."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.t0 = self.t1 = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)   # nvidia-smi's start-up
        self.t0 = time.time()
        return self

    def __exit__(self, *exc):
        self.t1 = time.time()
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    @staticmethod
    def parse(line):
        """(epoch seconds, SM MHz, max SM MHz, set of active reasons) of one sample, or None."""
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 10:
            return None
        try:
            ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            sm, smax = float(parts[2]), float(parts[3])
        except ValueError:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        return ts, sm, smax, {n for n, v in zip(names, parts[6:10]) if v.lower().startswith("active")}

    def summary(self):
        samples = [x for x in (self.parse(ln) for ln in self.lines) if x is not None]
        window = "timed region"
        inside = [x for x in samples if self.t0 is not None and self.t0 - 0.05 <= x[0] <= self.t1 + 0.05]
        if not inside:
            inside, window = samples, "whole sampler run (timed region shorter than one interval)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(x[1] for x in inside), "sm_max_mhz": max(x[2] for x in inside),
                "reasons": sorted(set().union(*(x[3] for x in inside))), "samples": len(inside),
                "interval_ms": 50, "window": window}


def gemm_source_hash():
    with open(os.path.join(ROOT, "mxfp8_block_scaled_rowwise_gb300", "csrc", "gemm.cu"), "rb") as f:
        return hashlib.sha1(f.read()).hexdigest()[:12]


# DRAM bytes (read + written) of one grouped-GEMM launch on the GEMM1 shape (131072 routed
# rows over 32 experts, N=4096, K=7168): the mean of three launches of a one-kernel ncu capture
# of `bench.py --only gemm` (command and figures in profiles/grouped_gemm_ffn.md), valid while
# gemm.cu is the source it was taken on.
RECORDED_GEMM1_TRAFFIC = {"gemm_cu_sha1": "1bc7ea395d3f", "bytes": 3842182485}


def recorded_traffic(kernel_hash: str):
    """DRAM bytes of one GEMM1-shape launch from the recorded capture, if it was taken on this
    exact kernel source (else None)."""
    if RECORDED_GEMM1_TRAFFIC["gemm_cu_sha1"] == kernel_hash:
        return RECORDED_GEMM1_TRAFFIC["bytes"]
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
    # bf16 input (the MoE path), then the same values as fp32 input (the input type of the pages'
    # bandwidth microbenchmark): bytes = input + (codes + 1/32 scale bytes) per output form
    xf = x.float()
    forms = (("row", mx.MX_ROWWISE, 1), ("col", mx.MX_COLWISE, 1), ("row+col", mx.MX_ROWWISE | mx.MX_COLWISE, 2))
    cases = [(name, mode, x, 2 + n * (1 + 1 / 32)) for name, mode, n in forms] + \
            [("f32_" + name, mode, xf, 4 + n * (1 + 1 / 32)) for name, mode, n in forms]
    for name, mode, xin, bpe in cases:
        out = mx.quantize_alloc(xin, mode)
        q = (out["q_row"], out["sf_row"], out["q_col"], out["sf_col"])
        dt = mx.MX_DTYPE_F32 if xin.dtype == torch.float32 else mx.MX_DTYPE_BF16

        def run():
            mx.mxfp8_quantize_ex(xin, dt, mx.MX_SCALE_FLOOR, rows, cols, mode, None, None, 0, out["ld_col"], *q, None)
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
    del x, xf, d
    return res


SKEWED_CFG = dict(T=4096, E=128, k=8, hidden=4096, inter=1536)


def fill_inputs_skewed(step, seed_base=1005):
    """Config-5 routing: top-8 of log p_e + Gumbel noise, p_e ~ rank^-1.2 with 4 experts never
    chosen (synth.zipf_ids); gates = softmax of N(0,1) draws per slot."""
    import torch
    from mxfp8_block_scaled_rowwise_gb300 import synth
    g = synth.generator(seed_base, step.dev)
    step.x.copy_(synth.randn_bf16(step.x.shape, g, device=step.dev))
    step.ids.copy_(synth.zipf_ids(step.T, step.E, step.k, synth.generator(seed_base + 7), device=step.dev))
    step.gate.copy_(torch.softmax(torch.randn(step.T, step.k, generator=g, device=step.dev), dim=1))
    step.w1.copy_(synth.randn_bf16(step.w1.shape, g, device=step.dev))
    step.w2.copy_(synth.randn_bf16(step.w2.shape, g, device=step.dev))
    step.dout.copy_(synth.randn_bf16(step.dout.shape, g, std=1e-2, device=step.dev))


def gemm_alg_bytes(step, P):
    """Algorithmic DRAM bytes of each GEMM launch of a step: operand codes, scales (B operands
    in the four-copy layout), outputs.  P = poff[E], the padded positions actually used."""
    R, E, H, I, I2 = step.R, step.E, step.H, step.I, step.I2

    def rows_gemm(k, n):     # A [R x k] rowwise, B [E*n x k] (or its columnwise form), C bf16 [R x n]
        return R * k + P * k // 32 + E * n * k + 4 * E * n * k // 32 + 2 * R * n

    def wgrad(n, k):         # A [n x P], B [k x P] columnwise, C fp32 [E x n x k]
        return n * P + n * P // 32 + k * P + 4 * k * P // 32 + 4 * E * n * k
    return {"fwd1": rows_gemm(H, I2), "fwd2": rows_gemm(I, H), "dgrad2": rows_gemm(H, I),
            "wgrad2": wgrad(H, I), "dgrad1": rows_gemm(I2, H), "wgrad1": wgrad(I2, H)}


def time_step(torch, step, steps, warmup, world=1, local=0, sample_clocks=False):
    """W untimed steps, then K steps between CUDA events on the current stream (barrier and
    synchronize on both sides); every GEMM launch timed with its own pair of events."""
    import torch.distributed as dist
    gemm_events = []

    def hook(name, fl, fn):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        gemm_events.append((name, fl, a, b))

    for _ in range(warmup):
        step.step()
    torch.cuda.synchronize()
    assert int(step.dev_err.item()) == 0, "device error %d" % int(step.dev_err.item())
    step.gemm_hook = hook
    launches0 = step.launches
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clk = ClockSampler(local) if sample_clocks else None
    if clk:
        clk.__enter__()
    t_start.record()
    for _ in range(steps):
        step.step()
    t_end.record()
    torch.cuda.synchronize()
    if clk:
        clk.__exit__(None, None, None)
    if world > 1:
        dist.barrier()
    step.gemm_hook = None
    assert int(step.dev_err.item()) == 0, "device error %d" % int(step.dev_err.item())
    per_kind = {}
    for name, fl, a, b in gemm_events:
        d = per_kind.setdefault(name, [0.0, 0, 0.0])
        d[0] += a.elapsed_time(b)
        d[1] += 1
        d[2] += fl
    return {"ms_total": t_start.elapsed_time(t_end), "launches": step.launches - launches0,
            "gemm_ms": sum(a.elapsed_time(b) for _, _, a, b in gemm_events),
            "gemm_fl": sum(fl for _, fl, _, _ in gemm_events), "n_gemm": len(gemm_events),
            "per_kind": per_kind, "clocks": clk.summary() if clk else None}


def run_skewed(torch, mx, dev, args, pk):
    """Config 5: the skewed small-group MoE layer step (T=4096, top-8 of E=128 Zipf(1.2) experts
    with 4 never chosen, hidden 4096, intermediate 1536), forward + dgrad + wgrad.  Its GEMMs are
    mixed-bound (the weight-gradient outputs are fp32 [128 x ...]), so each is held to the time
    max(FLOP / FP8 peak, algorithmic bytes / HBM peak)."""
    from mxfp8_block_scaled_rowwise_gb300.layer import MoEFFNStep
    step = MoEFFNStep(device=dev, **SKEWED_CFG)
    fill_inputs_skewed(step)
    torch.cuda.synchronize()
    r = time_step(torch, step, args.steps, args.warmup)
    counts = step.counts.cpu().numpy()
    P = int(step.poff[-1].item())
    fp8_peak = pk["bf16_tflops_sustained"] * FP8_OVER_BF16 * 1e12
    hbm = pk["hbm_gbs"] * 1e9
    nb = gemm_alg_bytes(step, P)
    per, t_roof, t_meas = {}, 0.0, 0.0
    for name, (ms, n, fl) in r["per_kind"].items():
        ms_one, fl_one = ms / n, fl / n
        roof_ms = max(fl_one / fp8_peak, nb[name] / hbm) * 1e3
        per[name] = {"ms": round(ms_one, 4), "TFLOP/s": round(fl_one / (ms_one * 1e-3) / 1e12, 1),
                     "GB/s_alg": round(nb[name] / (ms_one * 1e-3) / 1e9, 1),
                     "bound": "tensor" if fl_one / fp8_peak >= nb[name] / hbm else "hbm",
                     "roofline_ms": round(roof_ms, 4), "frac": round(roof_ms / ms_one, 4)}
        t_roof += roof_ms
        t_meas += ms_one
    ms_step = r["ms_total"] / args.steps
    step_flops = sum(step.gemm_flops().values())
    out = {"workload": "skewed MoE layer fwd+bwd step: T=4096, top-8 of E=128 (Zipf 1.2 popularity, %d experts "
                       "without tokens, %d groups not a multiple of 128 rows), hidden 4096, intermediate 1536"
                       % (int((counts == 0).sum()), int((counts % 128 != 0).sum())),
           "ms_per_step": round(ms_step, 4), "TFLOP/s": round(step_flops / (ms_step * 1e-3) / 1e12, 2),
           "gemm_roofline": {"bound": "max(FLOP/FP8 peak, alg bytes/HBM peak) per GEMM",
                             "roofline_ms": round(t_roof, 4), "measured_ms": round(t_meas, 4),
                             "frac": round(t_roof / t_meas, 4), "per_gemm": per}}
    R, H, I2, E = step.R, step.H, step.I2, step.E
    out["gemm_checks"] = grouped_vs_dense(torch, mx, step)
    out["gemm_checks"]["note"] = ("HBM-bound here: the dense E = 1 GEMM streams one 3072 x 4096 weight, the grouped "
                                  "one 124 of them, so the roofline fractions above are the comparison that holds; "
                                  "forward/dgrad public calls take single-CTA tiles at these group sizes")
    del step
    torch.cuda.empty_cache()
    return out


def time_hbm_kernels(torch, mx, step, pk, reps=10):
    """The step's HBM-bound launches one at a time on the step's own buffers (CUDA events,
    median of `reps`; every operand is larger than L2), with their algorithmic bytes: input
    read once, every output form written once (codes + 1/32 scale bytes per form).  The
    quantizes-on-gather also report the bytes with their input counted once per routed slot
    (what they move through L2: each slot reads its token's row)."""
    T, E, k, H, I, I2, R, pb = step.T, step.E, step.k, step.H, step.I, step.I2, step.R, step.pb
    RC = mx.MX_ROWWISE | mx.MX_COLWISE
    RC_B = RC | mx.MX_ROWWISE_X4 | mx.MX_COLWISE_X4
    RC_CB = RC | mx.MX_COLWISE_X4
    q2 = 2 * (1 + 1 / 32)   # both forms, codes + scales, per element
    dy = step.dy if step.dy is not None else torch.empty(R, H, dtype=torch.bfloat16, device=step.dev)
    runs = {
        "w1_quantize_row_col": (lambda: mx.mxfp8_quantize(step.w1, E * I2, H, RC_B, step.w1_seg, step.w1_seg, E, E * I2,
                                                         step.w1_q, step.w1_sf, step.w1c_q, step.w1c_sf, step.dev_err),
                                E * I2 * H * (2 + q2)),
        "x_quantize_on_gather": (lambda: mx.mxfp8_gather_quantize(step.x, T, H, RC_CB, step.src_row, step.off, step.poff,
                                                                  E, R, pb, step.a1_q, step.a1_sf, step.xpc_q,
                                                                  step.xpc_sf, step.dev_err),
                                 T * H * 2 + R * H * q2),
        "swiglu_fwd_quantize": (lambda: mx.mxfp8_swiglu_quantize(step.out1, R, I, RC_CB, step.off, step.poff, E, pb,
                                                                 step.h_q, step.h_sf, step.hc_q, step.hc_sf,
                                                                 step.dev_err),
                                R * I * (4 + q2)),
        "combine_fwd": (lambda: mx.moe_combine_fwd(step.out2, step.gate, step.dst_of, T, k, H, R, step.out,
                                                   step.dev_err), R * H * 2 + T * H * 2),
        "combine_bwd": (lambda: mx.moe_combine_bwd(step.dout, step.out2, step.gate, step.dst_of, T, k, H, R, dy,
                                                   step.dgate, step.dev_err), T * H * 2 + 2 * R * H * 2),
        "dy_quantize_row_col": (lambda: mx.mxfp8_quantize(dy, R, H, RC, step.off, step.poff, E, pb, step.dy_q, step.dy_sf,
                                                         step.dyc_q, step.dyc_sf, step.dev_err), R * H * (2 + q2)),
        "swiglu_bwd_quantize": (lambda: mx.mxfp8_swiglu_bwd_quantize(step.dh_in, step.out1, R, I, RC, step.off,
                                                                     step.poff, E, pb, step.dh_q, step.dh_sf,
                                                                     step.dhc_q, step.dhc_sf, step.dev_err),
                                R * I * 6 + R * I2 * q2),
    }
    if step.fuse_dy:
        # the step's backward forms dY on the fly: combine backward writes only dgate and each
        # routed row's gate; quantize-on-gather of dOut scales each routed row by its gate
        del runs["combine_bwd"], runs["dy_quantize_row_col"]
        runs["combine_bwd_dgate"] = (
            lambda: mx.moe_combine_bwd_ex(step.dout, step.out2, step.gate, step.dst_of, T, k, H, R, None, step.dgate,
                                          step.gate_rows, step.dev_err), T * H * 2 + R * H * 2 + T * k * 4 + R * 4)
        runs["dy_quantize_on_gather"] = (
            lambda: mx.mxfp8_gather_quantize_ex(step.dout, T, H, RC, step.src_row, step.gate_rows, step.off, step.poff,
                                                E, R, pb, step.dy_q, step.dy_sf, step.dyc_q, step.dyc_sf, step.dev_err),
            T * H * 2 + R * 4 + R * H * q2)
    out = {}
    for name, (fn, nbytes) in runs.items():
        ms = _timed(torch, fn, reps)
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[name] = {"ms": round(ms, 4), "GB/s": round(gbs, 1), "frac": round(gbs / pk["hbm_gbs"], 4)}
        if name in ("x_quantize_on_gather", "dy_quantize_on_gather"):
            out[name]["GB/s_input_per_slot"] = round(R * H * (2 + q2) / (ms * 1e-3) / 1e9, 1)
    torch.cuda.synchronize()
    assert int(step.dev_err.item()) == 0
    return out


def time_tiny(torch, mx, dev, reps=50):
    """Config 1 (T=512, K=256, E=4 top-1, W [4 x 512 x 256]): rowwise quantize of x and W,
    permutation (one launch at this size) with the fp8 row gather, grouped GEMM forward; median of
    `reps` timed runs, eager and replayed from one CUDA graph."""
    from mxfp8_block_scaled_rowwise_gb300 import synth
    d = synth.tiny(device=dev)
    T, K, E, N = d["T"], d["K"], d["E"], d["N"]
    err = mx.new_dev_err(dev)
    qx = mx.quantize_alloc(d["x"], mx.MX_ROWWISE, dev_err=err)
    qw = mx.quantize_alloc(d["w"].view(E * N, K), mx.MX_ROWWISE | mx.MX_ROWWISE_X4, dev_err=err)
    pm = mx.permute_alloc(d["ids"], E, qx["q_row"], qx["sf_row"], dev_err=err)
    C = torch.empty(T, N, dtype=torch.bfloat16, device=dev)

    def run():
        mx.mxfp8_quantize(d["x"], T, K, mx.MX_ROWWISE, None, None, 0, 0, qx["q_row"], qx["sf_row"], None, None, err)
        mx.mxfp8_quantize(d["w"].view(E * N, K), E * N, K, mx.MX_ROWWISE | mx.MX_ROWWISE_X4, None, None, 0, 0,
                          qw["q_row"], qw["sf_row"], None, None, err)
        mx.moe_permute(d["ids"], T, 1, E, pm["counts"], pm["off"], pm["poff"], pm["src_row"], pm["dst_of"],
                       qx["q_row"], qx["sf_row"], K, pm["q"], pm["sf"], pm["ws"], pm["ws"].numel(), err)
        mx.grouped_gemm_mxfp8_fwd(pm["q"], pm["sf"], qw["q_row"], qw["sf_row"], pm["off"], pm["poff"], E, T, N, K, C,
                                  err)
    for _ in range(5):
        run()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, b in ev:
        a.record()
        run()
        b.record()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ms = statistics.median(a.elapsed_time(b) for a, b in ev)
    c_eager = C.clone()
    # the same seven launches captured once in a CUDA graph and replayed (no per-launch host work
    # and no launch gaps between the short kernels)
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        run()
    torch.cuda.current_stream(dev).wait_stream(s)
    for _ in range(5):
        graph.replay()
    torch.cuda.synchronize()
    for a, b in ev:
        a.record()
        graph.replay()
        b.record()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(C.view(torch.int16), c_eager.view(torch.int16)), "graph replay differs from the eager run"
    ms_graph = statistics.median(a.elapsed_time(b) for a, b in ev)
    return {"workload": "tiny forward: T=512, K=256, E=4 top-1, N=512 (quantize x and W, permute + gather, "
                        "grouped GEMM; 5 launches)", "ms": round(ms, 4), "ms_graph": round(ms_graph, 4),
            "note": "launch-latency bound: 2*512*512*256 = 0.13 GFLOP; ms_graph: the same launches replayed "
                    "from one CUDA graph"}


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
        # one GEMM shape of the MoE FFN step alone on seeded synthetic E4M3 codes with unit
        # scales, for profiler captures: GEMM1 (131072 routed rows over 32 experts, N=4096,
        # K=7168; about 3 GB on the device) or wgrad1 (dW1 [32 x 4096 x 7168] fp32 over 4096
        # tokens per expert; about 5 GB); --raster-group G > 0 picks the tile order through the
        # internal test entry (G = 1: N tiles fastest), 0 = the public call
        g = torch.Generator(device=dev)
        g.manual_seed(17)
        E, T_e, N, K = CFG["E"], CFG["T"] * CFG["k"] // CFG["E"], 2 * CFG["inter"], CFG["hidden"]
        R = E * T_e

        def codes(r, c):
            t = torch.randint(0, 256, (r, c), dtype=torch.uint8, device=dev, generator=g)
            t[(t & 0x7F) == 0x7F] = 0x38   # no NaN codes
            return t
        off = torch.arange(0, (E + 1) * T_e, T_e, dtype=torch.int32, device=dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        G = args.raster_group
        # B codes row-major, or in 128 x 128 blocks of 16 KiB (random codes: the layout changes
        # only where the bytes sit, not the work)
        b_flags = mx.MX_GEMM_B_BLOCKED if args.gemm_b_layout == "blocked" else 0
        if args.gemm_shape == "skewed_fwd1":
            # GEMM1 of the skewed step: 32768 routed rows over 128 Zipf-popular experts (4 empty),
            # N = 3072, K = 4096; the 1.6 GB of W1 codes are streamed once (about 2 GB on the device)
            from mxfp8_block_scaled_rowwise_gb300 import synth
            c = SKEWED_CFG
            E, N, K = c["E"], 2 * c["inter"], c["hidden"]
            ids = synth.zipf_ids(c["T"], E, c["k"], synth.generator(1012))
            counts = torch.bincount(ids.reshape(-1), minlength=E)
            off = torch.zeros(E + 1, dtype=torch.int32)
            off[1:] = torch.cumsum(counts, 0)
            poff = torch.zeros(E + 1, dtype=torch.int32)
            poff[1:] = torch.cumsum((counts + 127) // 128 * 128, 0)
            R = int(off[-1])
            off, poff = off.to(dev), poff.to(dev)
            pb = mx.mx_padded_rows_bound(R, E)
            A, B = codes(R, K), codes(E * N, K)
            SFA = torch.full((mx.mx_sf_bytes(pb, K // 32),), 127, dtype=torch.uint8, device=dev)
            SFB = torch.full((mx.mx_sf_bytes_x4(E * N, K // 32),), 127, dtype=torch.uint8, device=dev)
            C = torch.empty(R, N, dtype=torch.bfloat16, device=dev)
            run = lambda: mx.grouped_gemm_mxfp8_fwd_ex(A, SFA, B, SFB, off, poff, E, R, N, K, C, b_flags, err)
        elif args.gemm_shape in ("fwd2", "dgrad2", "dgrad1", "wgrad2"):
            # the other GEMMs of the MoE FFN step at their own shapes, through the public calls
            # (the tile order and the B layout of the step's launches)
            H, I = CFG["hidden"], CFG["inter"]
            kind, N, K = {"fwd2": ("fwd", H, I), "dgrad2": ("dgrad", I, H), "dgrad1": ("dgrad", H, 2 * I),
                          "wgrad2": ("wgrad", H, I)}[args.gemm_shape]
            if G != 0 or b_flags != 0:
                raise SystemExit("--raster-group and --gemm-b-layout apply to fwd1 / wgrad1 only")
            if kind == "wgrad":
                A, B = codes(N, R), codes(K, R)
                SFA = torch.full((mx.mx_sf_bytes(N, R // 32),), 127, dtype=torch.uint8, device=dev)
                SFB = torch.full((mx.mx_sf_bytes_x4(K, R // 32),), 127, dtype=torch.uint8, device=dev)
                C = torch.empty(E, N, K, dtype=torch.float32, device=dev)
                run = lambda: mx.grouped_gemm_mxfp8_wgrad(A, SFA, B, SFB, off, off, E, N, K, R, C, err)
            else:
                pb = mx.mx_padded_rows_bound(R, E)
                A = codes(R, K)
                SFA = torch.full((mx.mx_sf_bytes(pb, K // 32),), 127, dtype=torch.uint8, device=dev)
                if kind == "fwd":   # B: the stacked weights [E*N x K], rowwise
                    B = codes(E * N, K)
                    SFB = torch.full((mx.mx_sf_bytes_x4(E * N, K // 32),), 127, dtype=torch.uint8, device=dev)
                else:               # B: their columnwise quantization [N x E*K]
                    B = codes(N, E * K)
                    SFB = torch.full((mx.mx_sf_bytes_x4(N, E * K // 32),), 127, dtype=torch.uint8, device=dev)
                C = torch.empty(R, N, dtype=torch.bfloat16, device=dev)
                fn = mx.grouped_gemm_mxfp8_fwd if kind == "fwd" else mx.grouped_gemm_mxfp8_dgrad
                run = lambda: fn(A, SFA, B, SFB, off, off, E, R, N, K, C, err)
        elif args.gemm_shape == "fwd1":
            A, B = codes(R, K), codes(E * N, K)
            pb = mx.mx_padded_rows_bound(R, E)
            SFA = torch.full((mx.mx_sf_bytes(pb, K // 32),), 127, dtype=torch.uint8, device=dev)
            SFB = torch.full((mx.mx_sf_bytes_x4(E * N, K // 32),), 127, dtype=torch.uint8, device=dev)
            C = torch.empty(R, N, dtype=torch.bfloat16, device=dev)
            if G == 0:
                run = lambda: mx.grouped_gemm_mxfp8_fwd_ex(A, SFA, B, SFB, off, off, E, R, N, K, C, b_flags, err)
            else:
                run = lambda: mx.testing_grouped_gemm(mx.MX_TESTING_FWD, A, SFA, B, SFB, off, off, E, R, N, K, 0, C,
                                                      err, flags=b_flags, raster_group=G)
        else:
            A, B = codes(N, R), codes(K, R)
            SFA = torch.full((mx.mx_sf_bytes(N, R // 32),), 127, dtype=torch.uint8, device=dev)
            SFB = torch.full((mx.mx_sf_bytes_x4(K, R // 32),), 127, dtype=torch.uint8, device=dev)
            C = torch.empty(E, N, K, dtype=torch.float32, device=dev)
            if G == 0:
                run = lambda: mx.grouped_gemm_mxfp8_wgrad_ex(A, SFA, B, SFB, off, off, E, N, K, R, C, b_flags, err)
            else:
                run = lambda: mx.testing_grouped_gemm(mx.MX_TESTING_WGRAD, A, SFA, B, SFB, off, off, E, 0, N, K, R, C,
                                                      err, flags=b_flags, raster_group=G)
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
            print(json.dumps({"gemm": args.gemm_shape, "b_layout": args.gemm_b_layout, "raster_group": G,
                              "ms": round(ms, 4),
                              "TFLOP/s": round(2.0 * R * N * K / (ms * 1e-3) / 1e12, 1)}), flush=True)
        return
    if args.only == "swiglu":
        # the fused SwiGLU kernels alone at the MoE FFN shape (131072 routed rows, intermediate 2048;
        # about 3 GB on the device), for profiler captures: forward then backward, 5 times each
        from mxfp8_block_scaled_rowwise_gb300 import synth
        R, I, E = CFG["T"] * CFG["k"], CFG["inter"], CFG["E"]
        g = synth.generator(23, dev)
        a = synth.randn_bf16((R, 2 * I), g, device=dev)
        dh = synth.randn_bf16((R, I), g, std=1e-2, device=dev)
        T_e = R // E
        off = torch.arange(0, (E + 1) * T_e, T_e, dtype=torch.int32, device=dev)
        RC = mx.MX_ROWWISE | mx.MX_COLWISE
        res = {}
        for bwd in (False, True):
            cols = 2 * I if bwd else I
            q_row = torch.empty(R, cols, dtype=torch.uint8, device=dev)
            sf_row = torch.empty(mx.mx_sf_bytes(R, cols // 32), dtype=torch.uint8, device=dev)
            q_col = torch.empty(cols, R, dtype=torch.uint8, device=dev)
            sf_col = torch.empty(mx.mx_sf_bytes(cols, R // 32), dtype=torch.uint8, device=dev)
            err = torch.zeros(1, dtype=torch.int32, device=dev)
            if bwd:
                fn = lambda: mx.mxfp8_swiglu_bwd_quantize(dh, a, R, I, RC, off, off, E, R, q_row, sf_row, q_col, sf_col,
                                                          err)
            else:
                fn = lambda: mx.mxfp8_swiglu_quantize(a, R, I, RC, off, off, E, R, q_row, sf_row, q_col, sf_col, err)
            ms = _timed(torch, fn, 5, )
            assert int(err.item()) == 0
            nbytes = R * I * 6 + R * 2 * I * 2 * (1 + 1 / 32) if bwd else R * I * (4 + 2 * (1 + 1 / 32))
            res["bwd" if bwd else "fwd"] = {"ms": round(ms, 4), "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1)}
        if rank == 0:
            print(json.dumps({"swiglu": res}), flush=True)
        return
    if args.only == "gather":
        # quantize-on-gather of x at the MoE FFN shape alone (16384 tokens x 7168, top-8 of 32
        # experts, row + col; about 2.5 GB on the device), for profiler captures: 3 + 10 launches
        from mxfp8_block_scaled_rowwise_gb300 import synth
        T, H, E, k = CFG["T"], CFG["hidden"], CFG["E"], CFG["k"]
        g = synth.generator(1003, dev)
        x = synth.randn_bf16((T, H), g, device=dev)
        ids = synth.topk_ids(torch.randn(T, E, generator=g, device=dev), k)
        err = mx.new_dev_err(dev)
        pm = mx.permute_alloc(ids, E, dev_err=err)
        R = T * k
        pb = mx.mx_padded_rows_bound(R, E)
        q_row = torch.empty(R, H, dtype=torch.uint8, device=dev)
        sf_row = torch.empty(mx.mx_sf_bytes(pb, H // 32), dtype=torch.uint8, device=dev)
        q_col = torch.empty(H, pb, dtype=torch.uint8, device=dev)
        sf_col = torch.empty(mx.mx_sf_bytes_x4(H, pb // 32), dtype=torch.uint8, device=dev)
        mode = mx.MX_ROWWISE | mx.MX_COLWISE | mx.MX_COLWISE_X4
        ms = _timed(torch, lambda: mx.mxfp8_gather_quantize(x, T, H, mode, pm["src_row"], pm["off"], pm["poff"], E,
                                                            R, pb, q_row, sf_row, q_col, sf_col, err))
        assert int(err.item()) == 0
        nbytes = T * H * 2 + R * H * 2 * (1 + 1 / 32)
        if rank == 0:
            print(json.dumps({"gather": {"ms": round(ms, 4), "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1),
                                         "GB/s_x_per_slot": round((nbytes + (R - T) * H * 2) / (ms * 1e-3) / 1e9, 1)}}),
                  flush=True)
        return
    if args.only == "combine":
        # combine forward and the dgate-only combine backward at the MoE FFN shape alone (16384
        # tokens x 7168, top-8 of 32 experts; about 2.7 GB on the device), for profiler captures:
        # 3 + 10 launches of each, forward first
        from mxfp8_block_scaled_rowwise_gb300 import synth
        T, H, E, k = CFG["T"], CFG["hidden"], CFG["E"], CFG["k"]
        R = T * k
        g = synth.generator(1004, dev)
        ids = synth.topk_ids(torch.randn(T, E, generator=g, device=dev), k)
        err = mx.new_dev_err(dev)
        pm = mx.permute_alloc(ids, E, dev_err=err)
        Y = synth.randn_bf16((R, H), g, device=dev)
        dout = synth.randn_bf16((T, H), g, std=1e-2, device=dev)
        gate = torch.softmax(torch.randn(T, k, generator=g, device=dev), dim=1)
        out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        dgate = torch.empty(T, k, dtype=torch.float32, device=dev)
        gate_rows = torch.empty(R, dtype=torch.float32, device=dev)
        fwd_ms = _timed(torch, lambda: mx.moe_combine_fwd(Y, gate, pm["dst_of"], T, k, H, R, out, err))
        bwd_ms = _timed(torch, lambda: mx.moe_combine_bwd_ex(dout, Y, gate, pm["dst_of"], T, k, H, R, None, dgate,
                                                             gate_rows, err))
        assert int(err.item()) == 0
        fwd_b, bwd_b = R * H * 2 + T * H * 2, T * H * 2 + R * H * 2 + T * k * 4 + R * 4
        if rank == 0:
            print(json.dumps({"combine": {
                "fwd": {"ms": round(fwd_ms, 4), "GB/s": round(fwd_b / (fwd_ms * 1e-3) / 1e9, 1)},
                "bwd_dgate": {"ms": round(bwd_ms, 4), "GB/s": round(bwd_b / (bwd_ms * 1e-3) / 1e9, 1)}}}),
                  flush=True)
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
    hbm = None
    if rank == 0:
        # the HBM-bound launches one at a time, after one untimed step and before the long GEMM runs
        step.step()
        with ClockSampler(local) as hclk:
            hbm = time_hbm_kernels(torch, mx, step, pk)
        hbm["clocks"] = hclk.summary()
    r = time_step(torch, step, args.steps, args.warmup, world, local, sample_clocks=True)
    launches = r["launches"]
    ms_total = max_over_ranks(r["ms_total"], dev)
    ms_step = ms_total / args.steps
    gemm_ms, gemm_fl, per_kind = r["gemm_ms"], r["gemm_fl"], r["per_kind"]
    clocks = r["clocks"]
    value = job_throughput(step_flops, world, ms_step * 1e-3) / 1e12
    alg_bytes = gemm_alg_bytes(step, int(step.poff[-1].item()))

    checks = gemm_checks(torch, mx, step) if rank == 0 else None
    assert int(step.dev_err.item()) == 0

    # e2e: same step through the public API with pinned host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(torch, step, args, step_flops, world)

    quant = time_quantizer(torch, mx, dev) if (rank == 0 and args.shape == "ffn") else {}
    tiny = time_tiny(torch, mx, dev) if (rank == 0 and args.shape == "ffn" and not args.no_tiny) else None
    skewed = None
    if rank == 0 and args.shape == "ffn" and not args.no_skewed:
        del step
        torch.cuda.empty_cache()
        step = None
        skewed = run_skewed(torch, mx, dev, args, pk)
    cpu = cpu_baseline(args) if (rank == 0 and world == 1 and not args.no_cpu_baseline) else None

    if rank == 0:
        fp8_peak = pk["bf16_tflops_sustained"] * FP8_OVER_BF16
        achieved = gemm_fl / (gemm_ms * 1e-3) / 1e12
        n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
        kh = gemm_source_hash()
        traffic = recorded_traffic(kh)
        n_launch = r["n_gemm"]
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
                         "traffic_scope": "DRAM read + write bytes of one GEMM1 launch (131072 x 4096 x 7168), "
                                          "one-kernel ncu capture; its algorithmic bytes: %d" % alg_bytes["fwd1"],
                         "frac_of_nominal": round(achieved / NOMINAL["fp8_tflops"], 4),
                         "frac_of_tensor_pipe": (round(achieved / (TENSOR_PIPE_FP8_FLOP_PER_CLK_SM * n_sm *
                                                                   clocks["sm_mhz"] * 1e6 / 1e12), 4)
                                                 if clocks and clocks.get("sm_mhz") else None),
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
                              "f32_*: the same values as fp32 input (the pages' microbenchmark input type), 4 bytes in; "
                              "peak = %s HBM copy %.1f GB/s" % (pk["source"], pk["hbm_gbs"]),
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clocks,
            "hbm_kernels": hbm,
            "hbm_kernels_note": "the step's HBM-bound launches timed one at a time on the step's buffers; bytes = "
                                "input read once + every output form written once; peak = %s HBM copy %.1f GB/s" % (
                                    pk["source"], pk["hbm_gbs"]),
            "skewed": skewed,
            "tiny": tiny,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_e2e(torch, step, args, step_flops, world):
    """The step through the public API with host buffers.  Per step: H2D of the layer's inputs
    (routing ids, gates and x, then the output gradient) from pinned memory, the step, D2H of
    the layer's outputs (forward output and input gradient, token order) into pinned memory.
    Copies run on their own streams and overlap the neighbouring steps' compute (double-buffered
    device inputs and outputs): the weights are quantized while the inputs arrive, the rest of the
    forward waits only for ids, gates and x, the backward for the output gradient, and the forward
    output leaves while the backward runs.  The timed region
    spans the first H2D to the last D2H."""
    in_names = ["ids", "gate", "x", "dout"]     # in copy order: what the forward needs first
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
    fwd_in_ready = [ev(), ev()]
    bwd_in_ready = [ev(), ev()]
    in_free = [ev(), ev()]
    fwd_done = [ev(), ev()]
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
                    if nm == "dout":
                        fwd_in_ready[sl].record(s_h2d)
                    slots_in[sl][nm].copy_(h_in[nm], non_blocking=True)
                bwd_in_ready[sl].record(s_h2d)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(out_free[sl])
                for nm in in_names:
                    setattr(step, nm, slots_in[sl][nm])
                for nm in out_names:
                    setattr(step, nm, slots_out[sl][nm])
                step.forward(before_inputs=lambda: s_cmp.wait_event(fwd_in_ready[sl]))
                fwd_done[sl].record(s_cmp)
                s_cmp.wait_event(bwd_in_ready[sl])
                step.backward()
                in_free[sl].record(s_cmp)
                done[sl].record(s_cmp)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(fwd_done[sl])
                h_out[sl]["out"].copy_(slots_out[sl]["out"], non_blocking=True)
                s_d2h.wait_event(done[sl])
                h_out[sl]["dx"].copy_(slots_out[sl]["dx"], non_blocking=True)
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
            "overlap": "H2D, compute and D2H on separate streams, double-buffered device inputs/outputs; the "
                       "weights quantized while ids, gates and x arrive, the forward output leaves during the backward"}


def _timed(torch, fn, reps=10):
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


def grouped_vs_dense(torch, mx, step):
    """Target checks on a step's GEMM1 shape (R routed rows x N=2I x K=H): the grouped GEMM vs an
    equal-FLOP dense GEMM (same kernel, E = 1), and 2-CTA pairs vs single-CTA tiles (chosen
    through the internal test entry)."""
    R, H, I2, E = step.R, step.H, step.I2, step.E
    dense_off = torch.tensor([0, R], dtype=torch.int32, device=step.dev)
    grouped = lambda: mx.grouped_gemm_mxfp8_fwd(step.a1_q, step.a1_sf, step.w1_q, step.w1_sf, step.off, step.poff, E,
                                                 R, I2, H, step.out1, step.dev_err)
    dense = lambda: mx.grouped_gemm_mxfp8_fwd(step.a1_q, step.a1_sf, step.w1_q, step.w1_sf, dense_off, dense_off, 1,
                                               R, I2, H, step.out1, step.dev_err)
    single = lambda: mx.testing_grouped_gemm(mx.MX_TESTING_FWD, step.a1_q, step.a1_sf, step.w1_q, step.w1_sf,
                                             step.off, step.poff, E, R, I2, H, 0, step.out1, step.dev_err,
                                             ctas_per_mma=1)
    fl = 2.0 * R * I2 * H
    t_g, t_d, t_1 = _timed(torch, grouped), _timed(torch, dense), _timed(torch, single)
    torch.cuda.synchronize()
    assert int(step.dev_err.item()) == 0
    tf = lambda ms: round(fl / (ms * 1e-3) / 1e12, 1)
    return {"shape": "GEMM1: %d routed rows over %d experts, N=%d, K=%d" % (R, E, I2, H),
            "grouped_tflops": tf(t_g), "dense_e1_tflops": tf(t_d), "grouped_over_dense": round(t_d / t_g, 4),
            "single_cta_tflops": tf(t_1), "two_cta_speedup": round(t_1 / t_g, 4)}


def gemm_checks(torch, mx, step):
    out = grouped_vs_dense(torch, mx, step)
    fl = 2.0 * step.R * step.I2 * step.H
    out["library_mxfp8"] = library_mxfp8(torch, step, lambda fn: _timed(torch, fn), fl,
                                         lambda ms: round(fl / (ms * 1e-3) / 1e12, 1))
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
def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:   # pragma: no cover
        return os.cpu_count() or 1


def cpu_baseline(args, budget_s: float = 12.0):
    """Time the CPU oracle (as it stands) on a bounded sample of the step's work and extrapolate
    the step time from the measured per-unit rates: once on one host thread, once on every host
    thread the process may use (independent oracle calls on separate threads; the C oracle runs
    without the Python lock).  The oracle's arithmetic is the same single-threaded code either way."""
    import numpy as np
    import torch
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    from mxfp8_block_scaled_rowwise_gb300 import synth
    oracle.build()
    T, E, k, H, I = CFG["T"], CFG["E"], CFG["k"], CFG["hidden"], CFG["inter"]
    I2, R = 2 * I, T * k
    g = synth.generator(7)
    t0 = time.perf_counter()
    nthr = host_threads()

    def rate(fn, units, seconds, threads):
        """units per second of fn on `threads` threads, each repeating it for `seconds`"""
        counts = [0] * threads
        t_start = time.perf_counter()
        stop = t_start + seconds

        def worker(i):
            while True:
                fn()
                counts[i] += 1
                if time.perf_counter() > stop:
                    return
        if threads == 1:
            worker(0)
        else:
            with ThreadPoolExecutor(threads) as ex:
                list(ex.map(worker, range(threads)))
        return sum(counts) * units / (time.perf_counter() - t_start), sum(counts)

    xb = synth.bf16_bits(synth.randn_bf16((1024, H), g))
    ids = synth.topk_ids(torch.randn(T, E, generator=g), k).numpy()
    qa, sa = oracle.quantize_rowwise(synth.bf16_bits(synth.randn_bf16((8, H), g)))
    qb, sb = oracle.quantize_rowwise(synth.bf16_bits(synth.randn_bf16((512, H), g)))
    # element counts of every quantization in the step, routed slots, GEMM FLOPs
    row_elems = E * I2 * H + E * H * I + T * H + R * I + R * H + R * I2
    col_elems = E * I2 * H + E * H * I + R * I + R * H + R * I2 + R * H
    step_flops = 3 * 2 * R * (I2 * H + H * I)
    legs = [("quant_row_elem_per_s", lambda: oracle.quantize_rowwise(xb), xb.size, 0.2),
            ("quant_col_elem_per_s", lambda: oracle.quantize_colwise_seg(xb, [0, 1024], [0, 1024], 1024), xb.size, 0.2),
            ("permute_slots_per_s", lambda: oracle.permute(ids, E), ids.size, 0.1),
            ("gemm_flop_per_s", lambda: oracle.gemm_nt(qa, sa, qb, sb), 2 * 8 * 512 * H, 0.5)]
    res = {}
    for threads in sorted({1, nthr}):
        rates, reps = {}, {}
        for name, fn, units, share in legs:
            rates[name], reps[name] = rate(fn, units, share * budget_s / 2, threads)
        t_step = (row_elems / rates["quant_row_elem_per_s"] + col_elems / rates["quant_col_elem_per_s"]
                  + R / rates["permute_slots_per_s"] + step_flops / rates["gemm_flop_per_s"])
        res[threads] = {"value": step_flops / t_step / 1e12, "extrapolated_step_s": round(t_step, 1),
                        "rates": {k_: round(v) for k_, v in rates.items()}, "reps": reps}
    best = res[nthr]
    return {"value": best["value"], "unit": "TFLOP/s", "cores": nthr, "host_cores": os.cpu_count(), "kind": "oracle",
            "sample": "C oracle on %d host threads (independent calls per thread) and on 1: rowwise and colwise "
                      "quantize of 1024x7168, the full top-8 permutation of 16384 tokens, fp64 GEMM of 8x512x7168, "
                      "each repeated for its share of the time; step time extrapolated from these rates (%.0f s "
                      "measured)" % (nthr, time.perf_counter() - t0),
            "extrapolated_step_s": best["extrapolated_step_s"], "extrapolated": True, "rates": best["rates"],
            "one_thread": {"value": res[1]["value"], "extrapolated_step_s": res[1]["extrapolated_step_s"],
                           "rates": res[1]["rates"]}}


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
        "cpu_baseline": {"kind": "oracle", "cores": res["cores"], "sample": res["sample"], "value": value,
                         "extrapolated": True, "one_thread": res["one_thread"]},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-skewed", action="store_true", help="skip the skewed 128-expert step (Zipf routing, experts of about 256 rows)")
    ap.add_argument("--only", default=None, choices=["quantizer", "gemm", "swiglu", "gather", "combine"],
                    help="run one kernel family alone at its MoE FFN shape (a few GB on the device; small cases "
                         "for profiler captures): the 16384 x 7168 quantizer, one grouped GEMM (--gemm-shape), "
                         "the SwiGLU kernels, the quantize-on-gather of x, or the combine kernels")
    ap.add_argument("--gemm-shape", default="fwd1",
                    choices=["fwd1", "fwd2", "dgrad2", "wgrad2", "dgrad1", "wgrad1", "skewed_fwd1"],
                    help="with --only gemm: one of the six GEMMs of the MoE FFN step at its own shape "
                         "(random codes, unit scales), or GEMM1 of the skewed 128-expert step")
    ap.add_argument("--gemm-b-layout", default="row", choices=["row", "blocked"],
                    help="with --only gemm: B codes row-major or in 128 x 128 blocks (MX_GEMM_B_BLOCKED)")
    ap.add_argument("--raster-group", type=int, default=0,
                    help="with --only gemm: tile order inside an expert (groups of G M tiles, M fastest; 0: default)")
    ap.add_argument("--no-tiny", action="store_true", help="skip the tiny forward timing (256 tokens, 8 experts)")
    ap.add_argument("--shape", default="ffn", choices=["ffn", "small"],
                    help="ffn: the MoE FFN workload (default); small: a reduced case for profiler captures")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
