"""Benchmark of the block-scaled low-precision linear layer on one GB300 (per rank).

One step = one pass of the layer's hot path over one batch of the dense
Qwen3-4B-shaped MLP projection (tokens M = 8192, hidden 2560, intermediate
9728), forward and backward:
    dual (row + transposed) 1x128 quantisation of X [8192, 2560] and of
    dY [8192, 9728], dual 128x128 quantisation of W [9728, 2560], then the
    fprop, dgrad and wgrad block-scaled FP8 GEMMs (3 x 408.02 GFLOP).
value = GEMM FLOPs of the step / step time (TFLOPS), inputs resident in HBM.
The same run measures, as separate sub-results, the quantise sweep on a
BF16 [8192, 4096] tensor (GB/s per granularity), the MoE grouped MXFP8 GEMM
(Qwen3-30B-A3B shapes) and the NVFP4 linear (Qwen2.5-32B shapes), each
against the roofline, plus the CPU oracle on a bounded sample of the step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

For N > 1, launch one rank per GPU with torchrun; every rank
runs its own batch (weak scaling, no collective on the data path) and rank 0
prints one JSON line.
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
sys.path.insert(0, ROOT)

M3, H3, I3 = 8192, 2560, 9728
GEMM_FLOP = 2 * M3 * H3 * I3                    # one of fprop / dgrad / wgrad
STEP_FLOP = 3 * GEMM_FLOP
FP8_PER_BF16 = 2.0                              # nominal dense ratio (4.5 / 2.25 PFLOP/s)
FP4_PER_BF16 = 6.0                              # nominal dense ratio (13.5 / 2.25 PFLOP/s)
METRIC = "block-scaled FP8 GEMM TFLOPS and quantize GB/s at 1 GB300 (% of roofline)"
# DRAM bytes (read + write) per blockwise-GEMM launch of the step, averaged
# over fprop, dgrad and wgrad, from one ncu capture of the step
# (ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum -k regex:gemm_blockwise
# on `bench.py --no-extras`), together with the SHA-256 (first 16 hex digits)
# of the kernel source it was taken on: once that source changes the figure
# no longer describes the kernel and the bench reports null.
GEMM_TRAFFIC = {"bytes": 140599296, "source_sha16": "08fbfd2a62900f2a"}
L2_FLUSH_BYTES = 512 << 20
TIMED_CALLS = 50                                # sub-benchmarks: median of this many calls


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extras", action="store_true", help="skip the sub-benchmarks")
    ap.add_argument("--sequential-gemms", action="store_true",
                    help="run the step's three GEMMs one after another on the step's stream")
    ap.add_argument("--kernel", default=None,
                    choices=["fprop", "dgrad", "wgrad", "fprop_pow2", "dgrad_pow2", "wgrad_pow2", "quant_1x128", "quant_dual_1x128", "quant_mxfp8",
                             "quant_per_tensor", "quant_nvfp4", "quant_nvfp4_row_4over6", "dequant_1x128",
                             "moe_gate_up", "moe_gather_quant",
                             "moe_swiglu_quant", "moe_quant_then_gather", "moe_layer", "nvfp4",
                             "mma_peak_e4m3", "mma_peak_mxfp8", "mma_peak_nvfp4"],
                    help="run only this piece of the path W+K times (for profiler captures); prints its time")
    return ap.parse_args()


def peaks():
    p = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            m = json.load(f)
        p.update({k: float(m[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained") if k in m})
        p["source"] = "measured"
    return p


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while active."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


# ---------------------------------------------------------------- inputs
def device_inputs(torch, seed: int, dev):
    """Seeded synthetic BF16 operands drawn on the device (same recipe as the
    tests' generators: N(0,1) activations with 1% outliers x50, N(0,0.02)
    weights), so that multi-GB workloads are built in milliseconds."""
    g = torch.Generator(device=dev)
    g.manual_seed(seed)

    def act(shape, frac, mult):
        z = torch.randn(shape, generator=g, device=dev, dtype=torch.float32)
        u = torch.rand(shape, generator=g, device=dev, dtype=torch.float32)
        return torch.where(u < frac, z * mult, z).to(torch.bfloat16)

    def wt(shape, std=0.02):
        return (torch.randn(shape, generator=g, device=dev, dtype=torch.float32) * std).to(torch.bfloat16)

    return act, wt


class DenseStep:
    """Buffers and launches of one fwd+bwd step of the blockwise FP8 linear.

    recipe "fp32": 1x128 / 128x128 FP32 scales, promoted in the GEMM epilogue;
    recipe "pow2": the same blocks with power-of-two (UE8M0) scales applied by
    the tensor core's block-scale path."""

    def __init__(self, torch, fp, dev, seed, recipe="fp32"):
        self.g_tok, self.g_blk = ("1x128", "128x128") if recipe == "fp32" else ("1x128_pow2", "128x128_pow2")
        act, wt = device_inputs(torch, seed, dev)
        self.torch, self.fp = torch, fp
        self.x = act((M3, H3), 0.01, 50.0)
        self.w = wt((I3, H3))
        self.dy = act((M3, I3), 0.01, 50.0)
        e = lambda *s, dt=torch.uint8: torch.empty(s, dtype=dt, device=dev)  # noqa: E731
        f32 = torch.float32 if recipe == "fp32" else torch.uint8
        self.qx, self.sx, self.qxt, self.sxt = e(M3, H3), e(M3, H3 // 128, dt=f32), e(H3, M3), e(H3, M3 // 128, dt=f32)
        self.qw, self.sw = e(I3, H3), e(I3 // 128, H3 // 128, dt=f32)
        self.qwt, self.swt = e(H3, I3), e(H3 // 128, I3 // 128, dt=f32)
        self.qdy, self.sdy, self.qdyt, self.sdyt = (e(M3, I3), e(M3, I3 // 128, dt=f32), e(I3, M3),
                                                    e(I3, M3 // 128, dt=f32))
        bf = torch.bfloat16
        self.y, self.dx, self.dw = e(M3, I3, dt=bf), e(M3, H3, dt=bf), e(I3, H3, dt=bf)
        self.ws = fp.workspace(dev)
        # The three GEMMs are independent once X, W and dY are quantised: with
        # the GEMM kernels' dynamic tile order they run concurrently, each on a
        # stream (and workspace) of its own, wgrad (longest tiles) first and
        # fprop (shortest) last, so fprop's tiles fill the SMs that dgrad's
        # last wave leaves idle.  Stream priorities keep that order when SMs
        # free up.
        self.concurrent = True
        self.ws_g = [fp.new_workspace(dev) for _ in range(3)]
        self.ws_q = [fp.new_workspace(dev) for _ in range(3)]
        lo, hi = torch.cuda.Stream.priority_range() if hasattr(torch.cuda.Stream, "priority_range") else (0, 0)
        # torch reports (lowest, highest) priority; a smaller number is a higher priority
        prio = [min(lo, hi) if i == 2 else (max(lo, hi) if i == 0 else (lo + hi) // 2) for i in range(3)]
        self.side = [torch.cuda.Stream(dev, priority=prio[i]) for i in range(3)]

    launches_per_step = 6

    def quantize(self):
        """X, W and dY, dual (row-wise and transposed).  With concurrent
        GEMMs the three quantisers also run concurrently, dY (the largest)
        on the highest-priority stream, each with a workspace of its own,
        joined back into the current stream before the GEMMs."""
        fp, torch = self.fp, self.torch
        jobs = ((self.dy, self.g_tok, self.qdyt, self.sdyt, self.qdy, self.sdy),
                (self.x, self.g_tok, self.qxt, self.sxt, self.qx, self.sx),
                (self.w, self.g_blk, self.qwt, self.swt, self.qw, self.sw))
        if not self.concurrent:
            for src, g, qt, st, q, s in jobs:
                fp.fp8_quantize_transposed(src, g, True, q_t=qt, scales_t=st, q=q, scales=s, ws=self.ws)
            return
        cur = torch.cuda.current_stream()
        ready = torch.cuda.Event()
        ready.record(cur)
        done = []
        for i, (src, g, qt, st, q, s) in enumerate(jobs):
            s_ = self.side[2 - i]            # dY on wgrad's (highest-priority) stream
            s_.wait_event(ready)
            with torch.cuda.stream(s_):
                fp.fp8_quantize_transposed(src, g, True, q_t=qt, scales_t=st, q=q, scales=s, ws=self.ws_q[i])
                e_ = torch.cuda.Event()
                e_.record(s_)
            done.append(e_)
        for e_ in done:
            cur.wait_event(e_)

    def ops(self):
        t, b = self.g_tok, self.g_blk
        return ((self.qx, self.sx, t, self.qw, self.sw, b, self.y),
                (self.qdy, self.sdy, t, self.qwt, self.swt, b, self.dx),
                (self.qdyt, self.sdyt, t, self.qxt, self.sxt, t, self.dw))

    def gemms(self, events=None):
        """fprop, dgrad, wgrad one after another on the current stream;
        events[i] (a start/end pair) brackets GEMM i."""
        for i, (a, sa, ga, b, sb, gb, out) in enumerate(self.ops()):
            if events is not None:
                events[i][0].record()
            self.fp.fp8_block_gemm(a, sa, ga, b, sb, gb, out=out, ws=self.ws_g[i])
            if events is not None:
                events[i][1].record()

    def gemms_concurrent(self, phase=None):
        """The three GEMMs on their own streams (wgrad, dgrad, fprop), joined
        back into the current stream; phase (a start/end pair) brackets them
        on the current stream."""
        torch, cur = self.torch, self.torch.cuda.current_stream()
        if phase is not None:
            phase[0].record(cur)
        ready = torch.cuda.Event()
        ready.record(cur)
        done = []
        ops = self.ops()
        for i in (2, 1, 0):
            a, sa, ga, b, sb, gb, out = ops[i]
            s_ = self.side[i]
            s_.wait_event(ready)
            with torch.cuda.stream(s_):
                self.fp.fp8_block_gemm(a, sa, ga, b, sb, gb, out=out, ws=self.ws_g[i])
                e_ = torch.cuda.Event()
                e_.record(s_)
            done.append(e_)
        for e_ in done:
            cur.wait_event(e_)
        if phase is not None:
            phase[1].record(cur)

    def run(self, events=None, phase=None):
        self.quantize()
        if self.concurrent and events is None:
            self.gemms_concurrent(phase)
        else:
            if phase is not None:
                phase[0].record()
            self.gemms(events)
            if phase is not None:
                phase[1].record()

    def status(self):
        return max(abs(self.fp.read_status(w)) for w in [self.ws] + self.ws_g + self.ws_q)


def max_over_ranks(torch, dist, value: float, device) -> float:
    """Largest value over all ranks (the job takes as long as its slowest rank)."""
    if dist is None or not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def flush_l2(torch, buf):
    """Leave L2 cold and clean: write all of buf (512 MB, larger than the
    129 MB L2), then read its first half back.  The write alone leaves L2
    full of dirty lines, and the timed kernel would pay for writing them back
    to HBM: a plain copy of 134 MB then reached about 0.75 of the measured
    copy bandwidth instead of about 1.0."""
    buf.zero_()
    buf[: buf.numel() // 2].max()


WARM_CALLS = 10                                 # sub-benchmarks: untimed calls first


def time_fn(torch, fn, reps=TIMED_CALLS, flush=None, warm=WARM_CALLS):
    """Median CUDA-event time (ms) of fn() on the current stream over `reps`
    calls, L2 flushed before each call; returns (median, samples)."""
    for _ in range(warm):
        fn()
    ts = []
    for _ in range(reps):
        if flush is not None:
            flush()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        fn()
        e.record()
        e.synchronize()
        ts.append(s.elapsed_time(e))
    return statistics.median(ts), ts


BATCH_SETS = 4                                  # rotating buffer sets for short kernels
BATCH_CALLS = 16                                # calls per timed sample (BATCH_SETS rounds)


def time_batched(torch, fns, reps=TIMED_CALLS, flush=None, warm=3):
    """Per-call CUDA-event time (ms) of short kernels: each of `reps` samples
    times BATCH_CALLS back-to-back calls that cycle through `fns` (one
    callable per buffer set, inputs and outputs distinct), after an L2
    flush, and divides by the count; returns (median, samples).  The event
    clock on GB300 advances in steps of about 2 us, a tenth of a 20 us
    quantiser, so one call per sample cannot resolve it.  With 4 sets of
    [8192, 4096] BF16 inputs and their outputs (about 400 MB), each set was
    last touched three calls (over 300 MB of traffic) earlier, more than the
    129 MB L2 holds, so every call still reads its input from HBM and its
    writes still reach HBM."""
    for _ in range(warm):            # warm rounds over every set (12 calls for 4 sets)
        for f in fns:
            f()
    ts = []
    for _ in range(reps):
        if flush is not None:
            flush()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for i in range(BATCH_CALLS):
            fns[i % len(fns)]()
        e.record()
        e.synchronize()
        ts.append(s.elapsed_time(e) / BATCH_CALLS)
    return statistics.median(ts), ts


def tensor_peaks(torch, fp):
    """Dense tensor-core rates measured by the library's own throughput loop
    (fp8bs_mma_peak: operands resident in shared memory, one thread issuing
    128 x 256 MMAs back to back on every SM): E4M3, MXFP8 and NVFP4.  Each is
    the best of 7 launches of about 2 ms after 3 warm-up launches (a burst
    figure, like MEASURED_PEAKS' bf16_tflops)."""
    out = {}
    for name, kind, iters in (("fp8_e4m3", 0, 16384), ("mxfp8", 1, 16384), ("nvfp4", 2, 8192)):
        flop = [0]

        def run():
            flop[0] = fp.mma_peak(kind, 256, iters)
        _, ts = time_fn(torch, run, reps=7, warm=3)
        out[name] = round(flop[0] / min(ts) / 1e9, 1)
    out["how"] = "fp8bs_mma_peak, N=256, random operands, best of 7 launches (~2 ms each), TFLOP/s"
    return out


# ---------------------------------------------------------------- sub-benchmarks
def quantize_sweep(torch, fp, dev, pk, flush):
    """Quantise sweep: BF16 [8192, 4096] at every granularity, row-wise and
    dual (row + transposed), GB/s of algorithmic bytes against HBM peak."""
    act, _ = device_inputs(torch, 100, dev)
    r, c = 8192, 4096
    x = act((r, c), 0.001, 100.0)
    e = r * c
    out = {}
    cases = {
        "1x128": 2 * e + e + 4 * e // 128,
        "128x128": 2 * e + e + 4 * (e // (128 * 128)),
        "mxfp8": 2 * e + e + e // 32,
        "per_tensor": 2 * 2 * e + e + 4,
        "nvfp4": 2 * 2 * e + e // 2 + e // 16 + 4,
    }
    ws = fp.workspace(dev)
    # BATCH_SETS copies of X (the first is the generated one); every timed
    # call below cycles through them with its own outputs per set
    xs = [x] + [x.clone() for _ in range(BATCH_SETS - 1)]
    # calibration: a plain device copy of X (the same read bytes, twice the
    # written ones) timed the same way.  "of_copy" below is its time over
    # the kernel's: on GB300 a read-only or write-only stream of this size
    # reaches only about half the copy's combined rate, so a quantiser that
    # reads X and writes fewer bytes is bound by the read, not by its total.
    xcs = [torch.empty_like(x) for _ in xs]
    copy_ms, _ = time_batched(torch, [lambda a=a, b=b: b.copy_(a) for a, b in zip(xs, xcs)], flush=flush)
    gbs = 4 * e / (copy_ms * 1e-3) / 1e9
    out["copy_calibration"] = {"gbs": round(gbs, 1), "us": round(copy_ms * 1e3, 2),
                               "frac": round(gbs / pk["hbm_gbs"], 3),
                               "what": "torch copy of the same [8192,4096] BF16 input, read + write bytes"}
    del xcs
    out["timing"] = (f"median of {TIMED_CALLS} samples; each sample {BATCH_CALLS} back-to-back calls over "
                     f"{BATCH_SETS} rotating input/output sets (~400 MB > 129 MB L2) after an L2 flush, "
                     f"divided by {BATCH_CALLS}")

    def row(nbytes, ms):
        gbs = nbytes / (ms * 1e-3) / 1e9
        return {"gbs": round(gbs, 1), "us": round(ms * 1e3, 2), "frac": round(gbs / pk["hbm_gbs"], 3),
                "of_copy": round(copy_ms / ms, 3)}

    for g, nbytes in cases.items():
        sets = [fp.fp8_quantize(xi, g, ws=ws) for xi in xs]
        fns = [lambda xi=xi, o=o: fp.fp8_quantize(xi, g, q=o[0], scales=o[1], tensor_scale=o[2], ws=ws)
               for xi, o in zip(xs, sets)]
        ms, _ = time_batched(torch, fns, flush=flush)
        out[g] = row(nbytes, ms)
        if g in ("per_tensor", "nvfp4"):
            # the same time against one read of X, the ideal if X could stay
            # on chip between the amax pass and the cast
            once = nbytes - 2 * e
            out[g]["frac_single_read_ideal"] = round(once / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], 3)
        if g in ("1x128", "mxfp8"):
            sbytes = {"1x128": 4 * e // 128, "mxfp8": e // 32}[g]
            xds = [torch.empty((r, c), dtype=torch.bfloat16, device=dev) for _ in xs]
            fns = [lambda o=o, xd=xd: fp.fp8_dequantize(o[0], o[1], g, cols=c, out=xd) for o, xd in zip(sets, xds)]
            ms, _ = time_batched(torch, fns, flush=flush)
            out["dequant_" + g] = row(e + sbytes + 2 * e, ms)
            del xds
        del sets, fns
    for g in ("1x128", "128x128", "mxfp8"):
        sets = [fp.fp8_quantize_transposed(xi, g, True, ws=ws) for xi in xs]
        sbytes = {"1x128": 4 * e // 128, "128x128": 4 * (e // 16384), "mxfp8": e // 32}[g]
        fns = [lambda xi=xi, o=o: fp.fp8_quantize_transposed(xi, g, True, q_t=o[0], scales_t=o[1], q=o[2],
                                                             scales=o[3], ws=ws)
               for xi, o in zip(xs, sets)]
        ms, _ = time_batched(torch, fns, flush=flush)
        out[g + "_dual"] = row(2 * e + 2 * e + 2 * sbytes, ms)
        del sets, fns
    return out


def moe_bench(torch, fp, dev, pk, flush):
    """The MoE expert MLP in MXFP8, Qwen3-30B-A3B shapes: gather + quantise of
    the routed tokens into expert order, grouped gate+up GEMM, SwiGLU +
    quantise, grouped down GEMM; each kernel alone and the four chained."""
    import synth
    tokens, experts, hidden, inter = 16384, 128, 2048, 768
    token_index, offsets = synth.moe_routing(tokens, experts, 8, seed=0)
    rows = int(offsets[-1])
    act, wt = device_inputs(torch, 200, dev)
    x = act((tokens, hidden), 0.001, 100.0)
    wgu = wt((experts * 2 * inter, hidden))
    wdn = wt((experts * hidden, inter))
    ws = fp.workspace(dev)
    idx = torch.from_numpy(token_index).to(dev)
    qa, sa = fp.fp8_quantize_gathered(x, idx, "mxfp8", ws=ws)
    qgu, sgu, _ = fp.fp8_quantize(wgu, "mxfp8", ws=ws)
    qdn, sdn, _ = fp.fp8_quantize(wdn, "mxfp8", ws=ws)
    qgu, sgu = qgu.view(experts, 2 * inter, hidden), sgu.view(experts, 2 * inter, hidden // 32)
    qdn, sdn = qdn.view(experts, hidden, inter), sdn.view(experts, hidden, inter // 32)
    off = torch.from_numpy(offsets).to(dev)
    d_gu = torch.empty((rows, 2 * inter), dtype=torch.bfloat16, device=dev)
    d_dn = torch.empty((rows, hidden), dtype=torch.bfloat16, device=dev)
    fp.fp8_grouped_gemm(qa, sa, qgu, sgu, off, "mxfp8", out=d_gu, ws=ws)
    qy, sy = fp.fp8_swiglu_quantize(d_gu, "mxfp8")
    f_gu = 2 * rows * 2 * inter * hidden
    f_dn = 2 * rows * hidden * inter
    run_ga = lambda: fp.fp8_quantize_gathered(x, idx, "mxfp8", q=qa, scales=sa, ws=ws)  # noqa: E731
    run_gu = lambda: fp.fp8_grouped_gemm(qa, sa, qgu, sgu, off, "mxfp8", out=d_gu, ws=ws)  # noqa: E731
    run_sw = lambda: fp.fp8_swiglu_quantize(d_gu, "mxfp8", q=qy, scales=sy)  # noqa: E731
    run_dn = lambda: fp.fp8_grouped_gemm(qy, sy, qdn, sdn, off, "mxfp8", out=d_dn, ws=ws)  # noqa: E731

    # the same dispatch as two launches: the token matrix quantised once, then
    # its code rows gathered into expert order (bit-identical to run_ga)
    qx_t, sx_t, _ = fp.fp8_quantize(x, "mxfp8", ws=ws)

    def run_qg():
        fp.fp8_quantize(x, "mxfp8", q=qx_t, scales=sx_t, ws=ws)
        fp.fp8_gather_rows(qx_t, sx_t, idx, "mxfp8", q=qa, scales=sa, ws=ws)

    def layer():
        run_ga(); run_gu(); run_sw(); run_dn()  # noqa: E702

    def layer_qg():
        run_qg(); run_gu(); run_sw(); run_dn()  # noqa: E702

    ms_qg, _ = time_fn(torch, run_qg, flush=flush)
    ms_layer_qg, _ = time_fn(torch, layer_qg, flush=flush)
    ms_ga, _ = time_fn(torch, run_ga, flush=flush)
    ms_gu, _ = time_fn(torch, run_gu, flush=flush)
    ms_sw, _ = time_fn(torch, run_sw, flush=flush)
    ms_dn, _ = time_fn(torch, run_dn, flush=flush)
    ms_layer, _ = time_fn(torch, layer, flush=flush)
    peak = pk["bf16_tflops"] * FP8_PER_BF16
    t_gu, t_dn = f_gu / ms_gu / 1e9, f_dn / ms_dn / 1e9
    # algorithmic bytes: x read once (the gathered re-reads of a token are L2 hits), the
    # index, the codes and UE8M0 scales written; SwiGLU reads [gate | up] once
    b_ga = tokens * hidden * 2 + rows * 8 + rows * hidden + rows * hidden // 32
    b_sw = rows * 2 * inter * 2 + rows * inter + rows * inter // 32
    g_ga, g_sw = b_ga / (ms_ga * 1e-3) / 1e9, b_sw / (ms_sw * 1e-3) / 1e9
    lp = pk.get("loop", {}).get("mxfp8")
    return {"gate_up": {"tflops": round(t_gu, 1), "ms": round(ms_gu, 3), "frac": round(t_gu / peak, 3),
                        "frac_of_mxfp8_loop_peak": round(t_gu / lp, 3) if lp else None},
            "down": {"tflops": round(t_dn, 1), "ms": round(ms_dn, 3), "frac": round(t_dn / peak, 3),
                     "frac_of_mxfp8_loop_peak": round(t_dn / lp, 3) if lp else None},
            "gather_quantize": {"gbs": round(g_ga, 1), "us": round(ms_ga * 1e3, 2),
                                "frac": round(g_ga / pk["hbm_gbs"], 3), "bytes": b_ga},
            "quantize_then_gather": {"gbs": round(b_ga / (ms_qg * 1e-3) / 1e9, 1), "us": round(ms_qg * 1e3, 2),
                                     "frac": round(b_ga / (ms_qg * 1e-3) / 1e9 / pk["hbm_gbs"], 3), "bytes": b_ga,
                                     "launches": 2},
            "layer_quantize_then_gather": {"ms": round(ms_layer_qg, 3),
                                           "tflops": round((f_gu + f_dn) / ms_layer_qg / 1e9, 1), "kernels": 5},
            "swiglu_quantize": {"gbs": round(g_sw, 1), "us": round(ms_sw * 1e3, 2),
                                "frac": round(g_sw / pk["hbm_gbs"], 3), "bytes": b_sw},
            "layer": {"ms": round(ms_layer, 3), "tflops": round((f_gu + f_dn) / ms_layer / 1e9, 1),
                      "kernels": 4},
            "peak_tflops": round(peak, 1), "peak_note": "measured bf16 burst x nominal fp8/bf16 ratio 2"}


def moe_nvfp4_bench(torch, fp, dev, pk, flush):
    """The MoE expert GEMMs in NVFP4 (Qwen3-30B-A3B shapes, the NVFP4 recipe's
    MoE): routed activations with per-token outer scales, each expert's
    weight with its own outer scale (gate and up sharing one)."""
    import synth
    tokens, experts, hidden, inter = 16384, 128, 2048, 768
    _, offsets = synth.moe_routing(tokens, experts, 8, seed=0)
    rows = int(offsets[-1])
    act, wt = device_inputs(torch, 400, dev)
    ws = fp.workspace(dev)
    off = torch.from_numpy(offsets).to(dev)

    def expert_weights(n, k):
        w = wt((experts, n, k))
        q = torch.empty((experts, n, k // 2), dtype=torch.uint8, device=dev)
        s = torch.empty((experts, n, k // 16), dtype=torch.uint8, device=dev)
        t = torch.empty((experts,), dtype=torch.float32, device=dev)
        for e in range(experts):
            fp.fp8_quantize(w[e], "nvfp4", q=q[e], scales=s[e], tensor_scale=t[e:e + 1], ws=ws)
        return q, s, t
    qgu, sgu, tgu = expert_weights(2 * inter, hidden)
    qdn, sdn, tdn = expert_weights(hidden, inter)
    qa, sa, ta = fp.fp8_quantize(act((rows, hidden), 0.001, 100.0), "nvfp4_row", ws=ws)
    qh, sh_, th = fp.fp8_quantize(act((rows, inter), 0.0, 1.0), "nvfp4_row", ws=ws)
    d_gu = torch.empty((rows, 2 * inter), dtype=torch.bfloat16, device=dev)
    d_dn = torch.empty((rows, hidden), dtype=torch.bfloat16, device=dev)
    run_gu = lambda: fp.fp8_grouped_gemm(qa, sa, qgu, sgu, off, "nvfp4_row", a_tensor_scale=ta,  # noqa: E731
                                         b_tensor_scale=tgu, k=hidden, out=d_gu, ws=ws)
    run_dn = lambda: fp.fp8_grouped_gemm(qh, sh_, qdn, sdn, off, "nvfp4_row", a_tensor_scale=th,  # noqa: E731
                                         b_tensor_scale=tdn, k=inter, out=d_dn, ws=ws)
    ms_gu, _ = time_fn(torch, run_gu, flush=flush)
    ms_dn, _ = time_fn(torch, run_dn, flush=flush)
    f_gu, f_dn = 2 * rows * 2 * inter * hidden, 2 * rows * hidden * inter
    peak = pk["bf16_tflops"] * FP4_PER_BF16
    lp = pk.get("loop", {}).get("nvfp4")
    out = {}
    for name, f, ms in (("gate_up", f_gu, ms_gu), ("down", f_dn, ms_dn)):
        t = f / ms / 1e9
        out[name] = {"tflops": round(t, 1), "ms": round(ms, 3), "frac": round(t / peak, 3),
                     "frac_of_nvfp4_loop_peak": round(t / lp, 3) if lp else None}
    out["note"] = "A per-token NVFP4 (nvfp4_row), B NVFP4 with one outer scale per expert"
    out["peak_note"] = "measured bf16 burst x nominal fp4/bf16 ratio 6"
    return out


def nvfp4_bench(torch, fp, dev, pk, flush):
    """NVFP4 linear, Qwen2.5-32B MLP shape X [16384,5120] x W [27648,5120]^T."""
    m, n, k = 16384, 27648, 5120
    act, wt = device_inputs(torch, 300, dev)
    x = act((m, k), 0.0, 1.0)
    w = wt((n, k))
    ws = fp.workspace(dev)
    qx, sx, tx = fp.fp8_quantize(x, "nvfp4", ws=ws)
    qw, sw, tw = fp.fp8_quantize(w, "nvfp4", ws=ws)
    d = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    run = lambda: fp.fp8_block_gemm(qx, sx, "nvfp4", qw, sw, "nvfp4", tx, tw, k=k, out=d, ws=ws)  # noqa: E731
    ms, _ = time_fn(torch, run, flush=flush)
    flop = 2 * m * n * k
    t = flop / ms / 1e9
    peak = pk["bf16_tflops"] * FP4_PER_BF16
    e = m * k
    # quantisers (tens of us): batched over rotating copies of X, each with
    # its own outputs (4 x 168 MB inputs)
    xs = [x] + [x.clone() for _ in range(BATCH_SETS - 1)]
    sets = [(qx, sx, tx)] + [fp.fp8_quantize(xi, "nvfp4", ws=ws) for xi in xs[1:]]
    qms, _ = time_batched(torch, [lambda xi=xi, o=o: fp.fp8_quantize(xi, "nvfp4", q=o[0], scales=o[1],
                                                                      tensor_scale=o[2], ws=ws)
                                  for xi, o in zip(xs, sets)], flush=flush)
    qgbs = (2 * 2 * e + e // 2 + e // 16) / (qms * 1e-3) / 1e9
    # the recipe's activation form: per-token outer scales, four-over-six blocks
    fos = fp.FLAG_NVFP4_4OVER6
    rsets = [fp.fp8_quantize(xi, "nvfp4_row", flags=fos, ws=ws) for xi in xs]
    qr, sr, tr = rsets[0]
    rms, _ = time_batched(torch, [lambda xi=xi, o=o: fp.fp8_quantize(xi, "nvfp4_row", q=o[0], scales=o[1],
                                                                      tensor_scale=o[2], flags=fos, ws=ws)
                                  for xi, o in zip(xs, rsets)], flush=flush)
    rgbs = (2 * e + e // 2 + e // 16 + 4 * m) / (rms * 1e-3) / 1e9       # one HBM read: the second pass hits L2
    run_r = lambda: fp.fp8_block_gemm(qr, sr, "nvfp4_row", qw, sw, "nvfp4", tr, tw, k=k, out=d, ws=ws)  # noqa: E731
    ms_r, _ = time_fn(torch, run_r, flush=flush)
    t_r = flop / ms_r / 1e9
    xds = [torch.empty_like(x) for _ in range(BATCH_SETS)]
    dms, _ = time_batched(torch, [lambda o=o, xd=xd: fp.fp8_dequantize(o[0], o[1], "nvfp4_row", cols=k,
                                                                        tensor_scale=o[2], out=xd)
                                  for o, xd in zip(rsets, xds)], flush=flush)
    dgbs = (e // 2 + e // 16 + 4 * m + 2 * e) / (dms * 1e-3) / 1e9
    lp = pk.get("loop", {}).get("nvfp4")
    return {"gemm": {"tflops": round(t, 1), "ms": round(ms, 3), "frac": round(t / peak, 3),
                     "frac_of_nvfp4_loop_peak": round(t / lp, 3) if lp else None},
            "gemm_row_scaled_a": {"tflops": round(t_r, 1), "ms": round(ms_r, 3), "frac": round(t_r / peak, 3),
                                  "frac_of_nvfp4_loop_peak": round(t_r / lp, 3) if lp else None},
            "peak_tflops": round(peak, 1), "peak_note": "measured bf16 burst x nominal fp4/bf16 ratio 6",
            "quantize_x": {"gbs": round(qgbs, 1), "us": round(qms * 1e3, 1), "frac": round(qgbs / pk["hbm_gbs"], 3)},
            "quantize_x_row_4over6": {"gbs": round(rgbs, 1), "us": round(rms * 1e3, 1),
                                      "frac": round(rgbs / pk["hbm_gbs"], 3)},
            "dequantize_x_bf16": {"gbs": round(dgbs, 1), "us": round(dms * 1e3, 1),
                                  "frac": round(dgbs / pk["hbm_gbs"], 3)}}


# ---------------------------------------------------------------- CPU oracle
def cpu_model() -> str:
    """The host CPU's model name: /proc/cpuinfo's (x86), lscpu's (Arm, whose
    /proc/cpuinfo has none), else the platform's."""
    import platform
    import subprocess
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.processor() or platform.machine()


def cpu_oracle_sample(rows: int = 4096):
    """The oracle on a bounded slice of the step: quantise `rows` token rows of
    X and dY and the whole weight W, run the three GEMMs for those rows
    (fprop: rows x I, dgrad: rows x H, wgrad: I x H over `rows` tokens).
    The default (half the step's tokens) is about 10-20 s of CPU work."""
    import numpy as np
    import synth
    from oracle import formats as OF
    from oracle import gemm as OG
    from oracle import quantize as OQ
    x = OF.bf16_bits_to_f32(synth.activations((rows, H3), seed=0))
    dy = OF.bf16_bits_to_f32(synth.activations((rows, I3), seed=2))
    w = OF.bf16_bits_to_f32(synth.weights((I3, H3), seed=1))
    t0 = time.perf_counter()
    qx, sx = OQ.quantize_1x128(x)
    qw, sw = OQ.quantize_128x128(w)
    qdy, sdy = OQ.quantize_1x128(dy)
    qwt, swt = OQ.transposed(OQ.quantize_128x128, w)
    qdyt, sdyt = OQ.transposed(OQ.quantize_1x128, dy)
    qxt, sxt = OQ.transposed(OQ.quantize_1x128, x)
    OG.block_gemm(qx, sx, "1x128", qw, sw, "128x128")
    OG.block_gemm(qdy, sdy, "1x128", qwt, swt, "128x128")
    OG.block_gemm(qdyt, sdyt, "1x128", qxt, sxt, "1x128")
    dt = time.perf_counter() - t0
    flop = 3 * 2 * rows * H3 * I3
    threads = int(os.environ.get("OMP_NUM_THREADS", "0")) or (os.cpu_count() or 1)
    return {"value": flop / dt / 1e12, "unit": "TFLOPS", "cores": threads, "kind": "oracle",
            "cpu": cpu_model(), "seconds": round(dt, 2),
            "sample": f"{rows} of {M3} token rows of the step (all three GEMMs, weight quantised in full); "
                      f"FLOPs counted for the sample only"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    # one bounded sample per step (about 3-7 s on a 16-core host), so that
    # --steps K ends within a few minutes
    res = [cpu_oracle_sample(256) for _ in range(max(1, args.steps))]
    v = statistics.mean(r["value"] for r in res)
    cb = dict(res[0])
    cb["value"] = v
    line = {"impl": "reference", "metric": METRIC,
            "value": v, "unit": "TFLOPS", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(args),
            "cpu_baseline": cb, "e2e": {"value": v, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                                        "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def gemm_source_sha16() -> str:
    """SHA-256 (first 16 hex digits) of the blockwise GEMM's source files."""
    import hashlib
    h = hashlib.sha256()
    for f in ("gemm_blockwise.cu", "sched.cuh", "ptx.cuh"):
        with open(os.path.join(ROOT, "fp8_block_scaled_03_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def workload_config(args):
    return {"workload": "dense blockwise FP8 linear fwd+bwd, Qwen3-4B MLP shape (tokens 8192, hidden 2560, "
                        "intermediate 9728); X,dY 1x128 FP32 scales (dual row+transposed), W 128x128 FP32 scales; "
                        "the three quantisers concurrently, then the three independent GEMMs concurrently "
                        "(wgrad, dgrad, fprop on streams of their own by priority, dynamic tile order)",
            "tokens": M3, "hidden": H3, "intermediate": I3, "parallelism": f"replicas x{args.gpus}",
            "l2": "inputs 250 MB and step working set ~630 MB, both > 129 MB L2; sub-benchmarks flush L2 "
                  "before each timed call (512 MB written, then 256 MB of it read back, so L2 starts cold and "
                  "clean); quantiser rows time 16 back-to-back calls over 4 rotating input/output sets "
                  "(~400 MB) after such a flush"}


# ---------------------------------------------------------------- main
def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    import torch
    import torch.distributed as dist
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    from fp8_block_scaled_03_gb300 import build as _build
    if rank == 0:
        _build.build()
    if world > 1:
        dist.barrier()
    import fp8_block_scaled_03_gb300 as fp
    fp.load_library()
    if args.kernel is not None:
        single_kernel(args, torch, fp, dev)
        return
    pk = peaks()
    step = DenseStep(torch, fp, dev, seed=1000 + rank)
    step.concurrent = not args.sequential_gemms
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush = lambda: flush_l2(torch, flush_buf)  # noqa: E731

    for _ in range(max(3, args.warmup)):
        step.run()
    torch.cuda.synchronize()

    # ---- timed region: exactly K steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    pev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(args.steps):
            ev[i][0].record()
            step.run(phase=pev[i])
            ev[i][1].record()
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        if world > 1:
            dist.barrier()
    ms_steps = [a.elapsed_time(b) for a, b in ev]
    ms_total = ms_steps and ev[0][0].elapsed_time(ev[-1][1])
    phase_ms = [a.elapsed_time(b) for a, b in pev]
    ms_total = max_over_ranks(torch, dist if world > 1 else None, ms_total, dev)
    ms_per_step = ms_total / args.steps
    value = world * STEP_FLOP / (ms_per_step * 1e-3) / 1e12
    assert step.status() == 0, "a device wait timed out during the bench"

    # ---- roofline of the dominant kernel (the blockwise GEMM), measured in the
    # timed region: the three GEMMs run concurrently there, so a launch's
    # average duration is a third of the GEMM phase (from the end of the
    # quantisers to the last GEMM, on the step's stream)
    avg_gemm_ms = statistics.mean(phase_ms) / 3
    achieved = GEMM_FLOP / (avg_gemm_ms * 1e-3) / 1e12
    # each GEMM alone, one after another (not timed in the step): for reference
    gev = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in range(3)]
           for _ in range(max(3, args.steps // 2))]
    for g in gev:
        step.gemms(g)
    torch.cuda.synchronize()
    per_gemm = [statistics.mean(g[j][0].elapsed_time(g[j][1]) for g in gev) for j in range(3)]
    assert step.status() == 0, "a device wait timed out during the bench"
    # the GEMMs run for well under a second here, so the burst BF16 figure is the denominator
    peak_fp8 = pk["bf16_tflops"] * FP8_PER_BF16
    sha = gemm_source_sha16()
    roofline = {"bound": "tensor", "kernel": "gemm_blockwise_kernel<1x128,128x128|1x128>",
                "achieved": round(achieved, 1), "peak": round(peak_fp8, 1), "unit": "TFLOP/s",
                "frac": round(achieved / peak_fp8, 3),
                "traffic": GEMM_TRAFFIC["bytes"] if GEMM_TRAFFIC["source_sha16"] == sha else None,
                "traffic_unit": "DRAM bytes read + written per launch (ncu), null if the kernel changed since",
                "kernel_source_sha16": sha,
                "peak_note": f"{pk['source']} bf16 burst x nominal fp8/bf16 ratio 2 (of {pk['source']})",
                "gemm_phase_ms": round(3 * avg_gemm_ms, 4),
                "per_gemm_ms": [round(x, 4) for x in per_gemm],
                "per_gemm_note": "fprop, dgrad, wgrad each alone on one stream, after the timed region",
                "recompute": "achieved = 2*8192*2560*9728 FLOP / (gemm_phase_ms / 3); frac = achieved / peak"}
    if rank == 0:
        loop = tensor_peaks(torch, fp)
        pk["loop"] = loop
        roofline["measured_fp8_loop_peak"] = loop["fp8_e4m3"]
        roofline["frac_of_fp8_loop_peak"] = round(achieved / loop["fp8_e4m3"], 3)

    line = {"metric": METRIC,
            "value": round(value, 1), "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": round(ms_per_step, 4), "wall_s": round(wall, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 (fp32 accum, bf16 out)",
            "data": "synthetic", "config": workload_config(args), "roofline": roofline,
            "gpu_launches": step.launches_per_step * args.steps, "clocks": clk.summary()}
    if rank == 0:
        line["tensor_peak_measured"] = pk["loop"]

    if rank == 0 and not args.no_extras:
        line["dense_pow2"] = pow2_step_bench(torch, fp, dev, args, pk)
        line["quantize"] = quantize_sweep(torch, fp, dev, pk, flush)
        line["moe_mxfp8"] = moe_bench(torch, fp, dev, pk, flush)
        line["nvfp4"] = nvfp4_bench(torch, fp, dev, pk, flush)
        line["moe_nvfp4"] = moe_nvfp4_bench(torch, fp, dev, pk, flush)
        line["e2e"] = e2e_bench(torch, fp, dev, step, reps=max(8, args.steps))
        line["cpu_baseline"] = cpu_oracle_sample()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def single_kernel(args, torch, fp, dev):
    """One piece of the path, W warm-up + K timed calls, inputs sized as in the
    step (used for ncu captures of a single kernel)."""
    act, wt = device_inputs(torch, 7, dev)
    ws = fp.workspace(dev)
    name = args.kernel
    if name in ("fprop", "dgrad", "wgrad", "fprop_pow2", "dgrad_pow2", "wgrad_pow2"):
        g = name.split("_")[0]
        sfx = "_pow2" if name.endswith("_pow2") else ""
        m, n, k = {"fprop": (M3, I3, H3), "dgrad": (M3, H3, I3), "wgrad": (I3, H3, M3)}[g]
        a = act((m, k), 0.01, 50.0)
        b = act((n, k), 0.01, 50.0) if g == "wgrad" else wt((n, k))
        ga = "1x128" + sfx
        gb = ("1x128" if g == "wgrad" else "128x128") + sfx
        qa, sa, _ = fp.fp8_quantize(a, ga, ws=ws)
        qb, sb, _ = fp.fp8_quantize(b, gb, ws=ws)
        out = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        fn = lambda: fp.fp8_block_gemm(qa, sa, ga, qb, sb, gb, out=out, ws=ws)  # noqa: E731
        work = 2 * m * n * k
    elif name.startswith("quant") or name.startswith("dequant"):
        x = act((8192, 4096), 0.001, 100.0)
        if name == "quant_nvfp4_row_4over6":
            fos = fp.FLAG_NVFP4_4OVER6
            q, s_, t_ = fp.fp8_quantize(x, "nvfp4_row", flags=fos, ws=ws)
            fn = lambda: fp.fp8_quantize(x, "nvfp4_row", q=q, scales=s_, tensor_scale=t_, flags=fos,  # noqa: E731
                                         ws=ws)
        elif name == "quant_nvfp4":
            q, s_, t_ = fp.fp8_quantize(x, "nvfp4", ws=ws)
            fn = lambda: fp.fp8_quantize(x, "nvfp4", q=q, scales=s_, tensor_scale=t_, ws=ws)  # noqa: E731
        elif name == "quant_per_tensor":
            q, s_, _ = fp.fp8_quantize(x, "per_tensor", ws=ws)
            fn = lambda: fp.fp8_quantize(x, "per_tensor", q=q, scales=s_, ws=ws)  # noqa: E731
        elif name == "dequant_1x128":
            q, s_, _ = fp.fp8_quantize(x, "1x128", ws=ws)
            xd = torch.empty_like(x)
            fn = lambda: fp.fp8_dequantize(q, s_, "1x128", cols=x.shape[1], out=xd)  # noqa: E731
        elif name == "quant_dual_1x128":
            bufs = fp.fp8_quantize_transposed(x, "1x128", True, ws=ws)
            fn = lambda: fp.fp8_quantize_transposed(x, "1x128", True, q_t=bufs[0], scales_t=bufs[1],  # noqa: E731
                                                    q=bufs[2], scales=bufs[3], ws=ws)
        else:
            g = "1x128" if name == "quant_1x128" else "mxfp8"
            q, s_, _ = fp.fp8_quantize(x, g, ws=ws)
            fn = lambda: fp.fp8_quantize(x, g, q=q, scales=s_, ws=ws)  # noqa: E731
        work = 0
    elif name == "moe_layer":
        # the four kernels of the expert MLP, as the bench's moe_mxfp8.layer times them
        import synth
        token_index, offsets = synth.moe_routing(16384, 128, 8, seed=0)
        rows = int(offsets[-1])
        x = act((16384, 2048), 0.001, 100.0)
        idx = torch.from_numpy(token_index).to(dev)
        off = torch.from_numpy(offsets).to(dev)
        qgu, sgu, _ = fp.fp8_quantize(wt((128 * 1536, 2048)), "mxfp8", ws=ws)
        qdn, sdn, _ = fp.fp8_quantize(wt((128 * 2048, 768)), "mxfp8", ws=ws)
        qgu, sgu = qgu.view(128, 1536, 2048), sgu.view(128, 1536, 64)
        qdn, sdn = qdn.view(128, 2048, 768), sdn.view(128, 2048, 24)
        qa, sa = fp.fp8_quantize_gathered(x, idx, "mxfp8", ws=ws)
        h = torch.empty((rows, 1536), dtype=torch.bfloat16, device=dev)
        out = torch.empty((rows, 2048), dtype=torch.bfloat16, device=dev)
        qy, sy = fp.fp8_swiglu_quantize(h, "mxfp8")

        def fn():
            fp.fp8_quantize_gathered(x, idx, "mxfp8", q=qa, scales=sa, ws=ws)
            fp.fp8_grouped_gemm(qa, sa, qgu, sgu, off, "mxfp8", out=h, ws=ws)
            fp.fp8_swiglu_quantize(h, "mxfp8", q=qy, scales=sy)
            fp.fp8_grouped_gemm(qy, sy, qdn, sdn, off, "mxfp8", out=out, ws=ws)
        work = 2 * rows * 1536 * 2048 + 2 * rows * 2048 * 768
    elif name in ("moe_gather_quant", "moe_swiglu_quant", "moe_quant_then_gather"):
        import synth
        token_index, offsets = synth.moe_routing(16384, 128, 8, seed=0)
        rows = int(offsets[-1])
        if name == "moe_quant_then_gather":
            x = act((16384, 2048), 0.001, 100.0)
            idx = torch.from_numpy(token_index).to(dev)
            qt, st, _ = fp.fp8_quantize(x, "mxfp8", ws=ws)
            q, s_ = fp.fp8_gather_rows(qt, st, idx, "mxfp8", ws=ws)

            def fn():
                fp.fp8_quantize(x, "mxfp8", q=qt, scales=st, ws=ws)
                fp.fp8_gather_rows(qt, st, idx, "mxfp8", q=q, scales=s_, ws=ws)
        elif name == "moe_gather_quant":
            x = act((16384, 2048), 0.001, 100.0)
            idx = torch.from_numpy(token_index).to(dev)
            q, s_ = fp.fp8_quantize_gathered(x, idx, "mxfp8", ws=ws)
            fn = lambda: fp.fp8_quantize_gathered(x, idx, "mxfp8", q=q, scales=s_, ws=ws)  # noqa: E731
        else:
            h = act((rows, 2 * 768), 0.0, 1.0)
            q, s_ = fp.fp8_swiglu_quantize(h, "mxfp8")
            fn = lambda: fp.fp8_swiglu_quantize(h, "mxfp8", q=q, scales=s_)  # noqa: E731
        work = 0
    elif name == "moe_gate_up":
        import synth
        _, offsets = synth.moe_routing(16384, 128, 8, seed=0)
        rows = int(offsets[-1])
        qa, sa, _ = fp.fp8_quantize(act((rows, 2048), 0.001, 100.0), "mxfp8", ws=ws)
        qb, sb, _ = fp.fp8_quantize(wt((128 * 1536, 2048)), "mxfp8", ws=ws)
        off = torch.from_numpy(offsets).to(dev)
        out = torch.empty((rows, 1536), dtype=torch.bfloat16, device=dev)
        fn = lambda: fp.fp8_grouped_gemm(qa, sa, qb.view(128, 1536, 2048), sb.view(128, 1536, 64), off,  # noqa: E731
                                         "mxfp8", out=out, ws=ws)
        work = 2 * rows * 1536 * 2048
    elif name.startswith("mma_peak"):
        # the tensor-core throughput loop behind the measured FP8 / FP4 peaks
        kind = {"mma_peak_e4m3": 0, "mma_peak_mxfp8": 1, "mma_peak_nvfp4": 2}[name]
        flop = [0]

        def fn():
            flop[0] = fp.mma_peak(kind, 256, 8192)
        fn()
        work = flop[0]
    else:  # nvfp4
        m, n, k = 16384, 27648, 5120
        qx, sx, tx = fp.fp8_quantize(act((m, k), 0.0, 1.0), "nvfp4", ws=ws)
        qw, sw, tw = fp.fp8_quantize(wt((n, k)), "nvfp4", ws=ws)
        out = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        fn = lambda: fp.fp8_block_gemm(qx, sx, "nvfp4", qw, sw, "nvfp4", tx, tw, k=k, out=out, ws=ws)  # noqa: E731
        work = 2 * m * n * k
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    ms, _ = time_fn(torch, fn, max(1, args.steps), None, warm=0)
    res = {"kernel": name, "ms": round(ms, 4)}
    if work:
        res["tflops"] = round(work / ms / 1e9, 1)
    assert fp.read_status() == 0
    print(json.dumps(res), flush=True)


def pow2_step_bench(torch, fp, dev, args, pk):
    """The same fwd+bwd step with power-of-two block scales (tensor-core
    block-scale path instead of FP32 promotion)."""
    step = DenseStep(torch, fp, dev, seed=2000, recipe="pow2")
    step.concurrent = not args.sequential_gemms
    for _ in range(max(3, args.warmup)):
        step.run()
    torch.cuda.synchronize()
    n = max(1, args.steps)
    # the GEMM phase of every step bracketed by events, read after the loop
    # (no host synchronisation inside the timed steps)
    pev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record()
    for i in range(n):
        step.run(phase=pev[i])
    s1.record()
    s1.synchronize()
    per_step = s0.elapsed_time(s1) / n
    avg = statistics.mean(a.elapsed_time(b) for a, b in pev) / 3
    # each GEMM alone, one after another, after the timed steps
    gev = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in range(3)]
           for _ in range(max(3, n // 2))]
    for g in gev:
        step.gemms(g)
    torch.cuda.synchronize()
    gms = [statistics.mean(g[j][0].elapsed_time(g[j][1]) for g in gev) for j in range(3)]
    assert step.status() == 0, "a device wait timed out during the power-of-two step"
    peak = pk["bf16_tflops"] * FP8_PER_BF16
    t = GEMM_FLOP / avg / 1e9
    lp = pk.get("loop", {}).get("mxfp8")
    return {"tflops_step": round(STEP_FLOP / per_step / 1e9, 1), "ms_per_step": round(per_step, 4),
            "gemm_tflops": round(t, 1), "gemm_frac": round(t / peak, 3),
            "gemm_frac_of_mxfp8_loop_peak": round(t / lp, 3) if lp else None,
            "peak_note": "measured bf16 burst x nominal fp8/bf16 ratio 2",
            "gemm_phase_ms": round(3 * avg, 4),
            "per_gemm_ms": [round(g, 4) for g in gms]}


def e2e_bench(torch, fp, dev, step, reps=8):
    """The step through the public API from pinned HOST buffers, with every
    host<->device copy inside the timed region: each step copies X, W and dY
    in and Y, dX and dW out.  The copies run on streams of their own, two
    buffer sets deep, so step i's outputs go out and step i+1's inputs come in
    while step i computes (as a training loop overlaps its transfers).
    Timed with CUDA events from the first input copy to the last output copy,
    over `reps` steps (the bench's --steps, at least 8): the pipeline's fill
    (the first input copy and compute) and drain (the last output copy) are
    inside the timed region and spread over those steps."""
    sets = [step, DenseStep(torch, fp, dev, seed=3000)]
    sets[1].concurrent = step.concurrent
    hx, hw, hdy = (t.cpu().pin_memory() for t in (step.x, step.w, step.dy))
    hout = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (s_.y, s_.dx, s_.dw)] for s_ in sets]
    s_in, s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def run(n, t_start=None, t_end=None):
        cmp_done, d2h_done = [None] * n, [None] * n
        if t_start is not None:
            t_start.record(s_in)
        for i in range(n):
            st = sets[i % 2]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(cmp_done[i - 2])        # this set's inputs are no longer read
                for h, d in zip((hx, hw, hdy), (st.x, st.w, st.dy)):
                    d.copy_(h, non_blocking=True)
                h2d_done = torch.cuda.Event()
                h2d_done.record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(h2d_done)
                if i >= 2:
                    s_cmp.wait_event(d2h_done[i - 2])       # this set's outputs have been copied out
                st.run()
                cmp_done[i] = torch.cuda.Event()
                cmp_done[i].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(cmp_done[i])
                for h, d in zip(hout[i % 2], (st.y, st.dx, st.dw)):
                    h.copy_(d, non_blocking=True)
                d2h_done[i] = torch.cuda.Event()
                d2h_done[i].record(s_out)
        if t_end is not None:
            t_end.record(s_out)

    # the host link on its own: one step's input copy, then one step's output copy
    def copy_gbs(pairs, stream, n=3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for dst, src in pairs:                          # one untimed round (first use of the pinned pages)
                dst.copy_(src, non_blocking=True)
            e0.record(stream)
            for _ in range(n):
                for dst, src in pairs:
                    dst.copy_(src, non_blocking=True)
            e1.record(stream)
        e1.synchronize()
        nbytes = n * sum(src.numel() * src.element_size() for _, src in pairs)
        return round(nbytes / (e0.elapsed_time(e1) * 1e-3) / 1e9, 1)

    torch.cuda.synchronize()
    h2d_gbs = copy_gbs([(d, h) for h, d in zip((hx, hw, hdy), (step.x, step.w, step.dy))], s_in)
    d2h_gbs = copy_gbs([(h, d) for h, d in zip(hout[0], (step.y, step.dx, step.dw))], s_out)
    run(2)
    torch.cuda.synchronize()
    # three timed runs of `reps` steps; the median is reported (the host link
    # is shared with the machine's other traffic, and one run can catch a
    # burst of it)
    runs = []
    for _ in range(3):
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        run(reps, t0, t1)
        t1.synchronize()
        torch.cuda.synchronize()
        runs.append(t0.elapsed_time(t1) / reps)
    ms = statistics.median(runs)
    h2d = sum(t.numel() * t.element_size() for t in (hx, hw, hdy))
    d2h = sum(t.numel() * t.element_size() for t in hout[0])
    return {"value": round(STEP_FLOP / (ms * 1e-3) / 1e12, 1), "unit": "TFLOPS", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 3),
            "ms_per_step_runs": [round(x, 3) for x in runs],
            "pipeline": f"2 buffer sets; H2D, compute and D2H on separate streams; {reps} steps timed, "
                        "median of 3 such runs",
            "host_link_gbs": {"h2d": h2d_gbs, "d2h": d2h_gbs}}


if __name__ == "__main__":
    main()
