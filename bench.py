"""Benchmark: block forward + fine-grained recompute + backward TFLOP/s on one GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                [--workload NAME] [--recompute fine|full|none|selective]

One step = one oases_stack_step call (forward, recompute, backward of the whole
block, weight gradients accumulated) on synthetic seeded inputs resident in HBM.
The default workload is the largest one that fits one GPU: the 4-layer GPT-style
stack, bf16, hidden 2560, ffn 10240, 20 heads of 128, causal, seq 2048, batch 8,
w = 4 simulated shards, 2 sub-batches.  FLOPs are algorithmic and counted for
the fine-grained schedule (FFN: 14 M H F; attention: 30 M H^2 + 9 B S^2 H with
causal halving), whatever mode is timed.  The headline percentage is of the
measured dense bf16 GEMM peak (burst); the percentage of the sustained rate is
given beside it.

L2: each timed step is bracketed by CUDA events on the call's first stream and
followed, outside the events, by a 256 MiB write that flushes the 129 MB L2.

roofline: the tcgen05 GEMM kernel (gemm_tc_kernel, every instantiation), which
has the largest share of the step's GPU time, timed alone launch by launch over
one sub-batch's GEMMs of one layer (L2 flushed before each); achieved = their
algorithmic FLOPs / their summed CUDA-event time.  roofline_attention_bwd: the
same for the attention backward (delta, dQ and dK/dV kernels).

--impl reference times the CPU oracle (fp64 numpy, oracle/) on this host's
cores on a bounded sample of the same workload; it is a deliberately slow
reference, not a competitor.

Under torchrun (N > 1) every rank runs an independent replica of the workload
on its own GPU (the block does not shard across GPUs here: all w shards live
on one device); value = total FLOPs of all ranks / max time over ranks.
"""
from __future__ import annotations

import argparse
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

METRIC = "block fwd+recompute+bwd TFLOP/s at 1 GB300; % of dense BF16 peak"
# ncu dram__bytes_read.sum + dram__bytes_write.sum of the roofline kernel's
# launches (one sub-batch's GEMMs of one layer, each launched once, cold L2),
# per launch, by workload, with the sha256 of the GEMM sources they were
# measured on (kernel_source_sha).  Reported only while those sources are
# unchanged.
NCU_TRAFFIC = {
    # the 14 GEMMs of one sub-batch of one layer, each launched twice (28 launches),
    # profiles/gemm_tc_stack4_h2560_traffic.md
    "stack4_bf16_h2560": {"source_sha256": "f92fa70c280c5ff2880fbcbca69ab84ef2764cc6bcd2976a8bb970ddfe724d1d",
                          "bytes_per_launch": 401570596},
}


GEMM_SOURCES = ("gemm_tc.cu", "common.cuh", "epilogue.cuh", "sm100_ptx.cuh")


def kernel_source_sha() -> str:
    """sha256 over the sources the tensor-core GEMM kernel is compiled from."""
    h = hashlib.sha256()
    for name in GEMM_SOURCES:
        with open(os.path.join(ROOT, "tensor_model_transformer_tp_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the roofline kernel from the ncu capture of
    this workload while the GEMM sources are unchanged; else None."""
    rec = NCU_TRAFFIC.get(workload)
    if rec and rec["source_sha256"] == kernel_source_sha():
        return rec["bytes_per_launch"]
    return None


def flops_fine(shape, mode="fine") -> float:
    """Algorithmic FLOPs of one step, counted for the FINE schedule: FFN
    fwd 4MHF + recompute 2MHF + bwd 8MHF; attention fwd 8MH^2 + 2BS^2H,
    recompute 6MH^2 + 2BS^2H, bwd 16MH^2 + 5BS^2H (causal; x2 without the
    mask).  NONE and SELECTIVE are credited only with what they execute (no
    recompute; SELECTIVE recomputes the attention operation); FULL's extra
    work is not credited."""
    M, H, B, S = shape.rows, shape.hidden, shape.batch, shape.seq
    bs2h = B * S * S * H * (1.0 if shape.causal else 2.0)
    f = 0.0
    if shape.kind in ("ffn", "layer"):
        f += (12.0 if mode in ("none", "selective") else 14.0) * M * H * shape.ffn
    if shape.kind in ("attn", "layer"):
        if mode == "none":
            f += 24.0 * M * H * H + 7.0 * bs2h
        elif mode == "selective":
            f += 24.0 * M * H * H + 9.0 * bs2h
        else:
            f += 30.0 * M * H * H + 9.0 * bs2h
    return f * shape.n_layers


def peaks():
    p = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
         "source": "fallback"}
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
            if k in d:
                p[k] = float(d[k])
        p["source"] = "measured"
    return p


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons every 50 ms.  The
    caller marks the timed regions (mark_start / mark_end, host wall clock
    around the synchronised regions); summary() keeps the samples taken inside
    them."""
    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}
    PERIOD_MS = 50

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.samples = []   # (host time, sm MHz, max MHz, reasons bitmask)
        self.windows = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                 "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)   # the first sample arrives before the timed region
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            try:
                self.samples.append((time.time(), float(parts[0]), float(parts[1]),
                                     int(parts[2], 16)))
            except (ValueError, IndexError):
                continue

    def mark_start(self):
        self.windows.append([time.time(), None])

    def mark_end(self):
        self.windows[-1][1] = time.time()

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        inside = [smp for smp in self.samples
                  if any(w0 <= smp[0] <= (w1 if w1 is not None else float("inf"))
                         for w0, w1 in self.windows)] if self.windows else list(self.samples)
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        reasons = set()
        for _, _, _, r in inside:
            for bit, name in self.REASONS.items():
                if r & bit and name != "gpu_idle":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(x[1] for x in inside), "sm_max_mhz": inside[-1][2],
                "reasons": sorted(reasons), "samples": len(inside),
                "period_ms": self.PERIOD_MS}


def max_over_ranks(value: float, device) -> float:
    """The largest value over all ranks (the whole job's step time); the value
    itself with one rank.  device: where the collective's tensor lives."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank: float, world: int, t_step_max: float) -> float:
    """Throughput of the whole job: every rank's replica does flops_per_rank per
    step, and the job's step takes the slowest rank's time."""
    return flops_per_rank * world / t_step_max / 1e12


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def oracle_product(shape):
    """Keyword arguments selecting the oracle's product for the workload's
    dtype: the MX-FP8 product for an mxfp8 block, the exact one otherwise."""
    if shape.dtype == "mxfp8":
        import oracle.fp8 as fp8
        return {"mm": fp8.mx_product_bf16}
    return {}


def oracle_rate(shape, recompute) -> float:
    """The oracle's FLOP/s on a small calibration sample of the workload (one
    sequence per sub-batch, at most 64 tokens).  Fixed costs weigh more on so
    small a sample, so the rate errs low and the samples sized from it small."""
    import oracle
    from synth import block_inputs
    cal = shape.replace(batch=shape.sub_batches, seq=min(shape.seq, 64))
    inp = block_inputs(cal, seed=0)
    t0 = time.perf_counter()
    oracle.run_step(cal, inp, mode=recompute, **oracle_product(shape))
    return flops_fine(cal, recompute) / max(time.perf_counter() - t0, 1e-6)


def oracle_sample(shape, recompute, seconds: float, rate: float):
    """The largest sample of the workload whose oracle step should take at most
    `seconds` at `rate` FLOP/s: its first sequences, a multiple of the
    sub-batch count; when one sequence per sub-batch is already too much, those
    sequences shortened (halved down to 8 tokens; the FFN is row-wise, the
    attention per sequence, so a shorter sequence is a smaller instance)."""
    fits = lambda s: flops_fine(s, recompute) / rate <= seconds
    s = shape.replace(batch=shape.sub_batches)
    while s.seq > 8 and not fits(s):
        s = s.replace(seq=max(8, s.seq // 2))
    nsb = shape.sub_batches
    while (s.seq == shape.seq and s.batch + nsb <= shape.batch
           and fits(s.replace(batch=s.batch + nsb))):
        s = s.replace(batch=s.batch + nsb)
    return s


def sample_text(sample, shape) -> str:
    return "%d of %d sequences, %d of %d tokens each" % (sample.batch, shape.batch, sample.seq,
                                                          shape.seq)


REFERENCE_SECONDS = 150.0  # the whole --impl reference run (warm-up and timed steps)


def run_reference(args, shape):
    """The oracle as it stands, on this host's cores, each step on a bounded
    sample sized so that all warm-up and timed steps take about
    REFERENCE_SECONDS."""
    import oracle
    from synth import block_inputs
    rank, world, _ = dist_env()
    if rank != 0:
        return
    per_step = REFERENCE_SECONDS / max(args.steps + args.warmup, 1)
    sample = oracle_sample(shape, args.recompute, per_step, oracle_rate(shape, args.recompute))
    inp = block_inputs(sample, seed=0)
    # the calibration rate can be off for the sample taken: time one step of it
    # (untimed, like the warm-up) and shrink it while it runs well over budget
    while True:
        t0 = time.perf_counter()
        oracle.run_step(sample, inp, mode=args.recompute, **oracle_product(shape))
        if time.perf_counter() - t0 <= 1.25 * per_step or (
                sample.batch == shape.sub_batches and sample.seq <= 8):
            break
        if sample.batch > shape.sub_batches:
            sample = sample.replace(batch=sample.batch - shape.sub_batches)
        else:
            sample = sample.replace(seq=max(8, sample.seq // 2))
        inp = block_inputs(sample, seed=0)
    for _ in range(args.warmup):
        oracle.run_step(sample, inp, mode=args.recompute, **oracle_product(shape))
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.run_step(sample, inp, mode=args.recompute, **oracle_product(shape))
    dt = (time.perf_counter() - t0) / args.steps
    value = flops_fine(sample, args.recompute) / dt / 1e12
    cores = len(os.sched_getaffinity(0))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": 0, "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded normal inputs, seed 0)",
            "config": {"workload": args.workload, "batch_sample": sample.batch,
                       "seq_sample": sample.seq, "recompute": args.recompute},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": sample_text(sample, shape) + " per step"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def cpu_baseline(shape, recompute):
    """Oracle timed on a bounded sample (rank 0, N = 1 only): whole steps on a
    sample of the workload of about 5 s each, repeated until about 10 s of host
    work."""
    import oracle
    from synth import block_inputs
    sample = oracle_sample(shape, recompute, 5.0, oracle_rate(shape, recompute))
    inp = block_inputs(sample, seed=0)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.run_step(sample, inp, mode=recompute, **oracle_product(shape))
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= 10.0 or reps >= 50:
            break
    return {"value": flops_fine(sample, recompute) * reps / dt / 1e12, "unit": "TFLOP/s",
            "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": "%d steps on %s (%.1f s, fp64 numpy)" % (
                reps, sample_text(sample, shape), dt)}


def _launch_aggregate(rows, family):
    """Aggregate of the kernel-table rows of one family: algorithmic work and
    CUDA-event time summed over its launches (one each)."""
    sel = [r for r in rows if r["family"] == family]
    work = sum(r["algorithmic"] for r in sel)
    t = sum(r["avg_us"] for r in sel) * 1e-6
    return sel, work, t


def roofline_entries(rows, pk, workload):
    """The roofline objects of the bench line, from the kernel table."""
    out = {}
    sel, fl, t = _launch_aggregate(rows, "gemm")
    if sel:
        n = len(sel)
        ach = fl / t / 1e12
        out["roofline"] = {
            "kernel": "gemm_tc_kernel (tcgen05 GEMM, all instantiations): one sub-batch's "
                      "%d GEMMs of one layer, each launched alone" % n,
            "bound": "tensor", "achieved": ach, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
            "frac": ach / pk["bf16_tflops"], "traffic": recorded_traffic(workload),
            "peak_source": pk["source"] + " bf16 GEMM (burst, kernel timed alone)",
            "algorithmic_flops_per_launch": fl / n, "avg_launch_s": t / n,
            "launches": [{"gemm": r["kernel"], "shape": r["shape"], "us": r["avg_us"],
                          "frac": r["frac"]} for r in sel]}
    sel, fl, t = _launch_aggregate(rows, "attn_bwd")
    if sel:
        ach = fl / t / 1e12
        out["roofline_attention_bwd"] = {
            "kernel": "attention backward (attn_delta_kernel + attn_bwd_dq_tc_kernel + "
                      "attn_bwd_dkv_tc_kernel), %s" % sel[0]["shape"],
            "bound": "tensor", "achieved": ach, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
            "frac": ach / pk["bf16_tflops"], "traffic": None,
            "algorithmic_flops_per_launch": fl, "avg_launch_s": t}
    sel, fl, t = _launch_aggregate(rows, "attn_fwd")
    if sel:
        out["roofline_attention_fwd_frac"] = fl / t / 1e12 / pk["bf16_tflops"]
    mx = [r for r in rows if r["family"] == "mx"]
    if mx:
        g = [r for r in mx if r["bound"] == "tensor"][0]
        out["fp8_gemm"] = {
            "kernel": "gemm_tc_kernel MX variant (tcgen05 kind::mxf8f6f4, block-32 UE8M0 "
                      "scales): %s" % g["kernel"], "shape": g["shape"], "bound": "tensor",
            "achieved": g["achieved"], "unit": "TFLOP/s", "peak": g["peak"], "frac": g["frac"],
            "peak_source": pk["source"] + " bf16 burst x 2 (nominal dense FP8 / BF16 rate)",
            "avg_launch_s": g["avg_us"] * 1e-6,
            "quantize": [{"kernel": r["kernel"], "shape": r["shape"], "us": r["avg_us"],
                          "GB/s": r["achieved"], "frac": r["frac"]} for r in mx
                         if r["bound"] == "hbm"]}
    return out


def mx_table(shape, pk, reps=20):
    """The MX-FP8 GEMM variant at the workload's FFN column-GEMM shape (per
    sub-batch): quantisers of the two operands (HBM-bound: read the bf16 rows,
    write codes + scales) and the block-scaled GEMM with the bias + GeLU
    epilogue, timed alone like kernel_table's rows.  The GEMM's peak is the
    measured bf16 burst peak times 2, the ratio of the nominal dense FP8 and
    BF16 tensor rates (4.5 / 2.25 PFLOP/s)."""
    import ctypes

    import torch

    import tensor_model_transformer_tp_gb300 as oz
    L = oz.lib()
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    L.oases_mx_scale_bytes.argtypes = [i32, i32]
    L.oases_mx_scale_bytes.restype = sz
    L.oases_mx_quantize.argtypes = [vp, i64, i32, i32, i32, i32, vp, i64, vp, vp]
    L.oases_mx_gemm.argtypes = [i32, i32, i32, vp, i64, vp, vp, i64, vp, i32, vp, i64, i32, vp, vp,
                                vp, i64, vp]
    dev = torch.device("cuda", torch.cuda.current_device())
    st = torch.cuda.current_stream(dev)
    sp = st.cuda_stream
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    Ms, H = shape.rows // shape.sub_batches, shape.hidden
    N = shape.ffn if shape.kind in ("ffn", "layer") else 3 * H
    u = torch.randn(Ms, H, device=dev).to(torch.bfloat16)
    w = (torch.randn(N, H, device=dev) * 0.02).to(torch.bfloat16)
    b = (torch.randn(N, device=dev) * 0.02).to(torch.bfloat16)
    qa = torch.empty(Ms, H, dtype=torch.uint8, device=dev)
    qb = torch.empty(N, H, dtype=torch.uint8, device=dev)
    sfa = torch.empty(L.oases_mx_scale_bytes(Ms, H), dtype=torch.uint8, device=dev)
    sfb = torch.empty(L.oases_mx_scale_bytes(N, H), dtype=torch.uint8, device=dev)
    C = torch.empty(Ms, N, dtype=torch.bfloat16, device=dev)
    rows = []

    def timed(name, dims, bound, work, peak, launch):
        assert launch() == 0, name
        torch.cuda.synchronize(dev)
        evs = []
        for _ in range(reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            assert launch() == 0, name
            e1.record(st)
            evs.append((e0, e1))
        torch.cuda.synchronize(dev)
        t = sum(a.elapsed_time(c) for a, c in evs) / reps * 1e-3
        unit = "GB/s" if bound == "hbm" else "TFLOP/s"
        ach = work / t / (1e9 if bound == "hbm" else 1e12)
        rows.append({"kernel": name, "shape": dims, "bound": bound, "family": "mx",
                     "avg_us": t * 1e6, "algorithmic": work, "achieved": ach, "unit": unit,
                     "peak": peak, "frac": ach / peak})

    def qbytes(R, K):
        return 2.0 * R * K + R * K + R * K / 32.0

    timed("mx_quantize (transposed, for a weight gradient)", "%dx%d" % (H, Ms), "hbm",
          qbytes(Ms, H), pk["hbm_gbs"],
          lambda: L.oases_mx_quantize(u.data_ptr(), H, H, Ms, 1, 1, qa.data_ptr(), Ms,
                                      sfa.data_ptr(), sp))
    timed("mx_quantize (activation rows)", "%dx%d" % (Ms, H), "hbm", qbytes(Ms, H), pk["hbm_gbs"],
          lambda: L.oases_mx_quantize(u.data_ptr(), H, Ms, H, 1, 0, qa.data_ptr(), H,
                                      sfa.data_ptr(), sp))
    timed("mx_quantize (weight rows)", "%dx%d" % (N, H), "hbm", qbytes(N, H), pk["hbm_gbs"],
          lambda: L.oases_mx_quantize(w.data_ptr(), H, N, H, 1, 0, qb.data_ptr(), H,
                                      sfb.data_ptr(), sp))
    timed("mx_gemm column GEMM + bias + GeLU (E4M3 x E4M3, fp32 accumulate)",
          "%dx%dx%d" % (Ms, N, H), "tensor", 2.0 * Ms * N * H, 2.0 * pk["bf16_tflops"],
          lambda: L.oases_mx_gemm(Ms, N, H, qa.data_ptr(), H, sfa.data_ptr(), qb.data_ptr(), H,
                                  sfb.data_ptr(), 2, C.data_ptr(), N, 1, None, b.data_ptr(),
                                  None, 0, sp))
    return rows


def kernel_table(shape, pk, reps=20):
    """Each kernel of one sub-batch's step (of one layer), launched alone through
    the kernel entry points (oases_debug.h) at the workload's per-sub-batch
    shape, L2 flushed before every launch, CUDA-event time averaged over reps
    launches.  HBM-bound kernels report algorithmic bytes / time against the
    measured HBM copy bandwidth; tensor-core kernels algorithmic FLOPs / time
    against the measured bf16 burst peak.  Returns one dict per kernel; its
    "family" is gemm, attn_fwd, attn_bwd or hbm."""
    import ctypes

    import torch

    import tensor_model_transformer_tp_gb300 as oz
    L = oz.lib()
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    L.oases_debug_gemm.argtypes = [i32, i32, i32, i32, vp, i64, i32, vp, i64, i32, i32, vp, i64,
                                   i32, vp, vp, vp, i64, i32, vp]
    L.oases_debug_layer_norm.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, f32, i32, vp]
    L.oases_debug_layer_norm_bwd_scratch_bytes.argtypes = [i32, i32]
    L.oases_debug_layer_norm_bwd_scratch_bytes.restype = sz
    L.oases_debug_layer_norm_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, vp,
                                             sz, vp]
    L.oases_debug_bias_grad_scratch_bytes.argtypes = [i32, i32]
    L.oases_debug_bias_grad_scratch_bytes.restype = sz
    L.oases_debug_bias_grad.argtypes = [vp, i64, i32, i32, i32, vp, vp, sz, vp]
    L.oases_debug_shard_sum.argtypes = [vp, i64, i32, vp, vp, vp, i32, i32, i32, vp]
    L.oases_debug_attention.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                        i32, vp]
    dev = torch.device("cuda", torch.cuda.current_device())
    st = torch.cuda.current_stream(dev)
    sp = st.cuda_stream
    bf = torch.bfloat16
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    Ms, H, w = shape.rows // shape.sub_batches, shape.hidden, shape.w
    rows = []

    def rnd(*dims, dtype=bf, scale=1.0):
        return (torch.randn(*dims, device=dev) * scale).to(dtype)

    def timed(name, dims, bound, work, launch, family):
        status = launch()
        assert status == 0, (name, status)
        torch.cuda.synchronize(dev)
        evs, bad = [], 0
        for _ in range(reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            bad += launch() != 0
            e1.record(st)
            evs.append((e0, e1))
        torch.cuda.synchronize(dev)
        assert bad == 0, (name, "failed launches", bad)
        t = sum(a.elapsed_time(b) for a, b in evs) / reps * 1e-3
        if bound == "hbm":
            ach, peak, unit = work / t / 1e9, pk["hbm_gbs"], "GB/s"
        else:
            ach, peak, unit = work / t / 1e12, pk["bf16_tflops"], "TFLOP/s"
        rows.append({"kernel": name, "shape": dims, "bound": bound, "family": family,
                     "avg_us": t * 1e6, "algorithmic": work, "achieved": ach, "unit": unit,
                     "peak": peak, "frac": ach / peak})

    def gemm(name, M, N, K, A, lda, ak, B, ldb, bk, epi, C, ldc, c_f32, C2=None, bias=None,
             aux=None, ld_aux=0):
        p = lambda t: t.data_ptr() if t is not None else None
        timed(name, "%dx%dx%d" % (M, N, K), "tensor", 2.0 * M * N * K,
              lambda: L.oases_debug_gemm(M, N, K, 1, p(A), lda, ak, p(B), ldb, bk, epi, p(C), ldc,
                                         0 if c_f32 else 1, p(C2), p(bias), p(aux), ld_aux, 2, sp),
              "gemm")

    x = rnd(Ms, H)
    gam, bet = rnd(H, scale=0.1) + 1, rnd(H, scale=0.1)
    u = torch.empty_like(x)
    mean = torch.empty(Ms, device=dev)
    rstd = torch.empty(Ms, device=dev)
    timed("ln_fwd", "%dx%d" % (Ms, H), "hbm", 4.0 * Ms * H + 4.0 * H + 8.0 * Ms,
          lambda: L.oases_debug_layer_norm(x.data_ptr(), gam.data_ptr(), bet.data_ptr(),
                                           u.data_ptr(), mean.data_ptr(), rstd.data_ptr(), Ms, H,
                                           1e-5, 1, sp), "hbm")
    dy = rnd(Ms, H)
    du = torch.empty(Ms, H, device=dev)
    if shape.kind in ("attn", "layer"):
        nh, d = shape.heads, H // shape.heads
        Bs, S = shape.batch // shape.sub_batches, shape.seq
        wqkv, bqkv = rnd(3 * H, H, scale=0.02), rnd(3 * H, scale=0.02)
        wo, bo = rnd(H, H, scale=0.02), rnd(H, scale=0.02)
        qkv = torch.empty(Ms, 3 * H, dtype=bf, device=dev)
        y = torch.empty(Ms, H, dtype=bf, device=dev)
        dwqkv = torch.zeros(3 * H, H, device=dev)
        dwo = torch.zeros(H, H, device=dev)
        gemm("qkv_gemm_bias (F_i fwd)", Ms, 3 * H, H, u, H, 1, wqkv, H, 1, 1, qkv, 3 * H, False,
             bias=bqkv)
        gemm("qkv_gemm_bias (R_i)", Ms, 3 * H, H, u, H, 1, wqkv, H, 1, 1, qkv, 3 * H, False,
             bias=bqkv)
        qkv.normal_()
        o = torch.empty(Ms, H, dtype=bf, device=dev)
        lse = torch.empty(nh, Ms, device=dev)
        do = rnd(Ms, H)
        delta = torch.empty(nh, Ms, device=dev)
        dqkv = torch.empty(Ms, 3 * H, dtype=bf, device=dev)
        causal = 1.0 if shape.causal else 2.0
        dims = "batch %d x seq %d, %d heads of %d" % (Bs, S, nh, d)
        timed("attention fwd (tcgen05)", dims, "tensor", 2.0 * Bs * S * S * H * causal,
              lambda: L.oases_debug_attention(qkv.data_ptr(), o.data_ptr(), lse.data_ptr(), None,
                                              None, None, Bs, S, nh, d, int(shape.causal), 1, 0, 2,
                                              sp), "attn_fwd")
        gemm("out_proj_shard_sum_bias_resid (F_j + C_i(F))", Ms, H, H, o, H, 1, wo, H, 1, 3, y, H,
             False, bias=bo, aux=x, ld_aux=H)
        gemm("dWo += dy^T o (fp32 reduce-add)", H, H, Ms, dy, H, 0, o, H, 0, 5, dwo, H, True)
        gemm("dO = dy Wo (B_j)", Ms, H, H, dy, H, 1, wo, H, 0, 0, do, H, False)
        timed("attention bwd (delta + dQ + dK/dV)", dims, "tensor", 5.0 * Bs * S * S * H * causal,
              lambda: L.oases_debug_attention(qkv.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                              do.data_ptr(), delta.data_ptr(), dqkv.data_ptr(), Bs,
                                              S, nh, d, int(shape.causal), 1, 1, 0, sp), "attn_bwd")
        gemm("dWqkv += dqkv^T u (fp32 reduce-add)", 3 * H, H, Ms, dqkv, 3 * H, 0, u, H, 0, 5,
             dwqkv, H, True)
        gemm("du = dqkv Wqkv (C_i(B), fp32)", Ms, H, 3 * H, dqkv, 3 * H, 1, wqkv, H, 0, 0, du, H,
             True)
        del wqkv, qkv, dwqkv, dwo, dqkv
    if shape.kind in ("ffn", "layer"):
        F = shape.ffn
        w1, b1 = rnd(F, H, scale=0.02), rnd(F, scale=0.02)
        w2, b2 = rnd(H, F, scale=0.02), rnd(H, scale=0.02)
        h, g_ = torch.empty(Ms, F, dtype=bf, device=dev), torch.empty(Ms, F, dtype=bf, device=dev)
        y = torch.empty(Ms, H, dtype=bf, device=dev)
        dw1 = torch.zeros(F, H, device=dev)
        dw2 = torch.zeros(H, F, device=dev)
        da = torch.empty(Ms, F, dtype=bf, device=dev)
        gemm("col_gemm_bias_gelu (F_i fwd)", Ms, F, H, u, H, 1, w1, H, 1, 2, h, F, False, bias=b1)
        gemm("col_gemm_bias_gelu+gelu' (R_i)", Ms, F, H, u, H, 1, w1, H, 1, 2, h, F, False, C2=g_,
             bias=b1)
        gemm("row_gemm_shard_sum_bias_resid (F_j + C_i(F))", Ms, H, F, h, F, 1, w2, F, 1, 3, y, H,
             False, bias=b2, aux=x, ld_aux=H)
        gemm("dW2 += dy^T h (fp32 reduce-add)", H, F, Ms, dy, H, 0, h, F, 0, 5, dw2, F, True)
        gemm("dA = (dy W2) * gelu' (B_j)", Ms, F, H, dy, H, 1, w2, F, 0, 4, da, F, False, aux=g_,
             ld_aux=F)
        gemm("dW1 += dA^T u (fp32 reduce-add)", F, H, Ms, da, F, 0, u, H, 0, 5, dw1, H, True)
        gemm("du = dA W1 (C_i(B), fp32)", Ms, H, F, da, F, 1, w1, H, 0, 0, du, H, True)
        db = torch.zeros(F, device=dev)
        nb = L.oases_debug_bias_grad_scratch_bytes(Ms, F)
        scratch = torch.empty(nb, dtype=torch.uint8, device=dev)
        timed("bias_grad db1 = colsum(dA)", "%dx%d" % (Ms, F), "hbm", 2.0 * Ms * F + 8.0 * F,
              lambda: L.oases_debug_bias_grad(da.data_ptr(), F, Ms, F, 1, db.data_ptr(),
                                              scratch.data_ptr(), nb, sp), "hbm")
        part = torch.randn(w, Ms, H, device=dev)
        timed("shard_sum (separate C_i(F), w=%d)" % w, "%dx%d" % (Ms, H), "hbm",
              4.0 * w * Ms * H + 2.0 * H + 4.0 * Ms * H,
              lambda: L.oases_debug_shard_sum(part.data_ptr(), Ms * H, w, b2.data_ptr(),
                                              x.data_ptr(), y.data_ptr(), Ms, H, 1, sp), "hbm")
        del w1, w2, h, g_, dw1, dw2, da, part
    dx = torch.empty(Ms, H, dtype=bf, device=dev)
    dgam, dbet = torch.zeros(H, device=dev), torch.zeros(H, device=dev)
    nl = L.oases_debug_layer_norm_bwd_scratch_bytes(Ms, H)
    lscr = torch.empty(nl, dtype=torch.uint8, device=dev)
    du.normal_()
    timed("ln_bwd (+ residual, dgamma, dbeta)", "%dx%d" % (Ms, H), "hbm",
          (4.0 + 3 * 2.0) * Ms * H + 8.0 * Ms + 2.0 * H + 16.0 * H,
          lambda: L.oases_debug_layer_norm_bwd(du.data_ptr(), x.data_ptr(), mean.data_ptr(),
                                               rstd.data_ptr(), gam.data_ptr(), dy.data_ptr(),
                                               dx.data_ptr(), dgam.data_ptr(), dbet.data_ptr(),
                                               Ms, H, 1, lscr.data_ptr(), nl, sp), "hbm")
    return rows


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="stack4_bf16_h2560")
    ap.add_argument("--recompute", default="fine", choices=["fine", "full", "none", "selective"])
    ap.add_argument("--sub-batches", type=int, default=None)
    ap.add_argument("--dtype", default=None, choices=["bf16", "mxfp8"],
                    help="override the workload's dtype (mxfp8: bf16 storage, MX-FP8 GEMMs); "
                         "the headline is the workload's own bf16")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch the step directly, not as a CUDA graph")
    ap.add_argument("--reduce", default="fused", choices=["fused", "separate"],
                    help="shard sums fused into the GEMMs or as separate reduction kernels")
    ap.add_argument("--kernels", action="store_true",
                    help="instead of the step: time each kernel alone at the workload's "
                         "per-sub-batch shape and print one JSON line per kernel")
    ap.add_argument("--reps", type=int, default=20,
                    help="--kernels: timed launches per kernel (after one untimed launch)")
    args = ap.parse_args()
    from synth import SHAPES
    shape = SHAPES[args.workload]
    if args.sub_batches:
        shape = shape.replace(sub_batches=args.sub_batches)
    if args.dtype:
        shape = shape.replace(dtype=args.dtype)
    if args.impl == "reference":
        run_reference(args, shape)
        return
    if args.kernels:
        import torch
        from tensor_model_transformer_tp_gb300 import build_library
        build_library()
        torch.cuda.set_device(0)
        pk = peaks()
        with ClockSampler(0) as clk:
            rows = kernel_table(shape, pk, reps=args.reps) + mx_table(shape, pk, reps=args.reps)
        for r in rows:
            r["workload"] = args.workload
            r["peak_source"] = pk["source"]
            print(json.dumps(r), flush=True)
        print(json.dumps({"clocks": clk.summary()}), flush=True)
        return

    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from synth import block_inputs
    from tensor_model_transformer_tp_gb300 import build_library, oases_last_launch_count
    from tensor_model_transformer_tp_gb300.device import DeviceBlock
    build_library()
    inp = block_inputs(shape, seed=0)
    blk = DeviceBlock(shape, inp["layers"], recompute=args.recompute,
                      device="cuda:%d" % local, reduce=args.reduce)
    x, g = blk.tensor(inp["x"]), blk.tensor(inp["g"])
    y, dx = blk.empty_like_io(), blk.empty_like_io()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def barrier():
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(max(3, args.warmup)):
        blk.step(x, g, y, dx)
    launches = oases_last_launch_count()
    # The timed step replays a CUDA graph captured from one oases_stack_step
    # call: the same kernels, stream fork/join and programmatic dependencies,
    # without the per-launch host cost.  Weight gradients keep accumulating.
    graph = None
    if not args.no_graph:
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        cap = blk.s0
        with torch.cuda.stream(cap):
            graph.capture_begin(capture_error_mode="relaxed")
            blk.step(x, g, y, dx)
            graph.capture_end()
        for _ in range(max(3, args.warmup)):
            graph.replay()
    xh = x.cpu().pin_memory()
    gh = g.cpu().pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    dxh = torch.empty_like(xh).pin_memory()
    for _ in range(2):
        blk.step(xh, gh, yh, dxh)
    barrier()
    # clocks are sampled over both timed regions (device-resident and end to end)
    with ClockSampler(local) as clk:
        clk.mark_start()
        evs = []
        for _ in range(args.steps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(blk.s0)
            if graph is not None:
                with torch.cuda.stream(blk.s0):
                    graph.replay()
            else:
                blk.step(x, g, y, dx)
            e1.record(blk.s0)
            evs.append((e0, e1))
            with torch.cuda.stream(blk.s0):
                flush.zero_()
        barrier()
        clk.mark_end()
        t_step = sum(a.elapsed_time(b) for a, b in evs) * 1e-3 / args.steps
        t_step = max_over_ranks(t_step, dev)

        # end to end: host (pinned) buffers through the same C-ABI call
        barrier()
        clk.mark_start()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(blk.s0)
        for _ in range(args.steps):
            blk.step(xh, gh, yh, dxh)
        e1.record(blk.s0)
        barrier()
        clk.mark_end()
    t_e2e = max_over_ranks(e0.elapsed_time(e1) * 1e-3 / args.steps, dev)
    fl = flops_fine(shape, args.recompute)
    value = whole_job_tflops(fl, world, t_step)
    io = shape.rows * shape.hidden * (4 if shape.dtype == "f32" else 2)

    pk = peaks()
    rows = kernel_table(shape, pk) + mx_table(shape, pk)
    out = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
           "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": t_step * 1e3,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": shape.dtype, "data": "synthetic (seeded normal inputs, seed 0)",
           "config": {"workload": args.workload, "kind": shape.kind, "batch": shape.batch,
                      "seq": shape.seq, "hidden": shape.hidden, "ffn": shape.ffn,
                      "heads": shape.heads, "w": shape.w, "sub_batches": shape.sub_batches,
                      "n_layers": shape.n_layers, "recompute": args.recompute,
                      "reduce": args.reduce,
                      "parallelism": "replicas" if world > 1 else "single-gpu",
                      "launch": "cuda-graph" if not args.no_graph else "direct",
                      "l2": "flushed between timed steps (256 MiB write)"},
           "pct_bf16_peak": 100.0 * value / world / pk["bf16_tflops"],
           "pct_bf16_peak_of": "%s dense bf16 GEMM peak (burst), %.1f TFLOP/s per GPU" % (
               pk["source"], pk["bf16_tflops"]),
           "pct_bf16_sustained": 100.0 * value / world / pk["bf16_tflops_sustained"],
           "pct_bf16_sustained_of": "%s sustained bf16 GEMM rate, %.1f TFLOP/s per GPU" % (
               pk["source"], pk["bf16_tflops_sustained"]),
           "e2e": {"value": whole_job_tflops(fl, world, t_e2e), "unit": "TFLOP/s",
                   "h2d_bytes_per_step": 2 * io, "d2h_bytes_per_step": 2 * io},
           "gpu_launches": launches * args.steps,
           "clocks": clk.summary()}
    out.update(roofline_entries(rows, pk, args.workload))
    if world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(shape, args.recompute)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
