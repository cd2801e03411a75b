"""Benchmark of the Fairy2i widely-linear 2-bit layer on B300.

Workload (the decode metric): batch-1 decode through the seven LLaMA-2-7B
projections of a decoder block (q/k/v/o 4096x4096, gate/up 11008x4096, down
4096x11008 as real matrices; T = 2), for 32 distinct blocks = the 224
projections of the 7B stack, 1.64 GB of packed codes and scales, far above
the 126 MB L2, so no flush is needed between steps.  One step = one token
through all 224 projections, one grouped launch per block (7 layers each).

value      = packed bytes streamed per step / device time per step (GB/s)
e2e        = the same bytes / time per step including the host->device copy of
             every projection's activation row and the device->host copy of
             every output row (pinned host buffers), the host waiting for the
             step's outputs; copies of a block overlap the other blocks' launches
roofline   = the decode kernel's average launch: packed bytes of one block
             (51,273,728 B) / launch time, against the measured HBM copy peak
cpu_baseline / --impl reference = the oracle (plain C, double precision,
             one thread) on a sample of output rows of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from bit_complex_valued_fairy2i_b300 import inputs  # noqa: E402

METRIC = "2-bit WL-complex GEMV weight GB/s vs HBM peak; prefill GEMM TFLOP/s"
UNIT = "GB/s"
T_STAGES = 2
BLOCKS = inputs.LLAMA2_7B_BLOCKS
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one decode launch of
# this workload per decode kernel, from ncu captures (must be re-measured whenever
# that kernel changes): linear_lut_kernel<2,1> (the capture in
# profiles/linear_lut_decode_llama2_7b_block_M1_T2.md) and linear_mma_kernel<4,1,16>.
DECODE_TRAFFIC_BYTES = {"lut": 51_394_048, "mma": 51_399_680, "auto": 51_399_680}
# decode kernel and arithmetic per --decode-algo (auto = the 2:4-sparse mma.sync decode at M = 1 on
# layout 2; lut = the table-lookup decode on layout 3)
DECODE_KERNELS = {
    "lut": ("linear_lut_kernel<2,1> (table lookup, layout 3)",
            "fp16 table entries (fp32 sums of 8 bf16 activations rounded once), fp32 accumulate"),
    "auto": ("linear_mma_kernel<4,1,16> (2:4-sparse mma.sync)",
             "bf16 (2:4-sparse mma.sync: code signs as bf16 +-2, bf16 x), fp32 accumulate"),
    "mma": ("linear_mma_kernel<4,1,16> (2:4-sparse mma.sync)",
            "bf16 (2:4-sparse mma.sync: code signs as bf16 +-2, bf16 x), fp32 accumulate"),
    "tcgen05_sp": ("linear_tc_decode_kernel (2:4-sparse tcgen05.mma.sp)",
                   "e4m3 (2:4-sparse tcgen05.mma.sp: code signs as e4m3 +-1, x as two exact e4m3 terms), "
                   "fp32 accumulate"),
    "addsub": ("linear_addsub_kernel (CUDA cores)", "fp32 adds/subtracts of bf16 x"),
}
WORKLOAD = ("llama2-7b decode GEMV, M=1, T=2: 7 projections per block x 32 distinct blocks "
            "(224 projections, 1.64 GB packed > L2), one grouped launch per block")


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        # raw samples go to $FAIRY2I_CLOCKS_DIR (default: the system temp directory); the JSON
        # line carries their summary
        out_dir = os.environ.get("FAIRY2I_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"fairy2i_clocks_gpu{index}_{os.getpid()}.csv")

    def one_shot(self):
        """One read of the same fields (the polling loop may take no sample in a short region)."""
        try:
            out = subprocess.run(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                  "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=10)
            with open(self.path, "a") as f:
                f.write(out.stdout)
        except (OSError, subprocess.SubprocessError):
            pass

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            open(self.path, "w").close()
            self.one_shot()
            self.fh = open(self.path, "a")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()
            self.one_shot()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not torch.distributed.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        torch.distributed.init_process_group(backend)
    return world, rank, local


def _barrier(world):
    if world > 1:
        torch.distributed.barrier()


def _max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# oracle on a sample of rows (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------
def _oracle_sample_setup(max_rows_per_proj: int, seed_config: int = 5, part: int = 0, parts: int = 1):
    """Oracle-quantized rows of block 0 (rows j = 0, s, 2s, ... of each projection; with
    `parts` > 1 only share `part` of them)."""
    import oracle
    samples = []
    for pi, (name, out_f, in_f) in enumerate(inputs.LLAMA2_7B_BLOCK):
        n, m = out_f // 2, in_f // 2
        step = max(1, n // max_rows_per_proj)
        rows = np.array_split(np.arange(0, n, step)[:max_rows_per_proj], parts)[part]
        if len(rows) == 0:
            continue
        R = inputs.weight_R(seed_config, pi, out_f, in_f)
        Rs = torch.cat([R[rows], R[n + rows]]).numpy()
        Uo, Wo = oracle.convert_f32(Rs)
        qU, qW = oracle.quantize(Uo, T_STAGES), oracle.quantize(Wo, T_STAGES)
        x = inputs.bf16_bits(inputs.activations(seed_config, pi, 1, in_f))
        # packed bytes these rows stand for: 2T planes of 2-bit codes + 4T fp32 scales per row
        nbytes = len(rows) * (2 * T_STAGES * m // 4 + 4 * T_STAGES * 4)
        samples.append((qU, qW, x, nbytes))
    return samples


def _oracle_run(samples):
    import oracle
    t0 = time.perf_counter()
    nbytes = 0
    for qU, qW, x, nb in samples:
        oracle.linear_mulfree(qU, qW, x)
        nbytes += nb
    return nbytes, time.perf_counter() - t0


def _oracle_worker(rows, part, parts, steps, warmup, ready, go, results):
    """One host core: its share of the sampled rows, `steps` timed passes after `go`."""
    samples = _oracle_sample_setup(rows, part=part, parts=parts)
    for _ in range(warmup):
        _oracle_run(samples)
    ready.put(part)
    go.wait()
    t0 = time.perf_counter()
    nb = 0
    for _ in range(steps):
        nb += _oracle_run(samples)[0]
    results.put((nb, time.perf_counter() - t0))


def _oracle_all_cores(rows: int, steps: int, warmup: int):
    """The oracle (unchanged, single-threaded loops) on every host core at once: one
    spawned process per core, each with its own share of the sampled rows, started
    together; returns (bytes, seconds of the slowest process, cores)."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    cores = os.cpu_count() or 1
    ready, results, go = ctx.Queue(), ctx.Queue(), ctx.Event()
    procs = [ctx.Process(target=_oracle_worker, args=(rows, i, cores, steps, warmup, ready, go, results))
             for i in range(cores)]
    for p in procs:
        p.start()
    for _ in procs:
        ready.get(timeout=600)
    go.set()
    out = [results.get(timeout=600) for _ in procs]
    for p in procs:
        p.join(timeout=60)
    return sum(o[0] for o in out), max(o[1] for o in out), cores


def _cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def cpu_baseline(target_s: float = 10.0):
    """The oracle on sampled rows of the workload: one thread, then the same rows
    dealt out to one process per host core (spawned; the oracle itself is unchanged)."""
    rows = 8
    samples = _oracle_sample_setup(rows)
    nb, dt = _oracle_run(samples)
    rows = max(1, min(2048, int(rows * target_s / max(dt, 1e-6))))
    samples = _oracle_sample_setup(rows)
    nb, dt = _oracle_run(samples)
    single = nb / dt / 1e9
    cores = os.cpu_count() or 1
    result = {"value": single, "unit": UNIT, "cores": 1, "kind": "oracle",
              "sample": f"oracle decode (plain C, fp64) of {rows} evenly spaced output rows of each of "
                        f"the 7 projections of block 0, M=1, T=2; {nb} packed-equivalent bytes",
              "cpu_model": _cpu_model(), "nproc": cores, "single_thread_GBps": single}
    if cores > 1:
        nbm, dtm, cores = _oracle_all_cores(rows, 1, 1)
        result.update({"value": nbm / dtm / 1e9, "cores": cores, "all_cores_GBps": nbm / dtm / 1e9,
                       "sample": result["sample"] + f"; then the same rows dealt out to {cores} processes"})
    return result


def run_reference(args, world, rank):
    """The oracle (the only executable statement of the method) on the machine's host cores:
    each step decodes a sample of output rows of the workload, dealt out to one spawned
    process per core (the oracle's own single-threaded loops, unchanged)."""
    if rank != 0:
        return
    steps_total = args.steps + args.warmup
    budget_s = 120.0
    cores = os.cpu_count() or 1
    rows = 4
    samples = _oracle_sample_setup(rows)
    nb, dt = _oracle_run(samples)
    per_row = dt / rows
    rows = max(1, min(2048, int(budget_s * cores / steps_total / max(per_row, 1e-9))))
    nbytes, dt, cores = _oracle_all_cores(rows, args.steps, args.warmup)
    value = nbytes / dt / 1e9
    sample = (f"each step: oracle decode (plain C, fp64) of {rows} evenly spaced output rows of each "
              f"of the 7 projections of block 0, M=1, T=2, rows dealt out to {cores} processes")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": sample},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
                         "cpu_model": _cpu_model()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def decode_layout(algo: str) -> int:
    return 3 if algo == "lut" else 2


# GPU clock cycles of the idle kernel queued ahead of a timed launch, so that the host has issued
# the launch (and its output allocations and argument checks) before the GPU reaches the first
# event: the events then bracket device work only (about 100 us at 2 GHz).
HOST_LEAD_CYCLES = 200_000


def build_stack(f2i, blocks: int, dev, T: int = T_STAGES, layout: int = 2):
    """Convert + quantize the stack on the GPU; times both (events around the launches, with an
    idle kernel queued ahead so that host work does not fall between the events)."""
    stack = []
    conv_ms = quant_ms = 0.0
    conv_bytes = quant_bytes = 0
    e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    # untimed warm-up of both kernels (the first launches of a process load them)
    name, out_f, in_f = inputs.LLAMA2_7B_BLOCK[0]
    R = inputs.weight_R(5, 0, out_f, in_f, device=dev)
    U, W = f2i.convert(R)
    f2i.quantize(U, W, T, check=False, layout=layout)
    torch.cuda.synchronize()
    del R, U, W
    for b in range(blocks):
        layers = []
        for pi, (name, out_f, in_f) in enumerate(inputs.LLAMA2_7B_BLOCK):
            R = inputs.weight_R(5, 7 * b + pi, out_f, in_f, device=dev)
            torch.cuda._sleep(HOST_LEAD_CYCLES)
            e[0].record()
            U, W = f2i.convert(R)
            e[1].record()
            q = f2i.quantize(U, W, T, check=False, layout=layout)
            e[2].record()
            e[2].synchronize()
            conv_ms += e[0].elapsed_time(e[1])
            quant_ms += e[1].elapsed_time(e[2])
            conv_bytes += R.numel() * 4 * 2  # read R, write U and W
            quant_bytes += R.numel() * 4 + q.nbytes  # read U and W, write codes + scales
            layers.append(q)
            del R, U, W
        stack.append(layers)
    f2i.sync_status()
    return stack, {"convert_GBps": conv_bytes / conv_ms / 1e6, "quantize_GBps": quant_bytes / quant_ms / 1e6,
                   "convert_ms_stack": conv_ms, "quantize_ms_stack": quant_ms}


def prefill_leg(f2i, dev, peaks, steps: int, warmup: int, M: int = 2048):
    """Prefill: the 7 projections of one block at M tokens (1 % outliers x10),
    one grouped call per step, three kernels: the ternary tcgen05 GEMM over
    layout 2 (16 n m T flops per token), and the dense GEMM of the dequantized
    matrix over layout 3 in its two forms: hi + lo bfloat16 terms (16 n m flops
    per token) and one fp16 term against an fp16 copy of x (8 n m flops per
    token; the copy is made by a conversion launch inside the timed call).
    Executed and dense-equivalent TFLOP/s for each; the faster leads."""
    qs2, qs3, xs, ys = [], [], [], []
    flops_tern = flops_dq = flops_dense = 0  # the fp16 form executes flops_dense
    for pi, (name, out_f, in_f) in enumerate(inputs.LLAMA2_7B_BLOCK):
        R = inputs.weight_R(4, pi, out_f, in_f, device=dev)
        U, W = f2i.convert(R)
        qs2.append(f2i.quantize(U, W, T_STAGES, check=False))
        qs3.append(f2i.quantize(U, W, T_STAGES, check=False, layout=3))
        del R, U, W
        xs.append(inputs.activations(4, pi, M, in_f, outliers=True, device=dev))
        ys.append(torch.empty((M, out_f), dtype=torch.float32, device=dev))
        n, m = out_f // 2, in_f // 2
        flops_tern += 16 * n * m * T_STAGES * M
        flops_dq += 16 * n * m * M
        flops_dense += 8 * n * m * M
    f2i.sync_status()
    stream = torch.cuda.current_stream()

    def timed(qs, algo):
        """ms per call over at least `steps` calls and 0.2 s (so that the clock sampler sees the
        sustained, power-capped state of a long prefill), with the clocks seen meanwhile."""
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(warmup):
            f2i.linear_group(qs, xs, ys, algo=algo)
        stop.record(stream)
        torch.cuda.synchronize()
        reps = max(steps, int(200.0 / max(start.elapsed_time(stop) / max(warmup, 1), 1e-3)) + 1)
        with ClockSampler(dev.index if dev.index is not None else 0) as clk:
            start.record(stream)
            for _ in range(reps):
                f2i.linear_group(qs, xs, ys, algo=algo)
            stop.record(stream)
            torch.cuda.synchronize()
        f2i.sync_status()
        return start.elapsed_time(stop) / reps, reps, clk.summary()

    legs = {}
    nt = 2 if M > 256 else 1
    for key, qs, algo, kernel, fl in (("ternary", qs2, "tcgen05", "linear_tcgen05_kernel<8>", flops_tern),
                                      ("dequantized", qs3, "tcgen05_dq", f"linear_dq_kernel<{T_STAGES},{nt},0,0>", flops_dq),
                                      ("dequantized_f16", qs3, "tcgen05_dq16",
                                       f"dq_x16_kernel + linear_dq_kernel<{T_STAGES},{nt},0,1>", flops_dense)):
        ms, reps, clocks = timed(qs, algo)
        tf = fl / (ms * 1e-3) / 1e12
        # the fp16 form runs on the same tensor-core rate as bfloat16 (kind::f16)
        legs[key] = {"algo": algo, "kernel": kernel, "layout": 2 if key == "ternary" else 3, "ms_per_block": ms,
                     "executed_flops_per_block": fl, "tflops_executed": tf,
                     "tflops_dense_equivalent": flops_dense / (ms * 1e-3) / 1e12,
                     "frac_of_bf16_peak": tf / peaks["bf16_tflops"],
                     "frac_of_bf16_sustained": tf / peaks["bf16_tflops_sustained"],
                     "tokens_per_s_per_block": M / (ms * 1e-3), "calls_timed": reps, "clocks": clocks}
    best = min(legs, key=lambda k: legs[k]["ms_per_block"])
    b = legs[best]
    return {"workload": f"llama2-7b block prefill, 7 projections, M={M}, T={T_STAGES}, 1% outliers x10, "
                        "one grouped launch", "kernel": b["kernel"], "algo": b["algo"], "ms_per_block": b["ms_per_block"],
            "executed_flops_per_block": b["executed_flops_per_block"],
            "dense_equivalent_flops_per_block": flops_dense, "tflops_executed": b["tflops_executed"],
            "tflops_dense_equivalent": b["tflops_dense_equivalent"],
            "peak_bf16_tflops": peaks["bf16_tflops"], "frac_of_bf16_peak": b["frac_of_bf16_peak"],
            "peak_bf16_tflops_sustained": peaks["bf16_tflops_sustained"],
            "frac_of_bf16_sustained": b["frac_of_bf16_sustained"], "clocks": b["clocks"],
            "calls_timed": b["calls_timed"],
            "peak_source": peaks["source"], "tokens_per_s_per_block": b["tokens_per_s_per_block"], "steps": steps,
            "by_kernel": legs}


SWEEP_ALGOS = ("lut", "tcgen05_dq", "tcgen05_dq16", "auto_layout3", "mma", "tcgen05", "auto", "tcgen05_sp")


def sweep_leg(f2i, dev, Ms=(1, 2, 4, 8, 16, 32, 64), reps: int = 10, blocks: int = 4, algos=SWEEP_ALGOS):
    """Batched decode sweep: per token count M and per algorithm, the 7 projections of
    `blocks` distinct blocks (205 MB at 4 blocks, above L2), one grouped call per block;
    time per block, weight GB/s and tokens/s-equivalent (eager calls; for AUTO on layout 3 also
    the same calls replayed as a CUDA graph).  "lut", "tcgen05_dq", "tcgen05_dq16" and
    "auto_layout3" read the same weights in layout 3 (the table lookup: one decode launch
    per 2 tokens at T = 2 (the first of 3 for odd M), each with its window-combining launch;
    the dequantized GEMM: one launch with N = M rounded up to 16, in the fp16 form after a
    conversion launch of the activations)."""
    stack, stack3, xs_full = [], [], []
    for b in range(blocks):
        qs, qs3, xb = [], [], []
        for pi, (name, out_f, in_f) in enumerate(inputs.LLAMA2_7B_BLOCK):
            R = inputs.weight_R(3, 7 * b + pi, out_f, in_f, device=dev)
            qs.append(f2i.convert_quantize(R, T_STAGES, check=False))
            qs3.append(f2i.convert_quantize(R, T_STAGES, check=False, layout=3))
            del R
            xb.append(inputs.activations(3, 7 * b + pi, max(Ms), in_f, device=dev))
        stack.append(qs)
        stack3.append(qs3)
        xs_full.append(xb)
    f2i.sync_status()
    nbytes = sum(q.nbytes for q in stack[0])
    out = []
    stream = torch.cuda.current_stream()
    for M in Ms:
        xs = [[x[:M].contiguous() for x in xb] for xb in xs_full]
        ys = [[torch.empty((M, 2 * q.n), dtype=torch.float32, device=dev) for q in qs] for qs in stack]
        row = {"M": M}
        for key in [a for a in algos if a != "tcgen05_sp" or M <= 8]:
            st = stack3 if key in ("lut", "tcgen05_dq", "tcgen05_dq16", "auto_layout3") else stack
            algo = "auto" if key == "auto_layout3" else key

            calls = [f2i.GroupCall(st[b], xs[b], ys[b], algo=algo) for b in range(blocks)]

            def step():
                for c in calls:
                    c()
            for _ in range(3):
                step()
            torch.cuda.synchronize()
            start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            start.record(stream)
            for _ in range(reps):
                step()
            stop.record(stream)
            torch.cuda.synchronize()
            us = start.elapsed_time(stop) / reps / blocks * 1e3
            row[key] = {"us_per_block": round(us, 2), "weight_GBps": round(nbytes / (us * 1e-6) / 1e9, 1),
                         "tokens_per_s_per_block": round(M / (us * 1e-6))}
            if key == "auto_layout3":
                # the same calls replayed as one CUDA graph: the device time per block, without
                # the per-call host work that bounds the eager figure at small M
                # (calls prepared inside the capture: a prepared call keeps the stream it was
                # built on, and the capture runs on a stream of its own)
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph):
                    for b in range(blocks):
                        f2i.GroupCall(st[b], xs[b], ys[b], algo=algo)()
                graph.replay()
                torch.cuda.synchronize()
                start.record(stream)
                for _ in range(reps):
                    graph.replay()
                stop.record(stream)
                torch.cuda.synchronize()
                gus = start.elapsed_time(stop) / reps / blocks * 1e3
                row[key]["graph_us_per_block"] = round(gus, 2)
                row[key]["graph_weight_GBps"] = round(nbytes / (gus * 1e-6) / 1e9, 1)
                row[key]["graph_tokens_per_s_per_block"] = round(M / (gus * 1e-6))
                del graph
        out.append(row)
    f2i.sync_status()
    return {"workload": f"llama2-7b blocks (7 projections each), T=2, {blocks} distinct blocks "
                        f"({blocks * nbytes / 1e6:.0f} MB > L2), one grouped launch per block",
            "bytes_per_block": nbytes, "rows": out}


def stack_leg(f2i, dev, T: int, blocks: int, steps: int, warmup: int, layout: int = 3):
    """The full 32-block LLaMA-2-7B linear stack at T stages: convert + quantize of all
    224 projections (timed per launch), then batch-1 decode of all of them per step
    (CUDA graph of one grouped call per block; layout 3 = the table-lookup decode)."""
    stack, offline = build_stack(f2i, blocks, dev, T, layout)
    nbytes = sum(q.nbytes for layers in stack for q in layers)
    # the same stack through the one-pass convert + quantize (codes written over the first ones)
    fused_ms, e = 0.0, [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    for b in range(blocks):
        for pi, (name, out_f, in_f) in enumerate(inputs.LLAMA2_7B_BLOCK):
            R = inputs.weight_R(5, 7 * b + pi, out_f, in_f, device=dev)
            torch.cuda._sleep(HOST_LEAD_CYCLES)
            e[0].record()
            f2i.convert_quantize(R, T, out=stack[b][pi], check=False, layout=layout)
            e[1].record()
            e[1].synchronize()
            fused_ms += e[0].elapsed_time(e[1])
            del R
    f2i.sync_status()
    offline["convert_quantize_fused_ms_stack"] = fused_ms
    offline["convert_quantize_fused_GBps"] = sum(4 * o * i for (_, o, i) in inputs.LLAMA2_7B_BLOCK) * blocks / (
        fused_ms * 1e6) + nbytes / (fused_ms * 1e6)
    xs = [[inputs.activations(5, 7 * b + pi, 1, inf, device=dev) for pi, (_, _, inf) in enumerate(inputs.LLAMA2_7B_BLOCK)]
          for b in range(blocks)]
    ys = [[torch.empty((1, outf), dtype=torch.float32, device=dev) for (_, outf, _) in inputs.LLAMA2_7B_BLOCK]
          for _ in range(blocks)]

    def step():
        for b in range(blocks):
            f2i.linear_group(stack[b], xs[b], ys[b])

    step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        graph.replay()
    stop.record(stream)
    torch.cuda.synchronize()
    f2i.sync_status()
    ms = start.elapsed_time(stop) / steps
    del graph, stack
    return {"T": T, "layout": layout, "packed_bytes": nbytes, "decode_ms_per_token": ms,
            "decode_GBps": nbytes / (ms * 1e-3) / 1e9, "tokens_per_s": 1e3 / ms, **offline}


def run_stack_only(args, world, rank, local):
    import bit_complex_valued_fairy2i_b300 as f2i
    from bit_complex_valued_fairy2i_b300 import build as f2i_build

    f2i_build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    rows = [stack_leg(f2i, dev, T, args.blocks, max(3, min(args.steps, 200)), args.warmup) for T in (1, 2, 3)]
    if rank == 0:
        print(json.dumps({"stack": {"workload": f"llama2-7b linear stack, {args.blocks} blocks x 7 projections, M=1",
                                    "rows": rows}}), flush=True)


def run_quantize_only(args, world, rank, local):
    """Offline weight preparation of `--blocks` blocks at T = 1, 2, 3 on layout 3: convert and
    quantize of every projection, each launch timed alone (CUDA events); GB/s of R read plus U, W
    written (convert) and U, W read plus codes and scales written (quantize)."""
    import bit_complex_valued_fairy2i_b300 as f2i
    from bit_complex_valued_fairy2i_b300 import build as f2i_build

    f2i_build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build_stack(f2i, 1, dev, 1, 3)  # warm-up (first launches, library load), discarded
    rows = []
    for T in (1, 2, 3):
        stack, offline = build_stack(f2i, args.blocks, dev, T, 3)
        del stack
        rows.append({"T": T, "layout": 3, **offline})
    if rank == 0:
        print(json.dumps({"quantize": {"workload": f"llama2-7b, {args.blocks} blocks x 7 projections, layout 3",
                                       "rows": rows}}), flush=True)


def run_grad_only(args, world, rank, local):
    """Input gradient dL/dx = U^^H g + W^^T conj(g) of every projection of the stack, M = 1, T = 2,
    one CUDA graph of all launches: packed bytes / device time.  Timed with one grouped launch per
    block (the reported figure) and with one launch per projection."""
    import bit_complex_valued_fairy2i_b300 as f2i
    from bit_complex_valued_fairy2i_b300 import build as f2i_build

    f2i_build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    blocks = args.blocks
    stack, _ = build_stack(f2i, blocks, dev)
    nbytes = sum(q.nbytes for layers in stack for q in layers)
    gs = [[torch.randn((1, 2 * q.n), device=dev) for q in layers] for layers in stack]
    gxs = [[torch.empty((1, 2 * q.m), device=dev) for q in layers] for layers in stack]

    def per_projection():
        for layers, gl, xl in zip(stack, gs, gxs):
            for q, g, gx in zip(layers, gl, xl):
                f2i.linear_grad_x(q, g, out=gx)

    def per_block():
        for layers, gl, xl in zip(stack, gs, gxs):
            f2i.linear_grad_x_group(layers, gl, outs=xl)

    steps = max(3, min(args.steps, 200))

    def time_graph(step):
        step()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize()
        stream = torch.cuda.current_stream()
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(steps):
            graph.replay()
        stop.record(stream)
        torch.cuda.synchronize()
        return start.elapsed_time(stop) / steps

    ms_proj = time_graph(per_projection)
    ms = time_graph(per_block)
    if rank == 0:
        print(json.dumps({"grad_x": {
            "workload": f"input gradient of llama2-7b projections, {blocks} blocks x 7, M=1, T={T_STAGES}, "
                        "one grouped launch per block",
            "kernel": "linear_grad_x_kernel (CUDA cores, 4-CTA clusters)",
            "ms_per_step": ms, "GBps": nbytes / (ms * 1e-3) / 1e9, "bytes_per_step": nbytes,
            "us_per_block": ms * 1e3 / blocks, "steps": steps,
            "one_launch_per_projection": {"us_per_block": ms_proj * 1e3 / blocks,
                                          "GBps": nbytes / (ms_proj * 1e-3) / 1e9}}}), flush=True)


def run_sweep_only(args, world, rank, local):
    import bit_complex_valued_fairy2i_b300 as f2i
    from bit_complex_valued_fairy2i_b300 import build as f2i_build

    f2i_build.build()
    torch.cuda.set_device(local)
    Ms = tuple(int(v) for v in args.sweep_ms.split(",")) if args.sweep_ms else (1, 2, 4, 8, 16, 32, 64)
    algos = tuple(args.sweep_algos.split(",")) if args.sweep_algos else SWEEP_ALGOS
    res = sweep_leg(f2i, torch.device("cuda", local), Ms=Ms, algos=algos)
    if rank == 0:
        print(json.dumps({"sweep": res}), flush=True)


def run_prefill_only(args, world, rank, local):
    import bit_complex_valued_fairy2i_b300 as f2i
    from bit_complex_valued_fairy2i_b300 import build as f2i_build

    f2i_build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    res = prefill_leg(f2i, dev, _peaks(), args.steps, args.warmup, args.prefill_tokens)
    if rank == 0:
        print(json.dumps({"prefill": res}), flush=True)


def run_ours(args, world, rank, local):
    import bit_complex_valued_fairy2i_b300 as f2i
    from bit_complex_valued_fairy2i_b300 import build as f2i_build

    f2i_build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks = _peaks()

    blocks = args.blocks
    algo = args.decode_algo
    stack, offline = build_stack(f2i, blocks, dev, layout=decode_layout(algo))
    bytes_per_block = sum(q.nbytes for q in stack[0])
    bytes_per_step = sum(q.nbytes for layers in stack for q in layers)

    # activations and outputs: one contiguous device buffer each, one row per projection
    x_sizes = [2 * q.m for layers in stack for q in layers]
    y_sizes = [2 * q.n for layers in stack for q in layers]
    x_all = torch.cat([inputs.activations(5, 7 * b + pi, 1, inf, device=dev).reshape(-1)
                       for b in range(blocks) for pi, (_, _, inf) in enumerate(inputs.LLAMA2_7B_BLOCK)])
    y_all = torch.empty(sum(y_sizes), dtype=torch.float32, device=dev)
    xv = list(torch.split(x_all, x_sizes))
    yv = list(torch.split(y_all, y_sizes))
    xs = [[xv[7 * b + i].view(1, -1) for i in range(7)] for b in range(blocks)]
    ys = [[yv[7 * b + i].view(1, -1) for i in range(7)] for b in range(blocks)]

    def step():
        for b in range(blocks):
            f2i.linear_group(stack[b], xs[b], ys[b], algo=algo)

    step()  # outside capture: first-use setup (shared-memory attributes)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()

    stream = torch.cuda.current_stream()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start.record(stream)
        for _ in range(args.steps):
            graph.replay()
        stop.record(stream)
        torch.cuda.synchronize()
    _barrier(world)
    total_ms = _max_over_ranks(start.elapsed_time(stop), world)
    ms_per_step = total_ms / args.steps
    launch_ms = ms_per_step / blocks  # every launch of the step is the decode kernel
    value = bytes_per_step * world / (ms_per_step * 1e-3) / 1e9

    # end to end: every step copies all activations in from pinned host memory and all outputs
    # back, then waits for them on the host.  One graph per step: block b's launch waits only for
    # its own activations (copy stream in), and its outputs go back (copy stream out) while the
    # next blocks run.
    x_host = torch.empty_like(x_all, device="cpu").pin_memory()
    x_host.copy_(x_all.cpu())
    y_host = torch.empty_like(y_all, device="cpu").pin_memory()
    h2d = x_all.numel() * x_all.element_size()
    d2h = y_all.numel() * y_all.element_size()
    xb_sizes = [sum(x_sizes[7 * b:7 * b + 7]) for b in range(blocks)]
    yb_sizes = [sum(y_sizes[7 * b:7 * b + 7]) for b in range(blocks)]
    x_dev_b, x_host_b = torch.split(x_all, xb_sizes), torch.split(x_host, xb_sizes)
    y_dev_b, y_host_b = torch.split(y_all, yb_sizes), torch.split(y_host, yb_sizes)
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(blocks)]
    ev_out = [torch.cuda.Event() for _ in range(blocks)]
    e2e_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(e2e_graph):
        main = torch.cuda.current_stream()
        s_in.wait_stream(main)
        s_out.wait_stream(main)
        with torch.cuda.stream(s_in):
            for b in range(blocks):
                x_dev_b[b].copy_(x_host_b[b], non_blocking=True)
                ev_in[b].record(s_in)
        for b in range(blocks):
            main.wait_event(ev_in[b])
            f2i.linear_group(stack[b], xs[b], ys[b], algo=algo)
            ev_out[b].record(main)
        with torch.cuda.stream(s_out):
            for b in range(blocks):
                s_out.wait_event(ev_out[b])
                y_host_b[b].copy_(y_dev_b[b], non_blocking=True)
        main.wait_stream(s_in)
        main.wait_stream(s_out)
    # the same copies with two waits: the first blocks' activations come in one copy, the rest
    # in a second that runs under those blocks; between the two waits every decode launch
    # depends on the previous kernel alone (it may start early, as in the device-only graph)
    head = min(4, blocks)
    x_head = sum(xb_sizes[:head])
    e2e_graph1 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(e2e_graph1):
        main = torch.cuda.current_stream()
        s_in.wait_stream(main)
        s_out.wait_stream(main)
        with torch.cuda.stream(s_in):
            x_all[:x_head].copy_(x_host[:x_head], non_blocking=True)
            ev_in[0].record(s_in)
            if head < blocks:
                x_all[x_head:].copy_(x_host[x_head:], non_blocking=True)
        main.wait_event(ev_in[0])
        for b in range(blocks):
            if b == head:
                main.wait_stream(s_in)
            f2i.linear_group(stack[b], xs[b], ys[b], algo=algo)
            ev_out[b].record(main)
        with torch.cuda.stream(s_out):
            for b in range(blocks):
                s_out.wait_event(ev_out[b])
                y_host_b[b].copy_(y_dev_b[b], non_blocking=True)
        main.wait_stream(s_out)

    def time_e2e(g):
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            g.replay()
            torch.cuda.current_stream().synchronize()
        return _max_over_ranks((time.perf_counter() - t0) / e2e_steps, world)

    e2e_steps = max(20, args.steps)  # host-timed: enough replays to average out wake-up jitter
    e2e_per_block_s = time_e2e(e2e_graph)
    e2e_one_wait_s = time_e2e(e2e_graph1)
    e2e_s = min(e2e_per_block_s, e2e_one_wait_s)
    e2e_value = bytes_per_step * world / e2e_s / 1e9

    # the same step issued eagerly (no graph): every call's host work (argument checks, launch
    # parameters, ctypes) is inside the timed region
    def eager_step():
        x_all.copy_(x_host, non_blocking=True)
        for b in range(blocks):
            f2i.linear_group(stack[b], xs[b], ys[b], algo=algo)
        y_host.copy_(y_all, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    for _ in range(3):
        eager_step()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        eager_step()
    e2e_eager_s = _max_over_ranks((time.perf_counter() - t0) / e2e_steps, world)

    # the same with each block's call prepared once (f2i.GroupCall): per step only the C call's
    # own host work (checks, launch parameters, the launches) remains
    calls = [f2i.GroupCall(stack[b], xs[b], ys[b], algo=algo) for b in range(blocks)]

    def prepared_step():
        x_all.copy_(x_host, non_blocking=True)
        for c in calls:
            c()
        y_host.copy_(y_all, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    for _ in range(3):
        prepared_step()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        prepared_step()
    e2e_prepared_s = _max_over_ranks((time.perf_counter() - t0) / e2e_steps, world)

    achieved = bytes_per_block / (launch_ms * 1e-3) / 1e9
    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": DECODE_KERNELS[algo][1],
        "data": "synthetic",
        "config": {"workload": WORKLOAD if blocks == BLOCKS else f"{blocks}-block cut of: {WORKLOAD}",
                   "M": 1, "T": T_STAGES, "blocks": blocks, "projections": 7 * blocks,
                   "bytes_per_step": bytes_per_step, "l2": "inputs larger than L2 (1.64 GB working set)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_s * 1e3, "ms_per_step_per_block_waits": e2e_per_block_s * 1e3,
                "ms_per_step_two_waits": e2e_one_wait_s * 1e3,
                "eager": {"value": bytes_per_step * world / e2e_eager_s / 1e9, "ms_per_step": e2e_eager_s * 1e3,
                          "note": "no CUDA graph: per-call host work included"},
                "eager_prepared": {"value": bytes_per_step * world / e2e_prepared_s / 1e9,
                                   "ms_per_step": e2e_prepared_s * 1e3,
                                   "note": "no CUDA graph, each block's call prepared once (GroupCall)"}},
        "gpu_launches": blocks * args.steps * (2 if algo == "lut" else 1),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"],
                     "traffic": DECODE_TRAFFIC_BYTES.get(algo),
                     "kernel": DECODE_KERNELS[algo][0], "bytes_per_launch": bytes_per_block,
                     "launch_us": launch_ms * 1e3, "peak_source": peaks["source"],
                     "frac_of_nominal_8TBps": achieved / 8000.0},
        "clocks": clk.summary(),
        "offline": offline,
    }
    del graph, e2e_graph, e2e_graph1
    # the prefill leg last among the GPU legs: for a second or two after its long tensor-core
    # load the next measurements ran up to 3x slower (55 against 19 us per block for the
    # table lookup at M = 1 in the sweep, 0.95 against 2.2 TB/s for the stack's T = 1
    # quantize), an after-effect of that leg, not of the kernels timed
    if not args.no_sweep:
        result["sweep"] = sweep_leg(f2i, dev)
    if not args.no_stack:
        del stack, x_all, y_all, xv, yv, xs, ys
        torch.cuda.empty_cache()
        result["stack"] = {"workload": f"llama2-7b linear stack, {blocks} blocks x 7 projections, M=1, layout 3 "
                                       "(table-lookup decode), T in {1, 2, 3}",
                           "rows": [stack_leg(f2i, dev, T, blocks, max(3, min(args.steps, 50)), 3) for T in (1, 2, 3)]}
    if not args.no_prefill:
        result["prefill"] = prefill_leg(f2i, dev, peaks, max(3, min(args.steps, 20)), 3, args.prefill_tokens)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    if rank == 0:
        print(json.dumps(result), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--mode", choices=["decode", "prefill", "sweep", "stack", "grad", "quantize"], default="decode",
                    help="prefill: time only the prefill leg (for profiling)")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-sweep", action="store_true", help="skip the batched-decode sweep (M = 1..64)")
    ap.add_argument("--no-stack", action="store_true", help="skip the T = 1, 2, 3 stack legs")
    ap.add_argument("--decode-algo", choices=sorted(DECODE_KERNELS), default="lut",
                    help="decode kernel of the default mode (lut = the table-lookup decode on layout 3; "
                         "auto = the library's choice on layout 2)")
    ap.add_argument("--prefill-tokens", type=int, default=2048)
    ap.add_argument("--sweep-ms", default="", help="--mode sweep: token counts, comma-separated (default 1..64)")
    ap.add_argument("--sweep-algos", default="",
                    help="--mode sweep: algorithms, comma-separated, from " + ",".join(SWEEP_ALGOS))
    ap.add_argument("--blocks", type=int, default=BLOCKS,
                    help="decoder blocks in the stack (32 = the full model; fewer only for profiling)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = _dist()
    if args.impl == "reference":
        run_reference(args, world, rank)
    elif args.mode == "prefill":
        run_prefill_only(args, world, rank, local)
    elif args.mode == "sweep":
        run_sweep_only(args, world, rank, local)
    elif args.mode == "stack":
        run_stack_only(args, world, rank, local)
    elif args.mode == "quantize":
        run_quantize_only(args, world, rank, local)
    elif args.mode == "grad":
        run_grad_only(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
