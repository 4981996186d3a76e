"""Benchmark of the QuaRot W4A4 hot path on GB300.

One step = one pass of every hot-path stage on synthetic, seeded inputs:
  1. quarot_rotate_quant_rowsum  X [2048, 12288] fp16 (H12 (x) H1024, random
                                 signs) -> packed INT4, fp16 scales, row code sums
  2. quarot_w4a4_gemm_rowsums    -> Y [2048, 4096] fp16 against W~ [4096, 12288]
                                 INT4 (its row code sums prepared with it)
  3. quarot_kv_write      append one token for 16 sequences (8 KV heads x 128)
  4. quarot_decode_attn   16 sequences x 32 query heads over 4096 cached tokens
The headline value is W4A4 layer tokens/s: 2048 tokens per step divided by
the device time of the step, inputs resident in HBM.

The step is a mixed batch: a 2048-token chunk through the down_proj layer
(1, 2) and a decode step of 16 other sequences (3, 4).  The two share no
data, so each step is one CUDA graph with two branches, rotate -> GEMM on the
launching stream and append -> decode on a forked stream, joined at the end.
The same step with the four kernels in one chain is timed beside it
("ms_per_step_serial"), and the bench checks that both give identical bytes.

Cold-L2 protocol.  Every device time is measured with CUDA events on the
launching stream over back-to-back launches that cycle through distinct sets
of input and output buffers, at least 4x the L2 size in all, so that no launch
finds its operands in L2 (a step moves ~178 MB; the per-stage sets are sized
the same way).  The older protocol, an L2 flush (a 2x L2 write) before every
launch outside the events, is reported beside it as "*_flush": it adds a fixed
~7 us per timed launch.  Warm-L2 numbers (one buffer set, back-to-back) are
reported separately and labelled.

--impl reference times the CPU oracle (dense Hadamard matrices, exact integer
GEMM, float64 attention) on the host cores over a bounded sample per step.
Multi-GPU (torchrun): every rank runs an independent replica (weak scaling);
the only cross-rank traffic is the barrier and the max of the step times.
"""
from __future__ import annotations

import argparse
import json
import math
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

M_TOK, K_DIM, N_OUT = 2048, 12288, 4096
# DRAM bytes (read + write) of one launch of the down_proj GEMM (the row-sum
# form the step runs, one accumulator), from one ncu capture of this kernel
# (37.838592 MB read + 0.232704 MB written); None whenever the kernel has
# changed since that capture.
GEMM_TRAFFIC_BYTES = 38_071_296
KV = W.CONFIGS["kv4"]
METRIC = "W4A4 layer tokens/s"
WORKLOAD = ("down_proj W4A4 layer 2048x12288->4096 (H12(x)H1024 rotate+quant, INT4 GEMM, fp16 out) "
            "+ KV4 decode step (append 1 token, GQA 32q/8kv x128 over 4096 cached tokens, batch 16)")
L2_CYCLE = 4  # buffer sets cover at least this many L2 sizes


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm": d.get("hbm_gbs", 6800.0), "bf16": d.get("bf16_tflops", 1900.0),
                "bf16_sustained": d.get("bf16_tflops_sustained", 1700.0), "source": "measured"}
    return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi sampled every 200 ms while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _job_time_ms(local_ms: float, ws: int, device) -> float:
    """The job's time for the timed region: the slowest rank's (every rank
    enters and leaves the region at a barrier).  One all-reduce (MAX)."""
    if ws <= 1:
        return float(local_ms)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _job_rate(tokens_per_rank_step: int, steps: int, ws: int, job_ms: float) -> float:
    """Whole-job throughput: the tokens all ranks processed over the job's time
    (replicas, weak scaling: every rank runs the full per-GPU workload)."""
    return ws * tokens_per_rank_step * steps / (job_ms / 1000.0)


# ============================================================================ CPU oracle baseline
# The oracle as it stands, in a pool of spawned processes (one BLAS thread
# each).  Workers are set up once (the packed weights; a decode cache of 4095
# tokens for one sequence, written by the oracle) outside the timed regions.
_CPU = {}
_ENV_1THREAD = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS")


def _cpu_init(wq, wsc, signs):
    import oracle as O

    T = KV["T"]
    k, v, qq = W.kv_inputs("kv4", B=1)
    caches = [np.zeros((1, KV["Hkv"], T, KV["d"] // 2), np.uint8), np.zeros((1, KV["Hkv"], T), np.float16),
              np.zeros((1, KV["Hkv"], T, KV["d"] // 2), np.uint8), np.zeros((1, KV["Hkv"], T), np.float16)]
    O.kv_write(k[:, :T - 1], v[:, :T - 1], 0, *caches)
    _CPU.update(wq=wq, wsc=wsc, signs=signs, caches=caches, k_new=np.ascontiguousarray(k[:, T - 1:]),
                v_new=np.ascontiguousarray(v[:, T - 1:]), q=qq)


def _cpu_ready(_):
    time.sleep(0.2)
    return os.getpid()


def _cpu_layer_task(arg):
    """rotate + quantize `x_rows`, then the exact INT GEMM against every output channel."""
    import oracle as O

    x_rows, fast = arg
    if fast:
        codes, sc = O.quantize_rows(O.rotate_fwht(x_rows, _CPU["signs"]), 1.0)
        aq = O.pack_int4(codes)
    else:
        aq, sc, _ = O.rotate_quant(x_rows, _CPU["signs"])
    _, y = O.w4a4_gemm(aq, sc, _CPU["wq"], _CPU["wsc"])
    return int(y.shape[0])


def _cpu_decode_task(_):
    """Append one token and run the decode attention of one sequence over 4096 tokens."""
    import oracle as O

    T = KV["T"]
    O.kv_write(_CPU["k_new"], _CPU["v_new"], T - 1, *_CPU["caches"])
    O.decode_attn(_CPU["q"], *_CPU["caches"], T=T)
    return 1


class OraclePool:
    """A spawned process pool running the oracle; `procs` workers, one thread each."""

    def __init__(self, procs: int):
        import oracle as O

        self.procs = procs
        _, w, s = W.layer_inputs("down_proj", M=1, N=N_OUT)
        # the weights are prepared offline, as on the GPU side (the fast mode
        # gives the same codes up to rounding ties; the GEMM time does not
        # depend on the code values)
        codes, wsc = O.quantize_rows(O.rotate_fwht(w, s), 1.0)
        wq = O.pack_int4(codes)
        saved = {k: os.environ.get(k) for k in _ENV_1THREAD}
        for k in _ENV_1THREAD:
            os.environ[k] = "1"
        try:
            self.pool = mp.get_context("spawn").Pool(procs, initializer=_cpu_init, initargs=(wq, wsc, s))
            self.pool.map(_cpu_ready, range(procs), chunksize=1)
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v

    def close(self):
        self.pool.close()
        self.pool.join()

    def step(self, rows_per_task: int, tasks: int, seqs: int, fast: bool = False):
        """Times `tasks` layer tasks of `rows_per_task` rows and `seqs` decode
        sequences, spread over the workers; returns (tokens/s of a whole step
        scaled linearly from the sample, layer seconds, decode seconds)."""
        rows = rows_per_task * tasks
        x = W.layer_inputs("down_proj", M=rows, N=0)[0]
        chunks = [(x[i * rows_per_task:(i + 1) * rows_per_task], fast) for i in range(tasks)]
        t0 = time.perf_counter()
        self.pool.map(_cpu_layer_task, chunks, chunksize=1)
        t1 = time.perf_counter()
        self.pool.map(_cpu_decode_task, range(seqs), chunksize=1)
        t2 = time.perf_counter()
        step_s = (t1 - t0) * (M_TOK / rows) + (t2 - t1) * (KV["B"] / seqs)
        return M_TOK / step_s, t1 - t0, t2 - t1


def _cores() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def cpu_baseline():
    """The oracle on the host cores: all cores (the reported value), one core,
    and the oracle's fast-transform mode on all cores; bounded samples scaled
    linearly to one step."""
    cores = _cores()
    pool = OraclePool(cores)
    try:
        pool.step(1, cores, cores)  # warm-up: first touches of the weights and caches
        v_all, tl, td = pool.step(4, cores, cores)
        v_fast, tlf, tdf = pool.step(4, cores, cores, fast=True)
        v_one, tl1, td1 = pool.step(4, 1, 1)
    finally:
        pool.close()
    return {
        "value": v_all, "unit": "tokens/s", "cores": cores, "kind": "oracle",
        "sample": (f"{4 * cores} of {M_TOK} layer rows (dense rotation + quant + exact INT GEMM against all "
                   f"{N_OUT} outputs, {tl:.2f} s) and {cores} of {KV['B']} decode sequences (append + attention "
                   f"over {KV['T']} tokens, {td:.2f} s) on {cores} single-threaded processes, each part scaled "
                   f"linearly to one step"),
        "single_thread": {"value": v_one, "cores": 1,
                          "sample": f"4 layer rows ({tl1:.2f} s) and 1 decode sequence ({td1:.2f} s), one process"},
        "fwht_mode": {"value": v_fast, "cores": cores,
                      "sample": (f"the oracle's O(d log d) fast-transform rotation in place of the dense product, "
                                 f"{4 * cores} layer rows ({tlf:.2f} s), {cores} decode sequences ({tdf:.2f} s)")},
    }


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    cores = _cores()
    pool = OraclePool(cores)
    try:
        for _ in range(args.warmup):
            pool.step(1, cores, cores)
        vals, layer_s, dec_s = [], [], []
        for _ in range(args.steps):
            v, tl, td = pool.step(1, cores, cores)
            vals.append(v)
            layer_s.append(tl)
            dec_s.append(td)
    finally:
        pool.close()
    value = statistics.median(vals)
    desc = (f"per step: {cores} of {M_TOK} layer rows (dense rotation + quant + exact INT GEMM against all {N_OUT} "
            f"outputs, median {statistics.median(layer_s):.2f} s) and {cores} of {KV['B']} decode sequences "
            f"(median {statistics.median(dec_s):.2f} s) on {cores} single-threaded processes, scaled linearly "
            f"to one step")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * M_TOK / value,
            "sample_ms_per_step": 1000.0 * statistics.median([a + b for a, b in zip(layer_s, dec_s)]),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64+int64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "l2": "n/a (CPU)"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ============================================================================ GPU timing helpers
class Timer:
    """CUDA-event timing on `stream` under the three protocols."""

    def __init__(self, q, stream, l2_bytes, flush):
        self.q, self.stream, self.l2, self.flush = q, stream, l2_bytes, flush

    def sets_for(self, bytes_per_set: int, cap: int = 128) -> int:
        return int(min(cap, max(2, math.ceil(L2_CYCLE * self.l2 / max(1, bytes_per_set)))))

    def _graph(self, fns):
        import torch

        for f in fns[:2]:  # eager first: one-time set-up (kernel attributes) stays out of the capture
            f()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for f in fns:
                f()
        return g

    def cycled(self, fns, launches_min: int = 40) -> float:
        """ms per call, back-to-back over the buffer sets of `fns` (one call each
        per graph replay)."""
        import torch

        g = self._graph(fns)
        reps = max(2, math.ceil(launches_min / len(fns)))
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(self.stream)
        for _ in range(reps):
            g.replay()
        b.record(self.stream)
        b.synchronize()
        self.q.quarot_check_error(self.stream)
        return a.elapsed_time(b) / (reps * len(fns))

    def warm(self, fn, launches: int = 40) -> float:
        """ms per call, back-to-back on one buffer set (operands warm in L2)."""
        return self.cycled([fn] * 8, launches)

    def flushed(self, fn, reps: int = 20) -> float:
        """ms per call, each launch preceded by an L2 flush outside its events."""
        import torch

        g = self._graph([fn])
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a, b in ev:
            self.flush.zero_()
            a.record(self.stream)
            g.replay()
            b.record(self.stream)
        torch.cuda.synchronize()
        self.q.quarot_check_error(self.stream)
        return float(np.mean([a.elapsed_time(b) for a, b in ev]))


def _gbs(nbytes, ms, hbm):
    g = nbytes / (ms / 1e3) / 1e9
    return {"ms": ms, "GB/s": g, "frac_hbm": g / hbm}


# ============================================================================ our arm
def run_ours(args):
    import torch

    import w4a4_rotated_quantized_gb300 as q
    from w4a4_rotated_quantized_gb300 import build as qbuild

    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or not os.path.exists(qbuild.LIB):
        qbuild.build()
    if ws > 1:
        dist.barrier()
    q.load()
    stream = torch.cuda.current_stream(dev)
    peaks = _peaks()
    hbm_peak = peaks["hbm"]
    fp8_peak = peaks["bf16"] * (4.5 / 2.25)  # kind::f8f6f4 executes the INT4 contraction
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty((max(2 * l2, 256 << 20),), dtype=torch.uint8, device=dev)
    tm = Timer(q, stream, l2, flush)

    # ---------------- inputs (seeded, synthetic), weights prepared offline
    x, w, s = W.layer_inputs("down_proj")
    k, v, qq = W.kv_inputs("kv4")
    B, T, Hkv, d = k.shape
    Hq = qq.shape[1]
    xt = torch.from_numpy(x).to(dev)
    st = torch.from_numpy(s).to(dev)
    wq, wsc, _ = q.quarot_rotate_quant(torch.from_numpy(w).to(dev), st)
    wrs = q.quarot_int4_rowsum(wq)  # the weight rows' code sums, prepared with the weights
    del w
    cache = q.new_kv_cache(B, Hkv, T, d, dev)
    q.quarot_kv_write(torch.from_numpy(k[:, :T - 1]).to(dev), torch.from_numpy(v[:, :T - 1]).to(dev), 0, *cache)
    k_new = torch.from_numpy(np.ascontiguousarray(k[:, T - 1:])).to(dev)
    v_new = torch.from_numpy(np.ascontiguousarray(v[:, T - 1:])).to(dev)
    q_dec = torch.from_numpy(qq).to(dev)
    ws_bytes = q.quarot_decode_workspace_bytes(B, Hq, d, T)
    torch.cuda.synchronize()

    # Buffer sets of one step: X, packed A + scales, W~ + scales, Y, the KV
    # cache, the new token, q, the decode output and workspace.  Every set
    # holds the same values in its own memory.
    def new_set(i):
        if i == 0:
            return dict(x=xt, aq=torch.empty((M_TOK, K_DIM // 2), dtype=torch.uint8, device=dev),
                        asx=torch.empty((M_TOK,), dtype=torch.float16, device=dev),
                        ars=torch.empty((M_TOK,), dtype=torch.int32, device=dev), wq=wq, wsc=wsc, wrs=wrs,
                        y=torch.empty((M_TOK, N_OUT), dtype=torch.float16, device=dev), cache=cache,
                        k_new=k_new, v_new=v_new, q=q_dec,
                        out=torch.empty((B, Hq, d), dtype=torch.float16, device=dev),
                        wsp=torch.empty((ws_bytes,), dtype=torch.uint8, device=dev))
        s0 = SETS[0]
        return {n: ([c.clone() for c in t] if isinstance(t, (list, tuple)) else t.clone()) for n, t in s0.items()}

    def set_bytes(sd):
        tot = 0
        for t in sd.values():
            for u in (t if isinstance(t, (list, tuple)) else [t]):
                tot += u.numel() * u.element_size()
        return tot

    SETS = [new_set(0)]
    n_sets = tm.sets_for(set_bytes(SETS[0]), cap=16)
    SETS += [new_set(i) for i in range(1, n_sets)]

    def stages_of(sd):
        return [
            lambda: q.quarot_rotate_quant_rowsum(sd["x"], st, q_out=sd["aq"], scale_out=sd["asx"], rowsum_out=sd["ars"]),
            lambda: q.quarot_w4a4_gemm_rowsums(sd["aq"], sd["asx"], sd["ars"], sd["wq"], sd["wsc"], sd["wrs"],
                                               y=sd["y"]),
            lambda: q.quarot_kv_write(sd["k_new"], sd["v_new"], T - 1, *sd["cache"]),
            lambda: q.quarot_decode_attn(sd["q"], *sd["cache"], T=T, out=sd["out"], workspace=sd["wsp"]),
        ]

    LAUNCHES_PER_STEP = 1 + 1 + 1 + 2
    side = torch.cuda.Stream(dev)

    def step_fn(sd):
        """The step's two independent branches: rotate -> GEMM on the current
        stream, KV append -> decode on `side`, joined before the step ends."""
        rot, gemm, kvw, dec = stages_of(sd)

        def f():
            cur = torch.cuda.current_stream(dev)
            side.wait_stream(cur)
            with torch.cuda.stream(side):
                kvw()
                dec()
            rot()
            gemm()
            cur.wait_stream(side)
        return f

    def serial_fn(sd):
        fns = stages_of(sd)

        def f():
            for g in fns:
                g()
        return f

    for sd in SETS:
        for _ in range(max(1, args.warmup // len(SETS) + 1)):
            step_fn(sd)()
    q.quarot_check_error(stream)
    g_steps, g_serial = [], []
    for sd in SETS:
        for fn, lst in ((step_fn, g_steps), (serial_fn, g_serial)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn(sd)()
            lst.append(g)
    for i in range(args.warmup):
        g_steps[i % n_sets].replay()
    torch.cuda.synchronize()
    q.quarot_check_error(stream)

    # ---------------- the timed region: K steps back-to-back over the buffer sets
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        e0.record(stream)
        for i in range(args.steps):
            g_steps[i % n_sets].replay()
        e1.record(stream)
        torch.cuda.synchronize()
        timed_samples = len(clocks.lines)
        # a short timed region may end before nvidia-smi reports: keep the same
        # load running (untimed) until a few samples exist
        t_end = time.time() + 3.0
        while len(clocks.lines) < timed_samples + 5 and time.time() < t_end:
            for i in range(60):
                g_steps[i % n_sets].replay()
            torch.cuda.synchronize()
    q.quarot_check_error(stream)
    total_ms = _job_time_ms(float(e0.elapsed_time(e1)), ws, dev)
    if ws > 1:
        dist.barrier()
    value = _job_rate(M_TOK, args.steps, ws, total_ms)

    # the same steps under the flush protocol (set 0, a 2x L2 write before each step)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in evs:
        flush.zero_()
        a.record(stream)
        g_steps[0].replay()
        b.record(stream)
    torch.cuda.synchronize()
    step_ms_flush = float(np.mean([a.elapsed_time(b) for a, b in evs]))

    # the same steps with the four kernels in one chain, cycled the same way
    for i in range(args.warmup):
        g_serial[i % n_sets].replay()
    e0.record(stream)
    for i in range(args.steps):
        g_serial[i % n_sets].replay()
    e1.record(stream)
    torch.cuda.synchronize()
    step_ms_serial = float(e0.elapsed_time(e1)) / args.steps
    # both forms of the step leave identical bytes in Y and the decode output
    s0 = SETS[0]
    g_serial[0].replay()
    torch.cuda.synchronize()
    y_ser, o_ser = s0["y"].clone(), s0["out"].clone()
    s0["y"].zero_()
    s0["out"].zero_()
    g_steps[0].replay()
    torch.cuda.synchronize()
    q.quarot_check_error(stream)
    if not (torch.equal(y_ser, s0["y"]) and torch.equal(o_ser, s0["out"])):
        raise RuntimeError("the two-branch step differs from the serial step")
    # the row-sum path against the plain entry points on the same input
    aq_p, as_p, _ = q.quarot_rotate_quant(s0["x"], st)
    y_p, _ = q.quarot_w4a4_gemm(aq_p, as_p, s0["wq"], s0["wsc"])
    torch.cuda.synchronize()
    if not (torch.equal(aq_p, s0["aq"]) and torch.equal(y_p, s0["y"])):
        raise RuntimeError("the row-sum step differs from quarot_rotate_quant + quarot_w4a4_gemm")
    del y_ser, o_ser, aq_p, as_p, y_p

    # ---------------- per-stage device times: back-to-back over the step's buffer sets
    stage_names = ["rotate_quant", "w4a4_gemm", "kv_write_append", "decode_attn"]
    per_set = [stages_of(sd) for sd in SETS]
    stage_ms, stage_ms_flush = [], []
    for j in range(4):
        stage_ms.append(tm.cycled([fs[j] for fs in per_set], launches_min=max(40, args.steps)))
        stage_ms_flush.append(tm.flushed(per_set[0][j], reps=max(10, min(args.steps, 50))))

    # ---------------- e2e: host buffers through the C ABI, copies inside the timed region
    # Every step copies its inputs (X, and the new K/V token with q as one
    # packed copy) from pinned host memory and reads its results (Y, the decode
    # output) back.  The steps are
    # pipelined the way a serving loop would run them: host-to-device copies on
    # one stream, the four kernels on the compute stream, device-to-host copies
    # on a third, with double-buffered device tensors, so step i+1's input copy
    # overlaps step i's kernels.  The per-step traffic (X 50 MB, W 25 MB, Y 17 MB,
    # KV cache 69 MB) exceeds L2, so no flush is needed between steps.
    s0 = SETS[0]
    x_h = torch.from_numpy(x).pin_memory()
    # the decode branch's three small inputs travel as one copy: a pinned host
    # buffer [k_new | v_new | q] and, per slot, a device buffer viewed as the
    # three tensors (each piece starts on a 256-byte boundary)
    small = [k_new, v_new, q_dec]
    offs, tot = [], 0
    for t_ in small:
        offs.append(tot)
        tot += (t_.numel() * t_.element_size() + 255) // 256 * 256
    small_h = torch.zeros(tot, dtype=torch.uint8).pin_memory()
    for t_, o_ in zip(small, offs):
        nb_ = t_.numel() * t_.element_size()
        small_h[o_:o_ + nb_].copy_(t_.cpu().contiguous().view(-1).view(torch.uint8))
    small_d = [torch.empty(tot, dtype=torch.uint8, device=dev) for _ in range(2)]

    def piece(buf, i):
        t_ = small[i]
        nb_ = t_.numel() * t_.element_size()
        return buf[offs[i]:offs[i] + nb_].view(t_.dtype).view(t_.shape)

    xd = [torch.empty_like(xt) for _ in range(2)]
    kd = [piece(small_d[i], 0) for i in range(2)]
    vd = [piece(small_d[i], 1) for i in range(2)]
    qd = [piece(small_d[i], 2) for i in range(2)]
    aqd = [torch.empty_like(s0["aq"]) for _ in range(2)]
    asd = [torch.empty_like(s0["asx"]) for _ in range(2)]
    ard = [torch.empty_like(s0["ars"]) for _ in range(2)]
    yd = [torch.empty_like(s0["y"]) for _ in range(2)]
    od = [torch.empty_like(s0["out"]) for _ in range(2)]
    y_h = [torch.empty_like(s0["y"], device="cpu").pin_memory() for _ in range(2)]
    o_h = [torch.empty_like(s0["out"], device="cpu").pin_memory() for _ in range(2)]
    h2d_st, d2h_st = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    dec_st = torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of the slot copied
    ev_comp = [torch.cuda.Event() for _ in range(2)]  # kernels of the slot done
    ev_out = [torch.cuda.Event() for _ in range(2)]   # results of the slot copied out

    def e2e_run(n):
        for i in range(n):
            sl = i % 2
            if i >= 2:
                h2d_st.wait_event(ev_comp[sl])  # slot's inputs no longer read
            with torch.cuda.stream(h2d_st):
                small_d[sl].copy_(small_h, non_blocking=True)
                xd[sl].copy_(x_h, non_blocking=True)
            ev_in[sl].record(h2d_st)
            stream.wait_event(ev_in[sl])
            if i >= 2:
                stream.wait_event(ev_out[sl])  # slot's results already read back
            dec_st.wait_stream(stream)  # the decode branch, forked as in the timed step
            q.quarot_kv_write(kd[sl], vd[sl], T - 1, *s0["cache"], stream=dec_st)
            q.quarot_decode_attn(qd[sl], *s0["cache"], T=T, out=od[sl], workspace=s0["wsp"], stream=dec_st)
            q.quarot_rotate_quant_rowsum(xd[sl], st, q_out=aqd[sl], scale_out=asd[sl], rowsum_out=ard[sl],
                                         stream=stream)
            q.quarot_w4a4_gemm_rowsums(aqd[sl], asd[sl], ard[sl], s0["wq"], s0["wsc"], s0["wrs"], y=yd[sl],
                                       stream=stream)
            stream.wait_stream(dec_st)
            ev_comp[sl].record(stream)
            d2h_st.wait_event(ev_comp[sl])
            with torch.cuda.stream(d2h_st):
                y_h[sl].copy_(yd[sl], non_blocking=True)
                o_h[sl].copy_(od[sl], non_blocking=True)
            ev_out[sl].record(d2h_st)

    e2e_run(max(2, args.warmup))
    torch.cuda.synchronize()
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    h2d_st.wait_event(e_start)
    e2e_run(args.steps)
    stream.wait_stream(d2h_st)
    e_end.record(stream)
    e_end.synchronize()
    q.quarot_check_error(stream)
    e2e_total = _job_time_ms(float(e_start.elapsed_time(e_end)), ws, dev)
    e2e_val = _job_rate(M_TOK, args.steps, ws, e2e_total)
    h2d = xd[0].numel() * xd[0].element_size() + small_h.numel()
    d2h = s0["y"].numel() * 2 + s0["out"].numel() * 2
    # the results of the last step match the device-resident step's
    torch.cuda.synchronize()
    g_steps[0].replay()
    torch.cuda.synchronize()
    sl = (args.steps - 1) % 2
    if not (torch.equal(y_h[sl], s0["y"].cpu()) and torch.equal(o_h[sl], s0["out"].cpu())):
        raise RuntimeError("e2e results differ from the device-resident step")

    # ---------------- roofline of the dominant kernel (GEMM, tensor pipe)
    gemm_ms = float(stage_ms[1])
    gemm_tflops = 2.0 * M_TOK * N_OUT * K_DIM / (gemm_ms / 1000.0) / 1e12
    rq_bytes = M_TOK * K_DIM * 2 + M_TOK * K_DIM // 2 + M_TOK * 2
    dec_bytes = B * Hkv * T * (d // 2) * 2 + B * Hkv * T * 2 * 2 + B * Hq * d * 2 * 2
    kvw_bytes = 2 * (B * Hkv * d * 2 + B * Hkv * (d // 2 + 2))
    stages = {
        "rotate_quant": dict(_gbs(rq_bytes, stage_ms[0], hbm_peak), ms_flush=stage_ms_flush[0]),
        "w4a4_gemm": {"ms": gemm_ms, "TOPS": gemm_tflops, "frac_fp8_peak": gemm_tflops / fp8_peak,
                      "ms_flush": stage_ms_flush[1]},
        "kv_write_append": {"ms": stage_ms[2], "GB/s": kvw_bytes / (stage_ms[2] / 1e3) / 1e9,
                            "ms_flush": stage_ms_flush[2]},
        "decode_attn": dict(_gbs(dec_bytes, stage_ms[3], hbm_peak), ms_flush=stage_ms_flush[3]),
    }
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "ms_per_step_flush": step_ms_flush,
        "ms_per_step_serial": step_ms_serial,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int4+f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "tokens_per_step": M_TOK,
                   "l2": (f"inputs larger than L2: steps cycle through {n_sets} distinct buffer sets "
                          f"({n_sets * set_bytes(SETS[0]) / 1e6:.0f} MB >= {L2_CYCLE}x L2 {l2 / 1e6:.0f} MB), "
                          f"back-to-back; ms_per_step_flush: one set, 2x L2 write before each step"),
                   "parallelism": f"replicas x{ws}",
                   "launch": ("CUDA graph per step, two branches joined: rotate+quant -> GEMM | "
                              "KV append -> decode (a mixed batch: the layer's 2048-token chunk and "
                              "16 decoding sequences share no data); ms_per_step_serial: one chain")},
        "roofline": {"bound": "tensor", "kernel": "w4a4_gemm", "achieved": gemm_tflops, "peak": fp8_peak,
                     "unit": "TFLOP/s", "frac": gemm_tflops / fp8_peak, "traffic": GEMM_TRAFFIC_BYTES,
                     "peak_source": f"{peaks['source']} bf16 burst x 2 (fp8/bf16 nominal ratio)"},
        "stages": stages,
        "e2e": {"value": e2e_val, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "pipeline": "per-step H2D, kernels (two branches, as in the timed step) and D2H on "
                            "four streams, double-buffered; no L2 flush (per-step traffic > L2)"},
        "gpu_launches": LAUNCHES_PER_STEP * args.steps,
        "clocks": dict(clocks.summary(), samples_in_timed_region=timed_samples),
    }
    if rank == 0 and not args.no_extra:
        extra = _other_configs(q, dev, stream, tm, hbm_peak, fp8_peak, s0, st, x, qq)
        line["other_configs"] = extra
    del SETS, g_steps, per_set
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


def _gemm_a8_case(q, tm, dev, g, M, N, K, wq_, ws_, fp8_peak, rot_ms):
    """quarot_w4a4_gemm_a8 (activations as operand bytes, seeded uniform codes)
    under the cycled protocol; the layer rate uses quarot_rotate_quant_a8."""
    import torch

    a8 = torch.randint(0, 16, (M, K), dtype=torch.uint8, generator=g).to(dev)
    rs = torch.randint(-8 * K // 16, 8 * K // 16, (M,), dtype=torch.int32, generator=g).to(dev)
    as_ = (torch.rand(M, generator=g) * 0.1 + 0.01).half().to(dev)
    nbytes = M * K + N * K // 2 + M * N * 2
    n = tm.sets_for(nbytes, cap=32)
    sets = [(a8.clone(), wq_.clone(), torch.empty((M, N), dtype=torch.float16, device=dev)) for _ in range(n)]
    fns = [(lambda a=a, w=w, y=y: q.quarot_w4a4_gemm_a8(a, rs, as_, w, ws_, y=y)) for a, w, y in sets]
    ms = tm.cycled(fns)
    tf = 2.0 * M * N * K / (ms / 1e3) / 1e12
    return {"ms": ms, "TOPS": tf, "frac_fp8_peak": tf / fp8_peak, "buffer_sets": n,
            "layer_tokens_per_s": M / ((ms + rot_ms) / 1e3)}


def _other_configs(q, dev, stream, tm, hbm_peak, fp8_peak, s0, st, x_dp, qq_kv):
    """The other measured workloads (rank 0), each under the cycled cold-L2
    protocol unless labelled warm: the HBM-roof rotate+quant of 2048 x 4096 and
    its M sweep, the fused RMSNorm and FP16-arithmetic variants, the cross-head
    transform, the bulk KV write of the whole kv4 cache, decode at batch 1, 4,
    16 and 64 (symmetric) and the asymmetric cache, causal prefill attention,
    the GEMM sweep, the legacy mma.sync integer rate, and the rotated vs naive
    W4A4 error on the down_proj inputs."""
    import torch

    res = {}

    def rot_case(name, fn_kind, x, s_t, extra=None):
        M, dd = x.shape
        xt = torch.from_numpy(x).to(dev)
        a8 = fn_kind == "a8"  # codes as operand bytes (d per row) plus int32 row sums
        nbytes = M * dd * 2 + (M * dd + M * 6 if a8 else M * dd // 2 + M * 2) + (M * 4 if fn_kind == "rs" else 0)
        n = tm.sets_for(nbytes)
        bufs = [(xt if i == 0 else xt.clone(), torch.empty((M, dd if a8 else dd // 2), dtype=torch.uint8, device=dev),
                 torch.empty((M,), dtype=torch.float16, device=dev)) for i in range(n)]
        rsb = torch.empty((M,), dtype=torch.int32, device=dev)

        def mk(b):
            xi, qo, so = b
            if a8:
                return lambda: q.quarot_rotate_quant_a8(xi, s_t, a8_out=qo, scale_out=so, rowsum_out=rsb)
            if fn_kind == "rotate":
                return lambda: q.quarot_rotate_quant(xi, s_t, q_out=qo, scale_out=so)
            if fn_kind == "rs":
                return lambda: q.quarot_rotate_quant_rowsum(xi, s_t, q_out=qo, scale_out=so, rowsum_out=rsb)
            if fn_kind == "rmsnorm":
                return lambda: q.quarot_rmsnorm_rotate_quant(xi, s_t, eps=1e-6, q_out=qo, scale_out=so)
            if fn_kind == "fp16":
                return lambda: q.quarot_rotate_quant_fp16(xi, s_t, q_out=qo, scale_out=so)
            return lambda: q.quarot_crosshead_rotate_quant(xi, 32, q_out=qo, scale_out=so)
        fns = [mk(b) for b in bufs]
        r = dict(_gbs(nbytes, tm.cycled(fns), hbm_peak), buffer_sets=n)
        if extra == "flush":
            r["ms_flush"] = tm.flushed(fns[0])
        if extra == "warm":
            r["ms_warm_l2"] = tm.warm(fns[0])
            r["GB/s_warm_l2"] = nbytes / (r["ms_warm_l2"] / 1e3) / 1e9
        res[name] = r
        return r["ms"]

    x4, _, s4 = W.layer_inputs("rotq4096")
    s4t = torch.from_numpy(s4).to(dev)
    rot_case("rotate_quant_2048x4096", "rotate", x4, s4t, extra="warm")
    rot_case("rmsnorm_rotate_quant_2048x4096", "rmsnorm", x4, s4t)
    rot_case("rmsnorm_rotate_quant_2048x12288", "rmsnorm", x_dp, st)
    rot_case("rotate_quant_fp16_2048x12288", "fp16", x_dp, st)
    rot_case("crosshead_rotate_quant_2048x32x128", "crosshead", W.query(2048, 32, 128, 77).reshape(2048, 4096), None)
    xs, _, ss = W.layer_inputs("sweep", M=8192)
    sst = torch.from_numpy(ss).to(dev)
    rot_ms = {M: rot_case(f"rotate_quant_{M}x4096", "rotate", np.ascontiguousarray(xs[:M]), sst)
              for M in (512, 2048, 8192)}
    # the tensor-core operand form (one byte per code, row sums) for the A8 GEMM
    rot8_ms = {M: rot_case(f"rotate_quant_a8_{M}x4096", "a8", np.ascontiguousarray(xs[:M]), sst)
               for M in (512, 2048, 8192)}
    rot8_dp = rot_case("rotate_quant_a8_2048x12288", "a8", x_dp, st)
    # packed codes plus int32 row code sums for the row-sum GEMM
    rotrs_ms = {M: rot_case(f"rotate_quant_rowsum_{M}x4096", "rs", np.ascontiguousarray(xs[:M]), sst)
                for M in (512, 2048, 8192)}

    # ---- KV cache: bulk write of the whole kv4 cache, decode batch sweep
    c = W.CONFIGS["kv4"]
    Hkv, Hq, d, T = c["Hkv"], c["Hq"], c["d"], c["T"]
    g = torch.Generator(device="cpu").manual_seed(4321)
    k, v, _ = W.kv_inputs("kv4")
    kt, vt = torch.from_numpy(k).to(dev), torch.from_numpy(v).to(dev)
    B = k.shape[0]
    in_b = 2 * kt.numel() * 2
    out_b = 2 * (B * Hkv * T * (d // 2 + 2))
    n = tm.sets_for(in_b + out_b)
    kv_sets = [((kt, vt) if i == 0 else (kt.clone(), vt.clone()), q.new_kv_cache(B, Hkv, T, d, dev)) for i in range(n)]
    fns = [(lambda a=a, cc=cc: q.quarot_kv_write(a[0], a[1], 0, *cc)) for a, cc in kv_sets]
    res["kv_write_bulk_B16xT4096"] = dict(_gbs(in_b + out_b, tm.cycled(fns, 20), hbm_peak), buffer_sets=n)
    del kv_sets, fns, kt, vt

    def rand_cache(Bd):
        kq_ = torch.randint(0, 256, (Bd, Hkv, T, d // 2), dtype=torch.uint8, generator=g).to(dev)
        vq_ = torch.randint(0, 256, (Bd, Hkv, T, d // 2), dtype=torch.uint8, generator=g).to(dev)
        ks_ = (torch.rand((Bd, Hkv, T), generator=g) * 0.45 + 0.05).half().to(dev)
        vs_ = (torch.rand((Bd, Hkv, T), generator=g) * 0.45 + 0.05).half().to(dev)
        return [kq_, ks_, vq_, vs_]

    for Bd in (1, 4, 16, 64):
        nbytes = Bd * Hkv * T * (d // 2) * 2 + Bd * Hkv * T * 2 * 2 + Bd * Hq * d * 2 * 2
        n = tm.sets_for(nbytes)
        base = rand_cache(Bd)
        qd = torch.randn((Bd, Hq, d), generator=g).half().to(dev)
        wsb = q.quarot_decode_workspace_bytes(Bd, Hq, d, T)
        sets = [([t if i == 0 else t.clone() for t in base], torch.empty((Bd, Hq, d), dtype=torch.float16, device=dev),
                 torch.empty((wsb,), dtype=torch.uint8, device=dev)) for i in range(n)]
        fns = [(lambda cc=cc, o=o, wsp=wsp: q.quarot_decode_attn(qd, *cc, T=T, out=o, workspace=wsp))
               for cc, o, wsp in sets]
        r = dict(_gbs(nbytes, tm.cycled(fns), hbm_peak), buffer_sets=n)
        if Bd == 16:
            r["ms_warm_l2"] = tm.warm(fns[0])
            r["GB/s_warm_l2"] = nbytes / (r["ms_warm_l2"] / 1e3) / 1e9
        res[f"decode_attn_B{Bd}_T4096"] = r
        del sets, fns, base
    # asymmetric cache (group 128, zero point, clip 0.95) at the kv4 size
    k, v, qq = W.kv_inputs("kv4")
    ac = q.new_kv_cache_asym(B, Hkv, T, d, dev)
    q.quarot_kv_write_asym(torch.from_numpy(k).to(dev), torch.from_numpy(v).to(dev), 0, *ac, stream=stream)
    qd = torch.from_numpy(qq).to(dev)
    nbytes = B * Hkv * T * (d // 2) * 2 + B * Hkv * T * (2 + 2) * 2 + B * Hq * d * 2 * 2
    n = tm.sets_for(nbytes)
    wsb = q.quarot_decode_workspace_bytes(B, Hq, d, T)
    sets = [([t if i == 0 else t.clone() for t in ac], torch.empty((B, Hq, d), dtype=torch.float16, device=dev),
             torch.empty((wsb,), dtype=torch.uint8, device=dev)) for i in range(n)]
    fns = [(lambda cc=cc, o=o, wsp=wsp: q.quarot_decode_attn_asym(qd, *cc, T=T, out=o, workspace=wsp))
           for cc, o, wsp in sets]
    res["decode_attn_asym_kv4"] = dict(_gbs(nbytes, tm.cycled(fns), hbm_peak), buffer_sets=n)
    del sets, fns, ac

    # ---- Init (prefill) attention over the INT4 cache: 4 prompts x 2048 tokens,
    # Hq 32 / Hkv 8, causal; flops are the useful ones (t <= i), 4 d per pair
    k, v, qp = W.prefill_inputs("prefill")
    Bp, Tp = k.shape[0], k.shape[1]
    pc = q.new_kv_cache(Bp, Hkv, Tp, d, dev)
    q.quarot_kv_write(torch.from_numpy(k).to(dev), torch.from_numpy(v).to(dev), 0, *pc, stream=stream)
    qpt = torch.from_numpy(qp).to(dev)
    nbytes = 2 * qpt.numel() * 2 + sum(t.numel() * t.element_size() for t in pc)
    n = tm.sets_for(nbytes)
    sets = [(qpt if i == 0 else qpt.clone(), [t if i == 0 else t.clone() for t in pc], torch.empty_like(qpt))
            for i in range(n)]
    fns = [(lambda a=a, cc=cc, o=o: q.quarot_prefill_attn(a, *cc, out=o)) for a, cc, o in sets]
    ms = tm.cycled(fns, 20)
    tf = 4.0 * Bp * Hq * d * (Tp * (Tp + 1) / 2) / (ms / 1e3) / 1e12
    res["prefill_attn_4x2048_h32kv8"] = {"ms": ms, "TFLOP/s": tf, "frac_f16_peak": tf / (fp8_peak / 2),
                                         "buffer_sets": n}
    del sets, fns, pc, qpt

    # ---- GEMM sweep M x 4096 x N (seeded uniform INT4 codes: GEMM speed does not
    # depend on the code values); layer rate M / (t_rotate_quant + t_gemm)
    K = 4096
    for N in (4096, 12288):
        wq_ = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, generator=g).to(dev)
        ws_ = (torch.rand(N, generator=g) * 0.01 + 0.001).half().to(dev)
        for M in (512, 2048, 8192):
            aq_ = torch.randint(0, 256, (M, K // 2), dtype=torch.uint8, generator=g).to(dev)
            as_ = (torch.rand(M, generator=g) * 0.1 + 0.01).half().to(dev)
            nbytes = M * K // 2 + N * K // 2 + M * N * 2
            n = tm.sets_for(nbytes, cap=32)
            sets = [(aq_.clone(), as_, wq_.clone(), ws_, torch.empty((M, N), dtype=torch.float16, device=dev))
                    for _ in range(n)]
            fns = [(lambda a=a, b=b, c_=c_, e=e, y=y: q.quarot_w4a4_gemm(a, b, c_, e, y=y)) for a, b, c_, e, y in sets]
            ms = tm.cycled(fns)
            tf = 2.0 * M * N * K / (ms / 1e3) / 1e12
            res[f"w4a4_gemm_{M}x{K}x{N}"] = {"ms": ms, "TOPS": tf, "frac_fp8_peak": tf / fp8_peak, "buffer_sets": n,
                                             "layer_tokens_per_s": M / ((ms + rot_ms[M]) / 1e3)}
            # both operands' row code sums given (quarot_rotate_quant_rowsum and
            # the weights' quarot_int4_rowsum, prepared outside the timing)
            ars_, wrs_ = q.quarot_int4_rowsum(aq_), q.quarot_int4_rowsum(wq_)
            fns = [(lambda a=a, b=b, c_=c_, e=e, y=y: q.quarot_w4a4_gemm_rowsums(a, b, ars_, c_, e, wrs_, y=y))
                   for a, b, c_, e, y in sets]
            ms = tm.cycled(fns)
            tf = 2.0 * M * N * K / (ms / 1e3) / 1e12
            res[f"w4a4_gemm_rowsums_{M}x{K}x{N}"] = {"ms": ms, "TOPS": tf, "frac_fp8_peak": tf / fp8_peak,
                                                     "buffer_sets": n,
                                                     "layer_tokens_per_s": M / ((ms + rotrs_ms[M]) / 1e3)}
            del sets, fns
            res[f"w4a4_gemm_a8_{M}x{K}x{N}"] = _gemm_a8_case(q, tm, dev, g, M, N, K, wq_, ws_, fp8_peak, rot8_ms[M])
    res["w4a4_gemm_a8_2048x12288x4096"] = _gemm_a8_case(q, tm, dev, g, M_TOK, N_OUT, K_DIM, s0["wq"], s0["wsc"],
                                                          fp8_peak, rot8_dp)
    # the bench GEMM with its operands warm in L2 (one buffer set, back-to-back)
    ms_w = tm.warm(lambda: q.quarot_w4a4_gemm_rowsums(s0["aq"], s0["asx"], s0["ars"], s0["wq"], s0["wsc"], s0["wrs"],
                                                      y=s0["y"]))
    tf = 2.0 * M_TOK * N_OUT * K_DIM / (ms_w / 1e3) / 1e12
    res["w4a4_gemm_2048x12288x4096_warm_l2"] = {"ms": ms_w, "TOPS": tf, "frac_fp8_peak": tf / fp8_peak}

    # ---- legacy warp-level integer MMA (mma.sync) rate on this GPU: the
    # instruction class of the pages' own 4-bit GEMM, reported as context
    sink = torch.zeros(1, dtype=torch.int32, device=dev)
    for bits, label in ((8, "s8 m16n8k32"), (4, "s4 m16n8k64")):
        for _ in range(2):
            q.quarot_legacy_imma_probe(bits, 256, sink)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        ops = q.quarot_legacy_imma_probe(bits, 8192, sink)
        b.record(stream)
        b.synchronize()
        tops = ops / (a.elapsed_time(b) / 1e3) / 1e12
        res[f"int{bits}_tc_legacy_mma_sync"] = {"TOPS": tops, "instruction": f"mma.sync {label}",
                                                "gemm_2048x12288x4096_frac_of_it": None}
    # the fp16 form (m16n8k16, fp32 accumulators): the instruction of the
    # decode and prefill attention kernels, whose tensor share it bounds
    for _ in range(2):
        q.quarot_legacy_imma_probe(16, 256, sink)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    ops = q.quarot_legacy_imma_probe(16, 8192, sink)
    b.record(stream)
    b.synchronize()
    res["f16_tc_legacy_mma_sync"] = {"TFLOPS": ops / (a.elapsed_time(b) / 1e3) / 1e12,
                                     "instruction": "mma.sync f16 m16n8k16, f32 accumulate"}
    gemm_tops = res.get("w4a4_gemm_2048x4096x12288", {}).get("TOPS")
    for bits in (8, 4):
        r = res[f"int{bits}_tc_legacy_mma_sync"]
        r["gemm_2048x12288x4096_frac_of_it"] = None if gemm_tops is None else gemm_tops / r["TOPS"]

    # ---- method effect on the down_proj inputs (the guide's naive vs rotated
    # W4A4 comparison), on 256 sampled rows, float64 on the GPU: the error of
    # our rotated W4A4 output and of naive per-token / per-channel INT4 without
    # rotation, both against the float product X W^T
    rows = torch.from_numpy(np.sort(np.random.default_rng(7).choice(M_TOK, 256, replace=False))).to(dev)
    _, wf, _ = W.layer_inputs("down_proj", M=1)
    xr = torch.from_numpy(x_dp).to(dev).index_select(0, rows).double()
    wd = torch.from_numpy(wf).to(dev).double()
    ref = xr @ wd.T

    def naive_q(t):
        sc = (torch.clamp(t.abs().amax(dim=1), min=1e-5) / 7.0).half().double()
        return torch.clamp(torch.round(t / sc[:, None]), -8, 7) * sc[:, None]
    y_naive = naive_q(xr) @ naive_q(wd).T
    y_rot = s0["y"].index_select(0, rows).double()

    def rel(a):
        return float(torch.linalg.norm(a - ref) / torch.linalg.norm(ref))
    res["method_effect_down_proj"] = {"rel_err_rotated_w4a4": rel(y_rot), "rel_err_naive_w4a4": rel(y_naive),
                                      "rows": 256, "reference": "float64 X W^T of the fp16 inputs"}
    del wd, xr, ref
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the other_configs lines")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
