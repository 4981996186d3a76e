"""Benchmark of the QuaRot W4A4 hot path on GB300.

One step = one pass of every hot-path stage on synthetic, seeded inputs:
  1. quarot_rotate_quant  X [2048, 12288] fp16 (H12 (x) H1024, random signs)
  2. quarot_w4a4_gemm     -> Y [2048, 4096] fp16 against W~ [4096, 12288] INT4
  3. quarot_kv_write      append one token for 16 sequences (8 KV heads x 128)
  4. quarot_decode_attn   16 sequences x 32 query heads over 4096 cached tokens
The headline value is W4A4 layer tokens/s: 2048 tokens per step divided by
the device time of the step (inputs resident in HBM, L2 flushed between
steps).  Per-stage times, HBM GB/s, GEMM TOPS and the roofline fraction come
from CUDA events on the launching stream in the same run.

--impl reference times the CPU oracle (dense Hadamard matrices, exact integer
GEMM, float64 attention) on the host cores over a bounded sample per step.
Multi-GPU (torchrun): every rank runs an independent replica (weak scaling);
the only cross-rank traffic is the barrier and the max of the step times.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

M_TOK, K_DIM, N_OUT = 2048, 12288, 4096
# DRAM bytes (read + write) of one launch of the down_proj GEMM, from an ncu
# capture of this bench (profiles/w4a4_gemm_pair_down_proj_2048x4096x12288.md);
# None whenever the kernel has changed since that capture.
GEMM_TRAFFIC_BYTES = 38_763_008  # 37.808384 MB read + 0.954624 MB written
KV = W.CONFIGS["kv4"]
METRIC = "W4A4 layer tokens/s"
WORKLOAD = ("down_proj W4A4 layer 2048x12288->4096 (H12(x)H1024 rotate+quant, INT4 GEMM, fp16 out) "
            "+ KV4 decode step (append 1 token, GQA 32q/8kv x128 over 4096 cached tokens, batch 16)")


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


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


def cpu_oracle_sample(rows: int = 8, seqs: int = 1):
    """Times the oracle on a bounded sample of one step; returns (tokens/s, seconds, description)."""
    import oracle as O

    x, w, s = W.layer_inputs("down_proj", M=rows, N=N_OUT)
    k, v, qq = W.kv_inputs("kv4", B=seqs)
    T = KV["T"]
    caches = [np.zeros((seqs, KV["Hkv"], T, KV["d"] // 2), np.uint8), np.zeros((seqs, KV["Hkv"], T), np.float16),
              np.zeros((seqs, KV["Hkv"], T, KV["d"] // 2), np.uint8), np.zeros((seqs, KV["Hkv"], T), np.float16)]
    # weights are prepared offline (not timed), as on the GPU side
    wq, wsc, _ = O.rotate_quant(w, s)
    O.kv_write(k[:, :T - 1], v[:, :T - 1], 0, *caches)
    t0 = time.perf_counter()
    aq, asc, _ = O.rotate_quant(x, s)
    O.w4a4_gemm(aq, asc, wq, wsc)
    t1 = time.perf_counter()
    O.kv_write(k[:, T - 1:], v[:, T - 1:], T - 1, *caches)
    O.decode_attn(qq, *caches, T=T)
    t2 = time.perf_counter()
    dt = t2 - t0
    # scale to a whole step: layer time with the rows, decode time with the batch
    step_s = (t1 - t0) * (M_TOK / rows) + (t2 - t1) * (KV["B"] / seqs)
    desc = (f"{rows} of {M_TOK} layer rows (rotate+quant + exact INT GEMM against all {N_OUT} outputs, "
            f"{t1 - t0:.2f} s) and {seqs} of {KV['B']} decode sequences (append + attention over {T} tokens, "
            f"{t2 - t1:.2f} s), each scaled linearly to one step")
    return M_TOK / step_s, dt, desc


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    for _ in range(args.warmup):
        cpu_oracle_sample(rows=1, seqs=1)
    vals, secs = [], 0.0
    desc = ""
    for _ in range(args.steps):
        v, dt, desc = cpu_oracle_sample(rows=2, seqs=1)
        vals.append(v)
        secs += dt
    value = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * M_TOK / value,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64+int64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "l2": "n/a (CPU)"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


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

    # ---------------- inputs (seeded, synthetic), weights prepared offline
    x, w, s = W.layer_inputs("down_proj")
    k, v, qq = W.kv_inputs("kv4")
    B, T, Hkv, d = k.shape
    Hq = qq.shape[1]
    xt = torch.from_numpy(x).to(dev)
    st = torch.from_numpy(s).to(dev)
    wq, wsc, _ = q.quarot_rotate_quant(torch.from_numpy(w).to(dev), st)
    del w
    cache = q.new_kv_cache(B, Hkv, T, d, dev)
    q.quarot_kv_write(torch.from_numpy(k[:, :T - 1]).to(dev), torch.from_numpy(v[:, :T - 1]).to(dev), 0, *cache)
    k_new = torch.from_numpy(np.ascontiguousarray(k[:, T - 1:])).to(dev)
    v_new = torch.from_numpy(np.ascontiguousarray(v[:, T - 1:])).to(dev)
    q_dec = torch.from_numpy(qq).to(dev)
    aq = torch.empty((M_TOK, K_DIM // 2), dtype=torch.uint8, device=dev)
    asx = torch.empty((M_TOK,), dtype=torch.float16, device=dev)
    y = torch.empty((M_TOK, N_OUT), dtype=torch.float16, device=dev)
    out = torch.empty((B, Hq, d), dtype=torch.float16, device=dev)
    wsp = torch.empty((q.quarot_decode_workspace_bytes(B, Hq, d, T),), dtype=torch.uint8, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty((max(2 * l2, 256 << 20),), dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()

    # The four stages of a step.  Each is launched through the C ABI on the
    # current stream; the timed loop replays them from CUDA graphs so that the
    # device time is not diluted by Python launch gaps.
    def s_rot():
        q.quarot_rotate_quant(xt, st, q_out=aq, scale_out=asx)

    def s_gemm():
        q.quarot_w4a4_gemm(aq, asx, wq, wsc, y=y)

    def s_kvw():
        q.quarot_kv_write(k_new, v_new, T - 1, *cache)

    def s_dec():
        q.quarot_decode_attn(q_dec, *cache, T=T, out=out, workspace=wsp)

    stages_fn = [s_rot, s_gemm, s_kvw, s_dec]
    LAUNCHES_PER_STEP = 1 + 1 + 1 + 2

    def step():
        for f in stages_fn:
            f()

    for _ in range(args.warmup):
        flush.zero_()
        step()
    q.quarot_check_error(stream)

    graphs = None
    try:
        g_step = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_step):
            step()
        g_stage = []
        for f in stages_fn:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                f()
            g_stage.append(g)
        graphs = (g_step, g_stage)
    except Exception as exc:  # graph capture unavailable: time direct launches
        print(f"# CUDA graph capture failed ({exc}); timing direct launches", file=sys.stderr)
    run_step = graphs[0].replay if graphs else step
    run_stage = [g.replay for g in graphs[1]] if graphs else stages_fn
    for _ in range(2):
        flush.zero_()
        run_step()
    torch.cuda.synchronize()
    q.quarot_check_error(stream)

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        for i in range(args.steps):
            flush.zero_()  # L2 flush between timed steps (outside the step's events)
            evs[i][0].record(stream)
            run_step()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        timed_samples = len(clocks.lines)
        # a short timed region may end before nvidia-smi reports: keep the same
        # load running (untimed) until a few samples exist
        t_end = time.time() + 3.0
        while len(clocks.lines) < timed_samples + 5 and time.time() < t_end:
            for _ in range(50):
                flush.zero_()
                run_step()
            torch.cuda.synchronize()
    q.quarot_check_error(stream)
    step_ms = np.array([a.elapsed_time(b) for a, b in evs])
    total_ms = _job_time_ms(float(step_ms.sum()), ws, dev)
    if ws > 1:
        dist.barrier()
    value = _job_rate(M_TOK, args.steps, ws, total_ms)

    # per-stage device times (same cold-L2 protocol, each stage replayed alone)
    reps = max(10, min(args.steps, 100))
    stage_ms = []
    for f in run_stage:
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            f()
            b.record(stream)
        torch.cuda.synchronize()
        stage_ms.append(float(np.mean([a.elapsed_time(b) for a, b in ev])))
    stage_ms = np.array(stage_ms)

    # ---------------- e2e: host buffers through the C ABI, copies inside the timed region
    # Every step copies its inputs (X, the new K/V token, q) from pinned host
    # memory and reads its results (Y, the decode output) back.  The steps are
    # pipelined the way a serving loop would run them: host-to-device copies on
    # one stream, the four kernels on the compute stream, device-to-host copies
    # on a third, with double-buffered device tensors, so step i+1's input copy
    # overlaps step i's kernels.  The per-step traffic (X 50 MB, W 25 MB, Y 17 MB,
    # KV cache 69 MB) exceeds L2, so no flush is needed between steps.
    x_h = torch.from_numpy(x).pin_memory()
    kn_h, vn_h, q_h = k_new.cpu().pin_memory(), v_new.cpu().pin_memory(), q_dec.cpu().pin_memory()
    xd = [torch.empty_like(xt) for _ in range(2)]
    kd = [torch.empty_like(k_new) for _ in range(2)]
    vd = [torch.empty_like(v_new) for _ in range(2)]
    qd = [torch.empty_like(q_dec) for _ in range(2)]
    aqd = [torch.empty_like(aq) for _ in range(2)]
    asd = [torch.empty_like(asx) for _ in range(2)]
    yd = [torch.empty_like(y) for _ in range(2)]
    od = [torch.empty_like(out) for _ in range(2)]
    y_h = [torch.empty_like(y, device="cpu").pin_memory() for _ in range(2)]
    o_h = [torch.empty_like(out, device="cpu").pin_memory() for _ in range(2)]
    h2d_st, d2h_st = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of the slot copied
    ev_comp = [torch.cuda.Event() for _ in range(2)]  # kernels of the slot done
    ev_out = [torch.cuda.Event() for _ in range(2)]   # results of the slot copied out

    def e2e_run(n):
        for i in range(n):
            sl = i % 2
            if i >= 2:
                h2d_st.wait_event(ev_comp[sl])  # slot's inputs no longer read
            with torch.cuda.stream(h2d_st):
                xd[sl].copy_(x_h, non_blocking=True)
                kd[sl].copy_(kn_h, non_blocking=True)
                vd[sl].copy_(vn_h, non_blocking=True)
                qd[sl].copy_(q_h, non_blocking=True)
            ev_in[sl].record(h2d_st)
            stream.wait_event(ev_in[sl])
            if i >= 2:
                stream.wait_event(ev_out[sl])  # slot's results already read back
            q.quarot_rotate_quant(xd[sl], st, q_out=aqd[sl], scale_out=asd[sl], stream=stream)
            q.quarot_w4a4_gemm(aqd[sl], asd[sl], wq, wsc, y=yd[sl], stream=stream)
            q.quarot_kv_write(kd[sl], vd[sl], T - 1, *cache, stream=stream)
            q.quarot_decode_attn(qd[sl], *cache, T=T, out=od[sl], workspace=wsp, stream=stream)
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
    h2d = (xd[0].numel() * 2 + kd[0].numel() * 2 + vd[0].numel() * 2 + qd[0].numel() * 2)
    d2h = y.numel() * 2 + out.numel() * 2
    # the results of the last step match the device-only path's
    torch.cuda.synchronize()
    sl = (args.steps - 1) % 2
    if not (torch.equal(y_h[sl], y.cpu()) and torch.equal(o_h[sl], out.cpu())):
        raise RuntimeError("e2e results differ from the device-resident step")

    # ---------------- roofline of the dominant kernel (GEMM, tensor pipe)
    hbm_peak, bf16_peak, peak_src = _peaks()
    fp8_peak = bf16_peak * (4.5 / 2.25)  # kind::f8f6f4 executes the INT4 contraction
    gemm_ms = float(stage_ms[1])
    gemm_tflops = 2.0 * M_TOK * N_OUT * K_DIM / (gemm_ms / 1000.0) / 1e12
    rq_bytes = M_TOK * K_DIM * 2 + M_TOK * K_DIM // 2 + M_TOK * 2
    dec_bytes = B * Hkv * T * (d // 2) * 2 + B * Hkv * T * 2 * 2 + B * Hq * d * 2 * 2
    kvw_bytes = 2 * (B * Hkv * d * 2 + B * Hkv * (d // 2 + 2))
    stages = {
        "rotate_quant": {"ms": float(stage_ms[0]), "GB/s": rq_bytes / (stage_ms[0] / 1e3) / 1e9,
                         "frac_hbm": rq_bytes / (stage_ms[0] / 1e3) / 1e9 / hbm_peak},
        "w4a4_gemm": {"ms": gemm_ms, "TOPS": gemm_tflops, "frac_fp8_peak": gemm_tflops / fp8_peak},
        "kv_write_append": {"ms": float(stage_ms[2]), "GB/s": kvw_bytes / (stage_ms[2] / 1e3) / 1e9},
        "decode_attn": {"ms": float(stage_ms[3]), "GB/s": dec_bytes / (stage_ms[3] / 1e3) / 1e9,
                        "frac_hbm": dec_bytes / (stage_ms[3] / 1e3) / 1e9 / hbm_peak},
    }
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int4+f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "tokens_per_step": M_TOK, "l2": "flushed between steps (2x L2 write)",
                   "parallelism": f"replicas x{ws}", "launch": "CUDA graph per step" if graphs else "direct"},
        "roofline": {"bound": "tensor", "kernel": "w4a4_gemm", "achieved": gemm_tflops, "peak": fp8_peak,
                     "unit": "TFLOP/s", "frac": gemm_tflops / fp8_peak, "traffic": GEMM_TRAFFIC_BYTES,
                     "peak_source": f"{peak_src} bf16 x 2 (fp8/bf16 nominal ratio)"},
        "stages": stages,
        "e2e": {"value": e2e_val, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "pipeline": "per-step H2D, kernels and D2H on three streams, double-buffered; no L2 flush "
                            "(per-step traffic > L2)"},
        "gpu_launches": LAUNCHES_PER_STEP * args.steps,
        "clocks": dict(clocks.summary(), samples_in_timed_region=timed_samples),
    }
    if rank == 0 and not args.no_extra:
        line["other_configs"] = _other_configs(q, W, dev, stream, flush, hbm_peak, fp8_peak)
    if rank == 0 and not args.no_cpu_baseline:
        import torch as _t  # noqa: F401

        cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
        v, dt, desc = cpu_oracle_sample(rows=32, seqs=2)
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc,
                                "sample_seconds": dt}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


def _other_configs(q, W, dev, stream, flush, hbm_peak, fp8_peak, reps=20):
    """The other measured workloads: rotate+quant of 2048 x 4096 (H_4096, HBM
    roof), the fused RMSNorm + rotate + quant at 2048 x 4096 and 2048 x 12288,
    decode over the asymmetric KV cache at the kv4 size, causal prefill attention
    (4 x 2048 tokens, fp16 tensor roof), and the GEMM sweep M in {512, 2048, 8192} x K 4096 x N in {4096, 12288}
    (tensor roof).  Same cold-L2 protocol as the stages; rank 0 only."""
    import torch

    def timed(f):
        for _ in range(3):
            f()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            f()
            b.record(stream)
        torch.cuda.synchronize()
        q.quarot_check_error(stream)
        return float(np.mean([a.elapsed_time(b) for a, b in ev]))

    res = {}
    x, _, s = W.layer_inputs("rotq4096")
    xt, st = torch.from_numpy(x).to(dev), torch.from_numpy(s).to(dev)
    M, d = x.shape
    qo = torch.empty((M, d // 2), dtype=torch.uint8, device=dev)
    so = torch.empty((M,), dtype=torch.float16, device=dev)
    ms = timed(lambda: q.quarot_rotate_quant(xt, st, q_out=qo, scale_out=so, stream=stream))
    nbytes = M * d * 2 + M * d // 2 + M * 2
    res["rotate_quant_2048x4096"] = {"ms": ms, "GB/s": nbytes / (ms / 1e3) / 1e9,
                                     "frac_hbm": nbytes / (ms / 1e3) / 1e9 / hbm_peak}
    ms = timed(lambda: q.quarot_rmsnorm_rotate_quant(xt, st, eps=1e-6, q_out=qo, scale_out=so, stream=stream))
    res["rmsnorm_rotate_quant_2048x4096"] = {"ms": ms, "GB/s": nbytes / (ms / 1e3) / 1e9,
                                             "frac_hbm": nbytes / (ms / 1e3) / 1e9 / hbm_peak}
    del xt, qo, so
    x, _, s = W.layer_inputs("down_proj", N=0)
    xt, st = torch.from_numpy(x).to(dev), torch.from_numpy(s).to(dev)
    M, d = x.shape
    qo = torch.empty((M, d // 2), dtype=torch.uint8, device=dev)
    so = torch.empty((M,), dtype=torch.float16, device=dev)
    ms = timed(lambda: q.quarot_rmsnorm_rotate_quant(xt, st, eps=1e-6, q_out=qo, scale_out=so, stream=stream))
    nbytes = M * d * 2 + M * d // 2 + M * 2
    res["rmsnorm_rotate_quant_2048x12288"] = {"ms": ms, "GB/s": nbytes / (ms / 1e3) / 1e9,
                                              "frac_hbm": nbytes / (ms / 1e3) / 1e9 / hbm_peak}
    # the FP16-arithmetic rotation variant on the same 2048 x 12288 rows
    ms = timed(lambda: q.quarot_rotate_quant_fp16(xt, st, q_out=qo, scale_out=so, stream=stream))
    res["rotate_quant_fp16_2048x12288"] = {"ms": ms, "GB/s": nbytes / (ms / 1e3) / 1e9,
                                           "frac_hbm": nbytes / (ms / 1e3) / 1e9 / hbm_peak}
    del xt, qo, so
    # cross-head Hadamard + INT4 of a prefill-sized attention output (2048 tokens x 32 heads x 128)
    zt = torch.from_numpy(W.query(2048, 32, 128, 77).reshape(2048, 4096)).to(dev)
    zq = torch.empty((2048, 2048), dtype=torch.uint8, device=dev)
    zs = torch.empty((2048,), dtype=torch.float16, device=dev)
    ms = timed(lambda: q.quarot_crosshead_rotate_quant(zt, 32, q_out=zq, scale_out=zs, stream=stream))
    nbytes = 2048 * 4096 * 2 + 2048 * 2048 + 2048 * 2
    res["crosshead_rotate_quant_2048x32x128"] = {"ms": ms, "GB/s": nbytes / (ms / 1e3) / 1e9,
                                                 "frac_hbm": nbytes / (ms / 1e3) / 1e9 / hbm_peak}
    del zt, zq, zs
    # asymmetric KV cache (group 128, zero point, clip 0.95): decode at the kv4 size
    k, v, qq = W.kv_inputs("kv4")
    B, T, Hkv, d = k.shape
    Hq = qq.shape[1]
    ac = q.new_kv_cache_asym(B, Hkv, T, d, dev)
    q.quarot_kv_write_asym(torch.from_numpy(k).to(dev), torch.from_numpy(v).to(dev), 0, *ac, stream=stream)
    qd = torch.from_numpy(qq).to(dev)
    od = torch.empty((B, Hq, d), dtype=torch.float16, device=dev)
    wsd = torch.empty((q.quarot_decode_workspace_bytes(B, Hq, d, T),), dtype=torch.uint8, device=dev)
    ms = timed(lambda: q.quarot_decode_attn_asym(qd, *ac, T=T, out=od, workspace=wsd, stream=stream))
    nbytes = B * Hkv * T * (d // 2) * 2 + B * Hkv * T * (2 + 2) * 2 + B * Hq * d * 2 * 2
    res["decode_attn_asym_kv4"] = {"ms": ms, "GB/s": nbytes / (ms / 1e3) / 1e9,
                                   "frac_hbm": nbytes / (ms / 1e3) / 1e9 / hbm_peak}
    del ac, qd, od, wsd
    # Init (prefill) attention over the INT4 cache: 4 prompts x 2048 tokens,
    # Hq 32 / Hkv 8, causal; flops are the useful ones (t <= i), 4 d per pair
    k, v, qq = W.prefill_inputs("prefill")
    B, T, Hkv, d = k.shape
    Hq = qq.shape[2]
    pc = q.new_kv_cache(B, Hkv, T, d, dev)
    q.quarot_kv_write(torch.from_numpy(k).to(dev), torch.from_numpy(v).to(dev), 0, *pc, stream=stream)
    qp = torch.from_numpy(qq).to(dev)
    op = torch.empty_like(qp)
    ms = timed(lambda: q.quarot_prefill_attn(qp, *pc, out=op, stream=stream))
    tf = 4.0 * B * Hq * d * (T * (T + 1) / 2) / (ms / 1e3) / 1e12
    res["prefill_attn_4x2048_h32kv8"] = {"ms": ms, "TFLOP/s": tf, "frac_f16_peak": tf / (fp8_peak / 2)}
    del pc, qp, op
    # rotate+quant of the sweep's activations (M x 4096, 8 outlier channels),
    # for the layer rate M / (t_rotate_quant + t_gemm) of each sweep shape
    xs, _, ss = W.layer_inputs("sweep", M=8192)
    rot_ms = {}
    sst = torch.from_numpy(ss).to(dev)
    for M in (512, 2048, 8192):
        xt = torch.from_numpy(np.ascontiguousarray(xs[:M])).to(dev)
        qo = torch.empty((M, 2048), dtype=torch.uint8, device=dev)
        so = torch.empty((M,), dtype=torch.float16, device=dev)
        rot_ms[M] = timed(lambda: q.quarot_rotate_quant(xt, sst, q_out=qo, scale_out=so, stream=stream))
        nb = M * 4096 * 2 + M * 2048 + M * 2
        res[f"rotate_quant_{M}x4096"] = {"ms": rot_ms[M], "GB/s": nb / (rot_ms[M] / 1e3) / 1e9,
                                         "frac_hbm": nb / (rot_ms[M] / 1e3) / 1e9 / hbm_peak}
        del xt, qo, so
    g = torch.Generator(device="cpu").manual_seed(1234)
    K = 4096
    for N in (4096, 12288):
        wq = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, generator=g).to(dev)
        ws_ = (torch.rand(N, generator=g) * 0.01 + 0.001).half().to(dev)
        for M in (512, 2048, 8192):
            aq = torch.randint(0, 256, (M, K // 2), dtype=torch.uint8, generator=g).to(dev)
            as_ = (torch.rand(M, generator=g) * 0.1 + 0.01).half().to(dev)
            y = torch.empty((M, N), dtype=torch.float16, device=dev)
            ms = timed(lambda: q.quarot_w4a4_gemm(aq, as_, wq, ws_, y=y, stream=stream))
            tf = 2.0 * M * N * K / (ms / 1e3) / 1e12
            res[f"w4a4_gemm_{M}x{K}x{N}"] = {"ms": ms, "TOPS": tf, "frac_fp8_peak": tf / fp8_peak,
                                               "layer_tokens_per_s": M / ((ms + rot_ms[M]) / 1e3)}
            del aq, as_, y
        del wq, ws_
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the rotate 2048x4096 and GEMM sweep lines")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
