"""Benchmark of the MXFP8 attention training step (forward + backward).

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl lpfa|reference]

A step is one pass of the whole hot path on one batch of synthetic input of
the B8 H32 S8192 D128 causal LLM training shape: MX quantization of Q, K (1x32)
and V (32 along tokens), the forward kernel, MX quantization of Q, K, dO
(32x32) and V (1x32), and the backward (D_i preprocess, main kernel).  Inputs
(512 MiB per bf16 tensor) are larger than L2, so no flush is needed.

Multi-GPU: every rank runs its own replica of the step on its own seeded
inputs (the path shards over (batch, head) with no exchange step); the time
is the max over ranks and the value counts the work of all ranks (weak
scaling).  --impl reference times the fp64 CPU oracle on a bounded sample of
the same workload (rank 0 only).

Beside the step the JSON line reports, each measured in the same run: the
bf16 variants of the forward and backward kernels on the same inputs (the
MXFP8 / bf16 ratio), the fused RMSNorm + MX quantizer, the tensor pipe's
block-scaled MMA rate, this library's and cuBLAS's MXFP8 GEMM 8192^3 (the
fastest of the two is the roofline's peak), the quantizing GEMM, the MXFP4,
NVFP4 and MXFP6 GEMMs, the jagged GEMM-Norm backward, the end-to-end rate
from pinned host memory with the copy rates that bound it, and the SM clocks
sampled by nvidia-smi during the run (raw samples in $LPFA_CLOCK_LOG_DIR,
default the system temp directory).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "MXFP8 attn fwd/bwd PFLOP/s (B8 H32 S8192 D128 causal); % of FP8 MMA peak"
WORKLOAD = "llm"
FP8_OVER_BF16 = 2.0      # nominal dense fp8 : bf16 tensor-core ratio
NORM_ITERS = 20          # timed launches of the fused RMSNorm + MX quantizer
E2E_MIN_STEPS = 40       # steps the end-to-end leg times at least


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            return json.load(fh)
    except (OSError, ValueError):
        return None


def smi_gpu_id(local: int) -> str:
    """The GPU's identity for nvidia-smi --id: its UUID (nvidia-smi numbers
    GPUs physically and ignores CUDA_VISIBLE_DEVICES, so the CUDA ordinal can
    name another process's GPU), else its PCI bus id, else the ordinal."""
    try:
        props = torch.cuda.get_device_properties(local)
        uuid = str(getattr(props, "uuid", "") or "")
        if uuid:
            return uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        if hasattr(props, "pci_bus_id"):
            return f"{props.pci_domain_id:08X}:{props.pci_bus_id:02X}:{props.pci_device_id:02X}.0"
    except Exception:
        pass
    return str(local)


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    def __init__(self, index):
        self.index = index
        self.proc = None
        # raw samples; the summary goes into the JSON line
        log_dir = os.environ.get("LPFA_CLOCK_LOG_DIR", tempfile.gettempdir())
        self.path = os.path.join(log_dir, f"bench_clocks_{os.getpid()}.csv")

    def __enter__(self):
        os.makedirs(os.path.dirname(self.path), exist_ok=True)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
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

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            for line in fh:
                f = [x.strip() for x in line.split(",")]
                if len(f) < 9:
                    continue
                try:
                    sm.append(float(f[1])); smax.append(float(f[2]))
                    power.append(float(f[3]))
                except ValueError:
                    continue
                for n, v in zip(names, f[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"],
                    "gpu": self.index}
        loaded = [s for s, p in zip(sm, power) if p > 0.5 * max(power)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax),
                "power_w_max": max(power), "samples": len(sm),
                "reasons": sorted(reasons), "gpu": self.index}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------- CPU oracle
def oracle_sample(rows: int, seed: int = 2):
    """Time the fp64 oracle (forward + backward) on one head of the workload
    restricted to the last ``rows`` queries (which see every earlier key) and
    the last ``rows`` keys.  Returns (flops of the sample, seconds, text)."""
    import numpy as np
    from oracle import attention as A
    w = workloads.get_config(WORKLOAD)
    g = torch.Generator().manual_seed(seed)
    S, D = w.seqlen, w.head_dim
    q, k, v, do = (torch.randn(1, S, 1, D, generator=g).to(torch.bfloat16)
                   for _ in range(4))
    r = np.arange(S - rows, S)
    t0 = time.perf_counter()
    fw = A.mx_attention_fwd(q, k, v, causal=True, softmax_scale=w.softmax_scale,
                            rows=r, kv_tile=A.FWD_KEY_TILE)
    o16 = torch.from_numpy(np.nan_to_num(fw["o"])).to(torch.bfloat16)
    A.mx_attention_bwd(q, k, v, o16, do, np.nan_to_num(fw["lse"]), causal=True,
                       softmax_scale=w.softmax_scale, q_rows=r, k_rows=r)
    dt = time.perf_counter() - t0
    visible = float(sum(i + 1 for i in r))          # (query, key) pairs
    flops = (4.0 + 10.0) * D * visible              # fwd + bwd convention
    text = (f"one head (b0,h0) of B8 H32 S8192 D128 causal: last {rows} query rows "
            f"(fwd, dQ) and last {rows} key rows (dK, dV), fp64 numpy oracle; "
            f"flops = 14*D*#(visible query,key) pairs of those query rows")
    return flops, dt, text


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    rows = 2048
    for _ in range(args.warmup):
        oracle_sample(rows)
    tot_f = tot_t = 0.0
    for _ in range(args.steps):
        f, t, text = oracle_sample(rows)
        tot_f += f; tot_t += t
    value = tot_f / tot_t / 1e15
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "PFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot_t / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16)",
        "config": {"workload": "llm: B8 H32 S8192 D128 causal, bounded sample",
                   "global_batch": 8, "seq_len": 8192, "parallelism": "none"},
        "cpu_baseline": {"value": value, "unit": "PFLOP/s", "cores": cores,
                         "kind": "oracle", "sample": text},
        "e2e": {"value": value, "unit": "PFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- GPU arm
def run_lpfa(args, world, rank, local):
    from mxfp8_block_scaled_quantizer_gb300 import build
    build()
    from mxfp8_block_scaled_quantizer_gb300 import lpfa as L

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = workloads.get_config(WORKLOAD)
    B, S, H, Hkv, D = w.batch, w.seqlen, w.heads_q, w.heads_kv, w.head_dim
    T = B * S
    # seeded synthetic inputs (workloads recipe), one replica per rank
    wr = workloads.custom(**{**w.__dict__, "seed": w.seed + rank})
    x = workloads.make_inputs(wr)
    host = {n: x[n].reshape(T, -1, D).contiguous().pin_memory()
            for n in ("q", "k", "v", "do")}
    q, k, v, do = (host[n].to(dev, non_blocking=True) for n in ("q", "k", "v", "do"))
    torch.cuda.synchronize()
    seqs = L.dense_seqs(B, S)
    desc = L.attn_desc(seqs, H, Hkv, D, w.causal, w.softmax_scale)
    fwd_flops, bwd_flops = workloads.attn_flops(w)

    # persistent buffers
    o = torch.empty((T, H, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((H, T), dtype=torch.float32, device=dev)
    fws = torch.empty(L.fwd_workspace_size(desc), dtype=torch.uint8, device=dev)
    dq = torch.empty((T, H, D), dtype=torch.float16, device=dev)
    dk = torch.empty((T, Hkv, D), dtype=torch.bfloat16, device=dev)
    dv = torch.empty((T, Hkv, D), dtype=torch.bfloat16, device=dev)
    bws = torch.empty(L.bwd_workspace_size(desc), dtype=torch.uint8, device=dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)
    launches_per_step = 3 + 1 + 4 + 2      # quantize x3, fwd, quantize x4, bwd x2

    def step(times=None):
        e = [ev() for _ in range(6)] if times is not None else None
        if e: e[0].record()
        mq, mk, mv = L.quantize_forward_operands(q, k, v, seqs)
        if e: e[1].record()
        L.attention_forward_mx(mq, mk, mv, desc, o, lse, fws)
        if e: e[2].record()
        bq, bk, bv, bdo = L.quantize_backward_operands(q, k, v, do, seqs)
        if e: e[3].record()
        L.attention_backward_mx(bq, bk, bv, bdo, o, do, lse, desc, dq, dk, dv, bws)
        if e:
            e[4].record()
            times.append(e)

    clk = ClockSampler(smi_gpu_id(local)).__enter__()   # warm-up to end of e2e
    time.sleep(1.0)                          # let the sampler start
    for _ in range(args.warmup):
        step()
    L.lpfa_check(fws)
    L.lpfa_check(bws)
    torch.cuda.synchronize()

    parts = []
    _barrier(world)
    torch.cuda.synchronize()
    t0, t1 = ev(), ev()
    t0.record()
    for _ in range(args.steps):
        step(parts)
    t1.record()
    torch.cuda.synchronize()
    _barrier(world)
    L.lpfa_check(fws)
    L.lpfa_check(bws)
    ms = t0.elapsed_time(t1) / args.steps
    ms_max = _max_over_ranks(ms, world)
    qf = statistics.mean(p[0].elapsed_time(p[1]) for p in parts)
    fw = statistics.mean(p[1].elapsed_time(p[2]) for p in parts)
    qb = statistics.mean(p[2].elapsed_time(p[3]) for p in parts)
    bw = statistics.mean(p[3].elapsed_time(p[4]) for p in parts)

    # ---- the bf16 variants of the same kernels on the same inputs, for the
    # MXFP8 / bf16 ratio (kernel against kernel; the MXFP8 side also with its
    # operand quantization)
    bf16 = {}
    try:
        ob, lb, fwsb = torch.empty_like(o), torch.empty_like(lse), torch.empty_like(fws)
        dqb, dkb, dvb = torch.empty_like(dq), torch.empty_like(dk), torch.empty_like(dv)
        bwsb = torch.empty_like(bws)
        fwd_b = lambda: L.attention_forward_bf16(q, k, v, desc, ob, lb, fwsb)
        bwd_b = lambda: L.attention_backward_bf16(q, k, v, ob, do, lb, desc, dqb, dkb, dvb, bwsb)
        for _ in range(2):
            fwd_b(); bwd_b()
        torch.cuda.synchronize()
        ts = []
        for _ in range(max(3, args.steps)):
            e = [ev() for _ in range(3)]
            e[0].record(); fwd_b(); e[1].record(); bwd_b(); e[2].record()
            ts.append(e)
        torch.cuda.synchronize()
        L.lpfa_check(fwsb)
        L.lpfa_check(bwsb)
        fb = statistics.mean(t[0].elapsed_time(t[1]) for t in ts)
        bb = statistics.mean(t[1].elapsed_time(t[2]) for t in ts)
        bf16 = {"fwd_tflops": fwd_flops / fb / 1e9, "bwd_tflops": bwd_flops / bb / 1e9,
                "fwd_ms": fb, "bwd_ms": bb,
                "mxfp8_over_bf16": {"fwd": fb / fw, "bwd": bb / bw,
                                    "fwd_incl_quantize": fb / (fw + qf),
                                    "bwd_incl_quantize": bb / (bw + qb)}}
        del ob, lb, fwsb, dqb, dkb, dvb, bwsb
    except Exception as exc:
        bf16 = {"error": repr(exc)[:200]}

    # ---- the fused RMSNorm + MX quantizer on the model's hidden state: Q
    # viewed as [T, H * D] (hidden 4096, 512 MiB, larger than L2), square
    # blocks with compact and both tensor-core scale layouts and rstd; beside
    # it, for context, the two-pass form (torch's bf16 rms_norm, then this
    # library's quantizer)
    wn = (1.0 + 0.1 * torch.randn(H * D, generator=torch.Generator().manual_seed(7)))
    wn = wn.bfloat16().to(dev)
    fused = lambda: L.rmsnorm_mx_quantize(q, wn, 1e-6, L.LPFA_BLK_32X32, seqs)
    two_pass = lambda: L.mx_quantize(
        torch.nn.functional.rms_norm(q.view(T, H * D), (H * D,), wn, 1e-6).view(T, H, D),
        L.LPFA_BLK_32X32, seqs)

    def _time(fn, iters=NORM_ITERS):
        for _ in range(3):
            res = fn()
        torch.cuda.synchronize()
        a_, b_ = ev(), ev()
        a_.record()
        for _ in range(iters):
            res = fn()
        b_.record()
        torch.cuda.synchronize()
        return a_.elapsed_time(b_) / iters, res

    norm_ms, (mn, rn) = _time(fused)
    norm_bytes = (q.numel() * 2 + wn.numel() * 2 + mn.data.numel() + mn.sf.numel()
                  + mn.sf_mma.numel() + mn.sf_mma_t.numel() + rn.numel() * 4)
    try:
        two_pass_ms = _time(two_pass)[0]
    except Exception:  # rms_norm missing from this torch
        two_pass_ms = None
    del mn, rn

    # ---- end to end through the public API with host buffers
    out_host = {"o": torch.empty((T, H, D), dtype=torch.bfloat16).pin_memory(),
                "dq": torch.empty((T, H, D), dtype=torch.float16).pin_memory(),
                "dk": torch.empty((T, Hkv, D), dtype=torch.bfloat16).pin_memory(),
                "dv": torch.empty((T, Hkv, D), dtype=torch.bfloat16).pin_memory()}

    # Copies overlap compute: inputs go up on their own stream into
    # triple-buffered device tensors (the upload of step i+2 may start as soon
    # as step i-1 is done, so the copy engine never waits for the step it
    # feeds), O comes back while the backward runs, dQ/dK/dV after it.  Every
    # copy of every timed step is inside the timed region, including the
    # first upload and the last download, which nothing overlaps; the e2e leg
    # times at least E2E_MIN_STEPS steps so that those two do not dominate.
    names = ("q", "k", "v", "do")
    nbuf = 3
    dev_in = [{n: torch.empty_like(host[n], device=dev) for n in names} for _ in range(nbuf)]
    cur = torch.cuda.current_stream()
    h2d_s, d2h_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    in_ready = [torch.cuda.Event() for _ in range(nbuf)]
    in_free = [torch.cuda.Event() for _ in range(nbuf)]
    for e in in_free:
        e.record(cur)

    def upload(i):
        b = i % nbuf
        with torch.cuda.stream(h2d_s):
            h2d_s.wait_event(in_free[b])
            for n in names:
                dev_in[b][n].copy_(host[n], non_blocking=True)
            in_ready[b].record(h2d_s)

    def e2e_step(i, nsteps):
        b = i % nbuf
        cur.wait_event(in_ready[b])
        if i + 2 < nsteps:
            upload(i + 2)
        x_ = dev_in[b]
        shp = lambda t, h: t.view(B, S, h, D)
        o_, lse_ = L.mx_attention_forward(shp(x_["q"], H), shp(x_["k"], Hkv), shp(x_["v"], Hkv),
                                          causal=w.causal, softmax_scale=w.softmax_scale,
                                          check=False)
        o_done = torch.cuda.Event()
        o_done.record(cur)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(o_done)
            o_.record_stream(d2h_s)
            out_host["o"].copy_(o_.view(T, H, D), non_blocking=True)
        dq_, dk_, dv_ = L.mx_attention_backward(shp(x_["q"], H), shp(x_["k"], Hkv),
                                                shp(x_["v"], Hkv), o_, shp(x_["do"], H), lse_,
                                                causal=w.causal, softmax_scale=w.softmax_scale,
                                                check=False)
        in_free[b].record(cur)
        g_done = torch.cuda.Event()
        g_done.record(cur)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(g_done)
            for t_, n in ((dq_, "dq"), (dk_, "dk"), (dv_, "dv")):
                t_.record_stream(d2h_s)
                out_host[n].copy_(t_.view(out_host[n].shape), non_blocking=True)

    def e2e_run(nsteps):
        for i in range(min(2, nsteps)):
            upload(i)
        for i in range(nsteps):
            e2e_step(i, nsteps)
        done = torch.cuda.Event()
        done.record(d2h_s)
        cur.wait_event(done)

    e2e_run(max(1, args.warmup))
    torch.cuda.synchronize()
    _barrier(world)
    e2e_steps = max(args.steps, E2E_MIN_STEPS)
    e0, e1 = ev(), ev()
    e0.record()
    e2e_run(e2e_steps)
    e1.record()
    torch.cuda.synchronize()
    clk.__exit__(None, None, None)
    e2e_ms = _max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in out_host.values())

    # the pinned-memory copy rates that bound the end-to-end leg: uploads
    # alone, downloads alone, and both at once on their two streams
    dev_out = {n: torch.empty(t.shape, dtype=t.dtype, device=dev) for n, t in out_host.items()}

    def _copies(up, down, reps=3):
        def once():
            h2d_s.wait_stream(cur)
            d2h_s.wait_stream(cur)
            if up:
                with torch.cuda.stream(h2d_s):
                    for n in names:
                        dev_in[0][n].copy_(host[n], non_blocking=True)
            if down:
                with torch.cuda.stream(d2h_s):
                    for n, t in dev_out.items():
                        out_host[n].copy_(t, non_blocking=True)
            cur.wait_stream(h2d_s)
            cur.wait_stream(d2h_s)
        once()                                  # untimed: first touch of the buffers
        torch.cuda.synchronize()
        c0, c1 = ev(), ev()
        c0.record(cur)
        for _ in range(reps):
            once()
        c1.record(cur)
        torch.cuda.synchronize()
        return c0.elapsed_time(c1) / reps

    t_up = _copies(True, False)
    t_down = _copies(False, True)
    t_both = _copies(True, True)
    copy_rates = {"h2d_gbs_alone": h2d / (t_up * 1e-3) / 1e9,
                  "d2h_gbs_alone": d2h / (t_down * 1e-3) / 1e9,
                  "both_ms": t_both, "h2d_ms_alone": t_up, "d2h_ms_alone": t_down,
                  "note": "2 GiB up + 2 GiB down per step; with both directions at "
                          "once the copies take both_ms, the floor of the e2e step"}
    del dev_out

    # ---- in-run MX MMA rates: the tensor pipe alone (lpfa_mma_peak), the
    # block-scaled GEMM 8192^3 of this library and of cuBLAS
    mma = {}
    try:
        mma["lpfa_mma_peak_tflops"] = L.lpfa_mma_peak() / 1e12
    except Exception as exc:
        mma["lpfa_mma_peak_tflops"] = None
        mma["mma_peak_note"] = repr(exc)[:160]
    try:
        M = N = K = 8192
        a = torch.randn(M, K, device=dev, dtype=torch.bfloat16)
        b = torch.randn(N, K, device=dev, dtype=torch.bfloat16)
        ga = L.mx_quantize(a.view(M, K // 128, 128), L.LPFA_BLK_1X32, L.dense_seqs(1, M), compact=False)
        gb = L.mx_quantize(b.view(N, K // 128, 128), L.LPFA_BLK_1X32, L.dense_seqs(1, N), compact=False)
        dmat = torch.empty(M, N, device=dev, dtype=torch.float32)
        A8, B8 = ga.data.view(M, K), gb.data.view(N, K)
        for _ in range(3):
            L.lpfa_mx_gemm(A8, ga.sf_mma, B8, gb.sf_mma, dmat)
        torch.cuda.synchronize()
        g0, g1 = ev(), ev()
        g0.record()
        for _ in range(10):
            L.lpfa_mx_gemm(A8, ga.sf_mma, B8, gb.sf_mma, dmat)
        g1.record()
        torch.cuda.synchronize()
        mma["lpfa_mx_gemm_tflops"] = 2.0 * M * N * K / (g0.elapsed_time(g1) / 10) / 1e9
        # the same GEMM with the quantizing epilogue (square blocks, compact
        # and both tensor-core scale layouts; no fp32 result)
        qo = torch.empty(M, N, device=dev, dtype=torch.uint8)
        qsf = torch.empty(M // 32, N // 32, device=dev, dtype=torch.uint8)
        qm = torch.empty(M // 128, N // 128, 512, device=dev, dtype=torch.uint8)
        qt = torch.empty(N // 128, M // 128, 512, device=dev, dtype=torch.uint8)
        gq = lambda: L.lpfa_mx_gemm_quantize(A8, ga.sf_mma, B8, gb.sf_mma, L.LPFA_BLK_32X32,
                                             qo, qsf, qm, qt)
        for _ in range(3):
            gq()
        torch.cuda.synchronize()
        g0.record()
        for _ in range(10):
            gq()
        g1.record()
        torch.cuda.synchronize()
        mma["lpfa_mx_gemm_quantize_32x32_tflops"] = 2.0 * M * N * K / (g0.elapsed_time(g1) / 10) / 1e9
        del qo, qsf, qm, qt
        try:
            a8 = A8.view(torch.float8_e4m3fn); b8 = B8.view(torch.float8_e4m3fn)
            sa = ga.sf_mma.view(torch.float8_e8m0fnu).reshape(-1)
            sb = gb.sf_mma.view(torch.float8_e8m0fnu).reshape(-1)
            for _ in range(3):
                torch._scaled_mm(a8, b8.t(), sa, sb, out_dtype=torch.bfloat16)
            torch.cuda.synchronize()
            g0.record()
            for _ in range(10):
                torch._scaled_mm(a8, b8.t(), sa, sb, out_dtype=torch.bfloat16)
            g1.record()
            torch.cuda.synchronize()
            mma["cublas_mxfp8_tflops"] = 2.0 * M * N * K / (g0.elapsed_time(g1) / 10) / 1e9
        except Exception as exc:  # library path not available in this torch
            mma["cublas_mxfp8_tflops"] = None
            mma["cublas_note"] = repr(exc)[:160]
        # the other block-scale formats on the same pair kernel (f3): dense
        # FP4 with MXFP4 and NVFP4 scales (kind::mxf4nvf4) and MXFP6 (E2M3)
        def _rate(fn):
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            g0.record()
            for _ in range(10):
                fn()
            g1.record()
            torch.cuda.synchronize()
            return 2.0 * M * N * K / (g0.elapsed_time(g1) / 10) / 1e9
        try:
            na, _, nsa = L.nvfp4_quantize(a)
            nb, _, nsb = L.nvfp4_quantize(b)
            mma["lpfa_nvfp4_gemm_tflops"] = _rate(
                lambda: L.lpfa_mx_gemm_fp4(na, nsa, nb, nsb, dmat, nvfp4=True))
            del na, nb, nsa, nsb
            fa = L.mx_quantize(a.view(M, K // 128, 128), L.LPFA_BLK_1X32, L.dense_seqs(1, M),
                               compact=False, fmt=L.LPFA_ELEM_E2M1)
            fb = L.mx_quantize(b.view(N, K // 128, 128), L.LPFA_BLK_1X32, L.dense_seqs(1, N),
                               compact=False, fmt=L.LPFA_ELEM_E2M1)
            pa4, pb4 = L.fp4_pack_dense(fa.data.view(M, K)), L.fp4_pack_dense(fb.data.view(N, K))
            mma["lpfa_mxfp4_gemm_tflops"] = _rate(
                lambda: L.lpfa_mx_gemm_fp4(pa4, fa.sf_mma, pb4, fb.sf_mma, dmat, nvfp4=False))
            del fa, fb, pa4, pb4
            sa6 = L.mx_quantize(a.view(M, K // 128, 128), L.LPFA_BLK_1X32, L.dense_seqs(1, M),
                                compact=False, fmt=L.LPFA_ELEM_E2M3)
            sb6 = L.mx_quantize(b.view(N, K // 128, 128), L.LPFA_BLK_1X32, L.dense_seqs(1, N),
                                compact=False, fmt=L.LPFA_ELEM_E2M3)
            pa6 = L.mx_pack_operand(sa6.data.view(M, K), L.LPFA_ELEM_E2M3)
            pb6 = L.mx_pack_operand(sb6.data.view(N, K), L.LPFA_ELEM_E2M3)
            mma["lpfa_mxfp6_gemm_tflops"] = _rate(
                lambda: L.lpfa_mx_gemm_fmt(pa6, sa6.sf_mma, pb6, sb6.sf_mma, dmat,
                                           L.LPFA_ELEM_E2M3, L.LPFA_ELEM_E2M3))
            del sa6, sb6, pa6, pb6
        except Exception as exc:
            mma["other_formats_note"] = repr(exc)[:160]
        del a, b, ga, gb, dmat
    except Exception as exc:
        mma["error"] = repr(exc)[:160]

    # ---- the jagged GEMM-Norm backward (16 jagged sequences, hidden 4096):
    # the RMSNorm backward fused with the 32x32 quantization of dY (both
    # orientations), then dX = dY W and dW = dY^T X on the block-scaled GEMM
    # with X and W kept quantized from the forward.  The rate counts the two
    # GEMMs' 4 T N K flops; the quantization of X and W is timed beside it.
    gn = {}
    try:
        cfg = workloads.GEMM_NORM
        lens = workloads.gemm_norm_lengths(cfg["batch"], cfg["len_min"], cfg["len_max"],
                                           cfg["seed"] + rank)
        Tn, Hn = int(lens.sum()), cfg["hidden"]
        gi = workloads.gemm_norm_inputs(Tn, Hn, Hn, cfg["seed"] + rank)
        xg, wg, gam, dzg = (gi[n].to(dev) for n in ("x", "w", "gamma", "dz"))
        del gi
        yg = xg @ wg.T                                   # the forward's bf16 Y
        rs = torch.rsqrt(yg.float().pow(2).mean(dim=1) + 1e-6)
        xq_, wq_ = L.mx_quantize_t(xg), L.mx_quantize_t(wg)
        ms_gn, _ = _time(lambda: L.gemm_norm_backward(xq_, wq_, yg, rs, gam, dzg), 10)
        ms_nq, _ = _time(lambda: L.rmsnorm_bwd_mx_quantize(yg, dzg, gam, rs), 10)
        ms_xw, _ = _time(lambda: (L.mx_quantize_t(xg), L.mx_quantize_t(wg)), 10)
        gflops = 4.0 * Tn * Hn * Hn
        nq_bytes = 6.0 * Tn * Hn                         # read Y, dZ; payload twice
        gn = {"workload": f"jagged: {cfg['batch']} sequences, lengths U[{cfg['len_min']}, "
                          f"{cfg['len_max']}] (T = {Tn}), hidden N = K = {Hn}",
              "ms": ms_gn, "tflops": gflops / ms_gn / 1e9,
              "norm_bwd_quantize_ms": ms_nq,
              "norm_bwd_quantize_gbs": nq_bytes / (ms_nq * 1e-3) / 1e9,
              "gemms_ms": ms_gn - ms_nq,
              "gemms_tflops": gflops / (ms_gn - ms_nq) / 1e9,
              "quantize_x_w_ms": ms_xw,
              "tflops_incl_quantize_x_w": gflops / (ms_gn + ms_xw) / 1e9,
              "context_pages_tflops": 1760.0,
              "context_note": "the pages' 1.76 PF/s is on other hardware and an unstated shape"}
        del xg, wg, gam, dzg, yg, rs, xq_, wq_
    except Exception as exc:
        gn = {"error": repr(exc)[:200]}

    peaks = _peaks()
    # Roofline denominator: the fastest dense block-scaled MXFP8 GEMM measured
    # in this run (this library's or cuBLAS's, M = N = K = 8192).  Beside it:
    # the tensor pipe's own rate (no memory traffic; an upper bound no GEMM
    # reaches), the measured burst bf16 GEMM rate x 2 (the nominal fp8:bf16
    # ratio) and the datasheet's ~4.5 PF/s.
    gemm_rates = {k: mma.get(k) for k in ("lpfa_mx_gemm_tflops", "cublas_mxfp8_tflops")
                  if mma.get(k)}
    bf16_burst_x2 = FP8_OVER_BF16 * (peaks or {}).get("bf16_tflops", 0.0) or None
    if gemm_rates:
        src_key = max(gemm_rates, key=gemm_rates.get)
        peak = gemm_rates[src_key]
        peak_src = {"lpfa_mx_gemm_tflops": "lpfa_mx_gemm",
                    "cublas_mxfp8_tflops": "cuBLAS MXFP8 (torch._scaled_mm)"}[src_key] + \
            " 8192^3, measured in this run (of measured)"
    elif bf16_burst_x2:
        peak = bf16_burst_x2
        peak_src = "measured bf16 burst x 2 (nominal fp8:bf16), MEASURED_PEAKS.json (of measured)"
    else:
        peak = 1900.0 * FP8_OVER_BF16
        peak_src = "fallback 1.9 PFLOP/s bf16 burst x 2 (of fallback)"
    pipe = mma.get("lpfa_mma_peak_tflops")
    hbm = peaks.get("hbm_gbs") if peaks else None
    hbm_src = "measured copy bandwidth, MEASURED_PEAKS.json (of measured)" if hbm else \
        "fallback 6.8 TB/s"
    hbm = hbm or 6800.0
    norm_gbs = norm_bytes / (norm_ms * 1e-3) / 1e9
    bwd_tflops = bwd_flops / bw / 1e9
    fwd_tflops = fwd_flops / fw / 1e9
    total = (fwd_flops + bwd_flops) * world
    value = total / (ms_max * 1e-3) / 1e15
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath):
        try:
            with open(tpath) as fh:
                traffic = json.load(fh).get("mx_attn_bwd_kernel_bytes_per_launch")
        except (OSError, ValueError):
            traffic = None
    line = {
        "metric": METRIC, "value": value, "unit": "PFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 (MXFP8, fp32 accumulate)", "data": "synthetic (seeded N(0,1) bf16)",
        "config": {"workload": "llm: B8 H32 S8192 D128 causal, fwd+bwd incl. MX quantization",
                   "global_batch": B * world, "seq_len": S, "heads": H, "head_dim": D,
                   "parallelism": f"replicas x{world} (shard over batch/heads, no collective)",
                   "l2": "no flush: every input tensor (512 MiB) is larger than L2"},
        "fwd": {"tflops": fwd_tflops, "ms": fw, "frac_of_peak": fwd_tflops / peak},
        "bwd": {"tflops": bwd_tflops, "ms": bw, "frac_of_peak": bwd_tflops / peak},
        "quantize_ms": {"fwd_operands": qf, "bwd_operands": qb},
        "bf16": bf16,
        "roofline": {"bound": "tensor",
                     "kernel": "mx_attn_bwd_kernel (lpfa_bwd call: D_i preprocess + main kernel)",
                     "achieved": bwd_tflops, "peak": peak, "unit": "TFLOP/s",
                     "frac": bwd_tflops / peak, "traffic": traffic,
                     "peak_source": peak_src,
                     "context": {
                         "mma_pipe_tflops": pipe,
                         "bwd_frac_of_pipe": bwd_tflops / pipe if pipe else None,
                         "fwd_frac_of_pipe": fwd_tflops / pipe if pipe else None,
                         "bf16_burst_x2_tflops": bf16_burst_x2,
                         "bwd_frac_of_bf16_burst_x2": bwd_tflops / bf16_burst_x2 if bf16_burst_x2 else None,
                         "datasheet_tflops": 4500.0}},
        "mma_rate_in_run": mma,
        "gemm_norm_bwd": gn,
        "rmsnorm_quantize": {
            "workload": f"x [{T}, {H * D}] bf16 (the llm Q tensor as hidden states), 32x32 blocks, "
                        "compact + both tensor-core scale layouts + rstd",
            "ms": norm_ms, "bytes_per_launch": norm_bytes, "achieved_gbs": norm_gbs,
            "peak_gbs": hbm, "frac": norm_gbs / hbm, "peak_source": hbm_src,
            "two_pass_ms": two_pass_ms,
            "two_pass": "torch bf16 rms_norm, then lpfa_mx_quantize (context)"},
        "e2e": {"value": total / (e2e_ms * 1e-3) / 1e15, "unit": "PFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms, "steps": e2e_steps, "copies": copy_rates},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    # clock-independent view: kernel time in SM clock cycles at the median
    # clock sampled under load
    mhz = line["clocks"].get("sm_mhz")
    if mhz:
        line["fwd"]["mcycles"] = fw * mhz * 1e-3
        line["bwd"]["mcycles"] = bw * mhz * 1e-3
        line["fwd"]["flop_per_cycle_per_sm"] = fwd_flops / (fw * mhz * 1e3) / \
            torch.cuda.get_device_properties(dev).multi_processor_count
        line["bwd"]["flop_per_cycle_per_sm"] = bwd_flops / (bw * mhz * 1e3) / \
            torch.cuda.get_device_properties(dev).multi_processor_count
    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
            f, t, text = oracle_sample(8192)
            cpu = {"value": f / t / 1e15, "unit": "PFLOP/s", "cores": cores,
                   "kind": "oracle", "sample": text, "seconds": t}
        line["cpu_baseline"] = cpu
        print(json.dumps(line))
    return 0


def run_profile_case(iters: int):
    """One small pass of the hot path for ncu captures: B4 H16 S8192 D128
    causal (128 MiB per bf16 tensor, larger than L2), the fused RMSNorm + MX
    quantizer on Q viewed as [32768, 2048], then fwd + bwd, ``iters`` times,
    no timing."""
    from mxfp8_block_scaled_quantizer_gb300 import build
    build()
    from mxfp8_block_scaled_quantizer_gb300 import lpfa as L
    B, S, H, D = 4, 8192, 16, 128
    g = torch.Generator(device="cuda").manual_seed(0)
    mk = lambda: torch.randn(B * S, H, D, device="cuda", dtype=torch.bfloat16, generator=g)
    q, k, v, do = mk(), mk(), mk(), mk()
    seqs = L.dense_seqs(B, S)
    desc = L.attn_desc(seqs, H, H, D, True, D ** -0.5)
    wn = torch.ones(H * D, device="cuda", dtype=torch.bfloat16)
    for _ in range(iters):
        L.rmsnorm_mx_quantize(q, wn, 1e-6, L.LPFA_BLK_32X32, seqs)
        mq, mk_, mv = L.quantize_forward_operands(q, k, v, seqs)
        o, lse, ws = L.attention_forward_mx(mq, mk_, mv, desc)
        bq, bk, bv, bdo = L.quantize_backward_operands(q, k, v, do, seqs)
        dq, dk, dv, bws = L.attention_backward_mx(bq, bk, bv, bdo, o, do, lse, desc)
    torch.cuda.synchronize()
    L.lpfa_check(ws)
    L.lpfa_check(bws)
    return 0


def run_profile_case_bf16(iters: int):
    """The bf16 forward (the two-query-tile kernel) on the profile case's
    attention shape, B4 H16 S8192 D128 causal, ``iters`` times, no timing."""
    from mxfp8_block_scaled_quantizer_gb300 import build
    build()
    from mxfp8_block_scaled_quantizer_gb300 import lpfa as L
    B, S, H, D = 4, 8192, 16, 128
    g = torch.Generator(device="cuda").manual_seed(0)
    mk = lambda: torch.randn(B * S, H, D, device="cuda", dtype=torch.bfloat16, generator=g)
    q, k, v = mk(), mk(), mk()
    seqs = L.dense_seqs(B, S)
    desc = L.attn_desc(seqs, H, H, D, True, D ** -0.5)
    for _ in range(iters):
        o, lse, ws = L.attention_forward_bf16(q, k, v, desc)
    torch.cuda.synchronize()
    L.lpfa_check(ws)
    return 0


def run_profile_case_gemm_norm(iters: int):
    """One small pass of the jagged GEMM-Norm backward for ncu captures: 4
    jagged sequences (lengths U[128, 8192], seed 5), hidden 4096 (X, Y, dZ
    larger than L2 together), ``iters`` times, no timing."""
    from mxfp8_block_scaled_quantizer_gb300 import build
    build()
    from mxfp8_block_scaled_quantizer_gb300 import lpfa as L
    lens = workloads.gemm_norm_lengths(4, 128, 8192, 5)
    T, H = int(lens.sum()), 4096
    g = torch.Generator(device="cuda").manual_seed(0)
    x = torch.randn(T, H, device="cuda", dtype=torch.bfloat16, generator=g)
    w = (torch.randn(H, H, device="cuda", generator=g) / H ** 0.5).bfloat16()
    gamma = torch.ones(H, device="cuda", dtype=torch.bfloat16)
    dz = torch.randn(T, H, device="cuda", dtype=torch.bfloat16, generator=g)
    y = x @ w.T
    rstd = torch.rsqrt(y.float().pow(2).mean(dim=1) + 1e-6)
    for _ in range(iters):
        xq, wq = L.mx_quantize_t(x), L.mx_quantize_t(w)
        L.gemm_norm_backward(xq, wq, y, rstd, gamma, dz)
    torch.cuda.synchronize()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="lpfa", choices=["lpfa", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-case", type=int, default=0, metavar="ITERS",
                    help="run the small ncu capture case ITERS times and exit")
    ap.add_argument("--case", default="attention", choices=["attention", "gemm_norm", "bf16_fwd"],
                    help="which small case --profile-case runs")
    args = ap.parse_args()
    if args.profile_case:
        if args.case == "gemm_norm":
            return run_profile_case_gemm_norm(args.profile_case)
        if args.case == "bf16_fwd":
            return run_profile_case_bf16(args.profile_case)
        return run_profile_case(args.profile_case)
    world, rank, local = _dist()
    try:
        if args.impl == "reference":
            return run_reference(args, world, rank)
        return run_lpfa(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
