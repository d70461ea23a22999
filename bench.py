#!/usr/bin/env python
"""Benchmark of the QLoRA NF4 frozen-base linear layer on B300.

One step = one pass of the whole hot path over one synthetic batch of the Llama-3-8B-shaped
attention projection (W 4096x4096 fp32 ~ N(0, 0.02), X/dY 4096x4096 bf16 ~ N(0, 1), r = 16,
alpha = 32): nf4_quantize -> nf4_dequantize -> qlora_linear_fwd -> qlora_linear_bwd.
value = (4 M N K + 6 M r (N + K)) / step time, in TFLOP/s (fwd+bwd model FLOPs; the
quantize/dequantize inside the step add time, not FLOPs).

--impl reference times the CPU oracle (the plain C restatement of the method) on a bounded
sample of the same workload, scaled to a whole step.

Prints one JSON line (rank 0).  Under torchrun (WORLD_SIZE > 1) every rank runs its own batch
(weak scaling) and the adapter gradients dA, dB are summed over ranks with one all-reduce per
step, the data-parallel exchange of the layer.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "QLoRA NF4 linear fwd+bwd TFLOP/s (Llama-8B shapes); NF4 dequant GB/s"
WORKLOAD = "llama3-8b-attn-proj: W 4096x4096 NF4 (blk64, double-quant blk256), M=4096 tokens, r=16, alpha=32"
L2_FLUSH_BYTES = 512 << 20


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return dict(hbm_gbs=p["hbm_gbs"], bf16_tflops=p["bf16_tflops"],
                    bf16_tflops_sustained=p.get("bf16_tflops_sustained"), source="measured")
    except Exception:
        return dict(hbm_gbs=6400.0, bf16_tflops=1800.0, bf16_tflops_sustained=1400.0, source="fallback")


def new_events(n):
    """n timing events whose CUDA handles exist (torch creates them on first record)."""
    import torch
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in ev:
        e.record()
    torch.cuda.synchronize()
    assert all(e.cuda_event for e in ev)
    return ev


def layer_flops(M, N, K, r):
    return 4.0 * M * N * K + 6.0 * M * r * (N + K)


# ---------------------------------------------------------------------------------------
# Clock sampling during the timed region (NVML, the library behind nvidia-smi)
# ---------------------------------------------------------------------------------------
REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
           0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
           0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}


class _NVML:
    """Minimal ctypes binding of NVML (the library nvidia-smi reads clocks from)."""
    CLOCK_SM = 1

    def __init__(self):
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")

    def handle(self, torch_dev):
        import torch
        h = ctypes.c_void_p()
        props = torch.cuda.get_device_properties(torch_dev)
        uuid = str(getattr(props, "uuid", "") or "")
        if uuid:
            u = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            if self.lib.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(h)) == 0:
                return h
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        idx = torch_dev.index or 0
        if vis and all(v.strip().isdigit() for v in vis.split(",")):
            idx = int(vis.split(",")[idx])
        if self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(idx), ctypes.byref(h)) != 0:
            raise RuntimeError("no NVML handle")
        return h

    def clock(self, h, max_clock=False):
        v = ctypes.c_uint()
        f = self.lib.nvmlDeviceGetMaxClockInfo if max_clock else self.lib.nvmlDeviceGetClockInfo
        return v.value if f(h, ctypes.c_int(self.CLOCK_SM), ctypes.byref(v)) == 0 else None

    def reasons(self, h):
        v = ctypes.c_ulonglong()
        f = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        return v.value if f(h, ctypes.byref(v)) == 0 else 0


class ClockSampler:
    def __init__(self, torch_dev):
        self.samples = []
        self.max_mhz = None
        self._stop = threading.Event()
        self._h = None
        try:
            self.nv = _NVML()
            self._h = self.nv.handle(torch_dev)
            self.max_mhz = self.nv.clock(self._h, max_clock=True)
        except Exception as e:  # no NVML: report it instead of inventing clocks
            self.error = repr(e)
            self._h = None

    def _run(self):
        while not self._stop.is_set():
            c = self.nv.clock(self._h)
            if c is not None:
                self.samples.append((c, self.nv.reasons(self._h)))
            time.sleep(0.002)

    def __enter__(self):
        if self._h is not None:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *a):
        if self._h is not None:
            self._stop.set()
            self._t.join()

    def summary(self):
        if self._h is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "error": getattr(self, "error", "no NVML")}
        mhz = [s[0] for s in self.samples]
        mask = 0
        for _, r in self.samples:
            mask |= r
        reasons = [name for bit, name in REASONS.items() if mask & bit and name != "gpu_idle"]
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(mhz), "source": "NVML (nvidia-smi's library), 2 ms polling during the timed steps"}


# ---------------------------------------------------------------------------------------
# CPU oracle sample (the reference arm and the cpu_baseline key)
# ---------------------------------------------------------------------------------------
def host_threads():
    """Host threads this process may run on (the affinity mask where the OS has one)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_threads(jobs, threads):
    """Run the callables on `threads` host threads and wait for all.  The oracle's routines are
    C functions called through ctypes, which releases the interpreter lock for the call, so the
    threads compute in parallel."""
    if threads <= 1:
        return [j() for j in jobs]
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(threads) as ex:
        return list(ex.map(lambda j: j(), jobs))


def oracle_step(inp, What_ref, tokens: int, threads: int):
    """The oracle's time for one whole step on `threads` host threads.
    quantize + dequantize of the whole weight matrix, its rows split evenly over the threads
    (each thread quantizes its rows as a matrix of their own: the same work per weight), then
    the layer forward and backward on `tokens` distinct tokens per thread, scaled to the step's
    M tokens.  Returns (seconds per whole step, description, seconds spent)."""
    import oracle
    M, N, K = inp.shape
    T = max(1, threads)
    chunk = -(-N // T)
    parts = [(a, min(N, a + chunk)) for a in range(0, N, chunk)]

    def qd(a, b):
        qz = oracle.nf4_quantize(inp.W[a:b])
        oracle.nf4_dequantize(qz["packed"], qz["qcode"], qz["c2"], qz["mu"], b - a, K)

    def layer(i):
        sel = (np.arange(tokens, dtype=np.int64) + i * tokens) % M
        oracle.layer_fwd_rows(What_ref, inp.X, inp.A, inp.B, inp.alpha, sel)
        oracle.layer_dx_rows(What_ref, inp.A, inp.B, inp.G, inp.alpha, sel)
        oracle.layer_adapter_grads(inp.X[sel], inp.A, inp.B, inp.G[sel], inp.alpha)

    t0 = time.perf_counter()
    run_threads([lambda a=a, b=b: qd(a, b) for a, b in parts], T)
    t_q = time.perf_counter() - t0
    t0 = time.perf_counter()
    run_threads([lambda i=i: layer(i) for i in range(T)], T)
    t_l = time.perf_counter() - t0
    done = tokens * T
    step_s = t_q + t_l * (M / done)
    desc = (f"oracle (plain C) on {T} host thread{'s' if T > 1 else ''}: quantize+dequantize of the whole {N}x{K} "
            f"matrix (not sampled; rows split over the threads), layer fwd+bwd on {done} of {M} tokens "
            f"({tokens} per thread) scaled x{M / done:g}")
    return step_s, desc, t_q + t_l


def oracle_baseline(inp, What_ref, flops, tokens=2):
    """The cpu_baseline key: the oracle single-threaded and over every host thread."""
    T = host_threads()
    s1, d1, sp1 = oracle_step(inp, What_ref, tokens, 1)
    sT, dT, spT = (s1, d1, 0.0) if T == 1 else oracle_step(inp, What_ref, tokens, T)
    return {"value": flops / sT / 1e12, "unit": "TFLOP/s", "cores": T, "kind": "oracle",
            "sample": dT + f" ({spT:.1f} s wall)", "ms_per_step": sT * 1e3,
            "single_core": {"value": flops / s1 / 1e12, "cores": 1, "ms_per_step": s1 * 1e3,
                            "sample": d1 + f" ({sp1:.1f} s)"},
            "parallel_speedup": s1 / sT}


def sweep_oracle_check(samples, threads):
    """For the sweep's sampled layers: the oracle's nf4_quantize + nf4_dequantize of the whole v
    matrix (codes, scale codes, c2, mu and the bf16 dequant compared bit for bit with the GPU's)
    and of 64 rows of up (codes compared), the layers spread over the host threads; returns
    the check and the oracle's own GB/s on that work."""
    import oracle
    if not samples:
        return None

    def one(smp):
        N, K = smp["v_shape"]
        t0 = time.perf_counter()
        ref = oracle.nf4_quantize(smp["v_W"])
        deq = oracle.nf4_dequantize(ref["packed"], ref["qcode"], ref["c2"], ref["mu"], N, K)
        rq = oracle.nf4_quantize(smp["up_W_rows"])
        dt = time.perf_counter() - t0
        codes, sc, c2, mu = smp["v_gpu"]
        ok_v = (np.array_equal(codes.view(np.uint8), ref["packed"]) and np.array_equal(sc.view(np.int8), ref["qcode"])
                and np.array_equal(c2.view(np.uint32), ref["c2"].view(np.uint32))
                and int(mu.view(np.uint32)[0]) == int(np.float32(ref["mu"]).view(np.uint32))
                and np.array_equal(smp["v_deq"].view(np.uint16), deq))
        ok_up = np.array_equal(smp["up_codes_rows"].reshape(-1), rq["packed"])
        byt = 4 * N * K + 2 * oracle.nf4_storage_bytes(N, K) + 2 * N * K + smp["up_W_rows"].size * 4.5
        return smp["layer"], ok_v, ok_up, dt, byt

    t0 = time.perf_counter()
    res = run_threads([lambda s=s: one(s) for s in samples], min(threads, len(samples)))
    wall = time.perf_counter() - t0
    return {"layers": [r[0] for r in res], "v_whole_bit_exact": all(r[1] for r in res),
            "up_rows_codes_bit_exact": all(r[2] for r in res),
            "what": "v 1024x8192 whole (codes, scale codes, c2, mu, bf16 dequant) and 64 rows of up (codes)",
            "oracle_GB/s": sum(r[4] for r in res) / wall / 1e9, "oracle_threads": min(threads, len(samples))}


def make_inputs():
    from bit_nf4_quantized_36_b300 import synth
    c = synth.LLAMA8B_ATTN
    return synth.layer_inputs(c["id"], c["M"], c["N"], c["K"], c["r"], c["alpha"]), c


def run_reference(args):
    """The reference arm: the CPU oracle, as it stands, on this host's cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    inp, c = make_inputs()
    M, N, K, r = c["M"], c["N"], c["K"], c["r"]
    ref = oracle.nf4_quantize(inp.W)
    What_ref = oracle.nf4_dequantize(ref["packed"], ref["qcode"], ref["c2"], ref["mu"], N, K)
    # size the per-step sample so that warm-up + timed steps take about two minutes
    T = host_threads()
    t1 = oracle_step(inp, What_ref, 1, T)[2]
    tokens = int(max(1, min(16, 120.0 / (args.steps + args.warmup) / max(t1, 1e-3))))
    for _ in range(args.warmup):
        oracle_step(inp, What_ref, tokens, T)
    steps = []
    desc = ""
    for _ in range(args.steps):
        s, desc, _ = oracle_step(inp, What_ref, tokens, T)
        steps.append(s)
    step_s = statistics.mean(steps)
    value = layer_flops(M, N, K, r) / step_s / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K, "r": r, "alpha": c["alpha"]},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": T, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------------------
def fused_kernel_source_sha():
    """sha256 of the fused kernel's source: gemm.cu from its first device helper up to the skinny
    LoRA products (the decode helpers and nf4_lora_gemm_kernel), so that edits elsewhere in the file
    do not void a profile taken of this kernel."""
    src = open(os.path.join(ROOT, "bit_nf4_quantized_36_b300", "csrc", "gemm.cu")).read()
    a = src.find("__device__ __forceinline__ uint32_t prmt(")
    b = src.find("// Skinny LoRA products")
    if a < 0 or b < a:
        return None
    return hashlib.sha256(src[a:b].encode()).hexdigest()


def traffic_from_profile(gemm_src_sha, name="fused_gemm_llama8b_attn"):
    """DRAM bytes per fused-kernel launch from the machine-readable sidecar of a committed ncu
    summary (profiles/<name>.json), if that capture was taken on the current kernel source;
    otherwise None."""
    path = os.path.join(ROOT, "profiles", name + ".json")
    try:
        with open(path) as f:
            kv = json.load(f)
        if kv.get("kernel_source_sha256") != gemm_src_sha:
            return None
        return float(kv["dram_bytes_per_launch_avg"])
    except (OSError, ValueError, KeyError, TypeError):
        return None


def host_link_ms(torch, s_in, s_out, ins, outs, reps=10):
    """Time of one step's host copies alone: every (device, pinned host) input pair copied in on
    s_in while every (pinned host, device) result pair is copied out on s_out."""
    ins, outs = list(ins), list(outs)
    cur = torch.cuda.current_stream()

    def once():
        s_in.wait_stream(cur)
        s_out.wait_stream(cur)
        with torch.cuda.stream(s_in):
            for d, h in ins:
                d.copy_(h, non_blocking=True)
        with torch.cuda.stream(s_out):
            for h, d in outs:
                h.copy_(d, non_blocking=True)
        cur.wait_stream(s_in)
        cur.wait_stream(s_out)

    for _ in range(2):
        once()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        once()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def run_ours(args):
    import torch

    import bit_nf4_quantized_36_b300 as q
    from bit_nf4_quantized_36_b300 import _lib, synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    # under torchrun (LOCAL_RANK set) the process group is formed even for one rank, so that the
    # multi-GPU path (NCCL group, barriers, all-reduces, max over ranks) runs as it would at N > 1
    if world > 1 or "LOCAL_RANK" in os.environ:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    L = _lib.load()
    peaks = load_peaks()

    c = synth.LLAMA8B_ATTN
    M, N, K, r, alpha = c["M"], c["N"], c["K"], c["r"], c["alpha"]
    inp = synth.layer_inputs(c["id"], M, N, K, r, alpha, sub=rank)  # each rank its own batch
    to_bf = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    W_h = torch.from_numpy(inp.W).pin_memory()
    X_h, A_h, B_h, G_h = (to_bf(t).pin_memory() for t in (inp.X, inp.A, inp.B, inp.G))
    W, X, A, B, G = (t.to(dev) for t in (W_h, X_h, A_h, B_h, G_h))

    qw = q.empty_nf4(N, K, dev)
    What = torch.empty((N, K), dtype=torch.bfloat16, device=dev)
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    U = torch.empty((M, r), dtype=torch.bfloat16, device=dev)
    dX = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    dA = torch.empty((r, K), dtype=torch.float32, device=dev)
    dB = torch.empty((N, r), dtype=torch.float32, device=dev)
    ws_q = torch.empty(q.quantize_workspace_bytes(N, K), dtype=torch.uint8, device=dev)
    ws_f = torch.empty(q.fwd_workspace_bytes(M, N, K, r), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(q.bwd_workspace_bytes(M, N, K, r), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    # Nothing in the step reads W^: the dequantization runs on a stream of its own beside the
    # layer's forward, forked after the quantization and joined at the end of the step (a fork and
    # join that graph capture records as edges).
    s_dq = torch.cuda.Stream()
    ev_fork, ev_join = torch.cuda.Event(), torch.cuda.Event()

    def step_on(ins, outs):
        W_, X_, A_, B_, G_ = ins
        What_, Y_, dX_, dA_, dB_ = outs
        cur = torch.cuda.current_stream()
        q.nf4_quantize(W_, out=qw, workspace=ws_q)
        ev_fork.record(cur)
        s_dq.wait_event(ev_fork)
        with torch.cuda.stream(s_dq):
            q.nf4_dequantize(qw, out=What_)
        ev_join.record(s_dq)
        q.qlora_linear_fwd(qw, X_, A_, B_, alpha, Y=Y_, U_save=U, workspace=ws_f)
        q.qlora_linear_bwd(qw, X_, A_, B_, alpha, G_, U, dX=dX_, dA=dA_, dB=dB_, workspace=ws_b)
        cur.wait_event(ev_join)
        if dist is not None:
            dist.all_reduce(dA_)
            dist.all_reduce(dB_)

    def step():
        step_on((W, X, A, B, G), (What, Y, dX, dA, dB))

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    q.check_device_error()

    # ---- timed region: K steps, L2 flushed between steps (outside the step events) ------
    Ksteps = args.steps
    use_graph = dist is None and not args.no_graph
    # events recorded inside a captured graph must be external to time its replays
    ev = [(torch.cuda.Event(enable_timing=True, external=use_graph), torch.cuda.Event(enable_timing=True, external=use_graph))
          for _ in range(Ksteps)]
    kev = new_events(4 * Ksteps)  # 2 fused launches per step
    kev_arr = (ctypes.c_void_p * len(kev))(*[e.cuda_event for e in kev])
    sampler = ClockSampler(dev)
    barrier()
    n0 = q.launch_count()
    if L.qlora_set_kernel_timer(ctypes.cast(kev_arr, ctypes.c_void_p), 2 * Ksteps) != 0:
        raise RuntimeError("qlora_set_kernel_timer rejected the events")

    def timed_steps():
        for i in range(Ksteps):
            flush.zero_()
            ev[i][0].record()
            step()
            ev[i][1].record()

    # One process on one GPU: the K timed steps (flushes and events included) are captured once
    # into a CUDA graph and replayed, as a training loop would replay its step; every kernel of
    # every step still runs.  Under torchrun the all-reduces stay outside a graph.
    graph_note = None
    if use_graph:
        try:
            cap = torch.cuda.Stream()
            cap.wait_stream(torch.cuda.current_stream())
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.stream(cap):
                with torch.cuda.graph(graph, stream=cap):
                    timed_steps()
            torch.cuda.current_stream().wait_stream(cap)
            barrier()
        except Exception as e:  # keep a measurement: the same steps launched on the stream
            use_graph = False
            graph_note = f"graph capture failed ({type(e).__name__}); stream launches"
            torch.cuda.synchronize()
            n0 = q.launch_count()
            L.qlora_set_kernel_timer(None, 0)
            if L.qlora_set_kernel_timer(ctypes.cast(kev_arr, ctypes.c_void_p), 2 * Ksteps) != 0:
                raise RuntimeError("qlora_set_kernel_timer rejected the events")
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(Ksteps)]
    with sampler:
        if use_graph:
            graph.replay()
        else:
            timed_steps()
        barrier()
    launches = q.launch_count() - n0
    nk = L.qlora_kernel_timer_count()
    L.qlora_set_kernel_timer(None, 0)
    q.check_device_error()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms_per_step = sum(step_ms) / Ksteps
    kt = [kev[2 * i].elapsed_time(kev[2 * i + 1]) for i in range(nk)]
    t_fwd = statistics.mean(kt[0::2]) if nk >= 2 else float("nan")
    t_dx = statistics.mean(kt[1::2]) if nk >= 2 else float("nan")
    if dist is not None:
        t = torch.tensor([ms_per_step, t_fwd, t_dx], device=dev, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_per_step, t_fwd, t_dx = t.tolist()

    flops = layer_flops(M, N, K, r)
    value = world * flops / (ms_per_step * 1e-3) / 1e12
    fl_fwd = 2.0 * M * N * K + 2.0 * M * N * r
    fl_dx = 2.0 * M * N * K + 2.0 * M * K * r
    achieved = (fl_fwd + fl_dx) / ((t_fwd + t_dx) * 1e-3) / 1e12
    src_sha = fused_kernel_source_sha()
    roofline = {"kernel": "nf4_lora_gemm_kernel (fused NF4-dequant tcgen05 GEMM; forward and dX launches)",
                "bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"], "traffic": traffic_from_profile(src_sha),
                "peak_source": f"{peaks['source']} bf16 dense (burst: the kernel runs ~0.1 ms at a time)",
                "launch_ms": {"forward": t_fwd, "dx": t_dx},
                "algorithmic_flops_per_launch": {"forward": fl_fwd, "dx": fl_dx}}
    clocks = sampler.summary()

    # ---- end to end through the C ABI with host buffers ------------------------------------
    # Every step copies its inputs (W, X, A, B, dY) from pinned host memory and its results
    # (W^, Y, dX, dA, dB) back.  Pipelined, as a training loop fed from the host runs: the copies
    # have streams of their own and two device buffer sets, so step i + 1's inputs come in and
    # step i - 1's results go out while step i computes; the timed region runs from the first
    # input copy to the last result copy.  Serial (reported beside it): the copies and the step
    # one after another on one stream.
    e2e_steps = min(Ksteps, 20)
    hosts_in = (W_h, X_h, A_h, B_h, G_h)
    outs_h = [torch.empty_like(t, device="cpu").pin_memory() for t in (What, Y, dX, dA, dB)]
    h2d = sum(t.numel() * t.element_size() for t in hosts_in)
    d2h = sum(t.numel() * t.element_size() for t in outs_h)
    ins = [(W, X, A, B, G), tuple(torch.empty_like(t) for t in (W, X, A, B, G))]
    outs = [(What, Y, dX, dA, dB), tuple(torch.empty_like(t) for t in (What, Y, dX, dA, dB))]
    s_comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    in_ready, comp_done, out_done = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))

    def e2e_pipelined(n, t0=None, t1=None):
        s_in.wait_stream(s_comp)
        if t0 is not None:
            t0.record(s_in)
        for i in range(n):
            sl = i % 2
            if i >= 2:
                s_in.wait_event(comp_done[sl])   # step i - 2 has read this input set
            with torch.cuda.stream(s_in):
                for d, h in zip(ins[sl], hosts_in):
                    d.copy_(h, non_blocking=True)
                in_ready[sl].record(s_in)
            s_comp.wait_event(in_ready[sl])
            if i >= 2:
                s_comp.wait_event(out_done[sl])  # step i - 2's results have left this output set
            step_on(ins[sl], outs[sl])
            comp_done[sl].record(s_comp)
            s_out.wait_event(comp_done[sl])
            with torch.cuda.stream(s_out):
                for h, d in zip(outs_h, outs[sl]):
                    h.copy_(d, non_blocking=True)
                out_done[sl].record(s_out)
        if t1 is not None:
            t1.record(s_out)
        s_comp.wait_stream(s_out)

    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(e2e_steps)]
    barrier()
    for i in range(e2e_steps):
        e2e_ev[i][0].record()
        for d, h in zip((W, X, A, B, G), hosts_in):
            d.copy_(h, non_blocking=True)
        step()
        for h, d in zip(outs_h, (What, Y, dX, dA, dB)):
            h.copy_(d, non_blocking=True)
        e2e_ev[i][1].record()
    barrier()
    serial_ms = sum(a.elapsed_time(b) for a, b in e2e_ev) / e2e_steps
    pipe_note = "pipelined: own copy streams, two device buffer sets; timed from the first input copy to the last result copy"
    try:
        e2e_pipelined(4)  # warm-up: the second buffer set and the copy streams
        barrier()
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e2e_pipelined(e2e_steps, p0, p1)
        barrier()
        e2e_ms = p0.elapsed_time(p1) / e2e_steps
    except Exception as e:  # keep the serial measurement as the end-to-end number
        if dist is not None:
            raise  # a rank that fell back alone would leave the others waiting at a barrier
        torch.cuda.synchronize()
        e2e_ms = serial_ms
        pipe_note = f"serial (the pipelined form failed: {type(e).__name__})"
    if dist is not None:
        t = torch.tensor([e2e_ms, serial_ms], device=dev, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_ms, serial_ms = t.tolist()
    e2e = {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "copies": pipe_note,
           "serial": {"value": world * flops / (serial_ms * 1e-3) / 1e12, "ms_per_step": serial_ms,
                      "copies": "inputs, step and results one after another on one stream"}}
    try:  # the bound of the end-to-end step: the same copies alone, both directions at once
        link_ms = host_link_ms(torch, s_in, s_out, zip(ins[1], hosts_in), zip(outs_h, outs[1]))
        e2e["link"] = {"ms_per_step": link_ms, "frac": link_ms / e2e_ms,
                       "what": "the step's input and result copies alone, in and out at once (no GPU work)"}
    except Exception as e:
        e2e["link"] = {"error": repr(e)}
    q.check_device_error()

    extras = {}
    sweep_samples = []
    if rank == 0 and not args.no_extras:
        try:
            extras = hbm_extras(q, _lib, L, dev, peaks, flush)
        except Exception as e:  # the headline line must still print
            extras = {"error": repr(e)}

    if rank == 0 and not args.no_extras:
        try:
            extras["concat_qkv"] = concat_extras(q, dev, flush)
        except Exception as e:
            extras["concat_qkv"] = {"error": repr(e)}
        try:
            extras["dropout_attn"] = dropout_extras(q, dev, flush, inp)
        except Exception as e:
            extras["dropout_attn"] = {"error": repr(e)}
        try:
            extras["paged_adamw"] = optim_extras(q, dev, peaks, flush)
        except Exception as e:
            extras["paged_adamw"] = {"error": repr(e)}
        try:
            extras["llama8b_mlp"] = mlp_extras(q, L, dev, peaks, flush)
        except Exception as e:
            extras["llama8b_mlp"] = {"error": repr(e)}
        try:
            extras["llama70b_sweep"], sweep_samples = sweep_extras(q, dev, peaks, flush)
        except Exception as e:
            extras["llama70b_sweep"] = {"error": repr(e)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        ref = oracle.nf4_quantize(inp.W)
        What_ref = oracle.nf4_dequantize(ref["packed"], ref["qcode"], ref["c2"], ref["mu"], N, K)
        cpu = oracle_baseline(inp, What_ref, flops, tokens=32)
        if sweep_samples:
            try:
                extras["llama70b_sweep"]["oracle_check"] = sweep_oracle_check(sweep_samples, host_threads())
            except Exception as e:
                extras["llama70b_sweep"]["oracle_check"] = {"error": repr(e)}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": Ksteps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": WORKLOAD, "M_per_gpu": M, "N": N, "K": K, "r": r, "alpha": alpha,
                           "step": ("nf4_quantize + nf4_dequantize + qlora_linear_fwd + qlora_linear_bwd "
                                    "(the dequantization on a forked stream beside the forward)"),
                           "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MiB write, outside the step events)",
                           "launch": ("the K timed steps captured in one CUDA graph, replayed once" if use_graph
                                      else graph_note or "stream launches"),
                           "parallelism": f"dp{world}"},
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
                "gpu_launches_per_step": launches / Ksteps, "clocks": clocks,
                "step_ms_min_max": [min(step_ms), max(step_ms)], "hbm_kernels": extras}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def replay_timed(torch, fn, flush, reps=10, L=None, kernel_events=None):
    """Device time of fn() with host enqueue kept out of the timing.  fn runs three times untimed
    (allocations, first-call set-up, clocks); then `reps` repetitions, each an L2 flush followed by
    fn() between two events, are captured into one CUDA graph and replayed twice, the events
    keeping the second replay's times: every kernel of every repetition runs, and the events see
    only device time.  With `kernel_events` (2 events
    per timed launch) the library's kernel timer is armed during the capture, so that its event
    pairs around each timed kernel become graph nodes too.  Returns (median call ms, the timed
    kernels' durations in launch order or None, how).  If the capture fails the repetitions run
    as stream launches and `how` says so."""
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True, external=True), torch.cuda.Event(enable_timing=True, external=True))
          for _ in range(reps)]

    def arm():
        if kernel_events is not None:
            arr = (ctypes.c_void_p * len(kernel_events))(*[e.cuda_event for e in kernel_events])
            if L.qlora_set_kernel_timer(ctypes.cast(arr, ctypes.c_void_p), len(kernel_events) // 2) != 0:
                raise RuntimeError("qlora_set_kernel_timer rejected the events")

    def body():
        for a, b in ev:
            flush.zero_()
            a.record()
            fn()
            b.record()

    how = "CUDA graph of the repetitions (L2 flush + call each), replayed once"
    arm()
    try:
        cap = torch.cuda.Stream()
        cap.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(graph, stream=cap):
                body()
        torch.cuda.current_stream().wait_stream(cap)
        torch.cuda.synchronize()
        # a first replay (graph upload, clocks up); the events, graph nodes like the kernel
        # timer's, keep the second replay's times
        graph.replay()
        torch.cuda.synchronize()
        graph.replay()
    except Exception as e:
        torch.cuda.synchronize()
        if kernel_events is not None:
            L.qlora_set_kernel_timer(None, 0)
            arm()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        how = f"stream launches (graph capture failed: {type(e).__name__}); host enqueue inside the events"
        body()
    torch.cuda.synchronize()
    tk = None
    if kernel_events is not None:
        nk = min(L.qlora_kernel_timer_count(), len(kernel_events) // 2)
        L.qlora_set_kernel_timer(None, 0)
        tk = [kernel_events[2 * i].elapsed_time(kernel_events[2 * i + 1]) for i in range(nk)] or None
    return statistics.median(a.elapsed_time(b) for a, b in ev), tk, how


def dropout_extras(q, dev, flush, inp, reps=10):
    """The bench layer (Llama-3-8B attention projection, M = 4096) fwd + bwd with LoRA dropout
    p = 0.05 on the adapter input, against the same call without dropout."""
    import torch
    W = torch.from_numpy(inp.W).to(dev)
    qw = q.nf4_quantize(W)
    X, A, B, G = (torch.from_numpy(np.ascontiguousarray(t).view(np.int16)).to(dev).view(torch.bfloat16)
                  for t in (inp.X, inp.A, inp.B, inp.G))

    def plain():
        _, U = q.qlora_linear_fwd(qw, X, A, B, inp.alpha)
        q.qlora_linear_bwd(qw, X, A, B, inp.alpha, G, U)

    def drop():
        _, U = q.qlora_linear_fwd_dropout(qw, X, A, B, inp.alpha, 0.05, 1234)
        q.qlora_linear_bwd_dropout(qw, X, A, B, inp.alpha, 0.05, 1234, G, U)

    t0, _, how = replay_timed(torch, plain, flush, reps)
    t1, _, _ = replay_timed(torch, drop, flush, reps)
    return {"p": 0.05, "plain_fwd_bwd_ms": t0, "dropout_fwd_bwd_ms": t1, "overhead": t1 / t0 - 1.0, "timing": how}


def optim_extras(q, dev, peaks, flush, reps=10):
    """The adapters' AdamW step with paged optimizer states, over every adapter of Llama-3-8B
    (rank 16 on all seven linear layers of 32 blocks: 41.9 M weights) in one launch: the step
    with the pages resident (reads p, g, m, v and writes p, m, v and the bf16 copy: 30 bytes per
    weight), paging the two fp32 moment buffers out to host memory and back in, and a step that
    finds its moments on the host and faults them in."""
    import torch
    from bit_nf4_quantized_36_b300 import synth
    n = synth.adapter_param_count()
    p, g, m0, v0 = synth.adamw_inputs_gpu(synth.LLAMA8B_ADAPTERS["id"], n, dev)
    opt = q.PagedAdamW(n)
    opt.m.tensor(torch.float32, n).copy_(m0)
    opt.v.tensor(torch.float32, n).copy_(v0)
    del m0, v0
    pb = torch.empty(n, dtype=torch.bfloat16, device=dev)
    opt.page_in()
    opt.step(p, g, pb)
    torch.cuda.synchronize()

    def ev(fn):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    t_res, _, how = replay_timed(torch, lambda: opt.step(p, g, pb), flush, reps)
    t_out, t_in, t_fault = [], [], []
    for _ in range(3):
        t_out.append(ev(opt.page_out))
        t_fault.append(ev(lambda: opt.step(p, g, pb)))     # moments on the host: migrated on demand
        opt.page_out()
        torch.cuda.synchronize()
        t_in.append(ev(opt.page_in))
    q.check_device_error()
    byt = 30 * n
    state = 8 * n
    return {"workload": synth.LLAMA8B_ADAPTERS["name"], "n": n, "kernel": "adamw_kernel",
            "step_ms_resident": t_res, "GB/s": byt / t_res / 1e6, "frac_hbm": byt / t_res / 1e6 / peaks["hbm_gbs"],
            "algorithmic_bytes": byt, "moment_bytes": state,
            "page_out_ms": statistics.median(t_out), "page_in_ms": statistics.median(t_in),
            "page_in_GB/s": state / statistics.median(t_in) / 1e6,
            "step_ms_faulting": statistics.median(t_fault), "timing": how,
            "timing_paging": "one event pair around each page-out, page-in and faulting step (stream launches)"}


def concat_extras(q, dev, flush, reps=10):
    """Llama-3-8B attention q/k/v (4096, 1024 and 1024 rows, K = 4096, 4096 tokens, r = 16 each):
    fwd + bwd of the three modules as three separate layer calls against one concatenated call
    (qlora_linear_fwd_cat / _bwd_cat)."""
    import torch
    from bit_nf4_quantized_36_b300 import synth
    M, K, r, alpha = 4096, 4096, 16, 32.0
    specs = [("q", 4096), ("k", 1024), ("v", 1024)]
    X = torch.randn((M, K), device=dev).to(torch.bfloat16)
    mods = []
    for i, (_, N) in enumerate(specs):
        W = synth.sweep_weight_gpu(0, i, N, K)
        A = (torch.randn((r, K), device=dev) / K ** 0.5).to(torch.bfloat16)
        B = (torch.randn((N, r), device=dev) * 0.01).to(torch.bfloat16)
        mods.append((q.nf4_quantize(W), A, B, alpha))
    Ncat = sum(N for _, N in specs)
    dY = torch.randn((M, Ncat), device=dev).to(torch.bfloat16)
    dYs = [dY[:, o:o + N].contiguous() for o, N in zip((0, 4096, 5120), (4096, 1024, 1024))]

    def separate():
        for (qw, A, B, a), g in zip(mods, dYs):
            _, U = q.qlora_linear_fwd(qw, X, A, B, a)
            q.qlora_linear_bwd(qw, X, A, B, a, g, U)

    def concatenated():
        _, U = q.qlora_linear_fwd_cat(mods, X)
        q.qlora_linear_bwd_cat(mods, X, dY, U)

    t_sep, _, how = replay_timed(torch, separate, flush, reps)
    t_cat, _, _ = replay_timed(torch, concatenated, flush, reps)
    fl = sum(4.0 * M * N * K + 6.0 * M * r * (N + K) for _, N in specs)
    return {"modules": "q 4096x4096, k 1024x4096, v 1024x4096; M=4096, r=16", "separate_ms": t_sep,
            "concatenated_ms": t_cat, "TFLOP/s_separate": fl / t_sep / 1e9, "TFLOP/s_concatenated": fl / t_cat / 1e9,
            "speedup": t_sep / t_cat, "timing": how}


def mlp_extras(q, L, dev, peaks, flush, reps=5):
    """Llama-3-8B MLP with adapters on all three linears (gate and up 4096 -> 14336, down
    14336 -> 4096; NF4 weights N(0, 0.02) with 0.1% +-U(0.2, 1.0) outliers), M = 8192 tokens,
    r = 64, alpha = 128: forward and backward (dX, dA, dB) of the three layers per step, graph
    replayed with an L2 flush before each step.  The fused GEMM's launches (a forward and a dX per
    layer) are timed by the library's kernel timer for the roofline."""
    import torch
    from bit_nf4_quantized_36_b300 import synth
    c = synth.LLAMA8B_MLP
    M, r, alpha = c["M"], c["r"], c["alpha"]
    g = torch.Generator(device=dev)
    g.manual_seed(synth.SEED_BASE + c["id"] * 0x1000 + 0x900)
    X = torch.randn((M, 4096), generator=g, device=dev).to(torch.bfloat16)     # MLP input (gate, up)
    H = torch.randn((M, 14336), generator=g, device=dev).to(torch.bfloat16)    # down's input
    mods = []
    for mi, (name, N, K) in enumerate(c["mats"]):
        W = synth.normal_weight_gpu(c["id"], mi, N, K, 0.02, outliers=True)
        qw = q.nf4_quantize(W)
        del W
        A = (torch.randn((r, K), generator=g, device=dev) / K ** 0.5).to(torch.bfloat16)
        B = (torch.randn((N, r), generator=g, device=dev) * 0.01).to(torch.bfloat16)
        G = torch.randn((M, N), generator=g, device=dev).to(torch.bfloat16)
        Xin = X if K == 4096 else H
        bufs = dict(Y=torch.empty((M, N), dtype=torch.bfloat16, device=dev),
                    U=torch.empty((M, r), dtype=torch.bfloat16, device=dev),
                    dX=torch.empty((M, K), dtype=torch.bfloat16, device=dev),
                    dA=torch.empty((r, K), dtype=torch.float32, device=dev),
                    dB=torch.empty((N, r), dtype=torch.float32, device=dev),
                    wf=torch.empty(q.fwd_workspace_bytes(M, N, K, r), dtype=torch.uint8, device=dev),
                    wb=torch.empty(q.bwd_workspace_bytes(M, N, K, r), dtype=torch.uint8, device=dev))
        mods.append((name, N, K, qw, Xin, A, B, G, bufs))
    torch.cuda.synchronize()

    def step():
        for name, N, K, qw, Xin, A, B, G, b in mods:
            q.qlora_linear_fwd(qw, Xin, A, B, alpha, Y=b["Y"], U_save=b["U"], workspace=b["wf"])
            q.qlora_linear_bwd(qw, Xin, A, B, alpha, G, b["U"], dX=b["dX"], dA=b["dA"], dB=b["dB"], workspace=b["wb"])

    kev = new_events(2 * 6 * reps)
    t, tks, how = replay_timed(torch, step, flush, reps, L=L, kernel_events=kev)
    q.check_device_error()
    flops = sum(layer_flops(M, N, K, r) for _, N, K in c["mats"])
    fused_fl = [fl for _, N, K in c["mats"] for fl in (2.0 * M * N * K + 2.0 * M * N * r, 2.0 * M * N * K + 2.0 * M * K * r)]
    res = {"workload": c["name"], "step": "qlora_linear_fwd + qlora_linear_bwd of gate, up and down",
           "ms_per_step": t, "TFLOP/s": flops / t / 1e9, "flops_per_step": flops, "timing": how}
    if tks and len(tks) >= 6:
        nrep = len(tks) // 6
        per = [statistics.median(tks[6 * i + j] for i in range(nrep)) for j in range(6)]
        ach = sum(fused_fl) / (sum(per) * 1e-3) / 1e12
        res["roofline"] = {"kernel": "nf4_lora_gemm_kernel (forward and dX launches of the three layers)",
                           "bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                           "frac": ach / peaks["bf16_tflops"], "traffic": None,
                           "peak_source": f"{peaks['source']} bf16 dense (burst)",
                           "launch_ms": dict(zip([f"{n}_{k}" for n, _, _ in c["mats"] for k in ("fwd", "dx")], per)),
                           "algorithmic_flops_per_launch": fused_fl,
                           "share_of_step": sum(per) / t}
    del mods
    torch.cuda.empty_cache()
    return res


def sweep_extras(q, dev, peaks, flush, layers=80, check_layers=(0, 40, 79)):
    """The whole-model sweep: 80 Llama-70B-shaped blocks (q, o 8192 x 8192; k, v 1024 x 8192;
    gate, up 28672 x 8192; down 8192 x 28672), fp32 weights N(0, 0.02) with 0.1% Student-t(3)
    entries generated per layer on the GPU (untimed), then nf4_quantize and nf4_dequantize to bf16
    of each matrix.  Each layer's 7 quantize + dequantize pairs are captured in a graph (an L2
    flush before each pair, an event pair around it) and replayed once.  For the layers in
    `check_layers` the v matrix (whole) and 64 rows of up are copied to the host with the
    GPU's results, for the check against the oracle in the CPU-baseline leg."""
    import torch
    from bit_nf4_quantized_36_b300 import synth
    c = synth.LLAMA70B_SWEEP
    shapes = sorted({(N, K) for _, N, K in c["mats"]})
    outs = {s: (q.empty_nf4(s[0], s[1], dev), torch.empty(s, dtype=torch.bfloat16, device=dev)) for s in shapes}
    ws = torch.empty(max(q.quantize_workspace_bytes(N, K) for N, K in shapes), dtype=torch.uint8, device=dev)
    per_layer_ms, byt_layer, samples = [], 0, []
    how = "per layer: a CUDA graph of the 7 (L2 flush, quantize + dequantize) pairs, replayed once"
    for layer in range(layers):
        Ws = [synth.sweep_weight_gpu(layer, mi, N, K, device=dev, std=c["w_std"]) for mi, (_, N, K) in enumerate(c["mats"])]
        ev = [(torch.cuda.Event(enable_timing=True, external=True), torch.cuda.Event(enable_timing=True, external=True))
              for _ in Ws]

        def body():
            for (a, b), W, (_, N, K) in zip(ev, Ws, c["mats"]):
                qw, What = outs[(N, K)]
                flush.zero_()
                a.record()
                q.nf4_quantize(W, out=qw, workspace=ws)
                q.nf4_dequantize(qw, out=What)
                b.record()

        torch.cuda.synchronize()
        try:
            cap = torch.cuda.Stream()
            cap.wait_stream(torch.cuda.current_stream())
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.stream(cap):
                with torch.cuda.graph(graph, stream=cap):
                    body()
            torch.cuda.current_stream().wait_stream(cap)
            graph.replay()
        except Exception as e:
            torch.cuda.synchronize()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in Ws]
            how = f"stream launches (graph capture failed: {type(e).__name__})"
            body()
        torch.cuda.synchronize()
        per_layer_ms.append(sum(a.elapsed_time(b) for a, b in ev))
        if layer == 0:
            byt_layer = sum(4 * N * K + 2 * q.nf4_storage_bytes(N, K) + 2 * N * K for _, N, K in c["mats"])
        # the v and up matrices' results are still in their shapes' output buffers (each is the
        # last matrix of its shape in the layer's order)
        if layer in check_layers:
            vq, vW = outs[(c["mats"][2][1], c["mats"][2][2])]
            uq, _ = outs[(c["mats"][5][1], c["mats"][5][2])]
            uN, uK = c["mats"][5][1], c["mats"][5][2]
            rows = torch.arange(0, uN, uN // 64, device=dev)[:64]
            samples.append({"layer": layer, "v_W": Ws[2].cpu().numpy(), "v_shape": (c["mats"][2][1], c["mats"][2][2]),
                            "v_gpu": [t.cpu().numpy() for t in (vq.codes, vq.scale_codes, vq.scale_scales, vq.scale_offset)],
                            "v_deq": vW.view(torch.int16).cpu().numpy(),
                            "up_rows": rows.cpu().numpy(), "up_W_rows": Ws[5][rows].cpu().numpy(),
                            "up_codes_rows": uq.codes.view(uN, uK // 2)[rows].cpu().numpy()})
        del Ws
    total_ms = sum(per_layer_ms)
    res = {"workload": c["name"], "layers": layers, "matrices_per_layer": len(c["mats"]),
           "weights_per_layer": sum(N * K for _, N, K in c["mats"]), "ms_total": total_ms,
           "ms_per_layer_median": statistics.median(per_layer_ms), "algorithmic_bytes_per_layer": byt_layer,
           "GB/s": layers * byt_layer / total_ms / 1e6, "frac_hbm": layers * byt_layer / total_ms / 1e6 / peaks["hbm_gbs"],
           "bytes": "quantize reads fp32 and writes the NF4 storage; dequantize reads the storage and writes bf16",
           "timing": how, "codes_checked": "in the CPU-baseline leg, layers " + ", ".join(map(str, check_layers))}
    del outs
    torch.cuda.empty_cache()
    return res, samples


def hbm_extras(q, _lib, L, dev, peaks, flush, reps=10):
    """Secondary numbers for the HBM-bound kernels on a Llama-70B MLP matrix (28672 x 8192):
    nf4_dequantize, nf4_quantize and adapter-merge GB/s, and the small-M forward (decode) GB/s on
    both 70B MLP matrices.  Every figure is device time of a graph-replayed call (replay_timed)."""
    import torch
    from bit_nf4_quantized_36_b300 import synth
    rows, cols = 28672, 8192
    n = rows * cols
    storage = q.nf4_storage_bytes(rows, cols)
    W = synth.sweep_weight_gpu(0, 4, rows, cols)
    qw = q.nf4_quantize(W)
    What = q.nf4_dequantize(qw)
    ws = torch.empty(q.quantize_workspace_bytes(rows, cols), dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()

    def gbs(name, t, byt, how, **kw):
        return {"matrix": f"{rows}x{cols}", "ms": t, "GB/s": byt / t / 1e6,
                "frac_hbm": byt / t / 1e6 / peaks["hbm_gbs"], "algorithmic_bytes": byt, "timing": how, **kw}

    out = {}
    t, _, how = replay_timed(torch, lambda: q.nf4_dequantize(qw, out=What), flush, reps)
    out["dequantize"] = gbs("dequantize", t, storage + 2 * n, how)
    t, _, how = replay_timed(torch, lambda: q.nf4_quantize(W, out=qw, workspace=ws), flush, reps)
    out["quantize"] = gbs("quantize", t, 4 * n + storage, how)
    # adapter merge W_m = bf16(W^ + (alpha/r) B A): codes and scales read, bf16 written
    for r_m in (16, 64):
        Am = (torch.randn((r_m, cols), device=dev) / cols ** 0.5).to(torch.bfloat16)
        Bm = (torch.randn((rows, r_m), device=dev) * 0.01).to(torch.bfloat16)
        t, _, how = replay_timed(torch, lambda: q.qlora_merge(qw, Am, Bm, 2.0 * r_m, out=What), flush, reps)
        out[f"merge_r{r_m}"] = gbs("merge", t, storage + 2 * n + 2 * r_m * (rows + cols), how)
    del W, What, qw, ws
    torch.cuda.empty_cache()
    # decode-like forward: M tokens through each 70B MLP matrix, r = 16, W ~ N(0, 0.015)
    c = synth.LLAMA70B_DECODE
    r, alpha = c["r"], c["alpha"]
    for mi, (name, N, K) in enumerate(c["mats"]):
        Wd = synth.normal_weight_gpu(c["id"], mi, N, K, c["w_std"])
        qd = q.nf4_quantize(Wd)
        del Wd
        A = (torch.randn((r, K), device=dev) / K ** 0.5).to(torch.bfloat16)
        B = (torch.randn((N, r), device=dev) * 0.01).to(torch.bfloat16)
        st = q.nf4_storage_bytes(N, K)
        dec = {}
        for M in c["Ms"]:
            X = torch.randn((M, K), device=dev).to(torch.bfloat16)
            Y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            U = torch.empty((M, r), dtype=torch.bfloat16, device=dev)
            wsf = torch.empty(q.fwd_workspace_bytes(M, N, K, r), dtype=torch.uint8, device=dev)
            kev = new_events(2 * reps)
            t, tks, how = replay_timed(torch, lambda: q.qlora_linear_fwd(qd, X, A, B, alpha, Y=Y, U_save=U,
                                                                         workspace=wsf),
                                       flush, reps, L=L, kernel_events=kev)
            tk = statistics.median(tks) if tks else None
            byt = st + 2 * r * (N + K) + 2 * M * (N + K)
            dec[f"M={M}"] = {"call_ms": t, "kernel": "nf4_gemv_kernel" if M <= 8 else "nf4_lora_gemm_small_kernel",
                             "kernel_ms": tk, "GB/s_kernel": byt / tk / 1e6 if tk else None,
                             "frac_hbm_kernel": byt / tk / 1e6 / peaks["hbm_gbs"] if tk else None,
                             "GB/s_call": byt / t / 1e6, "frac_hbm_call": byt / t / 1e6 / peaks["hbm_gbs"],
                             "algorithmic_bytes": byt, "timing": how}
        out[f"decode_forward_{name}_{N}x{K}_r{r}"] = dec
        del qd
    out["hbm_peak_GB/s"] = f"{peaks['hbm_gbs']} ({peaks['source']})"
    return out


def run_ncu_target(args):
    """A short, untimed run for profiler captures: three forward+backward passes of the layer on the
    bench workload (--ncu-target fused), three small-M forwards on a 70B MLP matrix
    (--ncu-target decode: the up projection 28672 x 8192; decode_down: the down projection
    8192 x 28672), three AdamW steps over the Llama-3-8B adapter set with the moments
    in plain device memory (--ncu-target adamw; the same kernel as with paged moments), or three
    quantizations, dequantizations or rank-16 adapter merges of a 28672 x 8192 matrix
    (--ncu-target quantize, dequantize, merge)."""
    import torch

    import bit_nf4_quantized_36_b300 as q
    from bit_nf4_quantized_36_b300 import synth
    dev = torch.device("cuda")
    if args.ncu_target in ("quantize", "dequantize", "merge"):
        W = synth.sweep_weight_gpu(0, 4, 28672, 8192)
        qw = q.nf4_quantize(W)
        What = q.nf4_dequantize(qw)
        Am = (torch.randn((16, 8192), device=dev) / 8192 ** 0.5).to(torch.bfloat16)
        Bm = (torch.randn((28672, 16), device=dev) * 0.01).to(torch.bfloat16)
        for _ in range(3):
            if args.ncu_target == "quantize":
                q.nf4_quantize(W, out=qw)
            elif args.ncu_target == "merge":
                q.qlora_merge(qw, Am, Bm, 32.0, out=What)
            else:
                q.nf4_dequantize(qw, out=What)
        torch.cuda.synchronize()
        q.check_device_error()
        print(json.dumps({"ncu_target": args.ncu_target, "rows": 28672, "cols": 8192, "ok": True}))
        return 0
    if args.ncu_target == "adamw":
        n = synth.adapter_param_count()
        p, g, m, v = synth.adamw_inputs_gpu(synth.LLAMA8B_ADAPTERS["id"], n, dev)
        pb = torch.empty(n, dtype=torch.bfloat16, device=dev)
        for t in range(1, 4):
            q.adamw_step(p, g, m, v, t, 2e-4, p_bf16=pb)
        torch.cuda.synchronize()
        q.check_device_error()
        print(json.dumps({"ncu_target": "adamw", "n": n, "ok": True}))
        return 0
    if args.ncu_target == "fused":
        c = synth.LLAMA8B_ATTN
        M, N, K, r, alpha = c["M"], c["N"], c["K"], c["r"], c["alpha"]
    elif args.ncu_target == "decode_down":
        M, N, K, r, alpha = args.decode_m, 8192, 28672, 16, 32.0
    else:
        M, N, K, r, alpha = args.decode_m, 28672, 8192, 16, 32.0
    g = torch.Generator(device=dev)
    g.manual_seed(synth.SEED_BASE + 7)
    W = torch.randn((N, K), generator=g, device=dev) * 0.02
    X = torch.randn((M, K), generator=g, device=dev).to(torch.bfloat16)
    A = (torch.randn((r, K), generator=g, device=dev) / K ** 0.5).to(torch.bfloat16)
    B = (torch.randn((N, r), generator=g, device=dev) * 0.01).to(torch.bfloat16)
    G = torch.randn((M, N), generator=g, device=dev).to(torch.bfloat16)
    qw = q.nf4_quantize(W)
    for _ in range(3):
        Y, U = q.qlora_linear_fwd(qw, X, A, B, alpha)
        if args.ncu_target == "fused":
            q.qlora_linear_bwd(qw, X, A, B, alpha, G, U)
    torch.cuda.synchronize()
    q.check_device_error()
    print(json.dumps({"ncu_target": args.ncu_target, "M": M, "N": N, "K": K, "r": r, "ok": True}))
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch the timed steps on the stream, not as a graph")
    ap.add_argument("--ncu-target", choices=["fused", "decode", "decode_down", "adamw", "quantize", "dequantize",
                                             "merge"],
                    default=None,
                    help="untimed short run of one kernel family, for profiler captures")
    ap.add_argument("--decode-m", type=int, default=1)
    args = ap.parse_args()
    if args.ncu_target:
        return run_ncu_target(args)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
