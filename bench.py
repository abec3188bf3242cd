#!/usr/bin/env python3
"""Benchmark of the lightning-attention hot path on GB300.

One "step" is one call of the prefill entry point over the MiniMax-01-shaped
layer: 1 sequence x 8192 tokens x 64 heads x d = 128, bf16 inputs, fp32
accumulation, bf16 output plus the fp32 final state [64, 128, 128].  The
JSON line's ``value`` is prefill tokens/s with inputs already resident in
HBM; ``decode`` holds the batched decode step (128 sequences x 64 heads,
fp32 state, 1000 consecutive steps); ``e2e`` repeats the prefill through the
same public call with the inputs in pinned host memory and the host<->device
copies inside the timed region; ``roofline`` relates the prefill kernel's
time to the HBM roofline (its bound) and ``tensor`` to the bf16 tensor peak;
``cpu_baseline`` is the fp64 CPU oracle timed on the host cores.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs an independent replica on its own GPU (the
path has no exchange step); rank 0 prints the line with the max time over
ranks and the tokens of all ranks.
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

METRIC = ("prefill tokens/s + % bf16 tensor peak; decode tokens/s + % HBM BW (1×GB300)")
# the files a kernel's code comes from (its traffic record is void once any changes)
_CSRC = os.path.join(ROOT, "lightning_attention_attn_gb300", "csrc")
PREFILL_KERNEL_SRC = [os.path.join(_CSRC, f) for f in ("prefill_tc.cu", "sm100_ptx.cuh")]
DECODE_KERNEL_SRC = [os.path.join(_CSRC, "decode.cu")]
CW_KERNEL_SRC = [os.path.join(_CSRC, f) for f in ("prefill_cw_tc.cu", "sm100_ptx.cuh")]


# ---------------------------------------------------------------- helpers
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return dict(hbm=float(j["hbm_gbs"]), bf16=float(j["bf16_tflops"]),
                    bf16_sustained=float(j.get("bf16_tflops_sustained", j["bf16_tflops"])),
                    source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


def fp32_alu_peak_tflops(sms):
    """FFMA peak of the CUDA cores: 128 fp32 lanes per SM, 2 flops per FMA,
    at the maximum SM clock of 2070 MHz."""
    return sms * 128 * 2 * 2.070e9 / 1e12


def cuda_core_roofline(flops, byts, ms, pk, sms):
    """The CUDA-core (FFMA) prefill is bound by fp32 arithmetic, not HBM."""
    peak = fp32_alu_peak_tflops(sms)
    tf = flops / (ms / 1e3) / 1e12
    return {"bound": "alu", "alg_flops": flops, "achieved": round(tf, 2),
            "peak": round(peak, 2), "unit": "TFLOP/s", "frac": round(tf / peak, 4),
            "peak_source": "derived: SMs x 128 fp32 lanes x 2 x 2070 MHz",
            "hbm_frac": round(byts / (ms / 1e3) / 1e9 / pk["hbm"], 4)}


def src_hash(paths):
    h = hashlib.sha256()
    for path in paths:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key, src):
    """DRAM bytes per launch from the committed ncu summary, only while the
    kernel source is the one that was profiled."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        j = json.load(f)
    e = j.get(kernel_key)
    if not e or e.get("source_sha256_16") != src_hash(src):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons in the background."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
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
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws):
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, ws):
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------- workload figures
def prefill_alg(T, H, d, B, nseq):
    """Algorithmic bytes and flops of one prefill launch.
    bytes: q, k, v read + o written (bf16) = 8 d per token-head, plus the fp32
    final state H d^2 4 per sequence.  flops: 4 d^2 (Q KV and K^T V) plus
    2 (B + 1) d (causal half of Q K^T and P V) per token-head."""
    byts = T * H * 8 * d + nseq * H * d * d * 4
    flops = T * H * (4 * d * d + 2 * (B + 1) * d)
    return byts, flops


def decode_alg(Bn, H, d):
    """State read + write (fp32) plus q, k, v read and o written (bf16)."""
    return Bn * H * (2 * d * d * 4 + 4 * d * 2)


# ------------------------------------------------------------- our arm
def cpu_baseline(inp, min_seconds=10.0):
    """The fp64 oracle (recurrent form) on the same 8K-token workload, all
    heads, repeated until at least min_seconds of CPU work."""
    import oracle
    threads = oracle.max_threads()
    T = inp.total_tokens
    t0 = time.perf_counter()
    n = 0
    while True:
        oracle.recurrent(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens.cpu())
        n += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds or n >= 20:
            break
    return {"value": n * T / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"full prefill_8k workload (1 x 8192 tokens x 64 heads x d=128, "
                      f"bf16 inputs upcast to fp64), recurrent form, {n} run(s), {dt:.1f} s"}


def run_ours(args, ws, rank, local):
    import torch
    import lightning_attention_attn_gb300 as la
    from lightning_attention_attn_gb300 import build as labuild
    from lightning_attention_attn_gb300 import workloads as wl

    la.load(labuild.build())
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    pk = peaks()

    cfg = wl.PREFILL_8K
    T, H, d = cfg["lengths"][0], cfg["num_heads"], cfg["head_dim"]
    B = 128
    inp = wl.prefill_inputs(cfg["lengths"], H, d, dtype=torch.bfloat16, seed=0, device=dev)
    out = torch.empty_like(inp.q)
    fs = torch.empty((1, H, d, d), dtype=torch.float32, device=dev)

    def step():
        la.prefill(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens, chunk=0, out=out,
                   final_state=fs, stream=stream)

    for _ in range(max(3, args.warmup)):
        step()
    la.device_status(stream)
    torch.cuda.synchronize()

    K = args.steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    # The same K launches captured once as a CUDA graph and replayed: the
    # way a fixed-shape serving or training loop issues them (no per-launch
    # host work).  Captured on a side stream (the legacy default stream
    # cannot capture).
    gstream = torch.cuda.Stream(device=dev)
    gstream.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=gstream):
        for _ in range(K):
            la.prefill(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens, chunk=0, out=out,
                       final_state=fs, stream=gstream)
    with torch.cuda.stream(gstream):
        graph.replay()
    torch.cuda.synchronize()
    g_start = torch.cuda.Event(enable_timing=True)
    g_end = torch.cuda.Event(enable_timing=True)

    def graph_ms(fn, n):
        """Mean ms per call of fn(stream), n calls captured as one CUDA graph
        and replayed (after one untimed replay)."""
        gstream.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=gstream):
            for _ in range(n):
                fn(gstream)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(gstream):
            g.replay()
            e0.record(gstream)
            g.replay()
            e1.record(gstream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        # untimed soak right before the timed steps, so the clock samples
        # (every 50 ms) cover the GPU under this load even when K steps
        # take only milliseconds
        t_soak = time.perf_counter()
        while time.perf_counter() - t_soak < 1.0:
            for _ in range(50):
                step()
            torch.cuda.synchronize()
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for i in range(K):
            evs[i][0].record(stream)
            step()
            evs[i][1].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
        with torch.cuda.stream(gstream):
            g_start.record(gstream)
            graph.replay()
            g_end.record(gstream)
        torch.cuda.synchronize()
    barrier(ws)
    la.device_status(stream)
    eager_ms = t_start.elapsed_time(t_end)
    launch_ms = [a.elapsed_time(b) for a, b in evs]
    eager_launch_s = sum(launch_ms) / K / 1e3
    # the timed region of `value`: the graph replay of the K launches; the
    # average launch duration is its span over K (gaps between launches
    # included)
    total_ms = g_start.elapsed_time(g_end)
    avg_launch_s = total_ms / K / 1e3
    total_ms = max_over_ranks(total_ms, ws)
    tokens = sum_over_ranks(float(T * K), ws)
    value = tokens / (total_ms / 1e3)

    byts, flops = prefill_alg(T, H, d, B, 1)
    achieved_gbs = byts / avg_launch_s / 1e9
    traffic = ncu_traffic("prefill_tc_kernel", PREFILL_KERNEL_SRC)
    roofline = {"bound": "hbm", "achieved": round(achieved_gbs, 1), "peak": pk["hbm"],
                "unit": "GB/s", "frac": round(achieved_gbs / pk["hbm"], 4),
                "traffic": traffic, "peak_source": pk["source"],
                "kernel": "prefill_tc_kernel", "alg_bytes_per_launch": byts,
                "launch_ms": round(avg_launch_s * 1e3, 4),
                "eager": {"ms_per_step": round(max_over_ranks(eager_ms, ws) / K, 5),
                          "launch_ms": round(eager_launch_s * 1e3, 4),
                          "frac": round(byts / eager_launch_s / 1e9 / pk["hbm"], 4)}}
    tflops = flops / avg_launch_s / 1e12
    t_roof = max(byts / (pk["hbm"] * 1e9), flops / (pk["bf16"] * 1e12))
    tensor = {"alg_flops_per_launch": flops, "achieved_tflops": round(tflops, 2),
              "peak_tflops": pk["bf16"], "frac_of_bf16_peak": round(tflops / pk["bf16"], 4),
              "frac_of_roofline": round(t_roof / avg_launch_s, 4)}

    # ---------------- the other prefill workloads of the benchmark set:
    # 128K-token context (chunk 128 on tensor cores; chunk 64 on the
    # CUDA-core kernel timed once) and the 16-sequence varlen batch
    def time_prefill(lengths, chunk, reps, dtype=torch.bfloat16):
        pin = wl.prefill_inputs(lengths, H, d, dtype=dtype, seed=0, device=dev)
        pout = torch.empty_like(pin.q)
        pfs = torch.empty((len(lengths), H, d, d), dtype=torch.float32, device=dev)

        def run():
            la.prefill(pin.q, pin.k, pin.v, pin.decay, pin.cu_seqlens, chunk=chunk, out=pout,
                       final_state=pfs, stream=stream)
        run()
        torch.cuda.synchronize()
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(reps):
            run()
        a1.record(stream)
        torch.cuda.synchronize()
        la.device_status(stream)
        ms = a0.elapsed_time(a1) / reps
        Tn = sum(lengths)
        if dtype == torch.float32:  # the CUDA-core (FFMA) kernel
            byts, flops = prefill_alg(Tn, H, d, chunk, len(lengths))
            byts += Tn * H * d * 8  # fp32 inputs and output: twice the bf16 bytes
            return {"ms_per_launch": round(ms, 4), "tokens_per_s": round(Tn / (ms / 1e3), 1),
                    "tokens": Tn, "chunk": chunk, "dtype": "f32",
                    "kernel": "prefill_simt_kernel (FFMA)",
                    "roofline": cuda_core_roofline(flops, byts, ms, pk, sms)}
        B = chunk if chunk else 128
        byts, flops = prefill_alg(Tn, H, d, B, len(lengths))
        return {"ms_per_launch": round(ms, 4), "tokens_per_s": round(Tn / (ms / 1e3), 1),
                "tokens": Tn, "chunk": chunk, "kernel": "prefill_tc_kernel",
                "tensor_tiles_per_128_tokens": 128 // B if B <= 128 else 1,
                "roofline": {"bound": "hbm", "alg_bytes": byts,
                             "achieved": round(byts / (ms / 1e3) / 1e9, 1), "peak": pk["hbm"],
                             "unit": "GB/s", "frac": round(byts / (ms / 1e3) / 1e9 / pk["hbm"], 4)}}

    def time_channel_decay(lengths, reps, chunk=64):
        """Per-channel decay (lambda_h scaled by 1 - 0.01 i / (d - 1) for key
        channel i): 64-token blocks run the tcgen05 kernel, 32-token blocks
        the CUDA-core kernel."""
        pin = wl.prefill_inputs(lengths, H, d, dtype=torch.bfloat16, seed=0, device=dev)
        lam_cw = pin.decay[:, None].repeat(1, d).contiguous()
        lam_cw = lam_cw * (1.0 - 0.01 * torch.linspace(0, 1, d, device=dev))[None, :]
        pout = torch.empty_like(pin.q)

        def run():
            la.prefill_channel_decay(pin.q, pin.k, pin.v, lam_cw, pin.cu_seqlens, chunk=chunk,
                                     out=pout, stream=stream)
        run()
        torch.cuda.synchronize()
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(reps):
            run()
        a1.record(stream)
        torch.cuda.synchronize()
        la.device_status(stream)
        ms = a0.elapsed_time(a1) / reps
        Tn = sum(lengths)
        byts, flops = prefill_alg(Tn, H, d, chunk, len(lengths))
        byts -= len(lengths) * H * d * d * 4  # no final state requested
        byts += H * d * 4                      # the decay table
        if chunk != 64:
            return {"ms_per_launch": round(ms, 3), "tokens_per_s": round(Tn / (ms / 1e3), 1),
                    "chunk": chunk, "kernel": "prefill_simt_kernel (FFMA), per-channel decay",
                    "roofline": cuda_core_roofline(flops, byts, ms, pk, sms)}
        return {"ms_per_launch": round(ms, 4), "tokens_per_s": round(Tn / (ms / 1e3), 1),
                "chunk": chunk, "kernel": "prefill_cw_tc_kernel (tcgen05), per-channel decay",
                "roofline": {"bound": "hbm", "alg_bytes": byts,
                             "achieved": round(byts / (ms / 1e3) / 1e9, 1), "peak": pk["hbm"],
                             "unit": "GB/s", "frac": round(byts / (ms / 1e3) / 1e9 / pk["hbm"], 4),
                             "traffic": ncu_traffic("prefill_cw_tc_kernel", CW_KERNEL_SRC)
                             if Tn == 8192 else None},  # the counters are of the 8K layer
                "tensor": {"alg_flops": flops,
                           "frac_of_bf16_peak": round(flops / (ms / 1e3) / 1e12 / pk["bf16"], 4),
                           "note": "the tensor pipe runs about 6x the algorithmic flops: hi/lo "
                                   "operand pairs stacked on the M rows, three decay slabs, "
                                   "diagonal sub-blocks as whole tiles, and the query-key "
                                   "products repeated in both value-slice CTAs of a head"}}

    def time_snapshots(lengths, interval, reps):
        """Prefill of the layer that also writes the state every `interval`
        tokens (per-block prefix cache)."""
        pin = wl.prefill_inputs(lengths, H, d, dtype=torch.bfloat16, seed=0, device=dev)
        pout = torch.empty_like(pin.q)
        pfs = torch.empty((len(lengths), H, d, d), dtype=torch.float32, device=dev)
        nsnap = la.snapshot_count(pin.cu_seqlens, interval)
        psn = torch.empty((nsnap, H, d, d), dtype=torch.float32, device=dev)

        def run():
            la.prefill_snapshots(pin.q, pin.k, pin.v, pin.decay, pin.cu_seqlens, interval,
                                 out=pout, final_state=pfs, snapshots=psn, stream=stream)
        run()
        torch.cuda.synchronize()
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(reps):
            run()
        a1.record(stream)
        torch.cuda.synchronize()
        la.device_status(stream)
        ms = a0.elapsed_time(a1) / reps
        Tn = sum(lengths)
        byts, _ = prefill_alg(Tn, H, d, 128, len(lengths))
        byts += nsnap * H * d * d * 4
        return {"ms_per_launch": round(ms, 4), "tokens_per_s": round(Tn / (ms / 1e3), 1),
                "snapshots": nsnap, "interval": interval,
                "roofline": {"bound": "hbm", "alg_bytes": byts,
                             "achieved": round(byts / (ms / 1e3) / 1e9, 1), "peak": pk["hbm"],
                             "unit": "GB/s", "frac": round(byts / (ms / 1e3) / 1e9 / pk["hbm"], 4)}}

    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    more = {"prefill_8k_channel_decay": time_channel_decay([8192], 10),
            "prefill_8k_channel_decay_cuda_cores": time_channel_decay([8192], 3, chunk=32),
            "prefill_128k_channel_decay": time_channel_decay([131072], 3),
            "prefill_8k_snapshots_every_1024": time_snapshots([8192], 1024, 10),
            "prefill_8k_snapshots_every_128": time_snapshots([8192], 128, 10),
            "prefill_8k_chunk64": time_prefill([8192], 64, 10),
            "prefill_8k_chunk32": time_prefill([8192], 32, 10),
            "prefill_8k_fp32_cuda_cores": time_prefill([8192], 64, 5, torch.float32),
            "prefill_128k": time_prefill([131072], 0, 5),
            "prefill_128k_chunk64": time_prefill([131072], 64, 3),
            "prefill_128k_chunk256": time_prefill([131072], 256, 5),
            "varlen_16": time_prefill(wl.varlen_lengths().tolist(), 0, 5)}
    torch.cuda.empty_cache()

    # ---------------- decode: 128 seqs x 64 heads, 1000 consecutive steps
    dcfg = wl.DECODE_128
    dsteps = dcfg["steps"]
    dinp = wl.decode_inputs(dcfg["batch"], dcfg["num_heads"], dcfg["head_dim"], steps=dsteps,
                            dtype=torch.bfloat16, seed=0, device=dev)
    dout = torch.empty_like(dinp.q[0])

    def dstep(t):
        la.decode(dinp.q[t], dinp.k[t], dinp.v[t], dinp.decay, dinp.state, out=dout,
                  stream=stream)

    for t in range(5):
        dstep(t)
    torch.cuda.synchronize()
    d0 = torch.cuda.Event(enable_timing=True)
    d1 = torch.cuda.Event(enable_timing=True)
    d0.record(stream)
    for t in range(dsteps):
        dstep(t)
    d1.record(stream)
    torch.cuda.synchronize()
    dms_eager = d0.elapsed_time(d1) / dsteps
    # the 1000 consecutive steps as one CUDA graph (fresh q, k, v per step)
    gstream.wait_stream(stream)
    dgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(dgraph, stream=gstream):
        for t in range(dsteps):
            la.decode(dinp.q[t], dinp.k[t], dinp.v[t], dinp.decay, dinp.state, out=dout,
                      stream=gstream)
    with torch.cuda.stream(gstream):
        dgraph.replay()
        d0.record(gstream)
        dgraph.replay()
        d1.record(gstream)
    torch.cuda.synchronize()
    la.device_status(stream)
    dms = d0.elapsed_time(d1) / dsteps
    del dgraph
    dbytes = decode_alg(dcfg["batch"], dcfg["num_heads"], dcfg["head_dim"])
    dgbs = dbytes / (dms / 1e3) / 1e9
    decode = {"value": round(dcfg["batch"] / (dms / 1e3), 1), "unit": "tokens/s",
              "ms_per_step": round(dms, 5), "steps": dsteps,
              "config": {"workload": "decode_128", "batch": dcfg["batch"], "heads": 64,
                         "head_dim": 128, "state": "fp32 [128,64,128,128]", "io": "bf16"},
              "roofline": {"bound": "hbm", "achieved": round(dgbs, 1), "peak": pk["hbm"],
                           "unit": "GB/s", "frac": round(dgbs / pk["hbm"], 4),
                           "traffic": ncu_traffic("decode_kernel", DECODE_KERNEL_SRC),
                           "kernel": "decode_kernel", "alg_bytes_per_launch": dbytes,
                           "eager": {"ms_per_step": round(dms_eager, 5),
                                     "frac": round(dbytes / (dms_eager / 1e3) / 1e9 / pk["hbm"],
                                                   4)}},
              "issue": "the 1000 steps replayed as one CUDA graph (eager under roofline.eager)"}
    # the channel-wise decay step on the same batch (one lambda per head and
    # key channel, read per state row): 200 consecutive steps
    lam_cw = dinp.decay[:, None].repeat(1, dcfg["head_dim"]).contiguous()
    lam_cw = lam_cw * (1.0 - 0.01 * torch.linspace(0, 1, dcfg["head_dim"], device=dev))[None, :]
    csteps = 200
    for t in range(5):
        la.decode_channel_decay(dinp.q[t], dinp.k[t], dinp.v[t], lam_cw, dinp.state, out=dout,
                                stream=stream)
    torch.cuda.synchronize()
    d0.record(stream)
    for t in range(csteps):
        la.decode_channel_decay(dinp.q[t], dinp.k[t], dinp.v[t], lam_cw, dinp.state, out=dout,
                                stream=stream)
    d1.record(stream)
    torch.cuda.synchronize()
    cms = d0.elapsed_time(d1) / csteps
    cgbs = dbytes / (cms / 1e3) / 1e9
    decode["channel_decay"] = {"ms_per_step": round(cms, 5), "steps": csteps,
                               "roofline": {"bound": "hbm", "achieved": round(cgbs, 1),
                                            "peak": pk["hbm"], "unit": "GB/s",
                                            "frac": round(cgbs / pk["hbm"], 4)}}
    la.device_status(stream)
    del dinp

    # ---------------- backward on the same 8K-token layer (training step of
    # the attention: one causal and two anti-causal tensor-core launches)
    g = torch.Generator(device=dev)
    g.manual_seed(1)
    dout = torch.randn(inp.q.shape, generator=g, device=dev).to(torch.bfloat16)
    dq, dk, dv = (torch.empty_like(inp.q) for _ in range(3))

    def bstep():  # the tensor-core path needs no workspace
        la.backward(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens, dout, dq=dq, dk=dk, dv=dv,
                    stream=stream)

    for _ in range(3):
        bstep()
    torch.cuda.synchronize()
    b0 = torch.cuda.Event(enable_timing=True)
    b1 = torch.cuda.Event(enable_timing=True)
    b0.record(stream)
    for _ in range(K):
        bstep()
    b1.record(stream)
    torch.cuda.synchronize()
    la.device_status(stream)
    bms_eager = b0.elapsed_time(b1) / K
    bms = graph_ms(lambda s_: la.backward(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens, dout,
                                          dq=dq, dk=dk, dv=dv, stream=s_), K)
    la.device_status(stream)
    bbytes = T * H * d * 2 * 7  # q, k, v, dout read; dq, dk, dv written (bf16)
    bgbs = bbytes / (bms / 1e3) / 1e9
    backward = {"value": round(T / (bms / 1e3), 1), "unit": "tokens/s", "ms_per_step": round(bms, 4),
                "config": {"workload": "prefill_8k backward (dq, dk, dv)",
                           "issue": "K steps replayed as one CUDA graph"},
                "eager_ms_per_step": round(bms_eager, 4),
                "launches_per_step": 3,
                "roofline": {"bound": "hbm", "achieved": round(bgbs, 1), "peak": pk["hbm"],
                             "unit": "GB/s", "frac": round(bgbs / pk["hbm"], 4),
                             "alg_bytes_per_step": bbytes,
                             "note": "algorithmic bytes of the gradients; the implementation "
                                     "runs 3 tensor-core launches, each reading 3 inputs and "
                                     "writing 1 (12 x T x H x d x 2 bytes moved)"}}
    del dout, dq, dk, dv

    # ---------------- mixed serving step (decode + prefill on two streams):
    # every sequence continues from a cached state; a few have several new
    # tokens, the rest one
    # the decode stream at a higher priority: its small blocks start before
    # the prefill's large ones take the SMs
    dstream = torch.cuda.Stream(device=dev, priority=-1)

    def measure_mixed(mlen, label, seed):
        minp = wl.prefill_inputs(mlen, H, d, dtype=torch.bfloat16, seed=seed, device=dev)
        mstate = wl.cached_states(len(mlen), H, d, seed=seed + 1, device=dev)
        mcu = minp.cu_seqlens.cpu().tolist()
        mout = torch.empty_like(minp.q)

        def mstep(two):
            if two:
                la.mixed_step(minp.q, minp.k, minp.v, minp.decay, minp.cu_seqlens, mstate,
                              out=mout, prefill_stream=stream, decode_stream=dstream,
                              cu_seqlens_host=mcu)
            else:  # the same update through one prefill launch for every sequence
                la.prefill(minp.q, minp.k, minp.v, minp.decay, minp.cu_seqlens, out=mout,
                           initial_state=mstate, final_state=mstate, stream=stream)

        res = {"config": {"workload": label}}
        for two in (True, False):
            for _ in range(3):
                mstep(two)
            torch.cuda.synchronize()
            m0 = torch.cuda.Event(enable_timing=True)
            m1 = torch.cuda.Event(enable_timing=True)
            m0.record(stream)
            for _ in range(K):
                mstep(two)
            m1.record(stream)
            torch.cuda.synchronize()
            res[("ms_two_streams" if two else "ms_one_prefill_launch") + "_eager"] = round(
                m0.elapsed_time(m1) / K, 4)
        # the same steps replayed as CUDA graphs (the decode stream joins the
        # capture through the step's fork and join events)
        res["ms_two_streams"] = round(graph_ms(
            lambda s_: la.mixed_step(minp.q, minp.k, minp.v, minp.decay, minp.cu_seqlens, mstate,
                                     out=mout, prefill_stream=s_, decode_stream=dstream,
                                     cu_seqlens_host=mcu), K), 4)
        res["ms_one_prefill_launch"] = round(graph_ms(
            lambda s_: la.prefill(minp.q, minp.k, minp.v, minp.decay, minp.cu_seqlens, out=mout,
                                  initial_state=mstate, final_state=mstate, stream=s_), K), 4)
        la.device_status(stream)
        mbytes = len(mlen) * H * d * d * 4 * 2 + sum(mlen) * H * d * 2 * 4
        res["tokens_per_s"] = round(sum(mlen) / (res["ms_two_streams"] / 1e3), 1)
        res["speedup_vs_one_launch"] = round(res["ms_one_prefill_launch"] /
                                             res["ms_two_streams"], 2)
        res["roofline"] = {"bound": "hbm", "alg_bytes_per_step": mbytes,
                           "achieved": round(mbytes / (res["ms_two_streams"] / 1e3) / 1e9, 1),
                           "peak": pk["hbm"], "unit": "GB/s"}
        res["roofline"]["frac"] = round(res["roofline"]["achieved"] / pk["hbm"], 4)
        return res

    mixed = measure_mixed([256 if s_ in (0, 77) else 1 for s_ in range(128)],
                          "mixed step: 128 sequences x 64 heads, 2 with 256 new tokens, "
                          "126 with 1, cached fp32 states", 2)
    # the serving batch the pages time their two-stream split on: 20 requests,
    # 2 with 50-token inputs, the rest decoding
    mixed["pages_batch"] = measure_mixed([50 if s_ in (3, 11) else 1 for s_ in range(20)],
                                         "20 sequences x 64 heads, 2 with 50 new tokens, "
                                         "18 with 1, cached fp32 states", 4)

    # short inputs alone: the tensor-core block (one partial 128-token chunk)
    # against the CUDA-core kernel at chunk 32 and 64
    sinp = wl.prefill_inputs([50, 50], H, d, dtype=torch.bfloat16, seed=6, device=dev)
    sst = wl.cached_states(2, H, d, seed=7, device=dev)
    sout = torch.empty_like(sinp.q)
    sfs = torch.empty_like(sst)
    short = {"config": {"workload": "2 sequences x 50 new tokens x 64 heads from cached states"}}
    for ch in (0, 32, 64):
        def sstep():
            la.prefill(sinp.q, sinp.k, sinp.v, sinp.decay, sinp.cu_seqlens, chunk=ch, out=sout,
                       initial_state=sst, final_state=sfs, stream=stream)
        for _ in range(3):
            sstep()
        torch.cuda.synchronize()
        s0_ = torch.cuda.Event(enable_timing=True)
        s1_ = torch.cuda.Event(enable_timing=True)
        s0_.record(stream)
        for _ in range(K):
            sstep()
        s1_.record(stream)
        torch.cuda.synchronize()
        short["ms_chunk_%d" % ch if ch else "ms_tensor_core_block_128"] = round(
            s0_.elapsed_time(s1_) / K, 4)
    la.device_status(stream)
    mixed["short_inputs"] = short
    del sinp, sst, sout, sfs

    # ---------------- end to end through the public call, host buffers.
    # Every step copies its inputs from pinned host memory, runs the prefill
    # and copies the output and final state back; steps are pipelined over
    # two device buffer sets and three streams (the copy-in of step k + 1
    # and the copy-out of step k - 1 overlap the prefill of step k).
    hq, hk, hv = (t.cpu().pin_memory() for t in (inp.q, inp.k, inp.v))
    sets = [(inp.q, inp.k, inp.v, out, fs)]
    sets.append(tuple(torch.empty_like(t) for t in sets[0]))
    hout = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    hfs = [torch.empty(fs.shape, dtype=fs.dtype).pin_memory() for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_run = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def e2e_step(k_):
        b = k_ % 2
        dq_, dk_, dv_, dout_, dfs_ = sets[b]
        if used[b]:
            s_in.wait_event(ev_run[b])      # the prefill of step k - 2 read these inputs
        with torch.cuda.stream(s_in):
            dq_.copy_(hq, non_blocking=True)
            dk_.copy_(hk, non_blocking=True)
            dv_.copy_(hv, non_blocking=True)
        ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        if used[b]:
            stream.wait_event(ev_out[b])    # step k - 2's outputs have been copied out
        la.prefill(dq_, dk_, dv_, inp.decay, inp.cu_seqlens, chunk=0, out=dout_,
                   final_state=dfs_, stream=stream)
        ev_run[b].record(stream)
        s_out.wait_event(ev_run[b])
        with torch.cuda.stream(s_out):
            hout[b].copy_(dout_, non_blocking=True)
            hfs[b].copy_(dfs_, non_blocking=True)
        ev_out[b].record(s_out)
        used[b] = True

    for k_ in range(4):
        e2e_step(k_)
    torch.cuda.synchronize()
    barrier(ws)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for s_ in (stream, s_out):
        s_.wait_event(e0)
    for k_ in range(K):
        e2e_step(k_)
    e1.record(s_out)
    torch.cuda.synchronize()
    e_ms = max_over_ranks(e0.elapsed_time(e1), ws)
    h2d = 3 * hq.numel() * hq.element_size()
    d2h = hout[0].numel() * hout[0].element_size() + hfs[0].numel() * hfs[0].element_size()
    # the host link alone: the same three input copies, back to back
    l0 = torch.cuda.Event(enable_timing=True)
    l1 = torch.cuda.Event(enable_timing=True)
    l0.record(s_in)
    for _ in range(3):
        with torch.cuda.stream(s_in):
            for dst, src in zip(sets[0][:3], (hq, hk, hv)):
                dst.copy_(src, non_blocking=True)
    l1.record(s_in)
    torch.cuda.synchronize()
    h2d_gbs = 3 * h2d / (l0.elapsed_time(l1) / 1e3) / 1e9
    e2e = {"value": round(tokens / (e_ms / 1e3), 1), "unit": "tokens/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "ms_per_step": round(e_ms / K, 4),
           "pipelining": "2 device buffer sets, copy-in / prefill / copy-out streams",
           "h2d_link_gbs": round(h2d_gbs, 1),
           "frac_of_h2d_bound": round((h2d / (h2d_gbs * 1e9)) / (e_ms / K / 1e3), 4)}
    del sets

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": ws,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(total_ms / K, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1); q, k scaled by d^-1/2; lambda_h = exp(-2^(-8(h+1)/64)))",
        "config": {"workload": "prefill_8k", "batch": 1, "seq_len": T, "heads": H,
                   "head_dim": d, "chunk": B, "value_slices_per_head": 2,
                   "inputs_vs_l2": "q, k, v = 384 MiB > 129 MB L2; no flush needed",
                   "parallelism": f"replicas x{ws}",
                   "issue": "the K launches replayed as one CUDA graph (eager numbers under "
                            "roofline.eager)"},
        "roofline": roofline, "tensor": tensor, "decode": decode, "backward": backward,
        "mixed": mixed, "more_prefill": more,
        "e2e": e2e,
        "gpu_launches": K,
    }
    clocks = clk.summary()
    line["clocks"] = clocks
    line["config"]["clocks_window"] = "1 s untimed soak of the same step + the timed steps"
    if rank == 0:
        host = wl.PrefillInputs(inp.q.cpu(), inp.k.cpu(), inp.v.cpu(), inp.decay.cpu(),
                                inp.cu_seqlens.cpu())
        line["cpu_baseline"] = cpu_baseline(host)
    # Compact copies of the secondary measurements, last in the line so that
    # a reader of only the line's tail still sees them.
    def frac(x):
        return x.get("roofline", {}).get("frac") if isinstance(x, dict) else x
    line["summary"] = {
        "decode_128": {"ms_per_step": decode["ms_per_step"], "tokens_per_s": decode["value"],
                       "hbm_frac": decode["roofline"]["frac"],
                       "eager_hbm_frac": decode["roofline"]["eager"]["frac"]},
        "backward_8k": {"ms_per_step": backward["ms_per_step"],
                        "tokens_per_s": backward["value"],
                        "hbm_frac": backward["roofline"]["frac"],
                        "launches_per_step": backward["launches_per_step"]},
        "prefill_8k": {"ms_per_launch": round(total_ms / K, 5), "hbm_frac": roofline["frac"],
                       "eager_hbm_frac": roofline["eager"]["frac"]},
        "chunk_sweep_hbm_frac": {k_: frac(more.get(k_)) for k_ in
                                 ("prefill_8k_chunk32", "prefill_8k_chunk64",
                                  "prefill_128k_chunk64", "prefill_128k",
                                  "prefill_128k_chunk256")},
        "varlen_16_hbm_frac": frac(more.get("varlen_16")),
        "channel_decay_8k": {
            "tensor_cores_ms": more["prefill_8k_channel_decay"]["ms_per_launch"],
            "tensor_cores_hbm_frac": frac(more["prefill_8k_channel_decay"]),
            "cuda_cores_ms": more["prefill_8k_channel_decay_cuda_cores"]["ms_per_launch"],
            "tensor_cores_128k_ms": more["prefill_128k_channel_decay"]["ms_per_launch"]},
    }
    return line


def run_only(args):
    """W + K back-to-back launches of one kernel on its measured workload
    (the 8K-token layer for prefill, the 128-sequence batch for decode), for
    profilers: no clocks, no e2e, no CPU baseline."""
    import torch
    import lightning_attention_attn_gb300 as la
    from lightning_attention_attn_gb300 import build as labuild
    from lightning_attention_attn_gb300 import workloads as wl
    la.load(labuild.build())
    if args.only == "prefill":
        cfg = wl.PREFILL_8K
        inp = wl.prefill_inputs(cfg["lengths"], cfg["num_heads"], cfg["head_dim"],
                                dtype=torch.bfloat16, seed=0, device="cuda")
        out = torch.empty_like(inp.q)
        fs = torch.empty((1, cfg["num_heads"], 128, 128), device="cuda")
        for _ in range(args.warmup + args.steps):
            la.prefill(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens, out=out, final_state=fs)
    elif args.only in ("channel_decay", "prefill_chunk64", "prefill_fp32"):
        # the 8K-token layer: per-channel decay on the tensor-core kernel
        # (lambda_h scaled by 1 - 0.01 i / (d - 1) for key channel i), the
        # scalar decay with 64-token blocks on the tensor cores, or fp32
        # inputs (chunk 64) on the CUDA-core kernel
        cfg = wl.PREFILL_8K
        inp = wl.prefill_inputs(cfg["lengths"], cfg["num_heads"], cfg["head_dim"],
                                dtype=torch.float32 if args.only == "prefill_fp32"
                                else torch.bfloat16, seed=0, device="cuda")
        d = cfg["head_dim"]
        lam_cw = inp.decay[:, None].repeat(1, d).contiguous()
        lam_cw = lam_cw * (1.0 - 0.01 * torch.linspace(0, 1, d, device="cuda"))[None, :]
        out = torch.empty_like(inp.q)
        for _ in range(args.warmup + args.steps):
            if args.only == "channel_decay":
                la.prefill_channel_decay(inp.q, inp.k, inp.v, lam_cw, inp.cu_seqlens, chunk=64,
                                         out=out)
            else:
                la.prefill(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens, chunk=64, out=out)
    elif args.only == "backward":
        cfg = wl.PREFILL_8K
        inp = wl.prefill_inputs(cfg["lengths"], cfg["num_heads"], cfg["head_dim"],
                                dtype=torch.bfloat16, seed=0, device="cuda")
        dout = torch.randn_like(inp.q, dtype=torch.float32).to(torch.bfloat16)
        for _ in range(args.warmup + args.steps):
            la.backward(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens, dout)
    else:
        cfg = wl.DECODE_128
        n = args.warmup + args.steps
        dinp = wl.decode_inputs(cfg["batch"], cfg["num_heads"], cfg["head_dim"], steps=n,
                                dtype=torch.bfloat16, seed=0, device="cuda")
        out = torch.empty_like(dinp.q[0])
        for t in range(n):
            la.decode(dinp.q[t], dinp.k[t], dinp.v[t], dinp.decay, dinp.state, out=out)
    torch.cuda.synchronize()
    la.device_status()
    return 0


# --------------------------------------------------------- reference arm
def run_reference(args, ws, rank):
    """The oracle (fp64, CPU, as it stands) on a bounded sample of the same
    workload: each step is the first 1024 tokens of the 8K layer, all 64
    heads, recurrent form.  Rank 0 only."""
    if rank != 0:
        return None
    import torch
    import oracle
    from lightning_attention_attn_gb300 import workloads as wl
    S = 1024
    inp = wl.prefill_inputs([S], 64, 128, dtype=torch.bfloat16, seed=0)
    threads = oracle.max_threads()
    for _ in range(args.warmup):
        oracle.recurrent(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.recurrent(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens)
    dt = time.perf_counter() - t0
    value = S * args.steps / dt
    sample = (f"first {S} tokens of the prefill_8k workload per step, all 64 heads, "
              f"fp64 recurrent form, {threads} threads")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tokens/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (same recipe as our arm)",
            "config": {"workload": "prefill_8k", "batch": 1, "seq_len": 8192, "heads": 64,
                       "head_dim": 128, "parallelism": "cpu oracle, rank 0"},
            "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--only", choices=["prefill", "decode", "backward", "channel_decay",
                                       "prefill_chunk64", "prefill_fp32"], default=None,
                    help="profiling aid: run just W + K launches of one kernel on its "
                         "workload and print nothing else")
    args = ap.parse_args(argv)
    if args.only:
        return run_only(args)
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        # the CPU oracle runs on rank 0 only; other ranks exit without work
        ws = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        line = run_reference(args, ws, rank)
        if rank == 0 and line is not None:
            print(json.dumps(line), flush=True)
        return
    ws, rank, local = dist_setup()
    line = run_ours(args, ws, rank, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
