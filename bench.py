"""Benchmark of the PSA attention step (fused forward + dQ + dK/dV backward) on GB300.

One step = psa_attention_fwd (QKV -> Out, LSE, extracted V) + psa_attention_bwd
(-> dQKV; for this sequence length one kernel per head computes dQ, dK and dV)
over one batch of the 'psa_fwdbwd_n400' workload: B=64, num_heads=4, KEY_DIM=32,
20x20 (N=400), bf16, synthetic seeded N(0,1) inputs.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--split-bwd]

--split-bwd times the two-kernel backward instead (psa_attention_bwd_dq then
psa_attention_bwd_dkdv), the form that long sequences use.

--sweep times the compute-bound cases instead, one JSON line each: the raw
FlashAttention-2 calls over BH=64, N in {1024, 4096, 16384}, d in {32, 64}
(forward, and dQ + dK/dV backward) and the N=1600 PSA step (B=32, 8 heads,
40x40), as TFLOP/s and as a fraction of the bf16 tensor peak.

--layout times the data-movement kernels instead (pack, its inverse, merge, its
inverse, extract) as GB/s against the measured HBM bandwidth, cold and hot L2,
and the unfused pack -> FA2 x 2 -> merge chain next to the fused calls.

--impl reference times the fp64 CPU oracle (the test oracle, untuned) on the
host cores, on a bounded sample of the same workload per step.

Under torchrun (N > 1) every rank runs its own replica of the workload (the path
has no exchange step: heads and batches are independent), so scaling is weak and
no collective touches the data path; only the timing uses a barrier and a max.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "psa_fwdbwd_n400"
METRIC = "PSA attention fwd+bwd tokens/s and TFLOP/s at N=400, KEY_DIM=32; % roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# DRAM bytes per call of each step part come from the ncu capture recorded in
# profiles/dram_traffic.json, which also records a hash of the kernel source the
# capture ran; a part whose source has changed since reports no traffic.
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")
CSRC = os.path.join(ROOT, "vision_transformer_attention_psapackqkv_gb300", "csrc")


def source_hash(files):
    """sha256 (first 16 hex digits) over the named kernel source files."""
    import hashlib

    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(part):
    """(bytes, note) of the recorded ncu capture of `part`, or (None, reason)."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)["parts"][part]
    except (OSError, KeyError, ValueError):
        return None, "no capture recorded"
    if source_hash(rec["sources"]) != rec["source_hash"]:
        return None, "kernel changed since the capture of " + rec["captured"]
    return rec["dram_bytes"], rec["kernel"] + ", ncu capture of " + rec["captured"]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        hbm = float(d.get("hbm_gbs") or d.get("hbm_GBps"))
        tf = float(d.get("bf16_tflops"))
        tfs = float(d.get("bf16_tflops_sustained", tf))
        return {"hbm_gbs": hbm, "bf16_tflops": tf, "bf16_tflops_sustained": tfs}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------- work model
def work_model(w):
    """Algorithmic FLOPs and HBM bytes of each kernel of one step (bf16 = 2 bytes).

    fwd   : S = Q K^T (2 N^2 KD) and O = P [V_lo|V_hi] (2 N^2 2KD) per head;
            reads QKV, writes Out, LSE and the extracted V.
    bwd_dq: S, dP = dO V^T (2 N^2 2KD), dQ = dS K (2 N^2 KD) per head; reads QKV
            (Q, K, V planes), Out, dOut, LSE; writes dQ and delta.
    bwd_dkdv: S^T, dP^T, dV = P^T dO (2 N^2 2KD), dK = dS^T Q (2 N^2 KD); reads QKV,
            dOut, LSE, delta; writes dK, dV.
    bwd   : the one-kernel backward: S^T, dP^T, dV, dK and dQ = dS K once each per
            head (2 N^2 (KD + 2KD + 2KD + KD + KD)); reads QKV, Out, dOut, LSE;
            writes dQKV.
    step  : the algorithmic total (S computed once in the forward and once in the
            backward): 192 N^2 + 448 N^2 FLOPs per head; bytes = QKV + Out + V
            written, QKV + Out + dOut read and dQKV written, LSE written and read.
    """
    N, BH, KD, B = w.N, w.BH, w.key_dim, w.B
    C, c = w.qkv_channels, w.out_channels
    e = 2
    n2 = float(N) * N * BH
    lse = BH * N * 4
    k = {
        "fwd": {"flops": n2 * (2 * KD + 2 * 2 * KD), "bytes": B * N * (C + c + c) * e + lse},
        "bwd_dq": {"flops": n2 * (2 * KD + 2 * 2 * KD + 2 * KD),
                   "bytes": B * N * (C + c + c + KD * w.num_heads) * e + 2 * lse},
        "bwd_dkdv": {"flops": n2 * (2 * KD + 2 * 2 * KD + 2 * 2 * KD + 2 * KD),
                     "bytes": B * N * (C + c + 3 * KD * w.num_heads) * e + 2 * lse},
        "bwd": {"flops": n2 * 2 * 7 * KD, "bytes": B * N * (C + c + c + C) * e + lse},
    }
    step = {"flops": n2 * (192 / 32 * KD + 448 / 32 * KD),
            "bytes": B * N * (C + c + c) * e + lse + B * N * (C + c + c + C) * e + lse}
    return k, step


# ----------------------------------------------------------------------------- ranks
def max_over_ranks(value, dist=None, device=None):
    """A per-rank float reduced to its maximum over all ranks (the job takes as long
    as its slowest replica); unchanged on a single process."""
    if dist is None:
        return float(value)
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_step, world, steps, ms):
    """Whole-job throughput: the units every replica processed over the job's time."""
    return units_per_step * world * steps / (ms / 1e3)


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML (read-only) in a thread."""

    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
               0x4: "sw_power_cap", 0x80: "hw_power_brake_slowdown", 0x1: "gpu_idle"}

    def __init__(self, index=0, period=0.002):
        self.samples, self.reasons, self.ok = [], 0, False
        self.period, self._stop = period, threading.Event()
        try:
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nv.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            if self.nv.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(self.h)) != 0:
                return
            mx = ctypes.c_uint()
            self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))
            self.max_mhz = int(mx.value)
            self.ok = True
        except OSError:
            pass

    def _sample(self):
        c = ctypes.c_uint()
        r = ctypes.c_ulonglong()
        if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(c)) == 0:
            self.samples.append(int(c.value))
        if self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h, ctypes.byref(r)) == 0:
            self.reasons |= int(r.value)

    def _run(self):
        while not self._stop.is_set():
            self._sample()
            time.sleep(self.period)

    def __enter__(self):
        if self.ok:
            self._sample()
            self.t = threading.Thread(target=self._run, daemon=True)
            self.t.start()
        return self

    def __exit__(self, *a):
        if self.ok:
            self._stop.set()
            self.t.join()
            self._sample()

    def summary(self):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvml unavailable"]}
        names = [n for bit, n in self.REASONS.items() if self.reasons & bit and n != "gpu_idle"]
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": names, "samples": len(self.samples)}


# ----------------------------------------------------------------------------- our arm
def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch

    from vision_transformer_attention_psapackqkv_gb300 import binding as B
    from vision_transformer_attention_psapackqkv_gb300.inputs import PSA_WORKLOADS, workload_inputs

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    w = PSA_WORKLOADS[WORKLOAD]
    scale = 1.0 / math.sqrt(w.key_dim)
    ins = workload_inputs(w)
    to_dev = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    qkv0, dout0 = to_dev(ins["qkv"]), to_dev(ins["dout"])
    shape = B.shape_of(qkv0, w.num_heads, w.key_dim)
    # rotate input/output sets whose footprint exceeds twice the L2 (129 MB)
    per_set = (qkv0.numel() * 2 * 2 + dout0.numel() * 2 * 3 + w.BH * w.N * 8)
    nsets = max(3, math.ceil(2 * 2 * 129e6 / per_set))
    sets = []
    for i in range(nsets):
        qkv = qkv0 if i == 0 else qkv0.roll(i, dims=0).contiguous()
        dout = dout0 if i == 0 else dout0.roll(i, dims=0).contiguous()
        sets.append({
            "qkv": qkv, "dout": dout,
            "out": torch.empty_like(dout), "vres": torch.empty_like(dout),
            "lse": torch.empty((w.BH, w.N), dtype=torch.float32, device="cuda"),
            "delta": torch.empty((w.BH, w.N), dtype=torch.float32, device="cuda"),
            "dqkv": torch.empty_like(qkv),
            "ws": torch.empty(B.psa_attention_bwd_workspace_size(shape), dtype=torch.uint8,
                              device="cuda"),
        })
    stream = torch.cuda.current_stream()

    def fwd(s, st=stream):
        B.psa_attention_fwd(s["qkv"], s["out"], s["lse"], s["vres"], shape, scale, st)

    def bwd_dq(s, st=stream):
        B.psa_attention_bwd_dq(s["qkv"], s["out"], s["dout"], s["lse"], s["delta"], s["dqkv"], shape,
                               scale, st)

    def bwd_dkdv(s, st=stream):
        B.psa_attention_bwd_dkdv(s["qkv"], s["dout"], s["lse"], s["delta"], None, s["dqkv"], shape, scale,
                                 st)

    def bwd(s, st=stream):
        B.psa_attention_bwd(s["qkv"], s["out"], s["dout"], s["lse"], None, s["dqkv"], s["ws"], shape,
                            scale, st)

    if args.split_bwd:
        parts = (("fwd", fwd), ("bwd_dq", bwd_dq), ("bwd_dkdv", bwd_dkdv))
    else:
        parts = (("fwd", fwd), ("bwd", bwd))
    # kernels per call: the forward (PsaExtractV fused) 1; psa_attention_bwd at this
    # sequence length 1 (one kernel per head, delta included); dQ 1; dK/dV 1
    launches = {"fwd": 1, "bwd": 1, "bwd_dq": 1, "bwd_dkdv": 1}
    launches_per_step = sum(launches[name] for name, _ in parts)

    def barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    for i in range(args.warmup):
        s = sets[i % nsets]
        for _, f in parts:
            f(s)
    barrier()
    if B.psa_get_last_device_error() != 0:
        raise RuntimeError("device error during warm-up")
    K = args.steps
    # The step loop is timed as a caller runs it: kernels back to back with no
    # event between them (the kernels use programmatic dependent launch, which an
    # event between two kernels would defeat).  The per-part times come from a
    # second pass of the same K steps with events around every part.
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local_rank)
    with sampler:
        start.record(stream)
        for i in range(K):
            s = sets[i % nsets]
            for _, f in parts:
                f(s)
        stop.record(stream)
        torch.cuda.synchronize()
    ms_total = start.elapsed_time(stop)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(parts) + 1)] for _ in range(K)]
    for i in range(K):
        s = sets[i % nsets]
        e = ev[i]
        e[0].record(stream)
        for j, (_, f) in enumerate(parts):
            f(s)
            e[j + 1].record(stream)
    torch.cuda.synchronize()
    per = {name: statistics.mean(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(K))
           for j, (name, _) in enumerate(parts)}
    ms_total = max_over_ranks(ms_total, dist, "cuda")
    if B.psa_get_last_device_error() != 0:
        raise RuntimeError("device error during the timed region")

    # end to end through the C ABI from pinned host buffers
    h_qkv = sets[0]["qkv"].cpu().pin_memory()
    h_dout = sets[0]["dout"].cpu().pin_memory()
    h_out = torch.empty(sets[0]["out"].shape, dtype=torch.bfloat16).pin_memory()
    h_vres = torch.empty_like(h_out).pin_memory()
    h_lse = torch.empty(sets[0]["lse"].shape, dtype=torch.float32).pin_memory()
    h_dqkv = torch.empty(sets[0]["dqkv"].shape, dtype=torch.bfloat16).pin_memory()
    Ke = max(3, min(K, 200))
    # Steps are pipelined the way a caller streaming batches would: the inputs of
    # step i+1 go up (copy stream `cin`) and the results of step i-1 come down
    # (`cout`) while step i computes on `cs`; two device sets alternate, and
    # events keep every copy and every call in order on its buffer.  The whole
    # sequence of Ke steps is captured once into a CUDA graph and replayed, so
    # host-side launch overhead stays out of the measurement.
    # Each direction is split over two streams (two copy engines at once).
    cs = torch.cuda.Stream()
    cins = (torch.cuda.Stream(), torch.cuda.Stream())
    couts = (torch.cuda.Stream(), torch.cuda.Stream())
    bufs = (sets[0], sets[1 % nsets])
    ev_in = [[torch.cuda.Event() for _ in range(2)] for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [[torch.cuda.Event() for _ in range(2)] for _ in range(2)]
    up = (lambda s: s["qkv"].copy_(h_qkv, non_blocking=True),
          lambda s: s["dout"].copy_(h_dout, non_blocking=True))

    def down0(s):
        h_dqkv.copy_(s["dqkv"], non_blocking=True)

    def down1(s):
        h_out.copy_(s["out"], non_blocking=True)
        h_vres.copy_(s["vres"], non_blocking=True)
        h_lse.copy_(s["lse"], non_blocking=True)
    down = (down0, down1)

    def e2e_steps(n):
        for c in cins + couts:
            c.wait_stream(cs)
        for i in range(n):
            bi = i % 2
            s = bufs[bi]
            for k in range(2):
                with torch.cuda.stream(cins[k]):
                    if i >= 2:
                        cins[k].wait_event(ev_comp[bi])  # step i-2 has read this set's inputs
                    up[k](s)
                    ev_in[k][bi].record(cins[k])
                cs.wait_event(ev_in[k][bi])
                if i >= 2:
                    cs.wait_event(ev_out[k][bi])  # step i-2's results have left this set
            for _, f in parts:
                f(s, cs)
            ev_comp[bi].record(cs)
            for k in range(2):
                with torch.cuda.stream(couts[k]):
                    couts[k].wait_event(ev_comp[bi])
                    down[k](s)
                    ev_out[k][bi].record(couts[k])
        for c in cins + couts:
            cs.wait_stream(c)

    barrier()
    with torch.cuda.stream(cs):
        e2e_steps(4)  # warm-up outside any graph
    torch.cuda.synchronize()
    e2e_mode = "cuda-graph"
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cs):
            e2e_steps(Ke)
        run_e2e = graph.replay
    except Exception as exc:  # capture unavailable: same sequence, launched eagerly
        e2e_mode = f"eager ({type(exc).__name__})"
        torch.cuda.synchronize()

        def run_e2e():
            with torch.cuda.stream(cs):
                e2e_steps(Ke)
    run_e2e()  # warm replay
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cs)
    with torch.cuda.stream(cs):
        run_e2e()
    e1.record(cs)
    torch.cuda.synchronize()
    if B.psa_get_last_device_error() != 0:
        raise RuntimeError("device error during the end-to-end run")
    ms_e2e = max_over_ranks(e0.elapsed_time(e1), dist, "cuda")
    h2d = h_qkv.numel() * 2 + h_dout.numel() * 2
    d2h = h_out.numel() * 2 * 2 + h_lse.numel() * 4 + h_dqkv.numel() * 2

    tokens_per_step = w.B * w.N
    kmodel, step_model = work_model(w)
    peaks, peak_src = load_peaks()
    ms_step = ms_total / K
    value = job_throughput(tokens_per_step, world, K, ms_total)
    tflops = job_throughput(step_model["flops"], world, K, ms_total) / 1e12
    # the dominant kernel (largest time share) and its roofline
    dom = max(per, key=per.get)
    km = kmodel[dom]
    t_s = per[dom] / 1e3
    t_flop = km["flops"] / (peaks["bf16_tflops"] * 1e12)
    t_byte = km["bytes"] / (peaks["hbm_gbs"] * 1e9)
    if t_byte >= t_flop:
        roof = {"bound": "hbm", "achieved": km["bytes"] / t_s / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": km["flops"] / t_s / 1e12, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"], roof["traffic_source"] = measured_traffic(dom)
    roof["kernel"] = dom
    roof["peak_source"] = peak_src
    step_roof_time = max(step_model["flops"] / (peaks["bf16_tflops_sustained"] * 1e12),
                         step_model["bytes"] / (peaks["hbm_gbs"] * 1e9))
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) QKV and dOut)",
        "config": {"workload": WORKLOAD, "B": w.B, "num_heads": w.num_heads, "key_dim": w.key_dim,
                   "H": w.H, "W": w.W, "N": w.N, "global_batch": w.B * world, "seq_len": w.N,
                   "parallelism": f"replicas x{world}",
                   "backward": "two kernels (dQ, dK/dV)" if args.split_bwd else "psa_attention_bwd",
                   "l2": f"rotating {nsets} input/output sets "
                   f"({nsets * per_set / 1e6:.0f} MB > 2 x L2)"},
        "tflops": tflops,
        "step_roofline": {"frac": step_roof_time / (ms_step / 1e3), "roofline_us": step_roof_time * 1e6,
                          "flops": step_model["flops"], "bytes": step_model["bytes"],
                          "peak_source": peak_src},
        "kernel_us": {k: v * 1e3 for k, v in per.items()},
        # consecutive kernels overlap their prologue with the previous kernel's tail
        # (programmatic dependent launch), so the parts, timed with events between
        # them, add up to more than ms_per_step
        "pdl": True,
        "roofline": roof,
        "e2e": {"value": job_throughput(tokens_per_step, world, Ke, ms_e2e), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": Ke,
                "pipelining": "H2D of step i+1 and D2H of step i-1 overlap step i",
                "launch": e2e_mode},
        "gpu_launches": launches_per_step * K,
        "clocks": sampler.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, scale, budget_s=args.cpu_seconds)
    if dist is not None:
        dist.destroy_process_group()
    return line


# ----------------------------------------------------------------------------- the oracle on CPU
def cpu_baseline(w, scale, budget_s=15.0, batches=None):
    """Times the fp64 oracle (PSA forward + backward) on the workload's inputs, on
    all host cores: the first `batches` batch items, grown (doubling) towards the
    whole batch, and the whole batch repeated until the timed sample lasts about
    two thirds of `budget_s`."""
    import oracle
    from vision_transformer_attention_psapackqkv_gb300.inputs import storage_to_f64, workload_inputs

    oracle.build()
    ins = workload_inputs(w)
    threads = oracle.default_threads()

    def run(nb, reps=1):
        q = storage_to_f64(ins["qkv"][:nb], w.dtype)
        d = storage_to_f64(ins["dout"][:nb], w.dtype)
        t0 = time.perf_counter()
        for _ in range(reps):
            oracle.psa_fwd(q, w.num_heads, w.key_dim, scale, nthreads=threads)
            oracle.psa_bwd(q, d, w.num_heads, w.key_dim, scale, nthreads=threads)
        return time.perf_counter() - t0

    reps = 1
    if batches is None:
        nb = max(1, math.ceil(threads / w.num_heads))
        t = run(nb)
        while t < budget_s / 4 and nb < w.B:
            nb = min(w.B, nb * 2)
            t = run(nb)
        if nb == w.B and t < budget_s / 3:
            reps = min(64, max(1, math.ceil(budget_s * 2 / 3 / max(t, 1e-3))))
            t = run(nb, reps)
    else:
        nb = batches
        t = run(nb)
    return {"value": reps * nb * w.N / t, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{reps} x {nb} of {w.B} batch items ({nb * w.num_heads} heads, "
                      f"{nb * w.N} tokens per pass), fp64 forward + backward, {t:.2f} s"}


# ----------------------------------------------------------------------------- sweep
def _time_loop(torch, fn, iters, warmup):
    for i in range(warmup):
        fn(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(iters):
        fn(i)
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / iters * 1e-3  # seconds per call


def _time_graph(torch, fn, iters, warmup):
    """Seconds per call of fn(i), i = 0 .. iters-1, replayed from a CUDA graph so the
    host's launch rate does not set the pace of short kernels."""
    for i in range(warmup):
        fn(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=s):
        for i in range(iters):
            fn(i)
    # replay() launches on the current stream (not the capture stream): time there
    with torch.cuda.stream(s):
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        g.replay()
        e1.record(s)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / iters * 1e-3


def run_sweep(args):
    """The long-sequence FA2 sweep and the N=1600 PSA step against the tensor peak.

    FLOPs are the algorithmic ones: FA2 forward 4 BH N^2 d, backward 10 BH N^2 d
    (S recomputed once); PSA step 192 N^2 + 448 N^2 per head (KD = 32).  The loops
    run for seconds, so the fraction is taken against the sustained bf16 peak.
    Inputs are seeded N(0,1) bf16 drawn on the device; enough input/output sets
    rotate to exceed twice the L2 where one set is smaller than that.
    """
    import torch

    from vision_transformer_attention_psapackqkv_gb300 import binding as B
    from vision_transformer_attention_psapackqkv_gb300.inputs import (FA2_SWEEP_BH, FA2_SWEEP_D,
                                                                      FA2_SWEEP_N, FA2_SWEEP_SEED,
                                                                      PSA_WORKLOADS)

    peaks, src = load_peaks()
    peak = peaks["bf16_tflops_sustained"]
    gen = torch.Generator(device="cuda")
    gen.manual_seed(FA2_SWEEP_SEED)
    rnd = lambda *shape: torch.randn(shape, generator=gen, device="cuda").to(torch.bfloat16)
    lines = []

    def emit(workload, part, flops, sec, extra):
        tf = flops / sec / 1e12
        line = {"metric": "attention TFLOP/s (algorithmic FLOPs)", "workload": workload,
                "part": part, "value": tf, "unit": "TFLOP/s", "us": sec * 1e6,
                "higher_is_better": True, "dtype": "bf16", "flops": flops,
                "tensor": {"peak": peak, "unit": "TFLOP/s", "frac": tf / peak,
                           "peak_source": f"{src}, sustained"}}
        line.update(extra)
        lines.append(line)
        print(json.dumps(line), flush=True)

    BH = FA2_SWEEP_BH
    for d in FA2_SWEEP_D:
        for N in FA2_SWEEP_N:
            if args.case not in (None, f"fa2_bh{BH}_n{N}_d{d}"):
                continue
            shp = (BH, N, d)
            per_set = 8 * BH * N * d * 2 + 2 * BH * N * 4
            nsets = max(1, math.ceil(2 * 129e6 / per_set) + (1 if per_set < 2 * 129e6 else 0))
            sets = []
            for _ in range(nsets):
                q, k, v, do = rnd(*shp), rnd(*shp), rnd(*shp), rnd(*shp)
                sets.append({"q": q, "k": k, "v": v, "do": do, "o": torch.empty_like(q),
                             "dq": torch.empty_like(q), "dk": torch.empty_like(q),
                             "dv": torch.empty_like(q),
                             "lse": torch.empty((BH, N), dtype=torch.float32, device="cuda"),
                             "delta": torch.empty((BH, N), dtype=torch.float32, device="cuda")})
            sc = 1.0 / math.sqrt(d)

            def fwd(i):
                s = sets[i % nsets]
                B.flash_attn2_fwd(s["q"], s["k"], s["v"], s["o"], s["lse"], sc)

            def bwd(i):
                s = sets[i % nsets]
                B.flash_attn2_bwd_dq(s["q"], s["k"], s["v"], s["o"], s["do"], s["lse"], s["delta"],
                                     s["dq"], sc)
                B.flash_attn2_bwd_dkdv(s["q"], s["k"], s["v"], s["do"], s["lse"], s["delta"],
                                       s["dk"], s["dv"], sc)

            ff, fb = 4.0 * BH * N * N * d, 10.0 * BH * N * N * d
            iters = max(5, min(400, int(3e13 / ff)))
            with ClockSampler() as clk:
                tfw = _time_loop(torch, fwd, iters, max(3, nsets))
                tbw = _time_loop(torch, bwd, iters, max(3, nsets))
            if B.psa_get_last_device_error() != 0:
                raise RuntimeError("device error in the sweep")
            extra = {"config": {"BH": BH, "N": N, "d": d, "iters": iters, "sets": nsets},
                     "clocks": clk.summary()}
            emit(f"fa2_bh{BH}_n{N}_d{d}", "fwd", ff, tfw, extra)
            emit(f"fa2_bh{BH}_n{N}_d{d}", "bwd (dQ + dK/dV)", fb, tbw, extra)
            del sets
            torch.cuda.empty_cache()

    w = PSA_WORKLOADS["psa_fwdbwd_n1600"]
    if args.case not in (None, w.name):
        return lines
    qkv = rnd(w.B, w.qkv_channels, w.H, w.W)
    dout = rnd(w.B, w.out_channels, w.H, w.W)
    shape = B.shape_of(qkv, w.num_heads, w.key_dim)
    sc = 1.0 / math.sqrt(w.key_dim)
    out, vres, dqkv = torch.empty_like(dout), torch.empty_like(dout), torch.empty_like(qkv)
    lse = torch.empty((w.BH, w.N), dtype=torch.float32, device="cuda")
    ws = torch.empty(B.psa_attention_bwd_workspace_size(shape), dtype=torch.uint8, device="cuda")
    pf = lambda i: B.psa_attention_fwd(qkv, out, lse, vres, shape, sc)
    pb = lambda i: B.psa_attention_bwd(qkv, out, dout, lse, None, dqkv, ws, shape, sc)
    n2 = float(w.N) * w.N * w.BH
    with ClockSampler() as clk:
        tpf = _time_loop(torch, pf, 100, 5)
        tpb = _time_loop(torch, pb, 100, 5)
    extra = {"config": {"B": w.B, "num_heads": w.num_heads, "key_dim": w.key_dim, "H": w.H,
                        "W": w.W, "N": w.N, "iters": 100, "sets": 1},
             "clocks": clk.summary()}
    emit(w.name, "fwd", 192 * n2, tpf, extra)
    emit(w.name, "bwd", 448 * n2, tpb, extra)
    emit(w.name, "fwd+bwd", 640 * n2, tpf + tpb, extra)
    return lines


def run_layout(args):
    """The data-movement kernels (PsaPackQkv, its inverse, PsaMergeAttn, its inverse,
    PsaExtractV) on the psa_fwdbwd_n400 workload, as GB/s of algorithmic bytes
    (every element read once and written once) against the measured HBM copy
    bandwidth, with L2 cold (enough buffer sets rotate to exceed twice the L2) and
    hot (one set, which fits in L2).  Then the unfused chain the pages describe
    (PsaPackQkv -> Flash Attention 2 on V_lo and on V_hi -> PsaMergeAttn, and
    PsaExtractV) next to the fused psa_attention_fwd, and the unfused backward
    (inverse merge -> dQ and dK/dV kernels per V half -> inverse pack; the sum of
    the two halves' dQ and dK has no kernel of its own and is left out) next to
    psa_attention_bwd.  One JSON line per case."""
    import torch

    from vision_transformer_attention_psapackqkv_gb300 import binding as B
    from vision_transformer_attention_psapackqkv_gb300.inputs import PSA_WORKLOADS

    peaks, src = load_peaks()
    hbm = peaks["hbm_gbs"]
    w = PSA_WORKLOADS[WORKLOAD]
    # every case is replayed from a CUDA graph of `iters` calls (short kernels would
    # otherwise wait on the host's launches)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(w.seed)
    rnd = lambda *shape: torch.randn(shape, generator=gen, device="cuda").to(torch.bfloat16)
    BH, N, KD = w.BH, w.N, w.key_dim
    scale = 1.0 / math.sqrt(KD)

    def make_set():
        qkv = rnd(w.B, w.qkv_channels, w.H, w.W)
        dout = rnd(w.B, w.out_channels, w.H, w.W)
        st = {"qkv": qkv, "dout": dout, "packed": torch.empty((4, BH, N, KD), dtype=torch.bfloat16, device="cuda"),
              "out": torch.empty_like(dout), "v": torch.empty_like(dout), "dqkv": torch.empty_like(qkv),
              "lse": torch.empty((BH, N), dtype=torch.float32, device="cuda"),
              "lse2": torch.empty((BH, N), dtype=torch.float32, device="cuda"),
              "delta": torch.empty((BH, N), dtype=torch.float32, device="cuda")}
        st["o"] = torch.empty((2, BH, N, KD), dtype=torch.bfloat16, device="cuda")
        st["do"] = torch.empty((2, BH, N, KD), dtype=torch.bfloat16, device="cuda")
        st["dpacked"] = torch.empty((4, BH, N, KD), dtype=torch.bfloat16, device="cuda")
        st["dqk_hi"] = torch.empty((2, BH, N, KD), dtype=torch.bfloat16, device="cuda")
        st["ws"] = torch.empty(B.psa_attention_bwd_workspace_size(B.shape_of(qkv, w.num_heads, KD)),
                               dtype=torch.uint8, device="cuda")
        return st

    per_set = sum(t.numel() * t.element_size() for t in make_set().values())
    nsets = max(3, math.ceil(2 * 2 * 129e6 / per_set))
    sets = [make_set() for _ in range(nsets)]
    shape = B.shape_of(sets[0]["qkv"], w.num_heads, KD)
    e = 2
    qkv_b, half_b = w.B * w.qkv_channels * N * e, w.B * w.out_channels * N * e
    cases = [
        ("psa_pack_qkv", 2 * qkv_b, lambda s: B.psa_pack_qkv(s["qkv"], s["packed"], shape)),
        ("psa_unpack_qkv", 2 * qkv_b, lambda s: B.psa_unpack_qkv(s["packed"], s["dqkv"], shape)),
        ("psa_merge_attn", 2 * half_b, lambda s: B.psa_merge_attn(s["o"][0], s["o"][1], s["out"], shape)),
        ("psa_unmerge_attn", 2 * half_b, lambda s: B.psa_unmerge_attn(s["dout"], s["do"][0], s["do"][1], shape)),
        ("psa_extract_v", 2 * half_b, lambda s: B.psa_extract_v(s["qkv"], s["v"], shape)),
    ]
    lines = []
    iters = args.iters
    for name, nbytes, fn in cases:
        for l2 in ("cold", "hot"):
            use = sets if l2 == "cold" else sets[:1]
            with ClockSampler() as clk:
                sec = _time_graph(torch, lambda i: fn(use[i % len(use)]), iters, min(2 * len(use), iters))
            gbs = nbytes / sec / 1e9
            line = {"metric": "layout kernel GB/s (algorithmic bytes)", "workload": WORKLOAD,
                    "kernel": name, "l2": l2, "value": gbs, "unit": "GB/s", "us": sec * 1e6,
                    "bytes": nbytes, "hbm": {"peak": hbm, "frac": gbs / hbm, "peak_source": src},
                    "clocks": clk.summary()}
            lines.append(line)
            print(json.dumps(line), flush=True)

    def fwd_chain(s):
        B.psa_pack_qkv(s["qkv"], s["packed"], shape)
        q, k, vlo, vhi = s["packed"]
        B.flash_attn2_fwd(q, k, vlo, s["o"][0], s["lse"], scale)
        B.flash_attn2_fwd(q, k, vhi, s["o"][1], s["lse2"], scale)
        B.psa_merge_attn(s["o"][0], s["o"][1], s["out"], shape)
        B.psa_extract_v(s["qkv"], s["v"], shape)

    def fwd_fused(s):
        B.psa_attention_fwd(s["qkv"], s["out"], s["lse"], s["v"], shape, scale)

    def bwd_chain(s):
        q, k, vlo, vhi = s["packed"]
        B.psa_unmerge_attn(s["dout"], s["do"][0], s["do"][1], shape)
        dq, dk, dvlo, dvhi = s["dpacked"]
        B.flash_attn2_bwd_dq(q, k, vlo, s["o"][0], s["do"][0], s["lse"], s["delta"], dq, scale)
        B.flash_attn2_bwd_dkdv(q, k, vlo, s["do"][0], s["lse"], s["delta"], dk, dvlo, scale)
        B.flash_attn2_bwd_dq(q, k, vhi, s["o"][1], s["do"][1], s["lse"], s["delta"], s["dqk_hi"][0], scale)
        B.flash_attn2_bwd_dkdv(q, k, vhi, s["do"][1], s["lse"], s["delta"], s["dqk_hi"][1], dvhi, scale)
        B.psa_unpack_qkv(s["dpacked"], s["dqkv"], shape)

    def bwd_fused(s):
        B.psa_attention_bwd(s["qkv"], s["out"], s["dout"], s["lse"], None, s["dqkv"], s["ws"], shape, scale)

    # the QKV 1x1 convolution of this block (c = nh*2*KD input channels -> nh*4*KD)
    gw = torch.Generator(device="cuda")
    gw.manual_seed(w.seed + 100)
    cin, cout = w.out_channels, w.qkv_channels
    conv_sets = [{"x": torch.randn((w.B, cin, w.H, w.W), generator=gw, device="cuda").to(torch.bfloat16),
                  "qkv": s["qkv"], "out": s["out"]} for s in sets]
    wt = (torch.randn((cout, cin), generator=gw, device="cuda") / math.sqrt(cin)).to(torch.bfloat16)
    bias = torch.randn((cout,), generator=gw, device="cuda") * 0.5
    conv_flops = 2.0 * w.B * cout * cin * N
    conv_bytes = (w.B * cin * N + cout * cin + w.B * cout * N) * 2 + cout * 4
    for name, fn, flops, nbytes in (
            ("psa_qkv_conv", lambda c: B.psa_qkv_conv(c["x"], wt, bias, c["qkv"]), conv_flops, conv_bytes),
            ("psa_qkv_conv -> psa_attention_fwd",
             lambda c: (B.psa_qkv_conv(c["x"], wt, bias, c["qkv"]),
                        B.psa_attention_fwd(c["qkv"], c["out"], None, None, shape, scale)),
             conv_flops + work_model(w)[0]["fwd"]["flops"], None)):
        with ClockSampler() as clk:
            sec = _time_graph(torch, lambda i: fn(conv_sets[i % nsets]), iters, min(2 * nsets, iters))
        line = {"metric": "QKV 1x1 conv (tensor cores)", "workload": WORKLOAD, "path": name,
                "config": {"B": w.B, "cin": cin, "cout": cout, "H": w.H, "W": w.W},
                "us": sec * 1e6, "tflops": flops / sec / 1e12, "l2": "cold", "clocks": clk.summary()}
        if nbytes:
            line["hbm"] = {"algorithmic_bytes": nbytes, "gbs": nbytes / sec / 1e9,
                           "frac": nbytes / sec / 1e9 / hbm, "peak_source": src}
            line["tensor"] = {"frac": flops / sec / 1e12 / peaks["bf16_tflops"], "peak_source": src}
        lines.append(line)
        print(json.dumps(line), flush=True)

    for st in sets:
        fwd_chain(st)
    kmodel, _ = work_model(w)
    for name, fn, nk, part in (("unfused forward chain", fwd_chain, 5, "fwd"),
                               ("psa_attention_fwd", fwd_fused, 1, "fwd"),
                               ("unfused backward chain (without the dQ / dK half sums)", bwd_chain, 6, "bwd"),
                               ("psa_attention_bwd", bwd_fused, 1, "bwd")):
        with ClockSampler() as clk:
            sec = _time_graph(torch, lambda i: fn(sets[i % nsets]), iters, min(2 * nsets, iters))
        km = kmodel[part]
        line = {"metric": "PSA attention step part, unfused chain vs fused", "workload": WORKLOAD,
                "path": name, "launches": nk, "us": sec * 1e6, "l2": "cold",
                "tflops": km["flops"] / sec / 1e12,
                "hbm": {"algorithmic_bytes": km["bytes"], "gbs": km["bytes"] / sec / 1e9,
                        "frac": km["bytes"] / sec / 1e9 / hbm, "peak_source": src},
                "clocks": clk.summary()}
        lines.append(line)
        print(json.dumps(line), flush=True)
    if B.psa_get_last_device_error() != 0:
        raise RuntimeError("device error in the layout bench")
    return lines


def run_reference(args):
    from vision_transformer_attention_psapackqkv_gb300.inputs import PSA_WORKLOADS

    w = PSA_WORKLOADS[WORKLOAD]
    scale = 1.0 / math.sqrt(w.key_dim)
    import oracle
    from vision_transformer_attention_psapackqkv_gb300.inputs import storage_to_f64, workload_inputs

    oracle.build()
    ins = workload_inputs(w)
    threads = oracle.default_threads()
    nb = 2  # batch items per step: 8 heads, 800 tokens
    q = storage_to_f64(ins["qkv"][:nb], w.dtype)
    d = storage_to_f64(ins["dout"][:nb], w.dtype)

    def step():
        oracle.psa_fwd(q, w.num_heads, w.key_dim, scale, nthreads=threads)
        oracle.psa_bwd(q, d, w.num_heads, w.key_dim, scale, nthreads=threads)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    t = time.perf_counter() - t0
    value = nb * w.N * args.steps / t
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) QKV and dOut)",
        "config": {"workload": WORKLOAD, "B": w.B, "num_heads": w.num_heads, "key_dim": w.key_dim,
                   "H": w.H, "W": w.W, "N": w.N, "step_sample_batches": nb},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"{nb} of {w.B} batch items per step ({nb * w.num_heads} heads)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--split-bwd", action="store_true")
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--layout", action="store_true",
                    help="time the data-movement kernels, the QKV conv and the unfused chain instead")
    ap.add_argument("--iters", type=int, default=200, help="with --layout: timed calls per case")
    ap.add_argument("--case", default=None,
                    help="with --sweep: run only the case of this name (e.g. fa2_bh64_n4096_d64)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if args.sweep:
        if rank == 0:
            run_sweep(args)
        return
    if args.layout:
        if rank == 0:
            run_layout(args)
        return
    line = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
