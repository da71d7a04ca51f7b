"""Benchmark of the weight-only quantized linear layer on GB300.

One step = one pass of the decode sweep: bits {5,6,7} x N {5120,17408} x
M {1,4,16}, K = 5120, group 128 (18 GEMMs, each on its own copy of the packed
weights, so a step streams ~0.78 GB of distinct weights: inputs larger than
L2). The value is whole-job decode throughput in GB/s of packed weight bytes.
The other rows (prefill sweep, W4A8, 8-bit lm_head, embedding gather, the
64-layer mixed-bit stack) are timed separately and reported under "extras",
each against its roofline.

    python bench.py [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs the same workload on its own GPU (replicas; the
layer needs no exchange between GPUs); the step time is the maximum over
ranks and the value sums the bytes of all ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode weight-stream GB/s (M≤16) and prefill TFLOPS (M≥4096), % of GB300 roofline"
K_DIM = 5120
DECODE_BITS = (5, 6, 7)
DECODE_N = (5120, 17408)
DECODE_M = (1, 4, 16)
WORKLOAD = ("decode sweep: bits {5,6,7} x N {5120,17408} x M {1,4,16}, K=5120, group=128, "
            "x bf16 N(0,1), codes uniform, scales 0.01|N(0,1)| with random sign")


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def _kernel_hash():
    h = hashlib.sha256()
    for f in ("decode2.cu", "wq_unpack.cuh", "wq_device.cuh", "wq_cluster.cuh"):
        h.update(open(os.path.join(ROOT, "weight_only_int2_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def _traffic_record():
    """DRAM bytes per launch of the decode kernel from a committed ncu summary,
    valid only while the kernel source is unchanged."""
    p = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    if d.get("kernel_hash") != _kernel_hash():
        return None
    return d


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- our arm

def _make_case_inputs(wq, torch, bits, N, M, seed):
    import wq_inputs as I

    codes = torch.from_numpy(I.make_codes(N, K_DIM, bits, seed)).cuda()
    s = I.make_scales(N, K_DIM // 128, seed + 1)
    s_dev = torch.from_numpy(s.view(np.int16)).view(torch.bfloat16).cuda()
    packed, s_dev = wq.wna16_repack(codes, s_dev, bits)
    del codes
    x = I.make_x(M, K_DIM, seed + 2)
    x_host = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory()
    return dict(bits=bits, N=N, M=M, packed=packed, scales=s_dev, x=x_host.cuda(), x_host=x_host,
                y=torch.empty((M, N), dtype=torch.bfloat16, device="cuda"),
                y_host=torch.empty((M, N), dtype=torch.bfloat16).pin_memory(),
                ws=torch.zeros(max(1, wq.wna16_workspace_bytes(M, N, K_DIM, bits)), dtype=torch.uint8,
                               device="cuda"),
                bytes=N * wq.packed_words_per_row(K_DIM, bits) * 4)


def _max_over_ranks(v: float, dist, device) -> float:
    """The maximum of v over all ranks (v itself without a process group)."""
    if dist is None:
        return float(v)
    import torch

    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _aggregate(step_bytes: float, ms_local: float, world: int, dist, device):
    """Whole-job throughput of replicas: every rank moves step_bytes per step;
    the job's step time is the slowest rank's. Returns (ms, GB/s)."""
    ms = _max_over_ranks(ms_local, dist, device)
    return ms, world * step_bytes / (ms * 1e-3) / 1e9


def run_ours(args, rank, world, dist):
    import torch

    import weight_only_int2_gb300 as wq
    from weight_only_int2_gb300 import _build

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    _build.build()
    wq.load()

    cases = []
    seed = 2000
    for bits in DECODE_BITS:
        for N in DECODE_N:
            for M in DECODE_M:
                if args.case is None or args.case == (bits, N, M):
                    cases.append(_make_case_inputs(wq, torch, bits, N, M, seed))
                seed += 10
    step_bytes = sum(c["bytes"] for c in cases)
    stream = torch.cuda.Stream()

    # one step's activations and outputs, each in one contiguous buffer on the
    # host (pinned) and on the device; every case works on its slice, so the
    # end-to-end step moves its inputs and its results in one copy each
    xs_numel = [c["x_host"].numel() for c in cases]
    ys_numel = [c["M"] * c["N"] for c in cases]
    x_host_all = torch.empty(sum(xs_numel), dtype=torch.bfloat16).pin_memory()
    y_host_all = torch.empty(sum(ys_numel), dtype=torch.bfloat16).pin_memory()
    x_all = torch.empty(sum(xs_numel), dtype=torch.bfloat16, device="cuda")
    y_all = torch.empty(sum(ys_numel), dtype=torch.bfloat16, device="cuda")
    xo = yo = 0
    for c, nx, ny in zip(cases, xs_numel, ys_numel):
        x_host_all[xo:xo + nx].copy_(c["x_host"].reshape(-1))
        c["x_host"] = x_host_all[xo:xo + nx].view(c["M"], K_DIM)
        c["x"] = x_all[xo:xo + nx].view(c["M"], K_DIM)
        c["y"] = y_all[yo:yo + ny].view(c["M"], c["N"])
        c["y_host"] = y_host_all[yo:yo + ny].view(c["M"], c["N"])
        xo += nx
        yo += ny
    x_all.copy_(x_host_all)

    def launch(c):
        wq.wna16_gemm(c["x"], c["packed"], c["scales"], c["N"], K_DIM, c["bits"], y=c["y"], ws=c["ws"])

    # one step as a CUDA graph (the timed region replays it back to back)
    with torch.cuda.stream(stream):
        for c in cases:  # first call sets up kernels outside the capture
            launch(c)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for c in cases:
            launch(c)
    # the same step with an event between launches, for the per-case table
    # (event nodes add their own gaps, so these durations are upper bounds)
    evs = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(len(cases) + 1)]
    graph_ev = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_ev, stream=stream):
        evs[0].record(stream)
        for i, c in enumerate(cases):
            launch(c)
            evs[i + 1].record(stream)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
        graph_ev.replay()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()

    with ClockSampler(local) as clk:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        with torch.cuda.stream(stream):
            t0.record(stream)
            for _ in range(args.steps):
                graph.replay()
            t1.record(stream)
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        # keep the GPU under the same load (untimed) until the clock sampler
        # has covered at least a second
        t_load = time.perf_counter()
        while time.perf_counter() - t_load < max(0.0, 1.0 - t0.elapsed_time(t1) * 1e-3):
            with torch.cuda.stream(stream):
                for _ in range(20):
                    graph.replay()
            torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        graph_ev.replay()
    torch.cuda.synchronize()
    per_launch = [[evs[i].elapsed_time(evs[i + 1])] for i in range(len(cases))]
    ms_per_step, value = _aggregate(step_bytes, t0.elapsed_time(t1) / args.steps, world, dist, "cuda")

    case_rows = []
    for i, c in enumerate(cases):
        us = 1000 * float(np.mean(per_launch[i]))
        case_rows.append({"bits": c["bits"], "N": c["N"], "M": c["M"], "us": round(us, 3),
                          "GBps": round(c["bytes"] / (us * 1e-6) / 1e9, 1)})

    # ---- end to end through the public API: pinned host x in, host y out
    e2e_ms = []
    h2d = x_host_all.numel() * 2
    d2h = y_host_all.numel() * 2
    with torch.cuda.stream(stream):
        for it in range(args.warmup + args.steps):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            x_all.copy_(x_host_all, non_blocking=True)
            for c in cases:
                launch(c)
            y_host_all.copy_(y_all, non_blocking=True)
            b.record(stream)
            stream.synchronize()
            if it >= args.warmup:
                e2e_ms.append(a.elapsed_time(b))
    _, e2e_value = _aggregate(step_bytes, float(np.mean(e2e_ms)), world, dist, "cuda")

    # the same step (copies and the 18 public calls) captured once as a CUDA
    # graph, as a serving loop would replay it: separates the copies' cost
    # from the host's per-call work in the eager figure above
    g_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_e2e, stream=stream):
        x_all.copy_(x_host_all, non_blocking=True)
        for c in cases:
            launch(c)
        y_host_all.copy_(y_all, non_blocking=True)
    e2e_graph_ms = []
    with torch.cuda.stream(stream):
        for it in range(args.warmup + args.steps):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g_e2e.replay()
            b.record(stream)
            stream.synchronize()
            if it >= args.warmup:
                e2e_graph_ms.append(a.elapsed_time(b))
    _, e2e_graph_value = _aggregate(step_bytes, float(np.mean(e2e_graph_ms)), world, dist, "cuda")

    # ---- the other rows (separate timed regions; reported, not the headline)
    extras = None
    if not args.no_prefill:
        extras = _time_extras(wq, torch, stream)

    hbm, bf16, bf16_sus, src = _peaks()
    # average launch duration = step time / launches (back-to-back graph
    # launches; the short gaps between kernels are counted against us)
    achieved = step_bytes / (ms_per_step * 1e-3) / 1e9
    tr = _traffic_record()
    traffic = None
    if tr is not None:
        # DRAM bytes of one launch of the b=6, N=17408, M=1 case, scaled to
        # the step's mean launch by packed bytes (traffic grows with them)
        ref_bytes = 17408 * 960 * 4
        traffic = round(tr["dram_bytes_per_launch"] * (step_bytes / len(cases)) / ref_bytes)
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4), "traffic": traffic,
                "kernel": "decode2_kernel (CTA pairs over K halves, TMA weight ring, warp MMA)",
                "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)" if src == "measured" else "fallback 6.8 TB/s",
                "algorithmic_bytes_per_launch": "N*K*bits/8 packed weight bytes",
                "duration": "CUDA events around back-to-back graph replays of the step, divided by launches"}
    return dict(value=value, ms_per_step=ms_per_step, cases=case_rows, e2e=dict(
        value=round(e2e_value, 1), unit="GB/s", h2d_bytes_per_step=h2d, d2h_bytes_per_step=d2h,
        method="eager public calls per step (pinned x in, y out, one copy each), synchronized",
        graph_value=round(e2e_graph_value, 1)),
        extras=extras, roofline=roofline, clocks=clk.summary(), launches=len(cases) * args.steps,
        bf16_peak=(bf16, bf16_sus, src))


def _event_ms(torch, stream, fn, reps):
    """Average device time of fn() over reps calls on stream (CUDA events)."""
    with torch.cuda.stream(stream):
        fn()
        stream.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        stream.synchronize()
    return a.elapsed_time(b) / reps


def _graph_ms(torch, stream, fn, reps):
    """Average device time of one replay of a CUDA graph that captured fn()."""
    with torch.cuda.stream(stream):
        fn()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        for _ in range(2):
            g.replay()
        stream.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            g.replay()
        b.record(stream)
        stream.synchronize()
    return a.elapsed_time(b) / reps


def _rand_layer(wq, torch, N, K, bits, gen):
    """Random codes (uniform) and scales (0.01 |N(0,1)|, random sign) on the
    device, repacked; for timing only (parity runs on the seeded host inputs)."""
    codes = torch.randint(0, 1 << bits, (N, K), dtype=torch.uint8, device="cuda", generator=gen)
    sc = torch.randn(N, K // 128, device="cuda", generator=gen) * 0.01
    packed, s = wq.wna16_repack(codes, sc.to(torch.bfloat16), bits)
    del codes
    return packed, s


L2_BYTES = 129 * 2**20
ROTATE_BYTES = 3 * L2_BYTES  # a timed rotation reads at least this much distinct data


def _sms(torch) -> int:
    return torch.cuda.get_device_properties(0).multi_processor_count


def _copies(nbytes: float) -> int:
    """Distinct copies of an input of nbytes that a timed rotation cycles
    through, so that each call reads its data from HBM, not from L2."""
    return max(1, int(-(-ROTATE_BYTES // max(1, int(nbytes)))))


def _rotation_ms(torch, stream, fns, reps):
    """Average device time of one call, over a CUDA graph that makes the calls
    fns[0..R-1] in turn (each on its own copy of the data), replayed reps
    times."""
    def step():
        for f in fns:
            f()
    return _graph_ms(torch, stream, step, reps) / len(fns)


def _mma_peaks(wq, torch, stream):
    """The warp-level tensor-core peaks (mma.sync) of this GPU, int8
    (m16n8k32, int32 accumulate) and bf16 (m16n8k16, fp32 accumulate), from
    the library's probe; each launch's checksums are verified exactly."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    blocks, iters = 4 * sms, 20000
    res = {}
    for kind, k, name in ((0, 32, "int8_mma_sync_tops"), (1, 16, "bf16_mma_sync_tflops")):
        out = torch.empty(blocks * 256, dtype=torch.int32, device="cuda")
        ms = _event_ms(torch, stream, lambda: wq.debug_mma_peak(kind, iters, blocks, out), 5)
        if not bool((out == 8 * 4 * k * iters).all()):
            raise RuntimeError(f"mma.sync probe kind {kind}: wrong checksums")
        ops = blocks * 8 * 8 * iters * 2 * 16 * 8 * k
        res[name] = round(ops / (ms * 1e-3) / 1e12, 1)
    return res


def _time_extras(wq, torch, stream, only=None):
    """The other rows of the scope table, each against its roofline: prefill
    sweep, the decode configuration's M = 64 cases, W4A8, the 8-bit lm_head,
    the embedding gather and the 64-layer mixed-bit stack (timed as one CUDA
    graph), the mma.sync peaks and the cost of the no-allocation entry point.
    Every row reads its weights from HBM: a row whose data fits L2 cycles
    through distinct copies of at least 3x L2; the others are larger than L2.
    Calls are timed in groups of at least 20. `only` names one row to time
    alone (profiling)."""

    def want(name):
        return only is None or only == name

    hbm, bf16, _, src = _peaks()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(1234)
    K = 5120
    out = {"peak_source": src}

    def gbs(nbytes, ms):
        v = nbytes / (ms * 1e-3) / 1e9
        return {"ms": round(ms, 4), "GBps": round(v, 1), "frac": round(v / hbm, 4)}

    def tfl(flops, ms):
        v = flops / (ms * 1e-3) / 1e12
        return {"ms": round(ms, 4), "TFLOPS": round(v, 1), "frac": round(v / bf16, 4)}

    N = 17408
    if want("prefill"):
        # prefill sweep: M in {2048, 8192} x bits in {5,6,7,8}, N = 17408
        rows = []
        for bits in (5, 6, 7, 8):
            packed, s = _rand_layer(wq, torch, N, K, bits, gen)
            for M in (2048, 8192):
                x = torch.randn(M, K, device="cuda", generator=gen).to(torch.bfloat16)
                y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
                ms = _event_ms(torch, stream, lambda: wq.wna16_gemm(x, packed, s, N, K, bits, y=y), 20)
                rows.append(dict(bits=bits, M=M, **tfl(2.0 * M * N * K, ms)))
            del packed, s
        out["prefill"] = rows

    if want("decode_m64"):
        # the decode configuration's M = 64 cases (outside the M <= 16 headline):
        # (streaming or tensor-core kernel by shape), on packed-weight bytes
        rows = []
        for bits in (5, 6, 7):
            for Nd in (5120, 17408):
                nb = Nd * K * bits / 8
                layers = [_rand_layer(wq, torch, Nd, K, bits, gen) for _ in range(_copies(nb))]
                x = torch.randn(64, K, device="cuda", generator=gen).to(torch.bfloat16)
                y = torch.empty(64, Nd, dtype=torch.bfloat16, device="cuda")
                ws = torch.zeros(max(1, wq.wna16_workspace_bytes(64, Nd, K, bits)), dtype=torch.uint8, device="cuda")
                fns = [lambda pk=pk, sc=sc: wq.wna16_gemm(x, pk, sc, Nd, K, bits, y=y, ws=ws) for pk, sc in layers]
                ms = _rotation_ms(torch, stream, fns, 20)
                rows.append(dict(bits=bits, N=Nd, M=64, copies=len(layers), **gbs(nb, ms)))
                del layers
        out["decode_m64"] = rows

    if want("w4a8"):
        # W4A8 (int8 activations quantized per token inside the call), against
        # the measured bf16 peak (the exact path multiplies on the bf16 tensor
        # cores) and beside it the measured int8 mma.sync peak
        peaks = _mma_peaks(wq, torch, stream)
        out["mma_sync_peaks"] = peaks
        nb = N * K * 4 / 8
        layers = [_rand_layer(wq, torch, N, K, 4, gen) for _ in range(_copies(nb))]
        packed, s = layers[0]
        rows = []
        for M in (1, 512, 8192):
            x = torch.randn(M, K, device="cuda", generator=gen).to(torch.bfloat16)
            y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
            if M == 1:
                fns = [lambda pk=pk, sc=sc: wq.w4a8_gemm(x, pk, sc, N, K, y=y) for pk, sc in layers]
                ms = _rotation_ms(torch, stream, fns, 20)
                rows.append(dict(M=M, copies=len(layers), **gbs(nb, ms)))
            else:
                ms = _event_ms(torch, stream, lambda: wq.w4a8_gemm(x, packed, s, N, K, y=y), 20)
                r = dict(M=M, **tfl(2.0 * M * N * K, ms))
                r["frac_int8_mma_sync"] = round(r["TFLOPS"] / peaks["int8_mma_sync_tops"], 4)
                rows.append(r)
        out["w4a8"] = rows
        del layers, packed, s

    if want("lm_head") or want("gather"):
        # lm_head: 8-bit, N = 248320 (1.27 GB packed), and the gather from the same table
        V = 248320
        packed, s = _rand_layer(wq, torch, V, K, 8, gen)
        if want("lm_head"):
            rows = []
            for M in (1, 4096):
                x = torch.randn(M, K, device="cuda", generator=gen).to(torch.bfloat16)
                y = torch.empty(M, V, dtype=torch.bfloat16, device="cuda")
                if M == 1:
                    ms = _graph_ms(torch, stream, lambda: wq.wna16_gemm(x, packed, s, V, K, 8, y=y), 20)
                    rows.append(dict(M=M, **gbs(V * K, ms)))
                else:
                    ms = _event_ms(torch, stream, lambda: wq.wna16_gemm(x, packed, s, V, K, 8, y=y), 20)
                    rows.append(dict(M=M, **tfl(2.0 * M * V * K, ms)))
            out["lm_head"] = rows
        if want("gather"):
            # distinct id sets and output buffers in turn (at least 3x L2 of
            # rows read and written), so that rows and outputs go through HBM
            T = 4096
            moved = T * (K + 2 * K // 128 + 2 * K + 4)  # packed row + scales in, bf16 row out, id
            R = _copies(moved)
            sets = [(torch.randint(0, V, (T,), dtype=torch.int32, device="cuda", generator=gen),
                     torch.empty(T, K, dtype=torch.bfloat16, device="cuda")) for _ in range(R)]
            fns = [lambda ids=ids, o=o: wq.qembed_gather(ids, packed, s, V, K, 8, out=o) for ids, o in sets]
            ms = _rotation_ms(torch, stream, fns, 20)
            # DRAM sees the reads within the launch; the written rows land in
            # L2 and reach HBM later (an ncu dram__bytes check)
            read = T * (K + 2 * K // 128 + 4)
            g = gbs(moved, ms)
            g["read_GBps"] = round(read / (ms * 1e-3) / 1e9, 1)
            g["read_frac"] = round(g["read_GBps"] / hbm, 4)
            out["gather"] = dict(T=T, bytes_moved=moved, bytes_read=read, id_sets=R, **g)
            del sets
        del packed, s

    if want("stack"):
        # 64-layer stack: layers 0-9 and 54-63 at 7 bits, 10-53 alternating 5 / 6
        layers = []
        for li in range(64):
            bits = 7 if (li < 10 or li >= 54) else (5 if (li - 10) % 2 == 0 else 6)
            packed, s = _rand_layer(wq, torch, N, K, bits, gen)
            layers.append((bits, packed, s))
        stack_bytes = sum(N * K * b / 8 for b, _, _ in layers)
        rows = []
        for M in (1, 4096):
            x = torch.randn(M, K, device="cuda", generator=gen).to(torch.bfloat16)
            ys = [torch.empty(M, N, dtype=torch.bfloat16, device="cuda") for _ in range(2)]

            def stack():
                for li, (b, pk, sc) in enumerate(layers):
                    wq.wna16_gemm(x, pk, sc, N, K, b, y=ys[li & 1])

            ms = _graph_ms(torch, stream, stack, 20)
            if M == 1:
                rows.append(dict(M=M, layers=64, packed_bytes=int(stack_bytes), **gbs(stack_bytes, ms)))
            else:
                rows.append(dict(M=M, layers=64, **tfl(2.0 * M * N * K * 64, ms)))
        out["stack"] = rows
        del layers

    if want("noalloc"):
        # the no-allocation entry point against the workspace one on a
        # split-K shape (16 tokens, K = 14336: the pair kernel's K half does
        # not fit): the difference is the scratch clear it queues per call
        Mn, Nn, Kn, bn = 16, 17408, 14336, 6
        nb = Nn * Kn * bn / 8
        layers = [_rand_layer(wq, torch, Nn, Kn, bn, gen) for _ in range(_copies(nb))]
        x = torch.randn(Mn, Kn, device="cuda", generator=gen).to(torch.bfloat16)
        y = torch.empty(Mn, Nn, dtype=torch.bfloat16, device="cuda")
        ws = torch.zeros(max(1, wq.wna16_workspace_bytes(Mn, Nn, Kn, bn)), dtype=torch.uint8, device="cuda")
        f_ws = [lambda pk=pk, sc=sc: wq.wna16_gemm(x, pk, sc, Nn, Kn, bn, y=y, ws=ws) for pk, sc in layers]
        f_na = [lambda pk=pk, sc=sc: wq.wna16_gemm_noalloc(x, pk, sc, Nn, Kn, bn, y=y) for pk, sc in layers]
        ms_ws = _rotation_ms(torch, stream, f_ws, 20)
        ms_na = _rotation_ms(torch, stream, f_na, 20)
        out["noalloc"] = dict(M=Mn, N=Nn, K=Kn, bits=bn, route=wq.debug_route(Mn, Nn, Kn, bn, _sms(torch)),
                              scratch_bytes=wq.wna16_workspace_bytes(Mn, Nn, Kn, bn),
                              ms_workspace=round(ms_ws, 4), ms_noalloc=round(ms_na, 4),
                              copies=len(layers))
        del layers
    torch.cuda.empty_cache()
    return out


def run_only(args):
    """One group of the other rows, timed alone (profiling): no decode sweep."""
    import torch

    import weight_only_int2_gb300 as wq
    from weight_only_int2_gb300 import _build

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    _build.build()
    wq.load()
    stream = torch.cuda.Stream()
    out = _time_extras(wq, torch, stream, only=args.only)
    wq.check_status()
    print(json.dumps({"only": args.only, **out}), flush=True)


def run_prefill_case(args):
    """One prefill shape on its own (bits, M; N = 17408, K = 5120): a small,
    self-contained workload for profiling the tensor-core kernel."""
    import torch

    import weight_only_int2_gb300 as wq
    from weight_only_int2_gb300 import _build

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    _build.build()
    wq.load()
    bits, M = args.prefill_case
    N, K = 17408, K_DIM
    gen = torch.Generator(device="cuda")
    gen.manual_seed(4321)
    packed, s = _rand_layer(wq, torch, N, K, bits, gen)
    x = torch.randn(M, K, device="cuda", generator=gen).to(torch.bfloat16)
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            wq.wna16_gemm(x, packed, s, N, K, bits, y=y)
    ms = _event_ms(torch, stream, lambda: wq.wna16_gemm(x, packed, s, N, K, bits, y=y), args.steps)
    wq.check_status()
    _, bf16, _, src = _peaks()
    tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
    print(json.dumps({"prefill_case": {"bits": bits, "M": M, "N": N, "K": K}, "ms": round(ms, 4),
                      "TFLOPS": round(tf, 1), "frac": round(tf / bf16, 4), "peak_source": src}), flush=True)


# ----------------------------------------------------------------------------- oracle arms

def _cpu_time_oracle(budget_s: float):
    """Times the CPU oracle (as it stands) on a bounded sample of the decode
    sweep: for each (bits, N) pair a row subset of W with all M tokens of the
    largest M. Returns (GB/s of packed weight bytes, cores used, sample text)."""
    import oracle as O
    import wq_inputs as I

    rows = 256
    done_bytes = 0
    t_wall0 = time.perf_counter()
    t_cpu0 = time.process_time()
    n = 0
    for bits in DECODE_BITS:
        for N in DECODE_N:
            q = I.make_codes(rows, K_DIM, bits, 3000 + bits)
            s = I.make_scales(rows, K_DIM // 128, 3001 + bits)
            p = O.pack(q, bits)                     # input preparation, untimed below
            x = I.make_x(16, K_DIM, 3002)
            t0 = time.perf_counter()
            codes = O.unpack(p, K_DIM, bits)
            for M in DECODE_M:
                O.wna16_ref(x[:M], codes, s, bits)
            done_bytes += rows * O.packed_words_per_row(K_DIM, bits) * 4 * len(DECODE_M)
            n += 1
            if time.perf_counter() - t_wall0 > budget_s:
                break
        if time.perf_counter() - t_wall0 > budget_s:
            break
    wall = time.perf_counter() - t_wall0
    cpu = time.process_time() - t_cpu0
    gbs = done_bytes / wall / 1e9
    sample = (f"{n} of 6 (bits, N) pairs, {rows} rows of W each, M in {{1,4,16}}: oracle unpack "
              f"(per-bit loops) + float64 dequant + matmul; {done_bytes} packed bytes")
    return gbs, max(1, round(cpu / wall)), sample


def run_reference(args, rank, world):
    if rank != 0:
        return
    hbm, _, _, _ = _peaks()
    vals = []
    sample = ""
    cores = 1
    for it in range(args.warmup + args.steps):
        gbs, cores, sample = _cpu_time_oracle(budget_s=8.0)
        if it >= args.warmup:
            vals.append(gbs)
    v = float(np.mean(vals))
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "arm": "CPU oracle (numpy float64) on host cores"},
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-prefill", "--no-extras", dest="no_prefill", action="store_true",
                    help="skip the other rows (prefill, W4A8, lm_head, gather, stack)")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--only", choices=["prefill", "decode_m64", "w4a8", "lm_head", "gather", "stack", "noalloc"],
                    default=None, help="time one group of the other rows alone, without the decode sweep")
    ap.add_argument("--prefill-case", type=str, default=None,
                    help="time one prefill shape 'bits,M' (N=17408, K=5120) alone (profiling)")
    ap.add_argument("--case", type=str, default=None,
                    help="restrict the decode sweep to one case 'bits,N,M' (profiling)")
    args = ap.parse_args()
    if args.case is not None:
        args.case = tuple(int(v) for v in args.case.split(","))
        if (len(args.case) != 3 or args.case[0] not in DECODE_BITS or args.case[1] not in DECODE_N
                or args.case[2] not in DECODE_M):
            ap.error(f"--case must name a case of the sweep: bits in {DECODE_BITS}, N in {DECODE_N}, "
                     f"M in {DECODE_M}")
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.only is not None:
        run_only(args)
        return
    if args.prefill_case is not None:
        args.prefill_case = tuple(int(v) for v in args.prefill_case.split(","))
        if len(args.prefill_case) != 2 or not 2 <= args.prefill_case[0] <= 8 or args.prefill_case[1] < 1:
            ap.error("--prefill-case wants 'bits,M' with bits in 2..8")
        run_prefill_case(args)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None

    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    if world > 1:
        import torch
        import torch.distributed as tdist

        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        tdist.init_process_group("nccl")
        dist = tdist
    r = run_ours(args, rank, world, dist)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        gbs, cores, sample = _cpu_time_oracle(budget_s=args.cpu_budget)
        cpu = {"value": round(gbs, 6), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample}
    if rank == 0:
        line = {"metric": METRIC, "value": round(r["value"], 1), "unit": "GB/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(r["ms_per_step"], 4),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic",
                "config": {"workload": WORKLOAD, "parallelism": f"replicas x{world}",
                           "l2": "inputs larger than L2: each step reads 0.78 GB of distinct packed weights",
                           "timing": "CUDA events around K back-to-back replays of a CUDA graph of one step (18 launches); the per-case table replays a second graph with events between launches"},
                "roofline": r["roofline"], "cpu_baseline": cpu, "e2e": r["e2e"],
                "gpu_launches": r["launches"], "clocks": r["clocks"], "extras": r["extras"],
                "cases": r["cases"]}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
