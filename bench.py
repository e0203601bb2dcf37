"""Benchmark of the structured-sparse GEMM path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One JSON line on rank 0. A step is one sparse GEMM Y = W_sparse . X over the
workload's activation batch, with the 2:4-compressed weight resident in HBM
(weights are pruned and compressed once; the per-step work is the GEMM). L2 is
flushed (a write of twice the device's L2, at least 256 MB) between timed steps;
each step is timed with CUDA events on the launching stream. The other hot-path rows (prune/compress, the
tile-wise prune, the TW/TVW gather GEMMs and the dense GEMM of the same kernel
family) are timed the same way and reported under "rows".

--impl reference times the CPU oracle (the test suite's reference
implementation) on this host's cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from structured_sparse_dnn_gb300 import inputs as I  # noqa: E402

METRIC = "effective TFLOP/s and % of 2:4-sparse tensor peak for sparse GEMM (1×GB300)"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "llm_ffn_e4m3"
FLUSH_BYTES = 256 << 20   # the least L2 flush; flush_bytes() takes twice the device's L2 if larger


def flush_bytes(dev) -> int:
    """Size of the buffer written between timed steps: twice the device's L2 (read from
    the device, not assumed), at least FLUSH_BYTES, rounded to 1 MB."""
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 0)
    return max(FLUSH_BYTES, (2 * l2 + (1 << 20) - 1) >> 20 << 20)


def peaks() -> dict:
    p = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            m = json.load(f)
        p.update({k: float(m[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained") if k in m})
        p["source"] = "measured"
    return p


def measured_traffic(workload: str):
    """DRAM bytes (read + write) per launch of the sparse GEMM on this workload from
    the committed ncu capture, if the kernel's sources (gemm.cu, ptx.cuh, common.cuh)
    are unchanged since; else None."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        tab = json.load(f)
    h = hashlib.sha256()
    for name in ("gemm.cu", "ptx.cuh", "common.cuh"):
        with open(os.path.join(ROOT, "structured_sparse_dnn_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    ent = tab.get(workload)
    if not ent or ent.get("kernel_src_sha256_16") != h.hexdigest()[:16]:
        return None
    return ent["dram_bytes_per_launch"]


def tensor_peak_effective(dt: str, pk: dict, sustained: bool = False) -> float:
    """2:4-sparse tensor peak in effective (nonzero) TFLOP/s: the sparse core runs
    twice the dense-equivalent rate, i.e. one dense peak of nonzero MACs. e4m3 is
    twice bf16 (nominal ratio)."""
    base = pk["bf16_tflops_sustained"] if sustained else pk["bf16_tflops"]
    return base * (2.0 if dt == "e4m3" else 1.0)


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self) -> dict:
        sm, mx, reasons = [], 0.0, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in getattr(self, "lines", []):
            parts = [x.strip() for x in ln.split(",")]
            try:
                sm.append(float(parts[0]))
                mx = max(mx, float(parts[1]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def barrier_max(value: float, ws: int) -> float:
    """Max of a per-rank scalar over all ranks (identity on one rank)."""
    if ws == 1:
        return value
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_step_per_rank: float, steps: int, ms_total_max: float, ws: int) -> float:
    """Weak scaling: every rank runs its own steps; the job's throughput is all
    ranks' work over the slowest rank's time."""
    return ws * flops_per_step_per_rank * steps / (ms_total_max * 1e-3) / 1e12


def timed_steps(fn, steps: int, warmup: int, flush: torch.Tensor, stream) -> list[float]:
    """ms per step: warmup untimed calls, then `steps` calls each between an L2
    flush and a pair of CUDA events on `stream`."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    # an untimed lead-in step keeps every SM busy (and the clocks up) while the host
    # enqueues the first timed steps, so that no step's events include launch latency
    flush.fill_(1)
    fn()
    evs = []
    for _ in range(steps):
        flush.fill_(1)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def pct(xs, q: float) -> float:
    """q-th percentile (linear interpolation) of a list."""
    return float(np.percentile(np.asarray(xs, dtype=np.float64), q))


def graph_ms(body, n: int, side) -> float:
    """ms per call of `body`: n calls captured in one CUDA graph on stream `side`,
    replayed three times after three untimed replays, best of the three."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        body()                                         # first call outside capture (library set-up)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=side, capture_error_mode="thread_local"):
            for _ in range(n):
                body()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(side)
        with torch.cuda.stream(side):
            g.replay()
        b.record(side)
        torch.cuda.synchronize()
        best = min(best, a.elapsed_time(b))
    del g
    return best / n


def flushed_graph_ms(fn, flush: torch.Tensor, dev, n: int = 20) -> float:
    """ms per call of `fn` with L2 flushed before each: n (flush, call) pairs in one
    graph minus n flushes alone (launch latency amortised)."""
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    return graph_ms(lambda: (flush.fill_(1), fn()), n, side) - graph_ms(lambda: flush.fill_(1), n, side)


def headline_protocol(step, flush, stream, dev, eff_flops) -> dict:
    """The headline kernel under three timings: 50 eager launches each after an L2
    flush (CUDA events around each: p10 / median / p90); 50 launches replayed from one
    CUDA graph with L2 warm (back to back); and 50 (flush, launch) pairs in one graph
    minus 50 flushes alone (L2 flushed, launch overhead amortised)."""
    n = 50
    eager = timed_steps(step, n, 10, flush, stream)
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream(dev))

    warm = graph_ms(step, n, side)
    with_flush = graph_ms(lambda: (flush.fill_(1), step()), n, side)
    flush_only = graph_ms(lambda: flush.fill_(1), n, side)
    cold = with_flush - flush_only
    tf = lambda ms: round(eff_flops / (ms * 1e-3) / 1e12, 1)
    return {"eager_l2_flushed": {"launches": n, "p10_ms": round(pct(eager, 10), 5),
                                 "median_ms": round(statistics.median(eager), 5), "p90_ms": round(pct(eager, 90), 5),
                                 "median_TFLOP/s": tf(statistics.median(eager))},
            "graph_l2_warm": {"launches": n, "ms_per_launch": round(warm, 5), "TFLOP/s": tf(warm)},
            "graph_l2_flushed": {"launches": n, "ms_per_launch": round(cold, 5), "TFLOP/s": tf(cold),
                                 "note": f"50 (flush of {flush.numel() * 4 >> 20} MB, GEMM) pairs in one graph minus "
                                         "50 flushes alone"}}


def host_link_rates(X_dev, X_host, Y_dev, Y_host, stream) -> dict:
    """Copy-engine rates of the host link for this step's buffers (pinned host X in,
    device Y out), GB/s, best of three: the floor the end-to-end number runs against."""
    out = {}
    for key, dst, src in (("h2d_gbs", X_dev, X_host), ("d2h_gbs", Y_host, Y_dev)):
        nbytes = src.numel() * src.element_size()
        ts = []
        for _ in range(3):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            dst.copy_(src, non_blocking=True)
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b))
        out[key] = round(nbytes / min(ts) / 1e6, 1)
    return out


def mma_microbench(ss, stream) -> dict:
    """Dense and 2:4-sparse tcgen05.mma rates with operands on chip (one CTA per
    SM), in dense-equivalent TFLOP/s, for the instruction shapes the GEMMs use."""
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    out = {}
    for dname, dt, eb in (("bf16", ss.BF16, 2), ("e4m3", ss.E4M3, 1)):
        for n in (192, 256):
            for sparse in (False, True):
                iters = 16384
                ss.mma_rate(dt, sparse, n, iters)
                torch.cuda.synchronize()
                ts = []
                for _ in range(3):
                    a = torch.cuda.Event(enable_timing=True)
                    b = torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    ss.mma_rate(dt, sparse, n, iters)
                    b.record(stream)
                    b.synchronize()
                    ts.append(a.elapsed_time(b))
                flops = sms * iters * 2.0 * 128 * n * (128 // eb)
                out[f"{dname}_{'sparse' if sparse else 'dense'}_n{n}"] = round(flops / (min(ts) * 1e-3) / 1e12, 1)
        for sparse in (False, True):  # SM pairs, M = 256, N = 256 (the large GEMM tiles' instruction)
            iters = 16384
            ss.mma_rate_pair(dt, sparse, iters)
            torch.cuda.synchronize()
            ts = []
            for _ in range(3):
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                ss.mma_rate_pair(dt, sparse, iters)
                b.record(stream)
                b.synchronize()
                ts.append(a.elapsed_time(b))
            flops = (sms // 2) * iters * 2.0 * 256 * 256 * (128 // eb)
            out[f"{dname}_{'sparse' if sparse else 'dense'}_pair_n256"] = round(flops / (min(ts) * 1e-3) / 1e12, 1)
    assert ss.check_device_error() == 0, "device error flag set by the MMA microbenchmark"
    return out


def make_sp24(wl, dev, ss):
    d = wl.make()
    Wd = I.torch_view(d["W"], wl.dt).to(dev)
    Xd = I.torch_view(d["X"], wl.dt).to(dev)
    form = ss.sp24_prune_compress(Wd, canonical_meta=False)
    return d, Wd, Xd, form


def run_gpu(args) -> None:
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from structured_sparse_dnn_gb300 import build
    if rank == 0 or not os.path.exists(build.LIB):
        build.build()
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    from structured_sparse_dnn_gb300 import ssdnn as ss

    pk = peaks()
    wl = I.WORKLOADS[args.workload]
    stream = torch.cuda.current_stream(dev)
    fbytes = flush_bytes(dev)
    flush = torch.empty(fbytes // 4, dtype=torch.float32, device=dev)
    d, Wd, Xd, form = make_sp24(wl, dev, ss)
    M, K, N = wl.M, wl.K, wl.N
    Y = torch.empty((M, N), dtype=torch.bfloat16 if wl.out_dt == "bf16" else torch.float16, device=dev)
    alpha = d["alpha"]
    eff_flops = 2.0 * M * N * K * 0.5

    def step():
        ss.sp24_gemm(form, Xd, alpha=alpha, out=Y)

    # ---- timed region: K steps, barrier + synchronize on both sides, clocks sampled
    # (the sampler also covers about half a second of untimed warm-up steps so that
    # it sees the GPU under load; they repeat the timed pattern, an L2 flush then the
    # GEMM, so that the power and clock state they leave is the timed steps' own)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    with ClockSampler(local) as clk:
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < 0.5:
            for _ in range(20):
                flush.fill_(1)
                step()
            torch.cuda.synchronize()
        times = timed_steps(step, args.steps, 0, flush, stream)
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    assert ss.check_device_error() == 0, "device error flag set"
    ms_total = barrier_max(sum(times), ws)
    ms_step = ms_total / args.steps
    value = whole_job_tflops(eff_flops, args.steps, ms_total, ws)
    kernel_ms = statistics.mean(times)
    achieved = eff_flops / (kernel_ms * 1e-3) / 1e12
    peak_eff = tensor_peak_effective(wl.dt, pk)

    # ---- end to end through the public call with host buffers (pinned)
    X_host = I.torch_view(d["X"], wl.dt).pin_memory()
    Y_host = torch.empty(Y.shape, dtype=Y.dtype).pin_memory()

    # the library's host-buffer call: X copied in, then Y computed in row blocks,
    # each block copied out on a second stream while the next one is computed
    copy_stream = torch.cuda.Stream(device=dev)
    e2e_rows = 2048

    def e2e_copies():
        ss.sp24_gemm_host(form, X_host, Y_host, Xd, Y, alpha=alpha, rows_per_block=e2e_rows, copy_stream=copy_stream)

    def e2e_direct():  # the epilogue stores Y into the pinned host buffer itself
        ss.sp24_gemm_host(form, X_host, Y_host, Xd, None, alpha=alpha)

    e2e_paths = {
        "copies": (e2e_copies, f"sp24_gemm_host (pinned host X and Y, {e2e_rows}-row blocks, "
                               "device Y copied out on a second stream)"),
        "direct": (e2e_direct, "sp24_gemm_host (pinned host X and Y, X copied in, the epilogue stores Y "
                               "into host memory)"),
    }
    e2e_ms = {}
    for key, (fn, _) in e2e_paths.items():
        e2e_ms[key] = statistics.mean(timed_steps(fn, max(3, args.steps // 2), 2, flush, stream))
    e2e_best = min(e2e_ms, key=e2e_ms.get)
    e2e_value = ws * eff_flops / (e2e_ms[e2e_best] * 1e-3) / 1e12
    link = host_link_rates(Xd, X_host, Y, Y_host, stream)
    x_bytes, y_bytes = Xd.numel() * Xd.element_size(), Y.numel() * Y.element_size()
    # the end-to-end floor: X in and Y out over the host link, the GEMM fully hidden
    link_ms = x_bytes / link["h2d_gbs"] / 1e6 + y_bytes / link["d2h_gbs"] / 1e6

    protocol = headline_protocol(step, flush, stream, dev, eff_flops) if rank == 0 else None

    rows = {}
    mma = None
    if not args.no_rows and rank == 0:
        rows = bench_rows(args, ss, dev, stream, flush, pk, d, wl, Wd, Xd, form)
        mma = mma_microbench(ss, stream)

    if rank == 0:
        clocks = clk.summary()
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": wl.dt, "data": "synthetic (seeded generator)",
            "config": {"workload": f"{wl.name}: W {M}x{K} N(0,{wl.sigma_w:g}) pruned 2:4, X {K}x{N} N(0,1), "
                                   f"{wl.dt} in, {wl.out_dt} out, fp32 accumulate",
                       "M": M, "K": K, "N": N, "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                       "l2": f"flushed between timed steps ({fbytes >> 20} MB write, >= 2x the device's L2)"},
            "step_ms": {"min": round(min(times), 5), "p10": round(pct(times, 10), 5),
                        "median": round(statistics.median(times), 5), "p90": round(pct(times, 90), 5),
                        "max": round(max(times), 5)},
            "timing_protocol": protocol,
            "pct_of_sparse_peak": round(100.0 * achieved / peak_eff, 2),
            "dense_equivalent_tflops": round(2 * achieved, 2),
            # the target's literal reading: this run's rate against the 2:4-sparse bf16 peak
            # (the bf16 run of the same shape is rows.sp24_gemm_bf16)
            "pct_of_sparse_bf16_peak_literal": round(100.0 * achieved / tensor_peak_effective("bf16", pk), 2),
            "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": round(peak_eff, 1),
                         "unit": "TFLOP/s", "frac": round(achieved / peak_eff, 4),
                         "traffic": measured_traffic(wl.name),
                         "peak_note": f"2:4-sparse {wl.dt} peak in nonzero-MAC TFLOP/s = "
                                      f"{'2 x ' if wl.dt == 'e4m3' else ''}{pk['source']} bf16 dense burst "
                                      f"{pk['bf16_tflops']}"},
            "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "path": e2e_paths[e2e_best][1],
                    "ms_per_step": {k: round(v, 4) for k, v in e2e_ms.items()},
                    "h2d_bytes_per_step": int(x_bytes), "d2h_bytes_per_step": int(y_bytes),
                    "host_link_gbs": link, "link_bound_ms": round(link_ms, 4),
                    "frac_of_link_bound": round(link_ms / e2e_ms[e2e_best], 4)},
            "mma_microbench_dense_equivalent_tflops": mma,
            "gpu_launches": args.steps,
            "clocks": clocks,
            "rows": rows,
        }
        key = f"{wl.dt}_sparse_pair_n256"
        if mma and key in mma:
            # the same ceiling as measured on chip at the headline's instruction shape
            # (SM pairs, M = 256, N = 256, one metadata copy per K stage;
            # effective = dense-equivalent / 2)
            mb = mma[key] / 2.0
            line["roofline"]["peak_sparse_mma_microbench"] = round(mb, 1)
            line["roofline"]["frac_of_microbench"] = round(achieved / mb, 4)
        if args.cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(wl, d, args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def bench_rows(args, ss, dev, stream, flush, pk, d, wl, Wd, Xd, form_main) -> dict:
    """Time the other hot-path rows on their own workloads."""
    rows = {}
    steps = max(5, args.steps // 2)
    M, K, N = wl.M, wl.K, wl.N
    eb = I.ELEM_BYTES[wl.dt]
    vb, mb, hb = ss.sp24_sizes(ss._DT[Wd.dtype], M, K)
    # a1: prune + compress (HBM bound): read W, write values + operand-order metadata
    form_c = ss.sp24_prune_compress(Wd, canonical_meta=False)
    compress = lambda: ss.sp24_prune_compress(Wd, canonical_meta=False, out=form_c)  # buffers reused
    t = statistics.mean(timed_steps(compress, steps, 2, flush, stream))
    tg = flushed_graph_ms(compress, flush, dev)
    nbytes = M * K * eb + vb + hb
    rows["sp24_prune_compress"] = {"workload": wl.name, "ms": round(t, 4), "GB/s": round(nbytes / t / 1e6, 1),
                                   "frac_of_hbm": round(nbytes / t / 1e6 / pk["hbm_gbs"], 3),
                                   "graph_l2_flushed": {"ms": round(tg, 4), "GB/s": round(nbytes / tg / 1e6, 1),
                                                        "frac_of_hbm": round(nbytes / tg / 1e6 / pk["hbm_gbs"], 3),
                                                        "note": "20 (L2 flush, call) pairs in one graph minus 20 "
                                                                "flushes alone"}}
    # a8: the dense GEMM of the same kernel family on the same shape
    Yd = torch.empty((M, N), dtype=torch.bfloat16 if wl.out_dt == "bf16" else torch.float16, device=dev)
    t = statistics.mean(timed_steps(lambda: ss.dense_gemm(Wd, Xd, alpha=d["alpha"], out=Yd), steps, 2, flush,
                                    stream))
    dense_tf = 2.0 * M * N * K / (t * 1e-3) / 1e12
    rows["dense_gemm"] = {"workload": wl.name, "ms": round(t, 4), "TFLOP/s": round(dense_tf, 1),
                          "frac_of_dense_peak": round(dense_tf / (pk["bf16_tflops"] * (2 if wl.dt == "e4m3" else 1)),
                                                      3)}
    # the fused layer epilogue on the same shape: per-row bias + GELU, e4m3 output
    # (the next layer's input), against the plain GEMM with its bf16 output
    if wl.dt == "e4m3":
        Y8 = torch.empty((M, N), dtype=torch.float8_e4m3fn, device=dev)
        bias = torch.linspace(-0.5, 0.5, M, dtype=torch.float32, device=dev)
        t_ep = statistics.mean(timed_steps(
            lambda: ss.sp24_gemm(form_main, Xd, alpha=d["alpha"], out=Y8, bias=bias, act="gelu", y_scale=8.0),
            steps, 2, flush, stream))
        t_plain = statistics.mean(timed_steps(lambda: ss.sp24_gemm(form_main, Xd, alpha=d["alpha"], out=Yd), steps,
                                              2, flush, stream))
        eff = M * N * K / (t_ep * 1e-3) / 1e12
        rows["sp24_gemm_bias_gelu_e4m3_out"] = {"workload": wl.name, "ms": round(t_ep, 4),
                                                "plain_bf16_out_ms": round(t_plain, 4),
                                                "effective_TFLOP/s": round(eff, 1)}
        del Y8, bias
    # a2 in bf16 on the same LLM FFN shape, when the headline is e4m3
    if wl.name == "llm_ffn_e4m3":
        wb = I.WORKLOADS["llm_ffn_bf16"]
        db, Wb, Xb, fb = make_sp24(wb, dev, ss)
        Yb = torch.empty((wb.M, wb.N), dtype=torch.bfloat16, device=dev)
        t = statistics.mean(timed_steps(lambda: ss.sp24_gemm(fb, Xb, out=Yb), steps, 2, flush, stream))
        eff = wb.M * wb.N * wb.K / (t * 1e-3) / 1e12
        rows["sp24_gemm_bf16"] = {"workload": wb.name, "ms": round(t, 4), "effective_TFLOP/s": round(eff, 1),
                                  "dense_equivalent_TFLOP/s": round(2 * eff, 1),
                                  "frac_of_sparse_bf16_peak": round(eff / pk["bf16_tflops"], 4)}
        t = statistics.mean(timed_steps(lambda: ss.dense_gemm(Wb, Xb, out=Yb), steps, 2, flush, stream))
        rows["dense_gemm_bf16"] = {"workload": wb.name, "ms": round(t, 4),
                                   "TFLOP/s": round(2.0 * wb.M * wb.N * wb.K / (t * 1e-3) / 1e12, 1)}
        del db, Wb, Xb, fb, Yb
    # a2 on the small workloads (toy, BERT FFN up/down, ResNet-50 1x1): one launch
    # after an L2 flush (events around it), and 20 launches back to back in one
    # CUDA graph (L2 warm, launch overhead amortised)
    small = {}
    for name in ("toy_fp16", "bert_ffn_up_bf16", "bert_ffn_down_bf16", "resnet50_1x1_fp16"):
        ws = I.WORKLOADS[name]
        dsm, Ws, Xs, fs = make_sp24(ws, dev, ss)
        Ys = torch.empty((ws.M, ws.N), dtype=Ws.dtype, device=dev)
        t_cold = statistics.median(timed_steps(lambda: ss.sp24_gemm(fs, Xs, out=Ys), steps, 3, flush, stream))
        t_dense = statistics.median(timed_steps(lambda: ss.dense_gemm(Ws, Xs, out=Ys), steps, 3, flush, stream))
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        t_warm = graph_ms(lambda: ss.sp24_gemm(fs, Xs, out=Ys), 20, side)
        vb_s, _, hb_s = ss.sp24_sizes(ss._DT[Ws.dtype], ws.M, ws.K)
        nbytes = vb_s + hb_s + ws.K * ws.N * 2 + ws.M * ws.N * 2
        small[name] = {"MxNxK": f"{ws.M}x{ws.N}x{ws.K}", "us_l2_flushed": round(t_cold * 1e3, 2),
                       "dense_us_l2_flushed": round(t_dense * 1e3, 2),
                       "us_graph_back_to_back": round(t_warm * 1e3, 2),
                       "effective_TFLOP/s_graph": round(ws.M * ws.N * ws.K / (t_warm * 1e-3) / 1e12, 1),
                       "GB/s_graph": round(nbytes / (t_warm * 1e-3) / 1e9, 1)}
        del dsm, Ws, Xs, fs, Ys
    rows["sp24_gemm_small_configs"] = small
    # a3-a7: tile-wise prune and the TW / TVW gather GEMMs vs the same-kernel dense GEMM
    tw = I.WORKLOADS["tile_wise_4096_bf16"]
    dt_ = tw.make()
    keep = dt_["keep"]
    keep4 = (keep // 4) * 4
    Wt = I.torch_view(dt_["W"], "bf16").to(dev)
    Xt = I.torch_view(dt_["X"], "bf16").to(dev)
    Yt = torch.empty((tw.M, tw.N), dtype=torch.bfloat16, device=dev)
    sz = ss.tw_sizes(ss.BF16, True, tw.M, tw.K, keep4)
    work = torch.empty(sz["workspace_bytes"], dtype=torch.uint8, device=dev)
    # the prune calls are timed writing into the buffers of an earlier result (out=),
    # so that no allocation of the Python helper is inside the timed region
    form_tvw = ss.tw_prune_compress(Wt, keep4, True, work)
    t_prune = statistics.mean(timed_steps(lambda: ss.tw_prune_compress(Wt, keep4, True, work, out=form_tvw), steps,
                                          2, flush, stream))
    form_tw = ss.tw_prune_compress(Wt, keep, False, work)
    t_tw = statistics.mean(timed_steps(lambda: ss.tvw_gemm(form_tw, Xt, out=Yt), steps, 2, flush, stream))
    t_tvw = statistics.mean(timed_steps(lambda: ss.tvw_gemm(form_tvw, Xt, out=Yt), steps, 2, flush, stream))
    t_dense = statistics.mean(timed_steps(lambda: ss.dense_gemm(Wt, Xt, out=Yt), steps, 2, flush, stream))
    # block-wise (NEXT-2) at the same per-tile kept fractions: 64-column blocks
    keep_b = (keep // 64).astype(np.int32)
    szb = ss.bw_sizes(ss.BF16, tw.M, tw.K, keep_b)
    work_b = torch.empty(szb["workspace_bytes"], dtype=torch.uint8, device=dev)
    form_bw = ss.bw_prune_compress(Wt, keep_b, work_b)
    t_bw_prune = statistics.mean(timed_steps(lambda: ss.bw_prune_compress(Wt, keep_b, work_b, out=form_bw), steps,
                                             2, flush, stream))
    t_bw = statistics.mean(timed_steps(lambda: ss.bw_gemm(form_bw, Xt, out=Yt), steps, 2, flush, stream))
    flops_bw = 2.0 * 128 * 64 * float(keep_b.sum()) * tw.N
    # element-wise / unstructured (NEXT-3): CSR x dense on the CUDA cores at 90 % and 95 % sparsity
    ew_rows = {}
    szw = ss.ew_sizes(ss.BF16, tw.M, tw.K, tw.K)
    work_e = torch.empty(szw["workspace_bytes"], dtype=torch.uint8, device=dev)
    for sparsity in (0.90, 0.95):
        k_e = round((1.0 - sparsity) * tw.K)
        form_e = ss.ew_prune_compress(Wt, k_e, work_e)
        t_ep = statistics.mean(timed_steps(lambda: ss.ew_prune_compress(Wt, k_e, work_e, out=form_e), 3, 1, flush,
                                           stream))
        t_e = statistics.mean(timed_steps(lambda: ss.ew_spmm(form_e, Xt, out=Yt), 5, 2, flush, stream))
        ew_rows[f"{int(sparsity * 100)}%"] = {
            "prune_ms": round(t_ep, 4), "spmm_ms": round(t_e, 4),
            "effective_TFLOP/s": round(2.0 * tw.M * k_e * tw.N / (t_e * 1e-3) / 1e12, 1),
            "speedup_over_dense": round(t_dense / t_e, 3)}
        del form_e
    del work_e
    dens = 128.0 * keep.sum() / (tw.M * tw.K)
    flops_tw = 2.0 * 128 * float(keep.sum()) * tw.N
    flops_tvw = 2.0 * 128 * float(keep4.sum()) * tw.N * 0.5
    # 3x3 convolutions of ResNet-50 (NEXT-4), batch 32, 2:4 vs dense filter, implicit GEMM
    conv_rows = {}
    for (H, Cin, Cout) in ((28, 128, 128), (14, 256, 256)):
        Nb = 32
        g = np.random.default_rng(7)
        Xc = torch.from_numpy(g.standard_normal((Nb, H, H, Cin)).astype(np.float32)).to(dev, torch.bfloat16)
        Wc = torch.from_numpy((g.standard_normal((Cout, 9 * Cin)) * (2.0 / (9 * Cin)) ** 0.5).astype(np.float32)
                              ).to(dev, torch.bfloat16)
        fc = ss.sp24_prune_compress(Wc, canonical_meta=False)
        Yc = torch.empty((Cout, Nb * H * H), dtype=torch.bfloat16, device=dev)
        t_sp = statistics.mean(timed_steps(lambda: ss.conv3x3(fc, Xc, out=Yc), steps, 2, flush, stream))
        t_dn = statistics.mean(timed_steps(lambda: ss.conv3x3(Wc, Xc, out=Yc), steps, 2, flush, stream))
        # tile-wise filter: each 128-channel tile keeps a quarter of its (tap, 64-channel) groups
        groups = 9 * Cin // 64
        keep_g = np.full((Cout + 127) // 128, max(1, round(0.25 * groups)), dtype=np.int32)
        ft = ss.bw_prune_compress(Wc, keep_g)
        t_twc = statistics.mean(timed_steps(lambda: ss.conv3x3(ft, Xc, out=Yc), steps, 2, flush, stream))
        flops = 2.0 * Cout * 9 * Cin * Nb * H * H
        kept = float(keep_g[0]) / groups
        conv_rows[f"{H}x{H}x{Cin}->{Cout}, batch {Nb}"] = {
            "sp24_ms": round(t_sp, 4), "dense_ms": round(t_dn, 4),
            "sp24_effective_TFLOP/s": round(0.5 * flops / (t_sp * 1e-3) / 1e12, 1),
            "dense_TFLOP/s": round(flops / (t_dn * 1e-3) / 1e12, 1), "speedup": round(t_dn / t_sp, 3),
            "tw_kept_fraction": round(kept, 4), "tw_ms": round(t_twc, 4),
            "tw_effective_TFLOP/s": round(kept * flops / (t_twc * 1e-3) / 1e12, 1),
            "tw_speedup": round(t_dn / t_twc, 3)}
        del Xc, Wc, fc, ft, Yc
    rows["conv3x3_resnet50"] = conv_rows
    rows["tile_wise"] = {
        "workload": tw.name, "kept_fraction": round(float(keep.sum()) / tw.K / len(keep), 4),
        "tw_prune_compress_ms (TVW)": round(t_prune, 4),
        "tw_gemm_ms": round(t_tw, 4), "tw_effective_TFLOP/s": round(flops_tw / (t_tw * 1e-3) / 1e12, 1),
        "tvw_gemm_ms": round(t_tvw, 4), "tvw_effective_TFLOP/s": round(flops_tvw / (t_tvw * 1e-3) / 1e12, 1),
        "dense_gemm_ms": round(t_dense, 4),
        "dense_TFLOP/s": round(2.0 * tw.M * tw.N * tw.K / (t_dense * 1e-3) / 1e12, 1),
        "tvw_speedup_over_dense": round(t_dense / t_tvw, 3), "tw_speedup_over_dense": round(t_dense / t_tw, 3),
        "bw_prune_compress_ms": round(t_bw_prune, 4), "bw_gemm_ms": round(t_bw, 4),
        "bw_effective_TFLOP/s": round(flops_bw / (t_bw * 1e-3) / 1e12, 1),
        "bw_kept_fraction": round(float(keep_b.sum()) * 64 / tw.K / len(keep_b), 4),
        "bw_speedup_over_dense": round(t_dense / t_bw, 3),
        "ew_unstructured": ew_rows,
        "sparsity": round(1 - float(dens), 4),
    }
    return rows


CPU_SAMPLE_ROWS = 1024


def cpu_sample(wl) -> np.ndarray:
    """The fixed CPU-oracle sample: CPU_SAMPLE_ROWS seeded random rows of W (all of
    X), the same for the GPU arm's cpu_baseline and for --impl reference."""
    rng = np.random.default_rng(0)
    return np.sort(rng.choice(wl.M, size=min(CPU_SAMPLE_ROWS, wl.M), replace=False))


def cpu_threads() -> int:
    """Threads the oracle's numpy math runs on (its BLAS pool when it can be read,
    else the CPUs this process may use)."""
    try:
        from threadpoolctl import threadpool_info
        n = [p["num_threads"] for p in threadpool_info() if p.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return len(os.sched_getaffinity(0))


def cpu_step(wl, d, sel) -> float:
    """One oracle step on the sample, as the oracle stands: 2:4 prune + compress of the
    sampled rows, decompress, decode of X, fp64 matmul, rounding to the output type.
    Returns seconds."""
    import oracle
    t0 = time.perf_counter()
    v, m = oracle.sp24.compress(d["W"][sel], wl.dt)
    oracle.gemm.gemm_sp24(v, m, wl.K, d["X"], wl.dt, wl.out_dt, d["alpha"])
    return time.perf_counter() - t0


def cpu_sample_desc(wl, n_rows: int) -> str:
    return (f"{n_rows} seeded random rows of W (all N={wl.N} columns of X, K={wl.K}) per step: prune + compress "
            f"+ decompress + decode of X + fp64 matmul + rounding, all timed")


def cpu_baseline(wl, d, seconds: float) -> dict:
    """The CPU oracle, as it stands, on the fixed row sample: steps repeated for about
    `seconds` (at least two), the median step time reported."""
    sel = cpu_sample(wl)
    cpu_step(wl, d, sel)                       # untimed first call (page-in, thread pool start)
    times = []
    while len(times) < 2 or sum(times) < seconds:
        times.append(cpu_step(wl, d, sel))
    per = statistics.median(times)
    eff = 2.0 * len(sel) * wl.N * wl.K * 0.5 / per / 1e12
    return {"value": eff, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
            "sample": cpu_sample_desc(wl, len(sel)) + f"; median of {len(times)} steps, {per:.2f} s each",
            "ms_per_sample_step": round(per * 1e3, 1)}


def run_reference(args) -> None:
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    wl = I.WORKLOADS[args.workload]
    d = wl.make()
    sel = cpu_sample(wl)
    for _ in range(args.warmup):
        cpu_step(wl, d, sel)
    times = [cpu_step(wl, d, sel) for _ in range(args.steps)]
    ms = 1e3 * statistics.mean(times)
    flops = 2.0 * len(sel) * wl.N * wl.K * 0.5
    value = flops * args.steps / sum(times) / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": wl.dt, "data": "synthetic (seeded generator)",
            "config": {"workload": wl.name, "M": wl.M, "K": wl.K, "N": wl.N, "sample_rows": int(len(sel)),
                       "step": "the CPU oracle on the fixed row sample (ms_per_step is that sample's measured time)"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
                             "sample": cpu_sample_desc(wl, len(sel))},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


PROFILE_CASES = ("headline", "headline_bf16", "compress", "tvw", "tw", "tw_prune", "dense_4096", "ew", "bw",
                 "conv_tw", "conv_sp24")


def run_profile_case(case: str) -> None:
    """Sets up one kernel of the bench on its workload and launches it four times
    (for an ncu capture of the last launches; prints nothing but a completion line)."""
    dev = torch.device("cuda", 0)
    from structured_sparse_dnn_gb300 import build
    build.build()
    from structured_sparse_dnn_gb300 import ssdnn as ss
    if case in ("headline", "headline_bf16", "compress"):
        wl = I.WORKLOADS["llm_ffn_bf16" if case == "headline_bf16" else DEFAULT_WORKLOAD]
        d, Wd, Xd, form = make_sp24(wl, dev, ss)
        Y = torch.empty((wl.M, wl.N), dtype=torch.bfloat16, device=dev)
        fn = ((lambda: ss.sp24_prune_compress(Wd, canonical_meta=False)) if case == "compress"
              else (lambda: ss.sp24_gemm(form, Xd, alpha=d["alpha"], out=Y)))
    elif case in ("conv_tw", "conv_sp24"):
        # ResNet-50 3x3 layers, batch 32: 28 x 28 x 128 -> 128 with the tile-wise filter (a
        # quarter of the (tap, 64-channel) groups), 14 x 14 x 256 -> 256 with the 2:4 filter
        H, Cin, Cout = (28, 128, 128) if case == "conv_tw" else (14, 256, 256)
        g = np.random.default_rng(7)
        Xc = torch.from_numpy(g.standard_normal((32, H, H, Cin)).astype(np.float32)).to(dev, torch.bfloat16)
        Wc = torch.from_numpy((g.standard_normal((Cout, 9 * Cin)) * (2.0 / (9 * Cin)) ** 0.5).astype(np.float32)
                              ).to(dev, torch.bfloat16)
        if case == "conv_tw":
            form = ss.bw_prune_compress(Wc, np.full((Cout + 127) // 128, round(0.25 * 9 * Cin // 64), dtype=np.int32))
        else:
            form = ss.sp24_prune_compress(Wc, canonical_meta=False)
        Yc = torch.empty((Cout, 32 * H * H), dtype=torch.bfloat16, device=dev)
        fn = lambda: ss.conv3x3(form, Xc, out=Yc)
    else:
        tw = I.WORKLOADS["tile_wise_4096_bf16"]
        d = tw.make()
        keep = d["keep"]
        keep4 = (keep // 4) * 4
        Wt = I.torch_view(d["W"], "bf16").to(dev)
        Xt = I.torch_view(d["X"], "bf16").to(dev)
        Yt = torch.empty((tw.M, tw.N), dtype=torch.bfloat16, device=dev)
        work = torch.empty(ss.tw_sizes(ss.BF16, True, tw.M, tw.K, keep4)["workspace_bytes"], dtype=torch.uint8,
                           device=dev)
        if case == "tw_prune":
            form = ss.tw_prune_compress(Wt, keep4, True, work)
            fn = lambda: ss.tw_prune_compress(Wt, keep4, True, work, out=form)
        elif case == "dense_4096":
            fn = lambda: ss.dense_gemm(Wt, Xt, out=Yt)
        elif case == "ew":  # the element-wise SpMM at 90 % sparsity
            form = ss.ew_prune_compress(Wt, round(0.1 * tw.K))
            fn = lambda: ss.ew_spmm(form, Xt, out=Yt)
        elif case == "bw":  # block-wise at the tile-wise kept fractions (64-column blocks)
            form = ss.bw_prune_compress(Wt, (keep // 64).astype(np.int32))
            fn = lambda: ss.bw_gemm(form, Xt, out=Yt)
        else:
            form = ss.tw_prune_compress(Wt, keep4 if case == "tvw" else keep, case == "tvw", work)
            fn = lambda: ss.tvw_gemm(form, Xt, out=Yt)
    for _ in range(4):
        fn()
    torch.cuda.synchronize()
    assert ss.check_device_error() == 0
    print(f"profile case {case}: done", flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(I.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-rows", action="store_true", help="skip the per-row sub-benchmarks")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--profile", choices=PROFILE_CASES,
                    help="run one kernel of the bench four times on its workload (for ncu) and exit")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)   # at least three untimed warm-up steps
    if args.profile:
        run_profile_case(args.profile)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
