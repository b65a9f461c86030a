"""Benchmark of the grouped matmul on GB300 (one JSON line on stdout).

Headline workload: the Mixtral-like MoE up-projection forward (8192 tokens,
top-2 of 8 experts -> 16384 rows; lhs [16384, 4096] bf16; rhs [8, 28672, 4096]
bf16 in the NT layout; bf16 out).  A step is one gmm call over that batch.
Metric: useful TFLOP/s = 2 * sum_g m_g * n * k / time.  Inputs (2.0 GB) are
larger than the 126 MB L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {gmm,reference}] [--no-suite]

Under torchrun every rank runs its own replica of the step (independent
batches: weak scaling, no collective on the data path); rank 0 prints the line.
--impl reference times the CPU oracle on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "grouped-GEMM useful TFLOP/s and % of GB300 dense peak (HBM GB/s for decode)"
UNIT = "TFLOP/s"
WORKLOAD = ("mixtral_up: gmm NT, lhs [16384,4096] bf16, rhs [8,28672,4096] bf16, "
            "group_sizes from softmax top-2 of 8 (seeded N(0,1) logits), bf16 out")
PROFILE = os.path.join(ROOT, "profiles", "gemm_bf16_2sm_nt_mixtral_up.md")
KERNEL_SRC = os.path.join(ROOT, "moe_grouped_matrix_gb300", "csrc", "gemm_bf16_2sm.cu")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


def kernel_hash() -> str:
    """Hash of the headline kernel's source, the headers it includes and the host code that
    picks its tile order."""
    h = hashlib.sha256()
    for path in (KERNEL_SRC, os.path.join(os.path.dirname(KERNEL_SRC), "ptx.cuh"),
                 os.path.join(os.path.dirname(KERNEL_SRC), "worklist.cuh"),
                 os.path.join(os.path.dirname(KERNEL_SRC), "gmm_api.cu")):
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profile_traffic():
    """DRAM bytes per launch recorded by the committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    if not os.path.exists(PROFILE):
        return None
    text = open(PROFILE).read()
    h = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    t = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not h or not t or h.group(1) != kernel_hash():
        return None
    return float(t.group(1))


# ---------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
            return
        t0 = time.time()
        while time.time() - t0 < 5 and os.path.getsize(self.path) == 0:
            time.sleep(0.05)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        with open(self.path) as f:
            out = summarize_clocks(f)
        os.unlink(self.path)
        return out


def summarize_clocks(lines):
    """nvidia-smi rows of ClockSampler.QUERY (CSV, no header, no units) -> the line's `clocks`:
    the median SM clock, the largest maximum clock, and the throttle reasons seen active in any
    sample; None without a complete row.  Fields that are not numbers ("[N/A]") are skipped."""
    rows = []
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) >= 9:
            rows.append(parts)
    if not rows:
        return None
    sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
    smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
    return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
            "reasons": reasons, "samples": len(rows)}


def headline_config(sizes, m, k, n, world):
    """The `config` of the headline line, the same for the GPU arm and the reference arm."""
    return {"workload": WORKLOAD, "m": int(m), "k": int(k), "n": int(n), "groups": int(sizes.size),
            "group_sizes": sizes.tolist(), "l2": "inputs larger than L2 (2.0 GB per step)",
            "parallelism": f"{world} independent replicas" if world > 1 else "single GPU"}


# ---------------------------------------------------------------- cpu baseline
def oracle_sample(lhs_cpu, rhs_cpu, group_sizes, rows_per_group, seed=123):
    import oracle
    from moe_grouped_matrix_gb300.workloads import sample_rows, stored_bits

    offs = oracle.group_offsets(group_sizes, lhs_cpu.shape[0])
    rng = np.random.Generator(np.random.PCG64(seed))
    rows = []
    for g in range(offs.size - 1):
        lo, hi = int(offs[g]), int(offs[g + 1])
        if hi > lo:
            rows.append(np.sort(rng.choice(hi - lo, size=min(rows_per_group, hi - lo), replace=False) + lo))
    rows = np.concatenate(rows).astype(np.int64)
    lb, rb = stored_bits(lhs_cpu), stored_bits(rhs_cpu)
    threads = oracle.default_threads()
    t0 = time.perf_counter()
    oracle.gmm(lb, rb, group_sizes, transpose_rhs=True, rows=rows, threads=threads)
    dt = time.perf_counter() - t0
    k = lhs_cpu.shape[1]
    n = rhs_cpu.shape[1]
    flops = 2.0 * rows.size * n * k
    full = float(np.asarray(group_sizes).sum()) / rows.size * dt
    return dict(value=flops / dt / 1e12, seconds=dt, rows=int(rows.size), threads=threads, full_seconds=full)


def _sample_rows(group_sizes, m, per_group, seed):
    """A seeded sample of up to `per_group` rows of every group (all rows of smaller groups)."""
    import oracle

    offs = oracle.group_offsets(group_sizes, m)
    rng = np.random.Generator(np.random.PCG64(seed))
    rows = [np.sort(rng.choice(int(offs[g + 1] - offs[g]), size=min(per_group, int(offs[g + 1] - offs[g])),
                               replace=False) + int(offs[g]))
            for g in range(offs.size - 1) if offs[g + 1] > offs[g]]
    return np.concatenate(rows).astype(np.int64) if rows else np.zeros(0, np.int64)


def oracle_baseline(run, flops_done, flops_full, sample):
    """Times `run()` (one oracle call, as it stands) on the host cores: the CPU baseline of one
    suite entry, with the full workload's time extrapolated by flops when `run` does part of it."""
    import oracle

    t0 = time.perf_counter()
    run()
    dt = time.perf_counter() - t0
    out = {"value": flops_done / dt / 1e12, "unit": UNIT, "cores": oracle.default_threads(), "kind": "oracle",
           "sample": sample, "seconds": dt}
    if flops_done < flops_full:
        out["full_seconds_extrapolated"] = dt * flops_full / flops_done
    return out


# ---------------------------------------------------------------- GPU arm
def run_gpu(args, rank, world):
    import torch
    import moe_grouped_matrix_gb300 as G
    from moe_grouped_matrix_gb300 import build as B
    from moe_grouped_matrix_gb300 import workloads as W
    from moe_grouped_matrix_gb300.sharding import max_over_ranks

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        B.build()
    if world > 1:
        torch.distributed.barrier()
    B.build()
    G.load_library()
    peaks = load_peaks()

    d = W.mixtral_up(dev)
    sizes = d["group_sizes"]
    m, k = d["lhs"].shape
    n = d["rhs"].shape[1]
    flops = 2.0 * float(sizes.sum()) * n * k
    gs = torch.tensor(sizes, dtype=torch.int32, device=dev)
    out = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    step = lambda: G.gmm(d["lhs"], d["rhs"], gs, transpose_rhs=True, out=out)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(local) if rank == 0 else None
    if clocks:
        clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for s, e in ev:
        s.record(stream)
        step()
        e.record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clock_info = clocks.stop() if clocks else None
    total_ms = t_start.elapsed_time(t_end)
    per_launch = [s.elapsed_time(e) for s, e in ev]
    total_ms = max_over_ranks(total_ms, device=dev)
    if G.read_device_errors() != 0:
        raise RuntimeError("device error flags set during the benchmark")

    ms_per_step = total_ms / args.steps
    value = flops * world * args.steps / (total_ms / 1e3) / 1e12
    kernel_ms = float(np.mean(per_launch))
    achieved = flops / (kernel_ms / 1e3) / 1e12

    # end to end: pinned host buffers, copies inside the timed region.  Every step copies its
    # activations and group sizes host -> device, runs gmm and copies its whole result device
    # -> host; the expert weights are model state, resident on the device (a second measurement,
    # `weights_copied_each_step`, also copies the 1.9 GB of weights every step).  Steps are
    # pipelined over two buffer sets and three streams, so step i + 1's input copy overlaps step
    # i's matmul and step i - 1's output copy (stream order keeps each buffer's reuse safe).
    e2e = None
    if True:
        h_lhs = d["lhs"].cpu().pin_memory()
        h_rhs = d["rhs"].cpu().pin_memory()
        h_gs = torch.from_numpy(sizes.copy()).pin_memory()
        h_out = [torch.empty((m, n), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        d_lhs = [torch.empty_like(d["lhs"]) for _ in range(2)]
        d_rhs = [d["rhs"], torch.empty_like(d["rhs"])]
        d_gs = [torch.empty_like(gs) for _ in range(2)]
        d_out = [out, torch.empty_like(out)]
        s_in, s_mm, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_mm = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]

        def run_e2e(copy_weights):
            used = [False, False]

            def e2e_step(i):
                sl = i % 2
                w_dev = d_rhs[sl] if copy_weights else d_rhs[0]
                with torch.cuda.stream(s_in):
                    if used[sl]:
                        s_in.wait_event(ev_mm[sl])  # step i - 2's matmul has read these inputs
                    d_lhs[sl].copy_(h_lhs, non_blocking=True)
                    if copy_weights:
                        w_dev.copy_(h_rhs, non_blocking=True)
                    d_gs[sl].copy_(h_gs, non_blocking=True)
                    ev_in[sl].record(s_in)
                with torch.cuda.stream(s_mm):
                    s_mm.wait_event(ev_in[sl])
                    if used[sl]:
                        s_mm.wait_event(ev_out[sl])  # step i - 2's result has left this buffer
                    G.gmm(d_lhs[sl], w_dev, d_gs[sl], transpose_rhs=True, out=d_out[sl], stream=s_mm)
                    ev_mm[sl].record(s_mm)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_mm[sl])
                    h_out[sl].copy_(d_out[sl], non_blocking=True)
                    ev_out[sl].record(s_out)
                used[sl] = True

            steps_e = max(4, min(args.steps, 10))
            e2e_step(0)
            e2e_step(1)
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s_in)
            for i in range(steps_e):
                e2e_step(i)
            s_out.wait_stream(s_in)
            s_out.wait_stream(s_mm)
            b.record(s_out)
            torch.cuda.synchronize()
            ms = max_over_ranks(a.elapsed_time(b) / steps_e, device=dev)
            h2d = h_lhs.numel() * 2 + h_gs.numel() * 4 + (h_rhs.numel() * 2 if copy_weights else 0)
            return {"value": flops * world / (ms / 1e3) / 1e12, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": int(h_out[0].numel() * 2), "ms_per_step": ms}

        e2e = run_e2e(False)
        e2e["pipelined"] = True
        e2e["weights"] = "resident on the device (model state); activations and group sizes copied each step"
        e2e["weights_copied_each_step"] = run_e2e(True)
        if G.read_device_errors(stream=s_mm) != 0:
            raise RuntimeError("device error flags set during the end-to-end measurement")
        del h_lhs, h_rhs, h_out, d_lhs, d_rhs, d_out

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = oracle_sample(d["lhs"][: m].cpu(), d["rhs"].cpu(), sizes, rows_per_group=args.cpu_rows)
        cpu = {"value": cb["value"], "unit": UNIT, "cores": cb["threads"], "kind": "oracle",
               "sample": f"{cb['rows']} rows ({args.cpu_rows} per group) of the workload, every column, "
                         f"fp64; {cb['seconds']:.1f} s",
               "seconds": cb["seconds"], "full_seconds_extrapolated": cb["full_seconds"]}

    suite = None
    if rank == 0 and world == 1 and not args.no_suite:
        del d, out
        torch.cuda.empty_cache()
        suite = run_suite(dev, peaks)

    traffic = profile_traffic()
    # A timed region of a quarter second or more runs under the power cap: its peak is the
    # sustained one (a seconds-long cuBLAS loop); a shorter one is compared with the burst peak.
    sustained = total_ms >= 250.0
    peak = peaks["bf16_sustained"] if sustained else peaks["bf16"]
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": headline_config(sizes, m, k, n, world),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peaks['source']} bf16 {'sustained' if sustained else 'burst'} "
                                    f"(timed region {total_ms:.0f} ms)",
                     "frac_of_burst": achieved / peaks["bf16"], "frac_of_sustained": achieved / peaks["bf16_sustained"],
                     "kernel": "gemm_bf16_2sm_kernel<NT, bf16 out>", "kernel_ms": kernel_ms,
                     "flops_per_launch": flops},
        "gpu_launches": args.steps,
        "clocks": clock_info,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    if suite is not None:
        line["suite"] = suite
    return line


def _flush_l2(flush):
    """Evicts every input from L2: writes `flush` (at least twice the L2), then reads it back, so
    that the lines left in L2 are clean and no write-back of the flush lands in a timed region."""
    flush.fill_(1)
    flush.view(-1, 1 << 20).amax(dim=1)


def _time_call(torch, fn, iters=20, warm=3, flush=None):
    """Mean time of fn() in ms over `iters` runs on the current stream.  With `flush` (a device
    buffer of at least twice the L2), L2 is flushed before every run, outside the timed events,
    so that no run finds its inputs in L2."""
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    if flush is None:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(iters):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / iters
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
    for a, b in ev:
        _flush_l2(flush)
        a.record()
        fn()
        b.record()
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in ev) / iters


def run_suite(dev, peaks):
    """Every other workload once: time, useful TFLOP/s, algorithmic GB/s and the fraction
    of the relevant roofline max(F / P_bf16, B / BW) / t."""
    import torch
    import moe_grouped_matrix_gb300 as G
    from moe_grouped_matrix_gb300 import workloads as W

    import oracle
    from moe_grouped_matrix_gb300.workloads import stored_bits

    res = {}
    # written before every timed run of the HBM-bound entries (2x the 126 MB L2)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    l2_note = "L2 flushed (256 MiB written, then read) before every timed run"

    def record(name, ms, flops, bytes_, cpu=None, flushed=True):
        t = ms / 1e3
        floor = max(flops / (peaks["bf16"] * 1e12), bytes_ / (peaks["hbm"] * 1e9))
        res[name] = {"ms": ms, "tflops": flops / t / 1e12, "gbs": bytes_ / t / 1e9,
                     "bound": "tensor" if flops / (peaks["bf16"] * 1e12) > bytes_ / (peaks["hbm"] * 1e9) else "hbm",
                     "roofline_frac": floor / t, "frac_of_bf16_peak": flops / t / 1e12 / peaks["bf16"],
                     "l2": l2_note if flushed else "inputs larger than L2, runs back to back"}
        if cpu is not None:
            res[name]["cpu_baseline"] = cpu

    # The tiny forward workload (512 rows, 8 groups, one empty; fp32 out), oracle in full.
    td = W.tiny(dev)
    tsizes = td["group_sizes"]
    tgs = torch.tensor(tsizes, dtype=torch.int32, device=dev)
    tm, tk = td["lhs"].shape
    tn = td["rhs"].shape[1]
    to = torch.empty((tm, tn), dtype=torch.float32, device=dev)
    ms = _time_call(torch, lambda: G.gmm(td["lhs"], td["rhs"], tgs, out=to), flush=flush)
    tfl = 2.0 * float(tsizes.sum()) * tn * tk
    tl, tr = stored_bits(td["lhs"]), stored_bits(td["rhs"])
    record("tiny_gmm_f32", ms, tfl, tm * tk * 2 + td["rhs"].numel() * 2 + tm * tn * 4,
           cpu=oracle_baseline(lambda: oracle.gmm(tl, tr, tsizes), tfl, tfl, "the whole workload, fp64"))
    del td, to

    # Context, not the reference arm: cuBLAS batched matmul on the dense equivalent of
    # the headline (8 experts x 2048 rows, k 4096 -> n 28672), same GPU, same run.
    a = W.normal((8, 2048, 4096), 1.0, 91, dev)
    wt = W.normal((8, 28672, 4096), 0.02, 92, dev)
    c = torch.empty((8, 2048, 28672), dtype=torch.bfloat16, device=dev)
    ms = _time_call(torch, lambda: torch.bmm(a, wt.transpose(1, 2), out=c), iters=10)
    record("cublas_bmm_dense_equivalent", ms, 2.0 * 8 * 2048 * 28672 * 4096,
           a.numel() * 2 + wt.numel() * 2 + c.numel() * 2, flushed=False)
    # ours on the same shapes (8 groups of 2048 rows), timed the same short way right after
    gs8 = torch.full((8,), 2048, dtype=torch.int32, device=dev)
    a2 = a.view(16384, 4096)
    c2 = c.view(16384, 28672)
    ms = _time_call(torch, lambda: G.gmm(a2, wt, gs8, transpose_rhs=True, out=c2), iters=10)
    record("gmm_same_shapes_as_cublas_line", ms, 2.0 * 8 * 2048 * 28672 * 4096,
           a.numel() * 2 + wt.numel() * 2 + c.numel() * 2, flushed=False)
    del a, wt, c, a2, c2
    torch.cuda.empty_cache()

    mo = W.moe128(dev)
    sizes = mo["group_sizes"]
    gs = torch.tensor(sizes, dtype=torch.int32, device=dev)
    rows = float(sizes.sum())
    live = int((sizes > 0).sum())
    mo_bits = {key: stored_bits(mo[key]) for key in ("lhs", "lhs_wo", "dout", "wi", "wo")}
    per_group = 16  # oracle sample: rows per group (forward) / k rows (tgmm)
    sample = _sample_rows(sizes, mo["lhs"].shape[0], per_group, seed=7)
    for name, lk, wk, trhs, n, k in [
        ("moe128_wi_nt", "lhs", "wi", True, 2048, 2048),
        ("moe128_wo_nt_k1024", "lhs_wo", "wo", True, 2048, 1024),
        ("moe128_wo_nn_n1024", "lhs", "wo", False, 1024, 2048),
        ("moe128_dlhs_nt", "dout", "wi", True, 2048, 2048),
    ]:
        lhs, w = mo[lk], mo[wk]
        o = torch.empty((lhs.shape[0], n), dtype=torch.bfloat16, device=dev)
        ms = _time_call(torch, lambda: G.gmm(lhs, w, gs, transpose_rhs=trhs, out=o), flush=flush)
        bytes_ = rows * k * 2 + live * n * k * 2 + lhs.shape[0] * n * 2
        cpu = oracle_baseline(lambda: oracle.gmm(mo_bits[lk], mo_bits[wk], sizes, transpose_rhs=trhs, rows=sample),
                              2.0 * sample.size * n * k, 2 * rows * n * k,
                              f"{sample.size} rows (up to {per_group} per group), every column, fp64")
        record(name, ms, 2 * rows * n * k, bytes_, cpu=cpu)
        del o
    k_rows = np.sort(np.random.Generator(np.random.PCG64(8)).choice(2048, size=4 * per_group, replace=False))
    tcpu = oracle_baseline(lambda: oracle.tgmm(mo_bits["lhs"], mo_bits["dout"], sizes, k_rows=k_rows),
                           2.0 * rows * k_rows.size * 2048, 2 * rows * 2048 * 2048,
                           f"{k_rows.size} of the 2048 output rows of every group, every column, fp64")
    dw = torch.empty((128, 2048, 2048), dtype=torch.float32, device=dev)
    ms = _time_call(torch, lambda: G.tgmm(mo["lhs"], mo["dout"], gs, out=dw), flush=flush)
    record("moe128_tgmm_f32", ms, 2 * rows * 2048 * 2048, rows * 2048 * 2 * 2 + dw.numel() * 4, cpu=tcpu)
    del dw
    dwb = torch.empty((128, 2048, 2048), dtype=torch.bfloat16, device=dev)
    ms = _time_call(torch, lambda: G.tgmm(mo["lhs"], mo["dout"], gs, out=dwb), flush=flush)
    record("moe128_tgmm_bf16", ms, 2 * rows * 2048 * 2048, rows * 2048 * 2 * 2 + dwb.numel() * 2)
    del mo, dwb, mo_bits
    torch.cuda.empty_cache()

    fd = W.fp8_decode(dev)
    sizes = fd["group_sizes"]
    gs = torch.tensor(sizes, dtype=torch.int32, device=dev)
    n, k = fd["rhs"].shape[1], fd["rhs"].shape[2]
    nb = fd["rhs_scale"].shape[1]
    o = torch.empty((fd["lhs"].shape[0], n), dtype=torch.bfloat16, device=dev)
    fd_bits = {key: stored_bits(fd[key]) for key in ("lhs", "rhs", "rhs_scale", "rhs_bias")}
    for go in (0, 32):
        rhs, sc, bi = fd["rhs"][go:], fd["rhs_scale"][go:], fd["rhs_bias"][go:]
        local = sizes[go:]
        rows = float(local.sum())
        live = int((local > 0).sum())
        call = lambda: G.gmm(fd["lhs"], rhs, gs, rhs_scale=sc, rhs_bias=bi, group_offset=go, out=o)
        # weights, scales and bias of non-empty local experts, their lhs rows, the whole output
        bytes_ = live * (n * k + nb * n * 4 + n * 2) + rows * k * 2 + fd["lhs"].shape[0] * n * 2
        cpu = oracle_baseline(
            lambda: oracle.gmm(fd_bits["lhs"], fd_bits["rhs"][go:], sizes, group_offset=go,
                               rhs_scale=fd_bits["rhs_scale"][go:], rhs_bias=fd_bits["rhs_bias"][go:]),
            2 * rows * n * k, 2 * rows * n * k, "the whole call, fp64")
        # the default: the activation rows split once by a pass, then the fp8 kernel
        record(f"fp8_decode_go{go}", _time_call(torch, call, flush=flush), 2 * rows * n * k, bytes_, cpu=cpu)
        # the same call with the split made inside the kernel for every weight tile
        with G.options(act_split="kernel"):
            record(f"fp8_decode_go{go}_split_in_kernel", _time_call(torch, call, flush=flush), 2 * rows * n * k,
                   bytes_)
    del fd_bits
    del fd, o
    torch.cuda.empty_cache()

    # bf16 weights with the same per-block scales and bias (the decoding kernel's bf16 path).
    fd = W.fp8_decode(dev)
    sizes = fd["group_sizes"]
    gs = torch.tensor(sizes, dtype=torch.int32, device=dev)
    w16 = fd["rhs"].to(torch.bfloat16)
    del fd["rhs"]
    o = torch.empty((fd["lhs"].shape[0], n), dtype=torch.bfloat16, device=dev)
    rows = float(sizes.sum())
    live = int((sizes > 0).sum())
    ms = _time_call(torch, lambda: G.gmm(fd["lhs"], w16, gs, rhs_scale=fd["rhs_scale"], rhs_bias=fd["rhs_bias"], out=o),
                    flush=flush)
    bytes_ = live * (n * k * 2 + nb * n * 4 + n * 2) + rows * k * 2 + fd["lhs"].shape[0] * n * 2
    record("decode_bf16_weights_scaled", ms, 2 * rows * n * k, bytes_)
    del fd, o, w16
    torch.cuda.empty_cache()

    # The decode workload with the other weight formats of the pages' dtype list (group_offset 0).
    for fmt in ("e5m2", "int8", "int4", "uint4", "e2m1"):
        fd = W.fp8_decode(dev, fmt=fmt)
        sizes = fd["group_sizes"]
        gs = torch.tensor(sizes, dtype=torch.int32, device=dev)
        o = torch.empty((fd["lhs"].shape[0], n), dtype=torch.bfloat16, device=dev)
        kw = {"rhs_format": fd["rhs_format"]} if fd["rhs_format"] else {}
        rows = float(sizes.sum())
        live = int((sizes > 0).sum())
        ms = _time_call(torch, lambda: G.gmm(fd["lhs"], fd["rhs"], gs, rhs_scale=fd["rhs_scale"],
                                             rhs_bias=fd["rhs_bias"], out=o, **kw), flush=flush)
        wbytes = n * k // 2 if fmt in W.PACKED else n * k
        bytes_ = live * (wbytes + nb * n * 4 + n * 2) + rows * k * 2 + fd["lhs"].shape[0] * n * 2
        record(f"decode_{fmt}_weights", ms, 2 * rows * n * k, bytes_)
        del fd, o
        torch.cuda.empty_cache()

    # W8A8 on the decode workload: per-token-group e4m3 quantisation of the activations
    # (128-wide groups), then the grouped matmul on e4m3 activations and e4m3 weights, with
    # f32 and with E8M0 weight scales; each kernel alone and the two in sequence.
    fd = W.fp8_decode(dev)
    sizes = fd["group_sizes"]
    gs = torch.tensor(sizes, dtype=torch.int32, device=dev)
    m = fd["lhs"].shape[0]
    rows = float(sizes.sum())
    live = int((sizes > 0).sum())
    q, a_scale = G.quantize_e4m3(fd["lhs"])
    o = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    ms = _time_call(torch, lambda: G.quantize_e4m3(fd["lhs"], out=q, scale=a_scale), flush=flush)
    record("w8a8_quantize_e4m3", ms, 0.0, m * k * 2 + m * k + m * (k // 128) * 4)
    e8 = torch.full(fd["rhs_scale"].shape, 120, dtype=torch.uint8, device=dev)
    for name, sc, sbytes in (("w8a8_decode_gmm", fd["rhs_scale"], 4), ("w8a8_decode_gmm_e8m0", e8, 1)):
        ms = _time_call(torch, lambda: G.gmm(q, fd["rhs"], gs, rhs_scale=sc, rhs_bias=fd["rhs_bias"], lhs_scale=a_scale,
                                             out=o), flush=flush)
        bytes_ = live * (n * k + nb * n * sbytes + n * 2) + rows * (k + (k // 128) * 4) + m * n * 2
        record(name, ms, 2 * rows * n * k, bytes_)

    def both():
        G.quantize_e4m3(fd["lhs"], out=q, scale=a_scale)
        G.gmm(q, fd["rhs"], gs, rhs_scale=fd["rhs_scale"], rhs_bias=fd["rhs_bias"], lhs_scale=a_scale, out=o)

    ms = _time_call(torch, both, flush=flush)
    bytes_ = live * (n * k + nb * n * 4 + n * 2) + m * k * 2 + m * n * 2
    record("w8a8_decode_quantize_plus_gmm", ms, 2 * rows * n * k, bytes_)
    del fd, o, q, a_scale, e8
    torch.cuda.empty_cache()

    # Microscaling weights on the decode workload (bf16 activations, the fp16-weight kernel):
    # MXFP8 (e4m3, an E8M0 scale per 32 k of a weight row) and NVFP4 (e2m1, an e4m3 scale per 16 k).
    for name, fmt, per in (("decode_mxfp8_weights", "e4m3", 32), ("decode_nvfp4_weights", "e2m1", 16)):
        fd = W.fp8_decode(dev, fmt=fmt)
        sizes = fd["group_sizes"]
        gs = torch.tensor(sizes, dtype=torch.int32, device=dev)
        L_ = fd["rhs"].shape[0]
        if fmt == "e4m3":
            bs = torch.full((L_, n, k // per), 127, dtype=torch.uint8, device=dev)
        else:
            bs = W.uniform((L_, n, k // per), 0.5, 2.0, 7, dev).to(torch.float8_e4m3fn)
        o = torch.empty((fd["lhs"].shape[0], n), dtype=torch.bfloat16, device=dev)
        kw = {"rhs_format": fd["rhs_format"]} if fd["rhs_format"] else {}
        rows = float(sizes.sum())
        live = int((sizes > 0).sum())
        ms = _time_call(torch, lambda: G.gmm(fd["lhs"], fd["rhs"], gs, rhs_block_scale=bs, rhs_bias=fd["rhs_bias"],
                                             out=o, **kw), flush=flush)
        wbytes = n * k // 2 if fmt == "e2m1" else n * k
        bytes_ = live * (wbytes + n * (k // per) + n * 2) + rows * k * 2 + fd["lhs"].shape[0] * n * 2
        record(name, ms, 2 * rows * n * k, bytes_)
        del fd, o, bs
        torch.cuda.empty_cache()
    del flush
    return res


# ---------------------------------------------------------------- ncu cases
def _ncu_gemm_small(torch, G, W, dev):
    # the headline kernel on a quarter of the workload's n (0.8 GB on the device, > L2)
    d = W.mixtral_up(dev)
    lhs, rhs = d["lhs"], d["rhs"][:, :7168].contiguous()
    gs = torch.tensor(d["group_sizes"], dtype=torch.int32, device=dev)
    out = torch.empty((lhs.shape[0], 7168), dtype=torch.bfloat16, device=dev)
    del d
    return lambda: G.gmm(lhs, rhs, gs, transpose_rhs=True, out=out)


def _ncu_tgmm(torch, G, W, dev):
    mo = W.moe128(dev, which=("lhs", "dout"))
    gs = torch.tensor(mo["group_sizes"], dtype=torch.int32, device=dev)
    dw = torch.empty((128, 2048, 2048), dtype=torch.float32, device=dev)
    return lambda: G.tgmm(mo["lhs"], mo["dout"], gs, out=dw)


def _ncu_fp8_decode(torch, G, W, dev):
    fd = W.fp8_decode(dev)
    gs = torch.tensor(fd["group_sizes"], dtype=torch.int32, device=dev)
    return lambda: G.gmm(fd["lhs"], fd["rhs"], gs, rhs_scale=fd["rhs_scale"], rhs_bias=fd["rhs_bias"])


def _ncu_decode_int4(torch, G, W, dev):
    fd = W.fp8_decode(dev, fmt="int4")
    gs = torch.tensor(fd["group_sizes"], dtype=torch.int32, device=dev)
    return lambda: G.gmm(fd["lhs"], fd["rhs"], gs, rhs_scale=fd["rhs_scale"], rhs_bias=fd["rhs_bias"],
                         rhs_format="int4")


def _ncu_decode_nvfp4(torch, G, W, dev):
    fd = W.fp8_decode(dev, fmt="e2m1")
    gs = torch.tensor(fd["group_sizes"], dtype=torch.int32, device=dev)
    L, n, k = fd["rhs"].shape[0], fd["rhs"].shape[1], fd["lhs"].shape[1]
    bs = W.uniform((L, n, k // 16), 0.0625, 16.0, 121, dev).to(torch.float8_e4m3fn)
    return lambda: G.gmm(fd["lhs"], fd["rhs"], gs, rhs_block_scale=bs, rhs_format="e2m1", rhs_bias=fd["rhs_bias"])


def _ncu_decode_int8(torch, G, W, dev):
    fd = W.fp8_decode(dev, fmt="int8")
    gs = torch.tensor(fd["group_sizes"], dtype=torch.int32, device=dev)
    return lambda: G.gmm(fd["lhs"], fd["rhs"], gs, rhs_scale=fd["rhs_scale"], rhs_bias=fd["rhs_bias"])


def _ncu_w8a8_decode(torch, G, W, dev):
    fd = W.fp8_decode(dev)
    gs = torch.tensor(fd["group_sizes"], dtype=torch.int32, device=dev)
    q, a_scale = G.quantize_e4m3(fd["lhs"])
    return lambda: G.gmm(q, fd["rhs"], gs, rhs_scale=fd["rhs_scale"], rhs_bias=fd["rhs_bias"], lhs_scale=a_scale)


def _ncu_moe128_wi(torch, G, W, dev):
    mo = W.moe128(dev, which=("lhs", "wi"))
    gs = torch.tensor(mo["group_sizes"], dtype=torch.int32, device=dev)
    out = torch.empty((32768, 2048), dtype=torch.bfloat16, device=dev)
    return lambda: G.gmm(mo["lhs"], mo["wi"], gs, out=out)


NCU_CASES = {"gemm_small": _ncu_gemm_small, "tgmm": _ncu_tgmm, "fp8_decode": _ncu_fp8_decode,
             "moe128_wi": _ncu_moe128_wi, "decode_int4": _ncu_decode_int4, "decode_int8": _ncu_decode_int8,
             "decode_nvfp4": _ncu_decode_nvfp4,
             "w8a8_decode": _ncu_w8a8_decode}


def run_ncu_case(name):
    import torch
    import moe_grouped_matrix_gb300 as G
    from moe_grouped_matrix_gb300 import build as B
    from moe_grouped_matrix_gb300 import workloads as W

    B.build()
    dev = torch.device("cuda", 0)
    fn = NCU_CASES[name](torch, G, W, dev)
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    if G.read_device_errors() != 0:
        raise RuntimeError("device error flags set")
    print(f"ncu case {name}: 3 launches ok")


# ---------------------------------------------------------------- reference arm
def run_reference(args, rank, world):
    """The CPU oracle, as it stands, on a bounded sample of the same workload each step."""
    import torch
    from moe_grouped_matrix_gb300 import workloads as W

    d = W.mixtral_up("cpu")
    sizes = d["group_sizes"]
    m, k = d["lhs"].shape
    n = d["rhs"].shape[1]
    for _ in range(args.warmup):
        oracle_sample(d["lhs"], d["rhs"], sizes, rows_per_group=1)
    times, vals, info = [], [], None
    for s in range(args.steps):
        info = oracle_sample(d["lhs"], d["rhs"], sizes, rows_per_group=args.ref_rows, seed=1000 + s)
        times.append(info["seconds"])
        vals.append(info["value"])
    total = sum(times)
    flops = 2.0 * info["rows"] * n * k
    value = flops * args.steps / total / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": headline_config(sizes, m, k, n, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": info["threads"], "kind": "oracle",
                         "sample": f"{info['rows']} rows ({args.ref_rows} per group) of the workload per step, "
                                   f"every column, fp64"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gmm", choices=["gmm", "reference"])
    ap.add_argument("--no-suite", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-rows", type=int, default=64, help="rows per group in the CPU-baseline sample")
    ap.add_argument("--ref-rows", type=int, default=1, help="rows per group per step of the reference arm")
    ap.add_argument("--ncu-case", choices=sorted(NCU_CASES), default=None,
                    help="run one small profiling case a few times and exit (for ncu captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.ncu_case:
        run_ncu_case(args.ncu_case)
        return

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return

    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", int(os.environ["LOCAL_RANK"])))
    line = run_gpu(args, rank, world)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
