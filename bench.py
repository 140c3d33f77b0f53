"""Benchmark: PASA attention forward TFLOP/s on GB300, fraction of the tensor-core peak.

One step = the whole hot path on one batch of synthetic input already resident in HBM:
the pseudo-average shift of K (kshift kernel) followed by the attention kernel, both
through the C ABI (pasa_kshift, pasa_attn_fwd_shifted). FLOPs follow the FlashAttention
convention (4 * B * Hq * visible (query, key) pairs * D). The e2e figure goes through
pasa_attn_fwd_host with pinned host buffers: every byte of q, k, v copied in and of o and
lse copied out lies inside the timed region, the copies overlapping the kernels piece by
piece.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--mode M]
  python bench.py --impl reference ...   # the fp64 CPU oracle on this host's cores

Prints one JSON line (rank 0). Under torchrun (N > 1) every rank runs its own replica of
the workload on its own GPU (weak scaling: the work is independent per (batch, head), so
there is no data-path collective); value = all ranks' FLOPs / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
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

import workloads as wl  # noqa: E402

METRIC = "PASA attn fwd TFLOP/s at 1 GB300; fraction of fp16 tensor peak; RMSE vs fp64"
DEFAULT_WORKLOAD = "kbias10_t3_b1h28g4_s32768_d128_causal"
# Each extra (workload, mode) of the default run: its TFLOP/s, fraction of the peak and
# relRMSE against the fp64 oracle. None = the mode of the headline line.
ALSO_RUNS = [
    ("kbias20_b1h28g4_s4096_d128_causal", None, False),
    ("resonance_a30_b2h5_s9216_d64", None, False),
    ("iid_b4h32g8_s8192_d128_causal", None, False),
    ("kbias10_t3_b1h28g4_s32768_d128_causal", 1, False),
    ("resonance_a30_b2h5_s9216_d64", 1, False),
    # the FP8 scores of the shift mode (e4m3 Q and K' with scales, fp32 accumulation): speed
    # on the 32K workload, and the 4K one, where the shift is what makes e4m3 scores usable
    ("kbias10_t3_b1h28g4_s32768_d128_causal", 5, False),
    ("kbias20_b1h28g4_s4096_d128_causal", 5, False),
    # the shift fused into the attention kernel (one launch, raw keys) on the same workloads
    ("kbias10_t3_b1h28g4_s32768_d128_causal", None, True),
    ("iid_b4h32g8_s8192_d128_causal", None, True),
]
DECODE_WORKLOAD = "kbias10_t3_b8h28g4_q1_s32768_d128_decode"
MODE_NAMES = {0: "shift_f16acc", 1: "shift_f32acc", 2: "naive_f16acc", 3: "noshift_f32acc", 4: "shift_f16all",
              5: "shift_fp8", 6: "naive_fp8"}
SHIFT_MODES = (0, 1, 4)     # a pseudo-average shift kernel (fp16 K') runs before the attention kernel
FP8_MODES = (5, 6)          # an e4m3 key-preparation kernel runs before it
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one attention-kernel launch
# on the 32K workload in mode 0, from an ncu capture of one full-size launch. Reported only
# while the kernel sources are the ones the counters were taken on.
TRAFFIC_WORKLOAD = "kbias10_t3_b1h28g4_s32768_d128_causal"
TRAFFIC_MODE = 0
TRAFFIC_BYTES = 738.26e6 + 198.99e6   # ncu prints MB to two decimals
TRAFFIC_KERNEL_SHA = "734e0f31415fb2e7"
# The same for one decode-kernel launch on the decode workload (an ncu capture at full
# size: 539.11 MB read + 2.97 MB written).
DECODE_TRAFFIC_BYTES = 539112960 + 2970368
DECODE_TRAFFIC_SHA = "0ff35ca3bb268cac"


def _source_sha(name):
    src = os.path.join(os.path.dirname(os.path.abspath(__file__)), "precision_flashattention_numerics_gb300",
                       "csrc", name)
    try:
        with open(src, "rb") as f:
            return hashlib.sha256(f.read()).hexdigest()[:16]
    except OSError:
        return None


def measured_traffic(w, mode):
    if TRAFFIC_BYTES is None or w.name != TRAFFIC_WORKLOAD or mode != TRAFFIC_MODE or \
            _source_sha("attn_fwd.cuh") != TRAFFIC_KERNEL_SHA:
        return None
    return round(TRAFFIC_BYTES)


def measured_decode_traffic(mode):
    if mode != 0 or _source_sha("decode_fwd.cuh") != DECODE_TRAFFIC_SHA:
        return None
    return DECODE_TRAFFIC_BYTES


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"pasa_bench_clocks_gpu{gpu_index}_{os.getpid()}.csv")

    def __enter__(self):
        os.makedirs(os.path.dirname(self.path), exist_ok=True)
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for _, _, flags in rows for n, f in zip(names, flags) if f.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def visible_pairs_rows(w: wl.Workload, rows: np.ndarray) -> np.ndarray:
    i = rows % w.Sq
    if not w.causal:
        return np.full(len(rows), w.Sk, np.int64)
    return np.clip(i + w.Sk - w.Sq + 1, 0, w.Sk)


def cpu_oracle_sample(w: wl.Workload, q, k, v, budget_s: float, seed: int = 0, keep: list | None = None):
    """Time the fp64 oracle on random rows of the workload for about `budget_s` seconds.
    With `keep`, the (rows, O_ref) pairs it computed are appended to it."""
    import oracle

    rng = np.random.default_rng(seed)
    total_rows = w.B * w.Hq * w.Sq
    n = 16
    elapsed, flops, rows_done = 0.0, 0.0, 0
    while elapsed < budget_s:
        rows = np.sort(rng.integers(0, total_rows, n)).astype(np.int64)
        t0 = time.perf_counter()
        o_ref, _ = oracle.attention(q, k, v, causal=w.causal, rows=rows)
        dt = time.perf_counter() - t0
        if keep is not None:
            keep.append((rows, o_ref))
        elapsed += dt
        flops += float(4.0 * w.D * visible_pairs_rows(w, rows).sum())
        rows_done += n
        n = int(min(max(n * 2, 16), max(16, n * (budget_s - elapsed) / max(dt, 1e-3))))
        if budget_s - elapsed < 0.2 * dt:
            break
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    threads = int(os.environ.get("OMP_NUM_THREADS", cores))
    return {
        "value": flops / elapsed / 1e12,
        "unit": "TFLOP/s",
        "cores": threads,
        "kind": "oracle",
        "sample": f"{rows_done} random query rows of {w.name} (fp64 oracle, all visible keys), {elapsed:.1f} s",
    }


def rmse_vs_oracle(o, pairs):
    """relRMSE / relMax (output scale) of device output `o` [B, H, S, D] against fp64 oracle
    rows: `pairs` is a list of (flat row indices, O_ref rows)."""
    import torch

    rows = np.concatenate([r for r, _ in pairs])
    ref = np.concatenate([x for _, x in pairs]).astype(np.float64)
    flat = o.reshape(-1, o.shape[-1])
    got = flat.index_select(0, torch.as_tensor(rows, device=o.device, dtype=torch.long)).double().cpu().numpy()
    if not np.isfinite(got).all():
        return {"rel_rmse": None, "rel_max": None, "rows": int(len(rows)), "nonfinite_rows": True}
    d = got - ref
    return {"rel_rmse": float(np.sqrt(np.mean(d * d)) / np.sqrt(np.mean(ref * ref))),
            "rel_max": float(np.abs(d).max() / np.abs(ref).max()), "rows": int(len(rows)),
            "vs": "fp64 oracle (plain attention) on the same fp16 inputs"}


def bench_gpu(args, w: wl.Workload, rank: int, world: int, local_rank: int, also: bool = False, mode=None,
              fused=None):
    import torch

    import precision_flashattention_numerics_gb300 as pasa

    mode = args.mode if mode is None else mode
    fused = args.fused if fused is None else fused
    if fused and (w.D != 128 or mode not in SHIFT_MODES):
        raise SystemExit("--fused needs D = 128 and a shift mode (0, 1, 4)")

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    q, k, v = wl.make_inputs(w, seed=w.seed + 7919 * rank)
    qt, kt, vt = (torch.from_numpy(x).to(dev) for x in (q, k, v))
    o = torch.empty_like(qt)
    lse = torch.empty((w.B, w.Hq, w.Sq), device=dev, dtype=torch.float32)
    if not also:
        # the e2e leg's pinned host buffers, allocated up front as an application would (the
        # host is then past the work of pinning ~0.5 GB before any timed copy)
        qh, kh, vh = (torch.from_numpy(x).pin_memory() for x in (q, k, v))
        oh = torch.empty(qt.shape, dtype=torch.float16).pin_memory()
        lh = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    nb = (w.Sk + pasa.block_rows(w.D) - 1) // pasa.block_rows(w.D)
    shift = mode in SHIFT_MODES
    fp8 = mode in FP8_MODES
    ks = torch.empty_like(kt) if shift else kt
    means = torch.empty((w.B, w.Hkv, nb, w.D), device=dev, dtype=torch.float16) if shift else None
    stream = torch.cuda.current_stream()
    prep = {}

    def prep_keys():
        if fused:
            return   # the attention kernel shifts the keys itself
        if shift:
            pasa.kshift(kt, out=ks, means=means)
        elif fp8:
            prep["k8"], prep["means"], prep["kscale"] = pasa.kprep_fp8(kt, mode=mode)

    def attention():
        if fused:
            pasa.attn_fwd_fused(qt, kt, vt, causal=w.causal, mode=mode, out=o, lse=lse)
        elif fp8:
            pasa.attn_fwd_fp8(qt, prep["k8"], prep["means"], prep["kscale"], vt, causal=w.causal, mode=mode,
                              out=o, lse=lse)
        else:
            pasa.attn_fwd_shifted(qt, ks, means, vt, causal=w.causal, mode=mode, out=o, lse=lse)

    def step():
        prep_keys()
        attention()

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    pasa.check_device_error()

    n = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    sampler = ClockSampler(local_rank) if not also else None
    if sampler:
        sampler.__enter__()
    barrier(world)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(n):
        ev[i][0].record(stream)
        prep_keys()
        ev[i][1].record(stream)
        attention()
        ev[i][2].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    if sampler:
        sampler.__exit__(None, None, None)
    pasa.check_device_error()
    total_ms = t_start.elapsed_time(t_end)
    total_ms = max_over_ranks(total_ms, world)
    attn_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(n)]
    kshift_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(n)] if ((shift or fp8) and not fused) else [0.0] * n
    flops = w.flops()
    finite = bool(torch.isfinite(o).all().item())
    res = {
        "total_ms": total_ms,
        "ms_per_step": total_ms / n,
        "attn_ms": statistics.mean(attn_ms),
        "kshift_ms": statistics.mean(kshift_ms),
        "flops": flops,
        "tflops": flops * n * world / (total_ms * 1e-3) / 1e12,
        "attn_tflops": flops / (statistics.mean(attn_ms) * 1e-3) / 1e12,
        "finite": finite,
        "clocks": sampler.summary() if sampler else None,
        "host": (q, k, v),
        "o": o,
    }
    if also:
        return res

    if shift and not fused:
        # The shift kernel on its own: back-to-back launches over four copies of the keys
        # (4 x (K + K') larger than L2, so each launch reads and writes DRAM), CUDA events
        # around the batch. The in-step events above also hold the gap after the attention
        # kernel.
        nbuf, n_iso = 4, max(8, n)
        kb_in = [kt] + [kt.clone() for _ in range(nbuf - 1)]
        kb_out = [ks] + [torch.empty_like(kt) for _ in range(nbuf - 1)]
        kb_m = [means] + [torch.empty_like(means) for _ in range(nbuf - 1)]
        for j in range(nbuf):
            pasa.kshift(kb_in[j], out=kb_out[j], means=kb_m[j])
        torch.cuda.synchronize()
        i0 = torch.cuda.Event(enable_timing=True)
        i1 = torch.cuda.Event(enable_timing=True)
        i0.record(stream)
        for it in range(n_iso):
            pasa.kshift(kb_in[it % nbuf], out=kb_out[it % nbuf], means=kb_m[it % nbuf])
        i1.record(stream)
        torch.cuda.synchronize()
        pasa.check_device_error()
        res["kshift_isolated_ms"] = i0.elapsed_time(i1) / n_iso
        res["kshift_isolated_launches"] = n_iso
        del kb_in, kb_out, kb_m

    # end to end through pasa_attn_fwd_host: q, k, v from pinned host memory, o and lse back
    # to it, every copy inside the timed region (overlapped with the kernels piece by piece)
    B, Hq, Sq, D = qt.shape
    Hkv, Sk = kt.shape[1], kt.shape[2]
    hbuf = torch.empty(pasa.host_device_bytes(B, Hq, Hkv, Sq, Sk, D, w.causal, mode, args.host_chunks),
                       dtype=torch.uint8, device=qt.device)

    def e2e_step():
        pasa.attn_fwd_host(qh, kh, vh, causal=w.causal, mode=mode, out=oh, lse=lh, chunks=args.host_chunks,
                           device_buffer=hbuf, sync=False)

    for _ in range(max(3, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    n_e2e = n
    barrier(world)
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e + 1)]
    marks[0].record(stream)
    for i in range(n_e2e):
        e2e_step()
        marks[i + 1].record(stream)
    torch.cuda.synchronize()
    pasa.check_device_error()
    e2e_ms = max_over_ranks(marks[0].elapsed_time(marks[-1]), world)
    step_ms = [marks[i].elapsed_time(marks[i + 1]) for i in range(n_e2e)]
    res["e2e"] = {
        "value": flops * n_e2e * world / (e2e_ms * 1e-3) / 1e12,
        "unit": "TFLOP/s",
        "h2d_bytes_per_step": int(q.nbytes + k.nbytes + v.nbytes),
        "d2h_bytes_per_step": int(oh.numel() * 2 + lh.numel() * 4),
        "ms_per_step": e2e_ms / n_e2e,
        # value and ms_per_step are over all timed steps; single steps of this path now and
        # then stall for several ms (host copy path), which these two make visible
        "median_step_ms": statistics.median(step_ms),
        "max_step_ms": max(step_ms),
    }
    return res


def bench_decode(args, w: wl.Workload, local_rank: int, sampler=None):
    """One decode step: refresh the cache's last block (where the new key row lands) and
    attend (decode kernel + split merge), in one call (pasa_attn_fwd_decode_step, or
    _step_fp8 for the e4m3 cache), whose decode kernel overlaps the refresh. attn_ms times
    the attend call alone. The cache is prepared once before timing, as a prefill would
    leave it."""
    import torch

    import precision_flashattention_numerics_gb300 as pasa

    dev = torch.device("cuda", local_rank)
    q, k, v = wl.make_inputs(w)
    qt, kt, vt = (torch.from_numpy(x).to(dev) for x in (q, k, v))
    mode = args.mode if args.mode in MODE_NAMES else 0
    shift = mode in SHIFT_MODES
    fp8 = mode in FP8_MODES
    kscale = None
    if fp8:   # e4m3 cache: codes, block scales, means (mode 5)
        ks, means, kscale = pasa.kprep_fp8(kt, mode=mode)
    else:
        ks, means = pasa.kshift(kt) if shift else (kt, None)
    o = torch.empty_like(qt)
    lse = torch.empty((w.B, w.Hq, w.Sq), device=dev, dtype=torch.float32)
    nbytes = pasa.decode_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D)
    ws = torch.empty(max(nbytes, 256), device=dev, dtype=torch.uint8)
    bn = pasa.block_rows(w.D)
    last = (w.Sk - 1) // bn
    stream = torch.cuda.current_stream()

    def attend():
        if fp8:
            pasa.attn_fwd_decode_fp8(qt, ks, means, kscale, vt, causal=w.causal, mode=mode, out=o, lse=lse,
                                     workspace=ws)
        else:
            pasa.attn_fwd_decode(qt, ks, means, vt, causal=w.causal, mode=mode, out=o, lse=lse, workspace=ws)

    def step():
        # one call: refresh and decode, the decode kernel overlapping the refresh
        if fp8:
            pasa.attn_fwd_decode_step_fp8(qt, kt, ks, means, kscale, vt, last, causal=w.causal, mode=mode, out=o,
                                          lse=lse, workspace=ws)
        else:
            pasa.attn_fwd_decode_step(qt, kt, ks, means, vt, last, causal=w.causal, mode=mode, out=o, lse=lse,
                                      workspace=ws)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    pasa.check_device_error()
    n = args.steps if args.decode else max(args.steps, 20)
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    if sampler:
        sampler.__enter__()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    marks[0].record(stream)
    for i in range(n):
        step()
        marks[i + 1].record(stream)
    torch.cuda.synchronize()
    wall_ms = (time.perf_counter() - t0) * 1e3 / n
    if sampler:
        sampler.__exit__(None, None, None)
    pasa.check_device_error()
    step_ms = marks[0].elapsed_time(marks[-1]) / n
    # the attend call alone (events around each call), for the kernel's roofline
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    for i in range(n):
        ev[i][0].record(stream)
        attend()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    pasa.check_device_error()
    attn_ms = statistics.mean(ev[i][0].elapsed_time(ev[i][1]) for i in range(n))
    nb = -(-w.Sk // bn)
    # algorithmic bytes of the attention: the cache (K' or K: fp16, or e4m3 codes and block
    # scales; V fp16), the block means, q, o, lse
    cache = w.B * w.Hkv * w.Sk * w.D * (1 if fp8 else 2) + w.B * w.Hkv * w.Sk * w.D * 2
    moved = cache + (w.B * w.Hkv * nb * w.D * 2 if (shift or mode == 5) else 0) + (w.B * w.Hkv * nb * 4 if fp8 else 0) \
        + 2 * w.B * w.Hq * w.Sq * w.D * 2 + w.B * w.Hq * w.Sq * 4
    gbs = moved / (attn_ms * 1e-3) / 1e9
    return {
        "workload": w.name, "mode": MODE_NAMES[mode], "tokens_per_s": round(w.B * w.Sq / (step_ms * 1e-3), 1),
        "ms_per_step": round(step_ms, 5), "attn_ms": round(attn_ms, 5), "host_ms_per_step": round(wall_ms, 5),
        "attn_bytes": moved, "attn_gbs": round(gbs, 1), "finite": bool(torch.isfinite(o).all().item()),
        "launches_per_step": (1 if (shift or fp8) else 0) + (2 if nbytes else 1),
        "merge": "combine_splits_kernel" if nbytes else "in the decode kernel (thread-block cluster)",
        "step_call": "pasa_attn_fwd_decode_step_fp8" if fp8 else "pasa_attn_fwd_decode_step",
    }


def _json_num(x):
    """A float for the JSON line; an overflowed accumulator (inf) is reported as "inf"."""
    x = float(x)
    return x if math.isfinite(x) else ("inf" if x > 0 else "nan" if x != x else "-inf")


def bench_stats(args, w: wl.Workload, local_rank: int):
    """The overflow diagnostic (pasa_attn_fwd_stats with per-key-block maxima): one step is the
    shift, the zeroing of the block maxima and the diagnostic variant of the attention kernel,
    which also tracks each block's score minimum and reduces both magnitudes per block."""
    import torch

    import precision_flashattention_numerics_gb300 as pasa

    dev = torch.device("cuda", local_rank)
    q, k, v = wl.make_inputs(w)
    qt, kt, vt = (torch.from_numpy(x).to(dev) for x in (q, k, v))
    mode = args.mode if args.mode in (0, 1, 2, 3, 4) else 0
    for _ in range(3):
        pasa.attn_fwd_stats(qt, kt, vt, causal=w.causal, mode=mode, block_stats=True)
    torch.cuda.synchronize()
    pasa.check_device_error()
    n = max(3, min(args.steps, 10))
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for i in range(n):
        ev[i][0].record(stream)
        pasa.attn_fwd_stats(qt, kt, vt, causal=w.causal, mode=mode, block_stats=True)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    pasa.check_device_error()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    # score magnitudes of the last call, over all query rows: what the score accumulator held
    # (S' with the shift, S without) and the recovered raw scores |S' + q.m|, against 65504
    _, _, st, _ = pasa.attn_fwd_stats(qt, kt, vt, causal=w.causal, mode=mode, block_stats=True)
    pasa.check_device_error()
    acc, rec = st[..., 0], st[..., 1]
    return {"workload": w.name, "mode": MODE_NAMES[mode], "ms_per_step": round(ms, 4),
            "tflops": round(w.flops() / (ms * 1e-3) / 1e12, 1), "steps": n,
            "step": "kshift + zeroing of the block maxima + diagnostic attention kernel",
            "max_abs_accumulated_score": _json_num(acc.max().item()),
            "max_abs_raw_score": _json_num(rec.max().item()),
            "rows_over_fp16_max": int((acc > 65504.0).sum().item()),
            "fp16_max": 65504.0}


def decode_main(args, rank: int, world: int, local_rank: int):
    """`--decode`: one JSON line for the decode step alone (tokens/s; roofline against HBM)."""
    w = wl.WORKLOADS[DECODE_WORKLOAD]
    if args.impl == "reference" or world > 1:
        if rank == 0:
            print(json.dumps({"impl": args.impl, "unavailable": "the decode line is single-GPU, pasa arm only"}))
        return
    import torch

    torch.cuda.set_device(local_rank)
    peaks, peak_src = load_peaks()
    sampler = ClockSampler(local_rank)
    dec = bench_decode(args, w, local_rank, sampler)
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    out = {
        "metric": "PASA decode tokens/s at 1 GB300 (one new query row per head per step)",
        "value": dec["tokens_per_s"], "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": dec["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3+f16" if args.mode in FP8_MODES else "f16",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Sq": w.Sq, "Sk": w.Sk, "D": w.D,
                   "mode": dec["mode"], "l2": "the K/V cache (537 MB) is larger than L2; no flush"},
        "roofline": {"kernel": "decode_fwd_kernel" + (" + combine_splits_kernel" if dec["launches_per_step"] > 2
                                                        else ""), "bound": "hbm",
                     "achieved": dec["attn_gbs"], "peak": hbm, "unit": "GB/s",
                     "frac": round(dec["attn_gbs"] / hbm, 4),
                     "traffic": measured_decode_traffic(args.mode),
                     "peak_source": f"{peak_src} copy bandwidth"},
        "gpu_launches": dec["launches_per_step"] * args.steps, "clocks": sampler.summary(),
        "finite_output": dec["finite"], "decode": dec,
    }
    print(json.dumps(out))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="pasa", choices=["pasa", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(wl.WORKLOADS))
    ap.add_argument("--mode", type=int, default=0, choices=[0, 1, 2, 3, 4, 5, 6])
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-also", action="store_true")
    ap.add_argument("--host-chunks", type=int, default=0,
                    help="pieces of the host-buffer (e2e) call; 0 = the library's automatic count")
    ap.add_argument("--fused", action="store_true",
                    help="time pasa_attn_fwd_fused (the shift inside the attention kernel) instead of the pre-pass path")
    ap.add_argument("--decode", action="store_true",
                    help="time only the decode step (refresh the cache's last block + attend) on the decode workload")
    args = ap.parse_args()

    rank, world, local_rank = dist_env()
    if args.decode:
        decode_main(args, rank, world, local_rank)
        return
    w = wl.WORKLOADS[args.workload]
    peaks, peak_src = load_peaks()
    config = {
        "workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Sq": w.Sq, "Sk": w.Sk, "D": w.D,
        "causal": w.causal, "inputs": w.kind, "mode": MODE_NAMES[args.mode],
        "path": "fused shift (pasa_attn_fwd_fused)" if args.fused else "shift pre-pass + attention",
        "l2": "inputs larger than L2 (129 MB); no flush between steps",
        "flop_convention": "4*B*Hq*visible_pairs*D",
    }

    if args.impl == "reference":
        if rank != 0:
            return
        q, k, v = wl.make_inputs(w)
        steps = []
        per_step_budget = max(1.0, min(args.cpu_budget, 60.0) / max(1, args.steps))
        for s in range(max(0, args.warmup) + args.steps):
            r = cpu_oracle_sample(w, q, k, v, budget_s=per_step_budget if s >= args.warmup else 0.5, seed=s)
            if s >= args.warmup:
                steps.append(r)
        val = statistics.mean(r["value"] for r in steps)
        out = {
            "impl": "reference", "metric": METRIC, "value": val,
            "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": None, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "config": config,
            "cpu_baseline": {**steps[-1], "value": val},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }
        print(json.dumps(out))
        return

    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    def peak_for(mode):
        peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))  # fp16 dense = bf16 dense rate
        note = f"{peak_src} bf16 dense burst (fp16 dense has the same nominal rate)"
        if mode in FP8_MODES:
            # half the FLOPs (QK) at the e4m3 rate, nominally 2x the 16-bit one, half (PV) at
            # fp16: the time at peak is 3/4 of the all-fp16 time
            peak = peak * 4.0 / 3.0
            note = (f"{peak_src} bf16 dense burst x 4/3: QK at the e4m3 rate (nominally 2x the 16-bit rate), "
                    "PV at the fp16 rate")
        return peak, note

    res = bench_gpu(args, w, rank, world, local_rank)
    also = {}
    if not args.no_also and world == 1:
        for name, amode, afused in ALSO_RUNS:
            amode = args.mode if amode is None else amode
            if name == w.name and amode == args.mode and afused == args.fused:
                continue
            wa = wl.WORKLOADS[name]
            if afused and (wa.D != 128 or amode not in SHIFT_MODES):
                continue
            ra = bench_gpu(args, wa, rank, world, local_rank, also=True, mode=amode, fused=afused)
            aq, ak, av = ra["host"]
            rows = wl.sample_rows(wa, 128)
            import oracle

            o_ref, _ = oracle.attention(aq, ak, av, causal=wa.causal, rows=rows)
            apeak, _ = peak_for(amode)
            attn_tf = ra["flops"] / (ra["attn_ms"] * 1e-3) / 1e12
            also[f"{name}/{MODE_NAMES[amode]}" + ("/fused" if afused else "")] = {
                "workload": name, "mode": MODE_NAMES[amode],
                "path": "fused shift (pasa_attn_fwd_fused, one launch)" if afused else "shift pre-pass + attention",
                "tflops": round(ra["tflops"], 1),
                "ms_per_step": round(ra["ms_per_step"], 4), "attn_ms": round(ra["attn_ms"], 4),
                "attn_tflops": round(attn_tf, 1), "attn_frac": round(attn_tf / apeak, 4),
                "kshift_ms": round(ra["kshift_ms"], 4), "finite": ra["finite"],
                "rmse": rmse_vs_oracle(ra["o"], [(rows, o_ref)]), "steps": args.steps,
                "warmup": max(3, args.warmup)}
            if amode in FP8_MODES:
                also[f"{name}/{MODE_NAMES[amode]}"]["note"] = (
                    "rmse is against plain fp64 attention, so it includes the e4m3 rounding of Q and K' "
                    "(3-bit mantissa); against attention on the same e4m3 values the kernel is within 2e-3 "
                    "(GPU tests)")
            del ra
        also[DECODE_WORKLOAD] = bench_decode(args, wl.WORKLOADS[DECODE_WORKLOAD], local_rank)
        if args.mode not in FP8_MODES:
            also["overflow_diagnostic"] = bench_stats(args, w, local_rank)

    peak, peak_note = peak_for(args.mode)
    traffic = measured_traffic(w, args.mode)
    attn_achieved = res["flops"] / (res["attn_ms"] * 1e-3) / 1e12
    roofline = {
        "kernel": "attn_fwd_kernel", "bound": "tensor", "achieved": round(attn_achieved, 1), "peak": peak,
        "unit": "TFLOP/s", "frac": round(attn_achieved / peak, 4), "traffic": traffic,
        "peak_source": peak_note,
    }
    kshift_kernel = None
    if (args.mode in SHIFT_MODES or args.mode in FP8_MODES) and not args.fused:
        import precision_flashattention_numerics_gb300 as pasa

        nbk = math.ceil(w.Sk / pasa.block_rows(w.D))
        if args.mode in FP8_MODES:   # K read, e4m3 codes, block scales (and means in mode 5) written
            kb = w.B * w.Hkv * (w.Sk * w.D * 3 + nbk * 4 + (nbk * w.D * 2 if args.mode == 5 else 0))
        else:
            kb = 2 * (w.B * w.Hkv * w.Sk * w.D * 2) + w.B * w.Hkv * nbk * w.D * 2
        gbs = kb / (res["kshift_ms"] * 1e-3) / 1e9
        hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        kshift_kernel = {"kernel": "kshift_kernel", "bound": "hbm", "achieved": round(gbs, 1), "peak": hbm,
                         "unit": "GB/s", "frac": round(gbs / hbm, 4), "bytes_per_launch": kb,
                         "ms": round(res["kshift_ms"], 5),
                         "timing": "events around its launch in each timed step (they also hold the gap "
                                   "after the attention kernel)"}
        if res.get("kshift_isolated_ms"):
            gi = kb / (res["kshift_isolated_ms"] * 1e-3) / 1e9
            kshift_kernel["isolated"] = {
                "achieved": round(gi, 1), "frac": round(gi / hbm, 4), "ms": round(res["kshift_isolated_ms"], 5),
                "timing": f"{res['kshift_isolated_launches']} back-to-back launches over 4 copies of the keys "
                          "(larger than L2), events around the batch"}
    dec = also.get(DECODE_WORKLOAD)
    if dec is not None:
        hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        dec["roofline"] = {"kernel": "decode_fwd_kernel" + (" + combine_splits_kernel" if dec["launches_per_step"] > 2
                                                            else ""), "bound": "hbm",
                           "achieved": dec["attn_gbs"], "peak": hbm, "unit": "GB/s",
                           "frac": round(dec["attn_gbs"] / hbm, 4),
                           "traffic": measured_decode_traffic(args.mode), "peak_source": f"{peak_src} copy bandwidth"}

    # accuracy of the timed steps' output: the oracle's rows from the cpu_baseline leg (or,
    # without it, a fixed sample of rows)
    cpu = None
    pairs = []
    if rank == 0:
        q, k, v = res["host"]
        if world == 1 and not args.no_cpu_baseline:
            cpu = cpu_oracle_sample(w, q, k, v, budget_s=args.cpu_budget, keep=pairs)
        else:
            import oracle

            rows = wl.sample_rows(w, 128)
            pairs = [(rows, oracle.attention(q, k, v, causal=w.causal, rows=rows)[0])]
    rmse = rmse_vs_oracle(res["o"], pairs) if rank == 0 else None

    if rank == 0:
        out = {
            "metric": METRIC,
            "value": round(res["tflops"], 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": round(res["ms_per_step"], 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3+f16" if args.mode in FP8_MODES else "f16",
            "data": "synthetic", "config": config,
            "roofline": roofline, "kshift": kshift_kernel, "cpu_baseline": cpu, "e2e": res["e2e"],
            "gpu_launches": args.steps * (2 if ((args.mode in SHIFT_MODES or args.mode in FP8_MODES) and not args.fused)
                                          else 1), "clocks": res["clocks"],
            "finite_output": res["finite"], "rmse": rmse, "also": also,
        }
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
