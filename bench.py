#!/usr/bin/env python
"""Benchmark of the block-sparse prefill attention path on GB300.

One step = one pass of the whole hot path over one layer of synthetic input:
fp_discover (K/V block means + block-score map) -> fp_select (threshold,
sink/local, CSR) -> fp_sparse_attn (paged, PackGQA, mean correction), each a
C-ABI call into libfprefill.

Default workload: the Qwen3-30B-A3B-shaped layer at 128K (batch 1,
L = 131072, 32 query / 4 kv heads, d = 128, 64-token shuffled pages, bf16,
alpha = 0.1, mean correction on), inputs from the seeded generator.  The
headline value is dense-equivalent TFLOP/s = 4 * d * H_q * (causal query-key
pairs) / (ms per layer); ms per layer is reported beside it.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With --gpus N > 1 (under torchrun) every rank runs an independent replica of
the layer (the path has no exchange step): weak scaling, value = the work of
all ranks / the slowest rank's time.  --impl reference times the float64 CPU
oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import shutil
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse prefill attn ms/layer + dense-equiv TFLOP/s at 128K BF16/FP8, 1×GB300"
UNIT = "TFLOP/s (dense-equivalent)"


# ----------------------------------------------------------------------------
# workload arithmetic
# ----------------------------------------------------------------------------

def causal_pairs(spec) -> int:
    return sum(lq * s + lq * (lq + 1) // 2 for lq, s in spec.requests)


def dense_equiv_flop(spec) -> float:
    return 4.0 * spec.d * spec.h_q * causal_pairs(spec)


def index_stats(spec, row_ptr: np.ndarray):
    """Kept blocks per row -> density over causal (I, J) pairs, the executed
    tile FLOPs of the attention kernel and its algorithmic FLOPs."""
    counts = np.diff(row_ptr.astype(np.int64))
    g = spec.h_q // spec.h_kv
    Is, rows = [], 0
    for lq, s in spec.requests:
        nqb = -(-lq // 128)
        I = s // 128 + np.arange(nqb)
        Is.append(np.repeat(I, spec.h_kv))
        rows += nqb * spec.h_kv
    I = np.concatenate(Is)
    causal = (I + 1).sum()
    kept = counts.sum()
    skipped = (I - (counts - 1)).clip(min=0)            # earlier blocks without a kept entry
    tile = 4.0 * spec.d * 128 * 128                      # S + PV of one 128x128 tile, one head
    kept_flop = tile * g * kept
    corr_flop = 4.0 * spec.d * 128 * g * skipped.sum()  # one mean token per skipped block per query
    return dict(density=float(kept / causal), nnz=int(kept), causal_pairs_blocks=int(causal),
                kept_flop=float(kept_flop), corr_flop=float(corr_flop),
                csr_bytes=int(4 * (len(row_ptr) + kept)))


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------

class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        exe = shutil.which("nvidia-smi")
        if exe:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen([exe, f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return None
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() in ("active", "1"):
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------

def max_over_ranks(ms: float, world: int, device=None) -> float:
    """The slowest rank's time (every rank calls this; a no-op at world 1)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(flop_per_replica: float, ms: float, world: int) -> float:
    """Dense-equivalent TFLOP/s of the whole job: every rank runs one replica
    of the layer (weak scaling), and the job takes the slowest rank's time."""
    return world * flop_per_replica / (ms * 1e-3) / 1e12


def cuda_time(fn, steps, stream):
    import torch
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        fn()
    b.record(stream)
    b.synchronize()
    return a.elapsed_time(b) / steps


def recorded_traffic(spec, logit_scale):
    """DRAM bytes per attention launch of this workload from the committed ncu
    record, or None when the record is for another workload or the kernel's
    sources changed since it was taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "attn_kernel_traffic_qwen30b_128k.md")
    if spec.name != "qwen30b-128k" or spec.dtype != "bf16" or logit_scale != 1.0 or not os.path.exists(path):
        return None
    rec = {}
    for line in open(path):
        if ":" in line and line.split(":")[0] in ("traffic_bytes_per_launch", "kernel_sources_sha256"):
            k, v = line.split(":", 1)
            rec[k.strip()] = v.strip()
    csrc = os.path.join(ROOT, "block_sparse_long_fp_gb300", "csrc")
    src = b"".join(open(os.path.join(csrc, f), "rb").read() for f in ("attn.cu", "sm100.cuh", "common.cuh", "launch.cuh"))
    if rec.get("kernel_sources_sha256") != hashlib.sha256(src).hexdigest():
        return None
    return int(float(rec["traffic_bytes_per_launch"]))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def measure_layer(layer, spec, steps, warmup, dense_steps, stream, fp8=False):
    """Time the whole step and each stage on one uploaded layer."""
    import torch
    flop = dense_equiv_flop(spec)
    for _ in range(warmup):
        _, _, (row_ptr, _, _) = layer.prefill()
    torch.cuda.synchronize()
    status = layer.device_status()
    stats = index_stats(spec, row_ptr.cpu().numpy())
    ms = cuda_time(lambda: layer.prefill(), steps, stream)
    k_mean, v_mean, score = layer.discover()
    rp, ci, nz = layer.select(score)
    reps = max(2, min(steps, 5))
    out_buf = torch.empty((layer.total_q, layer.h_q, 128), dtype=torch.bfloat16, device=layer.q.device)
    ms_disc = cuda_time(lambda: layer.discover(k_mean, v_mean, score), reps, stream)
    ms_sel = cuda_time(lambda: layer.select(score, rp, ci, nz), reps, stream)
    ms_attn = cuda_time(lambda: layer.sparse_attn(rp, ci, k_mean, v_mean, out=out_buf, want_lse=False), reps,
                        stream)
    # the fused fp_discover_select (no score map) in place of the first two stages
    km2, vm2, rp2, ci2, nz2 = layer.discover_select()
    ms_dsel = cuda_time(lambda: layer.discover_select(km2, vm2, None, rp2, ci2, nz2), reps, stream)
    ms_dense = None
    if dense_steps > 0:
        layer.dense_attn(out=out_buf, want_lse=False)
        ms_dense = cuda_time(lambda: layer.dense_attn(out=out_buf, want_lse=False), dense_steps, stream)
    peaks, peak_kind = load_peaks()
    peak = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) * (2.0 if fp8 else 1.0)
    attn_flop = stats["kept_flop"] + stats["corr_flop"]
    achieved = attn_flop / (ms_attn * 1e-3) / 1e12
    return dict(ms=ms, flop=flop, status=status, stats=stats, ms_disc=ms_disc, ms_sel=ms_sel, ms_attn=ms_attn,
                ms_dense=ms_dense, ms_dsel=ms_dsel, achieved=achieved, peak=peak, peak_kind=peak_kind)


def summary(m, spec, logit_scale, dtype):
    return {
        "dtype": dtype, "logit_scale": logit_scale,
        "ms_per_layer": round(m["ms"], 4),
        "dense_equiv_tflops": round(m["flop"] / (m["ms"] * 1e-3) / 1e12, 2),
        "stages_ms": {"discover": round(m["ms_disc"], 4), "select": round(m["ms_sel"], 4),
                      "sparse_attn": round(m["ms_attn"], 4), "discover_select_fused": round(m["ms_dsel"], 4)},
        "density": round(m["stats"]["density"], 5),
        "attn_tflops": round(m["achieved"], 2), "attn_peak_tflops": m["peak"],
        "attn_frac": round(m["achieved"] / m["peak"], 4),
        "dense_attn_ms": None if m["ms_dense"] is None else round(m["ms_dense"], 4),
        "speedup_vs_own_dense": None if m["ms_dense"] is None else round(m["ms_dense"] / m["ms"], 3),
        "device_status": m["status"],
    }


def selection_ablation(layer, spec, stream):
    """The max threshold against the top-k and top-p rules (the V1 summary's
    section 4.4 comparison), on one layer: kept density, attention time, and
    the relative error of O against the exact dense output (every 64th token)."""
    import torch
    from block_sparse_long_fp_gb300 import fprefill
    dense, _ = layer.dense_attn(want_lse=False)
    rows = torch.arange(0, layer.total_q, 64, device=dense.device)
    ref = dense[rows].float()
    k_mean, v_mean, score = layer.discover()
    saved = (layer.params.select_rule, layer.params.top_k, layer.params.top_p, layer.params.score_mode)
    out = {}
    rules = [("threshold_alpha_0.1", fprefill.FP_SELECT_THRESHOLD, 0, 0.0, fprefill.FP_SCORE_PACKED),
             ("top_k_64", fprefill.FP_SELECT_TOPK, 64, 0.0, fprefill.FP_SCORE_PACKED),
             ("top_p_0.9", fprefill.FP_SELECT_TOPP, 0, 0.9, fprefill.FP_SCORE_PACKED),
             ("top_p_0.5", fprefill.FP_SELECT_TOPP, 0, 0.5, fprefill.FP_SCORE_PACKED),
             ("head_union_alpha_0.1", fprefill.FP_SELECT_THRESHOLD, 0, 0.0, fprefill.FP_SCORE_HEAD_UNION)]
    for name, rule, k, p, mode in rules:
        layer.params.select_rule, layer.params.top_k, layer.params.top_p, layer.params.score_mode = rule, k, p, mode
        entry = {}
        if mode != fprefill.FP_SCORE_PACKED:
            k_mean, v_mean, score = layer.discover()
            entry["discover_ms"] = round(cuda_time(lambda: layer.discover(k_mean, v_mean, score), 3, stream), 4)
        rp, ci, nnz = layer.select(score)
        o, _ = layer.sparse_attn(rp, ci, k_mean, v_mean, want_lse=False)
        ms = cuda_time(lambda: layer.sparse_attn(rp, ci, k_mean, v_mean, out=o, want_lse=False), 3, stream)
        stats = index_stats(spec, rp.cpu().numpy())
        err = float(torch.linalg.vector_norm(o[rows].float() - ref) / torch.linalg.vector_norm(ref))
        entry.update({"density": round(stats["density"], 5), "attn_ms": round(ms, 4),
                      "rel_err_vs_dense": round(err, 5)})
        out[name] = entry
    (layer.params.select_rule, layer.params.top_k, layer.params.top_p, layer.params.score_mode) = saved
    return out


def chunk_variant(dev, stream, steps, dense_steps):
    """A chunked-prefill step at long context: 512 queries at position 130560
    (32/4 heads, the 128K layer's shape).  It has 64 work units for 152 SMs, so
    the attention splits each row's key list (split-KV) and merges the parts by
    LSE; timed with the automatic split and with splitting off."""
    from block_sparse_long_fp_gb300 import fprefill, synth
    spec = synth.Spec("chunk-512-at-128k", [(512, 130560)], 32, 4, page_size=64, layout="shuffled", n_needles=4,
                      config_id=6)
    case = synth.make_case(spec)
    out = {"workload": spec.name}
    for name, ks in (("auto_split", 0), ("no_split", 1)):
        layer = fprefill.layer_from_case(case, device=dev, params=fprefill.default_params(kv_splits=ks))
        res = summary(measure_layer(layer, spec, steps, 2, dense_steps, stream), spec, 1.0, "bf16")
        res["kv_splits"] = layer.kv_splits
        out[name] = res
        del layer
    a, n = out["auto_split"]["stages_ms"]["sparse_attn"], out["no_split"]["stages_ms"]["sparse_attn"]
    out["attn_speedup_from_split"] = round(n / a, 3)
    return out


def run_ours(args, rank, world):
    import torch
    import torch.distributed as dist
    from block_sparse_long_fp_gb300 import fprefill, synth

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    fp8 = args.dtype == "e4m3"
    spec = synth.config_spec(args.workload, dtype=args.dtype)
    t0 = time.time()
    case = synth.make_case(spec)
    gen_s = time.time() - t0
    layer = fprefill.layer_from_case(case, device=dev)
    if args.logit_scale != 1.0:
        # exact for powers of two; e4m3 codes carry the scale in the per-head query scales
        (layer.q_scale if fp8 else layer.q).mul_(args.logit_scale)
    stream = torch.cuda.current_stream()
    flop = dense_equiv_flop(spec)
    layer_splits = layer.kv_splits          # 1: no split-KV merge launch

    # --- warm-up and one index for the statistics ---
    for _ in range(args.warmup):
        out, _, (row_ptr, col_idx, nnz) = layer.prefill()
    torch.cuda.synchronize()
    status = layer.device_status()
    stats = index_stats(spec, row_ptr.cpu().numpy())

    # --- the timed region: K whole steps, barrier + sync on both sides ---
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        ms = cuda_time(lambda: layer.prefill(), args.steps, stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    ms = max_over_ranks(ms, world, dev)
    clocks = clk.summary()

    # --- per-stage breakdown, the attention kernel alone, the dense path ---
    m = measure_layer(layer, spec, min(args.steps, 5), 1, args.dense_steps, stream, fp8=fp8)
    ms_disc, ms_sel, ms_attn, ms_dense = m["ms_disc"], m["ms_sel"], m["ms_attn"], m["ms_dense"]

    # --- end to end through the C ABI with host buffers ---
    e2e = None
    if args.e2e_steps > 0:
        e2e = run_e2e(layer, args.e2e_steps, flop)

    # --- variants in the same line: the sparse regime and FP8-e4m3 ---
    variants = {}
    if args.variants and rank == 0 and not fp8:
        if args.logit_scale == 1.0:
            layer.q.mul_(16.0)                  # exact: a power of two
            variants["bf16_logit_scale_16"] = summary(
                measure_layer(layer, spec, min(args.steps, 5), 2, args.dense_steps, stream), spec, 16.0, "bf16")
            variants["bf16_logit_scale_16"]["selection_ablation"] = selection_ablation(layer, spec, stream)
            layer.q.div_(16.0)
        del layer
        torch.cuda.empty_cache()
        spec8 = synth.config_spec(args.workload, dtype="e4m3")
        case8 = synth.make_case(spec8)
        layer8 = fprefill.layer_from_case(case8, device=dev)
        variants["e4m3"] = summary(measure_layer(layer8, spec8, min(args.steps, 5), 2, args.dense_steps, stream,
                                                 fp8=True), spec8, 1.0, "e4m3")
        layer8.q_scale.mul_(16.0)               # the same sharper logits, exactly, through the scales
        variants["e4m3_logit_scale_16"] = summary(
            measure_layer(layer8, spec8, min(args.steps, 5), 2, args.dense_steps, stream, fp8=True), spec8, 16.0,
            "e4m3")
        del layer8, case8
        torch.cuda.empty_cache()
        variants["bf16_chunk_512_at_128k"] = chunk_variant(dev, stream, min(args.steps, 5), args.dense_steps)

    peaks, peak_kind = load_peaks()
    attn_flop = stats["kept_flop"] + stats["corr_flop"]
    achieved = attn_flop / (ms_attn * 1e-3) / 1e12
    # e4m3 runs kind::f8f6f4 MMAs: twice the measured bf16 rate (the nominal fp8 / bf16 ratio)
    peak = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) * (2.0 if fp8 else 1.0)
    value = whole_job_value(flop, ms, world)
    q_bytes = spec.total_q * spec.h_q * spec.d * (1 if fp8 else 2)
    res = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": args.dtype,
        "data": "synthetic (seeded block-coherent Q/K with sink and needles, V ~ N(0,1))",
        "config": {"workload": spec.name, "batch": spec.batch, "seq_len": spec.total_q,
                   "h_q": spec.h_q, "h_kv": spec.h_kv, "d": spec.d, "page_size": spec.page_size,
                   "page_layout": spec.layout, "alpha": 0.1, "sink_tokens": 256, "local_tokens": 512,
                   "block": 128, "mean_correction": True, "logit_scale": args.logit_scale,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": f"inputs larger than L2 (Q alone is {q_bytes / 2**20:.0f} MiB)"},
        "ms_per_layer": round(ms, 4),
        "stages_ms": {"discover": round(ms_disc, 4), "select": round(ms_sel, 4),
                      "sparse_attn": round(ms_attn, 4), "discover_select_fused": round(m["ms_dsel"], 4)},
        "density": round(stats["density"], 5), "nnz_blocks": stats["nnz"], "csr_bytes": stats["csr_bytes"],
        "dense_attn_ms": None if ms_dense is None else round(ms_dense, 4),
        "speedup_vs_own_dense": None if ms_dense is None else round(ms_dense / ms, 3),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": recorded_traffic(spec, args.logit_scale),
                     "kernel": "attn_kernel (fp_sparse_attn)",
                     "peak_source": f"{peak_kind} bf16 sustained (MEASURED_PEAKS.json)" + (" x 2 for e4m3" if fp8 else "")},
        "gpu_launches": (9 + (1 if layer_splits > 1 else 0)) * args.steps,
        "device_status": status,
        "clocks": clocks,
        "gen_seconds": round(gen_s, 1),
    }
    if variants:
        res["variants"] = variants
    if e2e:
        res["e2e"] = e2e
    return res, case


def run_e2e(layer, steps, flop):
    """Host pinned inputs -> device, the three C-ABI calls, output -> host."""
    import torch
    host = {n: getattr(layer, n).cpu().pin_memory() for n in ("q", "k_cache", "v_cache", "block_table")}
    out_dev = torch.empty((layer.total_q, layer.h_q, 128), dtype=torch.bfloat16, device=layer.q.device)
    out_host = torch.empty(out_dev.shape, dtype=torch.bfloat16).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_host.numel() * out_host.element_size()
    stream = torch.cuda.current_stream()

    def step():
        for n, t in host.items():
            getattr(layer, n).copy_(t, non_blocking=True)
        layer.prefill(out=out_dev)
        out_host.copy_(out_dev, non_blocking=True)

    step()
    torch.cuda.synchronize()
    ms = cuda_time(step, steps, stream)
    return {"value": round(flop / (ms * 1e-3) / 1e12, 3), "unit": UNIT, "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}


# ----------------------------------------------------------------------------
# the float64 oracle on a bounded sample (CPU baseline and reference arm)
# ----------------------------------------------------------------------------

def oracle_sample(case, seconds: float, seed: int = 0):
    """Time the oracle's full path (pool, score, select, attention) on query
    blocks of one kv head, adding blocks until `seconds` have elapsed; scale
    by the share of the layer's work they represent (work of a row is
    proportional to its causal length I+1)."""
    import oracle
    spec = case.spec
    r = max(range(spec.batch), key=lambda x: spec.requests[x][0])
    lq, start = spec.requests[r]
    hkv, g, B = spec.h_kv, spec.h_q // spec.h_kv, 128
    nqb = -(-lq // B)
    rng = np.random.default_rng(seed)
    t_all = time.perf_counter()
    k, v = oracle.request_kv(case, r)            # decode (not counted as method work)
    t0 = time.perf_counter()
    kbar, vbar = oracle.pool(k, B), oracle.pool(v, B)
    t_pool = time.perf_counter() - t0
    q0 = int(case.cu_seqlens_q[r])
    done_w, t_rows, nblocks = 0.0, 0.0, 0
    order = rng.permutation(nqb)
    h = 0
    for i in order:
        rows = slice(i * B, min(lq, (i + 1) * B))
        qs = oracle.decode(case.q[q0 + rows.start:q0 + rows.stop], spec.dtype) * \
            case.q_scale.astype(np.float64)[None, :, None]
        I = start // B + i
        qstart = start + i * B            # the block seen as a request starting at its first query
        t0 = time.perf_counter()
        s = oracle.score_rows(qs, qstart, hkv, B, 1 / math.sqrt(spec.d), kbar, [h])[0]
        keep_row, _ = oracle.select_row(s, I, 0.1, B, 256, 512)
        keep = np.zeros((1, hkv, kbar.shape[0]), np.uint8)
        keep[0, h, :I + 1] = keep_row
        n = rows.stop - rows.start
        qi = np.repeat(np.arange(n), g)
        qh = np.tile(np.arange(h * g, (h + 1) * g), n)
        oracle.attn_rows(qs, qstart, k, v, kbar, vbar, B, 1 / math.sqrt(spec.d), keep, True, qi, qh)
        t_rows += time.perf_counter() - t0
        done_w += (I + 1) * (rows.stop - rows.start)
        nblocks += 1
        if time.perf_counter() - t_all > seconds:
            break
    total_w = 0.0
    for lq_, st_ in spec.requests:
        total_w += hkv * sum((st_ // B + i + 1) * min(B, lq_ - i * B) for i in range(-(-lq_ // B)))
    est_ms = (t_rows * total_w / done_w + t_pool * spec.total_k / k.shape[0]) * 1e3
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return est_ms, dict(kind="oracle", cores=threads,
                        sample=f"{nblocks} query blocks x 1 kv head of request {r} (full pooling), "
                               f"scaled by causal work to the whole layer",
                        sampled_seconds=round(t_rows + t_pool, 2))


def run_reference(args, rank, world):
    from block_sparse_long_fp_gb300 import synth
    spec = synth.config_spec(args.workload)
    case = synth.make_case(spec)
    flop = dense_equiv_flop(spec)
    per = max(2.0, args.cpu_seconds / max(1, args.steps + args.warmup))
    for w in range(args.warmup):
        oracle_sample(case, per, seed=100 + w)
    times = []
    info = None
    for s in range(args.steps):
        est_ms, info = oracle_sample(case, per, seed=s)
        times.append(est_ms)
    ms = statistics.median(times)
    value = flop / (ms * 1e-3) / 1e12
    info["value"] = value
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": spec.name, "batch": spec.batch, "seq_len": spec.total_q, "h_q": spec.h_q,
                       "h_kv": spec.h_kv, "d": spec.d, "page_size": spec.page_size, "alpha": 0.1,
                       "mean_correction": True},
            "cpu_baseline": info,
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", type=int, default=3)
    ap.add_argument("--logit-scale", type=float, default=1.0)
    ap.add_argument("--dtype", default="bf16", choices=["bf16", "e4m3"],
                    help="arithmetic of the main workload (the variants run only with bf16)")
    ap.add_argument("--dense-steps", type=int, default=3)
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-variants", dest="variants", action="store_false",
                    help="skip the sparse-regime and FP8 variants")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            import oracle
            oracle.build()
            print(json.dumps(run_reference(args, rank, world)))
        return
    from block_sparse_long_fp_gb300 import build as _b
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
        if rank == 0:
            _b.build()
        dist.barrier()
    else:
        _b.build()
    res, case = run_ours(args, rank, world)
    if rank == 0 and args.cpu_seconds > 0:
        import oracle
        oracle.build()
        est_ms, info = oracle_sample(case, args.cpu_seconds)
        info["value"] = round(dense_equiv_flop(case.spec) / (est_ms * 1e-3) / 1e12, 6)
        info["unit"] = UNIT
        info["ms_per_layer_est"] = round(est_ms, 1)
        res["cpu_baseline"] = info
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
