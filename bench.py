#!/usr/bin/env python3
"""Benchmark: bf16 fused attention forward on the long-sequence causal
workload (B=2, h=16, T_q=T_k=8192, d_k=d_v=64, Q/K/V ~ N(0,1)), reported as
TFLOP/s with causal FLOPs halved (4*B*h*d*T^2/2) and as a fraction of the
measured dense bf16 tensor peak.

    python bench.py [--gpus N --steps K --warmup W] [--impl reference]

One JSON line on stdout (rank 0).  With N > 1 (launched by torchrun) every
rank runs an independent replica of the workload on its own GPU (attention
shards over (batch, head) with no exchange step); the time is the maximum over
ranks and the value counts the work of all ranks.

--impl reference times the fp64 CPU oracle on this host's cores on a bounded
sample of the same workload (a deliberately slow baseline, not the target).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import seeded_inputs as si  # noqa: E402

WORKLOAD = si.WORKLOADS[4]  # sdpa_causal_bf16_B2_h16_T8192_d64
METRIC = "attention fwd TFLOP/s (bf16, 1 GB300) and % of dense BF16 tensor peak"
UNIT = "TFLOP/s"
DATASHEET_BF16_TFLOPS = 2500.0  # GB300 NVL72 dense bf16 / 72 GPUs
NOMINAL_BF16_TFLOPS = 2250.0
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
ATTN_SOURCE = os.path.join(ROOT, "transformer_scaled_dot_softmax_gb300", "csrc", "attn_bf16.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "attn_fwd_bf16_causal_B2_h16_T8192_traffic.json")
L2_FLUSH_BYTES = 256 << 20


def attention_flops(w: si.Workload, key_lens=None) -> float:
    """Algorithmic FLOPs: 2*d_k per score plus 2*d_v per weighted value, over
    visible (query, key) pairs; causal counts T^2/2 as the target states."""
    if w.mask & si.MASK_CAUSAL:
        pairs = w.T_q * w.T_k / 2.0
    else:
        pairs = float(w.T_q * w.T_k)
    return 2.0 * (w.d_k + w.d_v) * w.B * w.h * pairs


def row_flops(w: si.Workload, t: np.ndarray) -> float:
    """FLOPs of the given causal query rows (row t sees t+1 keys)."""
    return float(2.0 * (w.d_k + w.d_v) * np.sum(np.minimum(t + 1, w.T_k)))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return FALLBACK_PEAKS, "fallback"


def source_digest(path: str) -> str:
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def measured_traffic():
    """DRAM bytes per launch from the committed ncu summary, or None once the
    kernel source has changed since the counters were taken."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        rec = json.load(f)
    if rec.get("source_sha256") != source_digest(ATTN_SOURCE):
        return None
    return rec.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[4:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for _, _, r in rows:
            for n, v in zip(names, r[1:]):
                if v.lower() == "active":
                    reasons.add(n)
        sm = sorted(x[0] for x in rows)
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(x[1] for x in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


# --------------------------------------------------------------- CPU oracle
def oracle_sample_rows(w: si.Workload, stride: int, offset: int = 0):
    """Flat row indices (b*h + head)*T_q + t for every head and t = offset,
    offset + stride, ... (rows spread over the whole causal triangle)."""
    t = np.arange(offset % stride, w.T_q, stride, dtype=np.int64)
    bh = np.arange(w.B * w.h, dtype=np.int64)
    return (bh[:, None] * w.T_q + t[None, :]).reshape(-1), t


def time_oracle(x, w: si.Workload, stride: int, offset: int = 0):
    import oracle  # the CPU baseline leg is the one place the bench runs the oracle
    rows, t = oracle_sample_rows(w, stride, offset)
    flops = row_flops(w, t) * w.B * w.h
    t0 = time.perf_counter()
    oracle.sdpa_rows(x["q"], x["k"], x["v"], rows, scale=w.scale, mask=w.mask)
    dt = time.perf_counter() - t0
    return flops / dt / 1e12, dt, len(rows), oracle.num_threads()


def visible_keys(w: si.Workload, key_lens, b: np.ndarray, t: np.ndarray) -> np.ndarray:
    """Visible keys of query row t of batch entry b."""
    L = np.full(len(b), w.T_k) if key_lens is None else np.clip(np.asarray(key_lens)[b], 0, w.T_k)
    return np.minimum(t + 1, L) if w.mask & si.MASK_CAUSAL else L


def oracle_attention_by_workload(target_flops: float = 1.5e9):
    """The oracle's scaled dot-product attention on the attention shapes of
    workloads 1-4 (seeded N(0,1) Q/K/V of the projected (B, h, T, 64) shape,
    the workload's mask and key lengths), timed on one thread and on all
    cores over the same row sample: every n-th row, n chosen so the sample
    holds about `target_flops` (about a second on one core)."""
    import oracle
    cores = oracle.num_threads()
    res = {}
    try:
        for idx in range(4):
            wl = si.WORKLOADS[idx]
            w = si.WORKLOADS[4].replace(B=wl.B, h=wl.h, T_q=wl.T_q, T_k=wl.T_k, d_k=wl.d_k,
                                        d_v=wl.d_v, mask=wl.mask, len_lo=wl.len_lo,
                                        len_hi=wl.len_hi, seed=wl.seed, name=wl.name)
            x = si.make_inputs(w)
            nrows = w.B * w.h * w.T_q
            b_of = np.arange(nrows) // (w.h * w.T_q)
            t_of = np.arange(nrows) % w.T_q
            per_row = 2.0 * (w.d_k + w.d_v) * visible_keys(w, x["key_lens"], b_of, t_of)
            stride = max(1, int(per_row.sum() / target_flops))
            rows = np.arange(0, nrows, stride, dtype=np.int64)
            fl = float(per_row[rows].sum())
            entry = {"rows": int(len(rows)), "of_rows": nrows}
            for threads in (1, cores):
                oracle.set_num_threads(threads)
                t0 = time.perf_counter()
                oracle.sdpa_rows(x["q"], x["k"], x["v"], rows, scale=w.scale, mask=w.mask,
                                 key_lens=x["key_lens"])
                dt = time.perf_counter() - t0
                entry["threads_%d" % threads] = {"tflops": fl / dt / 1e12, "seconds": dt}
            res[wl.name] = entry
    finally:
        oracle.set_num_threads(cores)
    return res


def run_reference(args, rank: int, world: int) -> int:
    if rank != 0:
        return 0
    w = WORKLOAD
    x = si.make_inputs(w)
    stride = args.oracle_stride
    for i in range(args.warmup):
        time_oracle(x, w, stride * 4, i)
    vals, secs, nrows = [], 0.0, 0
    cores = 1
    for i in range(args.steps):
        v, dt, n, cores = time_oracle(x, w, stride, i)
        vals.append(v)
        secs += dt
        nrows += n
    value = float(np.mean(vals))
    sample = ("each step: all %d (batch, head) pairs x every %d-th query row of the causal "
              "T=8192 triangle (%d rows/step), fp64" % (w.B * w.h, stride, nrows // args.steps))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w: si.Workload):
    return {"workload": w.name, "B": w.B, "h": w.h, "T_q": w.T_q, "T_k": w.T_k, "d_k": w.d_k,
            "d_v": w.d_v, "mask": "causal", "scale": w.scale,
            "inputs": "Q/K/V ~ N(0,1), SplitMix64+Box-Muller seed %d, bf16" % w.seed,
            "l2": "flushed between timed steps (256 MiB write)"}


# ---------------------------------------------------------------- GPU path
def max_over_ranks(x: float, dist=None, device=None) -> float:
    """The slowest rank's figure (all ranks must call it)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(flops_per_rank: float, world: int, ms_max: float) -> float:
    """TFLOP/s of all ranks together: every rank runs one replica."""
    return world * flops_per_rank / (ms_max * 1e-3) / 1e12


def run_gpu(args, rank: int, world: int, local_rank: int) -> int:
    import torch
    import transformer_scaled_dot_softmax_gb300 as tsds

    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", rank=rank, world_size=world)
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = WORKLOAD
    x = si.make_inputs(w)

    def to_dev(bits):
        return torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)

    q, k, v = to_dev(x["q_bits"]), to_dev(x["k_bits"]), to_dev(x["v_bits"])
    out = torch.empty_like(q)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    flops = attention_flops(w)

    def step():
        tsds.sdpa_forward(q, k, v, out, scale=w.scale, mask="causal", status=status,
                          stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError("kernel reported status %d" % int(status.item()))

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local_rank) as clocks:
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    ms = np.array([s.elapsed_time(e) for s, e in zip(starts, ends)])
    if int(status.item()) != 0:
        raise RuntimeError("kernel reported status %d" % int(status.item()))
    ms_mean = max_over_ranks(float(ms.mean()), dist, dev)
    value = whole_job_value(flops, world, ms_mean)

    # Beside the cold-L2 figure: the same launches back to back without the
    # flush (Q, K, V, O = 128 MiB, about the size of L2, stay partly resident).
    n_warm = min(args.steps, 100)
    ws_, we_ = ([torch.cuda.Event(enable_timing=True) for _ in range(n_warm)] for _ in range(2))
    for i in range(n_warm):
        ws_[i].record(stream)
        step()
        we_[i].record(stream)
    torch.cuda.synchronize(dev)
    warm_ms = max_over_ranks(float(np.mean([a.elapsed_time(b) for a, b in zip(ws_, we_)])), dist, dev)
    warm = {"ms_mean": warm_ms, "value": whole_job_value(flops, world, warm_ms), "unit": UNIT,
            "steps": n_warm, "l2": "not flushed between steps"}

    # End to end through the public API with host buffers: pinned host Q/K/V
    # -> device, attention, output -> pinned host, every step.
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, q, k, v, out, w, stream, dev, dist, flops, world)

    others = None
    if rank == 0 and not args.no_other_workloads:
        others = time_other_workloads(dev, stream, flush)
    if rank == 0:
        emit(args, w, x, ms, ms_mean, value, flops, world, clocks, e2e, others, warm)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def visible_pairs(w: si.Workload, key_lens) -> float:
    """Exact number of visible (query, key) pairs of a workload."""
    total = 0.0
    for b in range(w.B):
        L = w.T_k if key_lens is None else int(min(max(key_lens[b], 0), w.T_k))
        if w.mask & si.MASK_CAUSAL:
            i = np.arange(w.T_q)
            total += float(np.minimum(i + 1, L).sum())
        else:
            total += float(w.T_q) * L
    return total * w.h


def mha_flops(w: si.Workload, key_lens) -> float:
    """Projections (2 M K N each) plus attention over visible pairs."""
    hd = w.h * w.d_k
    proj = 2.0 * w.B * w.T_q * w.d_model * hd + 2.0 * 2 * w.B * w.T_k * w.d_model * hd \
        + 2.0 * w.B * w.T_q * hd * w.d_model
    return proj + 2.0 * (w.d_k + w.d_v) * visible_pairs(w, key_lens)


def time_other_workloads(dev, stream, flush, iters=20):
    """The other workloads of the table: fp32 SDPA latency, the three MHA
    forwards end to end (three launches; alone and with the residual +
    layer normalisation of the sublayer) and the decode step, device-resident
    inputs, L2 flushed between calls, CUDA events around each call."""
    import torch
    import transformer_scaled_dot_softmax_gb300 as tsds

    def dv(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(
            torch.bfloat16)

    def timed(fn):
        for _ in range(3):
            flush.zero_()
            fn()
        ev = []
        for _ in range(iters):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            ev.append((a, b))
        torch.cuda.synchronize(dev)
        return float(np.median([a.elapsed_time(b) for a, b in ev]))

    res = {}
    w = si.WORKLOADS[0]
    x = si.make_inputs(w)
    q, k, v = (torch.from_numpy(x[n].astype(np.float32)).to(dev) for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    ms = timed(lambda: tsds.sdpa_forward(q, k, v, o, scale=w.scale, stream=stream))
    res[w.name] = {"ms": ms, "us": 1e3 * ms, "kind": "fp32 SIMT SDPA (register kernel for T_k <= 32): one memory round trip + launch latency"}
    for w in si.WORKLOADS[1:4]:
        x = si.make_inputs(w)
        xq = dv(x["x_q_bits"])
        xkv = dv(x["x_kv_bits"]) if w.cross else xq
        wts = [dv(x[n + "_bits"]) for n in ("w_q", "w_k", "w_v", "w_o")]
        lens = None if x["key_lens"] is None else torch.from_numpy(x["key_lens"]).to(dev)
        out = torch.empty((w.B, w.T_q, w.d_model), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(tsds.mha_workspace_bytes(w.B, w.h, w.T_q, w.T_k), dtype=torch.uint8,
                         device=dev)
        ms = timed(lambda: tsds.mha_forward(xq, xkv, *wts, h=w.h, out=out, workspace=ws,
                                            scale=w.scale, mask=w.mask, key_lens=lens,
                                            stream=stream))
        fl = mha_flops(w, x["key_lens"])
        res[w.name] = {"ms": ms, "tflops": fl / (ms * 1e-3) / 1e12, "flops": fl,
                       "kind": "bf16 MHA forward: grouped QKV GEMM + fused attention + W^O GEMM"}
        ln = si.layernorm_params(w.seed, w.d_model)
        g, bt = dv(ln["gamma_bits"]), dv(ln["beta_bits"])
        ms_ln = timed(lambda: tsds.mha_forward_add_layernorm(
            xq, xkv, *wts, g, bt, h=w.h, out=out, workspace=ws, scale=w.scale, mask=w.mask,
            key_lens=lens, stream=stream))
        res[w.name + "_add_layernorm"] = {
            "ms": ms_ln, "tflops": fl / (ms_ln * 1e-3) / 1e12, "flops": fl,
            "kind": "LayerNorm(x + MHA(x)): W^O GEMM with residual add and normalisation "
                    "in its epilogue (cluster per 128-row block)"}
    # one encoder layer of the base model (attention + FFN sublayers, both normalised)
    w = si.WORKLOADS[6]
    x = si.make_inputs(w)
    F = si.ENCODER_D_FF
    ep = si.encoder_params(w.seed, w.d_model, F)
    params = {n: dv(ep[n + "_bits"]) for n in ("gamma1", "beta1", "w1", "b1", "w2", "b2", "gamma2",
                                               "beta2")}
    for n in ("w_q", "w_k", "w_v", "w_o"):
        params[n] = dv(x[n + "_bits"])
    xe = dv(x["x_q_bits"])
    lens = torch.from_numpy(x["key_lens"]).to(dev)
    oute = torch.empty_like(xe)
    wse = torch.empty(int(tsds.lib.encoder_layer_workspace_bytes(w.B, w.T_q, w.d_model, w.h, F)),
                      dtype=torch.uint8, device=dev)
    ms = timed(lambda: tsds.encoder_layer_forward(xe, params, w.h, oute, wse, scale=w.scale,
                                                  mask=w.mask, key_lens=lens, stream=stream))
    fl = mha_flops(w, x["key_lens"]) + 4.0 * w.B * w.T_q * w.d_model * F
    res[w.name] = {"ms": ms, "tflops": fl / (ms * 1e-3) / 1e12, "flops": fl,
                   "kind": "one post-LN encoder layer: MHA + FFN (d_ff 2048), 5 launches; "
                           "FLOPs = projections + visible-pair attention + the two FFN GEMMs"}
    del xe, oute, wse, params

    # backward of the headline workload (dq, dk, dv from q, k, v, o, lse, dO)
    w = si.WORKLOADS[4]
    x = si.make_inputs(w)
    q, k, v = dv(x["q_bits"]), dv(x["k_bits"]), dv(x["v_bits"])
    g = dv(si.f64_to_bf16_bits(si.round_bf16(si.normal(w.seed, si.TENSOR_IDS["dout"], q.shape))))
    o, lse = tsds.sdpa_forward_lse(q, k, v, scale=w.scale, mask="causal", stream=stream)
    ws = torch.empty(int(tsds.lib.sdpa_backward_workspace_bytes(w.B, w.h, w.T_q, w.T_k, 64, 64)),
                     dtype=torch.uint8, device=dev)
    dq, dk, dvv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ms = timed(lambda: tsds.sdpa_backward(q, k, v, o, g, lse, dq, dk, dvv, ws, scale=w.scale,
                                          mask="causal", stream=stream))
    fl = 2.5 * attention_flops(w)
    res[w.name + "_backward"] = {
        "ms": ms, "tflops": fl / (ms * 1e-3) / 1e12, "flops": fl,
        "kind": "bf16 attention backward (dq, dk, dv): 5 products per key/query tile pair = "
                "2.5x the forward's FLOPs; row terms + tcgen05 kernel + dq conversion"}
    del q, k, v, g, o, lse, ws, dq, dk, dvv

    w = si.WORKLOADS[5]
    x = si.make_inputs(w)
    q, k, v = dv(x["q_bits"]), dv(x["k_bits"]), dv(x["v_bits"])
    lens = torch.from_numpy(x["key_lens"]).to(dev)
    o = torch.empty_like(q)
    ms = timed(lambda: tsds.sdpa_decode_forward(q, k, v, lens, o, scale=w.scale, stream=stream))
    nbytes = decode_bytes(w, x["key_lens"])
    gbs = nbytes / (ms * 1e-3) / 1e9
    peaks, peak_kind = load_peaks()
    peak = peaks.get("hbm_gbs")
    res[w.name] = {"ms": ms, "us": 1e3 * ms, "gbs": gbs, "bytes": nbytes,
                   "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                                "frac": gbs / peak if peak else None,
                                "peak_source": peak_kind + " copy bandwidth"},
                   "kind": "bf16 decode attention: 8-CTA cluster per (b, h), HBM-bound"}
    return res


def decode_bytes(w, key_lens) -> int:
    """Algorithmic bytes of one decode call: every visible cached key and
    value row read once, the query rows read and the output rows written."""
    lens = np.full(w.B, w.T_k) if key_lens is None else np.clip(key_lens, 0, w.T_k)
    row = 2 * w.d_k
    return int(w.h * (lens.sum() * 2 * row + w.B * w.T_q * 2 * row))


def run_e2e(args, q, k, v, out, w, stream, dev, dist, flops, world):
    import torch
    import transformer_scaled_dot_softmax_gb300 as tsds
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    ws = torch.empty(tsds.sdpa_forward_host_workspace_bytes(w.B, w.h, w.T_q, w.T_k, w.d_k, w.d_v),
                     dtype=torch.uint8, device=dev)
    e2e_steps = max(3, min(args.steps, 20))

    def e2e_step():
        # one C-ABI call with host buffers: chunked host->device copies,
        # attention and device->host copy of the output, overlapped
        tsds.sdpa_forward_host(hq, hk, hv, hout, ws, scale=w.scale, mask="causal", stream=stream)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dist, dev)
    e2e_value = whole_job_value(flops, world, e2e_ms)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = hout.numel() * hout.element_size()
    return {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}


def emit(args, w, x, ms, ms_mean, value, flops, world, clocks, e2e, others=None, warm=None):
    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    achieved = flops / (float(ms.mean()) * 1e-3) / 1e12
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cv, cdt, cn, cores = time_oracle(x, w, args.oracle_stride)
        cpu = {"value": cv, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": "all %d (batch, head) pairs x every %d-th query row of the causal "
                         "T=8192 triangle (%d rows, %.1f s), fp64"
                         % (w.B * w.h, args.oracle_stride, cn, cdt),
               "attention_by_workload": oracle_attention_by_workload()}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_mean,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": workload_config(w),
        "pct_of_dense_bf16_peak": {
            "measured_%.1f" % peak: 100.0 * achieved / peak,
            "nominal_%.0f" % NOMINAL_BF16_TFLOPS: 100.0 * achieved / NOMINAL_BF16_TFLOPS,
            "datasheet_%.0f" % DATASHEET_BF16_TFLOPS: 100.0 * achieved / DATASHEET_BF16_TFLOPS},
        "roofline": {"kernel": "attn_fwd_bf16_kernel", "bound": "tensor",
                     "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "peak_source": peak_src + " burst bf16",
                     "flops_per_launch": flops, "traffic": measured_traffic()},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clocks.summary(),
        "ms_min": float(ms.min()), "ms_median": float(np.median(ms)),
        "warm_l2": warm,
        "other_workloads": others,
    }
    print(json.dumps(line), flush=True)


def parse(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--oracle-stride", type=int, default=1,
                    help="CPU baseline: time every n-th query row of every head")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="skip timing the fp32 SDPA and the three MHA workloads")
    ap.add_argument("--shape", default=None,
                    help="B,h,T override of the causal workload (profiling and sweeps only; "
                         "the reported line then names the changed workload)")
    return ap.parse_args(argv)


def main(argv=None) -> int:
    args = parse(argv)
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus and world != 1:
        raise SystemExit("--gpus %d does not match WORLD_SIZE %d" % (args.gpus, world))
    global WORKLOAD
    if args.shape:
        B, h, T = (int(v) for v in args.shape.split(","))
        WORKLOAD = WORKLOAD.replace(B=B, h=h, T_q=T, T_k=T,
                                    name="sdpa_causal_bf16_B%d_h%d_T%d_d64" % (B, h, T))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    return run_gpu(args, rank, world, local_rank)


if __name__ == "__main__":
    sys.exit(main())
