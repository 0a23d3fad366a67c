"""Benchmark of the decode-step hot path on GB300.

Workload (one "step"): one slow-AR decoder-layer step under continuous batching at bs=64:
RMSNorm+MXFP8 quantise -> QKV projection -> KV append -> GQA decode attention (32 q /
8 kv heads, head_dim 128, cap 32768, ragged kv_len ~ U[234, 4096] with a seeded
retire/refill schedule) -> quantise -> O projection + residual -> RMSNorm+quantise ->
MXFP8 SwiGLU MLP (Qwen3-4B shape 2560/9728) + residual -> prev_tokens_shift [64,16,10].

metric/unit: HBM GB/s = algorithmic bytes of the step / step time (the step's KV reads,
weights and activations, counted per kernel by the *_bytes functions below). The line also
carries the MLP-only sweep (M = 1..128: us and GB/s), the attention-only sweep (bs = 1..64:
GB/s), the paged-attention sweep (bs = 64, pages of 64/128/256), the MXFP8-KV attention sweep
(bs = 1..64 and paged), the prefill / extend attention sweep (TFLOP/s), the block-scaled FP8
(bsgemm) sweep and the square MXFP8 GEMM sweep, each timed the same way.

Timing: W untimed warm-up steps, then K steps each bracketed by CUDA events on the
launching stream, with an L2 flush between steps (outside the events: 256 MiB written, then
another 256 MiB read, so the step starts with clean, unrelated lines in the 129 MB L2);
barrier + synchronize around the timed loop; max over ranks.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs an independent replica (replicas only; no collective on
the data path) and rank 0 prints one JSON line.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MXFP8 SwiGLU-MLP decode µs + HBM GB/s (M=1–128); GQA decode attn GB/s"
BS, D_MODEL, D_FF, HQ, HKV, HD, CAP, W_WIN, CW = 64, 2560, 9728, 32, 8, 128, 32768, 16, 10
KV_LO, KV_HI, LIFE_HI, EPS = 234, 4096, 256, 1e-6
WORKLOAD = ("slow-AR decode-layer step, bs=64: RMSNorm+MXFP8 quant, QKV 2560->6144, KV append, GQA decode attn "
            "32q/8kv x128 over cap 32768 with ragged kv_len~U[234,4096] (seeded retire/refill), O 4096->2560 "
            "+res, RMSNorm+quant, MXFP8 SwiGLU MLP 2560/9728 +res, prev_tokens_shift [64,16,10]")


# --------------------------------------------------------------------------- byte counts
def mlp_bytes(M, d=D_MODEL, dff=D_FF, residual=False):
    """Algorithmic HBM bytes of the MXFP8 MLP: weights once, xq/xs read, hq/hs written and
    read back, y written (+ residual read)."""
    w = 2 * dff * d * (1 + 1 / 32) + d * dff * (1 + 1 / 32)
    act = M * d * (1 + 1 / 32) + 2 * M * dff * (1 + 1 / 32) + M * d * 2 + (M * d * 2 if residual else 0)
    return int(w + act)


def attn_bytes(kv_lens, Hq=HQ, Hkv=HKV, D=HD):
    """K and V rows of every active prefix once, plus q read and o written."""
    kv = int(np.sum(kv_lens)) * Hkv * D * 2 * 2
    return kv + len(kv_lens) * Hq * D * 2 * 2


def attn_kv_mxfp8_bytes(kv_lens, Hq=HQ, Hkv=HKV, D=HD):
    """MXFP8 K and V rows (E4M3 codes + one UE8M0 byte per 32) of every active prefix once,
    plus q read and o written (bf16)."""
    kv = int(np.sum(kv_lens)) * Hkv * (D + D // 32) * 2
    return kv + len(kv_lens) * Hq * D * 2 * 2


def prefill_flops(prefix, new, Hq=HQ, D=HD):
    """Causal prefill / extend attention flop: new token i of a sequence with P cached positions
    sees P + i + 1 keys, 2 D flop each for q.k and for p.v, per query head."""
    p, t = np.asarray(prefix, np.float64), np.asarray(new, np.float64)
    return float(np.sum(4.0 * D * Hq * (t * p + t * (t + 1) / 2)))


def gemm_bytes(M, N, K, residual=False):
    return int(N * K * (1 + 1 / 32) + M * K * (1 + 1 / 32) + M * N * 2 + (M * N * 2 if residual else 0))


def step_bytes(kv_lens, bs=BS):
    """Algorithmic HBM bytes of one decode-layer step, per fused kernel of the step."""
    d, qd = D_MODEL, HQ * HD
    nqkv = (HQ + 2 * HKV) * HD
    parts = {
        "rmsnorm_quant_1": bs * d * 2 + d * 2 + bs * d * (1 + 1 / 32),
        # weights + activations in; q written to the qkv buffer, K/V rows written to the cache
        "qkv_gemm_kv_append": gemm_bytes(bs, nqkv, d),
        # K/V prefixes + q in; o (bf16) and its MXFP8 copy out
        "attention_quant": attn_bytes(kv_lens) + bs * qd * (1 + 1 / 32),
        "o_gemm": gemm_bytes(bs, d, qd, residual=True),
        "rmsnorm_quant_2": bs * d * 2 + d * 2 + bs * d * (1 + 1 / 32),
        "mlp": mlp_bytes(bs, residual=True),
        "prev_shift": bs * W_WIN * CW * 4 * 2 + bs * CW * 4,
    }
    return {k: int(v) for k, v in parts.items()}


# --------------------------------------------------------------------------- distributed helpers
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a per-rank float over all ranks (identity when world == 1)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while active."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# DRAM traffic of the attention split kernel per algorithmic byte, from one ncu capture of the
# same kernel on a smaller cache (the bs-64, 4096-position capture: 634.68 MB of
# dram__bytes_read.sum + dram__bytes_write.sum for 622.54 MB of algorithmic bytes). Traffic
# grows in proportion to the prefix tokens read, so it is scaled to the step's launch. Set to
# None whenever the kernel changes until it is captured again.
ATTN_TRAFFIC_PER_ALG_BYTE = 634.677248e6 / 622538752


# --------------------------------------------------------------------------- measured peaks
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# --------------------------------------------------------------------------- our arm
def build_layer(dev, max_kv_len):
    import torch

    from mxfp8_mlp_gqa_gb300.step import DecodeLayer

    L = DecodeLayer(BS, D_MODEL, D_FF, HQ, HKV, HD, CAP, max_kv_len, W_WIN, CW, eps=EPS, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(0)

    def randn(shape, std=1.0, mean=0.0):
        return (torch.randn(shape, generator=g, device=dev, dtype=torch.float32) * std + mean).to(torch.bfloat16)

    nqkv = (HQ + 2 * HKV) * HD
    L.load_weights(randn((nqkv, D_MODEL), 0.02), randn((D_MODEL, HQ * HD), 0.02), randn((2 * D_FF, D_MODEL), 0.02),
                   randn((D_MODEL, D_FF), 0.02), randn((D_MODEL,), 0.1, 1.0), randn((D_MODEL,), 0.1, 1.0))
    # K/V ~ N(0,1) for the whole cache (prefixes and the rows later steps append into),
    # generated in slices to bound the temporary
    for c in (L.k_cache, L.v_cache):
        for b in range(BS):
            c[b].copy_(randn(c[b].shape))
    L.x.copy_(randn((BS, D_MODEL)))
    L.prev.copy_(torch.randint(0, 4096, (BS, W_WIN, CW), generator=g, device=dev, dtype=torch.int32))
    L.next_tokens.copy_(torch.randint(0, 4096, (BS, CW), generator=g, device=dev, dtype=torch.int32))
    return L


def timed_ops(L, ev):
    """The kernels of one step in order on one stream, with an event after each (the step
    proper forks the prev-window shift onto a second stream; here it runs last)."""
    from mxfp8_mlp_gqa_gb300 import api

    qd = L.Hq * L.D
    ev[0].record()
    api.rmsnorm_mxfp8_quantize(L.x, L.gamma1, L.eps, q=L.xq, s=L.xs)
    ev[1].record()
    api.mxfp8_gemm_qkv_kv_append(L.xq, L.xs, *L.wqkv, L.Hq, L.Hkv, L.k_cache, L.v_cache, L.kv_len, qkv=L.qkv,
                                 err=L.err)
    ev[2].record()
    api.gqa_decode_attn(L.qkv[:, :qd], L.k_cache, L.v_cache, L.kv_len, L.max_kv_len, L.scale, out=L.o, err=L.err,
                        workspace=L.ws_attn, oq=L.oq, os=L.os)
    ev[3].record()
    api.mxfp8_gemm(L.oq, L.os, *L.wo, residual=L.x, c=L.x1, workspace=L.ws_o)
    ev[4].record()
    api.rmsnorm_mxfp8_quantize(L.x1, L.gamma2, L.eps, q=L.hq_in, s=L.hs_in)
    ev[5].record()
    api.mlp_swiglu_mxfp8(L.hq_in, L.hs_in, *L.w13, *L.w2, residual=L.x1, y=L.y, workspace=L.ws_mlp)
    ev[6].record()
    api.prev_tokens_shift(L.prev, L.next_tokens)
    ev[7].record()


OP_NAMES = ["rmsnorm_quant_1", "qkv_gemm_kv_append", "attention_quant", "o_gemm", "rmsnorm_quant_2", "mlp",
            "prev_shift"]
NEV = len(OP_NAMES) + 1


def launches_per_step(max_kv_len):
    from mxfp8_mlp_gqa_gb300 import api

    attn = 2 if api.gqa_decode_attn_workspace(BS, HQ, HKV, HD, max_kv_len) > 0 else 1
    return 1 + 1 + attn + 1 + 1 + 2 + 1  # rmsnorm, qkv+append, attention(+combine), o, rmsnorm, mlp, shift


def run_ours(args, rank, local_rank, world):
    import torch

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    from mxfp8_mlp_gqa_gb300 import api, synth

    api.lib()
    total_steps = args.warmup + args.steps
    sched, refill = synth.slot_schedule(BS, total_steps + 1, KV_LO, KV_HI, LIFE_HI, seed=0)
    max_kv_len = int(sched.max())
    L = build_layer(dev, max_kv_len)
    sched_d = torch.from_numpy(sched).to(dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)

    def admit(s):
        # between steps (untimed): a slot retired by the schedule takes a new request -- its
        # prompt's K/V rows (positions 0 .. kv_len-2, what the prefill leaves) and a zeroed
        # prev window
        for b in np.nonzero(refill[s])[0]:
            n = int(sched[s][b]) - 1
            for c in (L.k_cache, L.v_cache):
                c[b, :, :n].copy_(torch.randn((HKV, n, HD), generator=gen, device=dev).to(torch.bfloat16))
            L.prev[b].zero_()
    flush = L2Flush(dev)
    peak_gbs, peak_src = measured_peaks()

    # one eager step (lazy initialisation), then the step is captured in a CUDA graph with a
    # timing event between consecutive kernels, so that per-kernel times are device times
    # without host enqueue gaps
    L.kv_len.copy_(sched_d[0])
    L.step()
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(NEV)]
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            timed_ops(L, evs)
    torch.cuda.current_stream().wait_stream(cap)
    plain = L.capture()  # the same step without event nodes: the headline timing
    for s in range(args.warmup):
        admit(s)
        L.kv_len.copy_(sched_d[s])
        plain.replay()
        graph.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    step_ms = []
    for i in range(args.steps):
        admit(args.warmup + i)                # retire / refill per the schedule, not timed
        L.kv_len.copy_(sched_d[args.warmup + i])   # schedule advance, not timed
        flush()                               # L2 flush, not timed
        e0.record()
        plain.replay()
        e1.record()
        e1.synchronize()
        step_ms.append(e0.elapsed_time(e1))
    # per-kernel device times: the evented graph over the same schedule rows
    per_op = {n: [] for n in OP_NAMES}
    ev_step_ms = []
    for i in range(args.steps):
        L.kv_len.copy_(sched_d[args.warmup + i])
        flush()
        graph.replay()
        evs[NEV - 1].synchronize()
        for k, n in enumerate(OP_NAMES):
            per_op[n].append(evs[k].elapsed_time(evs[k + 1]))
        ev_step_ms.append(evs[0].elapsed_time(evs[NEV - 1]))
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    assert int(L.err.item()) == 0, f"device error flag {int(L.err.item())}"

    tot_ms = max_over_ranks(sum(step_ms), world, dev)
    bytes_steps = [step_bytes(sched[args.warmup + i]) for i in range(args.steps)]
    tot_bytes = sum(sum(b.values()) for b in bytes_steps)
    value = world * tot_bytes / (tot_ms * 1e-3) / 1e9
    attn_bytes_avg = statistics.mean(b["attention_quant"] for b in bytes_steps)
    attn_ms = statistics.mean(per_op["attention_quant"])
    breakdown = {}
    for n in OP_NAMES:
        ms = statistics.mean(per_op[n])
        by = statistics.mean(b[n] for b in bytes_steps)
        breakdown[n] = {"us": round(ms * 1e3, 2), "GB_s": round(by / (ms * 1e-3) / 1e9, 1), "bytes": int(by)}

    # e2e through the public API with host buffers: every step one graph holding the copy of
    # the step's packed inputs (x, next tokens, kv_len) from pinned host memory, the step and
    # the copy of y back to pinned host memory; the host fills the input buffer between steps
    h_in, (x_h, nxt_h, lens_h), y_h = L.host_io()
    x_h.copy_(L.x.cpu())
    nxt_h.copy_(L.next_tokens.cpu())
    L.capture_io(h_in, y_h)
    for s in range(2):  # graph upload and first-launch costs stay out of the timing
        lens_h.copy_(torch.from_numpy(sched[args.warmup + s]))
        L.replay_io()
    torch.cuda.synchronize()
    e_ms = []
    for i in range(args.steps):
        lens_h.copy_(torch.from_numpy(sched[args.warmup + i]))
        flush()
        e0.record()
        L.replay_io()
        e1.record()
        e1.synchronize()
        e_ms.append(e0.elapsed_time(e1))
    e2e_ms = max_over_ranks(sum(e_ms), world, dev)
    h2d = h_in.numel()
    d2h = y_h.numel() * 2
    e2e = {"value": round(world * tot_bytes / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms / args.steps, 4)}

    # eager (uncaptured) launches of the same step, for context: includes host enqueue time
    g_ms = []
    for i in range(args.steps):
        L.kv_len.copy_(sched_d[args.warmup + i])
        flush()
        e0.record()
        L.step()
        e1.record()
        e1.synchronize()
        g_ms.append(e0.elapsed_time(e1))

    sweeps = {} if args.no_sweeps else run_sweeps(dev, flush)
    return {
        "value": value, "ms_per_step": tot_ms / args.steps, "clocks": clk, "breakdown": breakdown, "e2e": e2e,
        "eager_ms_per_step": statistics.mean(g_ms), "evented_ms_per_step": statistics.mean(ev_step_ms),
        "roofline": {"kernel": "gqa_split_kernel + gqa_combine_kernel (attention with fused MX quant)",
                     "bound": "hbm",
                     "achieved": round(attn_bytes_avg / (attn_ms * 1e-3) / 1e9, 1), "peak": peak_gbs,
                     "peak_source": peak_src, "unit": "GB/s",
                     "frac": round(attn_bytes_avg / (attn_ms * 1e-3) / 1e9 / peak_gbs, 4),
                     "traffic": (None if ATTN_TRAFFIC_PER_ALG_BYTE is None
                                 else int(attn_bytes_avg * ATTN_TRAFFIC_PER_ALG_BYTE)),
                     "traffic_unit": "bytes per launch (ncu, scaled from a smaller capture)",
                     "bytes_per_launch": int(attn_bytes_avg), "us_per_launch": round(attn_ms * 1e3, 2)},
        "gpu_launches": launches_per_step(max_kv_len) * args.steps,
        "sweeps": sweeps,
    }


class L2Flush:
    """Called between timed launches, outside the events: writes a 256 MiB buffer (the L2 holds
    129 MB), then reads a second 256 MiB buffer, so the timed kernels start with an L2 full of
    clean, unrelated lines -- their inputs are cold, and they are not charged for writing back
    the flush's own dirty lines (that write-back alone costs ~8 us of a decode step; a serving
    loop's previous layer leaves clean lines behind)."""

    def __init__(self, dev, mib=256):
        import torch

        self.w = torch.empty(mib << 20, dtype=torch.uint8, device=dev)
        self.r = torch.ones((mib << 20) // 8, dtype=torch.int64, device=dev)
        self.acc = torch.zeros(1, dtype=torch.int64, device=dev)

    def __call__(self):
        self.w.zero_()
        self.acc.add_(self.r.sum())


def _time_op(fn, flush, reps=30, warm=3):
    import torch

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(warm):
        fn()
    out = []
    for _ in range(reps):
        flush()
        # keep the GPU busy (~20 us) while the host enqueues fn, so that host-side work (argument
        # checks, tensor-map encoding, the launch) stays outside the device-timed interval
        torch.cuda._sleep(40000)
        e0.record()
        fn()
        e1.record()
        e1.synchronize()
        out.append(e0.elapsed_time(e1))
    # the event clock ticks in ~2 us steps on this part: the mean over many launches resolves
    # finer than any single interval (the median would stay on the grid)
    return statistics.fmean(out)


def run_sweeps(dev, flush):
    import torch

    from mxfp8_mlp_gqa_gb300 import api, synth

    g = torch.Generator(device=dev)
    g.manual_seed(1)
    rn = lambda shape, std=1.0: (torch.randn(shape, generator=g, device=dev) * std).to(torch.bfloat16)  # noqa: E731
    w13 = api.mxfp8_quantize(rn((2 * D_FF, D_MODEL), 0.02))
    w2 = api.mxfp8_quantize(rn((D_MODEL, D_FF), 0.02))
    mlp = {}
    for M in (1, 2, 4, 8, 16, 32, 64, 128):
        xq, xs = api.mxfp8_quantize(rn((M, D_MODEL)))
        y = torch.empty((M, D_MODEL), dtype=torch.bfloat16, device=dev)
        ws = torch.zeros(api.mlp_swiglu_mxfp8_workspace(M, D_MODEL, D_FF), dtype=torch.uint8, device=dev)
        ms = _time_op(lambda: api.mlp_swiglu_mxfp8(xq, xs, *w13, *w2, y=y, workspace=ws), flush)
        mlp[str(M)] = {"us": round(ms * 1e3, 2), "GB_s": round(mlp_bytes(M) / (ms * 1e-3) / 1e9, 1)}
    del w13, w2
    attn = {}
    cap = 32768
    K = torch.empty((64, HKV, cap, HD), dtype=torch.bfloat16, device=dev)
    V = torch.empty_like(K)
    for b in range(64):
        K[b].copy_(rn(K[b].shape))
        V[b].copy_(rn(V[b].shape))
    for bs in (1, 8, 16, 32, 64):
        lens = synth.kv_lens(bs, KV_LO, KV_HI, seed=0)
        q = rn((bs, HQ, HD))
        kl = torch.from_numpy(lens).to(dev)
        out = torch.empty((bs, HQ, HD), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(max(1, api.gqa_decode_attn_workspace(bs, HQ, HKV, HD, KV_HI)), dtype=torch.uint8, device=dev)
        Kb, Vb = K[:bs], V[:bs]
        ms = _time_op(lambda: api.gqa_decode_attn(q, Kb, Vb, kl, KV_HI, 1 / math.sqrt(HD), out=out, workspace=ws),
                      flush)
        attn[str(bs)] = {"us": round(ms * 1e3, 2), "GB_s": round(attn_bytes(lens) / (ms * 1e-3) / 1e9, 1)}
    del K, V
    return {"mlp_M": mlp, "attn_bs": attn, "attn_paged_bs64": paged_attn_sweep(dev, rn, flush),
            "attn_kv_mxfp8_bs": kv_mxfp8_attn_sweep(dev, rn, flush), "prefill": prefill_sweep(dev, rn, flush),
            "bsgemm": bsgemm_sweep(dev, rn, flush),
            "gemm_square": gemm_square_sweep(dev), "context": context_rows(dev, rn, flush)}


def context_rows(dev, rn, flush):
    """Context only, not targets: the same work through torch's own kernels on this machine.
    (1) The decode MLP in bf16 (F.linear, SiLU, F.linear: 2x the weight bytes of MXFP8) at
    M = 1 / 64 / 128. (2) Decode attention at bs = 8 through scaled_dot_product_attention with
    GQA: over the whole 32768-position cache with a mask (the baseline of the KV-cache write-up's
    section 4) and over the prefix up to the batch's longest kv_len, ragged rows masked (its
    section 5); both against this library's call on the same lengths."""
    import torch
    import torch.nn.functional as F

    from mxfp8_mlp_gqa_gb300 import api, synth

    out = {}
    w13 = rn((2 * D_FF, D_MODEL), 0.02)
    w2 = rn((D_MODEL, D_FF), 0.02)
    for M in (1, 64, 128):
        x = rn((M, D_MODEL))

        def mlp_bf16():
            gu = F.linear(x, w13)
            return F.linear(F.silu(gu[:, :D_FF]) * gu[:, D_FF:], w2)

        ms = _time_op(mlp_bf16, flush)
        out[f"torch_bf16_mlp_M{M}"] = {"us": round(ms * 1e3, 2)}
    del w13, w2
    bs, cap = 8, 32768
    lens = synth.kv_lens(bs, KV_LO, KV_HI, seed=0)
    K = rn((bs, HKV, cap, HD))
    V = rn((bs, HKV, cap, HD))
    q = rn((bs, HQ, HD))
    pos = torch.arange(cap, device=dev)
    kl = torch.from_numpy(lens).to(dev)
    scale = 1 / math.sqrt(HD)
    mask_full = (pos[None, :] < kl[:, None])[:, None, None, :]
    lmax = int(lens.max())
    mask_pre = mask_full[..., :lmax]
    q4 = q[:, :, None, :]
    try:
        ms_full = _time_op(lambda: F.scaled_dot_product_attention(q4, K, V, attn_mask=mask_full, scale=scale,
                                                                   enable_gqa=True), flush)
        ms_pre = _time_op(lambda: F.scaled_dot_product_attention(q4, K[:, :, :lmax], V[:, :, :lmax],
                                                                  attn_mask=mask_pre, scale=scale, enable_gqa=True),
                          flush)
        out["torch_sdpa_bs8_full_cache_masked"] = {"us": round(ms_full * 1e3, 2)}
        out["torch_sdpa_bs8_prefix_masked"] = {"us": round(ms_pre * 1e3, 2)}
    except Exception as ex:  # noqa: BLE001 - context only
        out["torch_sdpa"] = f"unavailable: {type(ex).__name__}"
    o = torch.empty((bs, HQ, HD), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(max(1, api.gqa_decode_attn_workspace(bs, HQ, HKV, HD, KV_HI)), dtype=torch.uint8, device=dev)
    ms = _time_op(lambda: api.gqa_decode_attn(q, K, V, kl, KV_HI, scale, out=o, workspace=ws), flush)
    out["ours_attn_bs8"] = {"us": round(ms * 1e3, 2)}
    return out


def bsgemm_bytes(M, N, K):
    """Block-scaled FP8 GEMM: E4M3 weights + one fp32 scale per 128x128 block, E4M3 activations
    + one fp32 scale per 1x128 block, bf16 out."""
    return int(N * K + ((N + 127) // 128) * (K // 128) * 4 + M * K + M * (K // 128) * 4 + M * N * 2)


def bsgemm_sweep(dev, rn, flush):
    """bsgemm recipe at the decode MLP's two weight shapes (gate/up 19456x2560, down
    2560x9728), next to the MXFP8 GEMM on the same shapes: us and GB/s of each format's bytes."""
    import torch

    from mxfp8_mlp_gqa_gb300 import api

    res = {}
    for name, (N, K) in {"gate_up": (2 * D_FF, D_MODEL), "down": (D_MODEL, D_FF)}.items():
        wb = rn((N, K), 0.02)
        wq, ws = api.bs_quantize_weight(wb)
        mq, ms_ = api.mxfp8_quantize(wb)
        del wb
        for M in (1, 16, 64, 128):
            x = rn((M, K))
            xq, xs = api.bs_quantize_act(x)
            mxq, mxs = api.mxfp8_quantize(x)
            out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            wsb = torch.empty(max(1, api.bs_gemm_workspace(M, N, K)), dtype=torch.uint8, device=dev)
            wsm = torch.zeros(max(1, api.lib().mxfp8_gemm_workspace(M, N, K)), dtype=torch.uint8, device=dev)
            t_bs = _time_op(lambda: api.bs_gemm(xq, xs, wq, ws, out=out, workspace=wsb), flush)
            t_mx = _time_op(lambda: api.mxfp8_gemm(mxq, mxs, mq, ms_, c=out, workspace=wsm), flush)
            res[f"{name}_M{M}"] = {"us": round(t_bs * 1e3, 2),
                                   "GB_s": round(bsgemm_bytes(M, N, K) / (t_bs * 1e-3) / 1e9, 1),
                                   "mxfp8_us": round(t_mx * 1e3, 2)}
        del wq, ws, mq, ms_
    return res


PREFILL_CASES = {"bs64_T234": ([0] * 64, [234] * 64), "bs1_T4096": ([0], [4096]),
                 "bs4_P2048_T2048": ([2048] * 4, [2048] * 4)}


def prefill_setup(dev, rn, prefix, new):
    """Device inputs of one causal prefill / extend call (caches already holding the new rows)."""
    import torch

    lens = np.asarray(prefix) + np.asarray(new)
    cap = int((lens.max() + 127) // 128 * 128)
    bs, total = len(new), int(np.sum(new))
    K = rn((bs, HKV, cap, HD))
    V = rn((bs, HKV, cap, HD))
    q = rn((total, HQ, HD))
    q_start = torch.from_numpy(np.concatenate([[0], np.cumsum(new)]).astype(np.int32)).to(dev)
    kl = torch.from_numpy(lens.astype(np.int32)).to(dev)
    out = torch.empty((total, HQ, HD), dtype=torch.bfloat16, device=dev)
    return q, K, V, q_start, kl, out, int(max(new))


def prefill_sweep(dev, rn, flush):
    """Causal prefill / extend attention (tcgen05): TFLOP/s of the causal flop count."""
    from mxfp8_mlp_gqa_gb300 import api

    res = {}
    for name, (prefix, new) in PREFILL_CASES.items():
        q, K, V, qs, kl, out, mq = prefill_setup(dev, rn, prefix, new)
        ms = _time_op(lambda: api.gqa_prefill_attn(q, K, V, qs, kl, mq, 1 / math.sqrt(HD), out=out), flush)
        res[name] = {"us": round(ms * 1e3, 2), "TFLOP_s": round(prefill_flops(prefix, new) / (ms * 1e-3) / 1e12, 1)}
        del q, K, V, out
    return res


def kv_mxfp8_attn_sweep(dev, rn, flush):
    """Decode attention over an MXFP8 K/V cache (contiguous, cap = 4096; and paged, 64-token
    pages) at bs = 1…64 over the bench's ragged lengths; GB/s over the MXFP8 algorithmic bytes."""
    import torch

    from mxfp8_mlp_gqa_gb300 import api, synth

    cap, bs_max = KV_HI, BS
    kc = torch.empty((bs_max, HKV, cap, HD), dtype=torch.uint8, device=dev)
    ks = torch.empty((bs_max, HKV, cap, HD // 32), dtype=torch.uint8, device=dev)
    vc, vs = torch.empty_like(kc), torch.empty_like(ks)
    for b in range(bs_max):
        for c, s in ((kc, ks), (vc, vs)):
            q8, s8 = api.mxfp8_quantize(rn((HKV * cap, HD)))
            c[b].copy_(q8.view(HKV, cap, HD))
            s[b].copy_(s8.view(HKV, cap, HD // 32))
    res = {}
    for bs in (1, 8, 16, 32, 64):
        lens = synth.kv_lens(bs, KV_LO, KV_HI, seed=0)
        q = rn((bs, HQ, HD))
        kl = torch.from_numpy(lens).to(dev)
        out = torch.empty((bs, HQ, HD), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(max(1, api.gqa_decode_attn_workspace(bs, HQ, HKV, HD, KV_HI)), dtype=torch.uint8, device=dev)
        a = (kc[:bs], ks[:bs], vc[:bs], vs[:bs])
        ms = _time_op(lambda: api.gqa_decode_attn_kv_mxfp8(q, *a, kl, KV_HI, 1 / math.sqrt(HD), out=out,
                                                           workspace=ws), flush)
        res[str(bs)] = {"us": round(ms * 1e3, 2), "GB_s": round(attn_kv_mxfp8_bytes(lens) / (ms * 1e-3) / 1e9, 1)}
    # paged, bs = 64: the contiguous arrays viewed as 64-token pages, visited in a seeded
    # random order
    ps = 64
    lens = synth.kv_lens(bs_max, KV_LO, KV_HI, seed=0)
    npg = cap // ps
    pools = [t.view(bs_max, HKV, npg, ps, -1).permute(0, 2, 1, 3, 4).contiguous().view(bs_max * npg, HKV, ps, -1)
             for t in (kc, ks, vc, vs)]
    table = np.random.default_rng(ps).permutation(bs_max * npg).astype(np.int32).reshape(bs_max, npg)
    tb = torch.from_numpy(table).to(dev)
    q = rn((bs_max, HQ, HD))
    kl = torch.from_numpy(lens).to(dev)
    out = torch.empty((bs_max, HQ, HD), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(max(1, api.gqa_decode_attn_workspace(bs_max, HQ, HKV, HD, KV_HI)), dtype=torch.uint8, device=dev)
    ms = _time_op(lambda: api.gqa_decode_attn_kv_mxfp8_paged(q, *pools, tb, kl, KV_HI, 1 / math.sqrt(HD), out=out,
                                                             workspace=ws), flush)
    res["paged64_bs64"] = {"us": round(ms * 1e3, 2), "GB_s": round(attn_kv_mxfp8_bytes(lens) / (ms * 1e-3) / 1e9, 1)}
    return res


def paged_attn_sweep(dev, rn, flush, bs=BS, page_sizes=(64, 128, 256)):
    """Paged decode attention at bs=64 over the bench's ragged lengths, pages placed at a seeded
    random permutation of the pool (with 10 % spare pages); GB/s over the same algorithmic bytes
    as the contiguous kernel."""
    import torch

    from mxfp8_mlp_gqa_gb300 import api, synth

    lens = synth.kv_lens(bs, KV_LO, KV_HI, seed=0)
    q = rn((bs, HQ, HD))
    kl = torch.from_numpy(lens).to(dev)
    out = torch.empty((bs, HQ, HD), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(max(1, api.gqa_decode_attn_workspace(bs, HQ, HKV, HD, KV_HI)), dtype=torch.uint8, device=dev)
    res = {}
    for ps in page_sizes:
        need = (lens.astype(np.int64) + ps - 1) // ps
        num_pages = int(need.sum() * 11 // 10)
        perm = np.random.default_rng(ps).permutation(num_pages).astype(np.int32)
        table = np.full((bs, (KV_HI + ps - 1) // ps), -1, np.int32)
        k = 0
        for b in range(bs):
            table[b, :need[b]] = perm[k:k + need[b]]
            k += int(need[b])
        Kp = rn((num_pages, HKV, ps, HD))
        Vp = rn((num_pages, HKV, ps, HD))
        tb = torch.from_numpy(table).to(dev)
        ms = _time_op(lambda: api.gqa_decode_attn_paged(q, Kp, Vp, tb, kl, KV_HI, 1 / math.sqrt(HD), out=out,
                                                        workspace=ws), flush)
        res[str(ps)] = {"us": round(ms * 1e3, 2), "GB_s": round(attn_bytes(lens) / (ms * 1e-3) / 1e9, 1)}
        del Kp, Vp
    return res


def fp8_peak_tflops():
    """Dense fp8 tensor peak used for config-5 fractions: the measured bf16 burst of
    MEASURED_PEAKS.json times the nominal fp8/bf16 ratio 2 (no fp8 figure is measured there)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return 2.0 * float(json.load(f)["bf16_tflops"]), "2 x measured bf16 burst"
    return 2.0 * 1900.0, "2 x fallback bf16"


def gemm_square_sweep(dev, sizes=(1024, 2048, 4096, 8192, 16384)):
    """Config-5 sweep: C = A' B'^T, A and B MXFP8 [N, N], bf16 C; TFLOP/s of 2 N^3 per call,
    median of 5 timed calls after 2 warm-up calls, as a fraction of the fp8 peak
    (fp8_peak_tflops). Alongside, cuBLAS's MXFP8 GEMM through torch._scaled_mm with UE8M0 block
    scales where this torch build supports it -- a library kernel's practical peak on this part,
    a measured lower bound of the fp8 peak -- and this kernel's ratio to it."""
    import torch

    from mxfp8_mlp_gqa_gb300 import api

    peak, peak_src = fp8_peak_tflops()

    g = torch.Generator(device=dev)
    g.manual_seed(5)
    out = {}
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timeit(fn, reps=5):
        for _ in range(2):
            fn()
        ts = []
        for _ in range(reps):
            e0.record()
            fn()
            e1.record()
            e1.synchronize()
            ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    for n in sizes:
        a = torch.randn((n, n), generator=g, device=dev).to(torch.bfloat16)
        aq, as_ = api.mxfp8_quantize(a)
        b = torch.randn((n, n), generator=g, device=dev).to(torch.bfloat16)
        bq, bs_ = api.mxfp8_quantize(b)
        del a, b
        c = torch.empty((n, n), dtype=torch.bfloat16, device=dev)
        ws = torch.zeros(max(1, api.mxfp8_gemm_workspace(n, n, n)), dtype=torch.uint8, device=dev)
        ms = timeit(lambda: api.mxfp8_gemm(aq, as_, bq, bs_, c=c, workspace=ws))
        tf = 2 * n ** 3 / (ms * 1e-3) / 1e12
        ent = {"us": round(ms * 1e3, 1), "TFLOP_s": round(tf, 1), "frac_of_fp8_peak": round(tf / peak, 3),
               "fp8_peak_TFLOP_s": round(peak, 1), "fp8_peak_source": peak_src}
        try:
            fa = aq.view(torch.float8_e4m3fn)
            fb = bq.view(torch.float8_e4m3fn)
            sa = torch.full((((n + 127) // 128) * 128 * ((n // 32 + 3) // 4) * 4,), 127, dtype=torch.uint8,
                            device=dev).view(torch.float8_e8m0fnu)
            sb = sa.clone()
            ms2 = timeit(lambda: torch._scaled_mm(fa, fb.t(), sa, sb, out_dtype=torch.bfloat16))
            ent["cublas_mxfp8_TFLOP_s"] = round(2 * n ** 3 / (ms2 * 1e-3) / 1e12, 1)
            ent["of_cublas_mxfp8"] = round(ms2 / ms, 3)
        except Exception as ex:  # noqa: BLE001 - context only
            ent["cublas_mxfp8"] = f"unavailable: {type(ex).__name__}"
        out[str(n)] = ent
        del aq, bq, c
    return out


def run_profile(args):
    """W + K launches of one entry point on synthetic device inputs (small ncu captures)."""
    import torch

    from mxfp8_mlp_gqa_gb300 import api, synth

    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev)
    g.manual_seed(2)
    rn = lambda shape, std=1.0: (torch.randn(shape, generator=g, device=dev) * std).to(torch.bfloat16)  # noqa: E731
    kind, _, arg = args.profile.partition(":")
    if kind == "mlp":
        M = int(arg)
        w13 = api.mxfp8_quantize(rn((2 * D_FF, D_MODEL), 0.02))
        w2 = api.mxfp8_quantize(rn((D_MODEL, D_FF), 0.02))
        xq, xs = api.mxfp8_quantize(rn((M, D_MODEL)))
        ws = torch.zeros(api.mlp_swiglu_mxfp8_workspace(M, D_MODEL, D_FF), dtype=torch.uint8, device=dev)
        y = torch.empty((M, D_MODEL), dtype=torch.bfloat16, device=dev)
        fn = lambda: api.mlp_swiglu_mxfp8(xq, xs, *w13, *w2, y=y, workspace=ws)  # noqa: E731
    elif kind == "attn":
        bs, _, capa = arg.partition(":")
        bs, cap = int(bs), int(capa or CAP)
        K = torch.empty((bs, HKV, cap, HD), dtype=torch.bfloat16, device=dev)
        V = torch.empty_like(K)
        for b in range(bs):
            K[b].copy_(rn(K[b].shape))
            V[b].copy_(rn(V[b].shape))
        lens = synth.kv_lens(bs, KV_LO, min(KV_HI, cap), seed=0)
        kl = torch.from_numpy(lens).to(dev)
        q = rn((bs, HQ, HD))
        ws = torch.empty(max(1, api.gqa_decode_attn_workspace(bs, HQ, HKV, HD, KV_HI)), dtype=torch.uint8, device=dev)
        out = torch.empty((bs, HQ, HD), dtype=torch.bfloat16, device=dev)
        fn = lambda: api.gqa_decode_attn(q, K, V, kl, KV_HI, 1 / math.sqrt(HD), out=out, workspace=ws)  # noqa: E731
    elif kind == "attn_mx":
        # decode attention over an MXFP8 K/V cache [bs, Hkv, cap, D] (+ scales)
        bs, _, capa = arg.partition(":")
        bs, cap = int(bs), int(capa or KV_HI)
        arrs = []
        for _ in range(2):
            c = torch.empty((bs, HKV, cap, HD), dtype=torch.uint8, device=dev)
            sc = torch.empty((bs, HKV, cap, HD // 32), dtype=torch.uint8, device=dev)
            for b in range(bs):
                q8, s8 = api.mxfp8_quantize(rn((HKV * cap, HD)))
                c[b].copy_(q8.view(HKV, cap, HD))
                sc[b].copy_(s8.view(HKV, cap, HD // 32))
            arrs += [c, sc]
        lens = synth.kv_lens(bs, KV_LO, min(KV_HI, cap), seed=0)
        kl = torch.from_numpy(lens).to(dev)
        q = rn((bs, HQ, HD))
        ws = torch.empty(max(1, api.gqa_decode_attn_workspace(bs, HQ, HKV, HD, KV_HI)), dtype=torch.uint8, device=dev)
        out = torch.empty((bs, HQ, HD), dtype=torch.bfloat16, device=dev)
        fn = lambda: api.gqa_decode_attn_kv_mxfp8(q, *arrs, kl, KV_HI, 1 / math.sqrt(HD), out=out,  # noqa: E731
                                                  workspace=ws)
    elif kind == "prefill":
        # causal prefill / extend attention, one of PREFILL_CASES
        prefix, new = PREFILL_CASES[arg]
        q, K, V, qs, kl, pout, mq = prefill_setup(dev, rn, prefix, new)
        fn = lambda: api.gqa_prefill_attn(q, K, V, qs, kl, mq, 1 / math.sqrt(HD), out=pout)  # noqa: E731
    elif kind == "gemm":
        M, N, K_ = (int(v) for v in arg.split("x"))
        aq, as_ = api.mxfp8_quantize(rn((M, K_)))
        bq, bs_ = api.mxfp8_quantize(rn((N, K_)))
        c = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        wsb = torch.zeros(max(1, api.mxfp8_gemm_workspace(M, N, K_)), dtype=torch.uint8, device=dev)
        fn = lambda: api.mxfp8_gemm(aq, as_, bq, bs_, c=c, workspace=wsb)  # noqa: E731
    elif kind == "bsgemm":
        # block-scaled FP8 GEMM (1x128 activation / 128x128 weight blocks, fp32 scales)
        M, N, K_ = (int(v) for v in arg.split("x"))
        xq, xs = api.bs_quantize_act(rn((M, K_)))
        wq, ws_ = api.bs_quantize_weight(rn((N, K_), 0.02))
        c = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        wsb = torch.zeros(max(1, api.bs_gemm_workspace(M, N, K_)), dtype=torch.uint8, device=dev)
        fn = lambda: api.bs_gemm(xq, xs, wq, ws_, out=c, workspace=wsb)  # noqa: E731
    elif kind == "cublas":
        # context only: cuBLAS's MXFP8 GEMM (torch._scaled_mm, UE8M0 block scales of 2^0) on
        # the same shape, for a side-by-side capture of a library kernel
        M, N, K_ = (int(v) for v in arg.split("x"))
        fa = api.mxfp8_quantize(rn((M, K_)))[0].view(torch.float8_e4m3fn)
        fb = api.mxfp8_quantize(rn((N, K_)))[0].view(torch.float8_e4m3fn)
        sa = torch.full((((M + 127) // 128) * 128 * ((K_ // 32 + 3) // 4) * 4,), 127, dtype=torch.uint8,
                        device=dev).view(torch.float8_e8m0fnu)
        sb = torch.full((((N + 127) // 128) * 128 * ((K_ // 32 + 3) // 4) * 4,), 127, dtype=torch.uint8,
                        device=dev).view(torch.float8_e8m0fnu)
        fn = lambda: torch._scaled_mm(fa, fb.t(), sa, sb, out_dtype=torch.bfloat16)  # noqa: E731
    else:
        raise SystemExit(f"unknown --profile {args.profile}")
    flush = L2Flush(dev)
    ms = _time_op(fn, flush, reps=args.steps, warm=args.warmup)
    out = {"profile": args.profile, "median_us": round(ms * 1e3, 2)}
    if kind == "attn":
        out["attn_bytes"] = attn_bytes(lens)
        out["sum_kv_len"] = int(lens.sum())
    if kind == "prefill":
        out["TFLOP_s"] = round(prefill_flops(*PREFILL_CASES[arg]) / (ms * 1e-3) / 1e12, 1)
    if kind == "attn_mx":
        out["attn_bytes"] = attn_kv_mxfp8_bytes(lens)
        out["sum_kv_len"] = int(lens.sum())
    return out


# --------------------------------------------------------------------------- oracle (CPU) arm
def oracle_weights(seed=0):
    """MXFP8 weights of the layer as the oracle quantises them (weight prep, untimed)."""
    from mxfp8_mlp_gqa_gb300 import synth
    from oracle import mx

    nqkv = (HQ + 2 * HKV) * HD

    def q(n, k, tid):
        # rows quantise independently: do it in row blocks to bound the fp64 temporaries
        wb = synth.weights(n, k, seed, synth.TID[tid])
        parts = [mx.mx_quantize(mx.bf16_to_f64(wb[i:i + 1024])) for i in range(0, n, 1024)]
        return np.concatenate([a for a, _ in parts]), np.concatenate([b for _, b in parts])

    return {"wqkv": q(nqkv, D_MODEL, "wqkv"), "wo": q(D_MODEL, HQ * HD, "wo"), "w13": q(2 * D_FF, D_MODEL, "w13"),
            "w2": q(D_MODEL, D_FF, "w2"), "g1": synth.gamma(D_MODEL, seed, synth.TID["gamma1"]),
            "g2": synth.gamma(D_MODEL, seed, synth.TID["gamma2"])}


def oracle_inputs(bs_sample, seed, kv_sched_row):
    """Per-step inputs of `bs_sample` sequences of the same workload (host)."""
    from mxfp8_mlp_gqa_gb300 import synth

    lens = np.asarray(kv_sched_row[:bs_sample])
    return {
        "x": synth.activations(bs_sample, D_MODEL, seed),
        "kp": synth.kv_prefix(bs_sample, HKV, HD, lens - 1, seed, synth.TID["k"]),
        "vp": synth.kv_prefix(bs_sample, HKV, HD, lens - 1, seed, synth.TID["v"]),
        "prev": synth.codes((bs_sample, W_WIN, CW), 4096, seed, synth.TID["prev"]),
        "next": synth.codes((bs_sample, CW), 4096, seed, synth.TID["next"]),
        "lens": lens,
    }


def oracle_step(w, inp):
    from oracle import ops

    return ops.decode_layer_step(inp["x"], w["g1"], w["g2"], w["wqkv"], w["wo"], w["w13"], w["w2"], inp["kp"],
                                 inp["vp"], inp["lens"], inp["prev"], inp["next"], HQ, HKV, HD, EPS,
                                 1 / math.sqrt(HD))


def sample_bytes(lens):
    return sum(step_bytes(lens, bs=len(lens)).values())


def run_cpu_baseline(bs_sample=1):
    """The oracle as it stands, one decode-layer step on a bounded sample of the workload."""
    from mxfp8_mlp_gqa_gb300 import synth

    sched, _ = synth.slot_schedule(BS, 1, KV_LO, KV_HI, LIFE_HI, seed=0)
    w = oracle_weights(0)
    inp = oracle_inputs(bs_sample, 0, sched[0])
    t0 = time.perf_counter()
    oracle_step(w, inp)
    sec = time.perf_counter() - t0
    by = sample_bytes(inp["lens"])
    return {"value": round(by / sec / 1e9, 4), "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"one oracle decode-layer step on {bs_sample} of the 64 sequences (kv_len "
                      f"{list(map(int, inp['lens']))}) with all weights: {sec:.2f} s; numpy fp64 (BLAS matmuls "
                      f"may use all cores, elementwise work is single-threaded)",
            "seconds": round(sec, 3), "bytes": by}


# The oracle per configuration (the pages' workloads, timed on this host's cores): each case runs
# in a child process so that the BLAS thread count is fixed before numpy loads -- once with one
# thread, once with every core.
CPU_CASES = ("config1_step", "config2_mlp_M1", "config2_mlp_M128", "config3_attn_bs64", "config5_gemm_4096_sampled")
THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS")


def cpu_case(name):
    """One timed oracle call of the named configuration; returns seconds, value, unit, sample."""
    from mxfp8_mlp_gqa_gb300 import synth
    from oracle import mx, ops

    def mxq(bits):
        return mx.mx_quantize(mx.bf16_to_f64(bits))

    if name == "config1_step":
        d, dff, hq, hkv, hd = 256, 768, 4, 2, 64
        w = {k: mxq(synth.weights(n, kk, 0, synth.TID[k])) for k, n, kk in
             (("wqkv", (hq + 2 * hkv) * hd, d), ("wo", d, hq * hd), ("w13", 2 * dff, d), ("w2", d, dff))}
        lens = np.array([100])
        args = (synth.activations(1, d, 0), synth.gamma(d, 0, synth.TID["gamma1"]),
                synth.gamma(d, 0, synth.TID["gamma2"]), w["wqkv"], w["wo"], w["w13"], w["w2"],
                synth.kv_prefix(1, hkv, hd, lens - 1, 0, synth.TID["k"]),
                synth.kv_prefix(1, hkv, hd, lens - 1, 0, synth.TID["v"]), lens,
                synth.codes((1, 8, 10), 1024, 0, synth.TID["prev"]), synth.codes((1, 10), 1024, 0, synth.TID["next"]),
                hq, hkv, hd, EPS, 1 / 8)
        t0 = time.perf_counter()
        ops.decode_layer_step(*args)
        sec = time.perf_counter() - t0
        return {"seconds": sec, "value": round(sec * 1e3, 3), "unit": "ms per step",
                "sample": "the whole tiny decode-layer step (d_model 256, d_ff 768, 4/2 heads x 64, kv_len 100)"}
    if name.startswith("config2_mlp_M"):
        M = int(name[len("config2_mlp_M"):])
        w13 = mxq(synth.weights(2 * D_FF, D_MODEL, 0, synth.TID["w13"]))
        w2 = mxq(synth.weights(D_MODEL, D_FF, 0, synth.TID["w2"]))
        xq, xs = mxq(synth.activations(M, D_MODEL, 0, outlier_frac=0.01))
        t0 = time.perf_counter()
        ops.swiglu_mlp(xq, xs, *w13, *w2)
        sec = time.perf_counter() - t0
        return {"seconds": sec, "value": round(mlp_bytes(M) / sec / 1e9, 4), "unit": "GB/s",
                "sample": f"the whole MLP at M = {M} (2560 / 9728, weights already MX-quantised)"}
    if name == "config3_attn_bs64":
        lens = synth.kv_lens(BS, KV_LO, KV_HI, seed=0)
        q = mx.bf16_to_f64(synth.normal_bf16((BS, HQ, HD), 1.0, 0, synth.TID["q"]))
        kp = [mx.bf16_to_f64(a) for a in synth.kv_prefix(BS, HKV, HD, lens, 0, synth.TID["k"])]
        vp = [mx.bf16_to_f64(a) for a in synth.kv_prefix(BS, HKV, HD, lens, 0, synth.TID["v"])]
        t0 = time.perf_counter()
        ops.gqa_decode_attention(q, kp, vp, 1 / math.sqrt(HD))
        sec = time.perf_counter() - t0
        return {"seconds": sec, "value": round(attn_bytes(lens) / sec / 1e9, 4), "unit": "GB/s",
                "sample": "GQA decode attention, bs 64, kv_len ~U[234, 4096] (sum %d)" % int(lens.sum())}
    if name == "config5_gemm_4096_sampled":
        N = 4096
        g = synth.rng(0, synth.TID["sample"])
        rows = np.sort(g.choice(N, 256, replace=False))
        cols = np.sort(g.choice(N, 256, replace=False))
        a = synth.normal_bf16((N, N), 1.0, 0, synth.TID["a"])[rows]
        b = synth.normal_bf16((N, N), 1.0, 0, synth.TID["b"])[cols]
        aq, bq = mxq(a), mxq(b)
        t0 = time.perf_counter()
        ops.mx_gemm(*aq, *bq)
        sec = time.perf_counter() - t0
        return {"seconds": sec, "value": round(2 * 256 * 256 * N / sec / 1e9, 3), "unit": "GFLOP/s",
                "sample": "256 sampled rows x 256 sampled columns of the 4096^3 MXFP8 GEMM (fp64 dot products)"}
    raise ValueError(name)


def run_cpu_cases():
    """Every CPU case twice in child processes: one BLAS thread, then all cores."""
    out = {}
    for name in CPU_CASES:
        row = {}
        for label, n in (("1_thread", "1"), ("all_cores", None)):
            env = dict(os.environ)
            for v in THREAD_VARS:
                if n is None:
                    env.pop(v, None)
                else:
                    env[v] = n
            r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-case", name], env=env,
                               capture_output=True, text=True, timeout=600)
            try:
                row[label] = json.loads(r.stdout.strip().splitlines()[-1])
            except (IndexError, ValueError):
                row[label] = {"error": (r.stderr or r.stdout)[-300:]}
        out[name] = row
    return {"cores": os.cpu_count(), "kind": "oracle", "cases": out}


def run_reference(args, rank, world):
    """--impl reference: the oracle timed on the host cores, on this workload, one bounded
    sample (one of the 64 sequences, all weights) per step. Rank 0 only."""
    if rank != 0:
        return None
    from mxfp8_mlp_gqa_gb300 import synth

    sched, _ = synth.slot_schedule(BS, args.warmup + args.steps, KV_LO, KV_HI, LIFE_HI, seed=0)
    bs_sample = 1
    w = oracle_weights(0)
    secs, by = [], 0
    for s in range(args.warmup + args.steps):
        inp = oracle_inputs(bs_sample, 0, sched[s])
        t0 = time.perf_counter()
        oracle_step(w, inp)
        dt = time.perf_counter() - t0
        if s >= args.warmup:
            secs.append(dt)
            by += sample_bytes(inp["lens"])
    tot = sum(secs)
    value = by / tot / 1e9
    sample = f"oracle decode-layer step on {bs_sample} of the 64 sequences per step, all weights"
    return {
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(tot / args.steps * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": {"workload": WORKLOAD, "sample": sample},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# --------------------------------------------------------------------------- main
def run_timeline(args):
    """The decode-layer step's CUDA graph on the instrumented library (libmxg_tl.so): per-launch
    device timeline (first entry, first return from the programmatic wait, last exit), medians
    over the timed steps, each step L2-flushed like the bench's."""
    import torch

    from mxfp8_mlp_gqa_gb300 import api, build as _build, synth, timeline

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    lib = api.lib(_build.build(timeline=True))
    total_steps = args.warmup + args.steps
    sched, _refill = synth.slot_schedule(BS, total_steps + 1, KV_LO, KV_HI, LIFE_HI, seed=0)
    L = build_layer(dev, int(sched.max()))
    sched_d = torch.from_numpy(sched).to(dev)
    rec = timeline.Recorder(lib)
    flush = L2Flush(dev)
    L.kv_len.copy_(sched_d[0])
    L.step()
    torch.cuda.synchronize()
    plain = L.capture()
    for s in range(args.warmup):
        L.kv_len.copy_(sched_d[s])
        plain.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    steps, ms = [], []
    for i in range(args.steps):
        L.kv_len.copy_(sched_d[args.warmup + i])
        flush()
        torch.cuda.synchronize()
        rec.reset()
        e0.record()
        plain.replay()
        e1.record()
        e1.synchronize()
        ms.append(e0.elapsed_time(e1))
        steps.append(rec.records())
    summ = timeline.summarize(steps)
    print(f"instrumented step: {statistics.median(ms) * 1e3:.1f} us (event-timed median of {args.steps})")
    print(timeline.format_table(summ))
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-sweeps", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-case", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--profile", default=None,
                    help="run one kernel family only (for ncu captures): mlp:<M> | attn:<bs>[:<cap>] | "
                         "gemm:<M>x<N>x<K> | cublas:<M>x<N>x<K> (library kernel, context)")
    ap.add_argument("--timeline", action="store_true",
                    help="print the decode step's per-launch device timeline from the instrumented library "
                         "(libmxg_tl.so) instead of the JSON line")
    args = ap.parse_args(argv)
    if args.cpu_case:  # child process of run_cpu_cases: one oracle timing, no GPU
        print(json.dumps(cpu_case(args.cpu_case)))
        return 0
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, local_rank, world = dist_env()

    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line))
        return 0

    import torch

    if args.timeline:
        return run_timeline(args)
    if args.profile:
        print(json.dumps(run_profile(args)))
        return 0
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res = run_ours(args, rank, local_rank, world)
    cpu = cpu_cases = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = run_cpu_baseline()
        cpu_cases = run_cpu_cases()
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(res["value"], 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(res["ms_per_step"], 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "mxfp8+bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "global_batch": BS * world, "parallelism": f"replicas x{world}",
                       "l2": "flushed between timed steps outside the events: 256 MiB written, then another 256 MiB "
                             "read, so the step starts with clean unrelated lines in L2; step footprint "
                             "~0.68 GB > 129 MB L2", "timing": "one captured CUDA graph per step, events around each replay on the launching "
                                           "stream; per-kernel breakdown from a second graph with timing events "
                                           "between its kernels"},
            "e2e": res["e2e"], "roofline": res["roofline"], "cpu_baseline": cpu,
            "cpu_baseline_configs": cpu_cases, "clocks": res["clocks"],
            "gpu_launches": res["gpu_launches"], "eager_ms_per_step": round(res["eager_ms_per_step"], 4),
            "evented_ms_per_step": round(res["evented_ms_per_step"], 4),
            "breakdown": res["breakdown"], "sweeps": res["sweeps"],
        }
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
