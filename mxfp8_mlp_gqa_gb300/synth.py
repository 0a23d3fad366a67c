"""Seeded synthetic inputs for the decode-step hot path.

This module is shared by the CUDA path's tests/bench and by the CPU oracle's
tests. It holds no arithmetic of the method itself (no MX quantisation, no
GEMM, no softmax): it only draws random numbers and rounds them to the storage
types the kernels take (bf16 bit patterns, int32 codes, int32 lengths).

Recipe (shapes and distributions of the pages' workloads, Qwen3-4B-shaped layer,
S2-Pro attention shape, see "How We Made Our Text-to-Speech API Free" -- Kernel
Benchmark Results, and "Fish Speech KV Cache 推理优化记录" -- §4):

* every tensor gets its own PCG64 stream, seeded by ``SeedSequence([seed, tid])``;
* weights: bf16 ~ N(0, 0.02); activations: bf16 ~ N(0, 1), optionally with 1 %
  of the channels (chosen by a seeded permutation, same for every row) scaled x20;
* RMSNorm gains: bf16 ~ N(1, 0.1) (a ones-gain would hide indexing bugs);
* q/K/V: bf16 ~ N(0, 1); ragged kv_len ~ U[lo, hi] (inclusive);
* codebook tokens: int32 uniform in [0, n_codes).

bf16 values are returned as ``numpy.uint16`` bit patterns (numpy has no bf16).
"""
from __future__ import annotations

import numpy as np

# tensor ids: one stream per logical tensor, so adding a tensor never shifts
# the values of another one.
TID = {
    "x": 1, "w13": 2, "w2": 3, "q": 4, "k": 5, "v": 6, "kv_len": 7,
    "prev": 8, "next": 9, "gamma1": 10, "gamma2": 11, "wqkv": 12, "wo": 13,
    "a": 14, "b": 15, "outlier": 16, "residual": 17, "sched": 18, "sample": 19,
}


def rng(seed: int, tid: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tid])))


def f32_to_bf16_bits(a) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); NaN kept quiet."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    # finite values are <= 0xFF7FFFFF, so adding at most 0x8000 cannot wrap a uint32
    r = ((u + (np.uint32(0x7FFF) + ((u >> 16) & np.uint32(1)))) >> 16).astype(np.uint16)
    nan = np.isnan(a)
    if nan.any():
        r = np.where(nan, np.uint16(0x7FC0), r)
    return r


def bf16_bits_to_f32(b) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def normal_bf16(shape, std: float, seed: int, tid: int, mean: float = 0.0) -> np.ndarray:
    g = rng(seed, tid)
    a = g.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    if mean != 0.0:
        a += np.float32(mean)
    return f32_to_bf16_bits(a)


def activations(M: int, K: int, seed: int = 0, outlier_frac: float = 0.0,
                outlier_scale: float = 20.0, tid: int = TID["x"]) -> np.ndarray:
    """bf16 [M, K] ~ N(0,1); round(outlier_frac*K) channels scaled by outlier_scale."""
    g = rng(seed, tid)
    a = g.standard_normal(size=(M, K), dtype=np.float32)
    n_out = int(round(outlier_frac * K))
    if n_out:
        ch = rng(seed, TID["outlier"]).permutation(K)[:n_out]
        a[:, ch] *= np.float32(outlier_scale)
    return f32_to_bf16_bits(a)


def weights(N: int, K: int, seed: int, tid: int, std: float = 0.02) -> np.ndarray:
    return normal_bf16((N, K), std, seed, tid)


def gamma(K: int, seed: int, tid: int) -> np.ndarray:
    return normal_bf16((K,), 0.1, seed, tid, mean=1.0)


def kv_lens(bs: int, lo: int, hi: int, seed: int, tid: int = TID["kv_len"]) -> np.ndarray:
    return rng(seed, tid).integers(lo, hi + 1, size=bs, dtype=np.int64).astype(np.int32)


def codes(shape, n_codes: int, seed: int, tid: int) -> np.ndarray:
    return rng(seed, tid).integers(0, n_codes, size=shape, dtype=np.int64).astype(np.int32)


def kv_prefix(bs: int, Hkv: int, D: int, lens, seed: int, tid: int) -> list:
    """Per-sequence active prefix [Hkv, kv_len_b, D] (bf16 bits), drawn sequence by
    sequence from one stream so that the values do not depend on the capacity."""
    g = rng(seed, tid)
    out = []
    for b in range(bs):
        a = g.standard_normal(size=(Hkv, int(lens[b]), D), dtype=np.float32)
        out.append(f32_to_bf16_bits(a))
    return out


def garbage_tail_value(i) -> np.ndarray:
    """Deterministic +-1e4 pattern for the never-read tail of a KV cache (bf16 bits)."""
    i = np.asarray(i, dtype=np.int64)
    return np.where(i % 2 == 0, np.uint16(0x461C), np.uint16(0xC61C)).astype(np.uint16)  # +-9984


def full_cache(bs: int, Hkv: int, cap: int, D: int, prefix: list) -> np.ndarray:
    """Host-side full cache [bs, Hkv, cap, D] with the prefix written and a +-1e4 tail
    (only for small capacities; large caches are filled on the device)."""
    c = garbage_tail_value(np.arange(bs * Hkv * cap * D)).reshape(bs, Hkv, cap, D)
    for b in range(bs):
        n = prefix[b].shape[1]
        c[b, :, :n, :] = prefix[b]
    return c


def slot_schedule(bs: int, steps: int, lo: int, hi: int, life_hi: int, seed: int):
    """Continuous-batching schedule: per step, kv_len [bs] (length after this step's
    append) and a refill mask. Each slot starts at kv_len ~ U[lo, hi], lives
    ~ U[1, life_hi] steps, then is retired and refilled with a fresh length."""
    g = rng(seed, TID["sched"])
    kv = g.integers(lo, hi + 1, size=bs)
    life = g.integers(1, life_hi + 1, size=bs)
    lens = np.zeros((steps, bs), np.int32)
    refill = np.zeros((steps, bs), bool)
    for s in range(steps):
        for b in range(bs):
            if life[b] == 0:
                kv[b] = g.integers(lo, hi + 1)
                life[b] = g.integers(1, life_hi + 1)
                refill[s, b] = True
        lens[s] = kv
        kv = kv + 1
        life = life - 1
    return lens, refill
