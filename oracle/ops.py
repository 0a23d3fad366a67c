"""fp64 restatement of the decode-step hot path -- oracle, test infrastructure only.

Each function is the plain definition of one step, with a library matmul as the
only primitive; no blocking, fusion or reordering beyond the definition.
"""
from __future__ import annotations

import numpy as np

from .mx import bf16_to_f64, f64_to_bf16, mx_dequantize, mx_quantize


# --------------------------------------------------------------------------- GEMM
def mx_gemm(aq, ascale, bq, bscale) -> np.ndarray:
    """C = A' B'^T in fp64, A' [M,K] and B' [N,K] the dequantised MX operands.

    [S2.1] "FP8 Quantization Strategy": the mxfp8 GEMM takes both operands as
    1x32-block MX tensors (E4M3 + UE8M0) along the contraction dimension K.
    """
    return mx_dequantize(aq, ascale) @ mx_dequantize(bq, bscale).T


def mx_gemm_sampled(aq, ascale, bq, bscale, rows, cols) -> np.ndarray:
    """C[rows][:, cols] of ``mx_gemm``: one fp64 dot product per sampled entry."""
    rows = np.asarray(rows)
    cols = np.asarray(cols)
    A = mx_dequantize(aq[rows], ascale[rows])
    B = mx_dequantize(bq[cols], bscale[cols])
    return A @ B.T


# --------------------------------------------------------------------------- MLP
def silu(g):
    """silu(g) = g / (1 + e^-g) (fp64)."""
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def swiglu_mlp(xq, xs, w13q, w13s, w2q, w2s, residual_bf16=None) -> dict:
    """Qwen3-4B-shaped SwiGLU MLP over MX operands ([S2.1] "Kernel Benchmark
    Results": quantise -> gate/up -> SwiGLU -> quantise -> down, with the SwiGLU
    fused into the down projection's activation quantisation so that no bf16
    intermediate exists).

    W13 = [W_gate; W_up] stacked along N (rows 0..d_ff-1 gate, d_ff..2d_ff-1 up).
    g, u = X' W_g'^T, X' W_u'^T; h = silu(g) * u; (hq, hs) = MX(h) along d_ff;
    y = H' W_d'^T (+ residual), rounded once to bf16.
    """
    d_ff = w13q.shape[0] // 2
    X = mx_dequantize(xq, xs)
    W13 = mx_dequantize(w13q, w13s)
    G = X @ W13[:d_ff].T
    U = X @ W13[d_ff:].T
    H = silu(G) * U
    hq, hs = mx_quantize(H)
    Y = mx_dequantize(hq, hs) @ mx_dequantize(w2q, w2s).T
    if residual_bf16 is not None:
        Y = Y + bf16_to_f64(residual_bf16)
    return {"g": G, "u": U, "h": H, "hq": hq, "hs": hs, "y": Y, "y_bf16": f64_to_bf16(Y)}


# --------------------------------------------------------------------------- RMSNorm
def rmsnorm_bf16(x_bf16, gamma_bf16, eps) -> np.ndarray:
    """RMSNorm of each row, rounded to bf16 (the input of the activation quantiser).

    y = x * rsqrt(mean(x^2) + eps) * gamma. The pages give no precision for this
    step; the reading used (both here and in the kernel, so that the bf16
    rounding that decides the quantised codes is taken at the same precision):
    mean(x^2) and rsqrt in fp64 (eps taken as the fp32 value passed by the
    caller), the factor rounded to fp32, then x*r and (x*r)*gamma in fp32, then
    bf16 round-to-nearest-even.
    """
    x = bf16_to_f64(x_bf16)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    r = (1.0 / np.sqrt(ms + np.float64(np.float32(eps)))).astype(np.float32)
    y = (x.astype(np.float32) * r) * bf16_to_f64(gamma_bf16).astype(np.float32)
    return f64_to_bf16(y.astype(np.float64))


def rmsnorm_mx_quantize(x_bf16, gamma_bf16, eps):
    return mx_quantize(bf16_to_f64(rmsnorm_bf16(x_bf16, gamma_bf16, eps)))


# --------------------------------------------------------------------------- attention
def gqa_decode_attention(q, k_prefix, v_prefix, scale) -> np.ndarray:
    """GQA decode attention over each sequence's active prefix (fp64 brute force).

    [FSKV] §5: the cache keeps its full capacity, and attention reads only the
    filled prefix K[:, :, :kv_len], V[:, :, :kv_len]; KV heads are shared by
    Hq/Hkv query heads (repeat_interleave(n_head // n_local_heads) in §5, i.e.
    query head h reads KV head floor(h / (Hq/Hkv))). The decode query sits at
    position kv_len-1, so no position inside the prefix is masked.

    q: [bs, Hq, D] (fp64 values); k_prefix[b], v_prefix[b]: [Hkv, kv_len_b, D].
    Returns o [bs, Hq, D] fp64 = softmax(scale * q K^T) V per (b, h).
    """
    bs, Hq, D = q.shape
    out = np.zeros((bs, Hq, D))
    for b in range(bs):
        K = np.asarray(k_prefix[b], dtype=np.float64)
        V = np.asarray(v_prefix[b], dtype=np.float64)
        Hkv = K.shape[0]
        grp = Hq // Hkv
        for h in range(Hq):
            g = h // grp
            s = scale * (K[g] @ q[b, h])
            p = np.exp(s - s.max())
            out[b, h] = (p @ V[g]) / p.sum()
    return out


def gqa_attention_full_cache_masked(q, k_cache, v_cache, kv_len, scale) -> np.ndarray:
    """The pre-fix formulation of [FSKV] §4: every query head attends over the
    full capacity with KV heads expanded by repeat_interleave and positions
    >= kv_len masked to -inf. Used only to check the invariant of [FSKV] §7
    (active prefix == full cache + mask)."""
    bs, Hq, D = q.shape
    Hkv, cap = k_cache.shape[1], k_cache.shape[2]
    K = np.repeat(np.asarray(k_cache, np.float64), Hq // Hkv, axis=1)
    V = np.repeat(np.asarray(v_cache, np.float64), Hq // Hkv, axis=1)
    s = scale * np.einsum("bhd,bhjd->bhj", q, K)
    mask = np.arange(cap)[None, :] >= np.asarray(kv_len)[:, None]
    s = np.where(mask[:, None, :], -np.inf, s)
    p = np.exp(s - s.max(axis=-1, keepdims=True))
    p = p / p.sum(axis=-1, keepdims=True)
    return np.einsum("bhj,bhjd->bhd", p, V)


# --------------------------------------------------------------------------- KV append
def kv_append(k_cache, v_cache, k_new, v_new, kv_len):
    """Write this step's K/V rows at position kv_len-1 of each sequence (in place
    update of the preallocated cache, [FSKV] §5 "kv_cache.update"); kv_len is the
    length after the append (prefill T, i-th decode T+i+1)."""
    k_cache = k_cache.copy()
    v_cache = v_cache.copy()
    for b, n in enumerate(np.asarray(kv_len)):
        k_cache[b, :, n - 1, :] = k_new[b]
        v_cache[b, :, n - 1, :] = v_new[b]
    return k_cache, v_cache


def paged_prefix(pool, block_table, kv_len, page_size) -> list:
    """Each sequence's active prefix [Hkv, kv_len_b, D] gathered from a paged pool
    [num_pages, Hkv, page_size, D]: position t of sequence b is row t % page_size of pool
    page block_table[b, t // page_size] ([S2.1] "What's Open Source": paged decode)."""
    out = []
    for b, n in enumerate(np.asarray(kv_len)):
        n = int(n)
        pref = np.zeros((pool.shape[1], n, pool.shape[3]), dtype=pool.dtype)
        for t in range(n):
            pref[:, t, :] = pool[int(block_table[b, t // page_size]), :, t % page_size, :]
        out.append(pref)
    return out


def gqa_decode_attention_paged(q, k_pool, v_pool, block_table, kv_len, page_size, scale) -> np.ndarray:
    """Decode attention over paged caches: the plain decode attention of each sequence's
    prefix gathered through its page table."""
    return gqa_decode_attention(q, paged_prefix(k_pool, block_table, kv_len, page_size),
                                paged_prefix(v_pool, block_table, kv_len, page_size), scale)


def kv_append_paged(k_pool, v_pool, block_table, k_new, v_new, kv_len, page_size):
    """kv_append into paged pools: position kv_len-1 of sequence b is row
    (kv_len-1) % page_size of page block_table[b, (kv_len-1) // page_size]."""
    k_pool = k_pool.copy()
    v_pool = v_pool.copy()
    for b, n in enumerate(np.asarray(kv_len)):
        pg = int(block_table[b, (int(n) - 1) // page_size])
        k_pool[pg, :, (int(n) - 1) % page_size, :] = k_new[b]
        v_pool[pg, :, (int(n) - 1) % page_size, :] = v_new[b]
    return k_pool, v_pool


# --------------------------------------------------------------------------- prefill / extend
def gqa_prefill_attention(q_new, k_prefix, v_prefix, scale) -> list:
    """Causal prefill / extend attention with native GQA ([S2.1] "What's Open Source":
    contiguous prefill and paged prefill (extend)). Sequence b holds kv_len_b rows in its cache,
    the last T_b of which belong to the new tokens; new token i sits at position
    kv_len_b - T_b + i and attends to positions 0 .. kv_len_b - T_b + i (T_b = kv_len_b is a
    prefill from scratch). q_new[b]: [T_b, Hq, D]; k_prefix[b], v_prefix[b]: [Hkv, kv_len_b, D].
    Returns o[b]: [T_b, Hq, D] fp64."""
    out = []
    for qb, K, V in zip(q_new, k_prefix, v_prefix):
        qb = np.asarray(qb, np.float64)
        K = np.asarray(K, np.float64)
        V = np.asarray(V, np.float64)
        T, Hq, D = qb.shape
        Hkv, n = K.shape[0], K.shape[1]
        grp = Hq // Hkv
        pos = n - T + np.arange(T)
        allowed = np.arange(n)[None, :] <= pos[:, None]
        o = np.zeros((T, Hq, D))
        for h in range(Hq):
            g = h // grp
            s = scale * (qb[:, h, :] @ K[g].T)
            s = np.where(allowed, s, -np.inf)
            p = np.exp(s - s.max(axis=1, keepdims=True))
            o[:, h, :] = (p @ V[g]) / p.sum(axis=1, keepdims=True)
        out.append(o)
    return out


def kv_append_extend(k_cache, v_cache, k_new, v_new, kv_len):
    """Write T_b new K/V rows per sequence (k_new[b], v_new[b]: [T_b, Hkv, D]) at positions
    kv_len_b - T_b .. kv_len_b - 1 of the cache [bs, Hkv, cap, D] ([FSKV] §5, kv_cache.update
    for a prefill or extend)."""
    k_cache = k_cache.copy()
    v_cache = v_cache.copy()
    for b, n in enumerate(np.asarray(kv_len)):
        T = k_new[b].shape[0]
        k_cache[b, :, n - T:n, :] = np.transpose(k_new[b], (1, 0, 2))
        v_cache[b, :, n - T:n, :] = np.transpose(v_new[b], (1, 0, 2))
    return k_cache, v_cache


# --------------------------------------------------------------------------- MXFP8 KV cache
def kv_rows_mx(rows):
    """K or V rows [..., D] (fp64 values of bf16 rows) MX-quantised along D: the 1x32-block
    format of [S2.1] "FP8 Quantization Strategy" (E4M3 elements, UE8M0 shared exponents),
    applied to the cache as the pages' MXFP8 FlashAttention reads it ("What's Open Source").
    Returns (codes uint8 [..., D], scale bytes uint8 [..., D/32])."""
    return mx_quantize(rows)


def kv_append_mxfp8(k_codes, k_scales, v_codes, v_scales, k_new, v_new, kv_len):
    """kv_append into an MXFP8 cache: the new rows k_new, v_new [bs, Hkv, D] (fp64 values of
    bf16) are MX-quantised along D and written at position kv_len-1 ([FSKV] §5)."""
    k_codes, k_scales, v_codes, v_scales = (a.copy() for a in (k_codes, k_scales, v_codes, v_scales))
    kq, ks = kv_rows_mx(k_new)
    vq, vs = kv_rows_mx(v_new)
    for b, n in enumerate(np.asarray(kv_len)):
        k_codes[b, :, n - 1, :] = kq[b]
        k_scales[b, :, n - 1, :] = ks[b]
        v_codes[b, :, n - 1, :] = vq[b]
        v_scales[b, :, n - 1, :] = vs[b]
    return k_codes, k_scales, v_codes, v_scales


def gqa_decode_attention_kv_mxfp8(q, k_codes, k_scales, v_codes, v_scales, scale) -> np.ndarray:
    """Decode attention over MXFP8 prefixes: every cached row is dequantised exactly
    (E4M3 value x 2^s of its 32-wide block) and the plain decode attention runs on those
    values. k_codes[b] [Hkv, kv_len_b, D] uint8, k_scales[b] [Hkv, kv_len_b, D/32] uint8."""
    K = [mx_dequantize(c, s) for c, s in zip(k_codes, k_scales)]
    V = [mx_dequantize(c, s) for c, s in zip(v_codes, v_scales)]
    return gqa_decode_attention(q, K, V, scale)


# --------------------------------------------------------------------------- prev window
def prev_tokens_shift(prev, next_tokens) -> np.ndarray:
    """Slide the Dual-AR previous-tokens window by one frame ([S2.1] "DualAR:
    S2-Specific Batching Constraints": prev int32 [bs, W, cw], next_tokens int32
    [bs, cw]). Reading: frame 0 is the oldest and is dropped, frames move down by
    one, and next_tokens becomes frame W-1."""
    prev = np.asarray(prev)
    nxt = np.asarray(next_tokens)
    out = np.empty_like(prev)
    out[:, :-1, :] = prev[:, 1:, :]
    out[:, -1, :] = nxt
    return out


# --------------------------------------------------------------------------- layer step
def decode_layer_step(x_bf16, gamma1, gamma2, wqkv, wo, w13, w2, k_prefix, v_prefix,
                      kv_len, prev, next_tokens, Hq, Hkv, D, eps, scale) -> dict:
    """One slow-AR decoder-layer step: RMSNorm -> MX quantise -> QKV projection ->
    KV append -> GQA decode attention -> MX quantise -> O projection + residual ->
    RMSNorm -> MX quantise -> SwiGLU MLP + residual; plus the prev-window shift.

    wqkv/wo/w13/w2 are (q, scale) MX pairs. k_prefix[b]/v_prefix[b] hold the
    kv_len[b]-1 rows already in the cache; the new row comes from the QKV
    projection. Every bf16 tensor the kernels store is rounded to bf16 here too.
    """
    bs = x_bf16.shape[0]
    xq, xs = rmsnorm_mx_quantize(x_bf16, gamma1, eps)
    qkv = f64_to_bf16(mx_gemm(xq, xs, *wqkv))
    qkv_f = bf16_to_f64(qkv)
    q = qkv_f[:, : Hq * D].reshape(bs, Hq, D)
    k_new = qkv_f[:, Hq * D:(Hq + Hkv) * D].reshape(bs, Hkv, D)
    v_new = qkv_f[:, (Hq + Hkv) * D:].reshape(bs, Hkv, D)
    kp = [np.concatenate([bf16_to_f64(k_prefix[b]), k_new[b][:, None, :]], axis=1) for b in range(bs)]
    vp = [np.concatenate([bf16_to_f64(v_prefix[b]), v_new[b][:, None, :]], axis=1) for b in range(bs)]
    for b in range(bs):
        assert kp[b].shape[1] == kv_len[b]
    o = f64_to_bf16(gqa_decode_attention(q, kp, vp, scale)).reshape(bs, Hq * D)
    oq, os_ = mx_quantize(bf16_to_f64(o))
    x1 = f64_to_bf16(bf16_to_f64(x_bf16) + mx_gemm(oq, os_, *wo))
    hq_in, hs_in = rmsnorm_mx_quantize(x1, gamma2, eps)
    mlp = swiglu_mlp(hq_in, hs_in, w13[0], w13[1], w2[0], w2[1], residual_bf16=x1)
    return {"qkv": qkv, "o": o, "x1": x1, "y": mlp["y"], "y_bf16": mlp["y_bf16"],
            "prev": prev_tokens_shift(prev, next_tokens)}
