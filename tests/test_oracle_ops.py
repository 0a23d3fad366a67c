"""Pins of the oracle's GEMM / MLP / RMSNorm / attention / prev-shift / step
(CPU only): brute force with independent decoding (torch float8 casts and plain
Python loops), closed forms, torch library routines, and the invariants stated
in the pages (active prefix == full cache + mask)."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from mxfp8_mlp_gqa_gb300 import synth
from oracle import mx, ops


def _dec_e4m3(q):
    return torch.from_numpy(np.ascontiguousarray(q)).view(torch.float8_e4m3fn).double().numpy()


def _dec_scale(s):
    return np.array([[2.0 ** (int(b) - 127) for b in row] for row in s])


def _brute_mx_dot(aq, as_, bq, bs_, i, j):
    """One output of C = A B^T as a plain Python loop over K (independent decode)."""
    a = _dec_e4m3(aq[i])
    b = _dec_e4m3(bq[j])
    tot = 0.0
    for k in range(aq.shape[1]):
        tot += (a[k] * 2.0 ** (int(as_[i, k // 32]) - 127)) * (b[k] * 2.0 ** (int(bs_[j, k // 32]) - 127))
    return tot


def _mx_operand(shape, seed, tid, std=1.0):
    x = mx.bf16_to_f64(synth.normal_bf16(shape, std, seed, tid))
    # distinct scales per block: multiply blocks by seeded powers of two
    g = synth.rng(seed, tid + 100)
    x = x * np.exp2(g.integers(-6, 7, (shape[0], shape[1] // 32))).repeat(32, axis=1)
    return mx.mx_quantize(x)


def test_mx_gemm_brute_force_nonsquare():
    aq, as_ = _mx_operand((5, 96), 0, 1)
    bq, bs_ = _mx_operand((7, 96), 0, 2)
    c = ops.mx_gemm(aq, as_, bq, bs_)
    for i in range(5):
        for j in range(7):
            assert math.isclose(c[i, j], _brute_mx_dot(aq, as_, bq, bs_, i, j), rel_tol=1e-12, abs_tol=1e-12)


def test_mx_gemm_transposed_scale_layout_is_detected():
    # the silent bug of [S2.1] "FP8 Quantization Strategy": reading the scales
    # with the wrong stride must change the result on non-square, non-uniform data
    aq, as_ = _mx_operand((4, 128), 1, 1)
    bq, bs_ = _mx_operand((4, 128), 1, 2)
    good = ops.mx_gemm(aq, as_, bq, bs_)
    bad = ops.mx_gemm(aq, as_, bq, np.ascontiguousarray(bs_.T).reshape(bs_.shape))
    assert np.linalg.norm(good - bad) > 0.1 * np.linalg.norm(good)


def test_mx_gemm_sampled_equals_full():
    aq, as_ = _mx_operand((33, 64), 2, 1)
    bq, bs_ = _mx_operand((29, 64), 2, 2)
    rows, cols = np.array([0, 5, 32, 7]), np.array([28, 0, 3])
    np.testing.assert_array_equal(ops.mx_gemm_sampled(aq, as_, bq, bs_, rows, cols),
                                  ops.mx_gemm(aq, as_, bq, bs_)[rows][:, cols])


def test_mx_gemm_identity_closed_form():
    # A = I (exact in E4M3 with scale 2^0) -> C = B'^T's columns, i.e. C[i, j] = B'[j, i]
    K = 64
    aq, as_ = mx.mx_quantize(np.eye(K))
    bq, bs_ = _mx_operand((10, K), 3, 2)
    np.testing.assert_array_equal(ops.mx_gemm(aq, as_, bq, bs_), mx.mx_dequantize(bq, bs_).T)


def _tiny_mlp(seed=0, d_model=64, d_ff=96, M=3):
    x = synth.activations(M, d_model, seed, outlier_frac=0.05)
    w13 = synth.weights(2 * d_ff, d_model, seed, synth.TID["w13"], std=0.2)
    w2 = synth.weights(d_model, d_ff, seed, synth.TID["w2"], std=0.2)
    xq, xs = mx.mx_quantize(mx.bf16_to_f64(x))
    w13q, w13s = mx.mx_quantize(mx.bf16_to_f64(w13))
    w2q, w2s = mx.mx_quantize(mx.bf16_to_f64(w2))
    res = synth.activations(M, d_model, seed, tid=synth.TID["residual"])
    return xq, xs, w13q, w13s, w2q, w2s, res


def test_swiglu_mlp_brute_force():
    xq, xs, w13q, w13s, w2q, w2s, res = _tiny_mlp()
    out = ops.swiglu_mlp(xq, xs, w13q, w13s, w2q, w2s, residual_bf16=res)
    M, d_ff, d_model = xq.shape[0], w13q.shape[0] // 2, xq.shape[1]
    for t in range(M):
        h = []
        for j in range(d_ff):
            g = _brute_mx_dot(xq, xs, w13q, w13s, t, j)
            u = _brute_mx_dot(xq, xs, w13q, w13s, t, d_ff + j)
            h.append(g / (1.0 + math.exp(-g)) * u)
        assert np.allclose(out["h"][t], h, rtol=1e-12, atol=1e-15)
        # requantise by brute force: per 32-block shared exponent, nearest E4M3 by search
        for blk in range(d_ff // 32):
            hb = np.array(h[32 * blk:32 * blk + 32])
            amax = np.abs(hb).max()
            s = -127 if amax == 0 else max(-127, min(127, math.floor(math.log2(amax)) - 8))
            assert out["hs"][t, blk] == s + 127
            grid = _dec_e4m3(np.arange(128, dtype=np.uint8))
            for k, v in enumerate(hb / 2.0 ** s):
                a = min(abs(v), 448.0)
                d = np.abs(np.nan_to_num(grid, nan=1e9) - a)
                cand = np.flatnonzero(d == d.min())
                code = int(cand[0] if cand.size == 1 else cand[cand % 2 == 0][0])
                assert out["hq"][t, 32 * blk + k] & 0x7F == code
        hd = _dec_e4m3(out["hq"][t]) * np.repeat(2.0 ** (out["hs"][t].astype(int) - 127), 32)
        for n in range(d_model):
            w = _dec_e4m3(w2q[n]) * np.repeat(2.0 ** (w2s[n].astype(int) - 127), 32)
            y = sum(hd[k] * w[k] for k in range(d_ff)) + mx.bf16_to_f64(res[t, n])
            assert math.isclose(out["y"][t, n], y, rel_tol=1e-12, abs_tol=1e-12)


def test_swiglu_mlp_zero_gate_is_residual():
    xq, xs, w13q, w13s, w2q, w2s, res = _tiny_mlp(1)
    w13q = w13q.copy()
    w13q[: w13q.shape[0] // 2] = 0
    out = ops.swiglu_mlp(xq, xs, w13q, w13s, w2q, w2s, residual_bf16=res)
    # h = silu(0) * u = +-0 (sign of u kept) -> codes 0x00 / 0x80, scale byte 0
    assert not (out["hq"] & 0x7F).any() and not out["hs"].any()
    np.testing.assert_array_equal(out["y_bf16"], res)


def test_silu_closed_form():
    g = np.array([0.0, 1.0, -1.0, 50.0, -800.0])
    np.testing.assert_allclose(ops.silu(g), [0.0, 1 / (1 + math.exp(-1)), -1 / (1 + math.e), 50.0, -0.0], rtol=1e-15)


def test_rmsnorm_against_torch():
    x = synth.activations(16, 2560, 0, outlier_frac=0.01)
    gam = synth.gamma(2560, 0, synth.TID["gamma1"])
    eps = 1e-6
    y = mx.bf16_to_f64(ops.rmsnorm_bf16(x, gam, eps))
    ref = F.rms_norm(torch.from_numpy(mx.bf16_to_f64(x)), (2560,), torch.from_numpy(mx.bf16_to_f64(gam)),
                     eps=float(np.float32(eps))).numpy()
    # one bf16 rounding (<= 2^-9 relative) plus fp32 products (~2^-23)
    assert np.all(np.abs(y - ref) <= np.abs(ref) * (2.0 ** -8) + 1e-30)


def test_rmsnorm_constant_row_closed_form():
    c = 3.0
    x = synth.f32_to_bf16_bits(np.full((1, 64), c, np.float32))
    one = synth.f32_to_bf16_bits(np.ones(64, np.float32))
    y = mx.bf16_to_f64(ops.rmsnorm_bf16(x, one, 0.0))
    np.testing.assert_array_equal(y, 1.0)


def _attn_case(bs, Hq, Hkv, D, cap, lens, seed=0):
    q = synth.normal_bf16((bs, Hq, D), 1.0, seed, synth.TID["q"])
    kp = synth.kv_prefix(bs, Hkv, D, lens, seed, synth.TID["k"])
    vp = synth.kv_prefix(bs, Hkv, D, lens, seed, synth.TID["v"])
    return q, kp, vp


def test_attention_prefix_equals_full_cache_with_mask():
    # [FSKV] §7 invariant: active prefix == full cache + mask (fp32 rtol 1e-5 /
    # atol 1e-6 in the pages; both sides are fp64 here)
    bs, Hq, Hkv, D, cap = 3, 8, 2, 32, 64
    lens = np.array([1, 17, 64])
    q, kp, vp = _attn_case(bs, Hq, Hkv, D, cap, lens)
    kc = synth.full_cache(bs, Hkv, cap, D, kp)
    vc = synth.full_cache(bs, Hkv, cap, D, vp)
    a = ops.gqa_decode_attention(mx.bf16_to_f64(q), [mx.bf16_to_f64(k) for k in kp],
                                 [mx.bf16_to_f64(v) for v in vp], 0.2)
    b = ops.gqa_attention_full_cache_masked(mx.bf16_to_f64(q), mx.bf16_to_f64(kc), mx.bf16_to_f64(vc), lens, 0.2)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


def test_attention_matches_torch_sdpa_gqa():
    bs, Hq, Hkv, D = 2, 8, 2, 64
    lens = np.array([5, 40])
    q, kp, vp = _attn_case(bs, Hq, Hkv, D, 64, lens, seed=1)
    qf = mx.bf16_to_f64(q)
    out = ops.gqa_decode_attention(qf, [mx.bf16_to_f64(k) for k in kp], [mx.bf16_to_f64(v) for v in vp], 0.125)
    for b in range(bs):
        K = torch.from_numpy(mx.bf16_to_f64(kp[b])).repeat_interleave(Hq // Hkv, dim=0)[None]
        V = torch.from_numpy(mx.bf16_to_f64(vp[b])).repeat_interleave(Hq // Hkv, dim=0)[None]
        ref = F.scaled_dot_product_attention(torch.from_numpy(qf[b])[None, :, None, :], K, V, scale=0.125)
        np.testing.assert_allclose(out[b], ref[0, :, 0].numpy(), rtol=1e-12, atol=1e-13)


def test_attention_mha_special_case_and_single_token():
    bs, H, D = 2, 4, 16
    lens = np.array([1, 9])
    q, kp, vp = _attn_case(bs, H, H, D, 16, lens, seed=2)
    out = ops.gqa_decode_attention(mx.bf16_to_f64(q), [mx.bf16_to_f64(k) for k in kp],
                                   [mx.bf16_to_f64(v) for v in vp], 0.3)
    # kv_len = 1 -> softmax weight 1 -> out = V_0 exactly
    np.testing.assert_array_equal(out[0], mx.bf16_to_f64(vp[0])[:, 0, :])
    # Hkv = Hq -> plain multi-head attention
    ref = F.scaled_dot_product_attention(torch.from_numpy(mx.bf16_to_f64(q[1]))[None, :, None, :],
                                         torch.from_numpy(mx.bf16_to_f64(kp[1]))[None],
                                         torch.from_numpy(mx.bf16_to_f64(vp[1]))[None], scale=0.3)
    np.testing.assert_allclose(out[1], ref[0, :, 0].numpy(), rtol=1e-12, atol=1e-13)


def test_attention_uniform_scores_give_mean():
    q = np.zeros((1, 2, 8))
    V = np.arange(2 * 5 * 8, dtype=float).reshape(2, 5, 8)
    K = np.ones((2, 5, 8))
    out = ops.gqa_decode_attention(q, [K[:1]], [V[:1]], 1.0)
    np.testing.assert_allclose(out[0, 0], V[0].mean(0), rtol=1e-15)
    np.testing.assert_allclose(out[0, 1], V[0].mean(0), rtol=1e-15)


def test_prev_tokens_shift_brute_force_and_special_cases():
    prev = synth.codes((3, 8, 10), 1024, 0, synth.TID["prev"])
    nxt = synth.codes((3, 10), 1024, 0, synth.TID["next"])
    out = ops.prev_tokens_shift(prev, nxt)
    for b in range(3):
        for w in range(8):
            for c in range(10):
                assert out[b, w, c] == (prev[b, w + 1, c] if w < 7 else nxt[b, c])
    # W = 1: the window becomes next_tokens
    np.testing.assert_array_equal(ops.prev_tokens_shift(prev[:, :1], nxt)[:, 0], nxt)
    # W shifts push every old frame out: the window holds the last W next_tokens in order
    win = prev.copy()
    hist = [synth.codes((3, 10), 1024, 9, 100 + i) for i in range(8)]
    for n in hist:
        win = ops.prev_tokens_shift(win, n)
    np.testing.assert_array_equal(win, np.stack(hist, axis=1))


def test_kv_append_brute_force():
    kc = np.zeros((2, 2, 6, 4))
    vc = np.zeros((2, 2, 6, 4))
    kn = np.arange(16.0).reshape(2, 2, 4)
    vn = -kn
    k2, v2 = ops.kv_append(kc, vc, kn, vn, np.array([1, 6]))
    assert np.array_equal(k2[0, :, 0], kn[0]) and np.array_equal(k2[1, :, 5], kn[1])
    assert np.array_equal(v2[1, :, 5], vn[1]) and np.count_nonzero(k2) == np.count_nonzero(kn)


def _scatter_to_pages(prefix, page_size, num_pages, rng):
    """Independent construction of a paged pool: each sequence's prefix cut into pages placed
    at random distinct pool pages, every other pool entry +-1e4."""
    Hkv, D = prefix[0].shape[0], prefix[0].shape[2]
    pool = np.where(np.arange(num_pages * Hkv * page_size * D) % 2 == 0, 1e4, -1e4).reshape(
        num_pages, Hkv, page_size, D)
    need = [(p.shape[1] + page_size - 1) // page_size for p in prefix]
    perm = rng.permutation(num_pages)[:sum(need)]
    table = np.full((len(prefix), max(need) + 1), -1, np.int32)
    k = 0
    for b, p in enumerate(prefix):
        for j in range(need[b]):
            seg = p[:, j * page_size:(j + 1) * page_size, :]
            pool[perm[k], :, :seg.shape[1], :] = seg
            table[b, j] = perm[k]
            k += 1
    return pool, table


def test_paged_attention_equals_contiguous_under_page_permutation():
    # the paged reading is the contiguous one on the same prefix: a random page placement
    # (and +-1e4 in every unused pool entry) changes nothing, bit for bit
    rng = np.random.default_rng(3)
    bs, Hq, Hkv, D, ps = 3, 8, 2, 16, 4
    lens = np.array([1, 9, 12])
    q = rng.standard_normal((bs, Hq, D))
    kp = [rng.standard_normal((Hkv, n, D)) for n in lens]
    vp = [rng.standard_normal((Hkv, n, D)) for n in lens]
    kpool, table = _scatter_to_pages(kp, ps, 16, np.random.default_rng(7))
    vpool, table_v = _scatter_to_pages(vp, ps, 16, np.random.default_rng(7))
    assert np.array_equal(table, table_v)
    got = ops.gqa_decode_attention_paged(q, kpool, vpool, table, lens, ps, 0.25)
    assert np.array_equal(got, ops.gqa_decode_attention(q, kp, vp, 0.25))
    # one page per sequence of the whole capacity, identity table: the contiguous cache
    cap = 16
    kc = np.stack([np.concatenate([k, np.full((Hkv, cap - k.shape[1], D), 7.0)], axis=1) for k in kp])
    vc = np.stack([np.concatenate([v, np.full((Hkv, cap - v.shape[1], D), 7.0)], axis=1) for v in vp])
    ident = np.arange(bs, dtype=np.int32)[:, None]
    assert np.array_equal(ops.gqa_decode_attention_paged(q, kc, vc, ident, lens, cap, 0.25), got)


def test_kv_append_paged_lands_where_the_gather_reads():
    rng = np.random.default_rng(5)
    Hkv, D, ps = 2, 8, 4
    prefix = [rng.standard_normal((Hkv, n, D)) for n in (3, 4, 8)]
    pool, table = _scatter_to_pages(prefix, ps, 12, np.random.default_rng(2))
    # give every sequence a page for its next position (the sequence of length 4 and 8 start one)
    free = [p for p in range(12) if p not in set(table[table >= 0].tolist())]
    for b, n in enumerate((3, 4, 8)):
        if table[b, n // ps] < 0:
            table[b, n // ps] = free.pop()
    kn = rng.standard_normal((3, Hkv, D))
    vn = rng.standard_normal((3, Hkv, D))
    lens = np.array([4, 5, 9])  # after the append
    k2, v2 = ops.kv_append_paged(pool, pool.copy(), table, kn, vn, lens, ps)
    gk = ops.paged_prefix(k2, table, lens, ps)
    gv = ops.paged_prefix(v2, table, lens, ps)
    for b in range(3):
        assert np.array_equal(gk[b][:, :-1], prefix[b]) and np.array_equal(gk[b][:, -1], kn[b])
        assert np.array_equal(gv[b][:, -1], vn[b])
    assert np.count_nonzero(k2 != pool) == np.count_nonzero(kn)


def _tiny_step(zero_paths=False, seed=0):
    bs, d, dff, Hq, Hkv, D = 2, 64, 96, 4, 2, 16
    x = synth.activations(bs, d, seed)
    g1 = synth.gamma(d, seed, synth.TID["gamma1"])
    g2 = synth.gamma(d, seed, synth.TID["gamma2"])
    wqkv = mx.mx_quantize(mx.bf16_to_f64(synth.weights((Hq + 2 * Hkv) * D, d, seed, synth.TID["wqkv"], 0.1)))
    wo_b = mx.bf16_to_f64(synth.weights(d, Hq * D, seed, synth.TID["wo"], 0.1))
    w13_b = mx.bf16_to_f64(synth.weights(2 * dff, d, seed, synth.TID["w13"], 0.1))
    if zero_paths:
        wo_b[:] = 0
        w13_b[:dff] = 0
    wo = mx.mx_quantize(wo_b)
    w13 = mx.mx_quantize(w13_b)
    w2 = mx.mx_quantize(mx.bf16_to_f64(synth.weights(d, dff, seed, synth.TID["w2"], 0.1)))
    lens = np.array([3, 10])
    kp = synth.kv_prefix(bs, Hkv, D, lens - 1, seed, synth.TID["k"])
    vp = synth.kv_prefix(bs, Hkv, D, lens - 1, seed, synth.TID["v"])
    prev = synth.codes((bs, 4, 10), 4096, seed, synth.TID["prev"])
    nxt = synth.codes((bs, 10), 4096, seed, synth.TID["next"])
    return ops.decode_layer_step(x, g1, g2, wqkv, wo, w13, w2, kp, vp, lens, prev, nxt,
                                 Hq, Hkv, D, 1e-6, 1 / math.sqrt(D)), x, kp, vp, prev, nxt


def test_decode_step_zero_projections_is_identity():
    out, x, *_ = _tiny_step(zero_paths=True)
    np.testing.assert_array_equal(out["x1"], x)
    np.testing.assert_array_equal(out["y_bf16"], x)


def test_decode_step_composition():
    out, x, kp, vp, prev, nxt = _tiny_step()
    np.testing.assert_array_equal(out["prev"], ops.prev_tokens_shift(prev, nxt))
    # the new K row written by the step is the projection's k slice
    qkv = mx.bf16_to_f64(out["qkv"])
    assert qkv.shape == (2, (4 + 4) * 16)
    assert np.isfinite(out["y"]).all() and not np.array_equal(out["y_bf16"], x)


def test_decode_step_closed_form():
    """The layer step on hand-built weights whose result is known in closed form, so that a
    wiring mistake in the composition (k and v slices swapped or offset, the new row appended
    at the wrong position or not at all, o used without its MX quantisation, the wrong
    residual) changes the result:

    x = 1 and gamma = 1, so RMSNorm gives 1.0 exactly and its MX codes are exact; the k rows
    of Wqkv are zero and every cached K row is zero, so all scores are 0 and attention is the
    plain mean of the V rows (kv_len rows, the appended one included); the v rows of Wqkv pick
    input channel j, so the appended V row is all ones; Wo is the identity and W13 is zero,
    so x1 = x + MX(o) and y = x1. The V prefix is chosen so that o hits E4M3 rounding ties at
    the block's scale (amax 1.75: codes step by 2^-3 in [1, 2), 2^-4 in [0.5, 1))."""
    bs, d, dff, Hq, Hkv, D = 2, 64, 32, 2, 1, 32
    E4M3_ONE = 0x38  # 1.0 = 2^(7-7) x 1.000
    x = np.full((bs, d), 0x3F80, np.uint16)     # bf16 1.0
    ones = np.full((d,), 0x3F80, np.uint16)
    wq = mx.mx_quantize(mx.bf16_to_f64(synth.weights(Hq * D, d, 0, synth.TID["wqkv"], 0.5)))
    wqkv_q = np.zeros(((Hq + 2 * Hkv) * D, d), np.uint8)
    wqkv_s = np.full(((Hq + 2 * Hkv) * D, d // 32), 127, np.uint8)
    wqkv_q[:Hq * D], wqkv_s[:Hq * D] = wq
    for j in range(D):                         # v row j = input channel j
        wqkv_q[(Hq + Hkv) * D + j, j] = E4M3_ONE
    wo_q = np.zeros((d, Hq * D), np.uint8)
    wo_q[np.arange(d), np.arange(d)] = E4M3_ONE
    wo_s = np.full((d, Hq * D // 32), 127, np.uint8)
    w13 = (np.zeros((2 * dff, d), np.uint8), np.full((2 * dff, d // 32), 127, np.uint8))
    w2 = mx.mx_quantize(mx.bf16_to_f64(synth.weights(d, dff, 0, synth.TID["w2"], 0.5)))
    # sequence 0: kv_len 4 (3 cached rows + the appended one), sequence 1: kv_len 2
    o0 = np.full(D, 0.25)
    o0[:5] = [1.75, 1.0625, 1.1875, 0.53125, -0.75]
    o1 = np.full(D, 0.5)
    o1[0] = -1.5
    lens = np.array([4, 2])
    vp0 = np.zeros((Hkv, 3, D))
    vp0[0, 0] = 4 * o0 - 1                      # mean over {4 o - 1, 0, 0, 1} = o
    vp1 = (2 * o1 - 1).reshape(Hkv, 1, D)       # mean over {2 o - 1, 1} = o
    kp = [np.zeros((Hkv, 3, D), np.uint16), np.zeros((Hkv, 1, D), np.uint16)]
    vp = [mx.f64_to_bf16(vp0), mx.f64_to_bf16(vp1)]
    prev = synth.codes((bs, 4, 10), 4096, 0, synth.TID["prev"])
    nxt = synth.codes((bs, 10), 4096, 0, synth.TID["next"])
    out = ops.decode_layer_step(x, ones, ones, (wqkv_q, wqkv_s), (wo_q, wo_s), w13, w2, kp, vp, lens, prev, nxt,
                                Hq, Hkv, D, 1e-6, 1 / math.sqrt(D))
    qkv = mx.bf16_to_f64(out["qkv"])
    np.testing.assert_array_equal(qkv[:, Hq * D:(Hq + Hkv) * D], 0.0)      # k of the new row
    np.testing.assert_array_equal(qkv[:, (Hq + Hkv) * D:], 1.0)           # v of the new row
    o = mx.bf16_to_f64(out["o"]).reshape(bs, Hq, D)
    for h in range(Hq):                                                    # both heads read kv head 0
        np.testing.assert_array_equal(o[0, h], o0)
        np.testing.assert_array_equal(o[1, h], o1)
    # MX(o) at block amax 1.75 (scale 2^-8): 1.0625 -> 1.0 and 1.1875 -> 1.25 (ties to the even
    # code), 0.53125 -> 0.5 (tie), the rest exact
    oq0 = np.full(D, 0.25)
    oq0[:5] = [1.75, 1.0, 1.25, 0.5, -0.75]
    x1 = mx.bf16_to_f64(out["x1"])
    np.testing.assert_array_equal(x1[0], 1.0 + np.tile(oq0, Hq))
    np.testing.assert_array_equal(x1[1], 1.0 + np.tile(o1, Hq))
    np.testing.assert_array_equal(out["y"], x1)                             # h = 0: y is the residual
    np.testing.assert_array_equal(out["y_bf16"], out["x1"])
