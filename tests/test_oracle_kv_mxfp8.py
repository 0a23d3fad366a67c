"""Pins of the MXFP8 KV-cache oracle (decode attention over E4M3 + UE8M0 K/V, the MX-quantising
append) against closed forms and the already-pinned bf16 attention, independent of the CUDA path."""
import numpy as np

from oracle import mx, ops


def _representable(rng, shape):
    """Values whose 1x32 blocks along the last axis quantise without error: an MX tensor's own
    dequantised values (re-quantising them gives the same codes and exponents)."""
    return mx.mx_dequantize(*mx.mx_quantize(rng.standard_normal(shape)))


def test_mx_quantisation_of_dequantised_rows_is_exact():
    rng = np.random.default_rng(0)
    x = _representable(rng, (5, 64))
    q, s = ops.kv_rows_mx(x)
    assert np.array_equal(mx.mx_dequantize(q, s), x)
    # a power-of-two factor per row only moves that row's exponents
    f = np.exp2(np.arange(5) * 13 - 30.0)[:, None]
    q2, s2 = ops.kv_rows_mx(x * f)
    assert np.array_equal(q2, q) and np.array_equal(s2.astype(int), s.astype(int) + (np.arange(5) * 13 - 30)[:, None])


def test_mx_kv_constant_v_rows_give_the_dequantised_row():
    # softmax weights sum to one: with every V row of a head equal to v, o = dequant(quant(v))
    rng = np.random.default_rng(1)
    Hq, Hkv, D, n = 4, 2, 64, 37
    q = rng.standard_normal((1, Hq, D))
    k = rng.standard_normal((Hkv, n, D))
    v_row = rng.standard_normal((Hkv, 1, D))
    v = np.repeat(v_row, n, axis=1)
    kc, ks = ops.kv_rows_mx(k)
    vc, vs = ops.kv_rows_mx(v)
    o = ops.gqa_decode_attention_kv_mxfp8(q, [kc], [ks], [vc], [vs], 0.125)
    vq = mx.mx_dequantize(*mx.mx_quantize(v_row))
    assert not np.array_equal(vq, v_row)  # the row is not representable: quantisation shows
    for h in range(Hq):
        np.testing.assert_allclose(o[0, h], vq[h // (Hq // Hkv), 0], rtol=0, atol=1e-13)


def test_mx_kv_blocks_run_along_the_head_dim():
    # K = 0 gives uniform weights, so o is the mean of the V rows. Rows spanning 2^-40 .. 2^40
    # quantise exactly only if each row (block of 32 along D) has its own exponent: blocks along
    # the token axis would flush the small rows.
    rng = np.random.default_rng(2)
    Hkv, n, D = 1, 9, 64
    base = _representable(rng, (Hkv, n, D))
    v = base * np.exp2(np.linspace(-40, 40, n))[None, :, None]
    kc, ks = ops.kv_rows_mx(np.zeros((Hkv, n, D)))
    vc, vs = ops.kv_rows_mx(v)
    assert np.array_equal(kc, np.zeros_like(kc)) and np.array_equal(ks, np.zeros_like(ks))
    o = ops.gqa_decode_attention_kv_mxfp8(np.ones((1, 2, D)), [kc], [ks], [vc], [vs], 1.0)
    ref = v[0].mean(axis=0)
    np.testing.assert_allclose(o[0, 0], ref, rtol=1e-14, atol=0)
    np.testing.assert_allclose(o[0, 1], ref, rtol=1e-14, atol=0)


def test_mx_kv_attention_is_the_bf16_attention_of_the_dequantised_cache():
    # the MX attention is the (SDPA-pinned) decode attention on the exact dequantised values
    rng = np.random.default_rng(3)
    lens = [1, 33, 70]
    q = rng.standard_normal((3, 8, 32))
    kp = [rng.standard_normal((2, n, 32)) for n in lens]
    vp = [rng.standard_normal((2, n, 32)) for n in lens]
    kq = [ops.kv_rows_mx(k) for k in kp]
    vq = [ops.kv_rows_mx(v) for v in vp]
    got = ops.gqa_decode_attention_kv_mxfp8(q, [c for c, _ in kq], [s for _, s in kq], [c for c, _ in vq],
                                            [s for _, s in vq], 0.2)
    ref = ops.gqa_decode_attention(q, [mx.mx_dequantize(c, s) for c, s in kq],
                                   [mx.mx_dequantize(c, s) for c, s in vq], 0.2)
    assert np.array_equal(got, ref)
    # and it is near the unquantised attention: E4M3 keeps 3 mantissa bits, so each V value moves
    # by at most 2^-4 of its block's largest magnitude (a single-token prefix shows that directly)
    exact = ops.gqa_decode_attention(q, kp, vp, 0.2)
    vmax = max(np.abs(v).max() for v in vp)
    assert np.abs(got - exact).max() < vmax / 8


def test_mx_kv_append_row_by_row_equals_quantising_the_prefix():
    rng = np.random.default_rng(4)
    bs, Hkv, cap, D, T = 2, 2, 10, 64, 7
    rows = rng.standard_normal((bs, Hkv, T, D))
    kc = np.full((bs, Hkv, cap, D), 0x7F, np.uint8)  # E4M3 NaN codes where nothing was written
    ks = np.full((bs, Hkv, cap, D // 32), 0xFF, np.uint8)
    vc, vs = kc.copy(), ks.copy()
    for t in range(T):
        kc, ks, vc, vs = ops.kv_append_mxfp8(kc, ks, vc, vs, rows[:, :, t], -rows[:, :, t], np.full(bs, t + 1))
    q_ref, s_ref = ops.kv_rows_mx(rows)
    assert np.array_equal(kc[:, :, :T], q_ref) and np.array_equal(ks[:, :, :T], s_ref)
    assert np.array_equal(vc[:, :, :T], q_ref ^ 0x80) and np.array_equal(vs[:, :, :T], s_ref)
    assert (kc[:, :, T:] == 0x7F).all() and (ks[:, :, T:] == 0xFF).all()
    # an all-zero row: exponent byte 0, codes +0
    zc, zs = ops.kv_rows_mx(np.zeros((1, D)))
    assert not zc.any() and not zs.any()


def test_mx_kv_paged_gather_equals_contiguous():
    rng = np.random.default_rng(5)
    Hkv, D, ps, lens = 2, 32, 4, np.array([3, 9])
    q = rng.standard_normal((2, 4, D))
    kp = [ops.kv_rows_mx(rng.standard_normal((Hkv, n, D))) for n in lens]
    vp = [ops.kv_rows_mx(rng.standard_normal((Hkv, n, D))) for n in lens]
    num_pages = 8
    perm = np.random.default_rng(9).permutation(num_pages)
    pools = [np.full((num_pages, Hkv, ps, w), 0x7F, np.uint8) for w in (D, D // 32, D, D // 32)]
    table = np.full((2, 3), -1, np.int32)
    k = 0
    for b, n in enumerate(lens):
        for j in range((n + ps - 1) // ps):
            sl = slice(j * ps, min(n, (j + 1) * ps))
            for pool, arr in zip(pools, (kp[b][0], kp[b][1], vp[b][0], vp[b][1])):
                pool[perm[k], :, :sl.stop - sl.start] = arr[:, sl]
            table[b, j] = perm[k]
            k += 1
    g = [ops.paged_prefix(pool, table, lens, ps) for pool in pools]
    got = ops.gqa_decode_attention_kv_mxfp8(q, g[0], g[1], g[2], g[3], 0.3)
    ref = ops.gqa_decode_attention_kv_mxfp8(q, [c for c, _ in kp], [s for _, s in kp], [c for c, _ in vp],
                                            [s for _, s in vp], 0.3)
    assert np.array_equal(got, ref)
