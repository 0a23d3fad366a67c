"""Pins of the block-scaled FP8 (bsgemm recipe) oracle: hand-worked blocks, the MX oracle at
unit scales, brute force, the quantiser's error bound and the block geometry."""
import numpy as np

from oracle import bs, mx


def test_hand_worked_activation_block():
    # amax 14 -> s = 14/448 = 2^-5 (exact). 14/s = 448 -> 0x7E; -7/s = -224 = -1.75*2^7 ->
    # exponent field 14, mantissa 6 -> 0xF6; 3.5/s = 112 = 1.75*2^6 -> 0x6E;
    # 0.1015625/s = 3.25 = 1.625*2^1 -> field 8, mantissa 5 -> 0x45; 0 -> 0x00; -0 -> 0x80
    x = np.zeros((1, 128))
    x[0, :6] = [14.0, -7.0, 3.5, 0.1015625, 0.0, -0.0]
    q, s = bs.bs_quantize_act(x)
    assert s.dtype == np.float32 and s[0, 0] == np.float32(2.0 ** -5)
    assert list(q[0, :6]) == [0x7E, 0xF6, 0x6E, 0x45, 0x00, 0x80]
    assert not q[0, 6:].any()


def test_non_power_of_two_scale_and_zero_block():
    x = np.zeros((2, 256))
    x[0, 0], x[0, 1] = 3.0, -1.0   # s = fp32(3/448); 3/s rounds to 448 -> 0x7E
    x[1, 128:] = 0.0               # second row: both blocks zero
    q, s = bs.bs_quantize_act(x)
    assert s[0, 0] == np.float32(3.0) / np.float32(448.0)
    assert q[0, 0] == 0x7E
    # -1/s = -149.33.. -> spacing 16 in [128, 256): -144 = -1.125*2^7 -> field 14, mantissa 1 -> 0xF1
    assert q[0, 1] == 0xF1
    assert s[0, 1] == 0 and s[1, 0] == 0 and s[1, 1] == 0 and not q[1].any()


def test_bs_gemm_at_unit_scales_is_the_mx_gemm_at_unit_scales():
    rng = np.random.default_rng(0)
    xq = rng.integers(0, 256, (5, 256)).astype(np.uint8) & 0x77   # no NaN codes
    wq = rng.integers(0, 256, (130, 256)).astype(np.uint8) & 0x77
    got = bs.bs_gemm(xq, np.ones((5, 2), np.float32), wq, np.ones((2, 2), np.float32))
    ref = mx.mx_dequantize(xq, np.full((5, 8), 127, np.uint8)) @ mx.mx_dequantize(
        wq, np.full((130, 8), 127, np.uint8)).T
    np.testing.assert_array_equal(got, ref)


def test_bs_gemm_brute_force():
    rng = np.random.default_rng(1)
    M, N, K = 3, 131, 256
    xq = rng.integers(0, 256, (M, K)).astype(np.uint8) & 0x77
    wq = rng.integers(0, 256, (N, K)).astype(np.uint8) & 0x77
    xs = rng.uniform(0.01, 2, (M, 2)).astype(np.float32)
    ws = rng.uniform(0.01, 2, (2, 2)).astype(np.float32)
    got = bs.bs_gemm(xq, xs, wq, ws)
    xv, wv = mx.e4m3_value(xq), mx.e4m3_value(wq)
    for m in range(M):
        for n in (0, 1, 127, 128, 130):
            acc = 0.0
            for kb in range(2):
                dot = sum(xv[m, k] * wv[n, k] for k in range(kb * 128, kb * 128 + 128))
                acc += float(xs[m, kb]) * float(ws[n // 128, kb]) * dot
            assert abs(got[m, n] - acc) <= 1e-12 * max(1.0, abs(acc))


def test_quantiser_error_bound_and_block_geometry():
    rng = np.random.default_rng(2)
    # weight rows in three 128-row blocks with very different magnitudes (last block short)
    w = rng.standard_normal((300, 256)) * np.repeat([1e-3, 1.0, 50.0], [128, 128, 44])[:, None]
    w = mx.bf16_to_f64(mx.f64_to_bf16(w))
    q, s = bs.bs_quantize_weight(w)
    assert s.shape == (3, 2)
    for i, (lo, hi) in enumerate(((0, 128), (128, 256), (256, 300))):
        for kb in range(2):
            blk = w[lo:hi, kb * 128:(kb + 1) * 128]
            assert s[i, kb] == np.float32(np.abs(blk).max()) / np.float32(448.0)
    deq = bs.bs_dequantize_weight(q, s)
    step = np.repeat(s.astype(np.float64)[np.arange(300) // 128], 128, axis=1)
    # half the E4M3 spacing at the top of the range (32 / 2) in units of the block scale
    assert np.all(np.abs(deq - w) <= 16.0 * step * (1 + 1e-6))
    xq, xs = bs.bs_quantize_act(w[:7])
    assert np.all(np.abs(bs.bs_dequantize_act(xq, xs) - w[:7]) <= 16.0 * np.repeat(xs, 128, axis=1) * (1 + 1e-6))
