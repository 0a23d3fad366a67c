"""Pins of the oracle's MX rules (CPU only) against hand-worked blocks, torch's
float8 casts (an independent library implementation of E4M3 / E8M0) and brute
force over the E4M3 code table."""
import math

import numpy as np
import pytest
import torch

from oracle import mx
from tests import golden

BLOCKS = golden.mx_blocks()


@pytest.mark.parametrize("name,vals,scale,codes", BLOCKS, ids=[b[0] for b in BLOCKS])
def test_hand_worked_blocks(name, vals, scale, codes):
    q, s = mx.mx_quantize(vals[None, :])
    assert int(s[0, 0]) == scale, name
    np.testing.assert_array_equal(q[0], codes, err_msg=name)


def test_hand_worked_inputs_are_bf16():
    for name, vals, _, _ in BLOCKS:
        t = torch.tensor(vals, dtype=torch.float64)
        assert torch.equal(t.to(torch.float32).to(torch.bfloat16).to(torch.float64), t), name


def test_e4m3_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = mx.e4m3_value(codes)
    nan = np.isnan(ref)
    np.testing.assert_array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    assert nan.sum() == 2  # 0x7F and 0xFF only


def test_e4m3_closed_form_landmarks():
    v = mx.e4m3_value(np.array([0x38, 0x7E, 0x01, 0x08, 0x07, 0x80, 0xB8], np.uint8))
    assert list(v[:5]) == [1.0, 448.0, 2.0 ** -9, 2.0 ** -6, 7 * 2.0 ** -9]
    assert v[5] == 0.0 and math.copysign(1, v[5]) == -1.0 and v[6] == -1.0


def test_e4m3_roundtrip_all_finite_codes():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    np.testing.assert_array_equal(mx.e4m3_encode(mx.e4m3_value(codes)), codes)


def test_e4m3_encode_matches_torch_in_range():
    g = np.random.default_rng(1)
    # fp32 values (torch's cast rounds from fp32 once) spread over the normal,
    # subnormal and underflow ranges, below the saturation threshold 464
    mag = np.exp2(g.uniform(-14, math.log2(463.9), 200000)).astype(np.float32)
    v = (mag * np.where(g.random(mag.size) < 0.5, -1, 1)).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = mx.e4m3_encode(v.astype(np.float64))
    np.testing.assert_array_equal(got, ref)


def test_e4m3_encode_saturates():
    v = np.array([448.0, 463.99, 464.0, 480.0, 1e6, -500.0, -1e30])
    np.testing.assert_array_equal(mx.e4m3_encode(v), [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE])


def _brute_force_e4m3(v):
    """Nearest finite E4M3 value by exhaustive search; ties -> even code; |v| above
    448 -> 448; the sign of zero kept."""
    finite = [c for c in range(128) if c != 0x7F]
    vals = [float(torch.tensor([c], dtype=torch.uint8).view(torch.float8_e4m3fn).float()) for c in finite]
    out = []
    for x in v:
        a = min(abs(x), 448.0)
        best = None
        for c, val in zip(finite, vals):
            d = abs(a - val)
            if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
                best = (d, c)
        out.append(best[1] | (0x80 if math.copysign(1, x) < 0 else 0))
    return np.array(out, np.uint8)


def test_e4m3_encode_brute_force():
    g = np.random.default_rng(2)
    v = np.concatenate([
        g.normal(0, 50, 300), g.normal(0, 0.01, 200),
        np.array([0.5 * 2 ** -9, 1.5 * 2 ** -9, 2.5 * 2 ** -9, 7.5 * 2 ** -9, 15.5 * 2 ** -9,
                  -0.0, 0.0, 17.0, 18.0, 19.0, 232.0, 240.0, 248.0, 464.0, 470.0]),
    ])
    np.testing.assert_array_equal(mx.e4m3_encode(v), _brute_force_e4m3(v))


def test_scale_decode_matches_torch_e8m0():
    b = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(b).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = mx.scale_value(b)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])


def test_mx_quantize_properties_random():
    g = np.random.default_rng(3)
    x = g.normal(0, 1, (64, 256)) * np.exp2(g.integers(-20, 20, (64, 1)))
    x = torch.tensor(x).to(torch.bfloat16).double().numpy()
    q, s = mx.mx_quantize(x)
    blk = x.reshape(64, 8, 32)
    amax = np.abs(blk).max(-1)
    # the scale is the largest power of two with amax / 2^s < 512 = 2^(emax+1)
    sv = s.astype(np.int64) - 127
    assert np.all(amax * np.exp2(-sv.astype(float)) < 512) and np.all(amax * np.exp2(-sv.astype(float)) >= 256)
    # dequantised error <= half an E4M3 step at each element's binade (or saturation 448 ... 512)
    d = mx.mx_dequantize(q, s).reshape(64, 8, 32)
    scaled = np.abs(blk) * np.exp2(-sv.astype(float))[..., None]
    step = np.exp2(np.maximum(np.floor(np.log2(np.maximum(scaled, 1e-300))), -6) - 3)
    err = np.abs(blk - d) * np.exp2(-sv.astype(float))[..., None]
    sat = scaled > 448
    assert np.all(err[~sat] <= step[~sat] / 2)
    assert np.all(np.abs(d[sat]) * np.exp2(-sv[..., None].repeat(32, -1)[sat].astype(float)) == 448)


def test_f64_to_bf16_matches_torch_for_fp32_values():
    g = np.random.default_rng(4)
    v = (g.normal(0, 1, 100000) * np.exp2(g.integers(-130, 120, 100000))).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(mx.f64_to_bf16(v.astype(np.float64)), ref)


def test_f64_to_bf16_single_rounding_brute_force():
    # fp64 values just above/below bf16 midpoints: a double rounding through
    # fp32 would get some of these wrong; exhaustive neighbour search decides
    g = np.random.default_rng(5)
    base = torch.tensor(g.normal(0, 1, 2000), dtype=torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    v = []
    for b in base:
        nb = float(torch.tensor([b]).to(torch.bfloat16).view(torch.int16).add(1).view(torch.bfloat16).double())
        mid = (b + nb) / 2
        v += [mid, mid + abs(mid) * 2.0 ** -40, mid - abs(mid) * 2.0 ** -40]
    v = np.array(v)
    got = mx.bf16_to_f64(mx.f64_to_bf16(v))
    for x, y in zip(v, got):
        lo = float(torch.tensor([x], dtype=torch.float64).to(torch.float32).to(torch.bfloat16).double())
        cands = set()
        for c in (lo,):
            i = int(torch.tensor([c]).to(torch.bfloat16).view(torch.int16))
            for d in (-1, 0, 1):
                cands.add(float(torch.tensor([i + d], dtype=torch.int16).view(torch.bfloat16).double()))
        best = min(cands, key=lambda c: (abs(c - x), int(torch.tensor([c]).to(torch.bfloat16).view(torch.int16)) & 1))
        assert y == best, (x, y, best)
