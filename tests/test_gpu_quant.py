"""GPU parity of the MX activation quantiser (bit-exact) and of RMSNorm+quantise
(bit-exact: both sides take the bf16 rounding that decides the codes at the same
precision -- fp64 mean of squares, fp32 products)."""
import numpy as np
import pytest
import torch

from mxfp8_mlp_gqa_gb300 import api, synth
from oracle import mx, ops
from tests import golden
from tests.gpu_util import dev_bf16

pytestmark = pytest.mark.gpu


def _quant_check(bits):
    q, s = api.mxfp8_quantize(dev_bf16(bits))
    oq, os_ = mx.mx_quantize(mx.bf16_to_f64(bits))
    np.testing.assert_array_equal(s.cpu().numpy(), os_)
    np.testing.assert_array_equal(q.cpu().numpy(), oq)


def test_hand_worked_blocks_bit_exact():
    blocks = golden.mx_blocks()
    vals = np.stack([b[1] for b in blocks])
    bits = synth.f32_to_bf16_bits(vals.astype(np.float32))
    q, s = api.mxfp8_quantize(dev_bf16(bits))
    for i, (name, _, scale, codes) in enumerate(blocks):
        assert int(s[i, 0]) == scale, name
        np.testing.assert_array_equal(q[i].cpu().numpy(), codes, err_msg=name)


@pytest.mark.parametrize("M,K", [(1, 256), (1, 2560), (3, 2560), (64, 2560), (128, 2560), (37, 9728), (64, 4096),
                                 (5, 32), (1, 96)])
def test_activations_bit_exact(M, K):
    _quant_check(synth.activations(M, K, seed=0, outlier_frac=0.01))


def test_weights_bit_exact_qwen3_shapes():
    # weight prep of the Qwen3-4B-shaped MLP: W13 [19456, 2560] and W2 [2560, 9728], N(0, 0.02)
    _quant_check(synth.weights(19456, 2560, 0, synth.TID["w13"]))
    _quant_check(synth.weights(2560, 9728, 0, synth.TID["w2"]))


def test_wide_dynamic_range_and_special_values():
    g = np.random.default_rng(7)
    a = g.standard_normal((96, 512)).astype(np.float32) * np.exp2(g.integers(-140, 126, (96, 1))).astype(np.float32)
    a[0] = 0.0
    a[1, ::2] = -0.0
    a[2] = np.float32(2.0 ** -133)   # bf16 subnormals
    a[3, :32] = 1.0
    bits = synth.f32_to_bf16_bits(a)
    bits[4] = 0x7F7F                 # bf16 max finite everywhere
    _quant_check(bits)


def test_strided_rows():
    x = synth.activations(8, 4096, seed=1)
    xt = dev_bf16(x)[:, 1024:3072]      # row stride 4096, K = 2048
    q, s = api.mxfp8_quantize(xt)
    oq, os_ = mx.mx_quantize(mx.bf16_to_f64(x[:, 1024:3072]))
    np.testing.assert_array_equal(q.cpu().numpy(), oq)
    np.testing.assert_array_equal(s.cpu().numpy(), os_)


def test_empty_input():
    q, s = api.mxfp8_quantize(torch.empty((0, 64), dtype=torch.bfloat16, device="cuda"))
    assert q.shape == (0, 64) and s.shape == (0, 2)


def test_binding_rejects_promotion_and_reshaping():
    with pytest.raises(TypeError):
        api.mxfp8_quantize(torch.zeros((1, 64), dtype=torch.float32, device="cuda"))
    with pytest.raises(ValueError):
        api.mxfp8_quantize(torch.zeros((64,), dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(api.MxgError):
        api.mxfp8_quantize(torch.zeros((1, 48), dtype=torch.bfloat16, device="cuda"))


@pytest.mark.parametrize("M,K", [(1, 256), (64, 2560), (7, 4096), (2, 32)])
def test_rmsnorm_quantize_bit_exact(M, K):
    x = synth.activations(M, K, seed=3, outlier_frac=0.01)
    gam = synth.gamma(K, 3, synth.TID["gamma1"])
    q, s = api.rmsnorm_mxfp8_quantize(dev_bf16(x), dev_bf16(gam), 1e-6)
    oq, os_ = ops.rmsnorm_mx_quantize(x, gam, 1e-6)
    np.testing.assert_array_equal(s.cpu().numpy(), os_)
    np.testing.assert_array_equal(q.cpu().numpy(), oq)


def test_rmsnorm_factor_near_a_rounding_midpoint():
    # Rows of ones with eps = 3 * 2^-24 put 1/sqrt(1 + eps) within ~2^-46 of the point halfway
    # between the fp32 numbers 1 - 2^-24 and 1 - 2^-23: the kernel's fp32 estimate of the factor
    # cannot decide that rounding and takes the fp64 sequence. Rows of other values and the
    # other eps take the estimate. Both must give the oracle's codes and scales bit for bit.
    K = 2560
    rng = np.random.default_rng(5)
    rows = [np.full(K, 1.0), np.full(K, -1.0)] + [rng.standard_normal(K) for _ in range(6)]
    x = mx.f64_to_bf16(np.array(rows))
    gam = synth.gamma(K, 5, synth.TID["gamma1"])
    for eps in (3 * 2.0 ** -24, 2.0 ** -24, 1e-6):
        eps32 = float(np.float32(eps))
        q, s = api.rmsnorm_mxfp8_quantize(dev_bf16(x), dev_bf16(gam), eps32)
        oq, os_ = ops.rmsnorm_mx_quantize(x, gam, eps32)
        np.testing.assert_array_equal(s.cpu().numpy(), os_)
        np.testing.assert_array_equal(q.cpu().numpy(), oq)
