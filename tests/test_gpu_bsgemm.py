"""GPU parity of the block-scaled FP8 (bsgemm recipe) quantisers (bit for bit) and GEMM
(rel. Frobenius <= 1e-2, max <= 3e-2 * rms, the MXFP8 GEMM's bound) against the fp64 oracle,
at decode shapes with split K, ragged M / N tails and a one-group K."""
import numpy as np
import pytest
import torch

from mxfp8_mlp_gqa_gb300 import api, synth
from oracle import bs, mx
from tests.gpu_util import assert_float_close, dev, dev_bf16, host_f64

pytestmark = pytest.mark.gpu


def _bits(shape, std, seed, tid, outliers=False):
    b = synth.normal_bf16(shape, std, seed, tid)
    if outliers:
        v = mx.bf16_to_f64(b)
        v[:, ::97] *= 20.0
        b = mx.f64_to_bf16(v)
    return b


def test_quantisers_bit_exact():
    x = _bits((7, 2560), 1.0, 1, synth.TID["x"], outliers=True)
    w = mx.bf16_to_f64(_bits((300, 256), 0.02, 2, synth.TID["w13"]))
    w[128:256, :128] = 0.0            # an all-zero 128x128 block
    w[256:, 128:] *= 1e4              # a short last row block with large values
    w = mx.f64_to_bf16(w)
    xq, xs = api.bs_quantize_act(dev_bf16(x))
    wq, ws = api.bs_quantize_weight(dev_bf16(w))
    torch.cuda.synchronize()
    oq, os_ = bs.bs_quantize_act(mx.bf16_to_f64(x))
    wq_o, ws_o = bs.bs_quantize_weight(mx.bf16_to_f64(w))
    np.testing.assert_array_equal(xq.cpu().numpy(), oq)
    np.testing.assert_array_equal(xs.cpu().numpy().view(np.uint32), os_.view(np.uint32))
    np.testing.assert_array_equal(wq.cpu().numpy(), wq_o)
    np.testing.assert_array_equal(ws.cpu().numpy().view(np.uint32), ws_o.view(np.uint32))
    assert ws_o[1, 0] == 0


@pytest.mark.parametrize("M,N,K", [(1, 2560, 9728), (16, 2560, 2560), (64, 4096, 2560), (128, 300, 512),
                                   (77, 200, 1024), (5, 128, 128), (33, 6144, 2560)])
def test_gemm_vs_oracle(M, N, K):
    x = _bits((M, K), 1.0, M, synth.TID["x"], outliers=True)
    w = _bits((N, K), 0.02, N, synth.TID["w13"])
    xq, xs = api.bs_quantize_act(dev_bf16(x))
    wq, ws = api.bs_quantize_weight(dev_bf16(w))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = api.bs_gemm(xq, xs, wq, ws, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    oq, os_ = bs.bs_quantize_act(mx.bf16_to_f64(x))
    wq_o, ws_o = bs.bs_quantize_weight(mx.bf16_to_f64(w))
    ref = bs.bs_gemm(oq, os_, wq_o, ws_o)
    assert_float_close(host_f64(out), ref)


def test_gemm_sampled_at_the_gate_up_shape():
    # M = 64 tokens through the Qwen3-4B gate/up weight (19456 x 2560): 256 sampled columns
    M, N, K = 64, 19456, 2560
    x = _bits((M, K), 1.0, 3, synth.TID["x"], outliers=True)
    w = _bits((N, K), 0.02, 4, synth.TID["w13"])
    xq, xs = api.bs_quantize_act(dev_bf16(x))
    wq, ws = api.bs_quantize_weight(dev_bf16(w))
    out = host_f64(api.bs_gemm(xq, xs, wq, ws))
    cols = np.sort(np.random.default_rng(0).choice(N, 256, replace=False))
    oq, os_ = bs.bs_quantize_act(mx.bf16_to_f64(x))
    wsub = mx.bf16_to_f64(w)
    wq_o, ws_o = bs.bs_quantize_weight(wsub)
    wsel = mx.e4m3_value(wq_o[cols]) * np.repeat(ws_o.astype(np.float64)[cols // 128], 128, axis=1)
    ref = bs.bs_dequantize_act(oq, os_) @ wsel.T
    assert_float_close(out[:, cols], ref)


def test_several_token_tiles_and_host_checks():
    M, N, K = 300, 640, 1024  # three 128-token tiles, a ragged last one
    x = _bits((M, K), 1.0, 9, synth.TID["x"])
    w = _bits((N, K), 0.02, 10, synth.TID["w13"])
    xq, xs = api.bs_quantize_act(dev_bf16(x))
    wq, ws = api.bs_quantize_weight(dev_bf16(w))
    out = api.bs_gemm(xq, xs, wq, ws)
    oq, os_ = bs.bs_quantize_act(mx.bf16_to_f64(x))
    wq_o, ws_o = bs.bs_quantize_weight(mx.bf16_to_f64(w))
    assert_float_close(host_f64(out), bs.bs_gemm(oq, os_, wq_o, ws_o))
    bad = torch.zeros((4, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(api.MxgError):  # K % 128 != 0
        api.bs_quantize_act(bad)
