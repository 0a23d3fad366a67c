"""Both GEMM kernel paths against the oracle: the tcgen05 block-scaled kernel (default where
K % 128 == 0) and the CUDA-core kernel (forced through mxg_set_tensor_core_path(0)), on
hand-built MX operands whose scales vary per row, per token and per 32-block -- a mapping
error of the scale factors in either kernel fails these."""
import numpy as np
import pytest
import torch

from mxfp8_mlp_gqa_gb300 import api, synth
from oracle import mx, ops
from tests.gpu_util import assert_float_close, assert_requant_close, dev_bf16, host_f64

pytestmark = pytest.mark.gpu


def _codes(shape, g):
    c = g.integers(0, 256, size=shape).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x38  # no NaN codes
    return c


@pytest.fixture(params=[True, False], ids=["tcgen05", "cuda-core"])
def path(request):
    prev = api.set_tensor_core_path(request.param)
    yield request.param
    api.set_tensor_core_path(prev)


@pytest.mark.parametrize("M,N,K", [(1, 256, 128), (16, 256, 512), (64, 2560, 4096), (77, 136, 256),
                                   (128, 6144, 2560), (200, 512, 384), (300, 1024, 1024), (1100, 264, 384),
                                   (2048, 520, 512), (2048, 256, 1024)])
def test_gemm_structured_scales(path, M, N, K):
    g = synth.rng(11, M * 7 + N)
    xq, wq = _codes((M, K), g), _codes((N, K), g)
    xs = (115 + (np.arange(M)[:, None] * 5 + np.arange(K // 32)[None, :]) % 23).astype(np.uint8)
    ws = (110 + (np.arange(N)[:, None] * 7 + np.arange(K // 32)[None, :] * 3) % 29).astype(np.uint8)
    res = synth.activations(M, N, 2, tid=synth.TID["residual"])
    d = lambda a: torch.from_numpy(a).cuda()  # noqa: E731
    c = api.mxfp8_gemm(d(xq), d(xs), d(wq), d(ws), residual=dev_bf16(res))
    ref = ops.mx_gemm(xq, xs, wq, ws) + mx.bf16_to_f64(res)
    # per-block scales spanning 2^-17..2^11 make the outputs heavy-tailed, so the bound on
    # the largest error is taken against max |ref| (bf16 output rounding is 2^-9 of that)
    got = host_f64(c)
    assert np.linalg.norm(got - ref) <= 1e-2 * np.linalg.norm(ref)
    assert np.abs(got - ref).max() <= 1e-2 * np.abs(ref).max()


@pytest.mark.parametrize("M", [1, 5, 33, 128, 130])
def test_mlp_both_paths(path, M):
    d_model, d_ff = 512, 1024
    x = synth.activations(M, d_model, 4, outlier_frac=0.01)
    w13 = synth.weights(2 * d_ff, d_model, 4, synth.TID["w13"])
    w2 = synth.weights(d_model, d_ff, 4, synth.TID["w2"])
    xq, xs = api.mxfp8_quantize(dev_bf16(x))
    g13, g2 = api.mxfp8_quantize(dev_bf16(w13)), api.mxfp8_quantize(dev_bf16(w2))
    hq, hs = api.mlp_gate_up_swiglu_mxfp8(xq, xs, *g13)
    y = api.mlp_swiglu_mxfp8(xq, xs, *g13, *g2)
    ref = ops.swiglu_mlp(*mx.mx_quantize(mx.bf16_to_f64(x)), *mx.mx_quantize(mx.bf16_to_f64(w13)),
                         *mx.mx_quantize(mx.bf16_to_f64(w2)))
    assert_requant_close(hq.cpu().numpy(), hs.cpu().numpy(), ref["hq"], ref["hs"])
    assert_float_close(host_f64(y), ref["y"])


def test_split_k_cluster_reduction_is_deterministic():
    # split-K partials are summed inside a thread-block cluster in a fixed order: repeated
    # calls give identical bits, and no workspace is needed
    M, N, K = 8, 1024, 4096
    g = synth.rng(3, 3)
    xq, wq = _codes((M, K), g), _codes((N, K), g)
    xs = np.full((M, K // 32), 124, np.uint8)
    ws = np.full((N, K // 32), 125, np.uint8)
    d = lambda a: torch.from_numpy(a).cuda()  # noqa: E731
    assert api.mxfp8_gemm_workspace(M, N, K) == 0
    outs = [api.mxfp8_gemm(d(xq), d(xs), d(wq), d(ws)).clone() for _ in range(3)]
    assert all(torch.equal(outs[0].view(torch.int16), o.view(torch.int16)) for o in outs[1:])
    assert_float_close(host_f64(outs[0]), ops.mx_gemm(xq, xs, wq, ws))


@pytest.mark.parametrize("M,N,K", [(1100, 264, 384), (2048, 520, 512), (1500, 1032, 256), (1025, 8, 128),
                                   (4100, 2056, 256), (3000, 4104, 384)])
def test_large_gemm_plain_store(M, N, K):
    # more than 1024 tokens and no residual: the persistent CTA-pair kernel writes its tiles
    # through staged copy-engine stores, clipped at ragged M / N edges (the last two shapes give
    # each pair two or more tiles, ragged ones included); every output element must be written
    g = synth.rng(12, M + N)
    xq, wq = _codes((M, K), g), _codes((N, K), g)
    xs = (115 + (np.arange(M)[:, None] * 5 + np.arange(K // 32)[None, :]) % 23).astype(np.uint8)
    ws = (110 + (np.arange(N)[:, None] * 7 + np.arange(K // 32)[None, :] * 3) % 29).astype(np.uint8)
    d = lambda a: torch.from_numpy(a).cuda()  # noqa: E731
    c = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    api.mxfp8_gemm(d(xq), d(xs), d(wq), d(ws), c=c)
    got = host_f64(c)
    assert not np.isnan(got).any()
    ref = ops.mx_gemm(xq, xs, wq, ws)
    assert np.linalg.norm(got - ref) <= 1e-2 * np.linalg.norm(ref)
    assert np.abs(got - ref).max() <= 1e-2 * np.abs(ref).max()
