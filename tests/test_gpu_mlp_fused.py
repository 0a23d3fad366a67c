"""The one-launch decode MLP kernel against the two-launch path (the gate/up + SwiGLU launch,
then the split-K down GEMM). Both split the down projection at the same K boundaries,
accumulate each split in the same order and sum the splits in split order, so y and the
workspace's hq / hs agree bit for bit; the two-launch path itself is held to the oracle in
test_gpu_mlp. Also: consecutive calls that share one workspace (its control words return to
zero after every call) and the status word of the bounded waits."""
import numpy as np
import pytest
import torch

from mxfp8_mlp_gqa_gb300 import api, synth
from oracle import mx, ops
from tests.gpu_util import assert_float_close, assert_requant_close, dev_bf16, host_f64

pytestmark = pytest.mark.gpu

_W = {}


def _weights(d_model, d_ff):
    key = (d_model, d_ff)
    if key not in _W:
        _W.clear()
        w13 = api.mxfp8_quantize(dev_bf16(synth.weights(2 * d_ff, d_model, 0, synth.TID["w13"])))
        w2 = api.mxfp8_quantize(dev_bf16(synth.weights(d_model, d_ff, 0, synth.TID["w2"])))
        _W[key] = (w13, w2)
    return _W[key]


def _inputs(M, d_model, seed, residual):
    x = synth.activations(M, d_model, seed, outlier_frac=0.01)
    xq, xs = api.mxfp8_quantize(dev_bf16(x))
    res = dev_bf16(synth.activations(M, d_model, seed, tid=synth.TID["residual"])) if residual else None
    return x, xq, xs, res


def _run(xq, xs, w13, w2, res, fused, ws=None):
    prev = api.lib().mxg_set_mlp_fused(1 if fused else 0)
    try:
        M, d_model = xq.shape
        if ws is None:
            ws = torch.zeros(api.mlp_swiglu_mxfp8_workspace(M, d_model, w2[0].shape[1]), dtype=torch.uint8,
                             device="cuda")
        y = api.mlp_swiglu_mxfp8(xq, xs, *w13, *w2, residual=res, workspace=ws)
    finally:
        api.lib().mxg_set_mlp_fused(prev)
    return y, ws


def _ctrl_bytes(d_model):
    return (d_model // 128 + 3) * 128


@pytest.mark.parametrize("M", [1, 2, 7, 16, 17, 32, 33, 64, 100, 128])
@pytest.mark.parametrize("residual", [False, True])
def test_one_launch_equals_two_launch(M, residual):
    d_model, d_ff = 2560, 9728
    w13, w2 = _weights(d_model, d_ff)
    _, xq, xs, res = _inputs(M, d_model, M, residual)
    y1, ws1 = _run(xq, xs, w13, w2, res, fused=True)
    y2, ws2 = _run(xq, xs, w13, w2, res, fused=False)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    nh = M * d_ff + M * d_ff // 32  # hq then hs at the start of the workspace
    assert torch.equal(ws1[:nh], ws2[:nh])
    assert not ws1[-_ctrl_bytes(d_model):].any()  # counters back at zero, status word clear


@pytest.mark.parametrize("M", [1, 5])
def test_one_launch_small_configuration(M):
    # the d_model 256 / d_ff 768 layer: 12 gate/up tiles, 2 row tiles x 6 splits
    d_model, d_ff = 256, 768
    w13, w2 = _weights(d_model, d_ff)
    x, xq, xs, res = _inputs(M, d_model, 3, True)
    y1, _ = _run(xq, xs, w13, w2, res, fused=True)
    y2, _ = _run(xq, xs, w13, w2, res, fused=False)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    ow13 = mx.mx_quantize(mx.bf16_to_f64(synth.weights(2 * d_ff, d_model, 0, synth.TID["w13"])))
    ow2 = mx.mx_quantize(mx.bf16_to_f64(synth.weights(d_model, d_ff, 0, synth.TID["w2"])))
    ref = ops.swiglu_mlp(*mx.mx_quantize(mx.bf16_to_f64(x)), *ow13, *ow2,
                         residual_bf16=synth.activations(M, d_model, 3, tid=synth.TID["residual"]))
    assert_float_close(host_f64(y1), ref["y"])


def test_back_to_back_calls_share_one_workspace():
    # four calls enqueued with no synchronisation between them, on one workspace: each call
    # finds its counters at zero (the previous call's last CTA reset them) and reads only the
    # h it wrote itself
    d_model, d_ff, M = 2560, 9728, 24
    w13, w2 = _weights(d_model, d_ff)
    ws = torch.zeros(api.mlp_swiglu_mxfp8_workspace(M, d_model, d_ff), dtype=torch.uint8, device="cuda")
    cases = [_inputs(M, d_model, 40 + k, k % 2 == 0) for k in range(4)]
    outs = [_run(xq, xs, w13, w2, res, fused=True, ws=ws)[0] for _, xq, xs, res in cases]
    torch.cuda.synchronize()
    assert not ws[-_ctrl_bytes(d_model):].any()
    for (_, xq, xs, res), y in zip(cases, outs):
        ref, _ = _run(xq, xs, w13, w2, res, fused=False)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16))


def test_one_launch_requant_matches_oracle():
    # the hq / hs the one-launch kernel leaves in its workspace are the oracle's re-quantised h
    d_model, d_ff, M = 2560, 9728, 64
    w13, w2 = _weights(d_model, d_ff)
    x, xq, xs, _ = _inputs(M, d_model, 9, False)
    _, ws = _run(xq, xs, w13, w2, None, fused=True)
    torch.cuda.synchronize()
    hq = ws[:M * d_ff].view(M, d_ff).cpu().numpy()
    hs = ws[M * d_ff:M * d_ff + M * d_ff // 32].view(M, d_ff // 32).cpu().numpy()
    ow13 = mx.mx_quantize(mx.bf16_to_f64(synth.weights(2 * d_ff, d_model, 0, synth.TID["w13"])))
    X = mx.mx_dequantize(*mx.mx_quantize(mx.bf16_to_f64(x)))
    W13 = mx.mx_dequantize(*ow13)
    H = ops.silu(X @ W13[:d_ff].T) * (X @ W13[d_ff:].T)
    rq, rs = mx.mx_quantize(H)
    assert_requant_close(hq, hs, rq, rs)
