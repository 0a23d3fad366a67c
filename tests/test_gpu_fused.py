"""The fused entry points of the decoder-layer step against the unfused calls they replace:
gqa_decode_attn_mxfp8 == gqa_decode_attn + mxfp8_quantize (bit-exact), and
mxfp8_gemm_qkv_kv_append == mxfp8_gemm + kv_append (bit-exact), including the error path
of an out-of-range kv_len; and the programmatic-dependent-launch chain of a weight quantiser
followed by a GEMM that reads the weight."""
import math

import numpy as np
import pytest
import torch

from mxfp8_mlp_gqa_gb300 import api, synth
from oracle import mx, ops
from tests.gpu_util import assert_float_close, dev, dev_bf16, host_f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("bs,mkv", [(8, 2048), (3, 64), (64, 2048)])
def test_attention_with_fused_quant_is_bit_exact(bs, mkv):
    Hq, Hkv, D, cap = 32, 8, 128, mkv
    lens = synth.kv_lens(bs, 1, mkv, seed=bs)
    lens[0] = 0 if bs > 3 else lens[0]  # an invalid sequence: zero output and zero codes
    q = dev_bf16(synth.normal_bf16((bs, Hq, D), 1.0, 7, synth.TID["q"]))
    K = dev_bf16(synth.normal_bf16((bs, Hkv, cap, D), 1.0, 7, synth.TID["k"]))
    V = dev_bf16(synth.normal_bf16((bs, Hkv, cap, D), 1.0, 7, synth.TID["v"]))
    kl = dev(lens)
    ref = api.gqa_decode_attn(q, K, V, kl, mkv, 1 / math.sqrt(D))
    rq, rs = api.mxfp8_quantize(ref.view(bs, Hq * D))
    oq = torch.empty((bs, Hq * D), dtype=torch.uint8, device="cuda")
    os_ = torch.empty((bs, Hq * D // 32), dtype=torch.uint8, device="cuda")
    out, oq, os_ = api.gqa_decode_attn(q, K, V, kl, mkv, 1 / math.sqrt(D), oq=oq, os=os_)
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(oq, rq) and torch.equal(os_, rs)


def test_qkv_projection_with_fused_kv_append_is_bit_exact():
    M, K, Hq, Hkv, D, cap = 16, 2560, 32, 8, 128, 256
    N = (Hq + 2 * Hkv) * D
    x = dev_bf16(synth.activations(M, K, 3))
    w = dev_bf16(synth.weights(N, K, 3, synth.TID["wqkv"]))
    xq, xs = api.mxfp8_quantize(x)
    wq, ws = api.mxfp8_quantize(w)
    lens = synth.kv_lens(M, 1, cap, seed=3)
    kc = dev_bf16(synth.normal_bf16((M, Hkv, cap, D), 1.0, 3, synth.TID["k"]))
    vc = dev_bf16(synth.normal_bf16((M, Hkv, cap, D), 1.0, 3, synth.TID["v"]))
    kc2, vc2 = kc.clone(), vc.clone()
    ref = api.mxfp8_gemm(xq, xs, wq, ws)
    api.kv_append(kc2, vc2, ref[:, Hq * D:(Hq + Hkv) * D], ref[:, (Hq + Hkv) * D:], dev(lens))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    qkv = api.mxfp8_gemm_qkv_kv_append(xq, xs, wq, ws, Hq, Hkv, kc, vc, dev(lens), err=err)
    assert int(err.item()) == 0
    assert torch.equal(qkv[:, :Hq * D].view(torch.int16), ref[:, :Hq * D].view(torch.int16))
    assert torch.equal(kc.view(torch.int16), kc2.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), vc2.view(torch.int16))
    # an out-of-range length: flagged, that sequence's rows untouched
    bad = lens.copy()
    bad[5] = cap + 1
    kc3 = kc.clone()
    api.mxfp8_gemm_qkv_kv_append(xq, xs, wq, ws, Hq, Hkv, kc3, vc, dev(bad), err=err)
    assert int(err.item()) == 7
    assert torch.equal(kc3[5].view(torch.int16), kc[5].view(torch.int16))


def test_back_to_back_weight_quantise_then_gemm():
    """mxfp8_quantize(W); mxfp8_quantize(x); mxfp8_gemm(x, W) enqueued with nothing in between:
    the GEMM may start copying W before its immediate predecessor (the x quantiser) has
    finished, but never before the W quantiser two launches back has completed. W's buffers
    first hold the codes of another matrix, so a read that came too early would show."""
    M, N, K = 16, 19456, 2560
    w_old = dev_bf16(synth.weights(N, K, 1, synth.TID["w13"], 0.5))
    w_new = synth.weights(N, K, 0, synth.TID["w13"])
    x = synth.activations(M, K, 0, outlier_frac=0.01)
    wq = torch.empty((N, K), dtype=torch.uint8, device="cuda")
    ws = torch.empty((N, K // 32), dtype=torch.uint8, device="cuda")
    xq = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    xs = torch.empty((M, K // 32), dtype=torch.uint8, device="cuda")
    c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    w_dev, x_dev = dev_bf16(w_new), dev_bf16(x)
    ref = ops.mx_gemm(*mx.mx_quantize(mx.bf16_to_f64(x)), *mx.mx_quantize(mx.bf16_to_f64(w_new)))
    for _ in range(3):
        api.mxfp8_quantize(w_old, q=wq, s=ws)
        torch.cuda.synchronize()
        api.mxfp8_quantize(w_dev, q=wq, s=ws)
        api.mxfp8_quantize(x_dev, q=xq, s=xs)
        api.mxfp8_gemm(xq, xs, wq, ws, c=c)
        torch.cuda.synchronize()
        assert_float_close(host_f64(c), ref)
