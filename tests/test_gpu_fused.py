"""The fused entry points of the decoder-layer step against the unfused calls they replace:
gqa_decode_attn_mxfp8 == gqa_decode_attn + mxfp8_quantize (bit-exact), and
mxfp8_gemm_qkv_kv_append == mxfp8_gemm + kv_append (bit-exact), including the error path
of an out-of-range kv_len; and programmatic-dependent-launch chains: a weight quantiser
followed by a GEMM that reads the weight, and a KV append, an extend append or a kv_len copy
followed by decode attention (which reads kv_len and the prefix before its own wait)."""
import math

import numpy as np
import pytest
import torch

from mxfp8_mlp_gqa_gb300 import api, synth
from oracle import mx, ops
from tests.gpu_util import assert_attn_close, assert_float_close, dev, dev_bf16, host_f64

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


# --- decode attention reads kv_len and the prefix below row kv_len - 1 before its wait ---

def _attn_ref(q, kp, vp, scale):
    return ops.gqa_decode_attention(mx.bf16_to_f64(q), [mx.bf16_to_f64(k) for k in kp],
                                    [mx.bf16_to_f64(v) for v in vp], scale)


def _cache(kp, bs, Hkv, cap, D, old=None):
    """Host bf16 bits [bs, Hkv, cap, D]: the prefixes, zeros past them; rows old[b] (a slice
    of positions) replaced by other values (what the cache held before the append)."""
    c = np.zeros((bs, Hkv, cap, D), np.uint16)
    for b in range(bs):
        c[b, :, :kp[b].shape[1]] = kp[b]
        if old is not None:
            sl = old[b]
            c[b, :, sl] = synth.normal_bf16((Hkv, sl.stop - sl.start, D), 4.0, b, synth.TID["v"])
    return c


def test_back_to_back_append_then_decode_attention():
    """kv_append (row kv_len - 1) and gqa_decode_attn enqueued with nothing in between: the
    attention issues its tiles below row kv_len - 1 while the append may still run, and the
    appended row only after it. That row first holds other values, so an early read shows."""
    bs, Hq, Hkv, D, cap, scale = 8, 32, 8, 128, 2048, 1 / math.sqrt(128)
    lens = synth.kv_lens(bs, 130, cap, seed=11)
    q = synth.normal_bf16((bs, Hq, D), 1.0, 11, synth.TID["q"])
    kp = synth.kv_prefix(bs, Hkv, D, lens, 11, synth.TID["k"])
    vp = synth.kv_prefix(bs, Hkv, D, lens, 11, synth.TID["v"])
    old = [slice(int(n) - 1, int(n)) for n in lens]
    k0, v0 = _cache(kp, bs, Hkv, cap, D, old), _cache(vp, bs, Hkv, cap, D, old)
    kn = dev_bf16(np.stack([k[:, -1] for k in kp]))  # [bs, Hkv, D]
    vn = dev_bf16(np.stack([v[:, -1] for v in vp]))
    K = torch.empty((bs, Hkv, cap, D), dtype=torch.bfloat16, device="cuda")
    V = torch.empty_like(K)
    qd, kl = dev_bf16(q), dev(lens)
    out = torch.empty((bs, Hq, D), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(max(1, api.gqa_decode_attn_workspace(bs, Hq, Hkv, D, cap)), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = _attn_ref(q, kp, vp, scale)
    for _ in range(3):
        K.copy_(dev_bf16(k0))
        V.copy_(dev_bf16(v0))
        torch.cuda.synchronize()
        api.kv_append(K, V, kn, vn, kl, err=err)
        api.gqa_decode_attn(qd, K, V, kl, cap, scale, out=out, err=err, workspace=ws)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_attn_close(host_f64(out), ref)


def test_back_to_back_extend_append_then_decode_attention():
    """kv_append_extend writes the last T rows of each prefix and lets its successor start
    only when it completes: decode attention enqueued right after it sees all T new rows
    (they first hold other values)."""
    bs, Hq, Hkv, D, cap, scale = 8, 32, 8, 128, 2048, 1 / math.sqrt(128)
    lens = synth.kv_lens(bs, 300, cap, seed=12)
    T = np.array([1, 64, 100, 200, 257, 33, 150, 299], np.int32)
    q = synth.normal_bf16((bs, Hq, D), 1.0, 12, synth.TID["q"])
    kp = synth.kv_prefix(bs, Hkv, D, lens, 12, synth.TID["k"])
    vp = synth.kv_prefix(bs, Hkv, D, lens, 12, synth.TID["v"])
    old = [slice(int(n) - int(t), int(n)) for n, t in zip(lens, T)]
    k0, v0 = _cache(kp, bs, Hkv, cap, D, old), _cache(vp, bs, Hkv, cap, D, old)
    kn = dev_bf16(np.concatenate([k[:, -int(t):].transpose(1, 0, 2) for k, t in zip(kp, T)]))  # [total, Hkv, D]
    vn = dev_bf16(np.concatenate([v[:, -int(t):].transpose(1, 0, 2) for v, t in zip(vp, T)]))
    q_start = dev(np.concatenate([[0], np.cumsum(T)]).astype(np.int32))
    K = torch.empty((bs, Hkv, cap, D), dtype=torch.bfloat16, device="cuda")
    V = torch.empty_like(K)
    qd, kl = dev_bf16(q), dev(lens)
    out = torch.empty((bs, Hq, D), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(max(1, api.gqa_decode_attn_workspace(bs, Hq, Hkv, D, cap)), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = _attn_ref(q, kp, vp, scale)
    for _ in range(3):
        K.copy_(dev_bf16(k0))
        V.copy_(dev_bf16(v0))
        torch.cuda.synchronize()
        api.kv_append_extend(K, V, kn, vn, q_start, kl, int(T.max()), err=err)
        api.gqa_decode_attn(qd, K, V, kl, cap, scale, out=out, err=err, workspace=ws)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_attn_close(host_f64(out), ref)


def test_back_to_back_kv_len_copy_then_decode_attention():
    """copy_bytes writing kv_len from pinned host memory, then decode attention with nothing in
    between: the attention reads kv_len before its own wait, which is safe because the copy
    lets its successor start only when it completes (kv_len first holds other lengths)."""
    bs, Hq, Hkv, D, cap, scale = 8, 32, 8, 128, 2048, 1 / math.sqrt(128)
    lens = synth.kv_lens(bs, 200, cap, seed=13)
    q = synth.normal_bf16((bs, Hq, D), 1.0, 13, synth.TID["q"])
    kp = synth.kv_prefix(bs, Hkv, D, lens, 13, synth.TID["k"])
    vp = synth.kv_prefix(bs, Hkv, D, lens, 13, synth.TID["v"])
    K, V = dev_bf16(_cache(kp, bs, Hkv, cap, D)), dev_bf16(_cache(vp, bs, Hkv, cap, D))
    kl = torch.empty(bs, dtype=torch.int32, device="cuda")
    host = torch.from_numpy(lens.copy()).pin_memory()
    qd = dev_bf16(q)
    out = torch.empty((bs, Hq, D), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(max(1, api.gqa_decode_attn_workspace(bs, Hq, Hkv, D, cap)), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = _attn_ref(q, kp, vp, scale)
    for _ in range(3):
        kl.copy_(dev(lens // 2))
        torch.cuda.synchronize()
        api.copy_bytes(kl, host)
        api.gqa_decode_attn(qd, K, V, kl, cap, scale, out=out, err=err, workspace=ws)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_attn_close(host_f64(out), ref)
