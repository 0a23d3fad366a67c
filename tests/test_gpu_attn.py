"""GPU parity of GQA decode attention over the active prefix (max |err| <= 2e-3 against
the fp64 oracle), at the tiny configuration (4/2 heads, head_dim 64, cap 1024,
kv_len 100) and the full S2-Pro shape (32/8 heads, head_dim 128, cap 32768, ragged
kv_len ~ U[234, 4096], bs 1..64), plus the invariants of the active-prefix reading: a
+-1e4 tail never changes a bit of the output, kv_len = 1 returns V_0, and out-of-range
lengths raise the device flag and zero that sequence."""
import math

import numpy as np
import pytest
import torch

from mxfp8_mlp_gqa_gb300 import api, synth
from oracle import mx, ops
from tests.gpu_util import assert_attn_close, dev, dev_bf16, host_f64

pytestmark = pytest.mark.gpu


def _device_cache(bs, Hkv, cap, D, prefix, tail="garbage"):
    """Device cache [bs, Hkv, cap, D]: the tail holds the +-1e4 pattern (or zeros), then the
    prefixes are copied in."""
    c = torch.empty((bs, Hkv, cap, D), dtype=torch.bfloat16, device="cuda")
    if tail == "garbage":
        v = c.view(torch.int16).view(-1, 2)
        v[:, 0] = int(np.int16(np.uint16(0x461C).view(np.int16)))
        v[:, 1] = int(np.uint16(0xC61C).view(np.int16))
    else:
        c.zero_()
    for b in range(bs):
        n = prefix[b].shape[1]
        if n:
            c[b, :, :n].copy_(dev_bf16(prefix[b]))
    return c


def _run(bs, Hq, Hkv, D, cap, lens, scale, max_kv_len=None, seed=0, tail="garbage", q_bits=None):
    lens = np.asarray(lens, np.int32)
    q = q_bits if q_bits is not None else synth.normal_bf16((bs, Hq, D), 1.0, seed, synth.TID["q"])
    kp = synth.kv_prefix(bs, Hkv, D, np.minimum(np.maximum(lens, 0), cap), seed, synth.TID["k"])
    vp = synth.kv_prefix(bs, Hkv, D, np.minimum(np.maximum(lens, 0), cap), seed, synth.TID["v"])
    K = _device_cache(bs, Hkv, cap, D, kp, tail)
    V = _device_cache(bs, Hkv, cap, D, vp, tail)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = api.gqa_decode_attn(dev_bf16(q), K, V, dev(lens), max_kv_len or cap, scale, err=err)
    torch.cuda.synchronize()
    return q, kp, vp, out, err


def _oracle(q, kp, vp, scale):
    return ops.gqa_decode_attention(mx.bf16_to_f64(q), [mx.bf16_to_f64(k) for k in kp],
                                    [mx.bf16_to_f64(v) for v in vp], scale)


def test_tiny_configuration():
    q, kp, vp, out, err = _run(1, 4, 2, 64, 1024, [100], 1 / 8)
    ref = _oracle(q, kp, vp, 1 / 8)
    assert_attn_close(host_f64(out), ref)
    assert int(err.item()) == 0


@pytest.mark.parametrize("bs", [1, 4, 8, 16, 32, 64])  # bs 4: 512-token splits (at most 32 (b, g) pairs)
def test_s2pro_shape_ragged(bs):
    lens = synth.kv_lens(bs, 234, 4096, seed=0)
    q, kp, vp, out, err = _run(bs, 32, 8, 128, 32768, lens, 1 / math.sqrt(128), max_kv_len=4096)
    ref = _oracle(q, kp, vp, 1 / math.sqrt(128))
    assert_attn_close(host_f64(out), ref)
    assert int(err.item()) == 0


def test_garbage_tail_is_never_read_bitwise():
    bs, cap = 8, 4096
    lens = synth.kv_lens(bs, 1, cap, seed=5)
    _, _, _, a, _ = _run(bs, 32, 8, 128, cap, lens, 0.0884, seed=5, tail="garbage")
    _, _, _, b, _ = _run(bs, 32, 8, 128, cap, lens, 0.0884, seed=5, tail="zero")
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("D,Hq,Hkv", [(128, 32, 8), (64, 4, 2), (128, 8, 8), (64, 16, 2), (128, 8, 1)])
def test_length_edges_and_group_sizes(D, Hq, Hkv):
    cap = 4096
    # tile (64), split and capacity boundaries
    lens = [1, 2, 63, 64, 65, 127, 128, 129, 511, 512, 513, 1000, 2047, 2048, 4095, 4096]
    q, kp, vp, out, err = _run(len(lens), Hq, Hkv, D, cap, lens, 1 / math.sqrt(D), seed=2)
    ref = _oracle(q, kp, vp, 1 / math.sqrt(D))
    got = host_f64(out)
    assert_attn_close(got, ref, floor_ulp=True)  # prefixes of 1..2 tokens: |o| ~ |V|
    # kv_len = 1: softmax weight 1, out = V_0 (rounded to bf16 once, as stored)
    g = Hq // Hkv
    for h in range(Hq):
        np.testing.assert_array_equal(got[0, h], mx.bf16_to_f64(vp[0])[h // g, 0])
    assert int(err.item()) == 0


def test_single_split_path():
    # a small max_kv_len bound -> one split per (b, g): the split kernel writes out directly
    lens = [1, 7, 40, 64]
    q, kp, vp, out, err = _run(4, 32, 8, 128, 256, lens, 0.09, max_kv_len=64, seed=3)
    assert_attn_close(host_f64(out), _oracle(q, kp, vp, 0.09), floor_ulp=True)
    assert api.gqa_decode_attn_workspace(4, 32, 8, 128, 64) == 0


def test_invalid_lengths_flag_and_zero():
    cap, mkv = 1024, 512
    lens = [0, 100, cap + 5, 600, 300]   # 0, > cap and > max_kv_len are invalid
    q, kp, vp, out, err = _run(5, 8, 2, 64, cap, lens, 0.125, max_kv_len=mkv, seed=4)
    assert int(err.item()) == 7
    got = host_f64(out)
    for b in (0, 2, 3):
        assert not got[b].any()
    ref = _oracle(q[[1, 4]], [kp[1], kp[4]], [vp[1], vp[4]], 0.125)
    assert_attn_close(got[[1, 4]], ref)


def test_strided_q_from_fused_projection():
    bs, Hq, Hkv, D, cap = 4, 32, 8, 128, 2048
    lens = synth.kv_lens(bs, 234, 2048, seed=6)
    fused = synth.normal_bf16((bs, (Hq + 2 * Hkv) * D), 1.0, 6, synth.TID["q"])
    kp = synth.kv_prefix(bs, Hkv, D, lens, 6, synth.TID["k"])
    vp = synth.kv_prefix(bs, Hkv, D, lens, 6, synth.TID["v"])
    K, V = _device_cache(bs, Hkv, cap, D, kp), _device_cache(bs, Hkv, cap, D, vp)
    out = api.gqa_decode_attn(dev_bf16(fused)[:, :Hq * D], K, V, dev(lens), cap, 0.0884)
    q = fused[:, :Hq * D].reshape(bs, Hq, D)
    assert_attn_close(host_f64(out), _oracle(q, kp, vp, 0.0884))
