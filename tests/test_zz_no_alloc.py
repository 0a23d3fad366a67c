"""The allocation-free attention entry point (gqa_decode_attn_noalloc).

It serves callers that cannot allocate device memory where attention runs (inside CUDA
graph capture, real-time threads, hosts that own the memory budget): its split-KV scratch is
a fixed device array inside the library. These tests call it through the C ABI and check it
against gqa_decode_attn (caller-provided workspace) on two calls in a row with different
shapes, so that scratch left behind by the first call cannot leak into the second. The file
is named to be collected last."""
import math

import numpy as np
import pytest
import torch

from mxfp8_mlp_gqa_gb300 import api, synth
from tests.gpu_util import dev, dev_bf16, host_f64

pytestmark = pytest.mark.gpu


def _case(bs, Hq, Hkv, D, cap, lo, hi, seed):
    lens = synth.kv_lens(bs, lo, hi, seed=seed)
    q = dev_bf16(synth.normal_bf16((bs, Hq, D), 1.0, seed, synth.TID["q"]))
    K = torch.empty((bs, Hkv, cap, D), dtype=torch.bfloat16, device="cuda")
    V = torch.empty_like(K)
    kp = synth.kv_prefix(bs, Hkv, D, lens, seed, synth.TID["k"])
    vp = synth.kv_prefix(bs, Hkv, D, lens, seed, synth.TID["v"])
    K.view(torch.int16).fill_(0x461C)
    V.view(torch.int16).fill_(-0x39E4)
    for b in range(bs):
        K[b, :, :lens[b]].copy_(dev_bf16(kp[b]))
        V[b, :, :lens[b]].copy_(dev_bf16(vp[b]))
    return q, K, V, dev(lens)


def test_noalloc_matches_workspace_entry_point_two_calls():
    for bs, Hq, Hkv, D, cap, lo, hi, seed in [(64, 32, 8, 128, 32768, 234, 4096, 0), (8, 16, 2, 64, 2048, 1, 2048, 1)]:
        q, K, V, kl = _case(bs, Hq, Hkv, D, cap, lo, hi, seed)
        scale = 1 / math.sqrt(D)
        ref = api.gqa_decode_attn(q, K, V, kl, hi, scale)
        got = torch.empty_like(ref)
        api.gqa_decode_attn_noalloc(q, K, V, kl, hi, scale, got)
        torch.cuda.synchronize()
        err = np.abs(host_f64(got) - host_f64(ref)).max()
        assert err <= 2e-3, err
        # same kernels, same split plan: the results agree bit for bit
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


def test_noalloc_rejects_problems_beyond_its_scratch():
    cap_bytes = api.lib().gqa_decode_attn_noalloc_capacity()
    assert cap_bytes == 8 << 20
    bs, Hq, Hkv, D, mkv = 512, 32, 8, 128, 4096
    assert api.gqa_decode_attn_workspace(bs, Hq, Hkv, D, mkv) > cap_bytes
    q = torch.zeros((bs, Hq, D), dtype=torch.bfloat16, device="cuda")
    K = torch.zeros((bs, Hkv, 16, D), dtype=torch.bfloat16, device="cuda")
    kl = torch.ones((bs,), dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(api.MxgError) as e:
        api.gqa_decode_attn_noalloc(q, K, K, kl, mkv, 0.1, out)
    assert e.value.status == 9
