"""Failure detection on the device, exercised without a fault: a bounded in-kernel wait is
made to run out and the kernel must report MXG_ETIMEOUT through the error flag, leave no
stale output behind and return, after which the context still works.

The library's test hook mxg_debug_stall_attn_loads(1) makes the split-KV decode attention's
copy warp issue no loads, so the consumer warps wait on pipeline stages that nothing fills (a
flag nobody sets). Their waits give up after the 2 s bound, the warps meet at the merge
barrier and leave together ([FSKV] §5 on bounds checks that report instead of trapping)."""
import math

import numpy as np
import pytest
import torch

from mxfp8_mlp_gqa_gb300 import api, synth
from oracle import ops
from tests.gpu_util import assert_attn_close, dev, dev_bf16, host_f64

pytestmark = pytest.mark.gpu

MXG_ETIMEOUT = 6


def _case(bs, Hq, Hkv, D, cap, lo, hi, seed):
    lens = synth.kv_lens(bs, lo, hi, seed=seed)
    qh = synth.normal_bf16((bs, Hq, D), 1.0, seed, synth.TID["q"])
    kp = synth.kv_prefix(bs, Hkv, D, lens, seed, synth.TID["k"])
    vp = synth.kv_prefix(bs, Hkv, D, lens, seed, synth.TID["v"])
    K = torch.zeros((bs, Hkv, cap, D), dtype=torch.bfloat16, device="cuda")
    V = torch.zeros_like(K)
    for b in range(bs):
        K[b, :, :lens[b]].copy_(dev_bf16(kp[b]))
        V[b, :, :lens[b]].copy_(dev_bf16(vp[b]))
    return dev_bf16(qh), K, V, dev(lens), qh, kp, vp


@pytest.mark.parametrize("shape", [
    (1, 4, 2, 64, 1024, 50, 64),      # one split (max_kv_len <= 64): the split kernel writes the output
    (1, 8, 2, 128, 1024, 300, 640),   # up to 10 splits of 64 tokens, merged by the combine kernel
])
@pytest.mark.parametrize("fused_mx", [False, True])
def test_attention_wait_runs_out_and_reports(shape, fused_mx):
    bs, Hq, Hkv, D, cap, lo, hi = shape
    q, K, V, kl, qh, kp, vp = _case(bs, Hq, Hkv, D, cap, lo, hi, 0)
    scale = 1 / math.sqrt(D)
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")
    out = torch.full((bs, Hq, D), 7.0, dtype=torch.bfloat16, device="cuda")
    oq = torch.full((bs, Hq * D), 0x55, dtype=torch.uint8, device="cuda") if fused_mx else None
    os_ = torch.full((bs, Hq * D // 32), 0x55, dtype=torch.uint8, device="cuda") if fused_mx else None
    assert api.lib().mxg_debug_stall_attn_loads(1) == 0
    try:
        api.gqa_decode_attn(q, K, V, kl, hi, scale, out=out, err=err, oq=oq, os=os_)
        torch.cuda.synchronize()
    finally:
        assert api.lib().mxg_debug_stall_attn_loads(0) == 0
    assert int(err.item()) == MXG_ETIMEOUT
    assert not out.float().abs().any()             # no stale or partial output
    if fused_mx:
        assert not oq.any() and not os_.any()
    # the context is healthy: the same call now runs to completion and matches the oracle
    err.zero_()
    api.gqa_decode_attn(q, K, V, kl, hi, scale, out=out, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    from oracle import mx
    ref = ops.gqa_decode_attention(mx.bf16_to_f64(qh), [mx.bf16_to_f64(k) for k in kp],
                                   [mx.bf16_to_f64(v) for v in vp], scale)
    assert_attn_close(host_f64(out), ref)
