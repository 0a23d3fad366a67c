"""GPU parity of prev_tokens_shift and kv_append (bit-exact), including the degenerate
cases and the device error flag for an out-of-range kv_len."""
import numpy as np
import pytest
import torch

from mxfp8_mlp_gqa_gb300 import api, synth
from oracle import ops
from tests.gpu_util import dev, dev_bf16, host_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("bs,W,cw,ncodes", [(1, 8, 10, 1024), (64, 16, 10, 4096), (3, 1, 10, 4096),
                                            (5, 7, 3, 1 << 31), (2, 1024, 12, 4096)])
def test_prev_tokens_shift_bit_exact(bs, W, cw, ncodes):
    prev = synth.codes((bs, W, cw), min(ncodes, 2 ** 31 - 1), 0, synth.TID["prev"])
    nxt = synth.codes((bs, cw), min(ncodes, 2 ** 31 - 1), 0, synth.TID["next"])
    p = dev(prev)
    ptr = p.data_ptr()
    api.prev_tokens_shift(p, dev(nxt))
    assert p.data_ptr() == ptr  # in place
    np.testing.assert_array_equal(p.cpu().numpy(), ops.prev_tokens_shift(prev, nxt))


def test_prev_tokens_shift_repeated_equals_history():
    bs, W, cw = 4, 16, 10
    p = dev(synth.codes((bs, W, cw), 4096, 1, synth.TID["prev"]))
    hist = [synth.codes((bs, cw), 4096, 1, 200 + i) for i in range(W)]
    for h in hist:
        api.prev_tokens_shift(p, dev(h))
    np.testing.assert_array_equal(p.cpu().numpy(), np.stack(hist, axis=1))


def test_prev_tokens_shift_contract():
    p = torch.zeros((2, 4, 10), dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        api.prev_tokens_shift(p, torch.zeros((2, 1, 10), dtype=torch.int32, device="cuda"))  # unsqueezed next
    with pytest.raises(TypeError):
        api.prev_tokens_shift(p, torch.zeros((2, 10), dtype=torch.int64, device="cuda"))     # promoted dtype
    with pytest.raises(TypeError):
        api.prev_tokens_shift(p.to(torch.int64), torch.zeros((2, 10), dtype=torch.int32, device="cuda"))


def test_kv_append_bit_exact_and_error_flag():
    bs, Hkv, D, cap = 4, 8, 128, 64
    kc = synth.normal_bf16((bs, Hkv, cap, D), 1.0, 0, synth.TID["k"])
    vc = synth.normal_bf16((bs, Hkv, cap, D), 1.0, 0, synth.TID["v"])
    # new rows as strided slices of a fused [bs, (Hq + 2 Hkv) * D] projection output
    qkv = synth.normal_bf16((bs, (32 + 2 * Hkv) * D), 1.0, 0, synth.TID["q"])
    lens = np.array([1, 17, 64, 30], np.int32)
    K, V = dev_bf16(kc), dev_bf16(vc)
    Q = dev_bf16(qkv)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.kv_append(K, V, Q[:, 32 * D:(32 + Hkv) * D], Q[:, (32 + Hkv) * D:], dev(lens), err=err)
    kn = qkv[:, 32 * D:(32 + Hkv) * D].reshape(bs, Hkv, D)
    vn = qkv[:, (32 + Hkv) * D:].reshape(bs, Hkv, D)
    ek, ev = ops.kv_append(kc, vc, kn, vn, lens)
    np.testing.assert_array_equal(host_bits(K), ek)
    np.testing.assert_array_equal(host_bits(V), ev)
    assert int(err.item()) == 0
    # kv_len out of [1, cap]: flagged, that sequence untouched, the others written
    bad = np.array([0, 5, cap + 1, 9], np.int32)
    api.kv_append(K, V, Q[:, 32 * D:(32 + Hkv) * D], Q[:, (32 + Hkv) * D:], dev(bad), err=err)
    assert int(err.item()) == 7
    got = host_bits(K)
    np.testing.assert_array_equal(got[0], ek[0])
    np.testing.assert_array_equal(got[2], ek[2])
    np.testing.assert_array_equal(got[1, :, 4], kn[1])
    np.testing.assert_array_equal(got[3, :, 8], kn[3])
