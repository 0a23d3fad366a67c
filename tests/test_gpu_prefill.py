"""GPU parity of causal prefill / extend attention (tcgen05) and of the prefill KV append.

The caches are filled on the GPU by kv_append_extend and checked bit for bit against the
oracle's append; attention is held against the fp64 oracle to the bound its arithmetic gives:
P enters the PV product in bf16, so |err| <= 2^-8 * max|V| + one bf16 step of the output."""
import math

import numpy as np
import pytest
import torch

from mxfp8_mlp_gqa_gb300 import api, synth
from oracle import mx, ops
from tests.gpu_util import bf16_ulp, dev, dev_bf16, host_bits, host_f64

pytestmark = pytest.mark.gpu
D = 128


def _garbage(shape):
    t = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    v = t.view(torch.int16).view(-1, 2)
    v[:, 0] = int(np.int16(np.uint16(0x461C).view(np.int16)))
    v[:, 1] = int(np.uint16(0xC61C).view(np.int16))
    return t


def _case(prefix, new, Hq, Hkv, seed):
    """bf16 bits of q [total_q, Hq, D], the whole K/V of each sequence [Hkv, P+T, D] and the
    new tokens' K/V rows [total_q, Hkv, D]."""
    lens = np.asarray(prefix) + np.asarray(new)
    total = int(np.sum(new))
    q = synth.normal_bf16((total, Hq, D), 1.0, seed, synth.TID["q"])
    kp = synth.kv_prefix(len(lens), Hkv, D, lens, seed, synth.TID["k"])
    vp = synth.kv_prefix(len(lens), Hkv, D, lens, seed, synth.TID["v"])
    kn = np.concatenate([np.transpose(k[:, k.shape[1] - t:], (1, 0, 2)) for k, t in zip(kp, new)])
    vn = np.concatenate([np.transpose(v[:, v.shape[1] - t:], (1, 0, 2)) for v, t in zip(vp, new)])
    q_start = np.concatenate([[0], np.cumsum(new)]).astype(np.int32)
    return q, kp, vp, kn, vn, q_start, lens.astype(np.int32)


def _caches(kp, vp, new, kn, vn, q_start, lens, cap, max_q):
    """Contiguous caches holding each prefix, then the new rows appended on the GPU (checked
    bit for bit against the oracle's append)."""
    bs, Hkv = len(kp), kp[0].shape[0]
    K, V = _garbage((bs, Hkv, cap, D)), _garbage((bs, Hkv, cap, D))
    for b in range(bs):
        P = kp[b].shape[1] - new[b]
        if P:
            K[b, :, :P].copy_(dev_bf16(kp[b][:, :P]))
            V[b, :, :P].copy_(dev_bf16(vp[b][:, :P]))
    k0, v0 = host_bits(K).astype(np.uint16), host_bits(V).astype(np.uint16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.kv_append_extend(K, V, dev_bf16(kn), dev_bf16(vn), dev(q_start), dev(lens), max_q, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    kc, vc = ops.kv_append_extend(k0, v0, [kn[q_start[b]:q_start[b + 1]] for b in range(bs)],
                                  [vn[q_start[b]:q_start[b + 1]] for b in range(bs)], lens)
    np.testing.assert_array_equal(host_bits(K), kc)
    np.testing.assert_array_equal(host_bits(V), vc)
    return K, V


def _check(out, q, kp, vp, q_start, scale, rows=None):
    got = host_f64(out)
    assert np.isfinite(got).all()
    qf = mx.bf16_to_f64(q)
    for b in range(len(kp)):
        K, V = mx.bf16_to_f64(kp[b]), mx.bf16_to_f64(vp[b])
        T = int(q_start[b + 1] - q_start[b])
        n = K.shape[1]
        idx = range(T) if rows is None else [i for i in rows if i < T]
        for i in idx:
            # new token i: an extend of one token over the prefix up to its own position
            pos = n - T + i
            (ref,) = ops.gqa_prefill_attention([qf[q_start[b] + i][None]], [K[:, :pos + 1]], [V[:, :pos + 1]], scale)
            bound = 2.0 ** -8 * np.abs(V[:, :pos + 1]).max() + bf16_ulp(ref[0])
            err = np.abs(got[q_start[b] + i] - ref[0])
            assert np.all(err <= bound), (b, i, float(err.max()))


@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (8, 8), (16, 8), (64, 8)])
def test_prefill_from_scratch(Hq, Hkv):
    new = [200, 77, 1, 129]
    q, kp, vp, kn, vn, q_start, lens = _case([0] * 4, new, Hq, Hkv, seed=Hq)
    K, V = _caches(kp, vp, new, kn, vn, q_start, lens, 256, 256)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = api.gqa_prefill_attn(dev_bf16(q), K, V, dev(q_start), dev(lens), 256, 1 / math.sqrt(D), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    _check(out, q, kp, vp, q_start, 1 / math.sqrt(D))


def test_extend_over_cached_prefixes():
    prefix, new = [100, 1000, 0, 383, 64], [50, 130, 128, 1, 64]
    q, kp, vp, kn, vn, q_start, lens = _case(prefix, new, 32, 8, seed=7)
    K, V = _caches(kp, vp, new, kn, vn, q_start, lens, 1536, 130)
    out = api.gqa_prefill_attn(dev_bf16(q), K, V, dev(q_start), dev(lens), 130, 0.08)
    _check(out, q, kp, vp, q_start, 0.08)


def test_paged_extend_is_bit_identical_to_contiguous():
    prefix, new, ps = [300, 64, 0], [200, 100, 257], 64
    q, kp, vp, kn, vn, q_start, lens = _case(prefix, new, 32, 8, seed=3)
    K, V = _caches(kp, vp, new, kn, vn, q_start, lens, 1024, 257)
    out_c = api.gqa_prefill_attn(dev_bf16(q), K, V, dev(q_start), dev(lens), 257, 0.09)
    # the same prefixes in randomly placed pages; new rows appended through the paged append
    need = [(int(n) + ps - 1) // ps for n in lens]
    num_pages = sum(need) + 4
    perm = np.random.default_rng(5).permutation(num_pages)
    kpool, vpool = _garbage((num_pages, 8, ps, D)), _garbage((num_pages, 8, ps, D))
    table = np.full((3, 1024 // ps), -1, np.int32)
    k = 0
    for b in range(3):
        P = int(prefix[b])
        for j in range(need[b]):
            table[b, j] = perm[k]
            lo, hi = j * ps, min(P, (j + 1) * ps)
            if hi > lo:
                kpool[int(perm[k]), :, :hi - lo].copy_(dev_bf16(kp[b][:, lo:hi]))
                vpool[int(perm[k]), :, :hi - lo].copy_(dev_bf16(vp[b][:, lo:hi]))
            k += 1
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    tb = dev(table)
    api.kv_append_extend_paged(kpool, vpool, tb, dev_bf16(kn), dev_bf16(vn), dev(q_start), dev(lens), 257, err=err)
    out_p = api.gqa_prefill_attn_paged(dev_bf16(q), kpool, vpool, tb, dev(q_start), dev(lens), 257, 0.09, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(out_p.view(torch.int16), out_c.view(torch.int16))
    _check(out_p, q, kp, vp, q_start, 0.09, rows=[0, 1, 63, 64, 127, 128, 199, 256])


def test_long_prefill_sampled_rows():
    # one 4096-token prefill (S2-Pro shape, 32 q / 8 kv heads): 32 tiles of 128 keys
    new = [4096]
    q, kp, vp, kn, vn, q_start, lens = _case([0], new, 32, 8, seed=11)
    K, V = _caches(kp, vp, new, kn, vn, q_start, lens, 4096, 4096)
    out = api.gqa_prefill_attn(dev_bf16(q), K, V, dev(q_start), dev(lens), 4096, 1 / math.sqrt(D))
    rows = sorted(set(np.random.default_rng(0).integers(0, 4096, 24).tolist()) | {0, 31, 32, 4095})
    _check(out, q, kp, vp, q_start, 1 / math.sqrt(D), rows=rows)


def test_inconsistent_lengths_set_the_flag():
    new = [40, 60]
    q, kp, vp, kn, vn, q_start, lens = _case([10, 0], new, 32, 8, seed=2)
    K, V = _caches(kp, vp, new, kn, vn, q_start, lens, 128, 60)
    bad = lens.copy()
    bad[1] = 30  # fewer cached positions than new tokens
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.zeros((100, 32, D), dtype=torch.bfloat16, device="cuda")
    api.gqa_prefill_attn(dev_bf16(q), K, V, dev(q_start), dev(bad), 60, 0.1, out=out, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 7
    assert not host_f64(out)[40:].any()  # the bad sequence was skipped
    _check(out[:40].contiguous(), q[:40], kp[:1], vp[:1], q_start[:2], 0.1)


def test_paged_bad_page_id_sets_the_flag():
    prefix, new, ps = [0, 0], [70, 130], 64
    q, kp, vp, kn, vn, q_start, lens = _case(prefix, new, 32, 8, seed=8)
    kpool, vpool = _garbage((8, 8, ps, D)), _garbage((8, 8, ps, D))
    table = np.array([[3, 6, -1], [0, 5, 1]], np.int32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.kv_append_extend_paged(kpool, vpool, dev(table), dev_bf16(kn), dev_bf16(vn), dev(q_start), dev(lens), 130,
                               err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    table[1, 2] = 99  # outside the pool: sequence 1's last 64 keys
    out = api.gqa_prefill_attn_paged(dev_bf16(q), kpool, vpool, dev(table), dev(q_start), dev(lens), 130, 0.09,
                                     err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 7
    assert np.isfinite(host_f64(out)).all()
    _check(out[:70].contiguous(), q[:70], kp[:1], vp[:1], q_start[:2], 0.09)


def test_host_checks():
    q = torch.zeros((4, 8, 64), dtype=torch.bfloat16, device="cuda")
    K = torch.zeros((1, 2, 64, 64), dtype=torch.bfloat16, device="cuda")
    qs, kl = dev(np.array([0, 4], np.int32)), dev(np.array([4], np.int32))
    with pytest.raises(api.MxgError):  # head dim 64: the tensor-core prefill needs 128
        api.gqa_prefill_attn(q, K, K, qs, kl, 4, 0.1)
