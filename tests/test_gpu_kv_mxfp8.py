"""GPU parity of decode attention over an MXFP8 K/V cache and of the MX-quantising KV append.

The cache contents on both sides come from the same seeded bf16 prefixes: the GPU quantises
them with its own kernel (mxfp8_quantize over rows of D, which must match the oracle's codes
bit for bit), the oracle with its own MX rule; attention is then held to max |err| <= 2e-3
against the fp64 oracle over the dequantised cache, the append bit for bit. Entries no
sequence owns hold E4M3 NaN codes (0x7F) and exponent bytes 0xFF."""
import math

import numpy as np
import pytest
import torch

from mxfp8_mlp_gqa_gb300 import api, synth
from mxfp8_mlp_gqa_gb300.api import MxgError
from oracle import mx, ops
from tests.gpu_util import assert_attn_close, bf16_ulp, dev, dev_bf16, host_f64

pytestmark = pytest.mark.gpu


def _filled(shape, byte):
    return torch.full(shape, byte, dtype=torch.uint8, device="cuda")


def _gpu_rows_mx(prefix_bits):
    """GPU MX quantisation of a prefix [Hkv, n, D] (bf16 bits) along D."""
    Hkv, n, D = prefix_bits.shape
    q, s = api.mxfp8_quantize(dev_bf16(prefix_bits.reshape(Hkv * n, D)))
    return q.view(Hkv, n, D), s.view(Hkv, n, D // 32)


def _oracle_rows_mx(prefix_bits):
    return ops.kv_rows_mx(mx.bf16_to_f64(prefix_bits))


def _mx_cache(prefix, cap):
    """Contiguous MXFP8 cache (codes, scales) [bs, Hkv, cap, D (/32)] holding the GPU-quantised
    prefixes; the oracle's codes are checked equal on the way."""
    bs, (Hkv, _, D) = len(prefix), prefix[0].shape
    c, s = _filled((bs, Hkv, cap, D), 0x7F), _filled((bs, Hkv, cap, D // 32), 0xFF)
    for b, p in enumerate(prefix):
        n = p.shape[1]
        if n:
            qg, sg = _gpu_rows_mx(p)
            qo, so = _oracle_rows_mx(p)
            assert np.array_equal(qg.cpu().numpy(), qo) and np.array_equal(sg.cpu().numpy(), so)
            c[b, :, :n].copy_(qg)
            s[b, :, :n].copy_(sg)
    return c, s


def _oracle(q, kp, vp, scale):
    kq = [_oracle_rows_mx(k) for k in kp]
    vq = [_oracle_rows_mx(v) for v in vp]
    return ops.gqa_decode_attention_kv_mxfp8(mx.bf16_to_f64(q), [c for c, _ in kq], [s for _, s in kq],
                                             [c for c, _ in vq], [s for _, s in vq], scale)


def _case(bs, Hq, Hkv, D, lens, seed):
    q = synth.normal_bf16((bs, Hq, D), 1.0, seed, synth.TID["q"])
    kp = synth.kv_prefix(bs, Hkv, D, lens, seed, synth.TID["k"])
    vp = synth.kv_prefix(bs, Hkv, D, lens, seed, synth.TID["v"])
    return q, kp, vp


@pytest.mark.parametrize("bs", [1, 4, 8, 64])  # bs 4: 512-token splits
def test_attention_vs_oracle_s2pro_shape(bs):
    Hq, Hkv, D, mkv, cap = 32, 8, 128, 4096, 4096
    lens = synth.kv_lens(bs, 234, mkv, seed=bs)
    q, kp, vp = _case(bs, Hq, Hkv, D, lens, bs)
    kc, ks = _mx_cache(kp, cap)
    vc, vs = _mx_cache(vp, cap)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    scale = 1 / math.sqrt(D)
    out = api.gqa_decode_attn_kv_mxfp8(dev_bf16(q), kc, ks, vc, vs, dev(lens), mkv, scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_attn_close(host_f64(out), _oracle(q, kp, vp, scale))


@pytest.mark.parametrize("D,Hq,Hkv", [(64, 4, 2), (128, 8, 8), (64, 16, 2), (128, 8, 1)])
def test_length_edges_and_group_sizes(D, Hq, Hkv):
    lens = np.array([1, 2, 63, 64, 65, 127, 128, 129, 500, 1024], np.int32)
    q, kp, vp = _case(len(lens), Hq, Hkv, D, lens, 11)
    kc, ks = _mx_cache(kp, 1024)
    vc, vs = _mx_cache(vp, 1024)
    out = api.gqa_decode_attn_kv_mxfp8(dev_bf16(q), kc, ks, vc, vs, dev(lens), 1024, 0.125)
    assert_attn_close(host_f64(out), _oracle(q, kp, vp, 0.125), floor_ulp=True)


def test_wide_dynamic_range_rows():
    # rows scaled token by token by 2^-6 .. 2^6 (K) and 2^-40 .. 2^40 (V): every block keeps its
    # own exponent, and the V exponents reach far outside f16's range on the P side
    bs, Hq, Hkv, D = 4, 8, 2, 128
    lens = np.array([37, 300, 640, 1000], np.int32)
    q, kp, vp = _case(bs, Hq, Hkv, D, lens, 21)
    f32 = lambda bits: mx.bf16_to_f64(bits)  # noqa: E731
    kp2, vp2 = [], []
    rng = np.random.default_rng(4)
    for k, v in zip(kp, vp):
        ek = rng.integers(-6, 7, size=(1, k.shape[1], 1))
        ev = rng.integers(-40, 41, size=(1, v.shape[1], 1))
        kp2.append(mx.f64_to_bf16(f32(k) * np.exp2(ek)))
        vp2.append(mx.f64_to_bf16(f32(v) * np.exp2(ev)))
    kc, ks = _mx_cache(kp2, 1024)
    vc, vs = _mx_cache(vp2, 1024)
    out = api.gqa_decode_attn_kv_mxfp8(dev_bf16(q), kc, ks, vc, vs, dev(lens), 1024, 0.05)
    ref = _oracle(q, kp2, vp2, 0.05)
    got = host_f64(out)
    assert np.isfinite(got).all()
    # relative to each output row's magnitude (V spans 2^80), floored at one bf16 step of the
    # element itself (the output is rounded to bf16)
    scale = np.abs(ref).max(axis=-1, keepdims=True)
    assert np.all(np.abs(got - ref) <= np.maximum(2e-3 * scale, bf16_ulp(ref)))


def test_paged_equals_contiguous_and_oracle():
    bs, Hq, Hkv, D, ps, mkv = 8, 32, 8, 128, 128, 2048
    lens = synth.kv_lens(bs, 1, mkv, seed=3)
    q, kp, vp = _case(bs, Hq, Hkv, D, lens, 3)
    need = [(int(n) + ps - 1) // ps for n in lens]
    num_pages = sum(need) + 3
    perm = np.random.default_rng(2).permutation(num_pages)
    pools = [_filled((num_pages, Hkv, ps, D), 0x7F), _filled((num_pages, Hkv, ps, D // 32), 0xFF),
             _filled((num_pages, Hkv, ps, D), 0x7F), _filled((num_pages, Hkv, ps, D // 32), 0xFF)]
    table = np.full((bs, mkv // ps), -1, np.int32)
    k = 0
    for b in range(bs):
        kq, ksc = _gpu_rows_mx(kp[b])
        vq, vsc = _gpu_rows_mx(vp[b])
        for j in range(need[b]):
            sl = slice(j * ps, min(int(lens[b]), (j + 1) * ps))
            w = sl.stop - sl.start
            for pool, arr in zip(pools, (kq, ksc, vq, vsc)):
                pool[int(perm[k]), :, :w].copy_(arr[:, sl])
            table[b, j] = perm[k]
            k += 1
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = api.gqa_decode_attn_kv_mxfp8_paged(dev_bf16(q), *pools, dev(table), dev(lens), mkv, 1 / math.sqrt(D),
                                             err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_attn_close(host_f64(out), _oracle(q, kp, vp, 1 / math.sqrt(D)))
    kc, ks = _mx_cache(kp, mkv)
    vc, vs = _mx_cache(vp, mkv)
    oc = api.gqa_decode_attn_kv_mxfp8(dev_bf16(q), kc, ks, vc, vs, dev(lens), mkv, 1 / math.sqrt(D))
    assert torch.equal(out.view(torch.int16), oc.view(torch.int16))


def test_out_of_range_kv_len_sets_flag_and_zeroes_that_sequence():
    lens = np.array([100, 5000, 0, 77], np.int32)
    safe = np.clip(lens, 0, 1024)
    q, kp, vp = _case(4, 8, 2, 64, safe, 5)
    kc, ks = _mx_cache(kp, 1024)
    vc, vs = _mx_cache(vp, 1024)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = api.gqa_decode_attn_kv_mxfp8(dev_bf16(q), kc, ks, vc, vs, dev(lens), 1024, 0.125, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 7
    got = host_f64(out)
    assert not got[1].any() and not got[2].any()
    ref = _oracle(q[[0, 3]], [kp[0], kp[3]], [vp[0], vp[3]], 0.125)
    assert_attn_close(got[[0, 3]], ref)


def test_host_checks():
    q = torch.zeros((1, 8, 128), dtype=torch.bfloat16, device="cuda")
    kc, ks = _filled((1, 2, 40, 128), 0), _filled((1, 2, 40, 4), 0)
    with pytest.raises(MxgError):  # cap % 16 != 0
        api.gqa_decode_attn_kv_mxfp8(q, kc, ks, kc, ks, dev(np.array([3], np.int32)), 40, 0.1)


def test_kv_append_mxfp8_bit_exact_contiguous_and_paged():
    bs, Hkv, D, cap, ps = 5, 8, 128, 256, 64
    lens = np.array([1, 64, 65, 200, 256], np.int32)
    kn = synth.normal_bf16((bs, Hkv, D), 1.0, 6, synth.TID["q"])
    vn = synth.normal_bf16((bs, Hkv, D), 3.0, 7, synth.TID["q"])
    bufs = [_filled((bs, Hkv, cap, D), 0x7F), _filled((bs, Hkv, cap, D // 32), 0xFF),
            _filled((bs, Hkv, cap, D), 0x7F), _filled((bs, Hkv, cap, D // 32), 0xFF)]
    host0 = [t.cpu().numpy() for t in bufs]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.kv_append_mxfp8(*bufs, dev_bf16(kn), dev_bf16(vn), dev(lens), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = ops.kv_append_mxfp8(*host0, mx.bf16_to_f64(kn), mx.bf16_to_f64(vn), lens)
    for t, r in zip(bufs, ref):
        np.testing.assert_array_equal(t.cpu().numpy(), r)
    # paged: the row of position n-1 lands in page table[b, (n-1) // ps] at (n-1) % ps
    num_pages = 12
    table = np.full((bs, cap // ps), -1, np.int32)
    perm = np.random.default_rng(1).permutation(num_pages)
    for b, n in enumerate(lens):
        table[b, (n - 1) // ps] = perm[b]
    pools = [_filled((num_pages, Hkv, ps, D), 0x7F), _filled((num_pages, Hkv, ps, D // 32), 0xFF),
             _filled((num_pages, Hkv, ps, D), 0x7F), _filled((num_pages, Hkv, ps, D // 32), 0xFF)]
    api.kv_append_mxfp8_paged(*pools, dev(table), dev_bf16(kn), dev_bf16(vn), dev(lens), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    kq, ksc = ops.kv_rows_mx(mx.bf16_to_f64(kn))
    vq, vsc = ops.kv_rows_mx(mx.bf16_to_f64(vn))
    got = [p.cpu().numpy() for p in pools]
    for b, n in enumerate(lens):
        pg, r = table[b, (n - 1) // ps], (n - 1) % ps
        for arr, want in zip(got, (kq[b], ksc[b], vq[b], vsc[b])):
            np.testing.assert_array_equal(arr[pg, :, r], want)
            arr[pg, :, r] = 0x7F if arr.shape[-1] == D else 0xFF
    assert all((a == (0x7F if a.shape[-1] == D else 0xFF)).all() for a in got)  # nothing else written


def test_paged_bad_page_id_sets_the_flag_other_sequences_intact():
    bs, Hq, Hkv, D, ps = 2, 8, 2, 128, 64
    lens = np.array([150, 90], np.int32)
    q, kp, vp = _case(bs, Hq, Hkv, D, lens, 13)
    num_pages = 6
    pools = [_filled((num_pages, Hkv, ps, D), 0x7F), _filled((num_pages, Hkv, ps, D // 32), 0xFF),
             _filled((num_pages, Hkv, ps, D), 0x7F), _filled((num_pages, Hkv, ps, D // 32), 0xFF)]
    table = np.array([[4, 0, 2, -1], [5, 1, -1, -1]], np.int32)
    for b in range(bs):
        kq, ksc = _gpu_rows_mx(kp[b])
        vq, vsc = _gpu_rows_mx(vp[b])
        for j in range((int(lens[b]) + ps - 1) // ps):
            sl = slice(j * ps, min(int(lens[b]), (j + 1) * ps))
            for pool, arr in zip(pools, (kq, ksc, vq, vsc)):
                pool[int(table[b, j]), :, :sl.stop - sl.start].copy_(arr[:, sl])
    table[1, 1] = num_pages + 3  # outside the pool
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = api.gqa_decode_attn_kv_mxfp8_paged(dev_bf16(q), *pools, dev(table), dev(lens), 256, 0.1, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 7
    assert np.isfinite(host_f64(out)).all()
    assert_attn_close(host_f64(out)[:1], _oracle(q[:1], kp[:1], vp[:1], 0.1))


def test_back_to_back_append_then_attention():
    """kv_append_mxfp8 (row kv_len - 1) and gqa_decode_attn_kv_mxfp8 enqueued with nothing in
    between: the attention issues its tiles (codes and scales) below row kv_len - 1 while the
    append may still run, the appended row only after it. That row first holds other codes
    (and the 0xFF scale), so a read that came too early would show."""
    bs, Hq, Hkv, D, cap, scale = 8, 32, 8, 128, 2048, 1 / math.sqrt(128)
    lens = synth.kv_lens(bs, 130, cap, seed=14)
    q, kp, vp = _case(bs, Hq, Hkv, D, lens, 14)
    kc, ks = _mx_cache([k[:, :-1] for k in kp], cap)  # the prefixes without their last row
    vc, vs = _mx_cache([v[:, :-1] for v in vp], cap)
    k0, s0, v0, t0 = kc.clone(), ks.clone(), vc.clone(), vs.clone()
    kn = dev_bf16(np.stack([k[:, -1] for k in kp]))  # [bs, Hkv, D]
    vn = dev_bf16(np.stack([v[:, -1] for v in vp]))
    qd, kl = dev_bf16(q), dev(lens)
    out = torch.empty((bs, Hq, D), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(max(1, api.gqa_decode_attn_workspace(bs, Hq, Hkv, D, cap)), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = _oracle(q, kp, vp, scale)
    for _ in range(3):
        for dst, src in ((kc, k0), (ks, s0), (vc, v0), (vs, t0)):
            dst.copy_(src)
        torch.cuda.synchronize()
        api.kv_append_mxfp8(kc, ks, vc, vs, kn, vn, kl, err=err)
        api.gqa_decode_attn_kv_mxfp8(qd, kc, ks, vc, vs, kl, cap, scale, out=out, err=err, workspace=ws)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_attn_close(host_f64(out), ref)
