"""GPU parity of paged decode attention and the paged KV append: against the fp64 oracle
(max |err| <= 2e-3), bit for bit against the contiguous kernel on the same prefixes, with
random page placement and +-1e4 in every pool entry no sequence owns."""
import math

import numpy as np
import pytest
import torch

from mxfp8_mlp_gqa_gb300 import api, synth
from oracle import mx, ops
from tests.gpu_util import assert_attn_close, dev, dev_bf16, host_f64

pytestmark = pytest.mark.gpu


def _garbage(shape):
    t = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    v = t.view(torch.int16).view(-1, 2)
    v[:, 0] = int(np.int16(np.uint16(0x461C).view(np.int16)))
    v[:, 1] = int(np.uint16(0xC61C).view(np.int16))
    return t


def _paged(prefix, page_size, extra_pages, seed, max_kv_len=0):
    """Device pool [num_pages, Hkv, page_size, D] holding each prefix at randomly placed pages,
    and the table [bs, max_pages] (unused entries -1) covering at least max_kv_len positions."""
    Hkv, D = prefix[0].shape[0], prefix[0].shape[2]
    need = [(p.shape[1] + page_size - 1) // page_size for p in prefix]
    num_pages = sum(need) + extra_pages
    perm = np.random.default_rng(seed).permutation(num_pages)
    pool = _garbage((num_pages, Hkv, page_size, D))
    width = max(max(need) + 1, (max_kv_len + page_size - 1) // page_size)
    table = np.full((len(prefix), width), -1, np.int32)
    k = 0
    for b, p in enumerate(prefix):
        pd = dev_bf16(p)
        for j in range(need[b]):
            seg = pd[:, j * page_size:(j + 1) * page_size, :]
            pool[int(perm[k]), :, :seg.shape[1], :].copy_(seg)
            table[b, j] = perm[k]
            k += 1
    return pool, table


def _contig(prefix, cap):
    Hkv, D = prefix[0].shape[0], prefix[0].shape[2]
    c = _garbage((len(prefix), Hkv, cap, D))
    for b, p in enumerate(prefix):
        c[b, :, :p.shape[1]].copy_(dev_bf16(p))
    return c


def _case(bs, Hq, Hkv, D, lens, seed):
    q = synth.normal_bf16((bs, Hq, D), 1.0, seed, synth.TID["q"])
    kp = synth.kv_prefix(bs, Hkv, D, lens, seed, synth.TID["k"])
    vp = synth.kv_prefix(bs, Hkv, D, lens, seed, synth.TID["v"])
    return q, kp, vp


@pytest.mark.parametrize("bs,page_size", [(1, 64), (8, 256), (64, 64), (64, 128)])
def test_paged_attention_vs_oracle_and_contiguous(bs, page_size):
    Hq, Hkv, D, mkv = 32, 8, 128, 4096
    lens = synth.kv_lens(bs, 234, mkv, seed=bs)
    q, kp, vp = _case(bs, Hq, Hkv, D, lens, bs)
    kpool, table = _paged(kp, page_size, 5, seed=1, max_kv_len=mkv)
    vpool, table_v = _paged(vp, page_size, 5, seed=1, max_kv_len=mkv)
    assert np.array_equal(table, table_v)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    scale = 1 / math.sqrt(D)
    out = api.gqa_decode_attn_paged(dev_bf16(q), kpool, vpool, dev(table), dev(lens), mkv, scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = ops.gqa_decode_attention(mx.bf16_to_f64(q), [mx.bf16_to_f64(k) for k in kp],
                                   [mx.bf16_to_f64(v) for v in vp], scale)
    assert_attn_close(host_f64(out), ref)
    # the same prefixes in a contiguous cache give the same bits (same tiles, same order)
    oc = api.gqa_decode_attn(dev_bf16(q), _contig(kp, mkv), _contig(vp, mkv), dev(lens), mkv, scale)
    assert torch.equal(out.view(torch.int16), oc.view(torch.int16))


def test_paged_length_edges_small_group():
    # tile / page boundaries and a group of 2 at D = 64
    Hq, Hkv, D, ps = 4, 2, 64, 64
    lens = np.array([1, 63, 64, 65, 128, 129, 500, 1024], np.int32)
    q, kp, vp = _case(len(lens), Hq, Hkv, D, lens, 9)
    kpool, table = _paged(kp, ps, 3, seed=4, max_kv_len=1024)
    vpool, _ = _paged(vp, ps, 3, seed=4, max_kv_len=1024)
    out = api.gqa_decode_attn_paged(dev_bf16(q), kpool, vpool, dev(table), dev(lens), 1024, 0.125)
    ref = ops.gqa_decode_attention(mx.bf16_to_f64(q), [mx.bf16_to_f64(k) for k in kp],
                                   [mx.bf16_to_f64(v) for v in vp], 0.125)
    assert_attn_close(host_f64(out), ref, floor_ulp=True)


def test_paged_bad_page_id_sets_the_flag():
    Hq, Hkv, D, ps = 8, 2, 64, 64
    lens = np.array([100, 70], np.int32)
    q, kp, vp = _case(2, Hq, Hkv, D, lens, 2)
    kpool, table = _paged(kp, ps, 1, seed=3)
    vpool, _ = _paged(vp, ps, 1, seed=3)
    table[1, 1] = kpool.shape[0] + 7  # outside the pool
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = api.gqa_decode_attn_paged(dev_bf16(q), kpool, vpool, dev(table), dev(lens), 128, 0.125, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 7
    ref = ops.gqa_decode_attention(mx.bf16_to_f64(q[:1]), [mx.bf16_to_f64(kp[0])], [mx.bf16_to_f64(vp[0])], 0.125)
    assert_attn_close(host_f64(out)[:1], ref)  # the other sequence is unaffected


def test_kv_append_paged_bit_exact():
    Hkv, D, ps = 8, 128, 64
    lens_before = np.array([63, 64, 200, 1], np.int32)
    kp = synth.kv_prefix(4, Hkv, D, lens_before, 6, synth.TID["k"])
    vp = synth.kv_prefix(4, Hkv, D, lens_before, 6, synth.TID["v"])
    kpool, table = _paged(kp, ps, 4, seed=8)
    vpool, _ = _paged(vp, ps, 4, seed=8)
    # pages for the positions the append reaches (the 64-long sequence starts a new page)
    used = set(table[table >= 0].tolist())
    free = [p for p in range(kpool.shape[0]) if p not in used]
    for b, n in enumerate(lens_before):
        if table[b, n // ps] < 0:
            table[b, n // ps] = free.pop()
    kn = synth.normal_bf16((4, Hkv, D), 1.0, 6, synth.TID["q"])
    vn = synth.normal_bf16((4, Hkv, D), 2.0, 7, synth.TID["q"])
    lens = lens_before + 1
    k0, v0 = kpool.view(torch.int16).cpu().numpy(), vpool.view(torch.int16).cpu().numpy()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.kv_append_paged(kpool, vpool, dev(table), dev_bf16(kn), dev_bf16(vn), dev(lens), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rk, rv = ops.kv_append_paged(k0, v0, table, kn.view(np.int16), vn.view(np.int16), lens, ps)
    np.testing.assert_array_equal(kpool.view(torch.int16).cpu().numpy(), rk)
    np.testing.assert_array_equal(vpool.view(torch.int16).cpu().numpy(), rv)
