"""Pins of the prefill / extend attention oracle: torch SDPA with a causal mask, the decode
attention for one new token, and prefill == prefix prefill followed by an extend."""
import numpy as np
import torch
import torch.nn.functional as F

from oracle import ops


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def test_prefill_from_scratch_matches_torch_sdpa_causal():
    rng = np.random.default_rng(0)
    T, Hq, Hkv, D = 37, 8, 2, 16
    q = _rand(rng, T, Hq, D)
    k = _rand(rng, Hkv, T, D)
    v = _rand(rng, Hkv, T, D)
    (o,) = ops.gqa_prefill_attention([q], [k], [v], 0.3)
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]                       # [1, Hq, T, D]
    kt = torch.from_numpy(k).repeat_interleave(Hq // Hkv, dim=0)[None]    # [1, Hq, T, D]
    vt = torch.from_numpy(v).repeat_interleave(Hq // Hkv, dim=0)[None]
    ref = F.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=0.3)[0].permute(1, 0, 2).numpy()
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)


def test_one_new_token_is_decode_attention():
    rng = np.random.default_rng(1)
    Hq, Hkv, D, lens = 4, 2, 8, [1, 5, 40]
    kp = [_rand(rng, Hkv, n, D) for n in lens]
    vp = [_rand(rng, Hkv, n, D) for n in lens]
    q = _rand(rng, 3, Hq, D)
    got = ops.gqa_prefill_attention([q[b:b + 1] for b in range(3)], kp, vp, 0.5)
    ref = ops.gqa_decode_attention(q, kp, vp, 0.5)
    for b in range(3):
        np.testing.assert_allclose(got[b][0], ref[b], rtol=0, atol=1e-13)


def test_extend_equals_the_tail_of_a_full_prefill():
    # a prefill of n tokens, split into a prefix of P and an extend of n - P: the extend's rows are
    # the last n - P rows of the one-shot prefill (same keys, same causal horizon)
    rng = np.random.default_rng(2)
    n, P, Hq, Hkv, D = 50, 31, 6, 3, 8
    q = _rand(rng, n, Hq, D)
    k = _rand(rng, Hkv, n, D)
    v = _rand(rng, Hkv, n, D)
    (full,) = ops.gqa_prefill_attention([q], [k], [v], 0.25)
    (ext,) = ops.gqa_prefill_attention([q[P:]], [k], [v], 0.25)
    np.testing.assert_allclose(ext, full[P:], rtol=0, atol=1e-13)
    # the first query of a prefill from scratch sees only itself: o = V_0
    np.testing.assert_allclose(full[0], np.repeat(v[:, 0], Hq // Hkv, axis=0), rtol=0, atol=1e-14)


def test_kv_append_extend_writes_the_last_rows():
    kc = np.zeros((2, 2, 8, 4))
    kn = [np.arange(24.0).reshape(3, 2, 4), -np.ones((1, 2, 4))]
    k2, v2 = ops.kv_append_extend(kc, kc, kn, kn, np.array([5, 8]))
    assert np.array_equal(k2[0, :, 2:5], np.transpose(kn[0], (1, 0, 2)))
    assert np.array_equal(k2[1, :, 7], kn[1][0]) and np.count_nonzero(k2) == 23 + 8
