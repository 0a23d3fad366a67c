"""Block-scaled FP8 ("bsgemm" recipe) in fp64 -- oracle, test infrastructure only.

Source: [S2.1] "FP8 Quantization Strategy" names bsgemm as 128x128 block-scaled FP8, and
"What's Open Source" gives its granularity: 1x128 blocks for activations, 128x128 blocks for
weights. The pages print no rule for the scale, so the plainest reading is taken: each block
keeps one fp32 scale s = fp32(amax / 448), computed in fp32, and its elements are
E4M3(fp32(v / s)) -- the fp32 quotient rounded once to E4M3, nearest-even, saturating at
+-448; a block whose amax is 0 gets s = 0 and elements E4M3(v) (signed zeros).
The product is C[m][n] = sum over 128-wide K blocks kb of
s_x[m][kb] * s_w[n // 128][kb] * sum_{k in kb} E4M3(xq[m][k]) * E4M3(wq[n][k]).
"""
from __future__ import annotations

import numpy as np

from .mx import E4M3_MAX, e4m3_encode, e4m3_value

BK = 128   # K width of an activation block and of a weight block
BN = 128   # N height of a weight block


def _quantize_blocks(blocks):
    """blocks [..., elements] (fp64 values of bf16) -> (codes uint8 [..., elements],
    scales float32 [...]) with one scale per block."""
    amax = np.max(np.abs(blocks), axis=-1)
    s = (amax.astype(np.float32) / np.float32(E4M3_MAX)).astype(np.float32)
    zero = s == 0
    div = np.where(zero, np.float32(1), s).astype(np.float32)
    q32 = (blocks.astype(np.float32) / div[..., None]).astype(np.float32)
    return e4m3_encode(q32.astype(np.float64)), s


def bs_quantize_act(x):
    """Activations [M, K] -> (codes uint8 [M, K], scales float32 [M, K/128]): 1x128 blocks."""
    x = np.asarray(x, dtype=np.float64)
    M, K = x.shape
    if K % BK:
        raise ValueError("K must be a multiple of 128")
    q, s = _quantize_blocks(x.reshape(M, K // BK, BK))
    return q.reshape(M, K), s


def bs_quantize_weight(w):
    """Weights [N, K] -> (codes uint8 [N, K], scales float32 [ceil(N/128), K/128]): 128x128
    blocks (the last row block may be shorter)."""
    w = np.asarray(w, dtype=np.float64)
    N, K = w.shape
    if K % BK:
        raise ValueError("K must be a multiple of 128")
    nb = (N + BN - 1) // BN
    q = np.zeros((N, K), dtype=np.uint8)
    s = np.zeros((nb, K // BK), dtype=np.float32)
    for i in range(nb):
        rows = w[i * BN:(i + 1) * BN]
        blk = rows.reshape(rows.shape[0], K // BK, BK).transpose(1, 0, 2).reshape(K // BK, -1)
        qb, sb = _quantize_blocks(blk)
        q[i * BN:(i + 1) * BN] = qb.reshape(K // BK, rows.shape[0], BK).transpose(1, 0, 2).reshape(rows.shape[0], K)
        s[i] = sb
    return q, s


def bs_dequantize_act(q, s):
    M, K = q.shape
    return (e4m3_value(q).reshape(M, K // BK, BK) * np.asarray(s, np.float64)[..., None]).reshape(M, K)


def bs_dequantize_weight(q, s):
    N, K = q.shape
    rows = np.arange(N) // BN
    return e4m3_value(q) * np.repeat(np.asarray(s, np.float64)[rows], BK, axis=1)


def bs_gemm(xq, xs, wq, ws) -> np.ndarray:
    """C = X' W'^T in fp64 over the dequantised block-scaled operands."""
    return bs_dequantize_act(xq, xs) @ bs_dequantize_weight(wq, ws).T
