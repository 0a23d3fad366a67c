"""Helpers shared by the GPU parity tests: host<->device moves of bf16 bit patterns and
the acceptance metrics of the hot path."""
import numpy as np
import torch

from oracle import mx

DEV = "cuda"


def dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(DEV)


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.to(DEV) if dtype is None else t.to(DEV, dtype)


def host_bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_f64(t):
    return mx.bf16_to_f64(host_bits(t))


def rel_frobenius(got, ref):
    return float(np.linalg.norm(got - ref) / np.linalg.norm(ref))


def assert_float_close(got, ref, rel_frob=1e-2, max_rel_rms=3e-2):
    """MLP / GEMM acceptance: relative Frobenius error <= 1e-2 and max |err| <= 3e-2 * rms(ref)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.isfinite(got).all()
    rf = rel_frobenius(got, ref)
    rms = float(np.sqrt(np.mean(ref * ref)))
    mx_err = float(np.abs(got - ref).max())
    assert rf <= rel_frob, f"relative Frobenius error {rf:.3e} > {rel_frob}"
    assert mx_err <= max_rel_rms * rms, f"max error {mx_err:.3e} > {max_rel_rms} * rms {rms:.3e}"
    return rf, mx_err / rms


def e4m3_ordinal(q):
    q = np.asarray(q).astype(np.int64)
    mag = q & 0x7F
    return np.where(q & 0x80, -mag, mag)


def assert_requant_close(hq_g, hs_g, hq_o, hs_o, frac=1e-3):
    """Down-projection input acceptance: per block the scale bytes agree except on <= frac of
    blocks (an amax at a power-of-two boundary may flip the shared exponent), and within
    same-scale blocks elements differ by <= 1 E4M3 step on <= frac of the elements."""
    hs_g, hs_o = np.asarray(hs_g), np.asarray(hs_o)
    flip = hs_g != hs_o
    assert flip.mean() <= frac, f"scale flips on {flip.mean():.2%} of blocks"
    M, n = np.asarray(hq_g).shape
    same = ~np.repeat(flip, 32, axis=1)
    d = np.abs(e4m3_ordinal(hq_g) - e4m3_ordinal(hq_o))[same]
    assert d.max(initial=0) <= 1, f"element off by {d.max()} E4M3 steps"
    assert (d > 0).mean() <= frac, f"{(d > 0).mean():.3%} of elements off by one step"
    # blocks with a flipped exponent: dequantised values still within one step of the larger scale
    if flip.any():
        vg = mx.mx_dequantize(hq_g, hs_g).reshape(M, -1, 32)[flip]
        vo = mx.mx_dequantize(hq_o, hs_o).reshape(M, -1, 32)[flip]
        step = np.exp2(np.maximum(hs_g, hs_o)[flip].astype(np.float64) - 127.0)[:, None] * 2.0 ** (8 - 3)
        assert np.all(np.abs(vg - vo) <= step)
    return float(flip.mean()), float((d > 0).mean())


def bf16_ulp(x):
    """Spacing of bf16 numbers at |x| (2^(floor(log2|x|) - 7)); 2^-133 at zero."""
    a = np.maximum(np.abs(np.asarray(x, np.float64)), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(a)) - 7)


def assert_attn_close(got, ref, floor_ulp=False):
    """Attention acceptance: max |err| <= 2e-3 against the fp64 oracle. With floor_ulp, the
    bound per element is max(2e-3, one bf16 step at |ref|): outputs of magnitude above 0.5
    (short prefixes, where o is close to a single V row) cannot be stored in bf16 closer
    than half a step, so 2e-3 alone is below the output format's resolution there."""
    err = np.abs(np.asarray(got, np.float64) - ref)
    tol = np.maximum(2e-3, bf16_ulp(ref)) if floor_ulp else 2e-3
    bad = err > tol
    assert not bad.any(), f"max err {err.max():.3e}; {bad.sum()} elements above the bound"
    return float(err.max())
