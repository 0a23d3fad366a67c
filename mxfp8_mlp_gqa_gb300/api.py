"""Python binding of libmxg (ctypes): the same entry points as ``include/mxg.h``.

Argument marshalling only: every step runs in the library's CUDA kernels. PyTorch
provides device memory and the current CUDA stream. Inputs are checked strictly
(dtype, rank, shape, contiguity, device); nothing is reshaped, unsqueezed or
promoted on the caller's behalf (the prev-window contract of [S2.1] "DualAR:
S2-Specific Batching Constraints"). Outputs may be passed in (stable addresses
for CUDA-graph capture) or are allocated with ``torch.empty``.

If the shared library is missing or cannot be loaded, every call raises: there
is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

from . import build as _build

_LIB = None

c_i64, c_f32, c_vp, c_sz = ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t

_SIGS = {
    "mxg_status_str": (ctypes.c_char_p, [ctypes.c_int]),
    "mxg_version": (ctypes.c_int, []),
    "mxg_set_tensor_core_path": (ctypes.c_int, [ctypes.c_int]),
    "mxg_debug_stall_attn_loads": (ctypes.c_int, [ctypes.c_int]),
    "mxfp8_quantize": (ctypes.c_int, [c_vp, c_i64, c_i64, c_i64, c_vp, c_vp, c_vp]),
    "rmsnorm_mxfp8_quantize": (ctypes.c_int, [c_vp, c_vp, c_f32, c_i64, c_i64, c_i64, c_vp, c_vp, c_vp]),
    "mxfp8_gemm_workspace": (c_sz, [c_i64, c_i64, c_i64]),
    "mxfp8_gemm": (ctypes.c_int, [c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, c_vp, c_vp, c_vp, c_sz, c_vp]),
    "mlp_gate_up_swiglu_mxfp8": (ctypes.c_int, [c_vp, c_vp, c_i64, c_i64, c_i64, c_vp, c_vp, c_vp, c_vp, c_vp]),
    "mlp_swiglu_mxfp8_workspace": (c_sz, [c_i64, c_i64, c_i64]),
    "mlp_swiglu_mxfp8": (ctypes.c_int, [c_vp, c_vp, c_i64, c_i64, c_i64, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp,
                                        c_vp, c_sz, c_vp]),
    "gqa_decode_attn_workspace": (c_sz, [c_i64, c_i64, c_i64, c_i64, c_i64]),
    "gqa_decode_attn": (ctypes.c_int, [c_vp, c_i64, c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, c_i64, c_i64, c_i64,
                                       c_f32, c_vp, c_vp, c_vp, c_sz, c_vp]),
    "gqa_decode_attn_mxfp8": (ctypes.c_int, [c_vp, c_i64, c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, c_i64, c_i64,
                                             c_i64, c_f32, c_vp, c_vp, c_vp, c_vp, c_vp, c_sz, c_vp]),
    "mxfp8_gemm_qkv_kv_append": (ctypes.c_int, [c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, c_i64, c_i64, c_vp,
                                                c_vp, c_vp, c_vp, c_i64, c_vp, c_vp]),
    "gqa_decode_attn_noalloc_capacity": (c_sz, []),
    "gqa_decode_attn_noalloc": (ctypes.c_int, [c_vp, c_i64, c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, c_i64, c_i64,
                                               c_i64, c_f32, c_vp, c_vp, c_vp]),
    "kv_append": (ctypes.c_int, [c_vp, c_vp, c_vp, c_vp, c_i64, c_vp, c_i64, c_i64, c_i64, c_i64, c_vp, c_vp]),
    "prev_tokens_shift": (ctypes.c_int, [c_vp, c_vp, c_i64, c_i64, c_i64, c_vp]),
    "copy_bytes": (ctypes.c_int, [c_vp, c_vp, c_i64, c_vp]),
    "gqa_decode_attn_paged": (ctypes.c_int, [c_vp, c_i64, c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, c_vp, c_i64, c_i64,
                                             c_i64, c_i64, c_i64, c_f32, c_vp, c_vp, c_vp, c_sz, c_vp]),
    "kv_append_paged": (ctypes.c_int, [c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, c_vp, c_vp, c_i64, c_vp, c_i64, c_i64,
                                       c_i64, c_vp, c_vp]),
    "gqa_decode_attn_kv_mxfp8": (ctypes.c_int, [c_vp, c_i64, c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, c_i64,
                                                c_i64, c_i64, c_f32, c_vp, c_vp, c_vp, c_sz, c_vp]),
    "gqa_decode_attn_kv_mxfp8_paged": (ctypes.c_int, [c_vp, c_i64, c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_i64,
                                                      c_vp, c_i64, c_i64, c_i64, c_i64, c_i64, c_f32, c_vp, c_vp, c_vp,
                                                      c_sz, c_vp]),
    "kv_append_mxfp8": (ctypes.c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_vp, c_i64, c_i64, c_i64, c_i64,
                                       c_vp, c_vp]),
    "kv_append_mxfp8_paged": (ctypes.c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, c_vp, c_vp, c_i64,
                                             c_vp, c_i64, c_i64, c_i64, c_vp, c_vp]),
    "gqa_prefill_attn": (ctypes.c_int, [c_vp, c_i64, c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, c_i64, c_i64, c_i64,
                                        c_i64, c_f32, c_vp, c_vp, c_vp]),
    "gqa_prefill_attn_paged": (ctypes.c_int, [c_vp, c_i64, c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, c_vp, c_vp, c_i64,
                                              c_i64, c_i64, c_i64, c_i64, c_i64, c_f32, c_vp, c_vp, c_vp]),
    "kv_append_extend": (ctypes.c_int, [c_vp, c_vp, c_vp, c_vp, c_i64, c_vp, c_vp, c_i64, c_i64, c_i64, c_i64, c_i64,
                                        c_i64, c_vp, c_vp]),
    "bs_quantize_act": (ctypes.c_int, [c_vp, c_i64, c_i64, c_i64, c_vp, c_vp, c_vp]),
    "bs_quantize_weight": (ctypes.c_int, [c_vp, c_i64, c_i64, c_vp, c_vp, c_vp]),
    "bs_gemm_workspace": (c_sz, [c_i64, c_i64, c_i64]),
    "bs_gemm": (ctypes.c_int, [c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, c_vp, c_vp, c_sz, c_vp, c_vp]),
    "kv_append_extend_paged": (ctypes.c_int, [c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, c_vp, c_vp, c_i64, c_vp, c_vp,
                                              c_i64, c_i64, c_i64, c_i64, c_i64, c_vp, c_vp]),
}


class MxgError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn}: {lib().mxg_status_str(status).decode()} (status {status})")


def header_functions() -> list:
    """Entry points declared in include/mxg.h."""
    src = open(os.path.join(_build.INCLUDE, "mxg.h")).read()
    return re.findall(r"^\s*(?:const char\*|int|size_t|mxg_status)\s+(\w+)\(", src, re.M)


def lib(path: str | None = None):
    """Load libmxg.so (once). Raises if it has not been built."""
    global _LIB
    if _LIB is None:
        p = path or _build.LIB
        if not os.path.exists(p):
            raise RuntimeError(f"libmxg.so not built at {p}: run __graft_entry__.build() first")
        L = ctypes.CDLL(p)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _LIB = L
    return _LIB


def set_tensor_core_path(enable: bool) -> bool:
    """Force (False) or allow (True, default) the tcgen05 GEMM kernels; returns the previous setting."""
    return bool(lib().mxg_set_tensor_core_path(1 if enable else 0))


def _call(name, *args):
    st = getattr(lib(), name)(*args)
    if st != 0:
        raise MxgError(name, st)


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(t, name, dtype, shape=None, ndim=None, contiguous=True):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype} (no implicit promotion)")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name}: rank {t.dim()}, expected {ndim} (no implicit reshaping)")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    return t


def _rows_view(t, name, dtype):
    """2-D tensor whose rows may be strided (last dim contiguous): returns the row stride."""
    _check(t, name, dtype, ndim=2, contiguous=False)
    if t.stride(1) != 1:
        raise ValueError(f"{name}: the last dimension must be contiguous")
    return t.stride(0)


def _out(t, name, dtype, shape, device):
    if t is None:
        return torch.empty(shape, dtype=dtype, device=device)
    return _check(t, name, dtype, shape)


# ------------------------------------------------------------------ quantisation
def mxfp8_quantize(x, q=None, s=None):
    """bf16 [M, K] -> (E4M3 bytes [M, K], UE8M0 scales [M, K/32])."""
    ld = _rows_view(x, "x", torch.bfloat16)
    M, K = x.shape
    q = _out(q, "q", torch.uint8, (M, K), x.device)
    s = _out(s, "s", torch.uint8, (M, K // 32), x.device)
    _call("mxfp8_quantize", _ptr(x), M, K, ld, _ptr(q), _ptr(s), _stream())
    return q, s


def rmsnorm_mxfp8_quantize(x, gamma, eps, q=None, s=None):
    ld = _rows_view(x, "x", torch.bfloat16)
    M, K = x.shape
    _check(gamma, "gamma", torch.bfloat16, (K,))
    q = _out(q, "q", torch.uint8, (M, K), x.device)
    s = _out(s, "s", torch.uint8, (M, K // 32), x.device)
    _call("rmsnorm_mxfp8_quantize", _ptr(x), _ptr(gamma), float(eps), M, K, ld, _ptr(q), _ptr(s), _stream())
    return q, s


# ------------------------------------------------------------------ GEMM / MLP
def mxfp8_gemm(aq, as_, bq, bs, residual=None, c=None, workspace=None):
    """C[M, N] = A' B'^T (+ residual) in bf16; A = (aq [M,K], as_ [M,K/32]), B = (bq [N,K], bs [N,K/32])."""
    _check(aq, "aq", torch.uint8, ndim=2)
    M, K = aq.shape
    _check(as_, "as", torch.uint8, (M, K // 32))
    _check(bq, "bq", torch.uint8, ndim=2)
    N = bq.shape[0]
    _check(bq, "bq", torch.uint8, (N, K))
    _check(bs, "bs", torch.uint8, (N, K // 32))
    if residual is not None:
        _check(residual, "residual", torch.bfloat16, (M, N))
    c = _out(c, "c", torch.bfloat16, (M, N), aq.device)
    need = lib().mxfp8_gemm_workspace(M, N, K)
    if workspace is None and need:
        workspace = torch.zeros(need, dtype=torch.uint8, device=aq.device)  # split-K counters start at 0
    ws_bytes = 0 if workspace is None else workspace.numel()
    _call("mxfp8_gemm", _ptr(aq), _ptr(as_), _ptr(bq), _ptr(bs), M, N, K, _ptr(residual), _ptr(c),
          _ptr(workspace), ws_bytes, _stream())
    return c


def mxfp8_gemm_qkv_kv_append(xq, xs, wq, ws, Hq, Hkv, k_cache, v_cache, kv_len, qkv=None, err=None):
    """QKV projection with the KV append fused: q columns -> qkv bf16 [M, (Hq+2Hkv)D]; K/V
    columns -> row kv_len[m]-1 of the caches [M, Hkv, cap, D]."""
    _check(xq, "xq", torch.uint8, ndim=2)
    M, K = xq.shape
    _check(xs, "xs", torch.uint8, (M, K // 32))
    _check(k_cache, "k_cache", torch.bfloat16, ndim=4)
    bs, Hkv_, cap, D = k_cache.shape
    if bs != M or Hkv_ != Hkv:
        raise ValueError("k_cache: expected [M, Hkv, cap, D]")
    _check(v_cache, "v_cache", torch.bfloat16, (M, Hkv, cap, D))
    N = (Hq + 2 * Hkv) * D
    _check(wq, "wq", torch.uint8, (N, K))
    _check(ws, "ws", torch.uint8, (N, K // 32))
    _check(kv_len, "kv_len", torch.int32, (M,))
    qkv = _out(qkv, "qkv", torch.bfloat16, (M, N), xq.device)
    if err is not None:
        _check(err, "err", torch.int32, (1,))
    _call("mxfp8_gemm_qkv_kv_append", _ptr(xq), _ptr(xs), _ptr(wq), _ptr(ws), M, K, Hq, Hkv, D, _ptr(qkv),
          _ptr(k_cache), _ptr(v_cache), _ptr(kv_len), cap, _ptr(err), _stream())
    return qkv


def mxfp8_gemm_workspace(M, N, K) -> int:
    return int(lib().mxfp8_gemm_workspace(M, N, K))


def mlp_gate_up_swiglu_mxfp8(xq, xs, w13q, w13s, hq=None, hs=None):
    _check(xq, "xq", torch.uint8, ndim=2)
    M, d_model = xq.shape
    _check(xs, "xs", torch.uint8, (M, d_model // 32))
    _check(w13q, "w13q", torch.uint8, ndim=2)
    d_ff = w13q.shape[0] // 2
    _check(w13q, "w13q", torch.uint8, (2 * d_ff, d_model))
    _check(w13s, "w13s", torch.uint8, (2 * d_ff, d_model // 32))
    hq = _out(hq, "hq", torch.uint8, (M, d_ff), xq.device)
    hs = _out(hs, "hs", torch.uint8, (M, d_ff // 32), xq.device)
    _call("mlp_gate_up_swiglu_mxfp8", _ptr(xq), _ptr(xs), M, d_model, d_ff, _ptr(w13q), _ptr(w13s), _ptr(hq),
          _ptr(hs), _stream())
    return hq, hs


def mlp_swiglu_mxfp8_workspace(M, d_model, d_ff) -> int:
    return int(lib().mlp_swiglu_mxfp8_workspace(M, d_model, d_ff))


def mlp_swiglu_mxfp8(xq, xs, w13q, w13s, w2q, w2s, residual=None, y=None, workspace=None):
    _check(xq, "xq", torch.uint8, ndim=2)
    M, d_model = xq.shape
    _check(xs, "xs", torch.uint8, (M, d_model // 32))
    d_ff = w13q.shape[0] // 2
    _check(w13q, "w13q", torch.uint8, (2 * d_ff, d_model))
    _check(w13s, "w13s", torch.uint8, (2 * d_ff, d_model // 32))
    _check(w2q, "w2q", torch.uint8, (d_model, d_ff))
    _check(w2s, "w2s", torch.uint8, (d_model, d_ff // 32))
    if residual is not None:
        _check(residual, "residual", torch.bfloat16, (M, d_model))
    y = _out(y, "y", torch.bfloat16, (M, d_model), xq.device)
    need = mlp_swiglu_mxfp8_workspace(M, d_model, d_ff)
    if workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=xq.device)  # split-K counters start at 0
    _check(workspace, "workspace", torch.uint8, ndim=1)
    _call("mlp_swiglu_mxfp8", _ptr(xq), _ptr(xs), M, d_model, d_ff, _ptr(w13q), _ptr(w13s), _ptr(w2q), _ptr(w2s),
          _ptr(residual), _ptr(y), _ptr(workspace), workspace.numel(), _stream())
    return y


# ------------------------------------------------------------------ attention / cache / window
def gqa_decode_attn_workspace(bs, Hq, Hkv, D, max_kv_len) -> int:
    return int(lib().gqa_decode_attn_workspace(bs, Hq, Hkv, D, max_kv_len))


def gqa_decode_attn(q, k_cache, v_cache, kv_len, max_kv_len, scale, out=None, err=None, workspace=None, oq=None,
                    os=None):
    """q bf16 [bs, Hq, D] (or a row-strided [bs, Hq*D] view), caches bf16 [bs, Hkv, cap, D],
    kv_len int32 [bs] on the device -> out bf16 [bs, Hq, D]. With oq/os given (uint8
    [bs, Hq*D] and [bs, Hq*D/32]) the output is also written MX-quantised (gqa_decode_attn_mxfp8)."""
    _check(k_cache, "k_cache", torch.bfloat16, ndim=4)
    bs, Hkv, cap, D = k_cache.shape
    _check(v_cache, "v_cache", torch.bfloat16, (bs, Hkv, cap, D))
    _check(kv_len, "kv_len", torch.int32, (bs,))
    if q.dim() == 3:
        _check(q, "q", torch.bfloat16, ndim=3)
        Hq = q.shape[1]
        _check(q, "q", torch.bfloat16, (bs, Hq, D))
        ld_q = Hq * D
    else:
        ld_q = _rows_view(q, "q", torch.bfloat16)
        if q.shape[0] != bs or q.shape[1] % D:
            raise ValueError("q: expected [bs, Hq*D]")
        Hq = q.shape[1] // D
    out = _out(out, "out", torch.bfloat16, (bs, Hq, D), k_cache.device)
    if err is not None:
        _check(err, "err", torch.int32, (1,))
    need = gqa_decode_attn_workspace(bs, Hq, Hkv, D, max_kv_len)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=k_cache.device)
    ws_bytes = 0 if workspace is None else workspace.numel()
    if oq is None and os is None:
        _call("gqa_decode_attn", _ptr(q), ld_q, _ptr(k_cache), _ptr(v_cache), _ptr(kv_len), bs, Hq, Hkv, D, cap,
              int(max_kv_len), float(scale), _ptr(out), _ptr(err), _ptr(workspace), ws_bytes, _stream())
        return out
    _check(oq, "oq", torch.uint8, (bs, Hq * D))
    _check(os, "os", torch.uint8, (bs, Hq * D // 32))
    _call("gqa_decode_attn_mxfp8", _ptr(q), ld_q, _ptr(k_cache), _ptr(v_cache), _ptr(kv_len), bs, Hq, Hkv, D, cap,
          int(max_kv_len), float(scale), _ptr(out), _ptr(oq), _ptr(os), _ptr(err), _ptr(workspace), ws_bytes,
          _stream())
    return out, oq, os


def gqa_decode_attn_paged(q, k_pool, v_pool, block_table, kv_len, max_kv_len, scale, out=None, err=None,
                          workspace=None):
    """Paged decode attention: q bf16 [bs, Hq, D]; pools bf16 [num_pages, Hkv, page_size, D];
    block_table int32 [bs, max_pages] (page ids) and kv_len int32 [bs] on the device."""
    _check(k_pool, "k_pool", torch.bfloat16, ndim=4)
    num_pages, Hkv, page_size, D = k_pool.shape
    _check(v_pool, "v_pool", torch.bfloat16, (num_pages, Hkv, page_size, D))
    _check(block_table, "block_table", torch.int32, ndim=2)
    bs, max_pages = block_table.shape
    _check(kv_len, "kv_len", torch.int32, (bs,))
    _check(q, "q", torch.bfloat16, ndim=3)
    Hq = q.shape[1]
    _check(q, "q", torch.bfloat16, (bs, Hq, D))
    out = _out(out, "out", torch.bfloat16, (bs, Hq, D), k_pool.device)
    if err is not None:
        _check(err, "err", torch.int32, (1,))
    need = gqa_decode_attn_workspace(bs, Hq, Hkv, D, max_kv_len)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=k_pool.device)
    ws_bytes = 0 if workspace is None else workspace.numel()
    _call("gqa_decode_attn_paged", _ptr(q), Hq * D, _ptr(k_pool), _ptr(v_pool), _ptr(block_table), max_pages,
          page_size, num_pages, _ptr(kv_len), bs, Hq, Hkv, D, int(max_kv_len), float(scale), _ptr(out), _ptr(err),
          _ptr(workspace), ws_bytes, _stream())
    return out


def kv_append_paged(k_pool, v_pool, block_table, k_new, v_new, kv_len, err=None):
    """kv_append into paged pools [num_pages, Hkv, page_size, D]; k_new/v_new bf16 [bs, Hkv, D]."""
    _check(k_pool, "k_pool", torch.bfloat16, ndim=4)
    num_pages, Hkv, page_size, D = k_pool.shape
    _check(v_pool, "v_pool", torch.bfloat16, (num_pages, Hkv, page_size, D))
    _check(block_table, "block_table", torch.int32, ndim=2)
    bs, max_pages = block_table.shape
    _check(kv_len, "kv_len", torch.int32, (bs,))
    _check(k_new, "k_new", torch.bfloat16, (bs, Hkv, D))
    _check(v_new, "v_new", torch.bfloat16, (bs, Hkv, D))
    if err is not None:
        _check(err, "err", torch.int32, (1,))
    _call("kv_append_paged", _ptr(k_pool), _ptr(v_pool), _ptr(block_table), max_pages, page_size, num_pages,
          _ptr(k_new), _ptr(v_new), Hkv * D, _ptr(kv_len), bs, Hkv, D, _ptr(err), _stream())


def _mx_cache(codes, scales, cname, sname):
    """MXFP8 cache arrays: codes uint8 [A, Hkv, T, D], scales uint8 [A, Hkv, T, D/32]."""
    _check(codes, cname, torch.uint8, ndim=4)
    A, Hkv, T, D = codes.shape
    if D % 32:
        raise ValueError(f"{cname}: D must be a multiple of 32")
    _check(scales, sname, torch.uint8, (A, Hkv, T, D // 32))
    return A, Hkv, T, D


def gqa_decode_attn_kv_mxfp8(q, k_codes, k_scales, v_codes, v_scales, kv_len, max_kv_len, scale, out=None, err=None,
                             workspace=None):
    """Decode attention over an MXFP8 cache: q bf16 [bs, Hq, D]; codes uint8 [bs, Hkv, cap, D],
    scales uint8 [bs, Hkv, cap, D/32]; kv_len int32 [bs] -> out bf16 [bs, Hq, D]."""
    bs, Hkv, cap, D = _mx_cache(k_codes, k_scales, "k_codes", "k_scales")
    _mx_cache(v_codes, v_scales, "v_codes", "v_scales")
    _check(v_codes, "v_codes", torch.uint8, (bs, Hkv, cap, D))
    _check(kv_len, "kv_len", torch.int32, (bs,))
    _check(q, "q", torch.bfloat16, ndim=3)
    Hq = q.shape[1]
    _check(q, "q", torch.bfloat16, (bs, Hq, D))
    out = _out(out, "out", torch.bfloat16, (bs, Hq, D), k_codes.device)
    if err is not None:
        _check(err, "err", torch.int32, (1,))
    need = gqa_decode_attn_workspace(bs, Hq, Hkv, D, max_kv_len)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=k_codes.device)
    ws_bytes = 0 if workspace is None else workspace.numel()
    _call("gqa_decode_attn_kv_mxfp8", _ptr(q), Hq * D, _ptr(k_codes), _ptr(k_scales), _ptr(v_codes), _ptr(v_scales),
          _ptr(kv_len), bs, Hq, Hkv, D, cap, int(max_kv_len), float(scale), _ptr(out), _ptr(err), _ptr(workspace),
          ws_bytes, _stream())
    return out


def gqa_decode_attn_kv_mxfp8_paged(q, k_codes, k_scales, v_codes, v_scales, block_table, kv_len, max_kv_len, scale,
                                   out=None, err=None, workspace=None):
    """Paged decode attention over MXFP8 pools: codes uint8 [num_pages, Hkv, page_size, D],
    scales uint8 [num_pages, Hkv, page_size, D/32]; block_table int32 [bs, max_pages]."""
    num_pages, Hkv, page_size, D = _mx_cache(k_codes, k_scales, "k_codes", "k_scales")
    _mx_cache(v_codes, v_scales, "v_codes", "v_scales")
    _check(v_codes, "v_codes", torch.uint8, (num_pages, Hkv, page_size, D))
    _check(block_table, "block_table", torch.int32, ndim=2)
    bs, max_pages = block_table.shape
    _check(kv_len, "kv_len", torch.int32, (bs,))
    _check(q, "q", torch.bfloat16, ndim=3)
    Hq = q.shape[1]
    _check(q, "q", torch.bfloat16, (bs, Hq, D))
    out = _out(out, "out", torch.bfloat16, (bs, Hq, D), k_codes.device)
    if err is not None:
        _check(err, "err", torch.int32, (1,))
    need = gqa_decode_attn_workspace(bs, Hq, Hkv, D, max_kv_len)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=k_codes.device)
    ws_bytes = 0 if workspace is None else workspace.numel()
    _call("gqa_decode_attn_kv_mxfp8_paged", _ptr(q), Hq * D, _ptr(k_codes), _ptr(k_scales), _ptr(v_codes),
          _ptr(v_scales), _ptr(block_table), max_pages, page_size, num_pages, _ptr(kv_len), bs, Hq, Hkv, D,
          int(max_kv_len), float(scale), _ptr(out), _ptr(err), _ptr(workspace), ws_bytes, _stream())
    return out


def kv_append_mxfp8(k_codes, k_scales, v_codes, v_scales, k_new, v_new, kv_len, err=None):
    """kv_append into an MXFP8 cache (codes [bs, Hkv, cap, D], scales [bs, Hkv, cap, D/32]);
    k_new/v_new bf16 [bs, Hkv, D] are MX-quantised on the way in."""
    bs, Hkv, cap, D = _mx_cache(k_codes, k_scales, "k_codes", "k_scales")
    _mx_cache(v_codes, v_scales, "v_codes", "v_scales")
    _check(v_codes, "v_codes", torch.uint8, (bs, Hkv, cap, D))
    _check(kv_len, "kv_len", torch.int32, (bs,))
    _check(k_new, "k_new", torch.bfloat16, (bs, Hkv, D))
    _check(v_new, "v_new", torch.bfloat16, (bs, Hkv, D))
    if err is not None:
        _check(err, "err", torch.int32, (1,))
    _call("kv_append_mxfp8", _ptr(k_codes), _ptr(k_scales), _ptr(v_codes), _ptr(v_scales), _ptr(k_new), _ptr(v_new),
          Hkv * D, _ptr(kv_len), bs, Hkv, D, cap, _ptr(err), _stream())


def kv_append_mxfp8_paged(k_codes, k_scales, v_codes, v_scales, block_table, k_new, v_new, kv_len, err=None):
    """kv_append_mxfp8 into paged MXFP8 pools [num_pages, Hkv, page_size, D (/32)]."""
    num_pages, Hkv, page_size, D = _mx_cache(k_codes, k_scales, "k_codes", "k_scales")
    _mx_cache(v_codes, v_scales, "v_codes", "v_scales")
    _check(v_codes, "v_codes", torch.uint8, (num_pages, Hkv, page_size, D))
    _check(block_table, "block_table", torch.int32, ndim=2)
    bs, max_pages = block_table.shape
    _check(kv_len, "kv_len", torch.int32, (bs,))
    _check(k_new, "k_new", torch.bfloat16, (bs, Hkv, D))
    _check(v_new, "v_new", torch.bfloat16, (bs, Hkv, D))
    if err is not None:
        _check(err, "err", torch.int32, (1,))
    _call("kv_append_mxfp8_paged", _ptr(k_codes), _ptr(k_scales), _ptr(v_codes), _ptr(v_scales), _ptr(block_table),
          max_pages, page_size, num_pages, _ptr(k_new), _ptr(v_new), Hkv * D, _ptr(kv_len), bs, Hkv, D, _ptr(err),
          _stream())


def _prefill_common(q, q_start, kv_len, max_q_len):
    _check(q, "q", torch.bfloat16, ndim=3)
    total_q, Hq, D = q.shape
    _check(q_start, "q_start", torch.int32, ndim=1)
    bs = q_start.shape[0] - 1
    _check(kv_len, "kv_len", torch.int32, (bs,))
    return total_q, Hq, D, bs


def gqa_prefill_attn(q, k_cache, v_cache, q_start, kv_len, max_q_len, scale, out=None, err=None):
    """Causal prefill / extend attention: q bf16 [total_q, Hq, 128] (new tokens of all sequences,
    sequence b at rows q_start[b] .. q_start[b+1]-1), caches bf16 [bs, Hkv, cap, 128] already
    holding the new rows, kv_len int32 [bs] counting them -> out bf16 [total_q, Hq, 128]."""
    total_q, Hq, D, bs = _prefill_common(q, q_start, kv_len, max_q_len)
    _check(k_cache, "k_cache", torch.bfloat16, ndim=4)
    _, Hkv, cap, _ = k_cache.shape
    _check(k_cache, "k_cache", torch.bfloat16, (bs, Hkv, cap, D))
    _check(v_cache, "v_cache", torch.bfloat16, (bs, Hkv, cap, D))
    out = _out(out, "out", torch.bfloat16, (total_q, Hq, D), q.device)
    if err is not None:
        _check(err, "err", torch.int32, (1,))
    _call("gqa_prefill_attn", _ptr(q), Hq * D, _ptr(k_cache), _ptr(v_cache), _ptr(q_start), _ptr(kv_len), bs,
          total_q, Hq, Hkv, D, cap, int(max_q_len), float(scale), _ptr(out), _ptr(err), _stream())
    return out


def gqa_prefill_attn_paged(q, k_pool, v_pool, block_table, q_start, kv_len, max_q_len, scale, out=None, err=None):
    """gqa_prefill_attn over paged pools bf16 [num_pages, Hkv, page_size, 128]."""
    total_q, Hq, D, bs = _prefill_common(q, q_start, kv_len, max_q_len)
    _check(k_pool, "k_pool", torch.bfloat16, ndim=4)
    num_pages, Hkv, page_size, _ = k_pool.shape
    _check(k_pool, "k_pool", torch.bfloat16, (num_pages, Hkv, page_size, D))
    _check(v_pool, "v_pool", torch.bfloat16, (num_pages, Hkv, page_size, D))
    _check(block_table, "block_table", torch.int32, ndim=2)
    if block_table.shape[0] != bs:
        raise ValueError("block_table: expected one row per sequence")
    max_pages = block_table.shape[1]
    out = _out(out, "out", torch.bfloat16, (total_q, Hq, D), q.device)
    if err is not None:
        _check(err, "err", torch.int32, (1,))
    _call("gqa_prefill_attn_paged", _ptr(q), Hq * D, _ptr(k_pool), _ptr(v_pool), _ptr(block_table), max_pages,
          page_size, num_pages, _ptr(q_start), _ptr(kv_len), bs, total_q, Hq, Hkv, D, int(max_q_len), float(scale),
          _ptr(out), _ptr(err), _stream())
    return out


def kv_append_extend(k_cache, v_cache, k_new, v_new, q_start, kv_len, max_q_len, err=None):
    """Write the new tokens' K/V rows (bf16 [total_q, Hkv, D]) into caches [bs, Hkv, cap, D] at
    positions kv_len[b] - T_b .. kv_len[b] - 1."""
    _check(k_cache, "k_cache", torch.bfloat16, ndim=4)
    bs, Hkv, cap, D = k_cache.shape
    _check(v_cache, "v_cache", torch.bfloat16, (bs, Hkv, cap, D))
    _check(k_new, "k_new", torch.bfloat16, ndim=3)
    total_q = k_new.shape[0]
    _check(k_new, "k_new", torch.bfloat16, (total_q, Hkv, D))
    _check(v_new, "v_new", torch.bfloat16, (total_q, Hkv, D))
    _check(q_start, "q_start", torch.int32, (bs + 1,))
    _check(kv_len, "kv_len", torch.int32, (bs,))
    if err is not None:
        _check(err, "err", torch.int32, (1,))
    _call("kv_append_extend", _ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new), Hkv * D, _ptr(q_start),
          _ptr(kv_len), bs, total_q, Hkv, D, cap, int(max_q_len), _ptr(err), _stream())


def kv_append_extend_paged(k_pool, v_pool, block_table, k_new, v_new, q_start, kv_len, max_q_len, err=None):
    """kv_append_extend into paged pools bf16 [num_pages, Hkv, page_size, D]."""
    _check(k_pool, "k_pool", torch.bfloat16, ndim=4)
    num_pages, Hkv, page_size, D = k_pool.shape
    _check(v_pool, "v_pool", torch.bfloat16, (num_pages, Hkv, page_size, D))
    _check(block_table, "block_table", torch.int32, ndim=2)
    bs, max_pages = block_table.shape
    _check(k_new, "k_new", torch.bfloat16, ndim=3)
    total_q = k_new.shape[0]
    _check(k_new, "k_new", torch.bfloat16, (total_q, Hkv, D))
    _check(v_new, "v_new", torch.bfloat16, (total_q, Hkv, D))
    _check(q_start, "q_start", torch.int32, (bs + 1,))
    _check(kv_len, "kv_len", torch.int32, (bs,))
    if err is not None:
        _check(err, "err", torch.int32, (1,))
    _call("kv_append_extend_paged", _ptr(k_pool), _ptr(v_pool), _ptr(block_table), max_pages, page_size, num_pages,
          _ptr(k_new), _ptr(v_new), Hkv * D, _ptr(q_start), _ptr(kv_len), bs, total_q, Hkv, D, int(max_q_len),
          _ptr(err), _stream())


# ------------------------------------------------------------------ block-scaled FP8 (bsgemm recipe)
def bs_quantize_act(x, q=None, s=None):
    """bf16 [M, K] -> (E4M3 codes [M, K], fp32 scales [M, K/128]): 1x128 blocks."""
    ld = _rows_view(x, "x", torch.bfloat16)
    M, K = x.shape
    q = _out(q, "q", torch.uint8, (M, K), x.device)
    s = _out(s, "s", torch.float32, (M, K // 128), x.device)
    _call("bs_quantize_act", _ptr(x), M, K, ld, _ptr(q), _ptr(s), _stream())
    return q, s


def bs_quantize_weight(w, q=None, s=None):
    """bf16 [N, K] -> (E4M3 codes [N, K], fp32 scales [ceil(N/128), K/128]): 128x128 blocks."""
    _check(w, "w", torch.bfloat16, ndim=2)
    N, K = w.shape
    q = _out(q, "q", torch.uint8, (N, K), w.device)
    s = _out(s, "s", torch.float32, ((N + 127) // 128, K // 128), w.device)
    _call("bs_quantize_weight", _ptr(w), N, K, _ptr(q), _ptr(s), _stream())
    return q, s


def bs_gemm_workspace(M, N, K):
    return int(lib().bs_gemm_workspace(M, N, K))


def bs_gemm(xq, xs, wq, ws, out=None, workspace=None, err=None):
    """out[M, N] (bf16) = block-scaled X' W'^T; xq/xs from bs_quantize_act, wq/ws from
    bs_quantize_weight."""
    _check(xq, "xq", torch.uint8, ndim=2)
    M, K = xq.shape
    _check(xs, "xs", torch.float32, (M, K // 128))
    _check(wq, "wq", torch.uint8, ndim=2)
    N = wq.shape[0]
    _check(wq, "wq", torch.uint8, (N, K))
    _check(ws, "ws", torch.float32, ((N + 127) // 128, K // 128))
    out = _out(out, "out", torch.bfloat16, (M, N), xq.device)
    if err is not None:
        _check(err, "err", torch.int32, (1,))
    need = bs_gemm_workspace(M, N, K)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=xq.device)
    ws_bytes = 0 if workspace is None else workspace.numel()
    _call("bs_gemm", _ptr(xq), _ptr(xs), _ptr(wq), _ptr(ws), M, N, K, _ptr(out), _ptr(workspace), ws_bytes, _ptr(err),
          _stream())
    return out


def gqa_decode_attn_noalloc(q, k_cache, v_cache, kv_len, max_kv_len, scale, out, err=None):
    """gqa_decode_attn without a workspace: for callers that cannot allocate device memory
    (inside CUDA-graph capture, real-time threads, hosts that own the memory budget). Its
    split-KV scratch is the library's fixed device array (gqa_decode_attn_noalloc_capacity()
    bytes, shared by all calls); `out` (and the optional int32 [1] device error flag `err`)
    must be passed in, so nothing is allocated here."""
    _check(k_cache, "k_cache", torch.bfloat16, ndim=4)
    bs, Hkv, cap, D = k_cache.shape
    _check(v_cache, "v_cache", torch.bfloat16, (bs, Hkv, cap, D))
    _check(kv_len, "kv_len", torch.int32, (bs,))
    _check(q, "q", torch.bfloat16, ndim=3)
    Hq = q.shape[1]
    _check(q, "q", torch.bfloat16, (bs, Hq, D))
    _check(out, "out", torch.bfloat16, (bs, Hq, D))
    if err is not None:
        _check(err, "err", torch.int32, (1,))
    _call("gqa_decode_attn_noalloc", _ptr(q), Hq * D, _ptr(k_cache), _ptr(v_cache), _ptr(kv_len), bs, Hq, Hkv, D,
          cap, int(max_kv_len), float(scale), _ptr(out), _ptr(err), _stream())
    return out


def kv_append(k_cache, v_cache, k_new, v_new, kv_len, err=None):
    """k_new/v_new: bf16 [bs, Hkv, D] or row-strided [bs, Hkv*D] views (e.g. slices of a fused QKV)."""
    _check(k_cache, "k_cache", torch.bfloat16, ndim=4)
    bs, Hkv, cap, D = k_cache.shape
    _check(v_cache, "v_cache", torch.bfloat16, (bs, Hkv, cap, D))
    _check(kv_len, "kv_len", torch.int32, (bs,))
    lds = []
    for t, name in ((k_new, "k_new"), (v_new, "v_new")):
        if t.dim() == 3:
            _check(t, name, torch.bfloat16, (bs, Hkv, D))
            lds.append(Hkv * D)
        else:
            lds.append(_rows_view(t, name, torch.bfloat16))
            if tuple(t.shape) != (bs, Hkv * D):
                raise ValueError(f"{name}: expected [bs, Hkv*D]")
    if lds[0] != lds[1]:
        raise ValueError("k_new and v_new must share a row stride")
    if err is not None:
        _check(err, "err", torch.int32, (1,))
    _call("kv_append", _ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new), lds[0], _ptr(kv_len), bs, Hkv, D,
          cap, _ptr(err), _stream())


def copy_bytes(dst, src):
    """dst <- src (same byte size, contiguous, 16-byte aligned, size a multiple of 16) by a
    kernel on the current stream; either side may be a pinned CPU tensor (mapped host memory)."""
    for t, name in ((dst, "dst"), (src, "src")):
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name}: expected a torch.Tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name}: must be contiguous")
        if not t.is_cuda and not t.is_pinned():
            raise ValueError(f"{name}: a CPU tensor must be pinned")
    n = dst.numel() * dst.element_size()
    if src.numel() * src.element_size() != n:
        raise ValueError("copy_bytes: dst and src differ in byte size")
    _call("copy_bytes", _ptr(dst), _ptr(src), n, _stream())
    return dst


def prev_tokens_shift(prev, next_tokens):
    """In place: prev int32 [bs, W, cw], next_tokens int32 [bs, cw] (exact shapes, no promotion)."""
    _check(prev, "prev", torch.int32, ndim=3)
    bs, W, cw = prev.shape
    _check(next_tokens, "next_tokens", torch.int32, (bs, cw))
    _call("prev_tokens_shift", _ptr(prev), _ptr(next_tokens), bs, W, cw, _stream())
    return prev
