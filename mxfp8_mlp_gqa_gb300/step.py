"""One slow-AR decoder-layer step under continuous batching, composed from the library's
entry points (every step runs in libmxg kernels; this module only owns buffers and the
call order):

    RMSNorm+MX-quantise -> QKV projection with the KV append fused in its epilogue ->
    GQA decode attention with the MX-quantised output fused in -> O projection + residual ->
    RMSNorm+MX-quantise -> SwiGLU MLP (gate/up + SwiGLU + requant, down + residual);
    the prev-window shift runs on a forked stream branch (it depends on nothing above)

The pages list the layer as RMSNorm -> attention -> RMSNorm -> MLP (Qwen3-style, [S2.1]
"The Real Reason Voice AI Costs Money" / "Kernel Benchmark Results", [FSKV] §2). The QKV
and O projections are the plainest way to join a 32x128-wide attention to a 2560-wide
residual stream; RoPE and QK-norm are not on the pages and are left out.

All buffers have stable addresses, so ``capture()`` records the step in a CUDA graph and
``replay()`` re-launches it; ``kv_len`` / ``next_tokens`` / ``x`` are updated in place
between replays. The three per-step inputs are views of one packed device buffer
(``inputs``), so a caller feeding the layer from the host moves them in one copy:
``host_io()`` returns pinned host buffers of the same layout and ``capture_io()`` records
that copy, the step and the copy of ``y`` back to the host as one graph.
"""
from __future__ import annotations

import math

import torch

from . import api


class DecodeLayer:
    def __init__(self, bs, d_model, d_ff, Hq, Hkv, D, cap, max_kv_len, W, cw, eps=1e-6, device="cuda"):
        self.bs, self.d_model, self.d_ff = bs, d_model, d_ff
        self.Hq, self.Hkv, self.D, self.cap = Hq, Hkv, D, cap
        self.max_kv_len, self.eps, self.scale = max_kv_len, eps, 1.0 / math.sqrt(D)
        dev = torch.device(device)
        u8, bf, i32 = torch.uint8, torch.bfloat16, torch.int32
        nqkv = (Hq + 2 * Hkv) * D
        self.nqkv = nqkv
        e = lambda shape, dt: torch.empty(shape, dtype=dt, device=dev)  # noqa: E731
        # caller-visible state; the per-step inputs x, next_tokens, kv_len are views of one
        # packed byte buffer (16-byte aligned sections) so that one copy brings them in
        self.cw = cw
        self.in_offsets, nbytes = self._input_layout(bs, d_model, cw)
        self.inputs = torch.zeros((nbytes,), dtype=u8, device=dev)
        self.x, self.next_tokens, self.kv_len = self._input_views(self.inputs)
        self.prev = e((bs, W, cw), i32)
        self.k_cache = e((bs, Hkv, cap, D), bf)
        self.v_cache = e((bs, Hkv, cap, D), bf)
        self.err = torch.zeros((1,), dtype=i32, device=dev)
        # weights (MXFP8, set by load_weights)
        self.wqkv = (e((nqkv, d_model), u8), e((nqkv, d_model // 32), u8))
        self.wo = (e((d_model, Hq * D), u8), e((d_model, Hq * D // 32), u8))
        self.w13 = (e((2 * d_ff, d_model), u8), e((2 * d_ff, d_model // 32), u8))
        self.w2 = (e((d_model, d_ff), u8), e((d_model, d_ff // 32), u8))
        self.gamma1 = e((d_model,), bf)
        self.gamma2 = e((d_model,), bf)
        # intermediates
        self.xq, self.xs = e((bs, d_model), u8), e((bs, d_model // 32), u8)
        self.qkv = e((bs, nqkv), bf)
        self.o = e((bs, Hq, D), bf)
        self.oq, self.os = e((bs, Hq * D), u8), e((bs, Hq * D // 32), u8)
        self.x1 = e((bs, d_model), bf)
        self.hq_in, self.hs_in = e((bs, d_model), u8), e((bs, d_model // 32), u8)
        self.y = e((bs, d_model), bf)
        self.ws_attn = e((max(1, api.gqa_decode_attn_workspace(bs, Hq, Hkv, D, max_kv_len)),), u8)
        self.ws_mlp = torch.zeros((api.mlp_swiglu_mxfp8_workspace(bs, d_model, d_ff),), dtype=u8, device=dev)
        self.ws_o = torch.zeros((max(1, api.mxfp8_gemm_workspace(bs, d_model, Hq * D)),), dtype=u8, device=dev)
        self.graph = None
        self.graph_io = None
        self.side = torch.cuda.Stream(device=dev)

    @staticmethod
    def _input_layout(bs, d_model, cw):
        """Byte offsets of x (bf16 [bs, d_model]), next_tokens (int32 [bs, cw]) and kv_len
        (int32 [bs]) in the packed input buffer, each section 16-byte aligned, and its size."""
        r16 = lambda n: (n + 15) // 16 * 16  # noqa: E731
        o_x = 0
        o_next = o_x + r16(bs * d_model * 2)
        o_len = o_next + r16(bs * cw * 4)
        return (o_x, o_next, o_len), o_len + r16(bs * 4)

    def _input_views(self, buf):
        o_x, o_next, o_len = self.in_offsets
        bs, d_model, cw = self.bs, self.d_model, self.cw
        x = buf[o_x:o_x + bs * d_model * 2].view(torch.bfloat16).view(bs, d_model)
        nxt = buf[o_next:o_next + bs * cw * 4].view(torch.int32).view(bs, cw)
        lens = buf[o_len:o_len + bs * 4].view(torch.int32)
        return x, nxt, lens

    def host_io(self):
        """Pinned host buffers for feeding the layer from the host: (packed input bytes, its x /
        next_tokens / kv_len views, y). Fill the views, then ``replay_io()``."""
        h_in = torch.zeros((self.inputs.numel(),), dtype=torch.uint8, pin_memory=True)
        h_y = torch.empty((self.bs, self.d_model), dtype=torch.bfloat16, pin_memory=True)
        return h_in, self._input_views(h_in), h_y

    def load_weights(self, wqkv_bf16, wo_bf16, w13_bf16, w2_bf16, gamma1, gamma2):
        """bf16 weights on the device -> MXFP8 once (weight prep, not part of a step)."""
        for src, dst in ((wqkv_bf16, self.wqkv), (wo_bf16, self.wo), (w13_bf16, self.w13), (w2_bf16, self.w2)):
            api.mxfp8_quantize(src, q=dst[0], s=dst[1])
        self.gamma1.copy_(gamma1)
        self.gamma2.copy_(gamma2)

    def step(self):
        Hq, Hkv, D = self.Hq, self.Hkv, self.D
        main = torch.cuda.current_stream()
        self.side.wait_stream(main)
        with torch.cuda.stream(self.side):
            api.prev_tokens_shift(self.prev, self.next_tokens)
        api.rmsnorm_mxfp8_quantize(self.x, self.gamma1, self.eps, q=self.xq, s=self.xs)
        api.mxfp8_gemm_qkv_kv_append(self.xq, self.xs, *self.wqkv, Hq, Hkv, self.k_cache, self.v_cache,
                                     self.kv_len, qkv=self.qkv, err=self.err)
        qd = Hq * D
        api.gqa_decode_attn(self.qkv[:, :qd], self.k_cache, self.v_cache, self.kv_len, self.max_kv_len, self.scale,
                            out=self.o, err=self.err, workspace=self.ws_attn, oq=self.oq, os=self.os)
        api.mxfp8_gemm(self.oq, self.os, *self.wo, residual=self.x, c=self.x1, workspace=self.ws_o)
        api.rmsnorm_mxfp8_quantize(self.x1, self.gamma2, self.eps, q=self.hq_in, s=self.hs_in)
        api.mlp_swiglu_mxfp8(self.hq_in, self.hs_in, *self.w13, *self.w2, residual=self.x1, y=self.y,
                             workspace=self.ws_mlp)
        main.wait_stream(self.side)
        return self.y

    def capture(self):
        """Record one step in a CUDA graph (run once eagerly first so lazy init is done)."""
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.graph, stream=s):
                self.step()
        torch.cuda.current_stream().wait_stream(s)
        return self.graph

    def replay(self):
        self.graph.replay()
        return self.y

    def capture_io(self, h_in, h_y, kernel_copy=True):
        """Record [packed inputs host -> device, one step, y device -> host] in one CUDA graph
        (h_in / h_y pinned, as from ``host_io()``). kernel_copy: move the bytes with the
        library's copy kernel through the host memory's device mapping (chained to the step's
        kernels); False: copy-engine copies."""
        if (not (h_in.is_pinned() and h_y.is_pinned()) or h_in.dtype != torch.uint8 or
                h_in.numel() != self.inputs.numel() or h_y.dtype != self.y.dtype or h_y.shape != self.y.shape or
                not (h_in.is_contiguous() and h_y.is_contiguous())):
            raise ValueError("capture_io needs the pinned buffers of host_io()")
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.graph_io = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.graph_io, stream=s):
                if kernel_copy:
                    api.copy_bytes(self.inputs, h_in)
                else:
                    self.inputs.copy_(h_in, non_blocking=True)
                self.step()
                if kernel_copy:
                    api.copy_bytes(h_y, self.y)
                else:
                    h_y.copy_(self.y, non_blocking=True)
        torch.cuda.current_stream().wait_stream(s)
        return self.graph_io

    def replay_io(self):
        """One step fed from and returning to the host buffers given to ``capture_io`` (the
        caller synchronises before reading y)."""
        self.graph_io.replay()
