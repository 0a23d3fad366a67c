"""CPU-only checks of the C ABI: the library loads, exports every entry point declared
in include/mxg.h, and rejects bad arguments on the host before touching the device."""
import ctypes
import subprocess

import pytest

from mxfp8_mlp_gqa_gb300 import api, build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return api.lib()


def test_header_declares_the_entry_points():
    names = set(api.header_functions())
    for n in ["mxfp8_quantize", "rmsnorm_mxfp8_quantize", "mxfp8_gemm", "mxfp8_gemm_workspace",
              "mlp_gate_up_swiglu_mxfp8", "mlp_swiglu_mxfp8", "mlp_swiglu_mxfp8_workspace", "gqa_decode_attn",
              "gqa_decode_attn_workspace", "kv_append", "prev_tokens_shift", "mxg_status_str", "mxg_version"]:
        assert n in names, n


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for n in api.header_functions():
        assert n in exported, n
        assert getattr(lib, n) is not None
    for n in api._SIGS:
        assert n in api.header_functions(), f"binding signature for undeclared {n}"


def test_status_strings(lib):
    assert lib.mxg_status_str(0) == b"ok"
    assert lib.mxg_status_str(3) == b"misaligned pointer or stride"
    assert lib.mxg_status_str(99) == b"unknown status"
    assert lib.mxg_version() >= 100


# Host-side validation returns before any CUDA call, so these run without a GPU.
FAKE = ctypes.c_void_p(0x10000)     # 16-byte aligned, never dereferenced
ODD = ctypes.c_void_p(0x10008)


def test_quantize_rejects_bad_shapes(lib):
    assert lib.mxfp8_quantize(None, 1, 32, 32, FAKE, FAKE, None) == 1
    assert lib.mxfp8_quantize(FAKE, 1, 48, 48, FAKE, FAKE, None) == 2       # K % 32
    assert lib.mxfp8_quantize(FAKE, 1, 32, 16, FAKE, FAKE, None) == 2       # ld < K
    assert lib.mxfp8_quantize(ODD, 1, 32, 32, FAKE, FAKE, None) == 3        # misaligned x
    assert lib.mxfp8_quantize(FAKE, 1, 32, 36, FAKE, FAKE, None) == 3       # ld % 8
    assert lib.mxfp8_quantize(FAKE, 0, 32, 32, FAKE, FAKE, None) == 0       # empty: nothing enqueued
    assert lib.rmsnorm_mxfp8_quantize(FAKE, FAKE, -1.0, 1, 32, 32, FAKE, FAKE, None) == 1
    assert lib.rmsnorm_mxfp8_quantize(FAKE, FAKE, 1e-6, 1, 17952, 17952, FAKE, FAKE, None) == 2


def test_gemm_and_mlp_reject_bad_shapes(lib):
    assert lib.mxfp8_gemm(FAKE, FAKE, FAKE, FAKE, 4, 16, 40, None, FAKE, None, 0, None) == 2   # K % 32
    assert lib.mxfp8_gemm(FAKE, FAKE, FAKE, FAKE, 4, 12, 64, None, FAKE, None, 0, None) == 2   # N % 8
    assert lib.mlp_gate_up_swiglu_mxfp8(FAKE, FAKE, 1, 256, 100, FAKE, FAKE, FAKE, FAKE, None) == 2
    ws = lib.mlp_swiglu_mxfp8_workspace(4, 256, 768)
    assert ws >= 4 * 768 + 4 * 24
    assert lib.mlp_swiglu_mxfp8(FAKE, FAKE, 4, 256, 768, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, ws - 1, None) == 4


def test_attention_and_cache_reject_bad_shapes(lib):
    args = dict(ld_q=4 * 64, bs=1, Hq=4, Hkv=2, D=64, cap=1024, mkv=1024)

    def call(**kw):
        a = {**args, **kw}
        return lib.gqa_decode_attn(FAKE, a["ld_q"], FAKE, FAKE, FAKE, a["bs"], a["Hq"], a["Hkv"], a["D"], a["cap"],
                                   a["mkv"], 0.125, FAKE, None, FAKE, 1 << 30, None)
    assert call(Hq=6, Hkv=4) == 2          # Hq % Hkv
    assert call(Hq=32, Hkv=2) == 2         # group > 8
    assert call(D=96) == 2                 # head_dim
    assert call(ld_q=100) == 2             # ld_q < Hq*D
    assert call(bs=65536, cap=32768, Hkv=8, Hq=32, ld_q=32 * 64) == 2  # bs*Hkv*cap >= 2^31
    assert lib.gqa_decode_attn(FAKE, 256, FAKE, FAKE, FAKE, 1, 4, 2, 64, 1024, 1024, -1.0, FAKE, None, FAKE, 1 << 30,
                               None) == 1  # scale
    need = lib.gqa_decode_attn_workspace(64, 32, 8, 128, 4096)
    assert need > 0 and lib.gqa_decode_attn_workspace(1, 4, 2, 64, 64) == 0
    assert lib.gqa_decode_attn(FAKE, 4096, FAKE, FAKE, FAKE, 64, 32, 8, 128, 32768, 4096, 0.1, FAKE, None, FAKE,
                               need - 1, None) == 4
    assert lib.kv_append(FAKE, FAKE, FAKE, FAKE, 100, FAKE, 1, 2, 64, 16, None, None) == 2   # ld_new < Hkv*D
    assert lib.prev_tokens_shift(FAKE, FAKE, 1, 0, 10, None) == 2
    assert lib.prev_tokens_shift(FAKE, FAKE, 1, 2000, 10, None) == 2                       # W*cw > 12288
    assert lib.prev_tokens_shift(None, FAKE, 1, 8, 10, None) == 1


def test_copy_bytes_host_checks(lib):
    # rejected on the host before anything is launched: null pointers, negative or ragged sizes
    st = ctypes.c_void_p(0)
    assert lib.copy_bytes(None, ctypes.c_void_p(16), 16, st) == 1         # MXG_EINVAL
    assert lib.copy_bytes(ctypes.c_void_p(16), ctypes.c_void_p(16), -16, st) == 1
    assert lib.copy_bytes(ctypes.c_void_p(16), ctypes.c_void_p(16), 0, st) == 0   # nothing to do
    assert lib.copy_bytes(ctypes.c_void_p(16), ctypes.c_void_p(16), 24, st) == 3  # MXG_EALIGN: 24 % 16
    assert lib.copy_bytes(ctypes.c_void_p(8), ctypes.c_void_p(16), 32, st) == 3   # unaligned dst


def test_decode_layer_input_layout():
    # x, next_tokens and kv_len share one packed buffer: sections in order, 16-byte aligned,
    # non-overlapping, and the bench shape's total is the bytes the host copies in per step
    from mxfp8_mlp_gqa_gb300.step import DecodeLayer
    for bs, d, cw in ((64, 2560, 10), (1, 256, 10), (3, 72, 7)):
        (o_x, o_n, o_l), total = DecodeLayer._input_layout(bs, d, cw)
        assert o_x == 0 and o_n >= bs * d * 2 and o_l >= o_n + bs * cw * 4 and total >= o_l + bs * 4
        assert o_n % 16 == 0 and o_l % 16 == 0 and total % 16 == 0
        assert total - (o_l + bs * 4) < 16
    assert DecodeLayer._input_layout(64, 2560, 10)[1] == 330496
