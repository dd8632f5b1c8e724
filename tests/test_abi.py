"""The C-ABI library loads, exports every function include/nvfp4.h declares,
and rejects bad arguments on the host before any launch (no GPU needed)."""
import ctypes
import os
import re

import pytest
import torch

import nvfp4_bit_block_02_b300 as nv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4.h")


@pytest.fixture(scope="module")
def L():
    from nvfp4_bit_block_02_b300 import build
    build.build()
    return nv.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(nvfp4_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["nvfp4_amax", "nvfp4_quantize", "nvfp4_quantize_grouped", "nvfp4_rht_quantize", "nvfp4_dequantize",
                     "nvfp4_transpose_2d", "nvfp4_gemm", "nvfp4_gemm_amax", "nvfp4_gemm_quantize",
                     "nvfp4_gemm_grouped", "nvfp4_w4a16_gemm", "nvfp4_codes_bytes", "nvfp4_scales_bytes", "nvfp4_sync_check",
                     "nvfp4_status_string", "nvfp4_last_error", "nvfp4_test_expire_next_wait"]:
        assert required in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
        assert ctypes.cast(getattr(L, name), ctypes.c_void_p).value


def test_size_queries(L):
    assert nv.codes_bytes(8192, 4096) == 8192 * 2048
    assert nv.scales_bytes(8192, 4096) == 8192 * 256
    assert nv.scales_bytes(130, 80) == 256 * 8         # rows padded to 128, blocks (5) to 4
    assert nv.scales_bytes(0, 64) == 0 and nv.codes_bytes(0, 64) == 0


def test_status_strings(L):
    for code, name in nv.STATUS.items():
        assert L.nvfp4_status_string(code).decode() == name


def _fake_tensor(rows, cols, base=0x10000):
    return nv.CTensor(base, base + 0x100000, base + 0x200000, base + 0x200100, rows, cols)


def _call_quantize(L, x_ptr, dtype, rows, cols, ld, cfg, out):
    return L.nvfp4_quantize(ctypes.c_void_p(x_ptr), dtype, rows, cols, ld, ctypes.byref(cfg), None,
                            ctypes.byref(out), None)


def test_quantize_argument_errors(L):
    cfg = nv.CQuantConfig(nv.BLOCK_1D, nv.ROUND_RNE, nv.SCALE_MAX6, 0, 0, 0)
    out = _fake_tensor(64, 64)
    # bad dtype / enums
    assert _call_quantize(L, 0x1000, 7, 64, 64, 64, cfg, out) == 1
    bad = nv.CQuantConfig(5, 0, 0, 0, 0, 0)
    assert _call_quantize(L, 0x1000, nv.BF16, 64, 64, 64, bad, out) == 1
    # output orientation mismatch
    assert _call_quantize(L, 0x1000, nv.BF16, 64, 64, 64, cfg, _fake_tensor(64, 32)) == 1
    # K not a multiple of 16
    assert _call_quantize(L, 0x1000, nv.BF16, 64, 40, 40, cfg, _fake_tensor(64, 40)) == 2
    # 2D needs rows % 16
    cfg2 = nv.CQuantConfig(nv.BLOCK_2D, 0, 0, 0, 0, 0)
    assert _call_quantize(L, 0x1000, nv.BF16, 24, 64, 64, cfg2, _fake_tensor(24, 64)) == 2
    # misaligned input / leading dimension
    assert _call_quantize(L, 0x1008, nv.BF16, 64, 64, 64, cfg, out) == 3
    assert _call_quantize(L, 0x1000, nv.BF16, 64, 64, 68, cfg, out) == 3
    # NULL buffers
    nul = nv.CTensor(0, 0x2000, 0x3000, 0x4000, 64, 64)
    assert _call_quantize(L, 0x1000, nv.BF16, 64, 64, 64, cfg, nul) == 1
    assert "codes" in L.nvfp4_last_error().decode()
    nul_g = nv.CTensor(0x2000, 0x2000, 0, 0x4000, 64, 64)
    assert _call_quantize(L, 0x1000, nv.BF16, 64, 64, 64, cfg, nul_g) == 1
    # the RHT path refuses 2D blocks
    assert L.nvfp4_rht_quantize(ctypes.c_void_p(0x1000), nv.BF16, 64, 64, 64, ctypes.byref(cfg2), 1, None,
                                ctypes.byref(out), None, None) == 2


def test_gemm_argument_errors(L):
    A = _fake_tensor(128, 256)
    B = _fake_tensor(256, 256, base=0x800000)
    D = ctypes.c_void_p(0x4000000)
    assert L.nvfp4_gemm(ctypes.byref(A), ctypes.byref(_fake_tensor(256, 512)), D, nv.BF16, 256, None) == 1
    # K must be a multiple of 64; M and N may be anything
    assert L.nvfp4_gemm(ctypes.byref(_fake_tensor(128, 96)), ctypes.byref(_fake_tensor(256, 96)), D, nv.BF16,
                        256, None) == 2
    assert "multiple of 64" in L.nvfp4_last_error().decode()
    # N * elsize must keep rows of D 16-byte aligned (ldd = N = 100 BF16: 200 bytes)
    assert L.nvfp4_gemm(ctypes.byref(_fake_tensor(100, 256)), ctypes.byref(_fake_tensor(100, 256, base=0x800000)), D,
                        nv.BF16, 100, None) == 3
    assert L.nvfp4_gemm(ctypes.byref(A), ctypes.byref(B), D, nv.BF16, 200, None) == 1       # ldd < N
    assert L.nvfp4_gemm(ctypes.byref(A), ctypes.byref(B), ctypes.c_void_p(0x4000008), nv.BF16, 256, None) == 3
    assert L.nvfp4_gemm(ctypes.byref(A), ctypes.byref(B), D, 9, 256, None) == 1
    assert L.nvfp4_gemm_grouped(nv.MAX_GROUPS + 1, None, None, None, nv.BF16, None) == 1
    assert L.nvfp4_gemm_grouped(0, None, None, None, nv.BF16, None) == 0


def test_amax_argument_errors(L):
    a = ctypes.c_void_p(0x4000)
    assert L.nvfp4_amax(ctypes.c_void_p(0x1000), 7, 4, 64, 64, a, None) == 1          # dtype
    assert L.nvfp4_amax(ctypes.c_void_p(0x1000), nv.BF16, 4, 64, 32, a, None) == 1    # ld < cols
    assert L.nvfp4_amax(ctypes.c_void_p(0x1000), nv.BF16, 4, 64, 64, None, None) == 1  # amax NULL
    assert L.nvfp4_amax(ctypes.c_void_p(0x1008), nv.BF16, 4, 64, 64, a, None) == 3    # misaligned x
    assert L.nvfp4_amax(ctypes.c_void_p(0x1000), nv.BF16, 4, 12, 64, a, None) == 3    # cols*2 % 16


def test_quantize_grouped_argument_errors(L):
    cfg = nv.CQuantConfig(nv.BLOCK_1D, nv.ROUND_RNE, nv.SCALE_MAX6, 0, 0, 0)
    n = 2
    X = (ctypes.c_void_p * n)(0x1000, 0x2000)
    R = (ctypes.c_int64 * n)(64, 64)
    C = (ctypes.c_int64 * n)(64, 40)
    O = (nv.CTensor * n)(_fake_tensor(64, 64), _fake_tensor(64, 40, base=0x800000))
    assert L.nvfp4_quantize_grouped(nv.MAX_GROUPS + 1, X, nv.BF16, R, C, C, ctypes.byref(cfg), O, None) == 1
    assert L.nvfp4_quantize_grouped(0, None, nv.BF16, None, None, None, ctypes.byref(cfg), None, None) == 0
    assert L.nvfp4_quantize_grouped(n, None, nv.BF16, R, C, C, ctypes.byref(cfg), O, None) == 1
    assert L.nvfp4_quantize_grouped(n, X, nv.BF16, R, C, C, ctypes.byref(cfg), O, None) == 2   # group 1: K % 16
    assert "group 1" in L.nvfp4_last_error().decode()


def test_transpose_2d_argument_errors(L):
    q = _fake_tensor(64, 128)
    qt = _fake_tensor(128, 64, base=0x800000)
    assert L.nvfp4_transpose_2d(None, ctypes.byref(qt), None) == 1
    assert L.nvfp4_transpose_2d(ctypes.byref(q), ctypes.byref(_fake_tensor(64, 128, base=0x800000)), None) == 1
    assert L.nvfp4_transpose_2d(ctypes.byref(_fake_tensor(40, 128)), ctypes.byref(_fake_tensor(128, 40, base=0x800000)),
                                None) == 2                                                  # rows % 16
    assert L.nvfp4_transpose_2d(ctypes.byref(q), ctypes.byref(_fake_tensor(128, 64)), None) == 1   # shares buffers
    mis = nv.CTensor(0x800008, 0x900000, 0xA00000, 0xA00100, 128, 64)
    assert L.nvfp4_transpose_2d(ctypes.byref(q), ctypes.byref(mis), None) == 3


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device error path")
def test_launch_without_a_device_reports_cuda_error(L):
    """With no GPU the first CUDA call fails; the API returns NVFP4_ERR_CUDA
    with a message instead of crashing (the pointers are never touched)."""
    cfg = nv.CQuantConfig(nv.BLOCK_1D, nv.ROUND_RNE, nv.SCALE_MAX6, 0, 0, 0)
    out = _fake_tensor(64, 64)
    st = _call_quantize(L, 0x1000, nv.BF16, 64, 64, 64, cfg, out)
    assert st == 4
    assert "cuda" in L.nvfp4_last_error().decode().lower()
    assert L.nvfp4_sync_check(None) == 4


def test_empty_tensors_are_ok_without_launch_for_gemm(L):
    A = _fake_tensor(0, 256)
    B = _fake_tensor(128, 256)
    assert L.nvfp4_gemm(ctypes.byref(A), ctypes.byref(B), ctypes.c_void_p(0x4000000), nv.BF16, 128, None) == 0


def test_gemm_amax_argument_errors(L):
    A = _fake_tensor(128, 256)
    B = _fake_tensor(256, 256, base=0x800000)
    D = ctypes.c_void_p(0x4000000)
    assert L.nvfp4_gemm_amax(ctypes.byref(A), ctypes.byref(B), D, nv.BF16, 256, None, None) == 1   # amax_out NULL
    assert L.nvfp4_gemm_amax(ctypes.byref(A), ctypes.byref(_fake_tensor(256, 512)), D, nv.BF16, 256,
                             ctypes.c_void_p(0x5000000), None) == 1                                  # K differs


def test_w4a16_argument_errors(L):
    W = _fake_tensor(256, 512)
    x, y = ctypes.c_void_p(0x4000000), ctypes.c_void_p(0x5000000)
    w = ctypes.byref(W)
    call = L.nvfp4_w4a16_gemm
    assert call(x, nv.F32, 4, 512, w, y, nv.BF16, 256, None) == 1                      # x must be BF16
    assert call(x, nv.BF16, 4, 512, w, y, 9, 256, None) == 1                           # output dtype
    assert call(x, nv.BF16, -1, 512, w, y, nv.BF16, 256, None) == 1                    # negative M
    assert call(x, nv.BF16, 4, 500, w, y, nv.BF16, 256, None) == 1                     # ldx < K
    assert call(x, nv.BF16, 4, 512, w, y, nv.BF16, 200, None) == 1                     # ldy < N
    assert call(x, nv.BF16, 4, 512, None, y, nv.BF16, 256, None) == 1                  # W NULL
    assert call(x, nv.BF16, 4, 40, ctypes.byref(_fake_tensor(256, 40)), y, nv.BF16, 256, None) == 2   # K % 16
    assert call(ctypes.c_void_p(0x4000008), nv.BF16, 4, 512, w, y, nv.BF16, 256, None) == 3          # x alignment
    assert call(x, nv.BF16, 4, 516, w, y, nv.BF16, 256, None) == 3                     # ldx % 8
    assert call(x, nv.BF16, 4, 512, w, ctypes.c_void_p(0x5000001), nv.BF16, 256, None) == 3          # y alignment
    assert call(x, nv.BF16, 4, 512, w, ctypes.c_void_p(0x5000002), nv.F32, 256, None) == 3
    assert call(x, nv.BF16, 4, 512, w, None, nv.BF16, 256, None) == 1                  # y NULL
    assert call(None, nv.BF16, 4, 512, w, y, nv.BF16, 256, None) == 1                  # x NULL
    assert call(x, nv.BF16, 0, 512, w, None, nv.BF16, 256, None) == 0                  # M = 0: nothing to do
    big = (1 << 28) + 16                                                                  # K beyond the kernel's offsets
    assert call(x, nv.BF16, 1, big, ctypes.byref(_fake_tensor(16, big)), y, nv.BF16, 16, None) == 2
    assert "too large" in L.nvfp4_last_error().decode()


def test_gemm_quantize_argument_errors(L):
    A = _fake_tensor(128, 256)
    B = _fake_tensor(256, 256, base=0x800000)
    out = _fake_tensor(128, 256, base=0xC00000)
    amax = ctypes.c_void_p(0x5000000)
    D = ctypes.c_void_p(0x4000000)
    call = L.nvfp4_gemm_quantize
    assert call(ctypes.byref(A), ctypes.byref(B), None, D, 256, None, ctypes.byref(out), None) == 1   # amax_in NULL
    assert call(ctypes.byref(A), ctypes.byref(B), amax, D, 256, None, None, None) == 1                # out NULL
    bad = _fake_tensor(128, 128, base=0xC00000)
    assert call(ctypes.byref(A), ctypes.byref(B), amax, D, 256, None, ctypes.byref(bad), None) == 1   # out not M x N
    B2, o2 = _fake_tensor(264, 256, base=0x800000), _fake_tensor(128, 264, base=0xC00000)
    assert call(ctypes.byref(A), ctypes.byref(B2), amax, None, 0, None, ctypes.byref(o2), None) == 2  # N % 16
    assert call(ctypes.byref(A), ctypes.byref(B), amax, D, 200, None, ctypes.byref(out), None) == 1   # ldd < N
    assert call(ctypes.byref(A), ctypes.byref(B), amax, ctypes.c_void_p(0x4000008), 256, None, ctypes.byref(out),
                None) == 3                                                                          # D misaligned
    assert call(ctypes.byref(A), ctypes.byref(B), amax, D, 256, amax, ctypes.byref(out), None) == 1   # aliasing


def test_wait_expiry_hook_arguments(L):
    # no launch happens here: arming only sets a process-wide flag
    assert L.nvfp4_test_expire_next_wait(0, 20_000_000) == 1
    assert L.nvfp4_test_expire_next_wait(3, 20_000_000) == 1
    assert L.nvfp4_test_expire_next_wait(1, 999_999) == 1
    assert L.nvfp4_test_expire_next_wait(2, 2_000_000_001) == 1
    for op in (1, 2):
        assert L.nvfp4_test_expire_next_wait(op, 20_000_000) == 0
        assert L.nvfp4_test_expire_next_wait(op, 0) == 0  # disarmed again
