"""NVFP4 quantizer and block-scaled GEMM for B300 (sm_103a).

Thin ctypes binding of ``libnvfp4.so`` (C ABI in ``include/nvfp4.h``): it only
turns torch tensors into pointers and the current CUDA stream into a handle.
Every step of the quantizer and the GEMM runs in the library's CUDA kernels;
there is no CPU fallback, and a missing or unloadable library raises.

Format ("NVIDIA Introduces a 4-Bit Pretraining Methodology Using NVFP4",
"Summary"): 16-element blocks of E2M1 codes, an E4M3 scale per block, an FP32
scale per tensor.  Recipe options ("Method"): 2D 16x16 weight blocks, 16x16
Random Hadamard Transform on Wgrad inputs, stochastic rounding on gradients;
Four-over-Six scaling (the hyper.ai story on the Nemotron 3 Ultra NVFP4
checkpoint).
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libnvfp4.so")

F32, BF16 = 0, 1
BLOCK_1D, BLOCK_2D = 0, 1
ROUND_RNE, ROUND_STOCHASTIC = 0, 1
SCALE_MAX6, SCALE_FOUR_OVER_SIX = 0, 1
STATUS = {0: "NVFP4_OK", 1: "NVFP4_ERR_INVALID_ARG", 2: "NVFP4_ERR_UNSUPPORTED_SHAPE", 3: "NVFP4_ERR_MISALIGNED",
          4: "NVFP4_ERR_CUDA", 5: "NVFP4_ERR_TIMEOUT"}
MAX_GROUPS = 128


class CTensor(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("global_scale", ctypes.c_void_p),
                ("amax", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64)]


class CQuantConfig(ctypes.Structure):
    _fields_ = [("block", ctypes.c_int), ("round", ctypes.c_int), ("scaling", ctypes.c_int),
                ("transpose", ctypes.c_int), ("seed", ctypes.c_uint64), ("offset", ctypes.c_uint64)]


class NVFP4Error(RuntimeError):
    def __init__(self, status: int, fn: str, msg: str):
        super().__init__(f"{fn}: {STATUS.get(status, status)}: {msg}")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """Load libnvfp4.so (raises if it is missing: there is no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing; build it with `python -m nvfp4_bit_block_02_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        P, I64, U64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64
        L.nvfp4_codes_bytes.argtypes = [I64, I64]
        L.nvfp4_codes_bytes.restype = ctypes.c_size_t
        L.nvfp4_scales_bytes.argtypes = [I64, I64]
        L.nvfp4_scales_bytes.restype = ctypes.c_size_t
        L.nvfp4_quantize.argtypes = [P, ctypes.c_int, I64, I64, I64, ctypes.POINTER(CQuantConfig), P,
                                     ctypes.POINTER(CTensor), P]
        L.nvfp4_rht_quantize.argtypes = [P, ctypes.c_int, I64, I64, I64, ctypes.POINTER(CQuantConfig), U64, P,
                                         ctypes.POINTER(CTensor), P, P]
        L.nvfp4_dequantize.argtypes = [ctypes.POINTER(CTensor), P, ctypes.c_int, P]
        L.nvfp4_transpose_2d.argtypes = [ctypes.POINTER(CTensor), ctypes.POINTER(CTensor), P]
        L.nvfp4_amax.argtypes = [P, ctypes.c_int, I64, I64, I64, P, P]
        L.nvfp4_quantize_grouped.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_void_p), ctypes.c_int,
                                             ctypes.POINTER(I64), ctypes.POINTER(I64), ctypes.POINTER(I64),
                                             ctypes.POINTER(CQuantConfig), ctypes.POINTER(CTensor), P]
        L.nvfp4_gemm.argtypes = [ctypes.POINTER(CTensor), ctypes.POINTER(CTensor), P, ctypes.c_int, I64, P]
        L.nvfp4_gemm_amax.argtypes = [ctypes.POINTER(CTensor), ctypes.POINTER(CTensor), P, ctypes.c_int, I64, P, P]
        L.nvfp4_gemm_quantize.argtypes = [ctypes.POINTER(CTensor), ctypes.POINTER(CTensor), P, P, I64, P,
                                          ctypes.POINTER(CTensor), P]
        L.nvfp4_gemm_grouped.argtypes = [ctypes.c_int, ctypes.POINTER(CTensor), ctypes.POINTER(CTensor),
                                         ctypes.POINTER(ctypes.c_void_p), ctypes.c_int, P]
        L.nvfp4_w4a16_gemm.argtypes = [P, ctypes.c_int, I64, I64, ctypes.POINTER(CTensor), P, ctypes.c_int, I64, P]
        L.nvfp4_sync_check.argtypes = [P]
        L.nvfp4_test_expire_next_wait.argtypes = [ctypes.c_int, ctypes.c_uint64]
        for fn in ("nvfp4_amax", "nvfp4_quantize", "nvfp4_quantize_grouped", "nvfp4_rht_quantize", "nvfp4_dequantize",
                   "nvfp4_transpose_2d", "nvfp4_gemm", "nvfp4_gemm_amax", "nvfp4_gemm_quantize", "nvfp4_gemm_grouped", "nvfp4_w4a16_gemm",
                   "nvfp4_sync_check", "nvfp4_test_expire_next_wait"):
            getattr(L, fn).restype = ctypes.c_int
        L.nvfp4_status_string.argtypes = [ctypes.c_int]
        L.nvfp4_status_string.restype = ctypes.c_char_p
        L.nvfp4_last_error.argtypes = []
        L.nvfp4_last_error.restype = ctypes.c_char_p
        _lib = L
    return _lib


def _check(status: int, fn: str):
    if status != 0:
        raise NVFP4Error(status, fn, lib().nvfp4_last_error().decode())


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return F32
    if dt == torch.bfloat16:
        return BF16
    raise TypeError(f"unsupported dtype {dt} (float32 or bfloat16)")


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def codes_bytes(rows: int, cols: int) -> int:
    return int(lib().nvfp4_codes_bytes(rows, cols))


def scales_bytes(rows: int, cols: int) -> int:
    return int(lib().nvfp4_scales_bytes(rows, cols))


@dataclass
class NVFP4Tensor:
    """A quantized rows x cols tensor (K = cols) on the device.

    codes: uint8 [rows, cols/2]; scales: uint8 [scales_bytes] in the
    tensor-core 128x4 atom layout; global_scale, amax: float32 [1].
    """
    codes: torch.Tensor
    scales: torch.Tensor
    global_scale: torch.Tensor
    amax: torch.Tensor
    rows: int
    cols: int

    @staticmethod
    def empty(rows: int, cols: int, device="cuda") -> "NVFP4Tensor":
        return NVFP4Tensor(torch.empty((rows, cols // 2), dtype=torch.uint8, device=device),
                           torch.empty(max(scales_bytes(rows, cols), 1), dtype=torch.uint8, device=device),
                           torch.empty(1, dtype=torch.float32, device=device),
                           torch.empty(1, dtype=torch.float32, device=device), rows, cols)

    def clone(self) -> "NVFP4Tensor":
        return NVFP4Tensor(self.codes.clone(), self.scales.clone(), self.global_scale.clone(), self.amax.clone(),
                           self.rows, self.cols)

    def c(self) -> CTensor:
        return CTensor(self.codes.data_ptr(), self.scales.data_ptr(), self.global_scale.data_ptr(),
                       self.amax.data_ptr(), self.rows, self.cols)


def _config(block, rounding, scaling, transpose, seed, offset) -> CQuantConfig:
    b = {"1d": BLOCK_1D, "2d": BLOCK_2D}[block]
    r = {"rne": ROUND_RNE, "stochastic": ROUND_STOCHASTIC}[rounding]
    s = {"max6": SCALE_MAX6, "four_over_six": SCALE_FOUR_OVER_SIX}[scaling]
    return CQuantConfig(b, r, s, int(bool(transpose)), seed, offset)


def _prep_input(x: torch.Tensor):
    if x.dim() != 2:
        raise ValueError("x must be 2D")
    if x.stride(1) != 1:
        raise ValueError("x must have unit column stride")
    return x.shape[0], x.shape[1], x.stride(0)


def amax(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """nvfp4_amax: max |x| as a device float32 [1]."""
    rows, cols, ld = _prep_input(x)
    if out is None:
        out = torch.empty(1, dtype=torch.float32, device=x.device)
    _check(lib().nvfp4_amax(_ptr(x), _dtype_code(x.dtype), rows, cols, ld, _ptr(out), _stream(stream)), "nvfp4_amax")
    return out


def quantize(x: torch.Tensor, *, block="1d", rounding="rne", scaling="max6", transpose=False, seed=0, offset=0,
             amax: torch.Tensor | None = None, out: NVFP4Tensor | None = None, stream=None) -> NVFP4Tensor:
    """nvfp4_quantize.  The result is in the output orientation: x (K = cols)
    or x^T (transpose=True, K = rows)."""
    rows, cols, ld = _prep_input(x)
    R, K = (cols, rows) if transpose else (rows, cols)
    if out is None:
        out = NVFP4Tensor.empty(R, K, device=x.device)
    cfg = _config(block, rounding, scaling, transpose, seed, offset)
    ct = out.c()
    _check(lib().nvfp4_quantize(_ptr(x), _dtype_code(x.dtype), rows, cols, ld, ctypes.byref(cfg), _ptr(amax),
                                ctypes.byref(ct), _stream(stream)), "nvfp4_quantize")
    return out


def quantize_grouped(xs: list, *, block="1d", rounding="rne", scaling="max6", transpose=False, seed=0, offset=0,
                     out: list | None = None, stream=None) -> list:
    """nvfp4_quantize_grouped: every tensor of ``xs`` (same dtype) quantized
    with its own amax, one amax and one encode launch per 64 tensors; group
    e draws SR bits at offset + e."""
    n = len(xs)
    if n == 0:
        return []
    dims = [_prep_input(x) for x in xs]
    if out is None:
        out = [NVFP4Tensor.empty(c if transpose else r, r if transpose else c, device=xs[0].device)
               for (r, c, _) in dims]
    cfg = _config(block, rounding, scaling, transpose, seed, offset)
    X = (ctypes.c_void_p * n)(*[x.data_ptr() for x in xs])
    R = (ctypes.c_int64 * n)(*[d[0] for d in dims])
    C = (ctypes.c_int64 * n)(*[d[1] for d in dims])
    L = (ctypes.c_int64 * n)(*[d[2] for d in dims])
    O = (CTensor * n)(*[o.c() for o in out])
    _check(lib().nvfp4_quantize_grouped(n, X, _dtype_code(xs[0].dtype), R, C, L, ctypes.byref(cfg), O,
                                        _stream(stream)), "nvfp4_quantize_grouped")
    return out


def rht_quantize(x: torch.Tensor, *, rht_seed: int, rounding="rne", scaling="max6", transpose=True, seed=0,
                 offset=0, amax: torch.Tensor | None = None, out: NVFP4Tensor | None = None,
                 transformed_debug: bool = False, stream=None):
    """nvfp4_rht_quantize: 16x16 RHT along K, then 1D quantization.  Returns
    (NVFP4Tensor, transformed fp32 [R][K] or None)."""
    rows, cols, ld = _prep_input(x)
    R, K = (cols, rows) if transpose else (rows, cols)
    if out is None:
        out = NVFP4Tensor.empty(R, K, device=x.device)
    dbg = torch.empty((R, K), dtype=torch.float32, device=x.device) if transformed_debug else None
    cfg = _config("1d", rounding, scaling, transpose, seed, offset)
    ct = out.c()
    _check(lib().nvfp4_rht_quantize(_ptr(x), _dtype_code(x.dtype), rows, cols, ld, ctypes.byref(cfg), rht_seed,
                                    _ptr(amax), ctypes.byref(ct), _ptr(dbg), _stream(stream)), "nvfp4_rht_quantize")
    return out, dbg


def dequantize(q: NVFP4Tensor, dtype=torch.float32, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """nvfp4_dequantize: fp32 (or BF16) [rows, cols]."""
    if out is None:
        out = torch.empty((q.rows, q.cols), dtype=dtype, device=q.codes.device)
    ct = q.c()
    _check(lib().nvfp4_dequantize(ctypes.byref(ct), _ptr(out), _dtype_code(out.dtype), _stream(stream)),
           "nvfp4_dequantize")
    return out


def transpose_2d(q: NVFP4Tensor, out: NVFP4Tensor | None = None, stream=None) -> NVFP4Tensor:
    """nvfp4_transpose_2d: the NVFP4 tensor of x^T (cols x rows) from that of
    x quantized with 2D 16x16 blocks (the Dgrad operand W^T), by repacking."""
    if out is None:
        out = NVFP4Tensor.empty(q.cols, q.rows, device=q.codes.device)
    cq, co = q.c(), out.c()
    _check(lib().nvfp4_transpose_2d(ctypes.byref(cq), ctypes.byref(co), _stream(stream)), "nvfp4_transpose_2d")
    return out


def gemm(a: NVFP4Tensor, b: NVFP4Tensor, out_dtype=torch.bfloat16, out: torch.Tensor | None = None,
         stream=None) -> torch.Tensor:
    """nvfp4_gemm: D [M, N] = A (M x K) * B (N x K)^T with the block scales."""
    if out is None:
        out = torch.empty((a.rows, b.rows), dtype=out_dtype, device=a.codes.device)
    ca, cb = a.c(), b.c()
    _check(lib().nvfp4_gemm(ctypes.byref(ca), ctypes.byref(cb), _ptr(out), _dtype_code(out.dtype), out.stride(0),
                            _stream(stream)), "nvfp4_gemm")
    return out


def gemm_amax(a: NVFP4Tensor, b: NVFP4Tensor, out_dtype=torch.bfloat16, out: torch.Tensor | None = None,
              amax_out: torch.Tensor | None = None, stream=None):
    """nvfp4_gemm_amax: D as nvfp4_gemm plus max |D| (as stored) reduced in the
    GEMM epilogue.  Returns (D, amax float32 [1])."""
    if out is None:
        out = torch.empty((a.rows, b.rows), dtype=out_dtype, device=a.codes.device)
    if amax_out is None:
        amax_out = torch.empty(1, dtype=torch.float32, device=a.codes.device)
    ca, cb = a.c(), b.c()
    _check(lib().nvfp4_gemm_amax(ctypes.byref(ca), ctypes.byref(cb), _ptr(out), _dtype_code(out.dtype), out.stride(0),
                                 _ptr(amax_out), _stream(stream)), "nvfp4_gemm_amax")
    return out, amax_out


def gemm_quantize(a: NVFP4Tensor, b: NVFP4Tensor, amax_in: torch.Tensor, out: NVFP4Tensor | None = None,
                  d: torch.Tensor | None = None, amax_out: torch.Tensor | None = None, stream=None) -> NVFP4Tensor:
    """nvfp4_gemm_quantize: D = A * B^T rounded to BF16 and encoded in the GEMM
    epilogue as the M x N NVFP4 tensor ``out`` (1D blocks along N, RNE,
    max-6, tensor amax ``amax_in``).  ``d`` (BF16 [M, N] view, optional)
    also receives D; ``amax_out`` (optional) receives max |D|."""
    if out is None:
        out = NVFP4Tensor.empty(a.rows, b.rows, device=a.codes.device)
    if d is not None and (d.dtype != torch.bfloat16 or d.stride(1) != 1):
        raise ValueError("d must be BF16 with unit column stride")
    ca, cb, co = a.c(), b.c(), out.c()
    _check(lib().nvfp4_gemm_quantize(ctypes.byref(ca), ctypes.byref(cb), _ptr(amax_in), _ptr(d),
                                     d.stride(0) if d is not None else b.rows, _ptr(amax_out), ctypes.byref(co),
                                     _stream(stream)), "nvfp4_gemm_quantize")
    return out


def gemm_grouped(a: list, b: list, out_dtype=torch.bfloat16, out: list | None = None, stream=None) -> list:
    """nvfp4_gemm_grouped: D[e] = A[e] * B[e]^T for every group, one launch
    (per 64 groups)."""
    n = len(a)
    if len(b) != n:
        raise ValueError("a and b differ in length")
    if out is None:
        out = [torch.empty((a[e].rows, b[e].rows), dtype=out_dtype, device=a[e].codes.device) for e in range(n)]
    CA = (CTensor * max(n, 1))(*[x.c() for x in a])
    CB = (CTensor * max(n, 1))(*[x.c() for x in b])
    D = (ctypes.c_void_p * max(n, 1))(*[o.data_ptr() for o in out])
    _check(lib().nvfp4_gemm_grouped(n, CA, CB, D, _dtype_code(out_dtype), _stream(stream)), "nvfp4_gemm_grouped")
    return out


def w4a16_gemm(x: torch.Tensor, w: NVFP4Tensor, out_dtype=torch.bfloat16, out: torch.Tensor | None = None,
               stream=None) -> torch.Tensor:
    """nvfp4_w4a16_gemm: y [M, N] = x (BF16, M x K) * W_hat^T, W_hat the BF16
    dequantization of the NVFP4 weight w (N x K), FP32 accumulation."""
    if x.dtype != torch.bfloat16 or x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be a 2D BF16 tensor with unit column stride")
    if out is None:
        out = torch.empty((x.shape[0], w.rows), dtype=out_dtype, device=x.device)
    cw = w.c()
    _check(lib().nvfp4_w4a16_gemm(_ptr(x), BF16, x.shape[0], x.stride(0), ctypes.byref(cw), _ptr(out),
                                  _dtype_code(out.dtype), out.stride(0), _stream(stream)), "nvfp4_w4a16_gemm")
    return out


def sync_check(stream=None):
    """Synchronise the stream and raise on a pending CUDA error or a pipeline
    timeout (GEMM or transposed encoder)."""
    _check(lib().nvfp4_sync_check(_stream(stream)), "nvfp4_sync_check")


TEST_GEMM, TEST_TRANSPOSED_ENCODER = 1, 2


def test_expire_next_wait(op: int, limit_ns: int):
    """nvfp4_test_expire_next_wait: failure-detection test support.  The next
    launch of the plain GEMM (op 1) or of the TMA-fed transposed encoder
    (op 2) waits on a barrier that never completes, so its bounded wait runs
    out after limit_ns and the next sync_check raises NVFP4_ERR_TIMEOUT."""
    _check(lib().nvfp4_test_expire_next_wait(op, limit_ns), "nvfp4_test_expire_next_wait")
