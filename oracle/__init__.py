"""Plain CPU oracle for the NVFP4 quantizer and block-scaled GEMM.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg import this package; the product path never does.
It shares no code with the CUDA library: the element/scale arithmetic lives in
``nvfp4_oracle.c`` (plain C, ``-O2 -ffp-contract=off``), the GEMM reference is
the definition written with numpy in float64.

What each function follows is stated in its docstring.  The pages behind the
method: "NVIDIA Introduces a 4-Bit Pretraining Methodology Using NVFP4"
("Summary": 16-element blocks, E4M3 block scales, FP32 per-tensor scale;
"Method": 2D 16x16 weight scaling, 16x16 RHT on Wgrad inputs, stochastic
rounding on gradients), the hyper.ai story "NVIDIA présente NVFP4" (two-level
micro-scaling, RHT against outliers, unbiased SR) and the hyper.ai story on
the Nemotron 3 Ultra NVFP4 checkpoint (Four-over-Six, W4A4 on Blackwell).

Parity unpinned: none.  Philox is pinned against an independent library
implementation (Triton's, run by its CPU interpreter) in the tests.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
                        -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0], dtype=np.float64)


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/liboracle.so`` (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-shared", "-fPIC",
               "-std=c11", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        U64 = ctypes.c_uint64
        lib.oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e2m1_decode.restype = ctypes.c_float
        lib.oracle_e2m1_encode_rne.argtypes = [ctypes.c_float]
        lib.oracle_e2m1_encode_rne.restype = ctypes.c_uint8
        lib.oracle_e2m1_encode_sr.argtypes = [ctypes.c_float, ctypes.c_uint32]
        lib.oracle_e2m1_encode_sr.restype = ctypes.c_uint8
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = ctypes.c_float
        lib.oracle_e4m3_encode_rne_sat.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode_rne_sat.restype = ctypes.c_uint8
        lib.oracle_philox4x32_10.argtypes = [P, P, P]
        lib.oracle_philox4x32_10.restype = None
        lib.oracle_sr_bits.argtypes = [U64, U64, U64]
        lib.oracle_sr_bits.restype = ctypes.c_uint32
        lib.oracle_rht_signs.argtypes = [U64, P]
        lib.oracle_rht_signs.restype = None
        lib.oracle_hadamard16.argtypes = [ctypes.c_int, ctypes.c_int]
        lib.oracle_hadamard16.restype = ctypes.c_int
        lib.oracle_rht16.argtypes = [P, P, P]
        lib.oracle_rht16.restype = None
        lib.oracle_quantize.argtypes = [P, I64, I64, I64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, U64, U64, U64, P, P, P, P, P, P, P]
        lib.oracle_quantize.restype = ctypes.c_int
        lib.oracle_dequantize.argtypes = [P, P, ctypes.c_float, I64, I64, P]
        lib.oracle_dequantize.restype = None
        lib.oracle_scales_bytes.argtypes = [I64, I64]
        lib.oracle_scales_bytes.restype = I64
        lib.oracle_swizzle_scales.argtypes = [P, I64, I64, P]
        lib.oracle_swizzle_scales.restype = None
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


# --------------------------------------------------------------------------
# element formats
# --------------------------------------------------------------------------
def e2m1_decode(code: int) -> float:
    return float(_load().oracle_e2m1_decode(code))


def e2m1_encode_rne(q: float) -> int:
    return int(_load().oracle_e2m1_encode_rne(q))


def e2m1_encode_sr(q: float, u16: int) -> int:
    return int(_load().oracle_e2m1_encode_sr(q, u16))


def e4m3_decode(b: int) -> float:
    return float(_load().oracle_e4m3_decode(b))


def e4m3_encode(t: float) -> int:
    return int(_load().oracle_e4m3_encode_rne_sat(t))


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact BF16 -> FP32 upcast of raw uint16 BF16 bit patterns."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------
# Philox and the random streams
# --------------------------------------------------------------------------
def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.asarray(ctr, dtype=np.uint32).copy()
    k = np.asarray(key, dtype=np.uint32).copy()
    out = np.zeros(4, dtype=np.uint32)
    _load().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def sr_bits(seed: int, offset: int, i: int) -> int:
    return int(_load().oracle_sr_bits(seed, offset, i))


def rht_signs(rht_seed: int) -> np.ndarray:
    out = np.zeros(16, dtype=np.int32)
    _load().oracle_rht_signs(rht_seed, _ptr(out))
    return out


def hadamard16() -> np.ndarray:
    lib = _load()
    return np.array([[lib.oracle_hadamard16(i, j) for j in range(16)] for i in range(16)], dtype=np.int64)


def rht16(x: np.ndarray, sigma: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    s = np.ascontiguousarray(sigma, dtype=np.int32)
    y = np.zeros(16, dtype=np.float32)
    _load().oracle_rht16(_ptr(x), _ptr(s), _ptr(y))
    return y


# --------------------------------------------------------------------------
# quantize / dequantize / scale layout
# --------------------------------------------------------------------------
class Quantized:
    """Oracle result in the output orientation R x K.

    codes: uint8 [R][K/2]; scales: logical uint8 [R][K/16] (E4M3 bytes);
    amax, g: floats; choice: uint8 [R][K/16] (1 = max-4 won) or None;
    transformed: fp32 [R][K] values that were encoded (after the RHT) or None.
    """

    def __init__(self, codes, scales, amax, g, choice, transformed, R, K):
        self.codes, self.scales, self.amax, self.g = codes, scales, amax, g
        self.choice, self.transformed, self.R, self.K = choice, transformed, R, K

    def physical_scales(self) -> np.ndarray:
        return swizzle_scales(self.scales, self.R, self.K)


def quantize(x: np.ndarray, *, transpose=False, block2d=False, stochastic=False, four_over_six=False,
             rht=False, seed=0, offset=0, rht_seed=0, amax=None, want_choice=False,
             want_transformed=False) -> Quantized:
    """Quantize a 2D array (fp32 values; pass BF16 through ``bf16_bits_to_f32``).

    Follows ``oracle_quantize`` in nvfp4_oracle.c step by step.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, cols = x.shape
    R, K = (cols, rows) if transpose else (rows, cols)
    codes = np.zeros((R, K // 2), dtype=np.uint8)
    scales = np.zeros((R, K // 16), dtype=np.uint8)
    choice = np.zeros((R, K // 16), dtype=np.uint8) if want_choice else None
    transformed = np.zeros((R, K), dtype=np.float32) if want_transformed else None
    amax_out = np.zeros(1, dtype=np.float32)
    g_out = np.zeros(1, dtype=np.float32)
    amax_in = None if amax is None else np.array([amax], dtype=np.float32)
    rc = _load().oracle_quantize(_ptr(x), rows, cols, cols, int(transpose), int(block2d), int(stochastic),
                                 int(four_over_six), int(rht), seed, offset, rht_seed, _ptr(amax_in),
                                 _ptr(codes), _ptr(scales), _ptr(amax_out), _ptr(g_out), _ptr(choice),
                                 _ptr(transformed))
    if rc != 0:
        raise ValueError(f"oracle_quantize rejected shape {x.shape} (transpose={transpose}, 2d={block2d})")
    return Quantized(codes, scales, float(amax_out[0]), float(g_out[0]), choice, transformed, R, K)


def dequantize(codes: np.ndarray, scales: np.ndarray, g: float) -> np.ndarray:
    """y = fl(fl(value(code) * s_b) * g), fp32 [R][K] from logical scales."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    R, K2 = codes.shape
    y = np.zeros((R, 2 * K2), dtype=np.float32)
    _load().oracle_dequantize(_ptr(codes), _ptr(scales), g, R, 2 * K2, _ptr(y))
    return y


def scales_bytes(R: int, K: int) -> int:
    return int(_load().oracle_scales_bytes(R, K))


def swizzle_scales(logical: np.ndarray, R: int, K: int) -> np.ndarray:
    logical = np.ascontiguousarray(logical, dtype=np.uint8)
    out = np.zeros(scales_bytes(R, K), dtype=np.uint8)
    _load().oracle_swizzle_scales(_ptr(logical), R, K, _ptr(out))
    return out


# --------------------------------------------------------------------------
# GEMM reference (definition in float64)
# --------------------------------------------------------------------------
def exact_values(codes: np.ndarray, scales: np.ndarray, g: float) -> np.ndarray:
    """Exact real value of every element, code * s_b * g, in float64 (exact:
    at most 6 + 24 significant bits)."""
    R, K2 = codes.shape
    K = 2 * K2
    lo = codes & 0x0F
    hi = codes >> 4
    c = np.empty((R, K), dtype=np.uint8)
    c[:, 0::2] = lo
    c[:, 1::2] = hi
    e4 = np.array([e4m3_decode(b) if (b & 0x7F) != 0x7F else 0.0 for b in range(256)], dtype=np.float64)
    s = np.repeat(e4[scales], 16, axis=1)
    return E2M1_VALUES[c] * s * np.float64(g)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """fp32 -> nearest BF16 value (ties to even), returned as fp32: keep the
    top 16 bits after adding 0x7FFF plus the lowest kept bit (finite inputs)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000).astype(np.uint32)
    return r.view(np.float32)


def w4a16_reference(x: np.ndarray, qw: Quantized, rows=None):
    """Y = X @ W_hat^T in float64 and the bound sum_k |x||w_hat|: the weight-only
    path, where the NVFP4 weight enters a BF16 GEMM as W_hat = BF16(decode),
    decode = fl(fl(value(code) * s_b) * g) (``dequantize``), rounded to the
    nearest BF16 (ties to even).  ``x``: the fp32 values of the BF16
    activations, M x K; ``qw``: N x K."""
    w = bf16_round(dequantize(qw.codes, qw.scales, qw.g)).astype(np.float64)
    a = np.asarray(x if rows is None else x[rows], dtype=np.float64)
    return a @ w.T, np.abs(a) @ np.abs(w).T


def gemm_reference(qa: Quantized, qb: Quantized, rows=None):
    """D = A_deq @ B_deq^T in float64 and the bound sum_k |a||b|.

    A is M x K, B is N x K (both in the quantizer's output orientation).  The
    NVFP4 GEMM is defined as the product of the dequantized operands; the
    matmul is the library primitive for the sum over k.  ``rows`` restricts
    the reference to a subset of output rows.
    """
    a = exact_values(qa.codes if rows is None else qa.codes[rows],
                     qa.scales if rows is None else qa.scales[rows], qa.g)
    b = exact_values(qb.codes, qb.scales, qb.g)
    return a @ b.T, np.abs(a) @ np.abs(b).T
