"""Helpers of the GPU parity tests: guarded device buffers, oracle runs on the
same bytes, and element-wise comparisons."""
from __future__ import annotations

import numpy as np
import torch

import nvfp4_bit_block_02_b300 as nv
import oracle

GUARD = 256          # bytes of canary before and after every output buffer
CANARY = 0xA5


class Guarded:
    """A uint8 device buffer with canary bands; .view is the payload."""

    def __init__(self, nbytes: int, device="cuda"):
        self.n = nbytes
        self.raw = torch.full((nbytes + 2 * GUARD,), CANARY, dtype=torch.uint8, device=device)
        self.view = self.raw[GUARD:GUARD + nbytes]

    def check(self):
        raw = self.raw.cpu().numpy()
        assert (raw[:GUARD] == CANARY).all(), "write before the buffer"
        assert (raw[GUARD + self.n:] == CANARY).all(), "write past the buffer"


def guarded_tensor(R: int, K: int):
    """An NVFP4Tensor whose codes, scales and scalars sit inside canary bands."""
    bufs = [Guarded(max(R * K // 2, 1)), Guarded(max(nv.scales_bytes(R, K), 1)), Guarded(4), Guarded(4)]
    t = nv.NVFP4Tensor(bufs[0].view[:R * K // 2].view(R, K // 2) if R * K else bufs[0].view[:0].view(R, K // 2),
                       bufs[1].view, bufs[2].view.view(torch.float32), bufs[3].view.view(torch.float32), R, K)
    return t, bufs


def to_numpy_f32(x: torch.Tensor) -> np.ndarray:
    """Exact fp32 values of a CPU bf16/f32 tensor."""
    return x.to(torch.float32).numpy()


def oracle_quantize_like(x_cpu: torch.Tensor, **kw) -> oracle.Quantized:
    return oracle.quantize(to_numpy_f32(x_cpu), **kw)


def assert_same_quantized(q: nv.NVFP4Tensor, ref: oracle.Quantized, what=""):
    codes = q.codes.cpu().numpy()
    scales = q.scales.cpu().numpy()
    amax = float(q.amax.cpu()[0])
    g = float(q.global_scale.cpu()[0])
    assert amax == ref.amax, f"{what}: amax {amax} != {ref.amax}"
    assert g == ref.g, f"{what}: g {g} != {ref.g}"
    phys = ref.physical_scales()
    if scales.size != phys.size:
        raise AssertionError(f"{what}: scale buffer size {scales.size} != {phys.size}")
    bad_s = np.nonzero(scales != phys)[0]
    assert bad_s.size == 0, f"{what}: {bad_s.size} scale bytes differ, first at {bad_s[:8]}"
    bad = np.argwhere(codes != ref.codes)
    assert bad.size == 0, (f"{what}: {len(bad)} code bytes differ, first {bad[:4].tolist()} "
                           f"gpu {codes[tuple(bad[0])]:#x} oracle {ref.codes[tuple(bad[0])]:#x}")


def unpack_codes(codes: np.ndarray) -> np.ndarray:
    out = np.empty((codes.shape[0], codes.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = codes & 15
    out[:, 1::2] = codes >> 4
    return out


def gemm_check(d_gpu: np.ndarray, d_ref: np.ndarray, bound: np.ndarray, bf16: bool, what=""):
    """|D - D_ref| <= 1e-5 * sum|a||b| (+ half a BF16 ulp of D_ref for BF16
    output, whose rounding alone exceeds the first term)."""
    tol = 1e-5 * bound
    if bf16:
        mag = np.abs(d_ref)
        e = np.floor(np.log2(np.where(mag > 0, mag, 1.0)))
        tol = tol + np.where(mag > 0, 2.0 ** (e - 8), 0.0)   # half ulp of an 8-bit significand
    err = np.abs(d_gpu.astype(np.float64) - d_ref)
    bad = np.argwhere(err > tol)
    assert bad.size == 0, (f"{what}: {len(bad)} outputs out of tolerance; first {bad[:3].tolist()} "
                           f"gpu {d_gpu[tuple(bad[0])]} ref {d_ref[tuple(bad[0])]} tol {tol[tuple(bad[0])]}")
    return float((err / np.maximum(bound, 1e-300)).max())
