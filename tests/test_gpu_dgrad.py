"""Dgrad path on the GPU: the repacked weight transpose (nvfp4_transpose_2d)
against the oracle, and dX = dY W through the block-scaled GEMM."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import nvfp4_bit_block_02_b300 as nv
import oracle
import synthetic
from tests.gpu_helpers import assert_same_quantized, gemm_check, guarded_tensor, oracle_quantize_like

pytestmark = pytest.mark.gpu


def _transpose_codes(codes: np.ndarray) -> np.ndarray:
    """Nibble-level transpose of packed codes [R][K/2] -> [K][R/2]."""
    full = np.empty((codes.shape[0], codes.shape[1] * 2), dtype=np.uint8)
    full[:, 0::2] = codes & 15
    full[:, 1::2] = codes >> 4
    t = full.T
    return (t[:, 0::2] | (t[:, 1::2] << 4)).astype(np.uint8)


@pytest.mark.parametrize("R,K", [(16, 16), (64, 128), (208, 336), (256, 512), (1040, 784)])
@pytest.mark.parametrize("scaling", ["max6", "four_over_six"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_transpose_2d_equals_quantizing_the_transpose(R, K, scaling, dtype):
    """RNE: repacking W's 2D quantization gives, bit for bit, the oracle's
    2D quantization of W^T, and the GPU's own transposed quantization."""
    rng = np.random.default_rng(R * 7 + K)
    x = torch.from_numpy(synthetic.with_entry_outliers(rng.standard_normal((R, K)).astype(np.float32), 0.01, 30.0,
                                                       R + K)).to(dtype)
    q = nv.quantize(x.cuda(), block="2d", scaling=scaling)
    qt, bufs = guarded_tensor(K, R)
    nv.transpose_2d(q, out=qt)
    direct = nv.quantize(x.cuda(), block="2d", scaling=scaling, transpose=True)
    nv.sync_check()
    for b in bufs:
        b.check()
    ref = oracle_quantize_like(x.t().contiguous(), block2d=True, four_over_six=scaling == "four_over_six")
    assert_same_quantized(qt, ref, f"transpose_2d {R}x{K} {scaling}")
    assert torch.equal(qt.codes, direct.codes)
    assert torch.equal(qt.scales, direct.scales)


def test_transpose_2d_keeps_stochastic_codes():
    """SR: the repack carries the codes drawn for W itself (the same quantized
    weight in both passes), i.e. the nibble transpose of W's codes."""
    rng = np.random.default_rng(5)
    R, K = 192, 320
    x = torch.from_numpy(rng.standard_normal((R, K)).astype(np.float32))
    q = nv.quantize(x.cuda(), block="2d", rounding="stochastic", seed=9, offset=3)
    qt = nv.transpose_2d(q)
    nv.sync_check()
    ref = oracle_quantize_like(x, block2d=True, stochastic=True, seed=9, offset=3)
    assert_same_quantized(q, ref, "W 2D SR")
    assert (qt.codes.cpu().numpy() == _transpose_codes(ref.codes)).all()
    # logical scales of W^T: entry (k, rb) is the scale of tile (rb, k / 16)
    tref = oracle.Quantized(_transpose_codes(ref.codes), np.repeat(ref.scales[::16, :].T, 16, axis=0), ref.amax,
                            ref.g, None, None, K, R)
    assert (qt.scales.cpu().numpy() == tref.physical_scales()).all()
    assert float(qt.amax.cpu()[0]) == ref.amax and float(qt.global_scale.cpu()[0]) == ref.g


def test_transpose_2d_empty():
    q = nv.quantize(torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda"), block="2d")
    qt = nv.transpose_2d(q)
    nv.sync_check()
    assert qt.rows == 64 and qt.cols == 0
    assert float(qt.amax.cpu()[0]) == 0.0 and float(qt.global_scale.cpu()[0]) == 1.0


def _dgrad_reference(dy_cpu, w_cpu, rows, seed):
    rd = oracle_quantize_like(dy_cpu, stochastic=True, seed=seed)
    rwt = oracle_quantize_like(w_cpu.t().contiguous(), block2d=True)
    return rd, rwt, oracle.gemm_reference(rd, rwt, rows=rows)


def test_dgrad_small():
    """dX [M][Kin] = dY [M][N] W [N][Kin]: dY 1D with SR, W 2D repacked."""
    rng = np.random.default_rng(11)
    M, N, Kin = 256, 512, 384
    dy = torch.from_numpy(synthetic.student_t((M, N), 4, 1e-3, 21)).to(torch.bfloat16)
    w = torch.from_numpy((0.02 * rng.standard_normal((N, Kin))).astype(np.float32)).to(torch.bfloat16)
    qd = nv.quantize(dy.cuda(), rounding="stochastic", seed=4)
    qwt = nv.transpose_2d(nv.quantize(w.cuda(), block="2d"))
    dx = nv.gemm(qd, qwt, out_dtype=torch.float32)
    nv.sync_check()
    rows = np.arange(M)
    rd, rwt, (ref, bound) = _dgrad_reference(dy, w, rows, 4)
    assert_same_quantized(qd, rd, "dY SR")
    assert_same_quantized(qwt, rwt, "W^T")
    gemm_check(dx.cpu().numpy(), ref, bound, False, "dgrad small")


def test_dgrad_llama8b_full_size_sampled():
    """Llama-3-8B MLP dgrad: dY 8192x14336 (1e-3 t(4), SR), W 14336x4096 (2D):
    dX 8192x4096 BF16, sampled rows against the oracle."""
    dy = synthetic.wgrad().tensors["dY"]
    w = synthetic.llama8b_fprop().tensors["W"]
    qd = nv.quantize(dy.cuda(), rounding="stochastic", seed=1)
    qwt = nv.transpose_2d(nv.quantize(w.cuda(), block="2d"))
    dx = nv.gemm(qd, qwt, out_dtype=torch.bfloat16)
    nv.sync_check()
    rng = np.random.default_rng(3)
    rows = np.concatenate([np.arange(0, 64), rng.choice(8192, 64, replace=False)])
    rd, rwt, (ref, bound) = _dgrad_reference(dy, w, rows, 1)
    assert (qwt.codes.cpu().numpy() == rwt.codes).all()
    gemm_check(dx[rows].float().cpu().numpy(), ref, bound, True, "8B dgrad")
