"""nvfp4_gemm_amax: the GEMM output unchanged, the amax reduced in its
epilogue equal to max |D| as stored, and the next quantization driven by it
equal to the one that reduces the amax itself."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import nvfp4_bit_block_02_b300 as nv
import synthetic

pytestmark = pytest.mark.gpu


def _operands(M, N, K, seed):
    rng = np.random.default_rng(seed)
    x = torch.from_numpy(synthetic.with_entry_outliers(rng.standard_normal((M, K)).astype(np.float32), 0.01, 30.0,
                                                       seed)).to(torch.bfloat16).cuda()
    w = torch.from_numpy((0.05 * rng.standard_normal((N, K))).astype(np.float32)).to(torch.bfloat16).cuda()
    # 2D weight blocks need whole 16-row groups; other N take 1D blocks
    return nv.quantize(x), nv.quantize(w, block="2d" if N % 16 == 0 else "1d")


@pytest.mark.parametrize("M,N,K", [(128, 128, 256), (384, 640, 512), (1024, 768, 1024), (256, 384, 2048)])
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_gemm_amax_matches(M, N, K, dt):
    qa, qb = _operands(M, N, K, M + N + K)
    d_ref = nv.gemm(qa, qb, out_dtype=dt)
    d, am = nv.gemm_amax(qa, qb, out_dtype=dt)
    nv.sync_check()
    assert torch.equal(d, d_ref)
    assert float(am.cpu()[0]) == float(d.float().abs().max().cpu())
    if dt == torch.bfloat16:
        q1 = nv.quantize(d, amax=am)
        q2 = nv.quantize(d)
        nv.sync_check()
        assert torch.equal(q1.codes, q2.codes) and torch.equal(q1.scales, q2.scales)
        assert torch.equal(q1.amax, q2.amax) and torch.equal(q1.global_scale, q2.global_scale)


def test_gemm_amax_llama8b_full_size():
    wl = synthetic.llama8b_fprop()
    qx = nv.quantize(wl.tensors["X"].cuda())
    qw = nv.quantize(wl.tensors["W"].cuda(), block="2d")
    d, am = nv.gemm_amax(qx, qw)
    ref = nv.gemm(qx, qw)
    nv.sync_check()
    assert torch.equal(d, ref)
    assert float(am.cpu()[0]) == float(d.float().abs().max().cpu())


@pytest.mark.parametrize("M,N,K", [(200, 130, 320), (77, 100, 64), (300, 200, 192), (129, 257, 128)])
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_gemm_amax_ragged(M, N, K, dt):
    """N not a multiple of 128 (an epilogue warp holds fewer than 128 valid
    columns) nor, for some, of a 16-byte unit (the row's last partial unit
    goes through plain stores): the amax covers exactly the stored outputs and
    nothing is written past them."""
    qa, qb = _operands(M, N, K, 7 * M + N + K)
    per16 = 16 // (2 if dt == torch.bfloat16 else 4)
    ld = -(-N // per16) * per16
    big_ref = torch.full((M + 1, ld + per16), -7.0, dtype=dt, device="cuda")
    big = big_ref.clone()
    nv.gemm(qa, qb, out=big_ref[:M, :N])
    _, am = nv.gemm_amax(qa, qb, out=big[:M, :N])
    nv.sync_check()
    assert torch.equal(big, big_ref)  # D identical, padding and the extra row untouched
    assert float(am.cpu()[0]) == float(big[:M, :N].float().abs().max().cpu())
