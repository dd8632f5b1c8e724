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
    return nv.quantize(x), nv.quantize(w, block="2d")


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
