"""nvfp4_amax on the GPU (the tensor amax alone, the input of the sharded
path) against the exact max |x|, and the single-process sharded quantize."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import nvfp4_bit_block_02_b300 as nv
from nvfp4_bit_block_02_b300.distributed import quantize_sharded

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("R,C,pad", [(1, 16, 0), (37, 64, 8), (1000, 4096, 0), (8192, 4096, 0), (3, 1024, 64)])
def test_amax_is_the_exact_max(dtype, R, C, pad):
    rng = np.random.default_rng(R + C)
    base = torch.from_numpy(rng.standard_normal((R, C + pad)).astype(np.float32)).to(dtype)
    base[R // 2, C // 3] = -1234.5 if dtype == torch.float32 else -1232.0
    base[0, C + pad - 1] = 1e6  # in the padding when pad > 0: must be ignored
    x = base.cuda()[:, :C]
    got = float(nv.amax(x).cpu()[0])
    want = float(base[:, :C].float().abs().max())
    assert got == want


def test_amax_empty_is_zero():
    assert float(nv.amax(torch.zeros((0, 64), device="cuda")).cpu()[0]) == 0.0


def test_sharded_quantize_on_one_process_equals_quantize():
    x = torch.randn(256, 512, device="cuda", dtype=torch.bfloat16)
    a = quantize_sharded(x, block="2d")
    b = nv.quantize(x, block="2d")
    nv.sync_check()
    assert torch.equal(a.codes, b.codes) and torch.equal(a.scales, b.scales) and torch.equal(a.amax, b.amax)
