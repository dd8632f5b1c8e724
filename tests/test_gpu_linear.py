"""The NVFP4 linear layer (autograd Function) against the oracle composed
step by step: fprop, dgrad and wgrad outputs element by element."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synthetic
from nvfp4_bit_block_02_b300.linear import NVFP4Linear, NVFP4LinearFunction
from tests.gpu_helpers import gemm_check, to_numpy_f32


def _oq(t: torch.Tensor, **kw):
    return oracle.quantize(to_numpy_f32(t), **kw)


@pytest.mark.gpu
@pytest.mark.parametrize("T,n_in,n_out", [(256, 256, 256), (512, 768, 512), (192, 320, 448)])
def test_linear_forward_backward_matches_oracle(T, n_in, n_out):
    rng = np.random.default_rng(T + n_in + n_out)
    x = torch.from_numpy(synthetic.with_channel_outliers(rng.standard_normal((T, n_in)).astype(np.float32), 0.01,
                                                         20.0, 7)).to(torch.bfloat16)
    w = torch.from_numpy((0.02 * rng.standard_normal((n_out, n_in))).astype(np.float32)).to(torch.bfloat16)
    dy = torch.from_numpy(synthetic.student_t((T, n_out), 4, 1e-3, 8)).to(torch.bfloat16)
    seed, offset, rht_seed = 17, 5, 3
    xg = x.cuda().requires_grad_(True)
    wg = w.cuda().requires_grad_(True)
    y = NVFP4LinearFunction.apply(xg, wg, seed, offset, rht_seed)
    y.backward(dy.cuda())
    torch.cuda.synchronize()
    all_rows = np.arange(T)
    # fprop: X 1D RNE, W 2D RNE
    ref, bound = oracle.gemm_reference(_oq(x), _oq(w, block2d=True), rows=all_rows)
    gemm_check(y.detach().float().cpu().numpy(), ref, bound, True, "fprop")
    # dgrad: dY 1D SR (offset 2*offset), W^T 2D
    ref, bound = oracle.gemm_reference(_oq(dy, stochastic=True, seed=seed, offset=2 * offset),
                                       _oq(w.t().contiguous(), block2d=True), rows=all_rows)
    gemm_check(xg.grad.float().cpu().numpy(), ref, bound, True, "dgrad")
    # wgrad: dY^T with RHT + SR (offset 2*offset+1), X^T with RHT, same sign vector
    ref, bound = oracle.gemm_reference(
        _oq(dy, transpose=True, rht=True, stochastic=True, seed=seed, offset=2 * offset + 1, rht_seed=rht_seed),
        _oq(x, transpose=True, rht=True, rht_seed=rht_seed), rows=np.arange(n_out))
    gemm_check(wg.grad.float().cpu().numpy(), ref, bound, True, "wgrad")


@pytest.mark.gpu
def test_linear_module_bf16_opt_out_and_stream_positions():
    torch.manual_seed(0)
    layer = NVFP4Linear(256, 256, device="cuda", seed=4)
    x = torch.randn(256, 256, device="cuda", dtype=torch.bfloat16)
    dy = torch.randn(256, 256, device="cuda", dtype=torch.bfloat16) * 1e-3   # not on the grid: SR draws matter
    layer(x).backward(dy)
    g1 = layer.weight.grad.clone()
    layer.weight.grad = None
    layer(x).backward(dy)
    # the second call draws from the next stream position: different rounding
    assert layer.calls == 2 and not torch.equal(g1, layer.weight.grad)
    layer.enabled = False
    y = layer(x)
    assert torch.equal(y, x @ layer.weight.t())


def test_linear_shape_rule_is_checked_on_the_host():
    x = torch.zeros(200, 256)
    w = torch.zeros(256, 256)
    with pytest.raises(ValueError, match="tokens"):
        NVFP4LinearFunction.apply(x, w, 0, 0, 1)
