"""nvfp4_quantize_grouped on the GPU: every group bit-exact with the
single-tensor call (same config, SR offset + e) and, for a sample of groups,
with the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import nvfp4_bit_block_02_b300 as nv
import synthetic
from tests.gpu_helpers import assert_same_quantized, oracle_quantize_like

pytestmark = pytest.mark.gpu


def _same(a: nv.NVFP4Tensor, b: nv.NVFP4Tensor, what: str):
    assert torch.equal(a.codes, b.codes), f"{what}: codes"
    assert torch.equal(a.scales, b.scales), f"{what}: scales"
    assert torch.equal(a.amax, b.amax) and torch.equal(a.global_scale, b.global_scale), f"{what}: scalars"


def _tensors(n, rng, dtype, transpose, b2d):
    xs = []
    for e in range(n):
        r = int(rng.choice([16, 48, 128, 272])) if (b2d or transpose) else int(rng.choice([1, 37, 128, 300]))
        c = int(rng.choice([16, 64, 208, 512]))
        scale = float(10.0 ** rng.uniform(-3, 2))
        x = synthetic.with_entry_outliers((scale * rng.standard_normal((r, c))).astype(np.float32), 0.01, 20.0, e)
        xs.append(torch.from_numpy(x).to(dtype))
    return xs


@pytest.mark.parametrize("count", [1, 3, 70])
@pytest.mark.parametrize("mode", ["1d", "2d", "1d_sr", "t_46", "t_sr_46", "2d_t"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_grouped_equals_single_calls(count, mode, dtype):
    rng = np.random.default_rng(count * 31 + len(mode))
    b2d = mode.startswith("2d")
    transpose = "t" in mode.split("_")[1:] or mode.startswith("t_")
    kw = dict(block="2d" if b2d else "1d", rounding="stochastic" if "sr" in mode else "rne",
              scaling="four_over_six" if "46" in mode else "max6", transpose=transpose, seed=5, offset=100)
    xs = [x.cuda() for x in _tensors(count, rng, dtype, transpose, b2d)]
    qs = nv.quantize_grouped(xs, **kw)
    nv.sync_check()
    for e, x in enumerate(xs):
        single = nv.quantize(x, **{**kw, "offset": kw["offset"] + e})
        _same(qs[e], single, f"group {e}")
    for e in sorted({0, count - 1}):
        ref = oracle_quantize_like(xs[e].cpu(), transpose=transpose, block2d=b2d, stochastic="sr" in mode,
                                   four_over_six="46" in mode, seed=5, offset=100 + e)
        assert_same_quantized(qs[e], ref, f"group {e} vs oracle")


@pytest.mark.parametrize("mode", ["1d", "t_46"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_grouped_row_strided_inputs(mode, dtype):
    """Groups given as column slices of wider buffers (row stride > cols): the
    amax pass walks such tiles row by row; every group bit-exact with the
    single call on the same view and, for two groups, with the oracle."""
    rng = np.random.default_rng(77 + len(mode))
    transpose = mode.startswith("t_")
    kw = dict(transpose=transpose, scaling="four_over_six" if "46" in mode else "max6", seed=3, offset=7)
    views = []
    for x in _tensors(9, rng, dtype, transpose, False):
        r, c = x.shape
        wide = torch.full((r, c + 64), 1e4, dtype=dtype)  # the columns past c must be ignored
        wide[:, :c] = x
        views.append(wide.cuda()[:, :c])
    assert all(v.stride(0) == v.shape[1] + 64 for v in views)
    qs = nv.quantize_grouped(views, **kw)
    nv.sync_check()
    for e, v in enumerate(views):
        _same(qs[e], nv.quantize(v, **{**kw, "offset": kw["offset"] + e}), f"group {e}")
    for e in (0, len(views) - 1):
        ref = oracle_quantize_like(views[e].cpu().contiguous(), transpose=transpose,
                                   four_over_six="46" in mode, seed=3, offset=7 + e)
        assert_same_quantized(qs[e], ref, f"group {e} vs oracle")


def test_grouped_with_empty_groups():
    xs = [torch.randn(64, 64, device="cuda"), torch.zeros((0, 64), device="cuda"), torch.randn(32, 128, device="cuda")]
    qs = nv.quantize_grouped(xs)
    nv.sync_check()
    _same(qs[0], nv.quantize(xs[0]), "group 0")
    _same(qs[2], nv.quantize(xs[2], offset=2), "group 2")
    assert float(qs[1].amax.cpu()[0]) == 0.0 and float(qs[1].global_scale.cpu()[0]) == 1.0


def test_grouped_moe_expert_weights_full_size():
    """The MoE workload: 64 expert weights W_e^T (1536 x 4096), Four-over-Six;
    every group against the single call, every 16th against the oracle."""
    W = synthetic.moe().tensors["W"]
    ws = [W[e].cuda() for e in range(W.shape[0])]
    qs = nv.quantize_grouped(ws, transpose=True, scaling="four_over_six")
    nv.sync_check()
    for e in range(len(ws)):
        _same(qs[e], nv.quantize(ws[e], transpose=True, scaling="four_over_six", offset=e), f"expert {e}")
    for e in range(0, len(ws), 16):
        ref = oracle_quantize_like(W[e], transpose=True, four_over_six=True)
        assert_same_quantized(qs[e], ref, f"expert {e} vs oracle")
