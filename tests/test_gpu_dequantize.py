"""Dequantizer parity on the GPU: fp32 output bit-exact with the oracle's
y = fl(fl(value(code) * s_b) * g); BF16 output = that fp32 value rounded to
nearest even."""
import numpy as np
import pytest
import torch

import nvfp4_bit_block_02_b300 as nv
import oracle
import synthetic
from tests.gpu_helpers import oracle_quantize_like

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape", [(256, 256), (130, 80), (1, 16), (384, 1040)])
@pytest.mark.parametrize("block", ["1d", "2d"])
def test_dequantize_parity(shape, block):
    rows, cols = shape
    if block == "2d" and rows % 16:
        pytest.skip("2D needs rows % 16")
    x = torch.from_numpy(synthetic.with_entry_outliers(synthetic.normal(shape, 1.0, 50), 0.01, 50, 51))
    q = nv.quantize(x.cuda(), block=block, scaling="four_over_six")
    y32 = nv.dequantize(q, torch.float32)
    y16 = nv.dequantize(q, torch.bfloat16)
    nv.sync_check()
    ref = oracle_quantize_like(x, block2d=block == "2d", four_over_six=True)
    yr = oracle.dequantize(ref.codes, ref.scales, ref.g)
    got = y32.cpu().numpy()
    assert (got.view(np.uint32) == yr.view(np.uint32)).all()
    assert torch.equal(y16.cpu(), torch.from_numpy(yr).to(torch.bfloat16))


def test_dequantize_round_trip_of_grid_values():
    """Values exactly on the grid of their block come back unchanged."""
    rng = np.random.default_rng(7)
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6], np.float32)
    v = rng.choice(grid, size=(64, 256)) * rng.choice([-1, 1], size=(64, 256))
    v[:, ::16] = 6.0
    v[0, 1] = 2688.0 / 448 * 6 / 6   # keep amax = 6: g = 6/2688, S_b = 448 g = 1 in every block
    x = torch.from_numpy(v.astype(np.float32))
    q = nv.quantize(x.cuda())
    y = nv.dequantize(q)
    nv.sync_check()
    ref = oracle_quantize_like(x)
    assert (y.cpu().numpy() == oracle.dequantize(ref.codes, ref.scales, ref.g)).all()


def test_dequantize_llama8b_weight_sampled():
    """The Llama-3-8B MLP weight (14336 x 4096, 2D blocks) decoded to BF16 in
    full on the GPU; sampled rows bit-exact with the oracle's decode of the
    same codes and scales rounded to BF16."""
    wl = synthetic.llama8b_fprop()
    q = nv.quantize(wl.tensors["W"].cuda(), block="2d")
    y = nv.dequantize(q, torch.bfloat16)
    nv.sync_check()
    rows = np.sort(np.random.default_rng(9).choice(14336, 256, replace=False))
    codes = q.codes.cpu().numpy()[rows]
    KB = 4096 // 16
    r = rows.astype(np.int64)[:, None]
    kb = np.arange(KB, dtype=np.int64)[None, :]
    phys = q.scales.cpu().numpy()
    scales = phys[((r >> 7) * (KB // 4) + (kb >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (kb & 3)]
    yr = oracle.dequantize(codes, scales, float(q.global_scale.cpu()[0]))
    assert torch.equal(y[torch.from_numpy(rows).cuda()].cpu(), torch.from_numpy(yr).to(torch.bfloat16))


def test_dequantize_grid_stride_wraps_rows():
    """More blocks than one pass of the grid (16 CTAs of 256 threads per SM) and
    a grid stride that is no multiple of the blocks per row (257 here), so every
    thread's walk carries from row to row at different block columns; the whole
    output bit-exact with the oracle."""
    rows, cols = 4800, 4112
    x = torch.from_numpy(synthetic.normal((rows, cols), 1.0, 52)).to(torch.bfloat16)
    q = nv.quantize(x.cuda())
    y32 = nv.dequantize(q, torch.float32)
    nv.sync_check()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert rows * (cols // 16) > sms * 16 * 256 and (sms * 16 * 256) % (cols // 16) != 0
    ref = oracle_quantize_like(x.float())
    yr = oracle.dequantize(ref.codes, ref.scales, ref.g)
    assert (y32.cpu().numpy().view(np.uint32) == yr.view(np.uint32)).all()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_dequantize_output_aligned_to_16_bytes_only(dtype):
    """An output that starts 16 bytes past a 32-byte boundary (the decoder's
    256-bit stores need 32): the 16-byte store path, bit-exact, and the bytes
    around the output untouched."""
    rows, cols = 96, 208
    x = torch.from_numpy(synthetic.normal((rows, cols), 1.0, 53))
    q = nv.quantize(x.cuda())
    es = 4 if dtype == torch.float32 else 2
    lead = 16 // es
    buf = torch.full((rows * cols + 2 * lead,), -3.0, dtype=dtype, device="cuda")
    y = buf[lead:lead + rows * cols].view(rows, cols)
    assert y.data_ptr() % 32 == 16
    nv.dequantize(q, dtype, out=y)
    nv.sync_check()
    ref = oracle_quantize_like(x)
    yr = oracle.dequantize(ref.codes, ref.scales, ref.g)
    if dtype == torch.float32:
        assert (y.cpu().numpy().view(np.uint32) == yr.view(np.uint32)).all()
    else:
        assert torch.equal(y.cpu(), torch.from_numpy(yr).to(torch.bfloat16))
    edges = torch.cat([buf[:lead], buf[lead + rows * cols:]]).float().cpu()
    assert (edges == -3.0).all()
