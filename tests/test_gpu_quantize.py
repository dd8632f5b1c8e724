"""Quantizer parity on the GPU: codes, physical scale bytes, amax and g must be
bit-exact with the oracle on the same seeded bytes (non-RHT paths)."""
import numpy as np
import pytest
import torch

import nvfp4_bit_block_02_b300 as nv
import oracle
import synthetic
from tests.gpu_helpers import assert_same_quantized, guarded_tensor, oracle_quantize_like, to_numpy_f32

pytestmark = pytest.mark.gpu

SHAPES = [(256, 256), (48, 80), (130, 1040), (384, 528), (16, 16), (1, 32)]
MODES = [
    dict(block="1d", rounding="rne", scaling="max6"),
    dict(block="1d", rounding="stochastic", scaling="max6", seed=1, offset=0),
    dict(block="1d", rounding="rne", scaling="four_over_six"),
    dict(block="1d", rounding="stochastic", scaling="four_over_six", seed=7, offset=3),
    dict(block="2d", rounding="rne", scaling="max6"),
    dict(block="2d", rounding="rne", scaling="four_over_six"),
    dict(block="2d", rounding="stochastic", scaling="four_over_six", seed=9, offset=1),
]


def oracle_kw(mode, transpose):
    return dict(transpose=transpose, block2d=mode["block"] == "2d", stochastic=mode["rounding"] == "stochastic",
                four_over_six=mode["scaling"] == "four_over_six", seed=mode.get("seed", 0),
                offset=mode.get("offset", 0))


def run_case(x_cpu, mode, transpose, amax=None):
    x = x_cpu.cuda()
    rows, cols = x.shape
    R, K = (cols, rows) if transpose else (rows, cols)
    q, bufs = guarded_tensor(R, K)
    amax_t = None if amax is None else torch.tensor([amax], dtype=torch.float32, device="cuda")
    nv.quantize(x, transpose=transpose, out=q, amax=amax_t, **mode)
    nv.sync_check()
    for b in bufs:
        b.check()
    ref = oracle_quantize_like(x_cpu, amax=amax, **oracle_kw(mode, transpose))
    return q, ref


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("transpose", [False, True])
@pytest.mark.parametrize("mode", MODES, ids=lambda m: f"{m['block']}-{m['rounding']}-{m['scaling']}")
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}x{s[1]}")
def test_quantize_parity(shape, mode, transpose, dtype):
    rows, cols = shape
    if transpose:
        rows, cols = cols, rows  # keep K = the second number of the shape
    R, K = (cols, rows) if transpose else (rows, cols)
    if K % 16 or (transpose and cols % 16) or (mode["block"] == "2d" and R % 16):
        pytest.skip("shape outside the format rules for this mode")
    x = synthetic.with_entry_outliers(synthetic.normal((rows, cols), 1.0, 31 + rows), 0.01, 50.0, 5)
    x_cpu = torch.from_numpy(x).to(dtype)
    q, ref = run_case(x_cpu, mode, transpose)
    assert_same_quantized(q, ref, f"{shape} {mode} T={transpose} {dtype}")


@pytest.mark.parametrize("transpose", [False, True])
def test_quantize_with_supplied_amax(transpose):
    x = torch.from_numpy(synthetic.normal((128, 256), 0.5, 3)).to(torch.bfloat16)
    amax = 7.25   # larger than max|x|: the producer's amax is taken as given
    q, ref = run_case(x, MODES[0], transpose, amax=amax)
    assert_same_quantized(q, ref, "supplied amax")
    assert float(q.amax.cpu()[0]) == amax


def _anchored(blocks: np.ndarray) -> np.ndarray:
    """Rows of 16-element blocks plus a row holding 2688, so g = 1."""
    x = np.zeros((blocks.shape[0] + 1, blocks.shape[1]), np.float32)
    x[:-1] = blocks
    x[-1, 0] = 2688.0
    return x


def test_e2m1_conversion_sweep_through_the_encoder():
    """g = 1 and every block holds a 6, so s_b = 1 and q = x exactly: the
    hardware E2M1 conversion meets the oracle on every bf16 value in [-8, 8],
    the ties, their float neighbours and signed zeros."""
    bf = (np.arange(0, 0x4101, dtype=np.uint32) << 16).view(np.float32)
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6], np.float32)
    mids = (grid[:-1] + grid[1:]) / 2
    near = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(9))])
    vals = np.concatenate([bf, -bf, near, -near, [0.0, -0.0, 1e-30, -1e-30, 5.9999995, 6.0000005, 100.0]])
    vals = vals.astype(np.float32)
    n = -(-vals.size // 15)
    pad = np.zeros(n * 15, np.float32)
    pad[:vals.size] = vals
    blocks = np.concatenate([np.full((n, 1), 6.0, np.float32), pad.reshape(n, 15)], axis=1)
    x = _anchored(blocks)
    x_cpu = torch.from_numpy(x)
    q, ref = run_case(x_cpu, MODES[0], False)
    assert_same_quantized(q, ref, "e2m1 sweep")


def test_e4m3_conversion_sweep_through_the_encoder():
    """g = 1 and block max 6t: t_b = t, so s_b is the hardware E4M3 rounding
    of t, for t over the whole E4M3 range, its ties and neighbours."""
    e4 = np.array([oracle.e4m3_decode(b) for b in range(0x7F)], np.float64)
    mids = (e4[:-1] + e4[1:]) / 2
    t = np.concatenate([e4, mids, mids * (1 + 2 ** -20), mids * (1 - 2 ** -20), np.exp2(np.linspace(-12, 8.9, 4000)),
                        [448.0, 449.0, 470.0, 1e-8]])
    t = t[t * 6 <= 2688.0]
    blocks = np.zeros((t.size, 16), np.float32)
    blocks[:, 0] = (t * 6).astype(np.float32)
    blocks[:, 1] = (t * 2.5).astype(np.float32)
    x_cpu = torch.from_numpy(_anchored(blocks))
    q, ref = run_case(x_cpu, MODES[0], False)
    assert_same_quantized(q, ref, "e4m3 sweep")


@pytest.mark.parametrize("case", ["zeros", "one_outlier", "denormals", "signed_zeros", "tiny_blocks"])
def test_edge_tensors(case):
    rows, cols = 64, 128
    x = np.zeros((rows, cols), np.float32)
    if case == "one_outlier":
        x = synthetic.normal((rows, cols), 1.0, 8)
        x[17, 33] = 1e6
    elif case == "denormals":
        x = synthetic.normal((rows, cols), 1e-39, 9)
        x[0, 0] = 1e-30   # amax above the supported floor, the rest denormal
    elif case == "signed_zeros":
        x[:, ::2] = -0.0
        x[5, 7] = 3.0
    elif case == "tiny_blocks":
        x = synthetic.normal((rows, cols), 1e-4, 10)
        x[0, 0] = 1e3
    for mode in [MODES[0], MODES[2], MODES[4], MODES[1]]:
        for tr in [False, True]:
            q, ref = run_case(torch.from_numpy(x), mode, tr)
            assert_same_quantized(q, ref, f"{case} {mode} T={tr}")


def test_quantize_is_deterministic():
    x = torch.from_numpy(synthetic.normal((512, 1024), 1.0, 11)).to(torch.bfloat16).cuda()
    outs = [nv.quantize(x, rounding="stochastic", scaling="four_over_six", seed=3) for _ in range(10)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o.codes, outs[0].codes) and torch.equal(o.scales, outs[0].scales)


def test_strided_input():
    full = torch.from_numpy(synthetic.normal((96, 256), 1.0, 12)).to(torch.bfloat16)
    x = full[:, :160]   # ld = 256
    q = nv.quantize(x.cuda())
    torch.cuda.synchronize()
    ref = oracle_quantize_like(x.contiguous())
    assert_same_quantized(q, ref, "strided")


def test_empty_tensor():
    x = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    q = nv.quantize(x)
    nv.sync_check()
    assert float(q.amax.cpu()[0]) == 0.0 and float(q.global_scale.cpu()[0]) == 1.0


# ---------------------------------------------------------------- full size --
def test_llama8b_fprop_operands_full_size():
    wl = synthetic.llama8b_fprop()
    for name, block in [("X", "1d"), ("W", "2d")]:
        x = wl.tensors[name]
        q = nv.quantize(x.cuda(), block=block)
        torch.cuda.synchronize()
        ref = oracle_quantize_like(x, block2d=block == "2d")
        assert_same_quantized(q, ref, f"8B {name}")
        del q


def test_moe_expert_weights_four_over_six_full_size_sample():
    """Every 8th expert of the MoE workload (W_e^T, Four-over-Six, K = 4096)."""
    wl = synthetic.moe()
    W = wl.tensors["W"]
    for e in range(0, W.shape[0], 8):
        q = nv.quantize(W[e].cuda(), transpose=True, scaling="four_over_six")
        torch.cuda.synchronize()
        ref = oracle_quantize_like(W[e], transpose=True, four_over_six=True)
        assert_same_quantized(q, ref, f"MoE expert {e}")


def test_wgrad_dy_stochastic_transposed_full_size():
    wl = synthetic.wgrad()
    dy = wl.tensors["dY"]
    q = nv.quantize(dy.cuda(), transpose=True, rounding="stochastic", seed=1, offset=0)
    torch.cuda.synchronize()
    ref = oracle_quantize_like(dy, transpose=True, stochastic=True, seed=1, offset=0)
    assert_same_quantized(q, ref, "wgrad dY^T SR")
