"""RHT quantizer on the GPU (the Wgrad operand path).

1. The transformed values (fp32 butterfly on the GPU) are within
   1e-6 * ||x_chunk||_2 of the oracle's fp64 transform, element by element.
2. The GPU's codes, scales, amax and g are bit-exact with the oracle's
   quantizer applied to the GPU's own transformed values.
3. Against the oracle's full RHT quantize, a code may differ only between
   neighbouring grid points whose boundary lies between the two transformed
   values; the flip count is reported.
"""
import numpy as np
import pytest
import torch

import nvfp4_bit_block_02_b300 as nv
import oracle
import synthetic
from tests.gpu_helpers import assert_same_quantized, to_numpy_f32, unpack_codes

pytestmark = pytest.mark.gpu

GRID = np.array([0, .5, 1, 1.5, 2, 3, 4, 6], np.float64)


def chunk_norms(V: np.ndarray) -> np.ndarray:
    R, K = V.shape
    n = np.linalg.norm(V.astype(np.float64).reshape(R, K // 16, 16), axis=2)
    return np.repeat(n, 16, axis=1)


def check_rht(x_cpu: torch.Tensor, transpose: bool, rounding="rne", scaling="max6", seed=1, offset=0, rht_seed=1):
    x = x_cpu.cuda()
    q, dbg = nv.rht_quantize(x, rht_seed=rht_seed, transpose=transpose, rounding=rounding, scaling=scaling,
                             seed=seed, offset=offset, transformed_debug=True)
    nv.sync_check()
    xf = to_numpy_f32(x_cpu)
    V = xf.T if transpose else xf
    sr, f46 = rounding == "stochastic", scaling == "four_over_six"
    full = oracle.quantize(xf, transpose=transpose, rht=True, rht_seed=rht_seed, stochastic=sr, four_over_six=f46,
                           seed=seed, offset=offset, want_transformed=True)
    y_gpu = dbg.cpu().numpy()
    # 1. transform tolerance
    err = np.abs(y_gpu.astype(np.float64) - full.transformed.astype(np.float64))
    tol = 1e-6 * chunk_norms(V)
    assert (err <= tol).all(), f"transform error {err.max()} above 1e-6 * chunk norm"
    # 2. bit-exact encode of the GPU's transformed values
    ref2 = oracle.quantize(y_gpu, stochastic=sr, four_over_six=f46, seed=seed, offset=offset)
    assert_same_quantized(q, ref2, "encode of transformed values")
    # 3. flips against the fp64-transform oracle
    cg = unpack_codes(q.codes.cpu().numpy())
    cr = unpack_codes(full.codes)
    flips = np.argwhere(cg != cr)
    if flips.size:
        same_scale = (np.repeat(ref2.scales, 16, 1) == np.repeat(full.scales, 16, 1))
        for r, k in flips[:2000]:
            if not same_scale[r, k]:
                continue  # the block scale itself moved by a boundary case of its own
            ig, ir = cg[r, k] & 7, cr[r, k] & 7
            assert abs(int(ig) - int(ir)) <= 1 or (cg[r, k] & 7) == 0 == (cr[r, k] & 7), (r, k, cg[r, k], cr[r, k])
    return len(flips), cg.size


@pytest.mark.parametrize("transpose", [True, False])
@pytest.mark.parametrize("rounding,scaling", [("rne", "max6"), ("stochastic", "max6"), ("rne", "four_over_six"),
                                              ("stochastic", "four_over_six")])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_rht_parity_small(transpose, rounding, scaling, dtype):
    x = synthetic.student_t((272, 144), 4, 1e-3, 21)
    x[3, 5] = 0.5  # one outlier the transform spreads
    flips, n = check_rht(torch.from_numpy(x).to(dtype), transpose, rounding, scaling)
    assert flips <= max(4, n // 1000)


def test_rht_signs_match_the_oracle_stream():
    """A unit impulse at chunk position i comes out as sigma_i * H[:, i] / 4."""
    H = oracle.hadamard16()
    sigma = oracle.rht_signs(5)
    x = np.zeros((16, 16), np.float32)
    for i in range(16):
        x[i, i] = 1.0            # column i holds e_i along K (transpose: K = rows)
    q, dbg = nv.rht_quantize(torch.from_numpy(x).cuda(), rht_seed=5, transpose=True, transformed_debug=True)
    torch.cuda.synchronize()
    y = dbg.cpu().numpy()
    for i in range(16):
        assert (y[i] == sigma[i] * H[:, i] / 4.0).all()


def test_wgrad_operands_full_size():
    """dY^T (SR, Philox seed 1) and X^T (RNE) of the Wgrad workload, RHT seed 1."""
    wl = synthetic.wgrad()
    for name, rounding in [("dY", "stochastic"), ("X", "rne")]:
        flips, n = check_rht(wl.tensors[name], True, rounding, "max6", seed=1, offset=0, rht_seed=1)
        print(f"{name}: {flips} code flips of {n} against the fp64-transform oracle")
        assert flips <= n // 10000
