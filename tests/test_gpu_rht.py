"""RHT quantizer on the GPU (the Wgrad operand path).

The transform is y = 1/4 * H16 * diag(sigma) * x per 16-chunk along K
("NVIDIA Introduces a 4-Bit Pretraining Methodology Using NVFP4", "Method":
16x16 Random Hadamard Transforms on Wgrad inputs).  The checks:

1. Transformed values within 1e-6 * ||x_chunk||_2 of the oracle's fp64
   transform, element by element.  The GPU rounds each value once from the
   exact one (an exact split of every input into a coarse and a fine part), so
   inside the documented exactness range (chunk magnitudes within 2^33 of
   each other for BF16, 2^17 for FP32) they must equal the oracle's values bit
   for bit; the count of values that differ anywhere is reported.
2. The GPU's codes, scales, amax and g are bit-exact with the oracle's
   quantizer applied to the GPU's own transformed values.
3. Against the oracle's full RHT quantize (fp64 transform), a code may differ
   only where both sides' pre-rounding values q = fl(y * r_b) lie within one
   fp32 ulp of the same rounding boundary of that element (an E2M1 midpoint
   for RNE, the element's threshold lo + u16 * step / 65536 for stochastic
   rounding), and a block scale only where t_b = fl(amax_b / fl(6 g)) lies
   within one ulp of an E4M3 rounding boundary or amax differs by one ulp.
   Every flip is checked and the counts are reported.
"""
import numpy as np
import pytest
import torch

import nvfp4_bit_block_02_b300 as nv
import oracle
import synthetic
from tests.gpu_helpers import assert_same_quantized, to_numpy_f32, unpack_codes

pytestmark = pytest.mark.gpu

E2M1_MAG = np.array([0, .5, 1, 1.5, 2, 3, 4, 6], np.float64)
RNE_BOUNDARIES = (E2M1_MAG[:-1] + E2M1_MAG[1:]) / 2            # 0.25, 0.75, ..., 5
E4M3_VALUES = np.array([oracle.e4m3_decode(b) for b in range(0x7F)], np.float64)
E4M3_BOUNDARIES = (E4M3_VALUES[:-1] + E4M3_VALUES[1:]) / 2


def ulp32(x: np.ndarray) -> np.ndarray:
    """Spacing of fp32 at |x| (the smallest subnormal at 0)."""
    a = np.abs(np.asarray(x, np.float32))
    return np.spacing(a).astype(np.float64)


def chunk_norms(V: np.ndarray) -> np.ndarray:
    R, K = V.shape
    n = np.linalg.norm(V.astype(np.float64).reshape(R, K // 16, 16), axis=2)
    return np.repeat(n, 16, axis=1)


def exact_range_mask(V: np.ndarray, bf16: bool) -> np.ndarray:
    """Elements whose chunk lies in the documented exactness range of the
    GPU transform: nonzero magnitudes within 2^33 (BF16) / 2^17 (FP32) of the
    chunk maximum, and the maximum below 2^124."""
    R, K = V.shape
    a = np.abs(V.astype(np.float64)).reshape(R, K // 16, 16)
    mx = a.max(axis=2)
    mn = np.where(a > 0, a, np.inf).min(axis=2)
    e_mx = np.floor(np.log2(np.where(mx > 0, mx, 1.0)))
    e_mn = np.floor(np.log2(np.where(np.isfinite(mn), mn, 1.0)))
    ok = (e_mx - e_mn <= (33 if bf16 else 17)) & (mx < 2.0 ** 124)
    return np.repeat(ok, 16, axis=1)


def block_reciprocals(q: oracle.Quantized) -> tuple[np.ndarray, np.ndarray]:
    """Per element (R x K): the block's decoded scale s and reciprocal
    r = fl(1 / fl(s * g)) (0 when s * g == 0), in fp32."""
    s = np.array([oracle.e4m3_decode(b) if b != 0x7F else 0.0 for b in range(256)], np.float32)[q.scales]
    S = (s * np.float32(q.g)).astype(np.float32)
    with np.errstate(divide="ignore"):
        r = np.where(S == 0, np.float32(0), (np.float32(1) / np.where(S == 0, np.float32(1), S)).astype(np.float32))
    return np.repeat(s, 16, 1), np.repeat(r.astype(np.float32), 16, 1)


def sr_thresholds(u16: int) -> np.ndarray:
    """The 7 points where stochastic rounding with draw u16 changes code:
    in [lo, hi) the element rounds up iff |q| > lo + u16 * (hi - lo) / 65536."""
    lo, hi = E2M1_MAG[:-1], E2M1_MAG[1:]
    return lo + u16 * (hi - lo) / 65536.0


def check_flip(qa: float, qb: float, boundaries: np.ndarray) -> bool:
    """Both |qa| and |qb| within one fp32 ulp of the same boundary that lies
    between them (or on one of them)."""
    a, b = abs(float(qa)), abs(float(qb))
    lo, hi = min(a, b), max(a, b)
    cands = boundaries[(boundaries >= lo - 1e-30) & (boundaries <= hi + 1e-30)]
    for beta in cands:
        u = float(ulp32(np.float32(beta)))
        if abs(a - beta) <= u and abs(b - beta) <= u:
            return True
    return False


def check_rht(x_cpu: torch.Tensor, transpose: bool, rounding="rne", scaling="max6", seed=1, offset=0, rht_seed=1):
    x = x_cpu.cuda()
    q, dbg = nv.rht_quantize(x, rht_seed=rht_seed, transpose=transpose, rounding=rounding, scaling=scaling,
                             seed=seed, offset=offset, transformed_debug=True)
    nv.sync_check()
    xf = to_numpy_f32(x_cpu)
    V = xf.T if transpose else xf
    sr, f46 = rounding == "stochastic", scaling == "four_over_six"
    full = oracle.quantize(xf, transpose=transpose, rht=True, rht_seed=rht_seed, stochastic=sr, four_over_six=f46,
                           seed=seed, offset=offset, want_transformed=True, want_choice=True)
    y_gpu = dbg.cpu().numpy()
    y_ref = full.transformed
    R, K = y_ref.shape
    # 1. transform tolerance, and bit-exactness inside the exactness range
    err = np.abs(y_gpu.astype(np.float64) - y_ref.astype(np.float64))
    tol = 1e-6 * chunk_norms(V)
    assert (err <= tol).all(), f"transform error {err.max()} above 1e-6 * chunk norm"
    differ = y_gpu.view(np.uint32) != y_ref.view(np.uint32)
    exact = exact_range_mask(V, x_cpu.dtype == torch.bfloat16)
    assert not (differ & exact).any(), (f"{int((differ & exact).sum())} transformed values inside the exactness "
                                        f"range are not the correctly rounded ones")
    # 2. bit-exact encode of the GPU's transformed values
    ref2 = oracle.quantize(y_gpu, stochastic=sr, four_over_six=f46, seed=seed, offset=offset, want_choice=True)
    assert_same_quantized(q, ref2, "encode of transformed values")
    # 3. every flip against the fp64-transform oracle sits on a rounding boundary
    cg = unpack_codes(q.codes.cpu().numpy())
    cr = unpack_codes(full.codes)
    code_flips = np.argwhere(cg != cr)
    scale_flips = np.argwhere(ref2.scales != full.scales)
    if ref2.amax != full.amax:
        assert abs(ref2.amax - full.amax) <= float(ulp32(np.float32(full.amax))), "amax moved by more than 1 ulp"
    s_g, r_g = block_reciprocals(ref2)
    s_r, r_r = block_reciprocals(full)
    g6_r = np.float32(6) * np.float32(full.g)
    for r, kb in scale_flips:
        amax_b = np.float32(np.abs(y_ref[r, 16 * kb:16 * kb + 16]).max())
        t = np.float32(amax_b / g6_r)
        assert ref2.amax != full.amax or check_flip(t, t, E4M3_BOUNDARIES) or \
            (ref2.choice[r, kb] != full.choice[r, kb]), f"block ({r}, {kb}) scale moved away from an E4M3 boundary"
    moved = np.repeat(ref2.scales != full.scales, 16, 1)
    for r, k in code_flips:
        if moved[r, k] or ref2.amax != full.amax:
            continue  # the block scale moved (checked above); its codes follow it
        qa = np.float32(np.float32(y_ref[r, k]) * r_r[r, k])
        qb = np.float32(np.float32(y_gpu[r, k]) * r_g[r, k])
        bounds = sr_thresholds(oracle.sr_bits(seed, offset, int(r) * K + int(k))) if sr else RNE_BOUNDARIES
        assert check_flip(qa, qb, np.concatenate([[0.0], bounds])), \
            f"code flip at ({r}, {k}): q {qa} (oracle) / {qb} (GPU) not within 1 ulp of one rounding boundary"
    n_diff = int(differ.sum())
    print(f"RHT {x_cpu.dtype} {tuple(x_cpu.shape)} transpose={transpose} {rounding}/{scaling}: "
          f"{n_diff} transformed values differ, {len(code_flips)} code flips, {len(scale_flips)} scale flips "
          f"of {R * K} elements")
    return len(code_flips), n_diff, R * K


@pytest.mark.parametrize("transpose", [True, False])
@pytest.mark.parametrize("rounding,scaling", [("rne", "max6"), ("stochastic", "max6"), ("rne", "four_over_six"),
                                              ("stochastic", "four_over_six")])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_rht_parity_small(transpose, rounding, scaling, dtype):
    x = synthetic.student_t((272, 144), 4, 1e-3, 21)
    x[3, 5] = 0.5  # one outlier the transform spreads
    check_rht(torch.from_numpy(x).to(dtype), transpose, rounding, scaling)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_rht_wide_chunks_are_correctly_rounded(dtype):
    """Chunks whose magnitudes span many binades (tiny values beside large
    ones) are where a plain fp32 butterfly rounds; the exact split must still
    give the correctly rounded transform."""
    rng = np.random.default_rng(31)
    x = synthetic.normal((256, 128), 1.0, 32)
    tiny = rng.random((256, 128)) < 0.2
    x[tiny] *= np.exp2(-rng.integers(8, 30, size=int(tiny.sum()))).astype(np.float32)
    for transpose in (True, False):
        check_rht(torch.from_numpy(x).to(dtype), transpose, "rne", "max6")


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
    """dY^T (SR, Philox seed 1) and X^T (RNE) of the Wgrad workload, RHT seed 1:
    every flip must sit on a rounding boundary (the helper checks each one)."""
    wl = synthetic.wgrad()
    for name, rounding in [("dY", "stochastic"), ("X", "rne")]:
        flips, n_diff, n = check_rht(wl.tensors[name], True, rounding, "max6", seed=1, offset=0, rht_seed=1)
        print(f"{name}: {flips} code flips and {n_diff} differing transformed values of {n}")
