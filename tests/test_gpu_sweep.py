"""A seeded sweep over random configurations, each checked against the oracle:
quantizer codes, scale bytes, amax and g bit-exact (every non-RHT mode, both
orientations and input dtypes, random shapes inside the format rules, random
value scales and outlier rates); GEMMs of random shapes (any M and N, K a
multiple of 64) within 1e-5 * sum|a||b|.  The draws come from fixed seeds, so
every case is reproducible by its id."""
import numpy as np
import pytest
import torch

import nvfp4_bit_block_02_b300 as nv
import oracle
import synthetic
from tests.gpu_helpers import assert_same_quantized, gemm_check, guarded_tensor, oracle_quantize_like

pytestmark = pytest.mark.gpu

N_QUANT, N_GEMM = 48, 24


def _quant_case(i):
    rng = np.random.default_rng(1000 + i)
    block = rng.choice(["1d", "2d"])
    rounding = rng.choice(["rne", "stochastic"])
    scaling = rng.choice(["max6", "four_over_six"])
    transpose = bool(rng.integers(0, 2))
    dtype = torch.bfloat16 if rng.integers(0, 2) else torch.float32
    # output orientation R x K: K % 16 == 0; 2D needs R % 16 == 0; transposed input needs R % 16 == 0 too
    K = 16 * int(rng.integers(1, 40))
    R = int(rng.integers(1, 400))
    if block == "2d" or transpose:
        R = 16 * max(1, R // 16)
    scale = float(10.0 ** rng.uniform(-6, 4))
    outliers = float(rng.choice([0.0, 0.001, 0.02]))
    seed, offset = int(rng.integers(0, 2**31)), int(rng.integers(0, 1000))
    return dict(block=block, rounding=rounding, scaling=scaling, transpose=transpose, dtype=dtype, R=R, K=K,
                scale=scale, outliers=outliers, seed=seed, offset=offset, data_seed=2000 + i)


@pytest.mark.parametrize("i", range(N_QUANT))
def test_quantize_sweep(i):
    c = _quant_case(i)
    rows, cols = (c["K"], c["R"]) if c["transpose"] else (c["R"], c["K"])
    x = synthetic.normal((rows, cols), c["scale"], c["data_seed"])
    if c["outliers"]:
        x = synthetic.with_entry_outliers(x, c["outliers"], 30.0, c["data_seed"] + 1)
    x_cpu = torch.from_numpy(x).to(c["dtype"])
    mode = dict(block=c["block"], rounding=c["rounding"], scaling=c["scaling"], seed=c["seed"], offset=c["offset"])
    q, bufs = guarded_tensor(c["R"], c["K"])
    nv.quantize(x_cpu.cuda(), transpose=c["transpose"], out=q, **mode)
    nv.sync_check()
    for b in bufs:
        b.check()
    ref = oracle_quantize_like(x_cpu, transpose=c["transpose"], block2d=c["block"] == "2d",
                               stochastic=c["rounding"] == "stochastic", four_over_six=c["scaling"] == "four_over_six",
                               seed=c["seed"], offset=c["offset"])
    assert_same_quantized(q, ref, f"sweep case {i}: {c}")


@pytest.mark.parametrize("i", range(N_GEMM))
def test_gemm_sweep(i):
    rng = np.random.default_rng(3000 + i)
    M, N = int(rng.integers(1, 700)), int(rng.integers(1, 700))
    K = 64 * int(rng.integers(1, 20))
    out_dtype = torch.bfloat16 if rng.integers(0, 2) else torch.float32
    a = torch.from_numpy(synthetic.normal((M, K), float(10.0 ** rng.uniform(-2, 2)), 4000 + i))
    b = torch.from_numpy(synthetic.normal((N, K), float(10.0 ** rng.uniform(-3, 1)), 5000 + i))
    b_block = "2d" if N % 16 == 0 and rng.integers(0, 2) else "1d"
    qa = nv.quantize(a.cuda())
    qb = nv.quantize(b.cuda(), block=b_block)
    # D's rows start on 16-byte boundaries (the boundary's rule for ldd); the
    # padding columns and an extra row keep a canary value
    per16 = 16 // (2 if out_dtype == torch.bfloat16 else 4)
    ld = -(-N // per16) * per16
    big = torch.full((M + 1, ld + per16), -7.0, dtype=out_dtype, device="cuda")
    d = big[:M, :N]
    nv.gemm(qa, qb, out=d)
    nv.sync_check()
    full = big.float().cpu().numpy()
    assert (full[:M, N:] == -7.0).all() and (full[M:] == -7.0).all(), "write outside D"
    ra = oracle_quantize_like(a)
    rb = oracle_quantize_like(b, block2d=b_block == "2d")
    assert_same_quantized(qa, ra, f"A of GEMM case {i}")
    assert_same_quantized(qb, rb, f"B of GEMM case {i}")
    ref, bound = oracle.gemm_reference(ra, rb)
    gemm_check(full[:M, :N], ref, bound, out_dtype == torch.bfloat16, f"GEMM case {i}: {M}x{N}x{K}")
