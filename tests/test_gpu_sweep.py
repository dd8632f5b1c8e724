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

N_QUANT, N_GEMM = 160, 96


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


@pytest.mark.parametrize("i", range(48))
def test_w4a16_sweep(i):
    """Random M, N, K (K % 16 == 0) and a padded output row; the padding keeps
    its canary."""
    from tests.test_gpu_w4a16 import activations_f32, bf16_activations, random_weight
    rng = np.random.default_rng(6000 + i)
    M, N, K = int(rng.integers(1, 41)), int(rng.integers(1, 600)), 16 * int(rng.integers(1, 300))
    out_dtype = torch.bfloat16 if rng.integers(0, 2) else torch.float32
    pad = int(rng.integers(0, 10))
    q, ref = random_weight(N, K, 7000 + i)
    x = bf16_activations(M, K, 8000 + i)
    big = torch.full((M + 1, N + pad), -7.0, dtype=out_dtype, device="cuda")
    nv.w4a16_gemm(x.cuda(), q, out=big[:M, :N])
    nv.sync_check()
    full = big.float().cpu().numpy()
    assert (full[:M, N:] == -7.0).all() and (full[M:] == -7.0).all(), "write outside y"
    y_ref, bound = oracle.w4a16_reference(activations_f32(x, K), ref)
    gemm_check(full[:M, :N], y_ref, bound, out_dtype == torch.bfloat16, f"W4A16 case {i}: {M}x{N}x{K}")


@pytest.mark.parametrize("i", range(24))
def test_gemm_grouped_sweep(i):
    """1..6 groups of random shapes (an empty group included at random); each
    group's rows a whole number of 16-byte units, as the grouped call requires."""
    rng = np.random.default_rng(9000 + i)
    out_dtype = torch.bfloat16 if rng.integers(0, 2) else torch.float32
    per16 = 8 if out_dtype == torch.bfloat16 else 4
    qa, qb, ra, rb = [], [], [], []
    for e in range(int(rng.integers(1, 7))):
        M = 0 if rng.random() < 0.15 else int(rng.integers(1, 300))
        N = per16 * int(rng.integers(1, 400 // per16))
        K = 64 * int(rng.integers(1, 9))
        a = torch.from_numpy(synthetic.normal((max(M, 1), K), 1.0, 9100 + 10 * i + e))[:M]
        b = torch.from_numpy(synthetic.normal((N, K), 0.05, 9200 + 10 * i + e))
        qa.append(nv.quantize(a.cuda()) if M else nv.NVFP4Tensor.empty(0, K))
        qb.append(nv.quantize(b.cuda()))
        ra.append(oracle_quantize_like(a) if M else None)
        rb.append(oracle_quantize_like(b))
    outs = nv.gemm_grouped(qa, qb, out_dtype=out_dtype)
    nv.sync_check()
    for e in range(len(qa)):
        if ra[e] is None:
            continue
        assert_same_quantized(qa[e], ra[e], f"A_{e}")
        ref, bound = oracle.gemm_reference(ra[e], rb[e])
        gemm_check(outs[e].float().cpu().numpy(), ref, bound, out_dtype == torch.bfloat16, f"grouped case {i} group {e}")


@pytest.mark.parametrize("i", range(48))
def test_gemm_quantize_sweep(i):
    """Random M, N (N % 16 == 0), K (K % 64 == 0) and tensor amax (exact,
    loose or saturating): the epilogue encoding equals the oracle's
    quantization of nvfp4_gemm's BF16 output; the stored D equals it."""
    rng = np.random.default_rng(10000 + i)
    M, N, K = int(rng.integers(1, 400)), 16 * int(rng.integers(1, 50)), 64 * int(rng.integers(1, 10))
    a = torch.from_numpy(synthetic.normal((M, K), 1.0, 10100 + i)).to(torch.bfloat16)
    b = torch.from_numpy(synthetic.normal((N, K), 0.02, 10200 + i)).to(torch.bfloat16)
    qa, qb = nv.quantize(a.cuda()), nv.quantize(b.cuda())
    d_ref, amax_true = nv.gemm_amax(qa, qb, out_dtype=torch.bfloat16)
    amax_in = amax_true * float(rng.choice([1.0, 3.0, 0.25]))
    out, bufs = guarded_tensor(M, N)
    store = bool(rng.integers(0, 2))
    d = torch.full((M + 1, N + 8), -7.0, dtype=torch.bfloat16, device="cuda")
    nv.gemm_quantize(qa, qb, amax_in, out=out, d=d[:M, :N] if store else None)
    nv.sync_check()
    for buf in bufs:
        buf.check()
    if store:
        assert torch.equal(d[:M, :N], d_ref)
    assert (d[:M, N:] == -7.0).all() and (d[M:] == -7.0).all(), "write outside D"
    ref = oracle.quantize(d_ref.float().cpu().numpy(), amax=float(amax_in.cpu()[0]))
    assert_same_quantized(out, ref, f"gemm_quantize case {i}: {M}x{N}x{K}")


@pytest.mark.parametrize("i", range(48))
def test_dequantize_sweep(i):
    """Random shapes, block modes and scalings; the FP32 output bit-exact with
    the oracle's decode, the BF16 output its nearest-even rounding."""
    rng = np.random.default_rng(11000 + i)
    block = "2d" if rng.integers(0, 2) else "1d"
    rows, cols = int(rng.integers(1, 500)), 16 * int(rng.integers(1, 80))
    if block == "2d":
        rows = 16 * max(1, rows // 16)
    scaling = "four_over_six" if rng.integers(0, 2) else "max6"
    x = torch.from_numpy(synthetic.normal((rows, cols), float(10.0 ** rng.uniform(-4, 3)), 11100 + i))
    q = nv.quantize(x.cuda(), block=block, scaling=scaling)
    y32 = nv.dequantize(q, torch.float32)
    y16 = nv.dequantize(q, torch.bfloat16)
    nv.sync_check()
    ref = oracle_quantize_like(x, block2d=block == "2d", four_over_six=scaling == "four_over_six")
    yr = oracle.dequantize(ref.codes, ref.scales, ref.g)
    assert (y32.cpu().numpy().view(np.uint32) == yr.view(np.uint32)).all()
    assert torch.equal(y16.cpu(), torch.from_numpy(yr).to(torch.bfloat16))


@pytest.mark.parametrize("i", range(64))
def test_rht_sweep(i):
    """Random RHT configurations (orientation, rounding, scaling, dtype, shape,
    value scale, wide-span chunks) under the RHT parity rules of
    tests/test_gpu_rht.py (check_rht)."""
    from tests.test_gpu_rht import check_rht
    rng = np.random.default_rng(12000 + i)
    transpose = bool(rng.integers(0, 2))
    rounding = "stochastic" if rng.integers(0, 2) else "rne"
    scaling = "four_over_six" if rng.integers(0, 2) else "max6"
    dtype = torch.bfloat16 if rng.integers(0, 2) else torch.float32
    # K = 16 * k along the transform; the transposed input needs its columns % 16
    rows, cols = 16 * int(rng.integers(1, 30)), 16 * int(rng.integers(1, 30))
    x = synthetic.student_t((rows, cols), 4, float(10.0 ** rng.uniform(-5, 1)), 12100 + i)
    if rng.integers(0, 2):  # some chunks with tiny neighbours of large values
        tiny = rng.random((rows, cols)) < 0.1
        x[tiny] *= np.exp2(-rng.integers(4, 24, size=int(tiny.sum()))).astype(np.float32)
    check_rht(torch.from_numpy(x).to(dtype), transpose, rounding, scaling)


@pytest.mark.parametrize("i", range(24))
def test_quantize_grouped_sweep(i):
    """1..70 tensors of random shapes in one grouped call (a second launch past
    64) with a random mode: every group bit-exact with the single-tensor call
    at offset + e, two groups against the oracle."""
    rng = np.random.default_rng(13000 + i)
    block = "2d" if rng.integers(0, 2) else "1d"
    transpose = bool(rng.integers(0, 2))
    rounding = "stochastic" if rng.integers(0, 2) else "rne"
    scaling = "four_over_six" if rng.integers(0, 2) else "max6"
    dtype = torch.bfloat16 if rng.integers(0, 2) else torch.float32
    count = int(rng.choice([1, 5, 33, 70]))
    kw = dict(block=block, rounding=rounding, scaling=scaling, transpose=transpose, seed=int(rng.integers(0, 1000)),
              offset=int(rng.integers(0, 1000)))
    xs = []
    for e in range(count):
        R, K = int(rng.integers(1, 200)), 16 * int(rng.integers(1, 20))
        if block == "2d" or transpose:
            R = 16 * max(1, R // 16)
        shape = (K, R) if transpose else (R, K)
        xs.append(torch.from_numpy(synthetic.normal(shape, float(10.0 ** rng.uniform(-3, 2)), 13100 + 100 * i + e))
                  .to(dtype).cuda())
    qs = nv.quantize_grouped(xs, **kw)
    nv.sync_check()
    for e, x in enumerate(xs):
        single = nv.quantize(x, **{**kw, "offset": kw["offset"] + e})
        assert torch.equal(qs[e].codes, single.codes) and torch.equal(qs[e].scales, single.scales), f"group {e}"
        assert torch.equal(qs[e].amax, single.amax) and torch.equal(qs[e].global_scale, single.global_scale)
    for e in sorted({0, count - 1}):
        ref = oracle_quantize_like(xs[e].cpu(), transpose=transpose, block2d=block == "2d",
                                   stochastic=rounding == "stochastic", four_over_six=scaling == "four_over_six",
                                   seed=kw["seed"], offset=kw["offset"] + e)
        assert_same_quantized(qs[e], ref, f"grouped case {i} group {e}")


@pytest.mark.parametrize("i", range(48))
def test_transpose_2d_sweep(i):
    """Random R x K (both % 16) and scaling, RNE: repacking the 2D quantization
    of W equals the oracle's 2D quantization of W^T bit for bit."""
    rng = np.random.default_rng(14000 + i)
    R, K = 16 * int(rng.integers(1, 60)), 16 * int(rng.integers(1, 60))
    scaling = "four_over_six" if rng.integers(0, 2) else "max6"
    dtype = torch.bfloat16 if rng.integers(0, 2) else torch.float32
    x = torch.from_numpy(synthetic.normal((R, K), float(10.0 ** rng.uniform(-3, 2)), 14100 + i)).to(dtype)
    q = nv.quantize(x.cuda(), block="2d", scaling=scaling)
    qt, bufs = guarded_tensor(K, R)
    nv.transpose_2d(q, out=qt)
    nv.sync_check()
    for b in bufs:
        b.check()
    ref = oracle_quantize_like(x.t().contiguous(), block2d=True, four_over_six=scaling == "four_over_six")
    assert_same_quantized(qt, ref, f"transpose_2d case {i}: {R}x{K} {scaling}")
