"""Block-scaled GEMM parity on the GPU against the oracle's float64 GEMM of
the dequantized operands: |D - D_ref| <= 1e-5 * sum_k |a||b| (plus half a
BF16 ulp of D_ref for BF16 output).  The operands are quantized on the GPU
and first checked bit-exact against the oracle's quantization, so both sides
multiply the same NVFP4 values."""
import numpy as np
import pytest
import torch

import nvfp4_bit_block_02_b300 as nv
import oracle
import synthetic
from tests.gpu_helpers import assert_same_quantized, gemm_check, oracle_quantize_like

pytestmark = pytest.mark.gpu


def quantize_both(x_cpu, **kw):
    q = nv.quantize(x_cpu.cuda(), **kw)
    torch.cuda.synchronize()
    okw = dict(transpose=kw.get("transpose", False), block2d=kw.get("block") == "2d",
               stochastic=kw.get("rounding") == "stochastic", four_over_six=kw.get("scaling") == "four_over_six",
               seed=kw.get("seed", 0), offset=kw.get("offset", 0))
    ref = oracle_quantize_like(x_cpu, **okw)
    assert_same_quantized(q, ref, "GEMM operand")
    return q, ref


def make_tensor_from_codes(codes: np.ndarray, logical_scales: np.ndarray, g: float) -> nv.NVFP4Tensor:
    R, K2 = codes.shape
    K = 2 * K2
    phys = oracle.swizzle_scales(logical_scales, R, K)
    return nv.NVFP4Tensor(torch.from_numpy(codes).cuda(), torch.from_numpy(phys).cuda(),
                          torch.tensor([g], dtype=torch.float32, device="cuda"),
                          torch.tensor([0.0], dtype=torch.float32, device="cuda"), R, K)


def test_gemm_pr1_256():
    wl = synthetic.pr1()
    qa, ra = quantize_both(wl.tensors["A"])
    qb, rb = quantize_both(wl.tensors["B"])
    d = nv.gemm(qa, qb, out_dtype=torch.float32)
    nv.sync_check()
    ref, bound = oracle.gemm_reference(ra, rb)
    gemm_check(d.cpu().numpy(), ref, bound, False, "PR1")


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (256, 512, 512), (384, 384, 768), (128, 128, 256),
                                   (512, 1280, 1024), (256, 256, 4096)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_gemm_shapes(M, N, K, out_dtype):
    a = torch.from_numpy(synthetic.normal((M, K), 1.0, M + K)).to(torch.bfloat16)
    b = torch.from_numpy(synthetic.normal((N, K), 0.02, N + K + 1)).to(torch.bfloat16)
    qa, ra = quantize_both(a)
    qb, rb = quantize_both(b, block="2d")
    d = nv.gemm(qa, qb, out_dtype=out_dtype)
    nv.sync_check()
    ref, bound = oracle.gemm_reference(ra, rb)
    gemm_check(d.float().cpu().numpy(), ref, bound, out_dtype == torch.bfloat16, f"{M}x{N}x{K}")


def test_gemm_all_ones_closed_form():
    M, N, K = 128, 256, 512
    a = make_tensor_from_codes(np.full((M, K // 2), 0x22, np.uint8), np.full((M, K // 16), 0x38, np.uint8), 1.0)
    b = make_tensor_from_codes(np.full((N, K // 2), 0x22, np.uint8), np.full((N, K // 16), 0x38, np.uint8), 1.0)
    d = nv.gemm(a, b, out_dtype=torch.float32)
    nv.sync_check()
    assert (d.cpu().numpy() == K).all()


def test_gemm_exact_integer_products():
    """Integer-valued codes, power-of-two scales, g = 1: the result is exact
    in fp32, so the GPU must match the oracle exactly."""
    rng = np.random.default_rng(5)
    M, N, K = 256, 512, 512
    ints = np.array([0, 2, 4, 5, 6, 7, 8, 10, 12, 13, 14, 15], np.uint8)
    pack = lambda c: (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)
    ca, cb = rng.choice(ints, (M, K)), rng.choice(ints, (N, K))
    sa = rng.choice(np.array([0x30, 0x38, 0x40], np.uint8), (M, K // 16))   # 0.5, 1, 2
    sb = rng.choice(np.array([0x30, 0x38, 0x40], np.uint8), (N, K // 16))
    a = make_tensor_from_codes(pack(ca), sa, 1.0)
    b = make_tensor_from_codes(pack(cb), sb, 1.0)
    d = nv.gemm(a, b, out_dtype=torch.float32)
    nv.sync_check()
    ra = oracle.Quantized(pack(ca), sa, 0, 1.0, None, None, M, K)
    rb = oracle.Quantized(pack(cb), sb, 0, 1.0, None, None, N, K)
    ref, _ = oracle.gemm_reference(ra, rb)
    got = d.cpu().numpy().astype(np.float64)
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{len(bad)} differ; first {bad[:3].tolist()} {got[tuple(bad[0])]} vs {ref[tuple(bad[0])]}"


def test_gemm_structured_scales_pin_the_layout():
    """Every code 1.0; A's block scales are distinct powers of two per (row,
    block) and B's per (column, block): each output is 16 * sum_kb sA * sB,
    exact, and any misplaced scale byte changes it."""
    rng = np.random.default_rng(6)
    M, N, K = 256, 512, 1024
    pows = np.array([0x28, 0x30, 0x38, 0x40, 0x48], np.uint8)   # 0.25 .. 4
    sa = rng.choice(pows, (M, K // 16))
    sb = rng.choice(pows, (N, K // 16))
    a = make_tensor_from_codes(np.full((M, K // 2), 0x22, np.uint8), sa, 1.0)
    b = make_tensor_from_codes(np.full((N, K // 2), 0x22, np.uint8), sb, 1.0)
    d = nv.gemm(a, b, out_dtype=torch.float32)
    nv.sync_check()
    dec = np.vectorize(oracle.e4m3_decode)
    ref = 16.0 * dec(sa).astype(np.float64) @ dec(sb).astype(np.float64).T
    got = d.cpu().numpy().astype(np.float64)
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{len(bad)} differ; first {bad[:3].tolist()}"


def test_gemm_is_deterministic():
    a = torch.from_numpy(synthetic.normal((256, 1024), 1.0, 40)).to(torch.bfloat16).cuda()
    b = torch.from_numpy(synthetic.normal((512, 1024), 1.0, 41)).to(torch.bfloat16).cuda()
    qa, qb = nv.quantize(a), nv.quantize(b)
    outs = [nv.gemm(qa, qb) for _ in range(5)]
    nv.sync_check()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


def test_gemm_ldd_larger_than_n():
    a = torch.from_numpy(synthetic.normal((128, 256), 1.0, 42)).to(torch.bfloat16)
    b = torch.from_numpy(synthetic.normal((256, 256), 1.0, 43)).to(torch.bfloat16)
    qa, ra = quantize_both(a)
    qb, rb = quantize_both(b)
    big = torch.full((128, 384), -7.0, dtype=torch.float32, device="cuda")
    nv.gemm(qa, qb, out=big[:, :256])
    nv.sync_check()
    ref, bound = oracle.gemm_reference(ra, rb)
    full = big.cpu().numpy()
    gemm_check(full[:, :256], ref, bound, False, "ldd")
    assert (full[:, 256:] == -7.0).all()


def _sampled_check(qa_ref, qb_ref, d, bf16, rows, what):
    ref, bound = oracle.gemm_reference(qa_ref, qb_ref, rows=rows)
    return gemm_check(d[rows].float().cpu().numpy(), ref, bound, bf16, what)


def test_gemm_llama8b_full_size_sampled():
    wl = synthetic.llama8b_fprop()
    qx, rx = quantize_both(wl.tensors["X"])
    qw, rw = quantize_both(wl.tensors["W"], block="2d")
    d = nv.gemm(qx, qw, out_dtype=torch.bfloat16)
    nv.sync_check()
    rng = np.random.default_rng(0)
    rows = np.concatenate([np.arange(0, 128), np.arange(8064, 8192), rng.choice(8192, 64, replace=False)])
    _sampled_check(rx, rw, d, True, rows, "8B fprop")


def test_gemm_wgrad_full_size_sampled():
    """dW = dY^T X with both operands RHT-transformed along the tokens, FP32 out."""
    wl = synthetic.wgrad()
    qd, _ = nv.rht_quantize(wl.tensors["dY"].cuda(), rht_seed=1, rounding="stochastic", seed=1)
    qx, _ = nv.rht_quantize(wl.tensors["X"].cuda(), rht_seed=1)
    d = nv.gemm(qd, qx, out_dtype=torch.float32)
    nv.sync_check()
    # the reference multiplies the GPU's own (separately verified) operands
    rd = oracle.Quantized(qd.codes.cpu().numpy(), None, 0, float(qd.global_scale.cpu()[0]), None, None, qd.rows, qd.cols)
    rx = oracle.Quantized(qx.codes.cpu().numpy(), None, 0, float(qx.global_scale.cpu()[0]), None, None, qx.rows, qx.cols)
    rd.scales = _logical_from_physical(qd.scales.cpu().numpy(), qd.rows, qd.cols)
    rx.scales = _logical_from_physical(qx.scales.cpu().numpy(), qx.rows, qx.cols)
    rng = np.random.default_rng(1)
    rows = np.concatenate([np.arange(0, 128), rng.choice(qd.rows, 64, replace=False)])
    _sampled_check(rd, rx, d, False, rows, "wgrad")


def _logical_from_physical(phys: np.ndarray, R: int, K: int) -> np.ndarray:
    """Inverse of the documented scale layout (index arithmetic only)."""
    KB = K // 16
    nka = (KB + 3) // 4
    r = np.arange(R)[:, None]
    kb = np.arange(KB)[None, :]
    off = ((r // 128) * nka + kb // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + kb % 4
    return phys[off]


def test_logical_from_physical_inverts_the_oracle_layout():
    rng = np.random.default_rng(2)
    R, K = 300, 1040
    logical = rng.integers(1, 255, (R, K // 16), dtype=np.uint8)
    assert (_logical_from_physical(oracle.swizzle_scales(logical, R, K), R, K) == logical).all()


@pytest.mark.parametrize("groups", [1, 3, 70])
def test_gemm_grouped_small(groups):
    rng = np.random.default_rng(groups)
    qa, qb, ra, rb = [], [], [], []
    for e in range(groups):
        M = int(rng.choice([128, 256]))
        N = int(rng.choice([128, 256, 384]))
        K = int(rng.choice([256, 512]))
        a = torch.from_numpy(synthetic.normal((M, K), 1.0, 100 + e)).to(torch.bfloat16)
        b = torch.from_numpy(synthetic.normal((N, K), 0.02, 200 + e)).to(torch.bfloat16)
        x, y = quantize_both(a)
        qa.append(x); ra.append(y)
        x, y = quantize_both(b, block="2d")
        qb.append(x); rb.append(y)
    outs = nv.gemm_grouped(qa, qb, out_dtype=torch.bfloat16)
    nv.sync_check()
    for e in range(groups):
        ref, bound = oracle.gemm_reference(ra[e], rb[e])
        gemm_check(outs[e].float().cpu().numpy(), ref, bound, True, f"group {e}")


def test_gemm_grouped_moe_full_size_sampled():
    """64 experts: X_e (512 x 4096, max-6) times W_e^T (1536 x 4096,
    Four-over-Six); every 8th expert checked on sampled rows."""
    wl = synthetic.moe()
    X, W = wl.tensors["X"], wl.tensors["W"]
    qx = [nv.quantize(X[e].cuda()) for e in range(X.shape[0])]
    qw = [nv.quantize(W[e].cuda(), transpose=True, scaling="four_over_six") for e in range(W.shape[0])]
    outs = nv.gemm_grouped(qx, qw, out_dtype=torch.bfloat16)
    nv.sync_check()
    rng = np.random.default_rng(3)
    for e in range(0, X.shape[0], 8):
        rx = oracle_quantize_like(X[e])
        rw = oracle_quantize_like(W[e], transpose=True, four_over_six=True)
        assert_same_quantized(qx[e], rx, f"X_{e}")
        assert_same_quantized(qw[e], rw, f"W_{e}")
        rows = rng.choice(512, 32, replace=False)
        _sampled_check(rx, rw, outs[e], True, rows, f"expert {e}")


def _rows_logical_scales(phys: np.ndarray, K: int, rows: np.ndarray) -> np.ndarray:
    """The logical scale bytes [len(rows)][K/16] of the given rows, read out of
    a physical buffer in the 128-row x 4-block atom layout of include/nvfp4.h."""
    KB = K // 16
    nka = (KB + 3) // 4
    r = rows.astype(np.int64)[:, None]
    kb = np.arange(KB, dtype=np.int64)[None, :]
    off = ((r >> 7) * nka + (kb >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (kb & 3)
    return phys[off]


def test_llama405b_full_size_sampled():
    """Llama-3.1-405B MLP fprop at full size: X 8192 x 16384 (1D), W 53248 x 16384
    (2D), GEMM with BF16 out, all on the GPU.  Sampled X rows and sampled
    16-row W groups are checked bit-exact against the oracle's quantization of
    those rows with the whole tensor's amax; the GEMM outputs at those rows and
    columns against the oracle's product of the same operands."""
    wl = synthetic.llama405b_fprop()
    X, W = wl.tensors["X"], wl.tensors["W"]
    K = X.shape[1]
    qx = nv.quantize(X.cuda())
    qw = nv.quantize(W.cuda(), block="2d")
    d = nv.gemm(qx, qw, out_dtype=torch.bfloat16)
    nv.sync_check()
    rng = np.random.default_rng(405)
    rx = np.unique(np.concatenate([np.arange(64), np.arange(8192 - 64, 8192), rng.choice(8192, 128, replace=False)]))
    groups = np.unique(np.concatenate([[0, 53248 // 16 - 1], rng.choice(53248 // 16, 14, replace=False)]))
    rw = (groups[:, None] * 16 + np.arange(16)[None, :]).reshape(-1)
    refs = {}
    for name, full, q, rows, b2d in (("X", X, qx, rx, False), ("W", W, qw, rw, True)):
        amax = float(torch.max(torch.abs(full)).float())
        ref = oracle.quantize(full[rows].float().numpy(), block2d=b2d, amax=amax)
        assert float(q.amax.cpu()[0]) == amax, f"405B {name}: amax"
        assert float(q.global_scale.cpu()[0]) == ref.g, f"405B {name}: g"
        codes = q.codes.cpu().numpy()[rows]
        assert (codes == ref.codes).all(), f"405B {name}: {int((codes != ref.codes).sum())} code bytes differ"
        sc = _rows_logical_scales(q.scales.cpu().numpy(), K, rows)
        assert (sc == ref.scales).all(), f"405B {name}: {int((sc != ref.scales).sum())} scale bytes differ"
        refs[name] = ref
    ref, bound = oracle.gemm_reference(refs["X"], refs["W"])
    got = d[torch.from_numpy(rx).cuda()][:, torch.from_numpy(rw).cuda()].float().cpu().numpy()
    gemm_check(got, ref, bound, True, "405B fprop")


# ---------------------------------------------------------------------------
# Shapes off the 128 x 128 x 256 tile grid: any M and N, K % 64 == 0.  The
# output sits inside a larger buffer (ldd > N, extra rows) filled with a
# sentinel, which must survive: the clipped stores write only M x N.
# ---------------------------------------------------------------------------
RAGGED = [(200, 72, 320), (1, 128, 256), (130, 1000, 64), (257, 136, 192), (129, 264, 448), (3, 8, 128),
          (384, 520, 832)]


def _ragged_operands(M, N, K, seed):
    a = torch.from_numpy(synthetic.normal((M, K), 1.0, seed)).to(torch.bfloat16)
    b = torch.from_numpy(synthetic.normal((N, K), 0.02, seed + 1)).to(torch.bfloat16)
    qa, ra = quantize_both(a)
    qb, rb = quantize_both(b, block="2d" if N % 16 == 0 else "1d")
    return qa, ra, qb, rb


@pytest.mark.parametrize("M,N,K", RAGGED)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_gemm_ragged_shapes(M, N, K, out_dtype):
    qa, ra, qb, rb = _ragged_operands(M, N, K, 7 * M + N + K)
    pad = 16 // (2 if out_dtype == torch.bfloat16 else 4)
    big = torch.full((M + 5, N + pad), -7.0, dtype=out_dtype, device="cuda")
    nv.gemm(qa, qb, out=big[:M, :N])
    nv.sync_check()
    full = big.float().cpu().numpy()
    ref, bound = oracle.gemm_reference(ra, rb)
    gemm_check(full[:M, :N], ref, bound, out_dtype == torch.bfloat16, f"{M}x{N}x{K}")
    assert (full[:M, N:] == -7.0).all(), "write past N"
    assert (full[M:] == -7.0).all(), "write past M"


@pytest.mark.parametrize("M,N,K", [(200, 72, 320), (130, 1000, 64), (1, 128, 256)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_gemm_amax_ragged(M, N, K, out_dtype):
    """The producer amax covers exactly the M x N stored values."""
    qa, ra, qb, rb = _ragged_operands(M, N, K, 11 * M + N + K)
    d, amax = nv.gemm_amax(qa, qb, out_dtype=out_dtype)
    nv.sync_check()
    assert float(amax.cpu()[0]) == float(d.float().abs().max().cpu())


def test_gemm_k_zero_writes_zeros():
    a, b = nv.NVFP4Tensor.empty(40, 0), nv.NVFP4Tensor.empty(24, 0)
    for t in (a, b):
        t.global_scale.fill_(1.0)
    big = torch.full((40, 32), -7.0, dtype=torch.float32, device="cuda")
    nv.gemm(a, b, out=big[:, :24])
    nv.sync_check()
    full = big.cpu().numpy()
    assert (full[:, :24] == 0).all() and (full[:, 24:] == -7.0).all()


def test_gemm_grouped_ragged_experts():
    """Routed experts with token counts that are not multiples of 128 (and one
    expert with no tokens), as MoE routing produces."""
    Ms = [1, 130, 0, 200, 512, 77, 384, 5]
    N, K = 136, 320
    qa, qb, ra, rb = [], [], [], []
    for e, M in enumerate(Ms):
        b = torch.from_numpy(synthetic.normal((N, K), 0.02, 300 + e)).to(torch.bfloat16)
        y, yr = quantize_both(b)
        qb.append(y); rb.append(yr)
        if M == 0:
            qa.append(nv.NVFP4Tensor.empty(0, K)); ra.append(None)
            qa[-1].global_scale.fill_(1.0)
            continue
        a = torch.from_numpy(synthetic.normal((M, K), 1.0, 400 + e)).to(torch.bfloat16)
        x, xr = quantize_both(a)
        qa.append(x); ra.append(xr)
    outs = [torch.full((M, N), -7.0, dtype=torch.bfloat16, device="cuda") for M in Ms]
    nv.gemm_grouped(qa, qb, out_dtype=torch.bfloat16, out=outs)
    nv.sync_check()
    for e, M in enumerate(Ms):
        if M == 0:
            continue
        ref, bound = oracle.gemm_reference(ra[e], rb[e])
        gemm_check(outs[e].float().cpu().numpy(), ref, bound, True, f"expert {e} (M={M})")
