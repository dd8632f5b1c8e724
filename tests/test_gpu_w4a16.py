"""Weight-only GEMM (W4A16) parity on the GPU against the oracle's float64
product of the BF16 activations with the BF16-rounded dequantized weights:
|y - y_ref| <= 1e-5 * sum_k |x||w_hat| (plus half a BF16 ulp of y_ref for BF16
output).  Weights come either from random code and scale bytes (every code,
every finite scale) or from the GPU quantizer checked bit-exact against the
oracle's quantization first, so both sides start from the same NVFP4 bytes."""
import numpy as np
import pytest
import torch

import nvfp4_bit_block_02_b300 as nv
import oracle
import synthetic
from tests.gpu_helpers import Guarded, assert_same_quantized, gemm_check, oracle_quantize_like

pytestmark = pytest.mark.gpu


def random_weight(N: int, K: int, seed: int, g: float = None):
    """Random NVFP4 bytes: all 16 codes, scale bytes 0..0x7E (0x7F is NaN)."""
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    scales = rng.integers(0, 0x7F, (N, K // 16), dtype=np.uint8)
    if g is None:
        g = float(np.float32(rng.uniform(1e-4, 1e-2)))
    ref = oracle.Quantized(codes, scales, 0.0, g, None, None, N, K)
    phys = oracle.swizzle_scales(scales, N, K)
    q = nv.NVFP4Tensor(torch.from_numpy(codes).cuda(), torch.from_numpy(phys).cuda(),
                       torch.tensor([g], dtype=torch.float32, device="cuda"),
                       torch.tensor([0.0], dtype=torch.float32, device="cuda"), N, K)
    return q, ref


def bf16_activations(M: int, ld: int, seed: int) -> torch.Tensor:
    return synthetic.to_bf16(synthetic.normal((M, ld), 1.0, seed))


def run(x_cpu: torch.Tensor, q: nv.NVFP4Tensor, out_dtype, ldy: int = None):
    """y = w4a16_gemm(x[:, :K], q) with x's row stride kept (ldx = x's width)
    and y written into an ldy-wide guarded buffer."""
    M, N, K = x_cpu.shape[0], q.rows, q.cols
    ldy = N if ldy is None else ldy
    es = 2 if out_dtype == torch.bfloat16 else 4
    buf = Guarded(max(M * ldy * es, 1))
    y_full = buf.view[:M * ldy * es].view(out_dtype).view(M, ldy)
    x = x_cpu.cuda()[:, :K]
    y = nv.w4a16_gemm(x, q, out=y_full[:, :N])
    nv.sync_check()
    buf.check()
    return y.float().cpu().numpy(), y_full


def activations_f32(x_cpu: torch.Tensor, K: int) -> np.ndarray:
    return synthetic.bf16_to_f32_numpy(x_cpu[:, :K].contiguous())


@pytest.mark.parametrize("M", [1, 3, 4, 5, 16, 40])
@pytest.mark.parametrize("N,K", [(1, 16), (200, 48), (256, 4096), (77, 4112), (77, 4160), (33, 96), (130, 288)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_w4a16_random_bytes(M, N, K, out_dtype):
    q, ref = random_weight(N, K, M * 1000 + N + K)
    x = bf16_activations(M, K, M + 7 * K)
    y, _ = run(x, q, out_dtype)
    y_ref, bound = oracle.w4a16_reference(activations_f32(x, K), ref)
    gemm_check(y, y_ref, bound, out_dtype == torch.bfloat16, f"W4A16 {M}x{N}x{K}")


def test_w4a16_identity_activations_reproduce_the_bf16_decode():
    """x = I: y[m][n] = W_hat[n][m] exactly (one nonzero product per sum),
    so the in-kernel decode must equal the BF16 dequantization bit for bit."""
    N, K = 200, 64
    q, ref = random_weight(N, K, 11)
    x = torch.eye(K, dtype=torch.bfloat16)
    y, _ = run(x, q, torch.float32)
    w_hat = oracle.bf16_round(oracle.dequantize(ref.codes, ref.scales, ref.g))
    np.testing.assert_array_equal(y, w_hat.T)


@pytest.mark.parametrize("K", [96, 80, 256])
def test_w4a16_unit_rows_reproduce_the_bf16_decode_at_small_m(K):
    """x = 8 rows of I at a time (the single-token-tile launches, K % 32 == 0
    or not): y[m][n] = W_hat[n][m0 + m] bit for bit, every K position once."""
    N = 72
    q, ref = random_weight(N, K, 13 + K)
    w_hat = oracle.bf16_round(oracle.dequantize(ref.codes, ref.scales, ref.g))
    eye = torch.eye(K, dtype=torch.bfloat16)
    for m0 in range(0, K, 8):
        y, _ = run(eye[m0:m0 + 8].contiguous(), q, torch.float32)
        np.testing.assert_array_equal(y, w_hat[:, m0:m0 + 8].T, err_msg=f"K={K} rows {m0}..{m0 + 7}")


def test_w4a16_closed_form_all_ones():
    """Codes 0x22 (value 1), scales 0x38 (1.0), g = 1, x = 1: y = K exactly."""
    N, K = 96, 2048
    codes = np.full((N, K // 2), 0x22, np.uint8)
    scales = np.full((N, K // 16), 0x38, np.uint8)
    q = nv.NVFP4Tensor(torch.from_numpy(codes).cuda(), torch.from_numpy(oracle.swizzle_scales(scales, N, K)).cuda(),
                       torch.tensor([1.0], device="cuda"), torch.tensor([0.0], device="cuda"), N, K)
    y, _ = run(torch.ones((5, K), dtype=torch.bfloat16), q, torch.float32)
    assert (y == K).all()


@pytest.mark.parametrize("block", ["1d", "2d"])
def test_w4a16_quantized_weight(block):
    """A weight quantized on the GPU (checked bit-exact against the oracle)
    times BF16 activations, strided x and y."""
    M, N, K = 9, 384, 1024
    w = synthetic.to_bf16(synthetic.normal((N, K), 0.02, 3))
    q = nv.quantize(w.cuda(), block=block)
    torch.cuda.synchronize()
    ref = oracle_quantize_like(w, block2d=block == "2d")
    assert_same_quantized(q, ref, "W4A16 weight")
    x = bf16_activations(M, K + 64, 4)
    y, y_full = run(x, q, torch.bfloat16, ldy=N + 8)
    y_ref, bound = oracle.w4a16_reference(activations_f32(x, K), ref)
    gemm_check(y, y_ref, bound, True, "W4A16 quantized weight")
    # the padding columns of y are not written
    pad = y_full[:, N:].contiguous().view(torch.uint8).cpu().numpy()
    assert (pad == 0xA5).all()


def test_w4a16_empty_and_zero_k():
    q, _ = random_weight(64, 64, 1)
    y = nv.w4a16_gemm(torch.empty((0, 64), dtype=torch.bfloat16, device="cuda"), q)
    nv.sync_check()
    assert y.shape == (0, 64)
    q0 = nv.NVFP4Tensor(torch.empty((32, 0), dtype=torch.uint8, device="cuda"),
                        torch.empty(0, dtype=torch.uint8, device="cuda"), torch.ones(1, device="cuda"),
                        torch.zeros(1, device="cuda"), 32, 0)
    y = nv.w4a16_gemm(torch.empty((3, 0), dtype=torch.bfloat16, device="cuda"), q0, out_dtype=torch.float32)
    nv.sync_check()
    assert (y.cpu() == 0).all()


@pytest.mark.parametrize("M", [1, 4, 16])
def test_w4a16_llama8b_decode_sampled(M):
    """The Llama-3-8B MLP up-projection weight (14336 x 4096) at decode-sized
    M, in the bench's launch configuration; every output column of a sample
    of 512 weight rows checked."""
    N, K = 14336, 4096
    q, ref = random_weight(N, K, 8 + M)
    x = bf16_activations(M, K, 80 + M)
    y = nv.w4a16_gemm(x.cuda(), q)
    nv.sync_check()
    y = y.float().cpu().numpy()
    sel = np.sort(np.random.default_rng(M).choice(N, 512, replace=False))
    sub = oracle.Quantized(ref.codes[sel], ref.scales[sel], 0.0, ref.g, None, None, len(sel), K)
    y_ref, bound = oracle.w4a16_reference(activations_f32(x, K), sub)
    gemm_check(y[:, sel], y_ref, bound, True, f"W4A16 8B decode M={M}")
