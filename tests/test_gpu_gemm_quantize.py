"""The GEMM whose epilogue emits the next layer's NVFP4 input (the producer
side of the recipe's just-in-time quantization; "NVIDIA Introduces a 4-Bit
Pretraining Methodology Using NVFP4").  Its codes, scales, g and amax must be
bit-exact with the oracle's quantization (1D, RNE, max-6) of the BF16 output
that nvfp4_gemm writes, with the same supplied tensor amax; the BF16 output
it stores must equal nvfp4_gemm's bit for bit."""
import numpy as np
import pytest
import torch

import nvfp4_bit_block_02_b300 as nv
import oracle
import synthetic
from tests.gpu_helpers import assert_same_quantized, guarded_tensor

pytestmark = pytest.mark.gpu


def _operands(M, N, K, seed):
    a = torch.from_numpy(synthetic.normal((M, K), 1.0, seed)).to(torch.bfloat16).cuda()
    b = torch.from_numpy(synthetic.normal((N, K), 0.02, seed + 1)).to(torch.bfloat16).cuda()
    return nv.quantize(a), nv.quantize(b, block="2d" if N % 16 == 0 else "1d")


def _rows_logical_scales(phys: np.ndarray, K: int, rows: np.ndarray) -> np.ndarray:
    KB = K // 16
    nka = (KB + 3) // 4
    r = rows.astype(np.int64)[:, None]
    kb = np.arange(KB, dtype=np.int64)[None, :]
    return phys[((r >> 7) * nka + (kb >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (kb & 3)]


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (200, 144, 320), (130, 1040, 64), (384, 528, 512), (1, 16, 64),
                                   (512, 1536, 1024)])
@pytest.mark.parametrize("amax_factor", [1.0, 2.0, 0.5])
def test_gemm_quantize_matches_quantize_of_the_bf16_output(M, N, K, amax_factor):
    qa, qb = _operands(M, N, K, 13 * M + N + K)
    d_ref, amax_true = nv.gemm_amax(qa, qb, out_dtype=torch.bfloat16)
    amax_in = amax_true * amax_factor          # exact bound, loose bound, or values that saturate
    out, bufs = guarded_tensor(M, N)
    d = torch.full((M, N + 8), -7.0, dtype=torch.bfloat16, device="cuda")
    amax_out = torch.zeros(1, dtype=torch.float32, device="cuda")
    nv.gemm_quantize(qa, qb, amax_in, out=out, d=d[:, :N], amax_out=amax_out)
    nv.sync_check()
    for b in bufs:
        b.check()
    assert torch.equal(d[:, :N], d_ref), "stored BF16 output differs from nvfp4_gemm's"
    assert (d[:, N:] == -7.0).all(), "write past N"
    assert float(amax_out.cpu()[0]) == float(amax_true.cpu()[0])
    ref = oracle.quantize(d_ref.float().cpu().numpy(), amax=float(amax_in.cpu()[0]))
    assert_same_quantized(out, ref, f"gemm_quantize {M}x{N}x{K} amax x{amax_factor}")


def test_gemm_quantize_without_storing_d():
    qa, qb = _operands(256, 512, 512, 5)
    d_ref, amax = nv.gemm_amax(qa, qb, out_dtype=torch.bfloat16)
    out = nv.gemm_quantize(qa, qb, amax)
    nv.sync_check()
    assert_same_quantized(out, oracle.quantize(d_ref.float().cpu().numpy(), amax=float(amax.cpu()[0])), "no D")


def test_gemm_quantize_llama8b_full_size_sampled():
    """Llama-3-8B fprop (8192 x 14336 x 4096): the epilogue encoding of the
    whole output, checked on sampled rows (all 14336 columns) against the
    oracle's quantization of the BF16 output with the producer amax."""
    wl = synthetic.llama8b_fprop()
    qx = nv.quantize(wl.tensors["X"].cuda())
    qw = nv.quantize(wl.tensors["W"].cuda(), block="2d")
    d, amax = nv.gemm_amax(qx, qw, out_dtype=torch.bfloat16)
    out = nv.gemm_quantize(qx, qw, amax)
    nv.sync_check()
    a = float(amax.cpu()[0])
    rng = np.random.default_rng(8)
    rows = np.unique(np.concatenate([np.arange(128), np.arange(8192 - 128, 8192), rng.choice(8192, 128, replace=False)]))
    ref = oracle.quantize(d[torch.from_numpy(rows).cuda()].float().cpu().numpy(), amax=a)
    assert float(out.amax.cpu()[0]) == a and float(out.global_scale.cpu()[0]) == ref.g
    codes = out.codes.cpu().numpy()[rows]
    assert (codes == ref.codes).all(), f"{int((codes != ref.codes).sum())} code bytes differ"
    sc = _rows_logical_scales(out.scales.cpu().numpy(), 14336, rows)
    assert (sc == ref.scales).all(), f"{int((sc != ref.scales).sum())} scale bytes differ"
