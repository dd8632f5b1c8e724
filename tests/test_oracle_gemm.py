"""Pins of the oracle GEMM reference: brute force on tiny inputs, exactly
representable products checked in integer arithmetic, and the closed form
of an all-ones product."""
import numpy as np
import torch

import oracle
from synthetic import normal


def _q(oracle_mod, codes, scales, g, R, K):
    return oracle_mod.Quantized(codes.astype(np.uint8), scales.astype(np.uint8), 0.0, g, None, None, R, K)


def test_gemm_all_ones_closed_form(oracle_mod):
    """Every code 1.0 (0x2), every scale 1.0 (0x38), g = 1: D = K."""
    for M, N, K in [(4, 3, 64), (2, 5, 256)]:
        a = _q(oracle_mod, np.full((M, K // 2), 0x22), np.full((M, K // 16), 0x38), 1.0, M, K)
        b = _q(oracle_mod, np.full((N, K // 2), 0x22), np.full((N, K // 16), 0x38), 1.0, N, K)
        d, bound = oracle_mod.gemm_reference(a, b)
        assert (d == K).all() and (bound == K).all()


def test_gemm_exact_integer_products(oracle_mod):
    """Codes restricted to integer values and scales to powers of two >= 1
    with power-of-two g: every product is an integer times a power of two, so
    the result is exact and must equal Python integer arithmetic."""
    rng = np.random.default_rng(4)
    M, N, K = 6, 7, 256
    int_codes = np.array([0, 2, 4, 5, 6, 7, 8, 10, 12, 13, 14, 15], np.uint8)   # 0, +-1, +-2, +-3, +-4, +-6
    ca = rng.choice(int_codes, size=(M, K))
    cb = rng.choice(int_codes, size=(N, K))
    pack = lambda c: (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)
    pow2_scales = np.array([0x38, 0x40, 0x48, 0x50], np.uint8)                 # 1, 2, 4, 8
    sa = rng.choice(pow2_scales, size=(M, K // 16))
    sb = rng.choice(pow2_scales, size=(N, K // 16))
    a = _q(oracle_mod, pack(ca), sa, 0.5, M, K)
    b = _q(oracle_mod, pack(cb), sb, 4.0, N, K)
    d, _ = oracle_mod.gemm_reference(a, b)
    val = {0: 0, 1: 1, 2: 2, 3: 3, 4: 4, 6: 6}
    mag = [0, None, 1, None, 2, 3, 4, 6]          # integer magnitudes only
    sdec = {0x38: 1, 0x40: 2, 0x48: 4, 0x50: 8}
    for m in range(M):
        for n in range(N):
            acc = 0
            for k in range(K):
                va = mag[ca[m, k] & 7] * (-1 if ca[m, k] & 8 else 1) * sdec[int(sa[m, k // 16])]
                vb = mag[cb[n, k] & 7] * (-1 if cb[n, k] & 8 else 1) * sdec[int(sb[n, k // 16])]
                acc += va * vb
            assert d[m, n] == acc * 0.5 * 4.0


def test_gemm_brute_force_tiny(oracle_mod):
    """Triple loop over the dequantized values (fp64) on quantized random data."""
    A = normal((5, 64), 1.0, 21)
    B = normal((3, 64), 0.02, 22)
    qa = oracle_mod.quantize(A)
    qb = oracle_mod.quantize(B)
    ya = oracle_mod.dequantize(qa.codes, qa.scales, qa.g).astype(np.float64)
    yb = oracle_mod.dequantize(qb.codes, qb.scales, qb.g).astype(np.float64)
    d, bound = oracle_mod.gemm_reference(qa, qb)
    for m in range(5):
        for n in range(3):
            s = 0.0
            t = 0.0
            for k in range(64):
                s += ya[m, k] * yb[n, k]
                t += abs(ya[m, k] * yb[n, k])
            # dequantize rounds code*s*g once to fp32: relative 2^-24 per term
            assert abs(d[m, n] - s) <= 2 ** -23 * t + 1e-300
            assert abs(bound[m, n] - t) <= 2 ** -23 * t
    # the rows= subset equals the corresponding rows of the full product (up to
    # the fp64 summation order of the matmul)
    d2, b2 = oracle_mod.gemm_reference(qa, qb, rows=np.array([4, 1]))
    assert (np.abs(d2 - d[[4, 1]]) <= 1e-14 * b2).all()


# ---------------------------------------------------------------------------
# W4A16 reference: BF16 rounding and the product with the BF16 weights
# ---------------------------------------------------------------------------
def test_bf16_round_matches_torch():
    rng = np.random.default_rng(11)
    x = np.concatenate([(rng.standard_normal(200000) * 10.0 ** rng.integers(-30, 30, 200000)).astype(np.float32),
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.005859375, 3.4e38, 1e-40], dtype=np.float32)])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    got = oracle.bf16_round(x)
    assert (got.view(np.uint32) == want.view(np.uint32)).all()


def test_w4a16_reference_brute_force():
    """Tiny case against a Python loop over exact rationals."""
    from fractions import Fraction
    rng = np.random.default_rng(12)
    M, N, K = 2, 3, 32
    x = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)).to(torch.bfloat16).float().numpy()
    qw = oracle.quantize(rng.standard_normal((N, K)).astype(np.float32))
    w = oracle.bf16_round(oracle.dequantize(qw.codes, qw.scales, qw.g))
    d, bound = oracle.w4a16_reference(x, qw)
    for m in range(M):
        for n in range(N):
            exact = sum(Fraction(float(x[m, k])) * Fraction(float(w[n, k])) for k in range(K))
            assert abs(float(exact) - d[m, n]) <= 1e-12 * max(1.0, bound[m, n])


def test_w4a16_reference_constant_weights_closed_form():
    """A constant weight tensor decodes to one value c everywhere, so each
    output is c times the row sum of X."""
    rng = np.random.default_rng(13)
    qw = oracle.quantize(np.full((48, 64), 0.3, dtype=np.float32))
    w = oracle.bf16_round(oracle.dequantize(qw.codes, qw.scales, qw.g))
    c = float(w[0, 0])
    assert (w == np.float32(c)).all() and abs(c - 0.3) < 0.3 / 64
    x = torch.from_numpy(rng.standard_normal((5, 64)).astype(np.float32)).to(torch.bfloat16).float().numpy()
    d, _ = oracle.w4a16_reference(x, qw)
    want = c * x.astype(np.float64).sum(axis=1)
    assert np.allclose(d, want[:, None], rtol=0, atol=1e-12)
