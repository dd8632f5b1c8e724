"""Pins of the oracle's element formats (E2M1, E4M3), the Philox stream and the
Hadamard transform against facts fixed outside the oracle: hand-worked
values, closed forms, an independent rounding construction, torch's FP8 cast
and Triton's Philox (run by its CPU interpreter)."""
import math
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


# ---------------------------------------------------------------- E2M1 ----
def test_e2m1_tie_table(oracle_mod):
    # midpoints between neighbours go to the even code (magnitude index)
    ties = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}
    for q, v in ties.items():
        code = oracle_mod.e2m1_encode_rne(q)
        assert oracle_mod.e2m1_decode(code) == v, (q, code)
        assert code & 1 == 0
        neg = oracle_mod.e2m1_encode_rne(-q)
        assert neg == (code | 8)


def test_e2m1_grid_saturation_and_sign(oracle_mod):
    for c, v in enumerate(GRID):
        assert oracle_mod.e2m1_encode_rne(v) == c
        assert oracle_mod.e2m1_decode(c) == v
        assert oracle_mod.e2m1_decode(c | 8) == -v
    for big in [6.0, 6.5, 7.0, 100.0, 3.0e38, math.inf]:
        assert oracle_mod.e2m1_encode_rne(big) == 7
        assert oracle_mod.e2m1_encode_rne(-big) == 15
    assert oracle_mod.e2m1_encode_rne(-0.1) == 8          # sign kept on a zero result
    assert oracle_mod.e2m1_encode_rne(-0.0) == 8
    assert oracle_mod.e2m1_encode_rne(0.0) == 0
    assert oracle_mod.e2m1_encode_rne(0.2499999) == 0
    assert oracle_mod.e2m1_encode_rne(0.2500001) == 1


def _e2m1_by_rint(a: np.ndarray) -> np.ndarray:
    """Independent construction: RNE onto the grid as three fixed-spacing
    pieces (0.5 on [0,2), 1 on [2,4), 2 on [4,6]) using numpy's rint
    (half to even integer), then saturation."""
    a = np.abs(a.astype(np.float64))
    v = np.where(a < 2.0, np.rint(a * 2.0) / 2.0, np.where(a < 4.0, np.rint(a), 2.0 * np.rint(a / 2.0)))
    # pieces meet at 2 and 4: rint(3.9*2)/2 = 4 etc. stay on the grid
    return np.minimum(v, 6.0)


def test_e2m1_against_independent_rounding(oracle_mod):
    rng = np.random.default_rng(11)
    # every bf16 value in [0, 8) plus random fp32 plus ties and their neighbours
    bf = (np.arange(0, 0x4100, dtype=np.uint32) << 16).view(np.float32)
    rnd = rng.uniform(0, 7, size=20000).astype(np.float32)
    mids = np.array([(GRID[i] + GRID[i + 1]) / 2 for i in range(7)], dtype=np.float32)
    near = np.concatenate([np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(10)), mids])
    qs = np.concatenate([bf, rnd, near]).astype(np.float32)
    want = _e2m1_by_rint(qs)
    got = np.array([oracle_mod.e2m1_decode(oracle_mod.e2m1_encode_rne(float(q))) for q in qs])
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(qs[i]), got[i], want[i]) for i in bad[:10]]


def test_e2m1_stochastic_exhaustive_probability(oracle_mod):
    """Over all 65536 values of u16 the up-probability is ceil(frac*2^16)/2^16:
    frac exactly on a value that is a multiple of 2^-16, unbiased to 2^-16."""
    lib = oracle_mod._load()
    cases = [0.1, 0.3, 0.6, 0.99, 1.2, 1.7, 2.25, 2.9, 3.3, 4.5, 5.99, 0.5 + 2 ** -20]
    u = np.arange(65536)
    for q in cases:
        q32 = float(np.float32(q))
        lo = max(v for v in GRID if v <= q32)
        hi = min(v for v in GRID if v > q32)
        frac = (q32 - lo) / (hi - lo)
        ups = sum(1 for x in u[::1] if oracle_mod.e2m1_decode(lib.oracle_e2m1_encode_sr(q32, int(x))) == hi)
        assert ups == math.ceil(frac * 65536), (q, ups, frac)
        mean = (ups * hi + (65536 - ups) * lo) / 65536
        assert 0 <= mean - q32 <= (hi - lo) * 2 ** -16 + 1e-12


def test_e2m1_stochastic_grid_values_never_move(oracle_mod):
    lib = oracle_mod._load()
    for c, v in enumerate(GRID):
        for u in [0, 1, 12345, 32768, 65535]:
            assert lib.oracle_e2m1_encode_sr(v, u) == c
            if v:
                assert lib.oracle_e2m1_encode_sr(-v, u) == (c | 8)
    for u in [0, 65535]:
        assert lib.oracle_e2m1_encode_sr(6.5, u) == 7
        assert lib.oracle_e2m1_encode_sr(1e30, u) == 7


# ---------------------------------------------------------------- E4M3 ----
def _e4m3_closed_form(b: int) -> float:
    e, m = (b >> 3) & 15, b & 7
    v = m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
    return -v if b & 0x80 else v


def test_e4m3_decode_all_codes(oracle_mod):
    for b in range(256):
        if b & 0x7F == 0x7F:
            assert math.isnan(oracle_mod.e4m3_decode(b))
        else:
            assert oracle_mod.e4m3_decode(b) == _e4m3_closed_form(b)
    assert oracle_mod.e4m3_decode(0x7E) == 448.0
    assert oracle_mod.e4m3_decode(0x01) == 2.0 ** -9


def test_e4m3_against_torch_cast_in_range(oracle_mod):
    """Cross-check with torch.float8_e4m3fn (RNE) for values below 464, where
    torch does not produce NaN."""
    rng = np.random.default_rng(5)
    vals = [_e4m3_closed_form(b) for b in range(0x7F)]
    mids = [(vals[i] + vals[i + 1]) / 2 for i in range(len(vals) - 1)]
    t = np.concatenate([
        (np.arange(0, 0x43E0, dtype=np.uint32) << 16).view(np.float32),  # bf16 values below 448
        rng.uniform(0, 460, 20000).astype(np.float32),
        np.exp2(rng.uniform(-14, 8.8, 20000)).astype(np.float32),
        np.array(mids, dtype=np.float32),
        np.nextafter(np.array(mids, dtype=np.float32), np.float32(0)),
        np.nextafter(np.array(mids, dtype=np.float32), np.float32(1000)),
    ]).astype(np.float32)
    t = t[t < 464]
    want = torch.from_numpy(t).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle_mod.e4m3_encode(float(x)) for x in t], dtype=np.uint8)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(t[i]), got[i], want[i]) for i in bad[:10]]


def test_e4m3_saturation_and_subnormals(oracle_mod):
    for big in [448.0, 448.5, 464.0, 465.0, 1e6, 3e38, math.inf]:
        assert oracle_mod.e4m3_encode(big) == 0x7E
    assert oracle_mod.e4m3_encode(2.0 ** -10) == 0x00          # tie 0 / 2^-9 -> even (0)
    assert oracle_mod.e4m3_encode(3 * 2.0 ** -10) == 0x02      # tie 2^-9 / 2^-8 -> even (2)
    assert oracle_mod.e4m3_encode(1.5 * 2.0 ** -10) == 0x01
    assert oracle_mod.e4m3_encode(0.0) == 0x00
    assert oracle_mod.e4m3_encode(1.0) == 0x38
    assert oracle_mod.e4m3_encode(1.0625) == 0x38              # tie 1 / 1.125 -> even
    assert oracle_mod.e4m3_encode(1.1875) == 0x3A              # tie 1.125 / 1.25 -> even


# ---------------------------------------------------------------- Philox --
_TRITON_SCRIPT = r"""
import os, sys, json
os.environ["TRITON_INTERPRET"] = "1"
import torch, triton, triton.language as tl

@triton.jit
def k(out_ptr, c_ptr, seed_lo, seed_hi, N: tl.constexpr):
    i = tl.arange(0, N)
    c0 = tl.load(c_ptr + i * 4 + 0); c1 = tl.load(c_ptr + i * 4 + 1)
    c2 = tl.load(c_ptr + i * 4 + 2); c3 = tl.load(c_ptr + i * 4 + 3)
    k0 = tl.full((N,), seed_lo, tl.uint32); k1 = tl.full((N,), seed_hi, tl.uint32)
    a, b, c, d = tl.random.philox_impl(c0.to(tl.uint32, bitcast=True), c1.to(tl.uint32, bitcast=True),
                                       c2.to(tl.uint32, bitcast=True), c3.to(tl.uint32, bitcast=True), k0, k1)
    tl.store(out_ptr + i * 4 + 0, a.to(tl.int32, bitcast=True))
    tl.store(out_ptr + i * 4 + 1, b.to(tl.int32, bitcast=True))
    tl.store(out_ptr + i * 4 + 2, c.to(tl.int32, bitcast=True))
    tl.store(out_ptr + i * 4 + 3, d.to(tl.int32, bitcast=True))

cases = json.loads(sys.stdin.read())
res = []
for key, ctrs in cases:
    c = torch.tensor(ctrs, dtype=torch.int64).to(torch.uint32).view(torch.int32).reshape(-1)
    n = len(ctrs)
    out = torch.zeros(n * 4, dtype=torch.int32)
    k[(1,)](out, c, key[0], key[1], N=n)
    res.append([x & 0xffffffff for x in out.tolist()])
print(json.dumps(res))
"""


def test_philox_against_triton_interpreter(oracle_mod):
    """Triton ships an independent Philox4x32-10 (the Salmon et al. rounds);
    its CPU interpreter runs it without a GPU."""
    import json
    rng = np.random.default_rng(3)
    cases = []
    for key in [(0, 0), (1, 0), (0xFFFFFFFF, 0xFFFFFFFF), (0x12345678, 0x9ABCDEF0)]:
        ctrs = [[0, 0, 0, 0], [1, 0, 0, 0], [0, 0x80000000, 0, 0], [0xFFFFFFFF] * 4]
        ctrs += rng.integers(0, 2 ** 32, size=(12, 4)).tolist()
        cases.append([list(key), ctrs])
    env = dict(os.environ, TRITON_INTERPRET="1")
    p = subprocess.run([sys.executable, "-c", _TRITON_SCRIPT], input=json.dumps(cases), capture_output=True,
                       text=True, env=env, timeout=600)
    if p.returncode != 0:
        pytest.fail("triton interpreter failed: " + p.stderr[-2000:])
    ref = json.loads(p.stdout.strip().splitlines()[-1])
    for (key, ctrs), words in zip(cases, ref):
        for j, ctr in enumerate(ctrs):
            got = oracle_mod.philox4x32_10(ctr, key).tolist()
            assert got == words[4 * j:4 * j + 4], (key, ctr)


def test_philox_sr_stream_uniform(oracle_mod):
    """The 16-bit rounding draws are uniform: chi-square over 16 bins of the
    top nibble, and a mean of u16 near 32767.5."""
    lib = oracle_mod._load()
    n = 40000
    u = np.array([lib.oracle_sr_bits(1, 0, i) for i in range(n)], dtype=np.int64)
    assert u.max() <= 0xFFFF
    hist = np.bincount(u >> 12, minlength=16)
    chi2 = ((hist - n / 16) ** 2 / (n / 16)).sum()
    assert chi2 < 45.0  # 15 dof, p ~ 1e-4
    assert abs(u.mean() - 32767.5) < 6 * 18918 / math.sqrt(n)
    # eight consecutive elements share one Philox call, halves low/high
    w = oracle_mod.philox4x32_10([0, 0, 0, 0], [1, 0])
    assert [int(x) for x in u[:8]] == [int(w[k // 2] >> (16 * (k & 1)) & 0xFFFF) for k in range(8)]


# ---------------------------------------------------------------- RHT -----
def test_hadamard_orthogonality(oracle_mod):
    H = oracle_mod.hadamard16()
    assert (H @ H.T == 16 * np.eye(16, dtype=np.int64)).all()
    assert (H == H.T).all()
    assert set(np.unique(H)) == {-1, 1}


def test_rht_unit_vectors_and_norm(oracle_mod):
    H = oracle_mod.hadamard16()
    sigma = oracle_mod.rht_signs(1)
    assert set(sigma.tolist()) <= {-1, 1}
    for i in range(16):
        e = np.zeros(16, np.float32)
        e[i] = 1.0
        y = oracle_mod.rht16(e, sigma)
        assert (y == sigma[i] * H[:, i] / 4.0).all()
    rng = np.random.default_rng(0)
    for _ in range(200):
        x = rng.standard_normal(16).astype(np.float32) * rng.uniform(1e-3, 1e3)
        y = oracle_mod.rht16(x, sigma).astype(np.float64)
        assert abs(np.linalg.norm(y) - np.linalg.norm(x.astype(np.float64))) <= 1e-6 * np.linalg.norm(x)


def test_rht_signs_depend_on_seed(oracle_mod):
    s = {tuple(oracle_mod.rht_signs(seed).tolist()) for seed in range(8)}
    assert len(s) == 8
