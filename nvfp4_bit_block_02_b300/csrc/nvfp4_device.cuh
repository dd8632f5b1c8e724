// Device helpers of the NVFP4 kernels (sm_103a).  Every fp32 operation that
// decides a code or a scale is an explicit IEEE intrinsic (__fmul_rn,
// __fdiv_rn, __frcp_rn, __fadd_rn, __fsub_rn, and one __fmaf_ru whose exact
// result is rounded upward on purpose) or a packed PTX operation with an
// explicit rounding mode (add/sub/mul/fma .rn.f32x2).  A packed product that
// rounds is never an operand of a later addition (where it could be fused):
// it feeds conversions, stores, bit-pattern arithmetic or the multiplicand of
// an fma; the packed products inside the transform are exact (by +-1 or
// +-1/4).  Where a rounded product feeds a difference (the Four-over-Six block
// error) the operations stay scalar.  The encoder's results are therefore
// fixed bit for bit by the sequence written in nvfp4.h.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace nvfp4 {

// --------------------------------------------------------------------------
// Element formats
// --------------------------------------------------------------------------

// Eight fp32 values -> eight E2M1 codes, round to nearest even, saturating at
// +-6.  Byte j of the result holds code(x[2j]) in its low nibble and
// code(x[2j+1]) in its high nibble (the cvt puts its first operand high).
__device__ __forceinline__ uint32_t e2m1x8_rne(const float* x) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]), "f"(x[7]));
  return r;
}

// fp32 (>= 0) -> E4M3 byte, round to nearest even, saturating at 448.
__device__ __forceinline__ uint32_t e4m3_rne_sat(float t) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(t));
  return r & 0xFFu;
}

// E4M3 byte (sign clear, not NaN) -> fp32, exact: the hardware conversion to
// f16 (every E4M3 value is an f16), then to f32.
__device__ __forceinline__ float e4m3_value(uint32_t b) {
  uint32_t h;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h) : "r"(b & 0xFFu));
  return __low2float(*reinterpret_cast<const __half2*>(&h));
}

// Stochastic rounding of a = |q| to an E2M1 magnitude index with a 16-bit
// uniform number u, given as nu = 65535 - u: neighbours lo <= a < hi on the
// grid, frac = (a - lo) / (hi - lo), round up iff u < fl(frac * 65536);
// a >= 6 saturates.  Write idx(a) for the grid position of a (0, 0.5, 1, 1.5,
// 2, 3, 4, 6 sit at 0..7; linear in between), so the result is
// floor(idx) + [u < frac * 65536] with frac = idx - floor(idx).  For an
// integer u that is (ceil(T) + 65535 - u) >> 16 with T = 65536 * idx (exact):
// ceil(T) + nu reaches the next multiple of 65536 iff ceil(frac * 65536) > u.
// T itself: on [0, 1) the grid is uniform, T = 131072 * a, and ceil(T) comes
// from one fma rounded upward onto the integer grid of [2^23, 2^24); on
// [1, 8) every binade holds two grid steps, so T is linear in the float's
// bit pattern: T = (bits(a) - bits(0.5)) / 64, ceil(T) = (bits(a) - bits(0.5)
// + 63) >> 6.  Above 6 (and at infinity) the min saturates to index 7.
__device__ __forceinline__ uint32_t e2m1_sr_index(float a, uint32_t nu) {
  const uint32_t tl = __float_as_uint(__fmaf_ru(a, 131072.0f, 8388608.0f)) - 0x4B000000u;
  const uint32_t tg = (__float_as_uint(a) - 0x3F000000u + 63u) >> 6;
  return min(((a < 1.0f ? tl : tg) + nu) >> 16, 7u);
}

// Decode: y = fl(fl(value(code) * s) * g), two codes at a time.  The values
// of a code byte come from one hardware conversion to f16x2 (every E2M1 value
// is an f16); value * s is formed in f32 by a mixed-precision fma with f16
// multiplicands, exact because every |value * s| lies in [2^-10, 2688] with at
// most 6 significant bits (adding -0 keeps the sign of a zero product); the
// product with g is one packed IEEE multiply.
//
// (s, s) in f16 from an E4M3 scale byte with its sign bit clear (exact).
__device__ __forceinline__ uint32_t e4m3_f16x2_splat(uint32_t b) {
  uint32_t h;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h) : "r"(b * 0x101u));
  return h;
}
// The 16 codes of a block (byte p = codes 2p, 2p+1, low nibble first) as 8
// f16x2 words of their values; the vector move hands each byte to its
// conversion without a shift.
__device__ __forceinline__ void e2m1x16_f16x2(uint2 c, uint32_t h[8]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3, b4, b5, b6, b7;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %8;\n\t"
      "mov.b32 {b4, b5, b6, b7}, %9;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t"
      "cvt.rn.f16x2.e2m1x2 %4, b4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %5, b5;\n\t"
      "cvt.rn.f16x2.e2m1x2 %6, b6;\n\t"
      "cvt.rn.f16x2.e2m1x2 %7, b7;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3]), "=r"(h[4]), "=r"(h[5]), "=r"(h[6]), "=r"(h[7])
      : "r"(c.x), "r"(c.y));
}
// fl(fl(v * s) * g) for the two values of f16x2 word h, s from e4m3_f16x2_splat.
__device__ __forceinline__ float2 decode_pair(uint32_t h, uint32_t s2, float2 g2) {
  float lo, hi;
  asm("{\n\t.reg .b16 v0, v1, sc, sd;\n\t"
      "mov.b32 {v0, v1}, %2;\n\t"
      "mov.b32 {sc, sd}, %3;\n\t"
      "fma.rn.f32.f16 %0, v0, sc, 0f80000000;\n\t"
      "fma.rn.f32.f16 %1, v1, sc, 0f80000000;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(h), "r"(s2));
  float2 p;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(p.x), "=f"(p.y)
      : "f"(lo), "f"(hi), "f"(g2.x), "f"(g2.y));
  return p;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// --------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): the published round
// multipliers and Weyl key increments.
// --------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

// The 16 rounding draws of the 16 elements starting at output-orientation
// linear index i0 (i0 % 16 == 0): element e draws half (e & 1) of word
// (e % 8) / 2 of the call with counter i0 / 8 + e / 8.  Returned
// complemented, nu[e] = 65535 - u[e], the form e2m1_sr_index takes.
__device__ __forceinline__ void sr_draws16(uint64_t seed, uint64_t offset, uint64_t i0, uint32_t nu[16]) {
  uint64_t j = i0 >> 3;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint64_t jj = j + h;
    uint4 w = philox4x32_10(make_uint4((uint32_t)jj, (uint32_t)(jj >> 32), (uint32_t)offset, (uint32_t)(offset >> 32)),
                            (uint32_t)seed, (uint32_t)(seed >> 32));
    const uint32_t c[4] = {~w.x, ~w.y, ~w.z, ~w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      nu[8 * h + 2 * k] = c[k] & 0xFFFFu;
      nu[8 * h + 2 * k + 1] = c[k] >> 16;
    }
  }
}

// Sign mask of the Hadamard transform: bit i set -> sigma_i = -1.
__device__ __forceinline__ uint32_t rht_sign_mask(uint64_t rht_seed) {
  uint4 w = philox4x32_10(make_uint4(0u, 0x80000000u, 0u, 0u), (uint32_t)rht_seed, (uint32_t)(rht_seed >> 32));
  return w.x & 0xFFFFu;
}

// Packed fp32x2 multiply, each lane an IEEE round-to-nearest-even product
// with subnormals kept (PTX with an explicit rounding mode).  Used only where
// the product feeds a conversion, never an addition, so no fused
// multiply-add can form from it.
__device__ __forceinline__ float2 mul2_rn(float2 a, float2 b) {
  float2 r;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
// Packed fp32x2 IEEE arithmetic (round to nearest even per lane).
__device__ __forceinline__ float2 add2_rn(float2 a, float2 b) {
  float2 r;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
__device__ __forceinline__ float2 sub2_rn(float2 a, float2 b) {
  float2 r;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
// a * b + c with one rounding per lane
__device__ __forceinline__ float2 fma2_rn(float2 a, float2 b, float2 c) {
  float2 r;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return r;
}

// In-place 16-point Walsh-Hadamard butterfly (Sylvester order) on two
// vectors at once (lanes .x and .y).
__device__ __forceinline__ void wht16x2(float2 v[16]) {
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; i += 2 * h) {
#pragma unroll
      for (int j = i; j < i + h; ++j) {
        const float2 a = v[j], b = v[j + h];
        v[j] = add2_rn(a, b);
        v[j + h] = sub2_rn(a, b);
      }
    }
  }
}

// Split constant of a chunk whose largest magnitude is m (finite, below
// 2^124): c = 1.5 * 2^(E+4), E the binary exponent of m.  For |x| <= m,
// x + c stays in c's binade, whose spacing is 2^(E-19).
__device__ __forceinline__ float rht_split_const(float m) {
  return __uint_as_float(((((__float_as_uint(m) >> 23) & 0xFFu) + 4u) << 23) | 0x400000u);
}

// Running maximum of |y| over the transformed chunks of a whole warp, exact,
// for the amax pass (every lane of the warp calls it together; `run_max` and
// the result are the same in every lane).  A plain fp32 butterfly comes
// first: with P = H16 * diag(sigma) * x (so y = P / 4), each of its outputs is
// within 2^-18 * max|x| of the exact P (four rounded stages over partial sums
// bounded by 16 * max|x|), and max|P| >= ||P||_2 / 4 = ||x||_2 >= max|x|
// (H16 * H16^T = 16 I), so the plain maximum m of |P| bounds the exact maximum
// of |y| by m / 4 * (1 + 2^-17).  Only when a lane's bound could reach the
// warp's exact maximum so far are that lane's chunks transformed exactly
// (rare once the maximum has grown).
__device__ __forceinline__ float rht16x2_absmax(float v[2][16], uint32_t sign_mask, float run_max);

// v[h] <- 1/4 * H16 * diag(sigma) * v[h] for the two 16-element chunks h = 0, 1,
// correctly rounded: every result is the fp32 value nearest the exact one.
//   Each input is split exactly as x = hi + lo, hi = x rounded to a multiple
//   of 2^(E-19) (E the exponent of the chunk's largest |x|, through
//   t = fl(sigma*x + c), c = 1.5 * 2^(E+4)), lo = sigma*x - hi.  hi has at most
//   20 significant bits below 2^(E+1), so every partial sum of its butterfly
//   (below 2^(E+5), a multiple of 2^(E-19)) is an fp32 value: the butterfly of
//   hi is exact.  |lo| <= 2^(E-20), and lo keeps the bits of x below the hi
//   grid, so the butterfly of lo is exact whenever the chunk's smallest
//   nonzero |x| is within 2^-33 (BF16 input) or 2^-17 (FP32 input) of its
//   largest.  The result is then fl(1/4 * Ylo + 1/4 * Yhi), one rounding of
//   the exact value.  (Outside that range the lo butterfly rounds at 2^-40
//   of the chunk maximum.)  The sign diagonal rides in the first fma.
__device__ __forceinline__ void rht16x2(float v[2][16], uint32_t sign_mask) {
  float m0 = 0.0f, m1 = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    m0 = fmaxf(m0, fabsf(v[0][i]));
    m1 = fmaxf(m1, fabsf(v[1][i]));
  }
  const float2 c = make_float2(rht_split_const(m0), rht_split_const(m1));
  float2 nh[16], lo[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float sg = ((sign_mask >> i) & 1u) ? -1.0f : 1.0f;
    const float2 x = make_float2(v[0][i], v[1][i]), sgn = make_float2(sg, sg);
    const float2 t = fma2_rn(x, sgn, c);  // fl(sigma*x + c)
    nh[i] = sub2_rn(c, t);                // -hi, exact (t and c share a binade)
    lo[i] = fma2_rn(x, sgn, nh[i]);       // sigma*x - hi, exact
  }
  wht16x2(nh);
  wht16x2(lo);
  const float2 q = make_float2(0.25f, 0.25f), nq = make_float2(-0.25f, -0.25f);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float2 y = fma2_rn(lo[i], q, mul2_rn(nh[i], nq));  // one rounding of (Ylo + Yhi) / 4
    v[0][i] = y.x;
    v[1][i] = y.y;
  }
}

__device__ __forceinline__ float rht16x2_absmax(float v[2][16], uint32_t sign_mask, float run_max) {
  float2 p[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float sg = ((sign_mask >> i) & 1u) ? -1.0f : 1.0f;
    p[i] = mul2_rn(make_float2(v[0][i], v[1][i]), make_float2(sg, sg));
  }
  wht16x2(p);
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) m = fmaxf(m, fmaxf(fabsf(p[i].x), fabsf(p[i].y)));
  // m / 4 is the plain maximum; the exact one is at most m / 4 * (1 + 2^-17)
  const bool need = __fmul_rn(m, 0.25f * (1.0f + 0x1p-16f)) >= run_max;
  if (__any_sync(0xFFFFFFFFu, need)) {
    float e = 0.0f;
    if (need) {
      rht16x2(v, sign_mask);
#pragma unroll
      for (int i = 0; i < 16; ++i) e = fmaxf(e, fmaxf(fabsf(v[0][i]), fabsf(v[1][i])));
    }
    // non-negative floats order like their bit patterns
    run_max = fmaxf(run_max, __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(e))));
  }
  return run_max;
}

// --------------------------------------------------------------------------
// Scale factors
// --------------------------------------------------------------------------

// Byte offset of logical scale (r, kb) in the 128x4-atom layout; n_katoms =
// ceil(K / 64).
__device__ __forceinline__ int64_t sf_offset(int64_t r, int64_t kb, int64_t n_katoms) {
  return ((r >> 7) * n_katoms + (kb >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (kb & 3);
}

// Per-tensor decode scale g = fl(amax / 2688), 1 for an all-zero tensor.
__device__ __forceinline__ float global_scale(float amax) { return amax == 0.0f ? 1.0f : __fdiv_rn(amax, 2688.0f); }

// One candidate block scale for grid maximum m: returns the E4M3 byte and
// sets its value s, the decode scale S = fl(s*g) and r = fl(1/S) (0 if S = 0).
__device__ __forceinline__ uint32_t block_scale(float amax_b, float mg, float g, float& s, float& rcp) {
  uint32_t b = e4m3_rne_sat(__fdiv_rn(amax_b, mg));
  s = e4m3_value(b);
  float S = __fmul_rn(s, g);
  rcp = (S == 0.0f) ? 0.0f : __frcp_rn(S);
  return b;
}

// Encode 16 values with block reciprocal rcp into two 32-bit words of codes
// (u: the complemented draws of sr_draws16, used only with SR).
// The products are paired into packed fp32x2 multiplies (each lane an IEEE
// round-to-nearest product, the same value as a scalar multiply).
template <bool SR>
__device__ __forceinline__ uint2 encode16(const float v[16], float rcp, const uint32_t* u) {
  float q[16];
  const float2 rr = make_float2(rcp, rcp);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float2 p = mul2_rn(make_float2(v[2 * i], v[2 * i + 1]), rr);
    q[2 * i] = p.x;
    q[2 * i + 1] = p.y;
  }
  const uint2 rne = make_uint2(e2m1x8_rne(q), e2m1x8_rne(q + 8));
  if constexpr (!SR) {
    return rne;
  } else {
    // magnitudes from stochastic rounding; each code's sign bit is q's sign,
    // which the round-to-nearest codes already carry (bit 3 of every nibble)
    uint32_t w0 = rne.x & 0x88888888u, w1 = rne.y & 0x88888888u;
#pragma unroll
    for (int i = 0; i < 8; ++i) w0 += e2m1_sr_index(fabsf(q[i]), u[i]) << (4 * i);
#pragma unroll
    for (int i = 0; i < 8; ++i) w1 += e2m1_sr_index(fabsf(q[8 + i]), u[8 + i]) << (4 * i);
    return make_uint2(w0, w1);
  }
}

// value * s for the two values of f16x2 word h (s from e4m3_f16x2_splat),
// exact in f32: mixed-precision fma with f16 multiplicands, adding -0.
__device__ __forceinline__ float2 scaled_pair(uint32_t h, uint32_t s2) {
  float2 r;
  asm("{\n\t.reg .b16 v0, v1, sc, sd;\n\t"
      "mov.b32 {v0, v1}, %2;\n\t"
      "mov.b32 {sc, sd}, %3;\n\t"
      "fma.rn.f32.f16 %0, v0, sc, 0f80000000;\n\t"
      "fma.rn.f32.f16 %1, v1, sc, 0f80000000;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "r"(h), "r"(s2));
  return r;
}

// Squared error of 16 encoded values against their decode fl(fl(v*s)*g),
// pairwise summed: ((e0+e1)+(e2+e3)) + ... over the 16 in order; s is the
// E4M3 scale byte.  Scalar IEEE operations with explicit rounding (a packed
// product feeding a packed difference was seen to change the result on the
// B300 for a few near-tie blocks, consistent with the two being fused).
__device__ __forceinline__ float block_sq_err16(const float v[16], uint2 codes, uint32_t sbyte, float g) {
  const uint32_t s2 = e4m3_f16x2_splat(sbyte & 0x7Fu);
  uint32_t h[8];
  e2m1x16_f16x2(codes, h);
  float e[16];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float2 vs = scaled_pair(h[j], s2);
    const float d0 = __fsub_rn(v[2 * j], __fmul_rn(vs.x, g));
    const float d1 = __fsub_rn(v[2 * j + 1], __fmul_rn(vs.y, g));
    e[2 * j] = __fmul_rn(d0, d0);
    e[2 * j + 1] = __fmul_rn(d1, d1);
  }
#pragma unroll
  for (int w = 1; w < 16; w <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; i += 2 * w) e[i] = __fadd_rn(e[i], e[i + w]);
  }
  return e[0];
}

}  // namespace nvfp4
