/*
 * Plain CPU oracle for the NVFP4 quantizer, dequantizer and the scale-factor
 * layout.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg load this file's library; the product path
 * never does.  It shares no code, header or table with the CUDA library.
 *
 * Sources (page title, then section):
 *  - "NVIDIA Introduces a 4-Bit Pretraining Methodology Using NVFP4 ..."
 *    (aissential.tech), "Summary": 16-element blocks, an E4M3 scale per block,
 *    an FP32 per-tensor scale.  "Method": 2D 16x16 weight scaling, 16x16
 *    Random Hadamard Transforms on Wgrad inputs, stochastic rounding on
 *    gradients.
 *  - hyper.ai story "NVIDIA présente NVFP4 ..." (single paragraph): two-level
 *    micro-scaling; the Hadamard transform smooths outliers; stochastic
 *    rounding keeps gradients unbiased.
 *  - hyper.ai story on the Nemotron 3 Ultra NVFP4 checkpoint (single
 *    paragraph): Four-over-Six scaling switches per block between two grid
 *    maxima to lower the rounding error.
 *  - Philox4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As
 *    Easy as 1, 2, 3", SC'11.
 *
 * Where the pages are silent the readings are written beside the code that
 * takes them.  Every float operation marked fl() below is one IEEE binary32
 * operation with round-to-nearest-even; the file is compiled with
 * -ffp-contract=off so that the compiler fuses none of them.
 *
 * Deliberately slow: every rounding is an exhaustive nearest search over the
 * target format's values, every transform a plain matrix-vector product.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* E2M1 element code: sign bit 3, magnitude index in bits 0..2.             */
/* Magnitude index c -> value: 0, 0.5, 1, 1.5, 2, 3, 4, 6.                  */
/* ------------------------------------------------------------------------ */
static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

float oracle_e2m1_decode(uint8_t code) {
  double m = E2M1_MAG[code & 7];
  return (float)((code & 8) ? -m : m);
}

/* Round-to-nearest, ties to the even code, saturating at 6: exhaustive search
 * over the 8 magnitudes.  The sign bit is copied from q, so -0.1 -> 0x8. */
uint8_t oracle_e2m1_encode_rne(float q) {
  uint8_t sign = signbit(q) ? 8 : 0;
  double a = fabs((double)q);
  if (!(a < 6.0)) return sign | 7; /* |q| >= 6 (and +-inf) saturate */
  int best = 0;
  double bestd = a; /* distance to 0 */
  for (int c = 1; c < 8; ++c) {
    double d = fabs(a - E2M1_MAG[c]);
    if (d < bestd || (d == bestd && (c & 1) == 0 && (best & 1) == 1)) {
      best = c;
      bestd = d;
    }
  }
  return sign | (uint8_t)best;
}

/* Stochastic rounding of q between its two neighbouring grid magnitudes.
 * Reading (the pages say only "stochastic rounding" and "unbiased"):
 *   lo <= |q| < hi neighbours on the grid, frac = fl(fl(|q|-lo)/fl(hi-lo))
 *   (both exact: the step is a power of two), round up iff
 *   u16 < fl(frac * 65536), u16 a uniform 16-bit integer.
 *   |q| >= 6 saturates to 6; a value on the grid never moves. */
uint8_t oracle_e2m1_encode_sr(float q, uint32_t u16) {
  uint8_t sign = signbit(q) ? 8 : 0;
  float a = fabsf(q);
  if (!(a < 6.0f)) return sign | 7;
  int lo = 0;
  for (int c = 1; c < 8; ++c)
    if ((double)a >= E2M1_MAG[c]) lo = c;
  int hi = lo + 1; /* exists: a < 6 */
  float flo = (float)E2M1_MAG[lo], fhi = (float)E2M1_MAG[hi];
  float frac = (a - flo) / (fhi - flo);
  float thr = frac * 65536.0f;
  int up = (float)u16 < thr;
  return sign | (uint8_t)(up ? hi : lo);
}

/* ------------------------------------------------------------------------ */
/* E4M3 (bias 7, no infinities, 0x7F is NaN): value of a byte.               */
/* ------------------------------------------------------------------------ */
float oracle_e4m3_decode(uint8_t b) {
  int e = (b >> 3) & 15, m = b & 7;
  double v;
  if ((b & 0x7F) == 0x7F) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9); /* subnormal: m * 2^-9 */
  else
    v = ldexp(1.0 + m / 8.0, e - 7);
  return (float)((b & 0x80) ? -v : v);
}

/* Round-to-nearest-even with saturation at 448 (never NaN); exhaustive search
 * over the 127 non-negative finite codes.  Codes are ordered like their
 * values, so "ties to even" means the even byte. */
uint8_t oracle_e4m3_encode_rne_sat(float t) {
  uint8_t sign = signbit(t) ? 0x80 : 0;
  double a = fabs((double)t);
  if (a >= 448.0) return sign | 0x7E;
  int best = 0;
  double bestd = a;
  for (int b = 1; b <= 0x7E; ++b) {
    double d = fabs(a - (double)oracle_e4m3_decode((uint8_t)b));
    if (d < bestd || (d == bestd && (b & 1) == 0 && (best & 1) == 1)) {
      best = b;
      bestd = d;
    }
  }
  return sign | (uint8_t)best;
}

/* ------------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon et al., SC'11): 10 rounds of the 4x32 S-box with the */
/* published multipliers and Weyl key increments.                          */
/* ------------------------------------------------------------------------ */
void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
  uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
  uint32_t k0 = key_in[0], k1 = key_in[1];
  for (int round = 0; round < 10; ++round) {
    uint64_t p0 = (uint64_t)M0 * c0;
    uint64_t p1 = (uint64_t)M1 * c2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    k0 += W0;
    k1 += W1;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Uniform 16-bit number for the element at output-orientation linear index i
 * (i = row * K + k).  Reading: eight elements share one Philox call with
 * counter (j_lo, j_hi, offset_lo, offset_hi), j = i / 8; element i takes
 * 16-bit half (i & 1) of word (i % 8) / 2, the high half for odd i. */
uint32_t oracle_sr_bits(uint64_t seed, uint64_t offset, uint64_t i) {
  uint64_t j = i / 8;
  uint32_t ctr[4] = {(uint32_t)j, (uint32_t)(j >> 32), (uint32_t)offset, (uint32_t)(offset >> 32)};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t w[4];
  oracle_philox4x32_10(ctr, key, w);
  uint32_t word = w[(i % 8) / 2];
  return (i & 1) ? (word >> 16) : (word & 0xFFFFu);
}

/* Random +-1 signs of the Hadamard transform.  Reading: one sign vector per
 * call, sigma_i = -1 iff bit i of word 0 of Philox(key = rht_seed,
 * ctr = (0, 0x80000000, 0, 0)); the rounding stream never reaches counter
 * word 1 = 2^31 (it would need 2^66 elements). */
void oracle_rht_signs(uint64_t rht_seed, int sign_out[16]) {
  uint32_t ctr[4] = {0u, 0x80000000u, 0u, 0u};
  uint32_t key[2] = {(uint32_t)rht_seed, (uint32_t)(rht_seed >> 32)};
  uint32_t w[4];
  oracle_philox4x32_10(ctr, key, w);
  for (int i = 0; i < 16; ++i) sign_out[i] = ((w[0] >> i) & 1u) ? -1 : 1;
}

/* Sylvester Hadamard entry H16[i][j] = (-1)^popcount(i & j). */
int oracle_hadamard16(int i, int j) {
  int p = __builtin_popcount((unsigned)(i & j));
  return (p & 1) ? -1 : 1;
}

/* y = 1/4 * H16 * diag(sigma) * x for one 16-chunk, in fp64, then rounded
 * once to fp32.  Reading: orthonormal scaling 1/4, sign diagonal applied
 * before H. */
void oracle_rht16(const float x[16], const int sigma[16], float y[16]) {
  for (int i = 0; i < 16; ++i) {
    double acc = 0.0;
    for (int j = 0; j < 16; ++j) acc += (double)oracle_hadamard16(i, j) * (double)sigma[j] * (double)x[j];
    y[i] = (float)(0.25 * acc);
  }
}

/* Pairwise sum in fp32 over n = 2^p terms: sum(a[0:n]) = sum(a[0:n/2]) +
 * sum(a[n/2:n]).  The CUDA side must use the same tree. */
static float pairwise_sum_f32(const float* a, int n) {
  if (n == 1) return a[0];
  float l = pairwise_sum_f32(a, n / 2);
  float r = pairwise_sum_f32(a + n / 2, n / 2);
  return l + r;
}

/* Logical element (r, k) of the output-orientation matrix. */
static inline float elem(const float* v, int64_t r, int64_t k, int64_t K) { return v[r * K + k]; }

/*
 * The quantizer.  Inputs are fp32 values (a BF16 input is upcast exactly by
 * the caller).  x is row-major [rows][ld].  The output orientation is
 * R x K with K = cols (transpose = 0) or R = cols, K = rows (transpose = 1,
 * i.e. x^T is quantized, its rows are the input's columns).
 *
 *  1. V = the output-orientation matrix; with rht != 0 every 16-chunk of a
 *     row of V along K is replaced by oracle_rht16 of it.
 *  2. amax = max |V| (or *amax_in), g = fl(amax / 2688) (g = 1 if amax = 0).
 *  3. Per block (1x16 along K, or a 16x16 tile when block2d):
 *       amax_b = max |v|;  candidates m = 6 (and m = 4 with four_over_six):
 *       s_m = E4M3(fl(amax_b / fl(m*g))), S_m = fl(s_m*g),
 *       r_m = S_m == 0 ? 0 : fl(1/S_m), code = E2M1(fl(v*r_m)) (RNE or SR).
 *     Four-over-Six keeps m = 4 iff err_4 < err_6, where
 *       err = pairwise sum over the block (row-major in a tile) of
 *             fl(d*d), d = fl(v - deq), deq = fl(fl(value(code)*s)*g).
 *  4. codes: byte (r, j) = code(r, 2j) | code(r, 2j+1) << 4;
 *     scales: logical [R][K/16] E4M3 bytes (a 2D tile's byte repeated on its
 *     16 rows).
 *
 * choice (nullable): per logical scale entry, 1 if max-4 won, else 0.
 * transformed (nullable): the fp32 matrix V that was encoded, [R][K].
 * Returns 0, or -1 on a shape the format does not allow.
 */
int oracle_quantize(const float* x, int64_t rows, int64_t cols, int64_t ld, int transpose, int block2d,
                    int stochastic, int four_over_six, int rht, uint64_t seed, uint64_t offset,
                    uint64_t rht_seed, const float* amax_in, uint8_t* codes, uint8_t* scales,
                    float* amax_out, float* g_out, uint8_t* choice, float* transformed) {
  int64_t R = transpose ? cols : rows;
  int64_t K = transpose ? rows : cols;
  if (K % 16 != 0 || (block2d && R % 16 != 0) || R < 0 || K < 0) return -1;
  int64_t KB = K / 16;

  /* step 1: V */
  float* V = (float*)malloc(sizeof(float) * (size_t)(R * K > 0 ? R * K : 1));
  if (!V) return -1;
  for (int64_t r = 0; r < R; ++r)
    for (int64_t k = 0; k < K; ++k) V[r * K + k] = transpose ? x[k * ld + r] : x[r * ld + k];
  if (rht) {
    int sigma[16];
    oracle_rht_signs(rht_seed, sigma);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r)
      for (int64_t kb = 0; kb < KB; ++kb) {
        float in[16], out[16];
        memcpy(in, V + r * K + kb * 16, sizeof in);
        oracle_rht16(in, sigma, out);
        memcpy(V + r * K + kb * 16, out, sizeof out);
      }
  }
  if (transformed) memcpy(transformed, V, sizeof(float) * (size_t)(R * K));

  /* step 2: per-tensor scale */
  float amax = 0.0f;
  if (amax_in) {
    amax = *amax_in;
  } else {
    for (int64_t e = 0; e < R * K; ++e) {
      float a = fabsf(V[e]);
      if (a > amax) amax = a;
    }
  }
  float g = (amax == 0.0f) ? 1.0f : amax / 2688.0f;
  *amax_out = amax;
  *g_out = g;

  /* step 3: blocks.  A block is a list of element positions (row-major). */
  int64_t TR = block2d ? R / 16 : R; /* block rows */
  int bh = block2d ? 16 : 1;         /* block height */
  int n = 16 * bh;                   /* elements per block */
#pragma omp parallel for schedule(static)
  for (int64_t br = 0; br < TR; ++br) {
    float vals[256];
    uint32_t ubits[256];
    uint8_t cand_codes[2][256];
    for (int64_t kb = 0; kb < KB; ++kb) {
      float amax_b = 0.0f;
      for (int i = 0; i < bh; ++i)
        for (int j = 0; j < 16; ++j) {
          int64_t r = br * bh + i, k = kb * 16 + j;
          float v = elem(V, r, k, K);
          vals[i * 16 + j] = v;
          if (fabsf(v) > amax_b) amax_b = fabsf(v);
          ubits[i * 16 + j] = stochastic ? oracle_sr_bits(seed, offset, (uint64_t)(r * K + k)) : 0u;
        }
      int ncand = four_over_six ? 2 : 1;
      const float mult[2] = {6.0f, 4.0f};
      uint8_t s_c[2];
      float err[2];
      for (int c = 0; c < ncand; ++c) {
        float mg = mult[c] * g;
        float t = amax_b / mg;
        uint8_t s = oracle_e4m3_encode_rne_sat(t);
        float sv = oracle_e4m3_decode(s);
        float S = sv * g;
        float rcp = (S == 0.0f) ? 0.0f : 1.0f / S;
        float sq[256];
        for (int e = 0; e < n; ++e) {
          float q = vals[e] * rcp;
          uint8_t code = stochastic ? oracle_e2m1_encode_sr(q, ubits[e]) : oracle_e2m1_encode_rne(q);
          cand_codes[c][e] = code;
          float deq = (oracle_e2m1_decode(code) * sv) * g;
          float d = vals[e] - deq;
          sq[e] = d * d;
        }
        s_c[c] = s;
        err[c] = pairwise_sum_f32(sq, n);
      }
      int pick = (four_over_six && err[1] < err[0]) ? 1 : 0;
      for (int i = 0; i < bh; ++i) {
        int64_t r = br * bh + i;
        scales[r * KB + kb] = s_c[pick];
        if (choice) choice[r * KB + kb] = (uint8_t)pick;
        for (int j = 0; j < 8; ++j) {
          uint8_t lo = cand_codes[pick][i * 16 + 2 * j];
          uint8_t hi = cand_codes[pick][i * 16 + 2 * j + 1];
          codes[r * (K / 2) + kb * 8 + j] = (uint8_t)(lo | (hi << 4));
        }
      }
    }
  }
  free(V);
  return 0;
}

/* Dequantize: y(r, k) = fl(fl(value(code) * s_b) * g) (the first product is
 * exact: at most 6 significant bits).  scales are logical [R][K/16]. */
void oracle_dequantize(const uint8_t* codes, const uint8_t* scales, float g, int64_t R, int64_t K, float* y) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < R; ++r)
    for (int64_t k = 0; k < K; ++k) {
      uint8_t byte = codes[r * (K / 2) + k / 2];
      uint8_t code = (k & 1) ? (byte >> 4) : (byte & 15);
      float sv = oracle_e4m3_decode(scales[r * (K / 16) + k / 16]);
      float p = oracle_e2m1_decode(code) * sv;
      y[r * K + k] = p * g;
    }
}

/*
 * Physical scale-factor layout (the tensor-core scale tile): the logical
 * [R][K/16] matrix is cut into 128-row x 4-column atoms of 512 bytes; atom
 * (R/128 index a_r, K/64 index a_k) starts at byte (a_r * ceil(K/64) + a_k) * 512
 * and holds entry (r, kb) at (r % 32) * 16 + ((r % 128) / 32) * 4 + kb % 4.
 * Padding rows/columns are zero.  Size: ceil(R/128)*128 * ceil(K/64)*4 bytes.
 */
int64_t oracle_scales_bytes(int64_t R, int64_t K) {
  int64_t rp = (R + 127) / 128 * 128;
  int64_t kbp = ((K / 16) + 3) / 4 * 4;
  return rp * kbp;
}

void oracle_swizzle_scales(const uint8_t* logical, int64_t R, int64_t K, uint8_t* physical) {
  int64_t KB = K / 16;
  int64_t n_ka = (KB + 3) / 4;
  memset(physical, 0, (size_t)oracle_scales_bytes(R, K));
  for (int64_t r = 0; r < R; ++r)
    for (int64_t kb = 0; kb < KB; ++kb) {
      int64_t atom = (r / 128) * n_ka + kb / 4;
      int64_t off = atom * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + kb % 4;
      physical[off] = logical[r * KB + kb];
    }
}
