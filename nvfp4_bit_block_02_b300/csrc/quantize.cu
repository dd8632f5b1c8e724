// NVFP4 quantizer kernels for sm_103a: tensor amax, row-wise (K = cols)
// and transposed (K = rows) encoders with 1D/2D blocks, stochastic rounding,
// Four-over-Six and the 16x16 Random Hadamard Transform, and the decoder.
//
// Format and recipe: "NVIDIA Introduces a 4-Bit Pretraining Methodology Using
// NVFP4" ("Summary": 16-element blocks, E4M3 block scales, FP32 tensor scale;
// "Method": 2D 16x16 weight blocks, RHT on Wgrad inputs, SR on gradients);
// Four-over-Six: the hyper.ai story on the Nemotron 3 Ultra NVFP4 checkpoint.
//
// The kernels are HBM-bound, except the encodes with stochastic rounding plus
// the RHT and with Four-over-Six, which are bound by ALU issue (Philox draws,
// the exact transform, two candidate encodes).  Each CTA of an encoder owns
// one 128-row x 4-block tile of the output orientation, i.e. exactly one
// 512-byte atom of the scale layout, so every scale byte (padding included)
// is written by the encoder and no memset is needed.  Loads are 16-byte
// vectors; the transposed encoder stages a 64 x 128 input tile in shared
// memory (through a TMA ring, one tensor map per tensor or group; through
// registers only when a group's map cannot be built) and reads it back as
// column pairs (32-bit words), conflict-free.
#include <atomic>

#include "gemm.h"
#include "nvfp4_device.cuh"
#include "quantize.h"

namespace nvfp4 {

// ---------------------------------------------------------------------------
// Tensor amax: max |x| as the max of the magnitude bit patterns (non-negative
// floats order like unsigned integers), one atomicMax per CTA.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t absmax_bits(uint4 w, float) {
  uint32_t a = max(w.x & 0x7FFFFFFFu, w.y & 0x7FFFFFFFu);
  uint32_t b = max(w.z & 0x7FFFFFFFu, w.w & 0x7FFFFFFFu);
  return max(a, b);
}
__device__ __forceinline__ uint32_t absmax_bits(uint4 w, __nv_bfloat16) {
  uint32_t m = __vmaxu2(__vmaxu2(w.x & 0x7FFF7FFFu, w.y & 0x7FFF7FFFu), __vmaxu2(w.z & 0x7FFF7FFFu, w.w & 0x7FFF7FFFu));
  return max(m & 0xFFFFu, m >> 16) << 16;
}

__device__ __forceinline__ void cta_max_to_global(uint32_t m, unsigned int* out) {
  __shared__ uint32_t red[32];
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) red[warp] = m;
  __syncthreads();
  if (warp == 0) {
    m = lane < (int)(blockDim.x >> 5) ? red[lane] : 0u;
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if (lane == 0 && m) atomicMax(out, m);
  }
}

template <typename T>
__global__ void __launch_bounds__(256) k_amax(const T* __restrict__ x, int64_t rows, int64_t nvec, int64_t ld_vec,
                                              unsigned int* __restrict__ out) {
  const uint4* base = reinterpret_cast<const uint4*>(x);
  uint32_t m = 0;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
    const uint4* row = base + r * ld_vec;
    int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    // 8 loads in flight per thread (128 B), then their maxima; the last
    // (partial) batch issues its loads together as well
    for (; v + 7 * stride < nvec; v += 8 * stride) {
      uint4 q[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) q[i] = __ldg(row + v + i * stride);
#pragma unroll
      for (int i = 0; i < 8; ++i) m = max(m, absmax_bits(q[i], T()));
    }
    if (v < nvec) {
      uint4 q[7];
#pragma unroll
      for (int i = 0; i < 7; ++i) q[i] = v + i * stride < nvec ? __ldg(row + v + i * stride) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int i = 0; i < 7; ++i) m = max(m, absmax_bits(q[i], T()));
    }
  }
  cta_max_to_global(m, out);
}

// Loop-safe CTA max + one atomicMax (callable repeatedly in a CTA-uniform loop).
__device__ __forceinline__ void cta_max_atomic(uint32_t m, unsigned int* out) {
  __shared__ uint32_t red[8];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  __syncthreads();  // the previous call's reads of red[] are done
  if (lane == 0) red[warp] = m;
  __syncthreads();
  if (warp == 0) {
    m = lane < (int)(blockDim.x >> 5) ? red[lane] : 0u;
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if (lane == 0 && m) atomicMax(out, m);
  }
}

// Grouped tensor amax: tiles of amax_rows[e] input rows of group e; a CTA
// reduces a tile and folds it into the group's accumulator.
template <typename T>
__global__ void __launch_bounds__(256) k_amax_grouped(const __grid_constant__ GroupQuant g) {
  constexpr int VEC = 16 / sizeof(T);
  const uint32_t total = g.amax_start[g.count];
  uint32_t e = 0;  // t only grows, so the group search resumes where it stopped
  for (uint32_t t = blockIdx.x; t < total; t += gridDim.x) {
    while (t >= g.amax_start[e + 1]) ++e;
    const QuantArgs& a = g.a[e];
    const int64_t nvec = a.C_in / VEC, ldv = a.ld / VEC;
    const int64_t r0 = (int64_t)(t - g.amax_start[e]) * g.amax_rows[e];
    const int64_t r1 = min(r0 + (int64_t)g.amax_rows[e], a.R_in);
    const uint4* base = reinterpret_cast<const uint4*>(a.x);
    uint32_t m = 0;
    if (ldv == nvec) {
      // contiguous rows: the tile is one run of vectors, 8 loads per thread in flight
      const uint4* run = base + r0 * nvec;
      const int64_t n = (r1 - r0) * nvec;
      for (int64_t v = threadIdx.x; v < n; v += 8 * (int64_t)blockDim.x) {
        uint4 q[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int64_t j = v + i * (int64_t)blockDim.x;
          q[i] = j < n ? __ldg(run + j) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) m = max(m, absmax_bits(q[i], T()));
      }
    } else {
      for (int64_t r = r0; r < r1; ++r)
        for (int64_t v = threadIdx.x; v < nvec; v += blockDim.x) m = max(m, absmax_bits(__ldg(base + r * ldv + v), T()));
    }
    cta_max_atomic(m, reinterpret_cast<unsigned int*>(a.amax_accum));
  }
}

__global__ void k_zero_group_amax(const __grid_constant__ GroupQuant g) {
  if ((int)threadIdx.x < g.count) *g.a[threadIdx.x].amax_accum = 0.0f;
}

// ---------------------------------------------------------------------------
// Raw 16-element block loads (kept packed until used, so a thread can hold
// the next tile's blocks in flight while it encodes the current one).
// ---------------------------------------------------------------------------
template <typename T>
struct RawBlock;
template <>
struct RawBlock<__nv_bfloat16> {
  uint4 w[2];
  __device__ __forceinline__ void load(const void* p) {
    const uint4* q = reinterpret_cast<const uint4*>(p);
    w[0] = __ldg(q);
    w[1] = __ldg(q + 1);
  }
  __device__ __forceinline__ void zero() { w[0] = w[1] = make_uint4(0, 0, 0, 0); }
  __device__ __forceinline__ void unpack(float v[16]) const {
    const uint32_t u[8] = {w[0].x, w[0].y, w[0].z, w[0].w, w[1].x, w[1].y, w[1].z, w[1].w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[2 * i] = bf16_lo(u[i]);
      v[2 * i + 1] = bf16_hi(u[i]);
    }
  }
};
template <>
struct RawBlock<float> {
  uint4 w[4];
  __device__ __forceinline__ void load(const void* p) {
    const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = __ldg(q + i);
  }
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = make_uint4(0, 0, 0, 0);
  }
  __device__ __forceinline__ void unpack(float v[16]) const {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[4 * i] = __uint_as_float(w[i].x);
      v[4 * i + 1] = __uint_as_float(w[i].y);
      v[4 * i + 2] = __uint_as_float(w[i].z);
      v[4 * i + 3] = __uint_as_float(w[i].w);
    }
  }
};

__device__ __forceinline__ float absmax16(const float v[16]) {
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(v[i]));
  return m;
}

// ---------------------------------------------------------------------------
// Persistent tile walk: tile t of a tiles_y x tiles_x grid is (t / tiles_x,
// t % tiles_x); a CTA visits blockIdx.x, blockIdx.x + G, ... by adding
// (G / tiles_x, G % tiles_x) with one carry, so the loop divides nothing.
// ---------------------------------------------------------------------------
struct TileWalk {
  uint32_t tiles_x, dy, dx;
  __device__ TileWalk(uint32_t tx) : tiles_x(tx), dy(gridDim.x / tx), dx(gridDim.x % tx) {}
  __device__ void start(uint32_t& y, uint32_t& x) const {
    y = blockIdx.x / tiles_x;
    x = blockIdx.x % tiles_x;
  }
  __device__ void next(uint32_t y, uint32_t x, uint32_t& ny, uint32_t& nx) const {
    nx = x + dx;
    ny = y + dy;
    if (nx >= tiles_x) {
      nx -= tiles_x;
      ++ny;
    }
  }
};

// Tile sources of the persistent encoders.  OneTensor walks one tensor's
// tile grid with TileWalk; Groups walks the concatenated tile lists of up to
// kQuantGroups tensors (tile_start[] prefix sums), each with its own args.
struct OneTensor {
  static constexpr bool kGrouped = false;
  struct Ref {
    uint32_t ty, tx;
  };
  const QuantArgs& a;
  uint32_t tiles_y;
  TileWalk walk;
  __device__ OneTensor(const QuantArgs& args, uint32_t tiles_x, uint32_t ty) : a(args), tiles_y(ty), walk(tiles_x) {}
  __device__ const QuantArgs& args(const Ref&) const { return a; }
  __device__ bool first(Ref& r) const {
    walk.start(r.ty, r.tx);
    return r.ty < tiles_y;
  }
  __device__ bool next(const Ref& c, Ref& n) const {
    walk.next(c.ty, c.tx, n.ty, n.tx);
    return n.ty < tiles_y;
  }
};

struct Groups {
  static constexpr bool kGrouped = true;
  struct Ref {
    uint32_t t, e, ty, tx;
  };
  const GroupQuant& g;
  __device__ explicit Groups(const GroupQuant& gq) : g(gq) {}
  __device__ const QuantArgs& args(const Ref& r) const { return g.a[r.e]; }
  // e0: a group at or before tile t's (a CTA's tiles only move forward, so
  // the search resumes from the previous tile's group)
  __device__ bool locate(uint32_t t, Ref& r, uint32_t e0 = 0) const {
    if (t >= g.tile_start[g.count]) return false;
    uint32_t e = e0;
    while (t >= g.tile_start[e + 1]) ++e;
    const uint32_t local = t - g.tile_start[e];
    r.t = t;
    r.e = e;
    r.ty = local / g.tiles_x[e];
    r.tx = local % g.tiles_x[e];
    return true;
  }
  __device__ bool first(Ref& r) const { return locate(blockIdx.x, r); }
  __device__ bool next(const Ref& c, Ref& n) const { return locate(c.t + gridDim.x, n, c.e); }
  // the first tile of a group publishes its g and amax
  __device__ bool owns_scalars(const Ref& r) const { return r.t == g.tile_start[r.e]; }
};

// ---------------------------------------------------------------------------
// Row-wise encoder: K = cols.  Persistent: CTA b handles tiles b, b + G, ...
// of 128 rows x 4 blocks; thread t owns blocks (row t/4 + 64h, block t%4) of
// the tile, h = 0, 1, and loads the next tile's blocks before encoding the
// current ones.  A 2D tile's 16 rows are the 8-row groups of warps 2i and
// 2i+1 (lane bits 2..4 = row bits 0..2).  Index arithmetic is 32-bit (rows
// and 16-element blocks each fit in 31 bits); byte offsets are 64-bit.
// ---------------------------------------------------------------------------
template <typename T, bool B2D, bool SR, bool F46, bool RHT, bool AMAX_ONLY, class Src>
__device__ __forceinline__ void quant_rows_body(const Src& src, const QuantArgs& a0) {
  __shared__ float xw[8][2][4];    // cross-warp exchange for 2D tiles
  __shared__ float xw4[8][2][4];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const uint32_t kbl = t & 3, rl = t >> 2;
  uint32_t mask = 0;
  if constexpr (RHT) mask = rht_sign_mask(a0.rht_seed);
  // per-tensor scale: once for one tensor, per tile (its group's) for groups
  float g = 1.0f, g6 = 6.0f, g4 = 4.0f;
  auto set_scale = [&](const QuantArgs& a, bool publish) {
    const float amax = *a.amax_in;
    g = global_scale(amax);
    g6 = __fmul_rn(6.0f, g);
    g4 = __fmul_rn(4.0f, g);
    if (publish && t == 0) {
      *a.g_out = g;
      if (a.amax_out != a.amax_in) *a.amax_out = amax;
    }
  };
  if constexpr (!AMAX_ONLY && !Src::kGrouped) set_scale(a0, blockIdx.x == 0);
  float run_max = 0.0f;
  [[maybe_unused]] uint32_t scale_group = 0xFFFFFFFFu;  // the group whose scale g, g6, g4 hold

  auto load = [&](const typename Src::Ref& ref, RawBlock<T> (&raw)[2]) {
    const QuantArgs& a = src.args(ref);
    const uint32_t R = (uint32_t)a.R, KB = (uint32_t)(a.K / 16);
    const uint32_t kb = ref.tx * 4 + kbl;
    const T* __restrict__ xp = reinterpret_cast<const T*>(a.x);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t r = ref.ty * 128 + rl + 64 * h;
      if (r < R && kb < KB) raw[h].load(xp + (int64_t)r * a.ld + kb * 16);
      else raw[h].zero();
    }
  };

  RawBlock<T> cur[2], nxt[2];
  typename Src::Ref ref;
  bool have = src.first(ref);
  if (have) load(ref, cur);
  while (have) {
    typename Src::Ref nref;
    const bool have_next = src.next(ref, nref);
    if (have_next) load(nref, nxt);
    const QuantArgs& a = src.args(ref);
    const uint32_t R = (uint32_t)a.R, KB = (uint32_t)(a.K / 16), nka = (KB + 3) / 4;
    if constexpr (!AMAX_ONLY && Src::kGrouped) {
      const bool owns = src.owns_scalars(ref);
      if (owns || ref.e != scale_group) set_scale(a, owns);
      scale_group = ref.e;
    }
    float v[2][16];
    bool valid[2];
    uint32_t r[2];
    const uint32_t kb = ref.tx * 4 + kbl;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      r[h] = ref.ty * 128 + rl + 64 * h;
      valid[h] = r[h] < R && kb < KB;
      cur[h].unpack(v[h]);
    }
    if constexpr (RHT && !AMAX_ONLY) rht16x2(v, mask);
    if constexpr (AMAX_ONLY) {
      if constexpr (RHT) run_max = rht16x2_absmax(v, mask, run_max);
      else run_max = fmaxf(run_max, fmaxf(absmax16(v[0]), absmax16(v[1])));
    } else {
      float ab[2] = {absmax16(v[0]), absmax16(v[1])};
      if constexpr (B2D) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float m = ab[h];
          m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
          m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 8));
          m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 16));
          if (lane < 4) xw[warp][h][kbl] = m;
          ab[h] = m;
        }
        __syncthreads();
#pragma unroll
        for (int h = 0; h < 2; ++h) ab[h] = fmaxf(ab[h], xw[warp ^ 1][h][kbl]);
      }
      uint2 codes[2], c4[2];
      uint32_t sbyte[2], b4[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t u[16];
        if constexpr (SR) sr_draws16(a.seed, a.offset, (uint64_t)r[h] * (uint64_t)a.K + kb * 16, u);
        float s6, r6;
        sbyte[h] = block_scale(ab[h], g6, g, s6, r6);
        codes[h] = encode16<SR>(v[h], r6, u);
        if constexpr (F46) {
          float s4, r4;
          b4[h] = block_scale(ab[h], g4, g, s4, r4);
          c4[h] = encode16<SR>(v[h], r4, u);
        }
      }
      if constexpr (F46) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float e6 = block_sq_err16(v[h], codes[h], sbyte[h], g);
          float e4 = block_sq_err16(v[h], c4[h], b4[h], g);
          if constexpr (B2D) {
#pragma unroll
            for (int o = 4; o <= 16; o <<= 1) {
              e6 = __fadd_rn(e6, __shfl_xor_sync(0xFFFFFFFFu, e6, o));
              e4 = __fadd_rn(e4, __shfl_xor_sync(0xFFFFFFFFu, e4, o));
            }
            __syncthreads();  // xw reuse: every thread has read the previous exchange
            if (lane < 4) {
              xw[warp][h][kbl] = e6;
              xw4[warp][h][kbl] = e4;
            }
            __syncthreads();
            // tile sum = rows 0..7 + rows 8..15 (fp add commutes)
            e6 = __fadd_rn(e6, xw[warp ^ 1][h][kbl]);
            e4 = __fadd_rn(e4, xw4[warp ^ 1][h][kbl]);
          }
          if (e4 < e6) {
            codes[h] = c4[h];
            sbyte[h] = b4[h];
          }
        }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (valid[h]) {
          *reinterpret_cast<uint2*>(a.codes + (int64_t)r[h] * (a.K / 2) + kb * 8) = codes[h];
          if (a.tdebug) {
            float4* d = reinterpret_cast<float4*>(a.tdebug + (int64_t)r[h] * a.K + kb * 16);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              d[i] = make_float4(v[h][4 * i], v[h][4 * i + 1], v[h][4 * i + 2], v[h][4 * i + 3]);
          }
        }
        a.scales[sf_offset(r[h], kb, nka)] = valid[h] ? (uint8_t)sbyte[h] : (uint8_t)0;
      }
      if constexpr (B2D) __syncthreads();  // the exchange buffers are reused by the next tile
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) cur[h] = nxt[h];
    ref = nref;
    have = have_next;
  }
  if constexpr (AMAX_ONLY) cta_max_to_global(__float_as_uint(run_max), reinterpret_cast<unsigned int*>(a0.amax_accum));
}

template <typename T, bool B2D, bool SR, bool F46, bool RHT, bool AMAX_ONLY>
__global__ void __launch_bounds__(256) k_quant_rows(QuantArgs a) {
  const uint32_t KB = (uint32_t)(a.K / 16);
  const OneTensor src(a, (KB + 3) / 4, (uint32_t)((a.R + 127) / 128));
  quant_rows_body<T, B2D, SR, F46, RHT, AMAX_ONLY>(src, a);
}

// The plain BF16 1D encode (RNE, max-6, no transform) fits 64 registers: 4
// CTAs per SM, so a tensor's tiles split into more, shorter rounds (the 8B
// activation X: 6.9 tiles per CTA instead of 9.2, 17.0 -> 16.0 us).  The 2D
// encode at 64 registers ran 17 % more instructions and stays at 3.
__global__ void __launch_bounds__(256, 4) k_quant_rows_plain(QuantArgs a) {
  const uint32_t KB = (uint32_t)(a.K / 16);
  const OneTensor src(a, (KB + 3) / 4, (uint32_t)((a.R + 127) / 128));
  quant_rows_body<__nv_bfloat16, false, false, false, false, false>(src, a);
}

template <typename T, bool B2D, bool SR, bool F46>
__global__ void __launch_bounds__(256) k_quant_rows_grouped(const __grid_constant__ GroupQuant g) {
  const Groups src(g);
  quant_rows_body<T, B2D, SR, F46, false, false>(src, g.a[0]);
}
// (the plain BF16 1D case at 4 CTAs per SM, as k_quant_rows_plain)
__global__ void __launch_bounds__(256, 4) k_quant_rows_grouped_plain(const __grid_constant__ GroupQuant g) {
  const Groups src(g);
  quant_rows_body<__nv_bfloat16, false, false, false, false, false>(src, g.a[0]);
}

// ---------------------------------------------------------------------------
// Transposed encoder: x is [Tt][N] row-major, the output orientation is
// N x Tt (K = Tt).  Persistent over tiles of 64 input rows x 128 columns: the
// tile is staged in shared memory and read back as column pairs; thread t
// then owns output rows n0 + 2*(t%64) + {0, 1} and block t/64 of the tile.  The
// next tile's global loads are issued before the current tile is encoded.  A
// 2D tile (16 output rows) is 8 consecutive lanes (lane bits 0..2 = row-pair
// bits).
// ---------------------------------------------------------------------------
template <typename T>
struct ColTile;
template <>
struct ColTile<__nv_bfloat16> {
  static constexpr int kRowBytes = 256;  // 128 columns
  __device__ static void pair(const uint8_t* s, int tok, int np, float& lo, float& hi) {
    uint32_t w = reinterpret_cast<const uint32_t*>(s + tok * kRowBytes)[np];
    lo = bf16_lo(w);
    hi = bf16_hi(w);
  }
};
template <>
struct ColTile<float> {
  static constexpr int kRowBytes = 512;
  __device__ static void pair(const uint8_t* s, int tok, int np, float& lo, float& hi) {
    float2 f = reinterpret_cast<const float2*>(s + tok * kRowBytes)[np];
    lo = f.x;
    hi = f.y;
  }
};

// TMA ring of the single-tensor transposed encoder: 64 x 128-element input
// tiles (16 KB in BF16, 32 KB in FP32), 64 KB per CTA, so that the bytes in
// flight do not depend on the registers the encode needs.
template <typename T>
constexpr int kColStages = 65536 / (64 * ColTile<T>::kRowBytes);
template <typename T>
constexpr int kColRingBytes = kColStages<T> * 64 * ColTile<T>::kRowBytes;

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void bar_init(uint64_t* b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(b)), "r"(n));
}
__device__ __forceinline__ bool bar_test(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait (`limit` ns of global time): false on timeout.
__device__ __forceinline__ bool bar_wait(uint64_t* b, uint32_t parity, unsigned long long limit) {
  if (bar_test(b, parity)) return true;
  unsigned long long t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (uint32_t it = 1;; ++it) {
    if (bar_test(b, parity)) return true;
    if ((it & 63u) == 0) {
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      if (t - t0 > limit) return false;
    }
  }
}
// One 2D tile of x into shared memory, completion counted on `b`.
__device__ __forceinline__ void tile_load(void* dst, const CUtensorMap* tm, int x, int y, uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(b)), "r"(bytes) : "memory");
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_addr(b))
      : "memory");
}

// TMA: input tiles through the ring, from the single tensor's map `tm` or from
// each tile's group's map in the group arguments; otherwise staged through
// registers (a group whose map could not be built).
// hold_tx and wait_ns: the failure-detection test's withheld bytes on each
// CTA's first tile and its wait limit (both 0 in normal launches: 2 s).
template <typename T, bool B2D, bool SR, bool F46, bool RHT, bool AMAX_ONLY, bool TMA, class Src>
__device__ __forceinline__ void quant_cols_body(const Src& src, const QuantArgs& a0, const CUtensorMap* tm = nullptr,
                                                uint32_t hold_tx = 0, unsigned long long wait_ns = 0) {
  constexpr int RB = ColTile<T>::kRowBytes;
  constexpr int VPR = RB / 16;                  // 16-byte vectors per tile row
  constexpr int NV = TMA ? 1 : (64 * VPR) / 256;  // vectors per thread (register path)
  constexpr int S = kColStages<T>;
  __shared__ __align__(16) uint8_t tile_s[TMA ? 16 : 64 * RB];
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ uint64_t full[TMA ? S : 1];
  __shared__ int abort_s;
  const int t = threadIdx.x;
  const int np = t & 63, kbl = t >> 6;
  uint32_t mask = 0;
  if constexpr (RHT) mask = rht_sign_mask(a0.rht_seed);
  float g = 1.0f, g6 = 6.0f, g4 = 4.0f;
  auto set_scale = [&](const QuantArgs& a, bool publish) {
    const float amax = *a.amax_in;
    g = global_scale(amax);
    g6 = __fmul_rn(6.0f, g);
    g4 = __fmul_rn(4.0f, g);
    if (publish && t == 0) {
      *a.g_out = g;
      if (a.amax_out != a.amax_in) *a.amax_out = amax;
    }
  };
  if constexpr (!AMAX_ONLY && !Src::kGrouped) set_scale(a0, blockIdx.x == 0);
  float run_max = 0.0f;
  [[maybe_unused]] uint32_t scale_group = 0xFFFFFFFFu;  // the group whose scale g, g6, g4 hold

  auto load = [&](const typename Src::Ref& ref, uint4 (&raw)[NV]) {
    const QuantArgs& a = src.args(ref);
    const uint32_t Tt = (uint32_t)a.R_in, N = (uint32_t)a.C_in;
    const T* __restrict__ xp = reinterpret_cast<const T*>(a.x);
    const uint32_t tok0 = ref.ty * 64, n0 = ref.tx * 128;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int idx = t + 256 * i, row = idx / VPR, cv = idx % VPR;
      const uint32_t col = n0 + (uint32_t)cv * (16 / sizeof(T));
      raw[i] = make_uint4(0, 0, 0, 0);
      if (tok0 + row < Tt && col < N)
        raw[i] = __ldg(reinterpret_cast<const uint4*>(xp + (int64_t)(tok0 + row) * a.ld + col));
    }
  };

  uint4 raw[NV];
  typename Src::Ref ref, iref;  // the tile to encode; (TMA) the next tile to request
  bool have = src.first(ref);
  [[maybe_unused]] bool have_i = have;
  [[maybe_unused]] uint32_t k = 0;    // this CTA's tile counter (TMA ring position)
  [[maybe_unused]] uint32_t req = 0;  // (thread 0) tiles requested so far
  [[maybe_unused]] const unsigned long long limit = wait_ns ? wait_ns : 2000000000ull;
  // the input map of a tile: the single tensor's, or the tile's group's
  [[maybe_unused]] auto map_of = [&](const typename Src::Ref& r) -> const CUtensorMap* {
    if constexpr (Src::kGrouped) return &src.g.tm[r.e];
    else return tm;
  };
  if constexpr (TMA) {
    if (t == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map_of(ref))) : "memory");
      abort_s = 0;
#pragma unroll
      for (int i = 0; i < S; ++i) bar_init(&full[i], 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      iref = ref;
      for (int i = 0; i < S && have_i; ++i) {
        tile_load(ring + i * 64 * RB, map_of(iref), (int)(iref.tx * 128), (int)(iref.ty * 64), &full[i],
                  64 * RB + (i == 0 ? hold_tx : 0u));
        ++req;
        typename Src::Ref n;
        have_i = src.next(iref, n);
        iref = n;
      }
    }
    __syncthreads();
  } else {
    if (have) load(ref, raw);
  }
  while (have) {
    const uint8_t* tile = tile_s;
    typename Src::Ref nref;
    const bool have_next = src.next(ref, nref);
    if constexpr (TMA) {
      if (!bar_wait(&full[k % S], (k / S) & 1, limit)) abort_s = 1;
      tile = ring + (k % S) * 64 * RB;
    } else {
      __syncthreads();  // the previous tile's readers are done with tile_s
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        int idx = t + 256 * i, row = idx / VPR, cv = idx % VPR;
        *reinterpret_cast<uint4*>(tile_s + row * RB + cv * 16) = raw[i];
      }
      __syncthreads();
      if (have_next) load(nref, raw);  // in flight during the encode
    }

    const QuantArgs& a = src.args(ref);
    const uint32_t Tt = (uint32_t)a.R_in, N = (uint32_t)a.C_in;
    const int64_t K = Tt;
    const uint32_t KB = Tt / 16, nka = (KB + 3) / 4;
    if constexpr (!AMAX_ONLY && Src::kGrouped) {
      const bool owns = src.owns_scalars(ref);
      if (owns || ref.e != scale_group) set_scale(a, owns);
      scale_group = ref.e;
    }
    const uint32_t n0 = ref.tx * 128;
    const uint32_t kb = ref.ty * 4 + kbl;
    float v[2][16];
#pragma unroll
    for (int e = 0; e < 16; ++e) ColTile<T>::pair(tile, 16 * kbl + e, np, v[0][e], v[1][e]);
    if constexpr (TMA) {
      // every thread has its values: the slot takes the tile S ahead
      __syncthreads();
      if (abort_s) break;  // a tile never landed (uniform after the barrier)
      if (t == 0 && have_i) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tile_load(ring + (k % S) * 64 * RB, map_of(iref), (int)(iref.tx * 128), (int)(iref.ty * 64), &full[k % S],
                  64 * RB);
        ++req;
        typename Src::Ref n;
        have_i = src.next(iref, n);
        if constexpr (Src::kGrouped) {  // the next request's map, when it is another group's
          if (have_i && n.e != iref.e)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&src.g.tm[n.e])) : "memory");
        }
        iref = n;
      }
      ++k;
    }
    if constexpr (RHT && !AMAX_ONLY) rht16x2(v, mask);
    bool valid[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) valid[h] = (n0 + 2 * np + h < N) && kb < KB;

    if constexpr (AMAX_ONLY) {
      if constexpr (RHT) run_max = rht16x2_absmax(v, mask, run_max);
      else run_max = fmaxf(run_max, fmaxf(absmax16(v[0]), absmax16(v[1])));
    } else {
      float ab[2] = {absmax16(v[0]), absmax16(v[1])};
      if constexpr (B2D) {
        float m = fmaxf(ab[0], ab[1]);
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
        ab[0] = ab[1] = m;
      }
      uint2 codes[2], c4[2];
      uint32_t sbyte[2], b4[2];
      float e6[2], e4[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t n = n0 + 2 * np + h;
        uint32_t u[16];
        if constexpr (SR) sr_draws16(a.seed, a.offset, (uint64_t)n * (uint64_t)K + kb * 16, u);
        float s6, r6;
        sbyte[h] = block_scale(ab[h], g6, g, s6, r6);
        codes[h] = encode16<SR>(v[h], r6, u);
        if constexpr (F46) {
          float s4, r4;
          b4[h] = block_scale(ab[h], g4, g, s4, r4);
          c4[h] = encode16<SR>(v[h], r4, u);
        }
      }
      if constexpr (F46) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          e6[h] = block_sq_err16(v[h], codes[h], sbyte[h], g);
          e4[h] = block_sq_err16(v[h], c4[h], b4[h], g);
        }
        if constexpr (B2D) {
          // tile rows 2p, 2p+1 are this thread's pair; then pairs of pairs ...
          float s6 = __fadd_rn(e6[0], e6[1]), s4 = __fadd_rn(e4[0], e4[1]);
#pragma unroll
          for (int o = 1; o <= 4; o <<= 1) {
            s6 = __fadd_rn(s6, __shfl_xor_sync(0xFFFFFFFFu, s6, o));
            s4 = __fadd_rn(s4, __shfl_xor_sync(0xFFFFFFFFu, s4, o));
          }
          e6[0] = e6[1] = s6;
          e4[0] = e4[1] = s4;
        }
#pragma unroll
        for (int h = 0; h < 2; ++h)
          if (e4[h] < e6[h]) {
            codes[h] = c4[h];
            sbyte[h] = b4[h];
          }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t n = n0 + 2 * np + h;
        if (valid[h]) {
          *reinterpret_cast<uint2*>(a.codes + (int64_t)n * (K / 2) + kb * 8) = codes[h];
          if (a.tdebug) {
            float4* d = reinterpret_cast<float4*>(a.tdebug + (int64_t)n * K + kb * 16);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              d[i] = make_float4(v[h][4 * i], v[h][4 * i + 1], v[h][4 * i + 2], v[h][4 * i + 3]);
          }
        }
        a.scales[sf_offset(n, kb, nka)] = valid[h] ? (uint8_t)sbyte[h] : (uint8_t)0;
      }
    }
    ref = nref;
    have = have_next;
  }
  if constexpr (TMA) {
    if (abort_s) {
      // a wait ran out: record it, let requested tiles land (bounded) and leave
      if (t == 0) {
        atomicOr(a0.err, 2u);
        for (uint32_t i = k; i < req; ++i) bar_wait(&full[i % S], (i / S) & 1, limit);
      }
      return;
    }
  }
  if constexpr (AMAX_ONLY) cta_max_to_global(__float_as_uint(run_max), reinterpret_cast<unsigned int*>(a0.amax_accum));
}

template <typename T, bool B2D, bool SR, bool F46, bool RHT, bool AMAX_ONLY>
__global__ void __launch_bounds__(256) k_quant_cols(const __grid_constant__ CUtensorMap tm, QuantArgs a, uint32_t hold_tx,
                                                   unsigned long long wait_ns) {
  const OneTensor src(a, (uint32_t)((a.C_in + 127) / 128), (uint32_t)((a.R_in + 63) / 64));
  quant_cols_body<T, B2D, SR, F46, RHT, AMAX_ONLY, true>(src, a, &tm, hold_tx, wait_ns);
}

// TMA: input tiles through the ring, each group's map in the parameters
// (else staged through registers).
template <typename T, bool B2D, bool SR, bool F46, bool TMA>
__global__ void __launch_bounds__(256) k_quant_cols_grouped(const __grid_constant__ GroupQuant g) {
  const Groups src(g);
  quant_cols_body<T, B2D, SR, F46, false, false, TMA>(src, g.a[0]);
}
// The TMA-fed encode without stochastic rounding fits 80 registers: 3 CTAs per
// SM (192 KB of rings) hide more of its ALU latency (MoE Four-over-Six
// weights 578 -> 561 us; with SR it spills and stays at 2).
template <typename T, bool B2D, bool F46>
__global__ void __launch_bounds__(256, 3) k_quant_cols_grouped3(const __grid_constant__ GroupQuant g) {
  const Groups src(g);
  quant_cols_body<T, B2D, false, F46, false, false, true>(src, g.a[0]);
}


// ---------------------------------------------------------------------------
// Decoder: one thread per block of 16 (grid-stride), the next block's codes
// and scale requested before the current one is decoded.  V8: the output is
// 32-byte aligned and each 32 bytes leave in one 256-bit store.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t w[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]),
               "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

template <typename TO, bool V8>
__global__ void __launch_bounds__(256) k_dequant(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                                                 const float* __restrict__ gptr, int64_t R, int64_t K, TO* __restrict__ y) {
  const float g = *gptr;
  const float2 g2 = make_float2(g, g);
  // thread -> block (r, kb) of the row-major block grid (adjacent threads,
  // adjacent blocks: coalesced code loads and output stores); the grid
  // stride is added as (rows, blocks) with one carry, so the loop divides once
  const uint32_t KB = (uint32_t)(K / 16), nka = (KB + 3) / 4;
  const uint64_t nblk = (uint64_t)R * KB;
  const uint64_t b0 = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x, step = (uint64_t)gridDim.x * blockDim.x;
  if (b0 >= nblk) return;
  uint64_t r = b0 / KB;
  uint32_t kb = (uint32_t)(b0 % KB);
  const uint64_t step_r = step / KB;
  const uint32_t step_kb = (uint32_t)(step % KB);
  uint2 c = __ldg(reinterpret_cast<const uint2*>(codes + r * (uint64_t)(K / 2) + kb * 8u));
  uint32_t sb = __ldg(scales + sf_offset((int64_t)r, kb, nka));
  for (uint64_t b = b0; b < nblk; b += step) {
    uint64_t nr = r + step_r;
    uint32_t nkb = kb + step_kb;
    if (nkb >= KB) {
      nkb -= KB;
      ++nr;
    }
    uint2 cn = make_uint2(0u, 0u);
    uint32_t sn = 0u;
    if (b + step < nblk) {
      cn = __ldg(reinterpret_cast<const uint2*>(codes + nr * (uint64_t)(K / 2) + nkb * 8u));
      sn = __ldg(scales + sf_offset((int64_t)nr, nkb, nka));
    }
    const uint32_t s2 = e4m3_f16x2_splat(sb & 0x7Fu);
    uint32_t h[8];
    e2m1x16_f16x2(c, h);
    float2 o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = decode_pair(h[i], s2, g2);
    TO* dst = y + r * (uint64_t)K + kb * 16u;
    if constexpr (sizeof(TO) == 4) {
      if constexpr (V8) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t w[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            w[2 * i] = __float_as_uint(o[4 * q + i].x);
            w[2 * i + 1] = __float_as_uint(o[4 * q + i].y);
          }
          st_global_v8(dst + 8 * q, w);
        }
      } else {
        float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
        for (int i = 0; i < 4; ++i) d[i] = make_float4(o[2 * i].x, o[2 * i].y, o[2 * i + 1].x, o[2 * i + 1].y);
      }
    } else {
      uint32_t w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        __nv_bfloat162 p = __floats2bfloat162_rn(o[i].x, o[i].y);
        w[i] = *reinterpret_cast<uint32_t*>(&p);
      }
      if constexpr (V8) {
        st_global_v8(dst, w);
      } else {
        uint4* d = reinterpret_cast<uint4*>(dst);
        d[0] = make_uint4(w[0], w[1], w[2], w[3]);
        d[1] = make_uint4(w[4], w[5], w[6], w[7]);
      }
    }
    c = cn;
    sb = sn;
    r = nr;
    kb = nkb;
  }
}

// Empty tensor: amax = 0, g = 1.
__global__ void k_empty_scalars(float* amax, float* g) {
  *amax = 0.0f;
  *g = 1.0f;
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------
static int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  return dev;
}

static int num_sms() {
  static std::atomic<int> cache[64] = {};
  const int dev = current_device();
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

cudaError_t launch_amax(const void* x, bool bf16, int64_t rows, int64_t cols, int64_t ld, float* amax_accum,
                        cudaStream_t s) {
  const int64_t vec = bf16 ? 8 : 4;
  int64_t r = rows, nvec = cols / vec, ldv = ld / vec;
  if (ld == cols) {  // contiguous: one flat row
    nvec = rows * cols / vec;
    r = 1;
    ldv = 0;
  }
  if (nvec == 0 || r == 0) return cudaSuccess;
  int64_t want = (nvec + 1023) / 1024;
  int64_t cap = (int64_t)num_sms() * 6;  // 6 CTAs per SM: measured best with 8 loads per thread
  unsigned gx = (unsigned)(want < 1 ? 1 : (want > cap ? cap : want));
  unsigned gy = (unsigned)(r > 65535 ? 65535 : r);
  if (gy > 1 && gx * gy > (unsigned)cap) gx = (unsigned)((cap + gy - 1) / gy);
  dim3 grid(gx ? gx : 1, gy);
  if (bf16)
    k_amax<__nv_bfloat16><<<grid, 256, 0, s>>>(reinterpret_cast<const __nv_bfloat16*>(x), r, nvec, ldv,
                                              reinterpret_cast<unsigned int*>(amax_accum));
  else
    k_amax<float><<<grid, 256, 0, s>>>(reinterpret_cast<const float*>(x), r, nvec, ldv,
                                      reinterpret_cast<unsigned int*>(amax_accum));
  return cudaGetLastError();
}

// Persistent grids: as many CTAs as fit on the GPU at once (occupancy of the
// instantiation with its dynamic shared memory), never more than there are
// tiles.  The resident count is cached per device in `cache`, one array per
// kernel (each launch site owns one).
using OccCache = std::atomic<int>[64];
template <class K>
static unsigned persistent_grid(K kernel, int64_t tiles, OccCache& cache, int smem = 0) {
  const int dev = current_device();
  int per_sm = cache[dev].load(std::memory_order_relaxed);
  if (per_sm <= 0) {
    if (smem > 48 * 1024) cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 256, smem) != cudaSuccess || per_sm <= 0)
      per_sm = 1;
    cache[dev].store(per_sm, std::memory_order_relaxed);
  }
  const int64_t cap = (int64_t)num_sms() * per_sm;
  return (unsigned)(tiles < cap ? (tiles > 0 ? tiles : 1) : cap);
}

template <typename T, bool B2D, bool SR, bool F46, bool RHT, bool AO>
static cudaError_t launch_q(const QuantArgs& a, bool transpose, cudaStream_t s) {
  if (!transpose) {
    const int64_t tiles = ((a.K / 16 + 3) / 4) * ((a.R + 127) / 128);
    if constexpr (sizeof(T) == 2 && !B2D && !SR && !F46 && !RHT && !AO) {
      auto k = k_quant_rows_plain;
      static OccCache occ = {};
      k<<<persistent_grid(k, tiles, occ), 256, 0, s>>>(a);
    } else {
      auto k = k_quant_rows<T, B2D, SR, F46, RHT, AO>;
      static OccCache occ = {};
      k<<<persistent_grid(k, tiles, occ), 256, 0, s>>>(a);
    }
  } else {
    // input tiles of 64 rows x 128 columns through the TMA ring
    CUtensorMap tm;
    if (!make_tile_map_2d(&tm, a.x, sizeof(T) == 2, a.R_in, a.C_in, a.ld, 128, 64)) return cudaErrorInvalidValue;
    const int64_t tiles = ((a.C_in + 127) / 128) * ((a.R_in + 63) / 64);
    auto k = k_quant_cols<T, B2D, SR, F46, RHT, AO>;
    constexpr int smem = kColRingBytes<T>;
    static OccCache occ = {};
    const unsigned grid = persistent_grid(k, tiles, occ, smem);
    const unsigned long long lim = take_armed_wait(2);  // failure-detection test only
    k<<<grid, 256, smem, s>>>(tm, a, lim ? 16u : 0u, lim);
  }
  return cudaGetLastError();
}

template <typename T, bool RHT, bool AO>
static cudaError_t dispatch_opts(const QuantArgs& a, bool transpose, bool b2d, bool sr, bool f46, cudaStream_t s) {
  if (AO) return launch_q<T, false, false, false, RHT, AO>(a, transpose, s);
  if (b2d) {
    if (sr) {
      if (f46) return launch_q<T, true, true, true, RHT, AO>(a, transpose, s);
      return launch_q<T, true, true, false, RHT, AO>(a, transpose, s);
    }
    if (f46) return launch_q<T, true, false, true, RHT, AO>(a, transpose, s);
    return launch_q<T, true, false, false, RHT, AO>(a, transpose, s);
  }
  if (sr) {
    if (f46) return launch_q<T, false, true, true, RHT, AO>(a, transpose, s);
    return launch_q<T, false, true, false, RHT, AO>(a, transpose, s);
  }
  if (f46) return launch_q<T, false, false, true, RHT, AO>(a, transpose, s);
  return launch_q<T, false, false, false, RHT, AO>(a, transpose, s);
}

template <typename T, bool B2D, bool SR, bool F46>
static void launch_qg(const GroupQuant& g, bool transpose, cudaStream_t s) {
  const uint32_t tiles = g.tile_start[g.count];
  if (!transpose) {
    if constexpr (sizeof(T) == 2 && !B2D && !SR && !F46) {
      auto k = k_quant_rows_grouped_plain;
      static OccCache occ = {};
      k<<<persistent_grid(k, tiles, occ), 256, 0, s>>>(g);
    } else {
      auto k = k_quant_rows_grouped<T, B2D, SR, F46>;
      static OccCache occ = {};
      k<<<persistent_grid(k, tiles, occ), 256, 0, s>>>(g);
    }
  } else if (g.use_tma) {
    constexpr int smem = kColRingBytes<T>;
    if constexpr (!SR) {
      auto k = k_quant_cols_grouped3<T, B2D, F46>;
      static OccCache occ = {};
      k<<<persistent_grid(k, tiles, occ, smem), 256, smem, s>>>(g);
    } else {
      auto k = k_quant_cols_grouped<T, B2D, SR, F46, true>;
      static OccCache occ = {};
      k<<<persistent_grid(k, tiles, occ, smem), 256, smem, s>>>(g);
    }
  } else {
    auto k = k_quant_cols_grouped<T, B2D, SR, F46, false>;
    static OccCache occ = {};
    k<<<persistent_grid(k, tiles, occ), 256, 0, s>>>(g);
  }
}

template <typename T>
static void dispatch_grouped(const GroupQuant& g, bool transpose, bool b2d, bool sr, bool f46, cudaStream_t s) {
  if (b2d) {
    if (sr) {
      if (f46) launch_qg<T, true, true, true>(g, transpose, s);
      else launch_qg<T, true, true, false>(g, transpose, s);
    } else {
      if (f46) launch_qg<T, true, false, true>(g, transpose, s);
      else launch_qg<T, true, false, false>(g, transpose, s);
    }
  } else {
    if (sr) {
      if (f46) launch_qg<T, false, true, true>(g, transpose, s);
      else launch_qg<T, false, true, false>(g, transpose, s);
    } else {
      if (f46) launch_qg<T, false, false, true>(g, transpose, s);
      else launch_qg<T, false, false, false>(g, transpose, s);
    }
  }
}

cudaError_t launch_quantize_grouped(GroupQuant& g, bool bf16, bool transpose, bool b2d, bool sr, bool f46,
                                    bool compute_amax, cudaStream_t s) {
  if (g.count <= 0) return cudaSuccess;
  const int64_t es = bf16 ? 2 : 4;
  uint32_t tiles = 0, atiles = 0;
  for (int e = 0; e < g.count; ++e) {
    const QuantArgs& a = g.a[e];
    g.tiles_x[e] = transpose ? (uint32_t)((a.C_in + 127) / 128) : (uint32_t)((a.K / 16 + 3) / 4);
    const uint32_t tiles_y = transpose ? (uint32_t)((a.R_in + 63) / 64) : (uint32_t)((a.R + 127) / 128);
    g.tile_start[e] = tiles;
    tiles += g.tiles_x[e] * tiles_y;
    const int64_t row_bytes = a.C_in * es;
    g.amax_rows[e] = (uint32_t)(row_bytes >= 65536 ? 1 : 65536 / row_bytes);
    g.amax_start[e] = atiles;
    atiles += (uint32_t)((a.R_in + g.amax_rows[e] - 1) / g.amax_rows[e]);
  }
  g.tile_start[g.count] = tiles;
  g.amax_start[g.count] = atiles;
  g.use_tma = 0;
  if (transpose) {  // the ring's input maps (64 tokens x 128 columns per tile)
    g.use_tma = 1;
    for (int e = 0; e < g.count && g.use_tma; ++e) {
      const QuantArgs& a = g.a[e];
      if (!make_tile_map_2d(&g.tm[e], a.x, bf16, a.R_in, a.C_in, a.ld, 128, 64)) g.use_tma = 0;
    }
  }
  if (compute_amax) {
    k_zero_group_amax<<<1, kQuantGroups, 0, s>>>(g);
    const unsigned cap = (unsigned)num_sms() * 8;
    const unsigned grid = atiles < cap ? atiles : cap;
    if (bf16) k_amax_grouped<__nv_bfloat16><<<grid, 256, 0, s>>>(g);
    else k_amax_grouped<float><<<grid, 256, 0, s>>>(g);
  }
  if (bf16) dispatch_grouped<__nv_bfloat16>(g, transpose, b2d, sr, f46, s);
  else dispatch_grouped<float>(g, transpose, b2d, sr, f46, s);
  return cudaGetLastError();
}

cudaError_t launch_quantize(const QuantArgs& a, bool bf16, bool transpose, bool b2d, bool sr, bool f46, bool rht,
                            bool amax_only, cudaStream_t s) {
  if (a.R == 0 || a.K == 0) return cudaSuccess;
  if (bf16) {
    if (rht) {
      if (amax_only) return dispatch_opts<__nv_bfloat16, true, true>(a, transpose, false, false, false, s);
      return dispatch_opts<__nv_bfloat16, true, false>(a, transpose, false, sr, f46, s);
    }
    return dispatch_opts<__nv_bfloat16, false, false>(a, transpose, b2d, sr, f46, s);
  }
  if (rht) {
    if (amax_only) return dispatch_opts<float, true, true>(a, transpose, false, false, false, s);
    return dispatch_opts<float, true, false>(a, transpose, false, sr, f46, s);
  }
  return dispatch_opts<float, false, false>(a, transpose, b2d, sr, f46, s);
}

cudaError_t launch_empty_scalars(float* amax, float* g, cudaStream_t s) {
  k_empty_scalars<<<1, 1, 0, s>>>(amax, g);
  return cudaGetLastError();
}

cudaError_t launch_dequantize(const uint8_t* codes, const uint8_t* scales, const float* g, int64_t R, int64_t K,
                              void* y, bool bf16_out, cudaStream_t s) {
  int64_t nblk = R * (K / 16);
  if (nblk == 0) return cudaSuccess;
  int64_t want = (nblk + 255) / 256, cap = (int64_t)num_sms() * 16;
  unsigned grid = (unsigned)(want > cap ? cap : want);
  const bool v8 = reinterpret_cast<uintptr_t>(y) % 32 == 0;  // rows are 32-byte multiples (K % 16 == 0)
  if (bf16_out) {
    __nv_bfloat16* yb = reinterpret_cast<__nv_bfloat16*>(y);
    if (v8) k_dequant<__nv_bfloat16, true><<<grid, 256, 0, s>>>(codes, scales, g, R, K, yb);
    else k_dequant<__nv_bfloat16, false><<<grid, 256, 0, s>>>(codes, scales, g, R, K, yb);
  } else {
    float* yf = reinterpret_cast<float*>(y);
    if (v8) k_dequant<float, true><<<grid, 256, 0, s>>>(codes, scales, g, R, K, yf);
    else k_dequant<float, false><<<grid, 256, 0, s>>>(codes, scales, g, R, K, yf);
  }
  return cudaGetLastError();
}

}  // namespace nvfp4
