// Weight-only NVFP4 GEMM (W4A16): Y = X * W_hat^T with BF16 activations X
// and NVFP4 weights W dequantized inside the kernel to the BF16 values a
// BF16 GEMM would take, W_hat = BF16(fl(fl(value(code) * s_b) * g)), FP32
// accumulation.  The serving variant the pages give for GPUs without FP4
// tensor cores (the hyper.ai story on the Nemotron 3 Ultra NVFP4 checkpoint:
// Blackwell computes W4A4, Hopper serving switches to W4A16; "BF16 vs NVFP4
// with Nemotron 3.5 Lightning", "Key takeaways": NVFP4 checkpoints run on
// Hopper and Ampere).  On B300 it is the decode-sized path: with few
// activation rows the kernel streams the weights once (0.5625 byte per
// weight instead of 2 for BF16).
//
// Layout of the work: a CTA of 4 warps owns 16 weight rows; warp w takes the
// K tiles w, w + 4, ...; the 4 partial results meet in shared memory.
// The products run on register-operand BF16 MMAs (m16n8k16, FP32
// accumulate): weight rows are the MMA's M, tokens its N (8 per MMA), the
// decoded BF16 pairs are the A fragment directly and the activations' BF16
// pairs the B fragment directly, so nothing is unpacked per token.  The sum
// over K does not depend on the order of its terms, so inside each K tile
// the K positions are permuted to suit the decode: lane (g, t) decodes
// whole 16-element blocks of rows g and g + 8 and feeds four MMAs per block
// with its own pairs; its B fragments are the activations at the same K
// positions (one 32-byte run per block).  With K % 32 == 0 a K tile is 128
// wide and lane t takes blocks 2t and 2t + 1 of it (16 code bytes and two
// adjacent scale bytes per row in one load each); otherwise a tile is 64
// wide and lane t takes block t (8 code bytes, one scale).
#include "nvfp4_device.cuh"
#include "quantize.h"

namespace nvfp4 {

// The 16 BF16 weights of one block as 8 bf16x2 words (word p = elements 2p,
// 2p+1): the decode fl(fl(value * s) * g) of each pair, rounded to BF16
// (nearest even).
__device__ __forceinline__ void w4a16_block(uint2 c, uint32_t sbyte, float2 g2, uint32_t w[8]) {
  const uint32_t s2 = e4m3_f16x2_splat(sbyte & 0x7Fu);
  uint32_t h[8];
  e2m1x16_f16x2(c, h);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float2 p = decode_pair(h[j], s2, g2);
    const __nv_bfloat162 b = __floats2bfloat162_rn(p.x, p.y);
    w[j] = *reinterpret_cast<const uint32_t*>(&b);
  }
}

// c += A (16 x 16, BF16, row-major fragment) * B (16 x 8, BF16), FP32.
__device__ __forceinline__ void mma_bf16_16816(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint2 ld_stream_u2(const uint8_t* p) {
  uint2 r;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}
__device__ __forceinline__ uint4 ld_stream_u4(const uint8_t* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// The codes (8 BPL bytes) and scales (BPL bytes) of a lane's BPL blocks of
// one row; block h's codes are words 2h, 2h + 1 and its scale byte h.
template <int BPL>
struct W4Blocks {
  uint32_t c[2 * BPL];
  uint32_t s;
  __device__ __forceinline__ void clear() {
#pragma unroll
    for (int i = 0; i < 2 * BPL; ++i) c[i] = 0u;
    s = 0u;
  }
  __device__ __forceinline__ void load(const uint8_t* codes, const uint8_t* scales) {
    if constexpr (BPL == 2) {
      const uint4 v = ld_stream_u4(codes);
      c[0] = v.x, c[1] = v.y, c[2] = v.z, c[3] = v.w;
      s = *reinterpret_cast<const uint16_t*>(scales);
    } else {
      const uint2 v = ld_stream_u2(codes);
      c[0] = v.x, c[1] = v.y;
      s = *scales;
    }
  }
};

constexpr int kW4Warps = 4;   // warps per CTA, splitting K
// K tiles per warp whose loads are issued together: two 64-wide tiles, or one
// 128-wide tile (the same bytes per lane)
template <int BPL>
constexpr int kW4Unroll = BPL == 2 ? 1 : 2;
constexpr int kW4AccMax = 2;  // independent accumulators per token tile (MMA j of a tile -> j % kW4Acc)

// NT = token tiles of 8 per pass over the weights (tokens m0 .. m0 + 8 NT - 1);
// BPL = blocks per lane and row in a K tile (the tile is 64 BPL wide).
// The 128-wide tiles hold more registers: 7 CTAs per SM (72 registers).
template <int NT, bool OUT_BF16, int BPL>
__global__ void __launch_bounds__(kW4Warps * 32, BPL == 1 ? 8 : 7)
    k_w4a16(const __nv_bfloat16* __restrict__ x, int64_t M, int64_t ldx, const uint8_t* __restrict__ codes,
            const uint8_t* __restrict__ scales, const float* __restrict__ gptr, int64_t N, int64_t K,
            void* __restrict__ y, int64_t ldy) {
  // two token tiles already give each warp two independent MMA chains (and one accumulator each avoids spills)
  constexpr int kW4Acc = NT == 1 ? kW4AccMax : 1;
  __shared__ float part[kW4Warps][NT][8][17];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int64_t n0 = (int64_t)blockIdx.x * 16;
  const int64_t ra = n0 + g;
  const bool va = ra < N, vb = ra + 8 < N;
  const float gs = *gptr;
  const float2 g2 = make_float2(gs, gs);
  const int KB = (int)(K / 16), KT = (KB + 4 * BPL - 1) / (4 * BPL), nka = (KB + 3) / 4;
  // block (row, kt * 4 BPL + BPL t + h) has its codes at row * K/2 +
  // kt * 32 BPL + 8 (BPL t + h) and its scale at sf_offset(row, BPL t + h) +
  // kt * 512 BPL (the BPL scales of a lane are adjacent bytes of one 128x4
  // atom); row ra + 8 lies in the same 32-row group as ra (16-row aligned
  // n0, g < 8), so its scales sit 128 bytes on and its codes 8 rows (4K
  // bytes) on.  With BPL = 2, K % 32 == 0: a lane's second block is valid
  // whenever its first is.
  const int64_t row8 = 4 * K;
  const uint8_t* pa = codes + ra * (K / 2) + 8 * BPL * t;
  const uint8_t* qa = scales + sf_offset(ra, BPL * t, nka);
  for (int64_t m0 = 0; m0 < M; m0 += 8 * NT) {
    float accj[NT][kW4Acc][4];
#pragma unroll
    for (int i = 0; i < NT; ++i)
#pragma unroll
      for (int j = 0; j < kW4Acc; ++j) accj[i][j][0] = accj[i][j][1] = accj[i][j][2] = accj[i][j][3] = 0.0f;
    const __nv_bfloat16* xr[NT];
    bool xv[NT];
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      const int64_t tok = m0 + 8 * i + g;
      xv[i] = tok < M;
      xr[i] = x + (xv[i] ? tok : 0) * ldx + 16 * BPL * t;
    }
    for (int kt0 = warp; kt0 < KT; kt0 += kW4Warps * kW4Unroll<BPL>) {
      W4Blocks<BPL> wa_in[kW4Unroll<BPL>], wb_in[kW4Unroll<BPL>];
#pragma unroll
      for (int u = 0; u < kW4Unroll<BPL>; ++u) {
        const int kt = kt0 + kW4Warps * u;
        const bool ok = kt < KT && kt * 4 * BPL + BPL * t < KB;
        wa_in[u].clear();
        wb_in[u].clear();
        if (ok && va) wa_in[u].load(pa + (uint32_t)kt * (32u * BPL), qa + (uint32_t)kt * (512u * BPL));
        if (ok && vb) wb_in[u].load(pa + row8 + (uint32_t)kt * (32u * BPL), qa + 128u + (uint32_t)kt * (512u * BPL));
      }
#pragma unroll
      for (int u = 0; u < kW4Unroll<BPL>; ++u) {
        const int kt = kt0 + kW4Warps * u;
        if (kt < KT) {  // warp-uniform
          const bool ok = kt * 4 * BPL + BPL * t < KB;
#pragma unroll
          for (int h = 0; h < BPL; ++h) {
            uint32_t wa[8], wb[8];
            w4a16_block(make_uint2(wa_in[u].c[2 * h], wa_in[u].c[2 * h + 1]), wa_in[u].s >> (8 * h), g2, wa);
            w4a16_block(make_uint2(wb_in[u].c[2 * h], wb_in[u].c[2 * h + 1]), wb_in[u].s >> (8 * h), g2, wb);
#pragma unroll
            for (int i = 0; i < NT; ++i) {
              uint4 xa = make_uint4(0u, 0u, 0u, 0u), xb = xa;
              if (xv[i] && ok) {
                const uint4* p = reinterpret_cast<const uint4*>(xr[i] + (uint32_t)kt * (64u * BPL) + 16 * h);
                xa = __ldg(p);
                xb = __ldg(p + 1);
              }
              mma_bf16_16816(accj[i][0 % kW4Acc], wa[0], wb[0], wa[1], wb[1], xa.x, xa.y);
              mma_bf16_16816(accj[i][1 % kW4Acc], wa[2], wb[2], wa[3], wb[3], xa.z, xa.w);
              mma_bf16_16816(accj[i][2 % kW4Acc], wa[4], wb[4], wa[5], wb[5], xb.x, xb.y);
              mma_bf16_16816(accj[i][3 % kW4Acc], wa[6], wb[6], wa[7], wb[7], xb.z, xb.w);
            }
          }
        }
      }
    }
    // C fragment: rows g, g + 8 (weight rows), columns 2t, 2t + 1 (tokens)
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      float c[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        c[e] = accj[i][0][e];
#pragma unroll
        for (int j = 1; j < kW4Acc; ++j) c[e] += accj[i][j][e];
      }
      part[warp][i][2 * t][g] = c[0];
      part[warp][i][2 * t + 1][g] = c[1];
      part[warp][i][2 * t][g + 8] = c[2];
      part[warp][i][2 * t + 1][g + 8] = c[3];
    }
    __syncthreads();
    for (int e = threadIdx.x; e < NT * 128; e += kW4Warps * 32) {
      const int i = e >> 7, tk = (e >> 4) & 7, row = e & 15;
      float v = part[0][i][tk][row];
#pragma unroll
      for (int w = 1; w < kW4Warps; ++w) v += part[w][i][tk][row];
      const int64_t tok = m0 + 8 * i + tk, n = n0 + row;
      if (tok < M && n < N) {
        if constexpr (OUT_BF16)
          reinterpret_cast<__nv_bfloat16*>(y)[tok * ldy + n] = __float2bfloat16_rn(v);
        else
          reinterpret_cast<float*>(y)[tok * ldy + n] = v;
      }
    }
    __syncthreads();
  }
}

cudaError_t launch_w4a16(const void* x, int64_t M, int64_t ldx, const uint8_t* codes, const uint8_t* scales,
                         const float* g, int64_t N, int64_t K, void* y, bool out_bf16, int64_t ldy, cudaStream_t s) {
  if (M == 0 || N == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((N + 15) / 16);
  const __nv_bfloat16* xp = reinterpret_cast<const __nv_bfloat16*>(x);
  const dim3 block(kW4Warps * 32);
  // 16-byte code loads need K % 32 == 0 (rows of 16-byte multiples); with
  // two token tiles the wide form would spill, so it serves M <= 8
#define NVFP4_W4_LAUNCH(NT, BF, BPL) k_w4a16<NT, BF, BPL><<<grid, block, 0, s>>>(xp, M, ldx, codes, scales, g, N, K, y, ldy)
  if (M <= 8 && K % 32 == 0) {
    if (out_bf16) NVFP4_W4_LAUNCH(1, true, 2);
    else NVFP4_W4_LAUNCH(1, false, 2);
  } else if (M <= 8) {
    if (out_bf16) NVFP4_W4_LAUNCH(1, true, 1);
    else NVFP4_W4_LAUNCH(1, false, 1);
  } else {
    if (out_bf16) NVFP4_W4_LAUNCH(2, true, 1);
    else NVFP4_W4_LAUNCH(2, false, 1);
  }
#undef NVFP4_W4_LAUNCH
  return cudaGetLastError();
}

}  // namespace nvfp4
