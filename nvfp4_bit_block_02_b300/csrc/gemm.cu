// Block-scaled NVFP4 x NVFP4 GEMM on the sm_103a tensor cores (tcgen05).
//
// D[m][n] = g_A * g_B * sum_k (a_mk * sA_{m,k/16}) (b_nk * sB_{n,k/16}), FP32
// accumulation in tensor memory: the W4A4 product the hyper.ai story on the
// Nemotron 3 Ultra NVFP4 checkpoint says Blackwell runs natively, on the
// format of "NVIDIA Introduces a 4-Bit Pretraining Methodology Using NVFP4"
// ("Summary").
//
// One CTA computes a 128 x 256 tile of D.  Warp roles:
//   warp 0      TMA producer: A and B code tiles (128 B of K = 256 elements
//               per row, 128B swizzle) by cp.async.bulk.tensor, the matching
//               scale atoms (contiguous 512-byte atoms of the 128x4 scale
//               layout) by cp.async.bulk, into a 4-stage ring.
//   warp 1      owns the tensor memory (512 columns: the 256-column FP32
//               accumulator and one scale-factor slot per stage) and issues,
//               from one thread, tcgen05.cp of the scale atoms into TMEM and
//               tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X
//               (M = 128, N = 256, K = 64 per instruction).
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (warp w reads TMEM
//               lanes 32*(w%4)..+31 = tile rows), scale by g_A*g_B, convert,
//               store.
// Every mbarrier wait is bounded (kWaitLimitNs).  On expiry the CTA records
// NVFP4 timeout in a device word, stops issuing, waits (bounded) for the
// copies and MMAs it has in flight, frees its tensor memory and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gemm.h"

namespace nvfp4 {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
#ifndef NVFP4_GEMM_MMA_N
#define NVFP4_GEMM_MMA_N 256
#endif
constexpr int MMA_N = NVFP4_GEMM_MMA_N;
constexpr int BKB = 128;  // bytes of K per stage per row = 256 FP4 elements
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BKB;
constexpr int B_BYTES = BN * BKB;
constexpr int SFA_BYTES = 4 * 512;               // 4 K-atoms of the 128-row tile
constexpr int SFB_BYTES = (BN / 128) * 4 * 512;  // per 128-row block of B
constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;
constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
constexpr int OFF_BAR = OFF_SFB + STAGES * SFB_BYTES;
constexpr int SMEM_BYTES = OFF_BAR + 128 + 1024;  // + barriers + alignment slack
constexpr int TMEM_COLS = 512;
constexpr int SF_COL0 = BN;                   // first scale-factor column
constexpr int SF_COLS_PER_STAGE = 16 + 32;    // SFA 4 atoms x 4 cols, SFB 8 atoms x 4 cols
constexpr int NUM_THREADS = 192;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s
static_assert(SF_COL0 + STAGES * SF_COLS_PER_STAGE <= TMEM_COLS, "TMEM budget");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// instruction descriptor: E2M1 x E2M1 (kind::mxf4nvf4 encoding 1), UE4M3
// scales, K-major A and B, dense K = 64, M and N fields.
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((uint32_t)(MMA_N >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ unsigned long long now_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: true when the phase completed; false on abort or timeout
// (a timeout raises the CTA's abort flag and the device error word).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned int* err, unsigned long long limit = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = now_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (now_ns() - t0 > limit) {
        *abort_flag = 1;
        atomicOr(err, 1u);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(kIdesc), "r"(acc), "r"(sfa), "r"(sfb)
      : "memory");
}

// K-major operand tile, 128-byte rows, 128B swizzle: 8-row atoms of 1024 B.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// One 512-byte scale atom: 32 rows x 16 B, no swizzle, 8x16 B core matrices.
__device__ __forceinline__ uint64_t desc_sf(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(128 >> 4) << 32) | ((uint64_t)1 << 46);
}

#define NVFP4_LD32(taddr, r)                                                                                         \
  asm volatile(                                                                                                      \
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"  \
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"                                                 \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), \
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),     \
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),    \
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])                  \
      : "r"(taddr))

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

struct TileJob {
  const CUtensorMap* tmA;
  const CUtensorMap* tmB;
  const uint8_t* sfa;  // scale buffer of A (128x4-atom layout)
  const uint8_t* sfb;
  const float* ga;
  const float* gb;
  void* d;
  int64_t ldd;
  int M, N, K;
  int m_tile, n_tile;
};

// One 128 x 256 output tile; called by all 192 threads of the CTA.
__device__ __forceinline__ void gemm_tile(const TileJob& j, bool out_bf16, uint8_t* smem, unsigned int* err) {
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + STAGES), accum = smem_u32(bars + 2 * STAGES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = j.K / 256;
  const int64_t n_katoms = j.K / 64;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_init(accum, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // valid 128-row blocks of B in this tile (N % 128 == 0)
  const int nb_valid = min(BN / 128, (j.N - j.n_tile * BN) / 128);
  const uint32_t stage_tx = A_BYTES + B_BYTES + SFA_BYTES + nb_valid * 2048;

  if (warp == 0 && lane == 0) {
    // ---------------- producer ----------------
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(j.tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(j.tmB)) : "memory");
    int issued = 0;
    for (int kt = 0; kt < nk; ++kt) {
      const int s = kt % STAGES;
      const uint32_t ph = (kt / STAGES) & 1;
      if (!mbar_wait(empty0 + 8 * s, ph ^ 1, abort_flag, err)) break;
      const uint32_t fb = full0 + 8 * s;
      mbar_expect_tx(fb, stage_tx);
      tma_load_2d(smem_u32(smem + OFF_A + s * A_BYTES), j.tmA, kt * BKB, j.m_tile * BM, fb);
      tma_load_2d(smem_u32(smem + OFF_B + s * B_BYTES), j.tmB, kt * BKB, j.n_tile * BN, fb);
      bulk_g2s(smem_u32(smem + OFF_SFA + s * SFA_BYTES), j.sfa + ((int64_t)j.m_tile * n_katoms + 4 * kt) * 512,
               SFA_BYTES, fb);
      for (int nb = 0; nb < nb_valid; ++nb)
        bulk_g2s(smem_u32(smem + OFF_SFB + s * SFB_BYTES + nb * 2048),
                 j.sfb + ((int64_t)(j.n_tile * (BN / 128) + nb) * n_katoms + 4 * kt) * 512, 2048, fb);
      issued = kt + 1;
    }
    if (*abort_flag) {
      // let every copy this thread started land before the CTA exits
      for (int kt = issued > STAGES ? issued - STAGES : 0; kt < issued; ++kt) {
        const unsigned long long t0 = now_ns();
        while (!mbar_try_wait(full0 + 8 * (kt % STAGES), (kt / STAGES) & 1) && now_ns() - t0 < 100000000ull) {
        }
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    for (int kt = 0; kt < nk; ++kt) {
      const int s = kt % STAGES;
      if (!mbar_wait(full0 + 8 * s, (kt / STAGES) & 1, abort_flag, err)) break;
      tc_fence_after();
      const uint32_t sfa_t = tmem + SF_COL0 + s * SF_COLS_PER_STAGE;
      const uint32_t sfb_t = sfa_t + 16;
      const uint32_t sa = smem_u32(smem + OFF_SFA + s * SFA_BYTES);
      const uint32_t sb = smem_u32(smem + OFF_SFB + s * SFB_BYTES);
#pragma unroll
      for (int ka = 0; ka < 4; ++ka) {
        tc_cp_sf(sfa_t + 4 * ka, desc_sf(sa + ka * 512));
#pragma unroll
        for (int nb = 0; nb < BN / 128; ++nb) tc_cp_sf(sfb_t + 8 * ka + 4 * nb, desc_sf(sb + nb * 2048 + ka * 512));
      }
      const uint32_t a0 = smem_u32(smem + OFF_A + s * A_BYTES);
      const uint32_t b0 = smem_u32(smem + OFF_B + s * B_BYTES);
#pragma unroll
      for (int ka = 0; ka < 4; ++ka) {
#pragma unroll
        for (int nh = 0; nh < BN / MMA_N; ++nh) {
          tc_mma(tmem + nh * MMA_N, desc_sw128(a0 + 32 * ka), desc_sw128(b0 + nh * MMA_N * BKB + 32 * ka),
                 sfa_t + 4 * ka, sfb_t + 8 * ka + 4 * (nh * MMA_N / 128), (kt | ka) != 0);
        }
      }
      tc_commit(empty0 + 8 * s);
    }
    tc_commit(accum);
    if (*abort_flag) {
      const unsigned long long t0 = now_ns();
      while (!mbar_try_wait(accum, 0) && now_ns() - t0 < 100000000ull) {
      }
    }
  } else if (warp >= 2) {
    // ---------------- epilogue ----------------
    const bool ok = mbar_wait(accum, 0, abort_flag, err);
    tc_fence_after();
    if (ok && !*abort_flag) {
      const int q = warp & 3;
      const int64_t row = (int64_t)j.m_tile * BM + q * 32 + lane;
      const float alpha = __fmul_rn(*j.ga, *j.gb);
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        const int col0 = j.n_tile * BN + c * 32;
        if (col0 >= j.N) break;  // warp-uniform
        uint32_t r[32];
        NVFP4_LD32(tbase + c * 32, r);
        tmem_ld_wait();
        if (out_bf16) {
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(j.d) + row * j.ldd + col0);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              __nv_bfloat162 p = __floats2bfloat162_rn(__fmul_rn(alpha, __uint_as_float(r[8 * v + 2 * i])),
                                                       __fmul_rn(alpha, __uint_as_float(r[8 * v + 2 * i + 1])));
              w[i] = *reinterpret_cast<uint32_t*>(&p);
            }
            dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(j.d) + row * j.ldd + col0);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            dst[v] = make_float4(__fmul_rn(alpha, __uint_as_float(r[4 * v])), __fmul_rn(alpha, __uint_as_float(r[4 * v + 1])),
                                 __fmul_rn(alpha, __uint_as_float(r[4 * v + 2])),
                                 __fmul_rn(alpha, __uint_as_float(r[4 * v + 3])));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS));
  }
}

__device__ __forceinline__ uint8_t* aligned_smem() {
  extern __shared__ uint8_t smem_raw[];
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, GemmArgs a) {
  TileJob j{&tmA, &tmB, a.sfa, a.sfb, a.ga, a.gb, a.d, a.ldd, a.M, a.N, a.K, (int)blockIdx.y, (int)blockIdx.x};
  gemm_tile(j, a.out_bf16 != 0, aligned_smem(), a.err);
}

__global__ void __launch_bounds__(NUM_THREADS, 1) k_gemm_grouped(const __grid_constant__ GroupedArgs g) {
  // find this CTA's group by the prefix sums of the tile counts
  int e = 0;
  while (e + 1 < g.count && (int)blockIdx.x >= g.tile_start[e + 1]) ++e;
  const int local = (int)blockIdx.x - g.tile_start[e];
  const int tn = (g.N[e] + BN - 1) / BN;
  TileJob j{&g.tmA[e], &g.tmB[e], g.sfa[e], g.sfb[e], g.ga[e], g.gb[e], g.d[e], (int64_t)g.N[e], g.M[e], g.N[e],
            g.K[e], local / tn, local % tn};
  gemm_tile(j, g.out_bf16 != 0, aligned_smem(), g.err);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
__device__ unsigned int g_device_error = 0;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// rows x (K/2) bytes, K-major, box = 128 B x box_rows, 128B swizzle
bool make_code_map(CUtensorMap* m, const uint8_t* codes, int64_t rows, int64_t K, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)(K / 2), (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
  cuuint32_t box[2] = {(cuuint32_t)BKB, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(codes), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool smem_configured(const void* fn) {
  return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) == cudaSuccess;
}

}  // namespace

unsigned int* device_error_word() {
  static unsigned int* p = nullptr;
  if (!p) {
    void* q = nullptr;
    if (cudaGetSymbolAddress(&q, g_device_error) == cudaSuccess) p = reinterpret_cast<unsigned int*>(q);
  }
  return p;
}

int gemm_tile_m() { return BM; }
int gemm_tile_n() { return BN; }

cudaError_t launch_gemm(const GemmOperand& A, const GemmOperand& B, void* D, int64_t ldd, bool out_bf16, cudaStream_t s,
                        const char** why) {
  CUtensorMap ta, tb;
  if (!make_code_map(&ta, A.codes, A.rows, A.K, BM) || !make_code_map(&tb, B.codes, B.rows, B.K, BN)) {
    *why = "cuTensorMapEncodeTiled failed (or driver entry point unavailable)";
    return cudaErrorInvalidValue;
  }
  unsigned int* err = device_error_word();
  if (!err) {
    *why = "device error word unavailable";
    return cudaErrorInvalidValue;
  }
  static bool cfg = false;
  if (!cfg) {
    if (!smem_configured(reinterpret_cast<const void*>(k_gemm))) {
      *why = "cudaFuncSetAttribute(max dynamic shared memory) failed";
      return cudaErrorInvalidValue;
    }
    cfg = true;
  }
  GemmArgs a{A.scales, B.scales, A.g, B.g, D, ldd, (int)A.rows, (int)B.rows, (int)A.K, out_bf16 ? 1 : 0, err};
  dim3 grid((unsigned)((B.rows + BN - 1) / BN), (unsigned)(A.rows / BM));
  k_gemm<<<grid, NUM_THREADS, SMEM_BYTES, s>>>(ta, tb, a);
  return cudaGetLastError();
}

cudaError_t launch_gemm_grouped(int count, const GemmOperand* A, const GemmOperand* B, void* const* D, bool out_bf16,
                                cudaStream_t s, const char** why) {
  unsigned int* err = device_error_word();
  if (!err) {
    *why = "device error word unavailable";
    return cudaErrorInvalidValue;
  }
  static bool cfg = false;
  if (!cfg) {
    if (!smem_configured(reinterpret_cast<const void*>(k_gemm_grouped))) {
      *why = "cudaFuncSetAttribute(max dynamic shared memory) failed";
      return cudaErrorInvalidValue;
    }
    cfg = true;
  }
  for (int base = 0; base < count; base += kGroupsPerLaunch) {
    const int n = count - base < kGroupsPerLaunch ? count - base : kGroupsPerLaunch;
    GroupedArgs g;
    g.count = n;
    g.out_bf16 = out_bf16 ? 1 : 0;
    g.err = err;
    int tiles = 0;
    for (int e = 0; e < n; ++e) {
      const GemmOperand& a = A[base + e];
      const GemmOperand& b = B[base + e];
      if (!make_code_map(&g.tmA[e], a.codes, a.rows, a.K, BM) || !make_code_map(&g.tmB[e], b.codes, b.rows, b.K, BN)) {
        *why = "cuTensorMapEncodeTiled failed (or driver entry point unavailable)";
        return cudaErrorInvalidValue;
      }
      g.sfa[e] = a.scales;
      g.sfb[e] = b.scales;
      g.ga[e] = a.g;
      g.gb[e] = b.g;
      g.d[e] = D[base + e];
      g.M[e] = (int)a.rows;
      g.N[e] = (int)b.rows;
      g.K[e] = (int)a.K;
      g.tile_start[e] = tiles;
      tiles += (int)(a.rows / BM) * (int)((b.rows + BN - 1) / BN);
    }
    if (tiles == 0) continue;
    k_gemm_grouped<<<tiles, NUM_THREADS, SMEM_BYTES, s>>>(g);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace nvfp4
