// Block-scaled NVFP4 x NVFP4 GEMM on the sm_103a tensor cores (tcgen05).
//
// D[m][n] = g_A * g_B * sum_k (a_mk * sA_{m,k/16}) (b_nk * sB_{n,k/16}), FP32
// accumulation in tensor memory: the W4A4 product the hyper.ai story on the
// Nemotron 3 Ultra NVFP4 checkpoint says Blackwell runs natively, on the
// format of "NVIDIA Introduces a 4-Bit Pretraining Methodology Using NVFP4"
// ("Summary").
//
// Persistent kernel on CTA pairs (clusters of 2, one CTA per SM).  A pair
// computes a 256 x 256 output tile with tcgen05.mma.cta_group::2 (M = 256,
// N = 256, K = 64 per instruction, kind::mxf4nvf4.block_scale.scale_vec::4X):
// CTA r of the pair holds rows 128r..128r+127 of the A tile and of the B tile
// in its shared memory and rows 128r.. of the accumulator in its tensor
// memory, so each SM loads a quarter of the tile's operand bytes.  Roles in
// each CTA (16 warps = 4 warpgroups):
//   warp 0       TMA producer: its A and B halves (128 B of K = 256 elements
//                per row, 128B swizzle; completion counted on the leader
//                CTA's barrier) into a 5-stage ring.
//   warp 1       tensor memory owner (both CTAs allocate together); in the
//                leader CTA one thread issues the pair's MMAs and commits to
//                both CTAs' barriers.
//   warp 2       scale producer: the stage's scale atoms by cp.async.bulk on a
//                barrier of their own (issuing them from warp 0 as well slowed
//                the operand stream by ~15%).
//   warp 3       idle after setup.
//   warps 4..7   scale warps: tcgen05.st of the stage's scale bytes into the
//                CTA's tensor memory.  For K-step j the MMA reads the 4 scales
//                of row r from lane r % 32, column (scale address + r / 32) of
//                every lane quarter (the layout tcgen05.cp .32x128b.warpx4
//                makes), scale address = slot + 4j (A), slot + 8j (B).
//   warps 8..15  epilogue: two warps per lane quarter drain the CTA's 128 x 256
//                accumulator half with tcgen05.ld (all 128 columns of a warp in
//                one round trip), release it, scale by g_A*g_B, convert, and
//                write 32 x 128-byte boxes through swizzled shared memory with
//                TMA stores while the next tile's mainloop runs.  The output
//                map covers the whole 16-byte units of a row (a TMA store is
//                clipped per 16-byte unit); a row's last partial unit is
//                written with plain stores.
// The two epilogue warpgroups raise their register limit (setmaxnreg) to hold
// a warp's 128 accumulator columns at once; the other two lower theirs to
// pay for it.
// Tensor maps are prefetched into the copy engine's descriptor cache during
// setup, and (grouped GEMM) the next group's while the current tile runs.
// Every mbarrier wait is bounded (kWaitLimitNs, or the limit a failure-
// detection test passes).  On expiry the CTA records a timeout in a device
// word, every role leaves its loop, in-flight copies and MMAs are waited for
// (bounded), both CTAs meet at a final cluster barrier, tensor memory is
// freed and the kernel returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "gemm.h"
#include "nvfp4_device.cuh"

namespace nvfp4 {
namespace {

constexpr int BM = 128;             // rows per CTA (the pair covers 256)
constexpr int BN = 256;             // output columns per tile
constexpr int BNH = BN / 2;         // B rows held by one CTA
constexpr int BKB = 128;            // bytes of K per stage per row = 256 FP4 elements
constexpr int STAGES = 5;
constexpr int A_BYTES = BM * BKB;   // 16 KB
constexpr int B_BYTES = BNH * BKB;  // 16 KB
constexpr int SFA_BYTES = 4 * 512;  // 4 K-atoms of the CTA's 128 A rows
constexpr int SFB_BYTES = 2 * 4 * 512;  // both 128-row blocks of B: each CTA's MMA half reads all 256 columns' scales
constexpr int EPI_WARPS = 8;
constexpr int EPI_BYTES = 32 * 128;  // one 32-row x 128-byte box per epilogue warp
constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;
constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
constexpr int OFF_EPI = OFF_SFB + STAGES * SFB_BYTES;
constexpr int OFF_BAR = OFF_EPI + EPI_WARPS * EPI_BYTES;
constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;  // + barriers + alignment slack
constexpr int TMEM_COLS = 512;
constexpr int SFA_COL0 = BN;                             // 16 columns per stage
constexpr int SFB_COL0 = (SFA_COL0 + 16 * STAGES + 31) / 32 * 32;  // 32 columns per stage
constexpr int NUM_WARPS = 8 + EPI_WARPS;  // warpgroups 0-1: producers, MMA, scale warps; 2-3: epilogue
constexpr int NUM_THREADS = 32 * NUM_WARPS;
// Register split: the kernel is launched with kRegsLaunch per thread; after
// setup warpgroups 0-1 drop to kRegsLow and the epilogue warpgroups rise to
// kRegsHigh.  setmaxnreg.inc waits until the registers exist, so the split
// must add up to exactly what the block was launched with (the host checks
// the compiled count before the first launch).
constexpr int kRegsLaunch = 65536 / NUM_THREADS;  // 128
constexpr int kRegsLow = 88, kRegsHigh = 168;
static_assert(NUM_WARPS == 16 && EPI_WARPS == 8, "role layout: four whole warpgroups, the last two the epilogue");
static_assert(2 * 128 * kRegsLow + 2 * 128 * kRegsHigh == NUM_THREADS * kRegsLaunch, "setmaxnreg split");
static_assert(kRegsLow % 8 == 0 && kRegsHigh % 8 == 0 && kRegsHigh <= 256, "setmaxnreg operands");
constexpr int GROUP_M = 8;  // raster: bands of 8 pair rows
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s
static_assert(SFB_COL0 + 32 * STAGES <= TMEM_COLS, "TMEM budget");
static_assert(SFA_COL0 % 16 == 0 && SFB_COL0 % 32 == 0, "tcgen05.st .x16/.x32 need aligned columns");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(OFF_EPI % 1024 == 0 && OFF_B % 1024 == 0, "swizzled buffers need 1024-byte alignment");

// instruction descriptor: E2M1 x E2M1 (kind::mxf4nvf4 encoding 1), UE4M3
// scales, K-major A and B, dense K = 64, N = 256, M = 256 (the pair).
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)((2 * BM) >> 4) << 24);

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ unsigned long long now_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t num_clusters() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// shared::cluster address of the same shared-memory offset in CTA `rank`
__device__ __forceinline__ uint32_t peer_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// arrive on a barrier given by its shared::cluster address (own or peer CTA).
// Relaxed: what it publishes is tensor-memory state already completed by
// tcgen05.wait::ld/st and ordered by tcgen05.fence::before_thread_sync; a
// release at cluster scope would add a full memory fence on the scale path
// of every K-step (measured: the pair kernel ran at half speed with it).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cbar) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cbar) : "memory");
}
// CTA-scope poll: every barrier here guards tensor-memory or async-proxy data
// (TMA, tensor core), ordered by the tcgen05 fences around the waits, not
// generic memory of the peer; a cluster-scope acquire cost ~130 cycles a poll.
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
// one non-blocking test of a phase
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: true when the phase completed; false on abort or timeout
// (a timeout raises the CTA's abort flag and the device error word).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, unsigned int* err,
                                          unsigned long long limit) {
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

// Short bounded wait used only on the way out.
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = now_ns();
  while (!mbar_try_wait(bar, parity) && now_ns() - t0 < 100000000ull) {
  }
}

// TMA load into this CTA's shared memory; completion is counted on the
// barrier at shared::cluster address `cbar` (the leader CTA's, for the pair).
__device__ __forceinline__ void tma_load_pair(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t cbar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(cbar)
      : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(src)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// Bring a tensor map (kernel parameter) into the copy engine's descriptor
// cache ahead of its first use.
__device__ __forceinline__ void prefetch_tensor_map(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// arrive (once, when this thread's MMAs complete) on the barrier at the same
// offset in both CTAs of the pair
__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"((uint16_t)3)
      : "memory");
}
__device__ __forceinline__ void tc_mma_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t sfa, uint32_t sfb,
                                            uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(kIdesc), "r"(acc), "r"(sfa), "r"(sfb)
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

#define NVFP4_LD32(taddr, r)                                                                                         \
  asm volatile(                                                                                                      \
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"  \
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"                                                 \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), \
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),     \
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),    \
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])                  \
      : "r"(taddr)                                                                                                   \
      : "memory")

// The registers written by a tcgen05.ld are only valid after tcgen05.wait::ld;
// this empty asm names them as read-write after the wait, so no use of them
// can be scheduled before it.
#define NVFP4_LD_FENCE(r)                                                                                            \
  asm volatile(""                                                                                                    \
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),    \
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),           \
                 "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),         \
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),         \
                 "+r"(r[29]), "+r"(r[30]), "+r"(r[31])                                                              \
               :                                                                                                     \
               : "memory")

// K-major operand tile, 128-byte rows, 128B swizzle: 8-row atoms of 1024 B.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 p = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&p);
}

// One pair tile (256 x 256 outputs) and the operands it reads.
struct Tile {
  const CUtensorMap* tmA;
  const CUtensorMap* tmB;
  const CUtensorMap* tmD;
  const uint8_t* sfa;
  const uint8_t* sfb;
  const float* ga;
  const float* gb;
  int M, N, K;
  int pm, pn;  // pair-row (256-row) and column (256-col) tile indices
  int n_tma;   // columns the output map covers (whole 16-byte units of a row)
  void* d;     // D and its leading dimension, for the columns past n_tma
  int64_t ldd;
};

// Raster order: bands of GROUP_M pair rows; inside a band columns advance
// slowest, so the pairs working at one time share A and B rows in L2.
__device__ __forceinline__ void raster(int t, int mt, int nt, int& pm, int& pn) {
  const int band_tiles = GROUP_M * nt;
  const int band = t / band_tiles, in = t % band_tiles;
  const int rows = min(GROUP_M, mt - band * GROUP_M);
  pm = band * GROUP_M + in % rows;
  pn = in / rows;
}

struct SingleSched {
  static constexpr bool kMapsVary = false;  // one set of tensor maps for every tile
  const CUtensorMap* tmA;
  const CUtensorMap* tmB;
  const CUtensorMap* tmD;
  const GemmArgs* a;
  __device__ int num_tiles() const { return ((a->M + 2 * BM - 1) / (2 * BM)) * ((a->N + BN - 1) / BN); }
  __device__ Tile get(int t) const {
    Tile x{tmA, tmB, tmD, a->sfa, a->sfb, a->ga, a->gb, a->M, a->N, a->K, 0, 0, a->n_tma, a->d, a->ldd};
    raster(t, (a->M + 2 * BM - 1) / (2 * BM), (a->N + BN - 1) / BN, x.pm, x.pn);
    return x;
  }
};

struct GroupedSched {
  static constexpr bool kMapsVary = true;  // one set of tensor maps per group
  const GroupedArgs* g;
  __device__ int num_tiles() const { return g->tile_start[g->count]; }
  __device__ Tile get(int t) const {
    int e = 0, hi = g->count - 1;  // the last group whose first tile is <= t (binary search)
    while (e < hi) {
      const int mid = (e + hi + 1) >> 1;
      if (g->tile_start[mid] <= t) e = mid;
      else hi = mid - 1;
    }
    // (every group's row is a whole number of 16-byte units: ldd = N_e)
    Tile x{&g->tmA[e], &g->tmB[e], &g->tmD[e], g->sfa[e], g->sfb[e], g->ga[e], g->gb[e], g->M[e], g->N[e], g->K[e], 0, 0,
           g->N[e], nullptr, 0};
    raster(t - g->tile_start[e], (g->M[e] + 2 * BM - 1) / (2 * BM), (g->N[e] + BN - 1) / BN, x.pm, x.pn);
    return x;
  }
};

// Encode one epilogue thread's row segment of BF16 outputs (128 columns from
// col0, packed two per word) as NVFP4 with 1D blocks along N: exactly the
// encoder's max-6 / round-to-nearest-even sequence (include/nvfp4.h) with g
// from the supplied amax.  Codes go to row r of the [M][N/2] code matrix; the
// two 4-block scale words to their atoms (zeros for rows >= M and blocks past
// N, which are the layout's padding).
__device__ __forceinline__ void encode_row_segment(const GemmQuantOut& qo, const uint32_t (&pk)[64], int r, int col0,
                                                   int M, int N, float g, float g6) {
  const int KB = N >> 4, nka = (KB + 3) >> 2;
  const bool row_ok = r < M;
  uint32_t sw[2] = {0u, 0u};
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int kb = (col0 >> 4) + j;
    if (row_ok && kb < KB) {
      float v[16];
      uint32_t mx = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t w = pk[8 * j + i];
        v[2 * i] = bf16_lo(w);
        v[2 * i + 1] = bf16_hi(w);
        mx = __vmaxu2(mx, w & 0x7FFF7FFFu);
      }
      const float amax_b = __uint_as_float(max(mx & 0xFFFFu, mx >> 16) << 16);
      float sv, rcp;
      const uint32_t sb = block_scale(amax_b, g6, g, sv, rcp);
      *reinterpret_cast<uint2*>(qo.codes + (int64_t)r * (N >> 1) + kb * 8) = encode16<false>(v, rcp, nullptr);
      sw[j >> 2] |= sb << (8 * (j & 3));
    }
  }
#pragma unroll
  for (int a = 0; a < 2; ++a) {
    const int ka = (col0 >> 6) + a;
    if (ka < nka)
      *reinterpret_cast<uint32_t*>(qo.scales + ((int64_t)(r >> 7) * nka + ka) * 512 + (r & 31) * 16 +
                                   ((r >> 5) & 3) * 4) = sw[a];
  }
}

// hold_tx and wait_ns: the failure-detection test's withheld bytes and wait
// limit (both 0 in normal launches).
// OUT_BF16: BF16 output (else FP32); a compile-time choice so that each
// kernel holds one epilogue.
template <class Sched, bool QOUT, bool OUT_BF16>
__device__ __forceinline__ void gemm_pairs(const Sched& sched, unsigned int* err,
                                           unsigned int* amax_out, const GemmQuantOut* qo = nullptr,
                                           uint32_t hold_tx = 0, unsigned long long wait_ns = 0) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  // per CTA: full[S] (leader: A/B bytes of both CTAs + the 8 scale warps of
  // the pair, so the MMA thread polls one barrier per stage), sf_full[S] (own
  // scale bytes), empty[S], accum_full, accum_empty (leader: 16 epilogue
  // warps), drain
  const uint32_t full0 = smem_u32(bars), sff0 = full0 + 8 * STAGES, empty0 = sff0 + 8 * STAGES;
  const uint32_t accum_full = empty0 + 8 * STAGES, accum_empty = accum_full + 8, drain = accum_empty + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * STAGES + 3);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int num_tiles = sched.num_tiles();
  const int first = (int)cluster_id(), step = (int)num_clusters();
  const unsigned long long limit = wait_ns ? wait_ns : kWaitLimitNs;

  if constexpr (QOUT) {
    if (blockIdx.x == 0 && threadIdx.x == 0) {  // the encoded tensor's scalars
      const float amax = *qo->amax_in;
      *qo->global_scale = global_scale(amax);
      *qo->amax = amax;
    }
  }
  if (threadIdx.x == 32 * 3 && first < num_tiles) {
    // the first tile's maps start their way into the copy engine during setup
    const Tile x0 = sched.get(first);
    prefetch_tensor_map(x0.tmA);
    prefetch_tensor_map(x0.tmB);
    // (a zero map when D is not stored, or when no row holds a whole 16-byte unit)
    if ((!QOUT || qo->store_d) && x0.n_tma > 0) prefetch_tensor_map(x0.tmD);
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1 + 8);
      mbar_init(sff0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_init(accum_full, 1);
    mbar_init(accum_empty, 2 * EPI_WARPS);
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {  // both CTAs: the pair's tensor memory is allocated together
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers are initialised before any remote signal
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the register split: each warpgroup executes one setmaxnreg together, and
  // only the epilogue code follows the increase
  if (warp < 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
    if (warp == 0) {
      // ---------------- TMA producer (each CTA: its halves) ----------------
      if (lane == 0) {
        uint32_t it = 0;
        const uint32_t lead_full0 = peer_addr(full0, 0);
        for (int t = first; t < num_tiles && !*abort_flag; t += step) {
          const Tile x = sched.get(t);
          if (Sched::kMapsVary && t + step < num_tiles) {  // the next tile's maps (another group's)
            const Tile xn = sched.get(t + step);
            if (xn.tmA != x.tmA) prefetch_tensor_map(xn.tmA);
            if (xn.tmB != x.tmB) prefetch_tensor_map(xn.tmB);
          }
          const int nk = (x.K + 255) / 256;  // the last stage's box is zero-filled past K
          const int m_tile = 2 * x.pm + (int)rank;               // this CTA's 128 A rows
          const bool a_valid = m_tile * BM < x.M;
          const int nb_mine = 2 * x.pn + (int)rank;              // this CTA's 128 B rows
          const bool b_valid = nb_mine * 128 < x.N;
          // the leader's halves always exist; the peer's may not (M or N % 256 == 128)
          const uint32_t ab_tx = A_BYTES * (1 + ((2 * x.pm + 1) * BM < x.M)) + B_BYTES * (1 + ((2 * x.pn + 1) * 128 < x.N));
          for (int kt = 0; kt < nk; ++kt, ++it) {
            const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
            if (!mbar_wait(empty0 + 8 * s, ph ^ 1, abort_flag, err, limit)) break;
            // A/B: the leader expects both CTAs' bytes on its own barrier
            if (leader) mbar_expect_tx(full0 + 8 * s, ab_tx + (it == 0 ? hold_tx : 0u));
            const uint32_t fb = lead_full0 + 8 * s;
            if (a_valid) tma_load_pair(smem_u32(smem + OFF_A + s * A_BYTES), x.tmA, kt * BKB, m_tile * BM, fb);
            if (b_valid) tma_load_pair(smem_u32(smem + OFF_B + s * B_BYTES), x.tmB, kt * BKB, nb_mine * 128, fb);
          }
        }
        if (*abort_flag) {
          // Copies already issued must land before the pair leaves.  They
          // complete on the leader's full barriers, which the leader drains
          // (bounded: a phase whose scale-warp arrivals were abandoned never
          // completes); the peer cannot observe them and waits 2 ms instead.
          if (leader) {
            for (uint32_t i = it > STAGES ? it - STAGES : 0; i < it; ++i)
              mbar_drain(full0 + 8 * (i % STAGES), (i / STAGES) & 1);
          } else {
            const unsigned long long t0 = now_ns();
            while (now_ns() - t0 < 2000000ull) {
            }
          }
        }
      }
    } else if (warp == 1) {
      // ---------------- MMA issuer (leader CTA) ----------------
      if (leader && lane == 0) {
        // the MMA issue queue is shallow, so every cycle spent between stages
        // idles the tensor pipe: one barrier poll per stage, stage and phase kept
        // incrementally, descriptors advanced by adding to their address field
        // (K-step j is 32 bytes = 2 units further; a stage is A_BYTES / 16 units)
        // The next stage's barrier is tested between the MMAs of the current
        // one, while the tensor pipe is busy, so a ready stage costs no poll.
        const uint64_t da0 = desc_sw128(smem_u32(smem + OFF_A)), db0 = desc_sw128(smem_u32(smem + OFF_B));
        uint32_t s = 0, ph = 0, ti = 0;
        bool ok = true, next_ready = false;
        for (int t = first; t < num_tiles && ok; t += step, ++ti) {
          const Tile x = sched.get(t);
          const int nk = (x.K + 255) / 256, nkc = x.K / 64;
          if (!mbar_wait(accum_empty, (ti & 1) ^ 1, abort_flag, err, limit)) break;
          tc_fence_after();
          for (int kt = 0; kt < nk; ++kt) {
            if (!next_ready && !mbar_wait(full0 + 8 * s, ph, abort_flag, err, limit)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sn = s + 1 == STAGES ? 0 : s + 1, phn = s + 1 == STAGES ? ph ^ 1 : ph;
            const uint64_t da = da0 + (uint64_t)(s * (A_BYTES >> 4)), db = db0 + (uint64_t)(s * (B_BYTES >> 4));
            const uint32_t sfa = tmem + SFA_COL0 + 16 * s, sfb = tmem + SFB_COL0 + 32 * s;
            const int kc = nkc - 4 * kt;  // K-steps of 64 left: 4 or more except in a K-tail stage
            if (kc >= 4) {
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                tc_mma_pair(tmem, da + 2 * j, db + 2 * j, sfa + 4 * j, sfb + 8 * j, (kt | j) != 0);
                if (j == 2) next_ready = mbar_test(full0 + 8 * sn, phn);
              }
            } else {
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                if (j < kc) tc_mma_pair(tmem, da + 2 * j, db + 2 * j, sfa + 4 * j, sfb + 8 * j, (kt | j) != 0);
                if (j == 2) next_ready = mbar_test(full0 + 8 * sn, phn);
              }
            }
            tc_commit_pair(empty0 + 8 * s);
            s = sn;
            ph = phn;
          }
          next_ready = next_ready && ok;
          if (ok) tc_commit_pair(accum_full);
        }
        tc_commit_pair(drain);  // arrives when every MMA this thread issued has completed
        mbar_drain(drain, 0);
      }
    } else if (warp >= 4) {
      // ---------------- scale warps: shared memory -> TMEM ----------------
      const uint32_t q = warp & 3;
      const uint32_t lane_base = (q * 32) << 16;
      const uint32_t lead_full0 = peer_addr(full0, 0);
      uint32_t it = 0;
      bool ok = true;
      for (int t = first; t < num_tiles && ok; t += step) {
        const Tile x = sched.get(t);
        const int nk = (x.K + 255) / 256;
        for (int kt = 0; kt < nk; ++kt, ++it) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
          // warp vote: the tcgen05.st below is warp-collective
          if (!__all_sync(0xFFFFFFFFu, mbar_wait(sff0 + 8 * s, ph, abort_flag, err, limit))) {
            ok = false;
            break;
          }
          // the slot's previous MMAs completed before these bytes were copied
          // (the scale producer waited for them): order the stores after them
          tc_fence_after();
          // lane l: row l of every 512-byte atom = 16 bytes = 4 consecutive columns
          const uint4* sa = reinterpret_cast<const uint4*>(smem + OFF_SFA + s * SFA_BYTES) + lane;
          const uint4* sb = reinterpret_cast<const uint4*>(smem + OFF_SFB + s * SFB_BYTES) + lane;
          uint32_t va[16], vb[32];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint4 wa = sa[j * 32];
            va[4 * j] = wa.x; va[4 * j + 1] = wa.y; va[4 * j + 2] = wa.z; va[4 * j + 3] = wa.w;
            const uint4 w0 = sb[j * 32];        // B rows 0..127 of the tile
            const uint4 w1 = sb[128 + j * 32];  // B rows 128..255
            vb[8 * j] = w0.x; vb[8 * j + 1] = w0.y; vb[8 * j + 2] = w0.z; vb[8 * j + 3] = w0.w;
            vb[8 * j + 4] = w1.x; vb[8 * j + 5] = w1.y; vb[8 * j + 6] = w1.z; vb[8 * j + 7] = w1.w;
          }
          tmem_st16(tmem + lane_base + SFA_COL0 + 16 * s, va);
          tmem_st32(tmem + lane_base + SFB_COL0 + 32 * s, vb);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(lead_full0 + 8 * s);
        }
      }
    } else if (warp == 2) {
      // ---------------- scale producer (each CTA: its scale atoms) ----------------
      if (lane == 0) {
        uint32_t it = 0;
        for (int t = first; t < num_tiles && !*abort_flag; t += step) {
          const Tile x = sched.get(t);
          const int nk = (x.K + 255) / 256;
          const int nka = x.K / 64;  // 4-block scale atoms per 128 rows (K % 64 == 0)
          const int m_tile = 2 * x.pm + (int)rank;
          const bool a_valid = m_tile * BM < x.M;
          // 128-row scale blocks of B that exist (the buffer is padded to 128 rows)
          const int sfb_blocks = min(2, (x.N - x.pn * BN + 127) / 128);
          const int sfb_first = 2 * x.pn;
          for (int kt = 0; kt < nk; ++kt, ++it) {
            const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
            if (!mbar_wait(empty0 + 8 * s, ph ^ 1, abort_flag, err, limit)) break;
            // the atoms of this stage's K-steps: 4, or fewer at a K tail (the
            // next atoms in memory belong to the next 128 rows)
            const uint32_t bytes = (uint32_t)min(4, nka - 4 * kt) * 512;
            const uint32_t sb = sff0 + 8 * s;
            mbar_expect_tx(sb, (a_valid ? bytes : 0) + sfb_blocks * bytes);
            if (a_valid)
              bulk_g2s(smem_u32(smem + OFF_SFA + s * SFA_BYTES), x.sfa + ((int64_t)m_tile * nka + 4 * kt) * 512,
                       bytes, sb);
            for (int nb = 0; nb < sfb_blocks; ++nb)
              bulk_g2s(smem_u32(smem + OFF_SFB + s * SFB_BYTES + nb * 2048),
                       x.sfb + ((int64_t)(sfb_first + nb) * nka + 4 * kt) * 512, bytes, sb);
          }
        }
        // copies already issued land on this CTA's own scale barriers: drain
        // the last round of every slot before the CTA leaves
        if (*abort_flag)
          for (uint32_t i = it > STAGES ? it - STAGES : 0; i < it; ++i) mbar_drain(sff0 + 8 * (i % STAGES), (i / STAGES) & 1);
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
    // ---------------- epilogue (each CTA: its 128 accumulator rows) ----------------
    const int e = warp - 8;
    const uint32_t q = warp & 3, half = e >> 2;
    const uint32_t taddr0 = tmem + ((q * 32) << 16) + half * 128;
    uint8_t* stage = smem + OFF_EPI + e * EPI_BYTES;
    const uint32_t stage_u32 = smem_u32(stage);
    const uint32_t lead_accum_empty = peer_addr(accum_empty, 0);
    uint32_t ti = 0;
    [[maybe_unused]] const CUtensorMap* prev_d = nullptr;
    for (int t = first; t < num_tiles; t += step, ++ti) {
      const Tile x = sched.get(t);
      if constexpr (Sched::kMapsVary) {
        if (x.tmD != prev_d) {  // the group's output map, fetched while the mainloop runs
          if (e == 0 && lane == 0) prefetch_tensor_map(x.tmD);
          prev_d = x.tmD;
        }
      }
      // warp vote: tcgen05.ld is warp-collective
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(accum_full, ti & 1, abort_flag, err, limit))) break;
      tc_fence_after();
      const float alpha = __fmul_rn(*x.ga, *x.gb);
      const int col0 = x.pn * BN + half * 128;
      const int row0 = (2 * x.pm + (int)rank) * BM + q * 32;
      // warp-uniform: this warp's 32 rows x 128 columns hold at least one
      // output; stores of partial boxes are clipped by the tensor map, and
      // boxes wholly past N are skipped
      const bool active = col0 < x.N && row0 < x.M;
      const int ncols = x.N - col0;           // valid columns of this warp's 128 (may exceed 128)
      const bool row_ok = row0 + lane < x.M;  // this thread's row exists
      if constexpr (QOUT || OUT_BF16) {  // (the quantizing variant always forms BF16 outputs)
        uint32_t pk[64];
        if (active) {
          // the warp's 128 columns in one round trip; the accumulator is
          // released as soon as they are in registers, before converting
          uint32_t r0[32], r1[32], r2[32], r3[32];
          NVFP4_LD32(taddr0, r0);
          NVFP4_LD32(taddr0 + 32, r1);
          NVFP4_LD32(taddr0 + 64, r2);
          NVFP4_LD32(taddr0 + 96, r3);
          tmem_ld_wait();
          NVFP4_LD_FENCE(r0);
          NVFP4_LD_FENCE(r1);
          NVFP4_LD_FENCE(r2);
          NVFP4_LD_FENCE(r3);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(lead_accum_empty);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            pk[i] = pack_bf16(__fmul_rn(alpha, __uint_as_float(r0[2 * i])), __fmul_rn(alpha, __uint_as_float(r0[2 * i + 1])));
            pk[16 + i] =
                pack_bf16(__fmul_rn(alpha, __uint_as_float(r1[2 * i])), __fmul_rn(alpha, __uint_as_float(r1[2 * i + 1])));
            pk[32 + i] =
                pack_bf16(__fmul_rn(alpha, __uint_as_float(r2[2 * i])), __fmul_rn(alpha, __uint_as_float(r2[2 * i + 1])));
            pk[48 + i] =
                pack_bf16(__fmul_rn(alpha, __uint_as_float(r3[2 * i])), __fmul_rn(alpha, __uint_as_float(r3[2 * i + 1])));
          }
        }
        if (!active) {  // nothing was loaded: release right away
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(lead_accum_empty);
        }
        if (amax_out && active) {
          // producer amax of the stored BF16 values: |x| bit patterns order
          // like unsigned integers, two per word (word i = columns 2i, 2i+1);
          // elements outside M x N are left out
          uint32_t mx = 0;
          if (ncols >= 128) {
#pragma unroll
            for (int i = 0; i < 64; ++i) mx = __vmaxu2(mx, pk[i] & 0x7FFF7FFFu);
          } else {
#pragma unroll
            for (int i = 0; i < 64; ++i) {
              const uint32_t keep = 2 * i + 1 < ncols ? 0x7FFF7FFFu : (2 * i < ncols ? 0x00007FFFu : 0u);
              mx = __vmaxu2(mx, pk[i] & keep);
            }
          }
          if (!row_ok) mx = 0;
          uint32_t m = max(mx & 0xFFFFu, mx >> 16) << 16;
          m = __reduce_max_sync(0xFFFFFFFFu, m);
          if (lane == 0 && m) atomicMax(amax_out, m);
        }
        if constexpr (QOUT) {
          // the next layer's NVFP4 input from the BF16 values just formed; a
          // CTA whose 128 rows start below M owns its scale atoms' padding too
          if ((2 * x.pm + (int)rank) * BM < x.M && col0 < x.N) {
            const float g = global_scale(*qo->amax_in);
            encode_row_segment(*qo, pk, row0 + lane, col0, x.M, x.N, g, __fmul_rn(6.0f, g));
          }
        }
        if (active && (!QOUT || qo->store_d)) {
          // this warp's columns inside whole 16-byte units (all of them when quantizing: N % 16 == 0)
          const int ntma = QOUT ? ncols : x.n_tma - col0;
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {  // 64 columns = one 128-byte box row
            if (64 * cc >= ntma) break;
            if (lane == 0) bulk_wait_read0();
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 8; ++i)
              *reinterpret_cast<uint4*>(stage + lane * 128 + ((i ^ (lane & 7)) << 4)) =
                  make_uint4(pk[32 * cc + 4 * i], pk[32 * cc + 4 * i + 1], pk[32 * cc + 4 * i + 2], pk[32 * cc + 4 * i + 3]);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(x.tmD, stage_u32, col0 + 64 * cc, row0);
              bulk_commit();
            }
          }
          // (the quantizing variant has N % 16 == 0: whole units only)
          if (!QOUT && ntma < ncols && ntma < 128 && row_ok) {
            // the last partial 16-byte unit of the row (1..7 columns from t0,
            // a multiple of 8): its 4 words picked without dynamic indexing
            const int t0 = max(ntma, 0), cnt = min(ncols, 128) - t0, gsel = t0 >> 3;
            uint32_t w4[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int gi = 0; gi < 16; ++gi)
              if (gi == gsel) {
                w4[0] = pk[4 * gi];
                w4[1] = pk[4 * gi + 1];
                w4[2] = pk[4 * gi + 2];
                w4[3] = pk[4 * gi + 3];
              }
            unsigned short* dst =
                reinterpret_cast<unsigned short*>(x.d) + (int64_t)(row0 + lane) * x.ldd + col0 + t0;
#pragma unroll
            for (int j = 0; j < 7; ++j)
              if (j < cnt) dst[j] = (unsigned short)(w4[j >> 1] >> (16 * (j & 1)));
          }
        }
      } else {
        // the warp's 128 columns in one round trip, then the accumulator is
        // released before the four 32-column boxes are staged and stored
        uint32_t r0[32], r1[32], r2[32], r3[32];
        if (active) {
          NVFP4_LD32(taddr0, r0);
          NVFP4_LD32(taddr0 + 32, r1);
          NVFP4_LD32(taddr0 + 64, r2);
          NVFP4_LD32(taddr0 + 96, r3);
          tmem_ld_wait();
          NVFP4_LD_FENCE(r0);
          NVFP4_LD_FENCE(r1);
          NVFP4_LD_FENCE(r2);
          NVFP4_LD_FENCE(r3);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(lead_accum_empty);
        const int ntma = x.n_tma - col0;
        // one 32-column chunk: scaled in place (one product per output), then
        // the producer amax, the TMA box and the row's partial last unit
        auto chunk = [&](uint32_t (&r)[32], const int c) {
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__fmul_rn(alpha, __uint_as_float(r[i])));
          if (amax_out && active) {
            uint32_t m = 0;
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (32 * c + i < ncols) m = max(m, r[i] & 0x7FFFFFFFu);
            if (!row_ok) m = 0;
            m = __reduce_max_sync(0xFFFFFFFFu, m);
            if (lane == 0 && m) atomicMax(amax_out, m);
          }
          if (active && 32 * c < ntma) {
            if (lane == 0) bulk_wait_read0();
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 8; ++i)
              *reinterpret_cast<uint4*>(stage + lane * 128 + ((i ^ (lane & 7)) << 4)) =
                  make_uint4(r[4 * i], r[4 * i + 1], r[4 * i + 2], r[4 * i + 3]);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(x.tmD, stage_u32, col0 + 32 * c, row0);
              bulk_commit();
            }
          }
          // the last partial 16-byte unit of the row (1..3 columns from t0, a
          // multiple of 4), when it lies in this 32-column chunk
          const int t0 = max(ntma, 0);
          if (!QOUT && active && row_ok && ntma < ncols && ntma < 128 && (t0 >> 5) == c) {
            const int cnt = min(ncols, 128) - t0, osel = (t0 & 31) >> 2;
            uint32_t v4[3] = {0u, 0u, 0u};
#pragma unroll
            for (int oi = 0; oi < 8; ++oi)
              if (oi == osel) {
                v4[0] = r[4 * oi];
                v4[1] = r[4 * oi + 1];
                v4[2] = r[4 * oi + 2];
              }
            uint32_t* dst = reinterpret_cast<uint32_t*>(x.d) + (int64_t)(row0 + lane) * x.ldd + col0 + t0;
#pragma unroll
            for (int j = 0; j < 3; ++j)
              if (j < cnt) dst[j] = v4[j];
          }
        };
        chunk(r0, 0);
        chunk(r1, 1);
        chunk(r2, 2);
        chunk(r3, 3);
      }
    }
    if (lane == 0) bulk_wait0();
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still signal it
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS));
  }
}

template <bool OUT_BF16>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
           const __grid_constant__ CUtensorMap tmD, const __grid_constant__ GemmArgs a) {
  SingleSched s{&tmA, &tmB, &tmD, &a};
  gemm_pairs<SingleSched, false, OUT_BF16>(s, a.err, a.amax_out, nullptr, a.hold_tx, a.wait_ns);
}

// The GEMM with the NVFP4 encoding of its BF16 output in the epilogue.
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_gemm_quant(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmD, const __grid_constant__ GemmArgs a) {
  SingleSched s{&tmA, &tmB, &tmD, &a};
  gemm_pairs<SingleSched, true, true>(s, a.err, a.amax_out, &a.q);
}

template <bool OUT_BF16>
__global__ void __launch_bounds__(NUM_THREADS, 1) k_gemm_grouped(const __grid_constant__ GroupedArgs g) {
  GroupedSched s{&g};
  gemm_pairs<GroupedSched, false, OUT_BF16>(s, g.err, nullptr);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// Timeout word of the pipeline waits (one per device, shared by every GEMM
// launched on it) and the slot that nvfp4_sync_check's exchange reads back.
__device__ unsigned int g_device_error = 0;
__device__ unsigned int g_device_error_taken = 0;

__global__ void k_take_error() { g_device_error_taken = atomicExch(&g_device_error, 0u); }

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::atomic<EncodeTiledFn> cached{nullptr};
  EncodeTiledFn fn = cached.load(std::memory_order_acquire);
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<EncodeTiledFn>(p);
      cached.store(fn, std::memory_order_release);
    }
  }
  return fn;
}

// rows x (K/2) bytes, K-major, box = 128 B x 128 rows, 128B swizzle.  Boxes
// reaching past the last row or past K are zero-filled by the copy engine.
bool make_code_map(CUtensorMap* m, const uint8_t* codes, int64_t rows, int64_t K) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)(K / 2), (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
  cuuint32_t box[2] = {(cuuint32_t)BKB, 128};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(codes), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// D: rows x cols of bf16/fp32 with leading dimension ldd; box = 128 B x 32 rows,
// 128B swizzle.  Stores of boxes reaching past the tensor are clipped.
bool make_out_map(CUtensorMap* m, void* d, int64_t rows, int64_t cols, int64_t ldd, bool bf16) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const int es = bf16 ? 2 : 4;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(ldd * es)};
  cuuint32_t box[2] = {(cuuint32_t)(128 / es), 32};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, d, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Per-device launch state.  Everything here depends on the device (symbol
// addresses live in each device's context, the shared-memory opt-in is a
// per-device function attribute), so it is cached per device ordinal;
// concurrent first calls compute the same values, and the atomics make the
// publication safe.
constexpr int kMaxDevices = 64;
enum KernelId { kSingleF32 = 0, kSingleBf16, kSingleQuant, kGroupedF32, kGroupedBf16, kNumKernels };
struct DeviceState {
  std::atomic<unsigned int*> err{nullptr};
  std::atomic<unsigned int*> err_taken{nullptr};
  std::atomic<int> sms{0};
  std::atomic<int> max_pairs[kNumKernels] = {};
  std::atomic<bool> smem_ok[kNumKernels] = {};
};
DeviceState g_dev[kMaxDevices];

DeviceState* device_state() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  return &g_dev[dev];
}

unsigned int* symbol_addr(const unsigned int& sym) {
  void* q = nullptr;
  return cudaGetSymbolAddress(&q, sym) == cudaSuccess ? reinterpret_cast<unsigned int*>(q) : nullptr;
}

int num_sms(DeviceState* st) {
  int n = st->sms.load(std::memory_order_relaxed);
  if (n <= 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    st->sms.store(n, std::memory_order_relaxed);
  }
  return n;
}

// The shared-memory opt-in, and the check that the kernel was compiled to
// kRegsLaunch registers per thread: the setmaxnreg split inside it adds up to
// exactly that many, and with fewer the epilogue's increase would wait for
// registers that never come.
bool kernel_configured(DeviceState* st, KernelId k, const void* fn, const char** why) {
  if (st->smem_ok[k].load(std::memory_order_acquire)) return true;
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess || fa.numRegs != kRegsLaunch) {
    *why = "GEMM kernel not compiled to the register count its setmaxnreg split assumes";
    return false;
  }
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) != cudaSuccess) {
    *why = "cudaFuncSetAttribute failed";
    return false;
  }
  st->smem_ok[k].store(true, std::memory_order_release);
  return true;
}

// grid of CTA pairs: one pair per two SMs, no more pairs than tiles
template <class... Args>
cudaError_t launch_pairs(void (*kernel)(Args...), int pair_tiles, DeviceState* st, KernelId k, cudaStream_t s,
                         Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int max_pairs = st->max_pairs[k].load(std::memory_order_relaxed);
  if (max_pairs <= 0) {  // pairs that can be resident at once (clusters live inside one GPC)
    cfg.gridDim = dim3(2 * (unsigned)(num_sms(st) / 2), 1, 1);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(kernel), &cfg) != cudaSuccess || n <= 0)
      n = num_sms(st) / 2;
    max_pairs = n;
    st->max_pairs[k].store(n, std::memory_order_relaxed);
  }
  const int pairs = pair_tiles < max_pairs ? pair_tiles : max_pairs;
  cfg.gridDim = dim3((unsigned)(2 * (pairs > 0 ? pairs : 1)), 1, 1);
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace

bool make_tile_map_2d(CUtensorMap* m, const void* base, bool bf16, int64_t rows, int64_t cols, int64_t ld,
                      uint32_t box_cols, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const int es = bf16 ? 2 : 4;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(ld * es)};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base),
            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

unsigned int* device_error_word() {
  DeviceState* st = device_state();
  if (!st) return nullptr;
  unsigned int* p = st->err.load(std::memory_order_acquire);
  if (!p) {
    p = symbol_addr(g_device_error);
    if (p) st->err.store(p, std::memory_order_release);
  }
  return p;
}

cudaError_t take_device_error(cudaStream_t s, unsigned int* value) {
  DeviceState* st = device_state();
  if (!st) return cudaErrorInvalidDevice;
  unsigned int* p = st->err_taken.load(std::memory_order_acquire);
  if (!p) {
    p = symbol_addr(g_device_error_taken);
    if (!p) return cudaErrorInvalidSymbol;
    st->err_taken.store(p, std::memory_order_release);
  }
  k_take_error<<<1, 1, 0, s>>>();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaMemcpyAsync(value, p, sizeof(unsigned int), cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(s);
}

namespace {
std::atomic<unsigned long long> g_armed_wait[3];  // [op]: armed wait limit in ns, 0 = not armed
}  // namespace

void arm_wait_expiry(int op, unsigned long long limit_ns) {
  if (op >= 1 && op <= 2) g_armed_wait[op].store(limit_ns, std::memory_order_release);
}
unsigned long long take_armed_wait(int op) {
  if (op < 1 || op > 2) return 0;
  // cheap test first: the normal launch path never writes the flag
  if (g_armed_wait[op].load(std::memory_order_relaxed) == 0) return 0;
  return g_armed_wait[op].exchange(0, std::memory_order_acq_rel);
}

int gemm_tile_m() { return 2 * BM; }
int gemm_tile_n() { return BN; }

cudaError_t launch_gemm(const GemmOperand& A, const GemmOperand& B, void* D, int64_t ldd, bool out_bf16, cudaStream_t s,
                        const char** why, float* amax_out, const GemmQuantOut* q) {
  CUtensorMap ta, tb, td = {};
  // the output map covers the whole 16-byte units of each row (TMA clips a
  // store per 16-byte unit); the kernel writes the remaining columns itself
  const int es = out_bf16 ? 2 : 4;
  const int64_t n_tma = (B.rows * es / 16) * 16 / es;
  if (!make_code_map(&ta, A.codes, A.rows, A.K) || !make_code_map(&tb, B.codes, B.rows, B.K) ||
      (D && n_tma > 0 && !make_out_map(&td, D, A.rows, n_tma, ldd, out_bf16))) {
    *why = "cuTensorMapEncodeTiled failed (or driver entry point unavailable)";
    return cudaErrorInvalidValue;
  }
  DeviceState* st = device_state();
  unsigned int* err = device_error_word();
  if (!st || !err) {
    *why = "device error word unavailable";
    return cudaErrorInvalidValue;
  }
  const KernelId kid = q ? kSingleQuant : out_bf16 ? kSingleBf16 : kSingleF32;
  auto kernel = q ? k_gemm_quant : out_bf16 ? k_gemm<true> : k_gemm<false>;
  if (!kernel_configured(st, kid, reinterpret_cast<const void*>(kernel), why)) return cudaErrorInvalidValue;
  GemmArgs a{A.scales, B.scales, A.g, B.g, (int)A.rows, (int)B.rows, (int)A.K, err,
             reinterpret_cast<unsigned int*>(amax_out), q ? *q : GemmQuantOut{}, D, ldd, (int)n_tma, 0u, 0ull};
  if (!q) {
    const unsigned long long lim = take_armed_wait(1);
    if (lim) {  // failure-detection test: 16 bytes that no copy delivers
      a.hold_tx = 16;
      a.wait_ns = lim;
    }
  }
  const int tiles = (int)((A.rows + 2 * BM - 1) / (2 * BM)) * (int)((B.rows + BN - 1) / BN);
  cudaError_t e = launch_pairs(kernel, tiles, st, kid, s, ta, tb, td, a);
  if (e != cudaSuccess) *why = "cudaLaunchKernelEx (cluster of 2) failed";
  return e;
}

cudaError_t launch_gemm_grouped(int count, const GemmOperand* A, const GemmOperand* B, void* const* D, bool out_bf16,
                                cudaStream_t s, const char** why) {
  DeviceState* st = device_state();
  unsigned int* err = device_error_word();
  if (!st || !err) {
    *why = "device error word unavailable";
    return cudaErrorInvalidValue;
  }
  const KernelId kid = out_bf16 ? kGroupedBf16 : kGroupedF32;
  auto kernel = out_bf16 ? k_gemm_grouped<true> : k_gemm_grouped<false>;
  if (!kernel_configured(st, kid, reinterpret_cast<const void*>(kernel), why)) return cudaErrorInvalidValue;
  GroupedArgs g;
  int n = 0, tiles = 0;
  auto flush = [&]() -> cudaError_t {
    if (n == 0) return cudaSuccess;
    g.count = n;
    g.err = err;
    g.tile_start[n] = tiles;
    const int t = tiles;
    n = 0;
    tiles = 0;
    if (t == 0) return cudaSuccess;
    cudaError_t e = launch_pairs(kernel, t, st, kid, s, g);
    if (e != cudaSuccess) *why = "cudaLaunchKernelEx (cluster of 2) failed";
    return e;
  };
  for (int i = 0; i < count; ++i) {
    const GemmOperand& a = A[i];
    const GemmOperand& b = B[i];
    if (a.rows == 0 || b.rows == 0) continue;  // an empty product: nothing to write
    if (!make_code_map(&g.tmA[n], a.codes, a.rows, a.K) || !make_code_map(&g.tmB[n], b.codes, b.rows, b.K) ||
        !make_out_map(&g.tmD[n], D[i], a.rows, b.rows, b.rows, out_bf16)) {
      *why = "cuTensorMapEncodeTiled failed (or driver entry point unavailable)";
      return cudaErrorInvalidValue;
    }
    g.sfa[n] = a.scales;
    g.sfb[n] = b.scales;
    g.ga[n] = a.g;
    g.gb[n] = b.g;
    g.M[n] = (int)a.rows;
    g.N[n] = (int)b.rows;
    g.K[n] = (int)a.K;
    g.tile_start[n] = tiles;
    tiles += (int)((a.rows + 2 * BM - 1) / (2 * BM)) * (int)((b.rows + BN - 1) / BN);
    if (++n == kGroupsPerLaunch) {
      cudaError_t e = flush();
      if (e != cudaSuccess) return e;
    }
  }
  return flush();
}

}  // namespace nvfp4
