// Internal launch interface of the block-scaled GEMM (not part of the C ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace nvfp4 {

struct GemmOperand {
  const uint8_t* codes;   // [rows][K/2]
  const uint8_t* scales;  // 128x4-atom layout
  const float* g;         // per-tensor decode scale (device)
  int64_t rows, K;
};

// The epilogue's NVFP4 encoding of the BF16-rounded output (the next layer's
// input): 1D blocks of 16 along N, round to nearest even, max-6, with the
// tensor amax supplied.
struct GemmQuantOut {
  uint8_t* codes;         // [M][N/2]
  uint8_t* scales;        // 128 x 4-block atoms, ceil(M/128)*128 x ceil(N/64)*4 bytes
  float* global_scale;    // written: g = fl(amax / 2688) (1 if amax = 0)
  float* amax;            // written: the amax used
  const float* amax_in;   // read: the tensor amax to encode with
  int store_d;            // 0: D itself is not written
};

struct GemmArgs {
  const uint8_t* sfa;
  const uint8_t* sfb;
  const float* ga;
  const float* gb;
  int M, N, K;
  unsigned int* err;
  unsigned int* amax_out;  // nullable: atomicMax of |D| (as stored) over the output, float bits
  GemmQuantOut q;          // used by the quantizing variant only
  // D for the columns past the last whole 16-byte unit of a row (the output
  // tensor map covers n_tma = those whole units; its clipping is per 16-byte
  // unit, so the rest of the row goes through plain stores)
  void* d;
  int64_t ldd;
  int n_tma;
  // Failure-detection test only (0 in every normal launch): extra bytes the
  // leader CTA of each pair expects on its first stage's barrier, which no
  // copy delivers, and the wait limit in ns (0: the default limit).
  unsigned int hold_tx;
  unsigned long long wait_ns;
};

constexpr int kGroupsPerLaunch = 64;

struct GroupedArgs {
  CUtensorMap tmA[kGroupsPerLaunch];
  CUtensorMap tmB[kGroupsPerLaunch];
  CUtensorMap tmD[kGroupsPerLaunch];
  const uint8_t* sfa[kGroupsPerLaunch];
  const uint8_t* sfb[kGroupsPerLaunch];
  const float* ga[kGroupsPerLaunch];
  const float* gb[kGroupsPerLaunch];
  int M[kGroupsPerLaunch], N[kGroupsPerLaunch], K[kGroupsPerLaunch];
  int tile_start[kGroupsPerLaunch + 1];
  int count;
  unsigned int* err;
};

unsigned int* device_error_word();
// A 2D tiled tensor map over a row-major [rows][ld] BF16/FP32 matrix (first
// `cols` columns), box = box_cols x box_rows elements, no swizzle; boxes past
// the edges are zero-filled.  False when the driver entry point is missing
// or the encoding is rejected.
bool make_tile_map_2d(CUtensorMap* m, const void* base, bool bf16, int64_t rows, int64_t cols, int64_t ld,
                      uint32_t box_cols, uint32_t box_rows);
// Read and clear the current device's timeout word in one atomic exchange
// (ordered on `s`), then synchronise `s` and return the value read.
cudaError_t take_device_error(cudaStream_t s, unsigned int* value);
// Failure-detection test support: arm the next launch of the plain GEMM
// (op 1) or of the TMA-fed transposed encoder (op 2) made by this process so
// that one of its pipeline barriers is never completed and the bounded wait
// on it runs out after limit_ns.  take_armed_wait returns the armed limit
// for `op` and disarms it (0 when not armed).
void arm_wait_expiry(int op, unsigned long long limit_ns);
unsigned long long take_armed_wait(int op);
int gemm_tile_m();
int gemm_tile_n();
cudaError_t launch_gemm(const GemmOperand& A, const GemmOperand& B, void* D, int64_t ldd, bool out_bf16, cudaStream_t s,
                        const char** why, float* amax_out = nullptr, const GemmQuantOut* q = nullptr);
cudaError_t launch_gemm_grouped(int count, const GemmOperand* A, const GemmOperand* B, void* const* D, bool out_bf16,
                                cudaStream_t s, const char** why);

}  // namespace nvfp4
