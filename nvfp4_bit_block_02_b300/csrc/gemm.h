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

struct GemmArgs {
  const uint8_t* sfa;
  const uint8_t* sfb;
  const float* ga;
  const float* gb;
  int M, N, K;
  int out_bf16;
  unsigned int* err;
  unsigned int* amax_out;  // nullable: atomicMax of |D| (as stored) over the output, float bits
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
  int out_bf16;
  unsigned int* err;
};

unsigned int* device_error_word();
// Read and clear the current device's timeout word in one atomic exchange
// (ordered on `s`), then synchronise `s` and return the value read.
cudaError_t take_device_error(cudaStream_t s, unsigned int* value);
int gemm_tile_m();
int gemm_tile_n();
cudaError_t launch_gemm(const GemmOperand& A, const GemmOperand& B, void* D, int64_t ldd, bool out_bf16, cudaStream_t s,
                        const char** why, float* amax_out = nullptr);
cudaError_t launch_gemm_grouped(int count, const GemmOperand* A, const GemmOperand* B, void* const* D, bool out_bf16,
                                cudaStream_t s, const char** why);

}  // namespace nvfp4
