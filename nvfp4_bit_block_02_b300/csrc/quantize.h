// Internal launch interface of the quantizer kernels (not part of the C ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace nvfp4 {

struct QuantArgs {
  const void* x;        // input, row-major [R_in][ld]
  int64_t R_in, C_in;   // input rows / cols
  int64_t ld;           // input leading dimension (elements)
  int64_t R, K;         // output orientation
  const float* amax_in; // tensor amax the encoder uses
  float* amax_out;      // copy of it (may alias amax_in)
  float* amax_accum;    // atomicMax target of the amax-only passes
  float* g_out;
  uint8_t* codes;
  uint8_t* scales;
  float* tdebug;        // fp32 [R][K] transformed values, or nullptr
  uint64_t seed, offset, rht_seed;
  unsigned int* err;    // device timeout word (bounded waits of the TMA-fed encoder)
};

// Up to kQuantGroups tensors quantized by one amax launch and one encode
// launch (the MoE experts): per group its own args and tensor amax, and (the
// transposed encoder) its input tensor map.
constexpr int kQuantGroups = 64;
struct GroupQuant {
  CUtensorMap tm[kQuantGroups];  // transposed encoder: 64 x 128-element input tiles of each group's x
  QuantArgs a[kQuantGroups];
  uint32_t tiles_x[kQuantGroups];         // encoder tile-grid width per group
  uint32_t tile_start[kQuantGroups + 1];  // encoder tiles, prefix sums
  uint32_t amax_rows[kQuantGroups];       // amax pass: input rows per tile
  uint32_t amax_start[kQuantGroups + 1];  // amax tiles, prefix sums
  int count;
  int use_tma;  // transposed encoder: every group's map was built (else register staging)
};

// Fills the tile tables of g (count and a[] set by the caller), then
// launches: zero the amax accumulators and reduce every group's amax (when
// compute_amax), and the encoder over all groups' tiles.
cudaError_t launch_quantize_grouped(GroupQuant& g, bool bf16, bool transpose, bool b2d, bool sr, bool f46,
                                    bool compute_amax, cudaStream_t s);

cudaError_t launch_amax(const void* x, bool bf16, int64_t rows, int64_t cols, int64_t ld, float* amax_accum,
                        cudaStream_t s);
cudaError_t launch_quantize(const QuantArgs& a, bool bf16, bool transpose, bool b2d, bool sr, bool f46, bool rht,
                            bool amax_only, cudaStream_t s);
cudaError_t launch_empty_scalars(float* amax, float* g, cudaStream_t s);
cudaError_t launch_dequantize(const uint8_t* codes, const uint8_t* scales, const float* g, int64_t R, int64_t K,
                              void* y, bool bf16_out, cudaStream_t s);
cudaError_t launch_w4a16(const void* x, int64_t M, int64_t ldx, const uint8_t* codes, const uint8_t* scales,
                         const float* g, int64_t N, int64_t K, void* y, bool out_bf16, int64_t ldy, cudaStream_t s);
cudaError_t launch_transpose_2d(const uint8_t* codes, const uint8_t* scales, const float* g, const float* amax,
                                int64_t R, int64_t K, uint8_t* codes_t, uint8_t* scales_t, float* g_t, float* amax_t,
                                cudaStream_t s);

}  // namespace nvfp4
