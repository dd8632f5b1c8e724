// Transpose of a 2D-block-quantized tensor: the Dgrad operand W^T from the
// weight's own NVFP4 codes ("NVIDIA Introduces a 4-Bit Pretraining
// Methodology Using NVFP4", "Method": 16x16 weight blocks keep the forward
// and backward quantization of W consistent).  A 16x16 block has one scale
// and its elements keep their codes under transposition, so W^T's NVFP4
// tensor is a pure data movement of W's: codes nibble-transposed, scales
// re-laid out.  No value is re-encoded.
#include "nvfp4_device.cuh"
#include "quantize.h"

namespace nvfp4 {

// Codes: in [R][K/2] (element 2j of a row in the low nibble of byte j) ->
// out [K][R/2].  A CTA moves a 64-row x 128-column tile: 64 x 64 input bytes
// staged in shared memory (8-byte loads; K % 16 == 0 keeps every 8-byte
// chunk whole), then thread t assembles output row t/2, bytes 16(t%2)..+15,
// from input rows 2j and 2j+1 (8-byte stores; R % 16 == 0).
__global__ void __launch_bounds__(256) k_transpose_codes(const uint8_t* __restrict__ in, int64_t R, int64_t K,
                                                         uint8_t* __restrict__ out) {
  constexpr int PITCH = 68;  // 64 bytes + 4: the column reads below hit distinct banks
  __shared__ __align__(16) uint8_t tile[64 * PITCH];
  const int t = threadIdx.x;
  const int64_t r0 = (int64_t)blockIdx.y * 64, k0 = (int64_t)blockIdx.x * 128;
  const int64_t in_row_bytes = K / 2, out_row_bytes = R / 2;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int idx = t + 256 * i, row = idx >> 3, chunk = idx & 7;
    const int64_t r = r0 + row, b = k0 / 2 + 8 * chunk;
    uint2 v = make_uint2(0, 0);
    if (r < R && b < in_row_bytes) v = *reinterpret_cast<const uint2*>(in + r * in_row_bytes + b);
    *reinterpret_cast<uint32_t*>(tile + row * PITCH + 8 * chunk) = v.x;
    *reinterpret_cast<uint32_t*>(tile + row * PITCH + 8 * chunk + 4) = v.y;
  }
  __syncthreads();
  const int kl = t >> 1, jb = 16 * (t & 1);       // output row (local), first output byte (local)
  const int col = kl >> 1, shift = 4 * (kl & 1);  // input byte column and nibble of element kl
  uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const uint32_t lo = (tile[(2 * (jb + j)) * PITCH + col] >> shift) & 15u;
    const uint32_t hi = (tile[(2 * (jb + j) + 1) * PITCH + col] >> shift) & 15u;
    w[j >> 2] |= (lo | (hi << 4)) << (8 * (j & 3));
  }
  const int64_t k = k0 + kl, b = r0 / 2 + jb;
  if (k < K) {
    uint8_t* dst = out + k * out_row_bytes + b;
    if (b < out_row_bytes) *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
    if (b + 8 < out_row_bytes) *reinterpret_cast<uint2*>(dst + 8) = make_uint2(w[2], w[3]);
  }
}

// Scales: every byte of the output's physical scale buffer (K rows x R/16
// blocks, 128x4 atoms), padding written as 0.  Logical entry (k, rb) of the
// output is the scale of input tile (rb, k/16), read at input row 16*rb.
// Thread 0 also copies the per-tensor scalars.
__global__ void __launch_bounds__(256) k_transpose_scales(const uint8_t* __restrict__ in, int64_t R, int64_t K,
                                                          uint8_t* __restrict__ out, int64_t out_bytes,
                                                          const float* __restrict__ g_in, const float* __restrict__ amax_in,
                                                          float* __restrict__ g_out, float* __restrict__ amax_out) {
  const int64_t KB_in = K / 16, RB = R / 16;
  const int64_t nka_in = (KB_in + 3) / 4, nka_out = (RB + 3) / 4;
  const int64_t o = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (o == 0) {
    *g_out = *g_in;
    *amax_out = *amax_in;
  }
  if (o >= out_bytes) return;
  const int64_t atom = o >> 9, w = o & 511;
  const int64_t k = (atom / nka_out) * 128 + ((w & 15) >> 2) * 32 + (w >> 4);
  const int64_t rb = (atom % nka_out) * 4 + (w & 3);
  out[o] = (k < K && rb < RB) ? in[sf_offset(16 * rb, k / 16, nka_in)] : (uint8_t)0;
}

cudaError_t launch_transpose_2d(const uint8_t* codes, const uint8_t* scales, const float* g, const float* amax,
                                int64_t R, int64_t K, uint8_t* codes_t, uint8_t* scales_t, float* g_t, float* amax_t,
                                cudaStream_t s) {
  if (R > 0 && K > 0) {
    dim3 grid((unsigned)((K + 127) / 128), (unsigned)((R + 63) / 64));
    k_transpose_codes<<<grid, 256, 0, s>>>(codes, R, K, codes_t);
  }
  // output: K rows (padded to 128) x R/16 blocks (padded to 4)
  const int64_t out_bytes = (R > 0 && K > 0) ? ((K + 127) / 128) * 128 * ((R / 16 + 3) / 4) * 4 : 0;
  const int64_t blocks = out_bytes > 0 ? (out_bytes + 255) / 256 : 1;
  k_transpose_scales<<<(unsigned)blocks, 256, 0, s>>>(scales, R, K, scales_t, out_bytes, g, amax, g_t, amax_t);
  return cudaGetLastError();
}

}  // namespace nvfp4
