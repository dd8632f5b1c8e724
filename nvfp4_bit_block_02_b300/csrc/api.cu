// C ABI of the NVFP4 library (declared in include/nvfp4.h): argument checks on
// the host, then kernel launches on the caller's stream.  No allocation, no
// synchronisation (except nvfp4_sync_check).
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <string>

#include "gemm.h"
#include "nvfp4.h"
#include "quantize.h"

namespace {

thread_local std::string g_last_error;

nvfp4_status fail(nvfp4_status s, const std::string& msg) {
  g_last_error = msg;
  return s;
}

nvfp4_status cuda_fail(cudaError_t e, const char* what) {
  return fail(NVFP4_ERR_CUDA, std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")");
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

nvfp4_status check_tensor_buffers(const nvfp4_tensor* t, const char* name) {
  if (!t) return fail(NVFP4_ERR_INVALID_ARG, std::string(name) + " is NULL");
  if (t->rows < 0 || t->cols < 0) return fail(NVFP4_ERR_INVALID_ARG, std::string(name) + " has a negative size");
  if (!t->global_scale || !t->amax)
    return fail(NVFP4_ERR_INVALID_ARG, std::string(name) + " has a NULL buffer (global_scale, amax)");
  if ((!t->codes || !t->scales) && t->rows > 0 && t->cols > 0)
    return fail(NVFP4_ERR_INVALID_ARG, std::string(name) + " has a NULL buffer (codes, scales)");
  if (!aligned16(t->codes) || !aligned16(t->scales))
    return fail(NVFP4_ERR_MISALIGNED, std::string(name) + " codes/scales must be 16-byte aligned");
  return NVFP4_OK;
}

// Validation shared by nvfp4_quantize and nvfp4_rht_quantize.
nvfp4_status check_quantize(const void* x, nvfp4_dtype xt, int64_t rows, int64_t cols, int64_t ld,
                            const nvfp4_quant_config* cfg, const nvfp4_tensor* out, bool rht) {
  if (!cfg) return fail(NVFP4_ERR_INVALID_ARG, "cfg is NULL");
  if (xt != NVFP4_F32 && xt != NVFP4_BF16) return fail(NVFP4_ERR_INVALID_ARG, "input dtype must be F32 or BF16");
  if (cfg->block != NVFP4_BLOCK_1D && cfg->block != NVFP4_BLOCK_2D) return fail(NVFP4_ERR_INVALID_ARG, "bad block mode");
  if (cfg->round != NVFP4_ROUND_RNE && cfg->round != NVFP4_ROUND_STOCHASTIC)
    return fail(NVFP4_ERR_INVALID_ARG, "bad rounding mode");
  if (cfg->scaling != NVFP4_SCALE_MAX6 && cfg->scaling != NVFP4_SCALE_FOUR_OVER_SIX)
    return fail(NVFP4_ERR_INVALID_ARG, "bad scaling mode");
  if (cfg->transpose != 0 && cfg->transpose != 1) return fail(NVFP4_ERR_INVALID_ARG, "transpose must be 0 or 1");
  if (rht && cfg->block != NVFP4_BLOCK_1D) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "the RHT path uses 1D blocks");
  if (rows < 0 || cols < 0) return fail(NVFP4_ERR_INVALID_ARG, "negative size");
  if (ld < cols) return fail(NVFP4_ERR_INVALID_ARG, "ld < cols");
  nvfp4_status st = check_tensor_buffers(out, "out");
  if (st != NVFP4_OK) return st;
  const int64_t R = cfg->transpose ? cols : rows, K = cfg->transpose ? rows : cols;
  if (out->rows != R || out->cols != K)
    return fail(NVFP4_ERR_INVALID_ARG, "out->rows/cols must be the output orientation (" + std::to_string(R) + " x " +
                                           std::to_string(K) + ")");
  if (K % 16) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "K (the contraction length) must be a multiple of 16");
  if (cfg->transpose && cols % 16) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "transpose needs cols % 16 == 0");
  if (cfg->block == NVFP4_BLOCK_2D && R % 16) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "2D blocks need rows % 16 == 0");
  if (R == 0 || K == 0) return NVFP4_OK;
  if (!x) return fail(NVFP4_ERR_INVALID_ARG, "x is NULL");
  const int64_t es = xt == NVFP4_BF16 ? 2 : 4;
  if (!aligned16(x) || (ld * es) % 16) return fail(NVFP4_ERR_MISALIGNED, "x must be 16-byte aligned with ld*elsize % 16 == 0");
  // launch geometry: row-wise grid.y = ceil(R/128), transposed grid.y = ceil(K/64)
  if ((!cfg->transpose && cdiv(R, 128) > 65535) || (cfg->transpose && cdiv(K, 64) > 65535) ||
      cdiv(K / 16, 4) > ((int64_t)1 << 31) - 1 || cdiv(R, 128) > ((int64_t)1 << 31) - 1)
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "tensor too large for one launch");
  return NVFP4_OK;
}

nvfp4_status run_quantize(const void* x, nvfp4_dtype xt, int64_t rows, int64_t cols, int64_t ld,
                          const nvfp4_quant_config* cfg, bool rht, uint64_t rht_seed, const float* amax_in,
                          nvfp4_tensor* out, float* tdebug, void* stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool bf16 = xt == NVFP4_BF16;
  const int64_t R = out->rows, K = out->cols;
  if (R == 0 || K == 0) {
    cudaError_t e = nvfp4::launch_empty_scalars(out->amax, out->global_scale, s);
    return e == cudaSuccess ? NVFP4_OK : cuda_fail(e, "empty-tensor scalars");
  }
  if (tdebug && !aligned16(tdebug)) return fail(NVFP4_ERR_MISALIGNED, "transformed_debug must be 16-byte aligned");
  const float* amax = amax_in;
  nvfp4::QuantArgs a{};
  a.x = x;
  a.R_in = rows;
  a.C_in = cols;
  a.ld = ld;
  a.R = R;
  a.K = K;
  a.amax_out = out->amax;
  a.amax_accum = out->amax;
  a.g_out = out->global_scale;
  a.codes = out->codes;
  a.scales = out->scales;
  a.tdebug = tdebug;
  a.seed = cfg->seed;
  a.offset = cfg->offset;
  a.rht_seed = rht_seed;
  a.err = nvfp4::device_error_word();
  if (!a.err) return cuda_fail(cudaGetLastError(), "device error word (cudaGetSymbolAddress)");
  const bool tr = cfg->transpose != 0, b2d = cfg->block == NVFP4_BLOCK_2D,
             sr = cfg->round == NVFP4_ROUND_STOCHASTIC, f46 = cfg->scaling == NVFP4_SCALE_FOUR_OVER_SIX;
  if (!amax) {
    cudaError_t e = cudaMemsetAsync(out->amax, 0, sizeof(float), s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(amax)");
    if (rht) {
      a.amax_in = out->amax;
      e = nvfp4::launch_quantize(a, bf16, tr, false, false, false, true, true, s);
    } else {
      e = nvfp4::launch_amax(x, bf16, rows, cols, ld, out->amax, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "amax launch");
    amax = out->amax;
  }
  a.amax_in = amax;
  cudaError_t e = nvfp4::launch_quantize(a, bf16, tr, b2d, sr, f46, rht, false, s);
  if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
  return NVFP4_OK;
}

nvfp4_status check_gemm_operands(const nvfp4_tensor* A, const nvfp4_tensor* B) {
  nvfp4_status st = check_tensor_buffers(A, "A");
  if (st != NVFP4_OK) return st;
  st = check_tensor_buffers(B, "B");
  if (st != NVFP4_OK) return st;
  if (A->cols != B->cols) return fail(NVFP4_ERR_INVALID_ARG, "A and B must have the same K (cols)");
  if (A->cols % 64) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "K must be a multiple of 64");
  if (A->rows > ((int64_t)1 << 30) || B->rows > ((int64_t)1 << 30) || A->cols > ((int64_t)1 << 30))
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "GEMM dimension too large");
  return NVFP4_OK;
}

nvfp4::GemmOperand operand(const nvfp4_tensor* t) {
  return nvfp4::GemmOperand{t->codes, t->scales, t->global_scale, t->rows, t->cols};
}

}  // namespace

extern "C" {

size_t nvfp4_codes_bytes(int64_t rows, int64_t cols) {
  if (rows <= 0 || cols <= 0) return 0;
  return (size_t)(rows * (cols / 2));
}

size_t nvfp4_scales_bytes(int64_t rows, int64_t cols) {
  if (rows <= 0 || cols <= 0) return 0;
  return (size_t)(cdiv(rows, 128) * 128 * cdiv(cols / 16, 4) * 4);
}

nvfp4_status nvfp4_quantize(const void* x, nvfp4_dtype xt, int64_t rows, int64_t cols, int64_t ld,
                            const nvfp4_quant_config* cfg, const float* amax_in, nvfp4_tensor* out, void* stream) {
  nvfp4_status st = check_quantize(x, xt, rows, cols, ld, cfg, out, false);
  if (st != NVFP4_OK) return st;
  return run_quantize(x, xt, rows, cols, ld, cfg, false, 0, amax_in, out, nullptr, stream);
}

nvfp4_status nvfp4_rht_quantize(const void* x, nvfp4_dtype xt, int64_t rows, int64_t cols, int64_t ld,
                                const nvfp4_quant_config* cfg, uint64_t rht_seed, const float* amax_in,
                                nvfp4_tensor* out, float* transformed_debug, void* stream) {
  nvfp4_status st = check_quantize(x, xt, rows, cols, ld, cfg, out, true);
  if (st != NVFP4_OK) return st;
  return run_quantize(x, xt, rows, cols, ld, cfg, true, rht_seed, amax_in, out, transformed_debug, stream);
}

nvfp4_status nvfp4_amax(const void* x, nvfp4_dtype xt, int64_t rows, int64_t cols, int64_t ld, float* amax,
                        void* stream) {
  if (xt != NVFP4_F32 && xt != NVFP4_BF16) return fail(NVFP4_ERR_INVALID_ARG, "input dtype must be F32 or BF16");
  if (rows < 0 || cols < 0) return fail(NVFP4_ERR_INVALID_ARG, "negative size");
  if (ld < cols) return fail(NVFP4_ERR_INVALID_ARG, "ld < cols");
  if (!amax) return fail(NVFP4_ERR_INVALID_ARG, "amax is NULL");
  const int64_t es = xt == NVFP4_BF16 ? 2 : 4;
  if (rows > 0 && cols > 0) {
    if (!x) return fail(NVFP4_ERR_INVALID_ARG, "x is NULL");
    if (!aligned16(x) || (ld * es) % 16 || (cols * es) % 16)
      return fail(NVFP4_ERR_MISALIGNED, "x must be 16-byte aligned with ld*elsize and cols*elsize % 16 == 0");
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float), s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(amax)");
  if (rows == 0 || cols == 0) return NVFP4_OK;
  e = nvfp4::launch_amax(x, xt == NVFP4_BF16, rows, cols, ld, amax, s);
  return e == cudaSuccess ? NVFP4_OK : cuda_fail(e, "amax launch");
}

nvfp4_status nvfp4_quantize_grouped(int count, const void* const* x, nvfp4_dtype xt, const int64_t* rows,
                                    const int64_t* cols, const int64_t* ld, const nvfp4_quant_config* cfg,
                                    nvfp4_tensor* out, void* stream) {
  if (count < 0 || count > NVFP4_MAX_GROUPS)
    return fail(NVFP4_ERR_INVALID_ARG, "count must be in [0, " + std::to_string(NVFP4_MAX_GROUPS) + "]");
  if (count == 0) return NVFP4_OK;
  if (!x || !rows || !cols || !ld || !out) return fail(NVFP4_ERR_INVALID_ARG, "a host array is NULL");
  for (int e = 0; e < count; ++e) {
    nvfp4_status st = check_quantize(x[e], xt, rows[e], cols[e], ld[e], cfg, &out[e], false);
    if (st != NVFP4_OK) return fail(st, "group " + std::to_string(e) + ": " + g_last_error);
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool bf16 = xt == NVFP4_BF16, tr = cfg->transpose != 0, b2d = cfg->block == NVFP4_BLOCK_2D,
             sr = cfg->round == NVFP4_ROUND_STOCHASTIC, f46 = cfg->scaling == NVFP4_SCALE_FOUR_OVER_SIX;
  nvfp4::GroupQuant gq{};  // kernel parameters of one launch (~9 KB, copied at launch)
  nvfp4::GroupQuant* gp = &gq;
  int n = 0;
  auto flush = [&]() -> nvfp4_status {
    if (n == 0) return NVFP4_OK;
    gp->count = n;
    cudaError_t e = nvfp4::launch_quantize_grouped(*gp, bf16, tr, b2d, sr, f46, true, s);
    n = 0;
    return e == cudaSuccess ? NVFP4_OK : cuda_fail(e, "grouped quantize launch");
  };
  nvfp4_status st = NVFP4_OK;
  for (int e = 0; e < count && st == NVFP4_OK; ++e) {
    nvfp4_tensor* o = &out[e];
    if (o->rows == 0 || o->cols == 0) {
      cudaError_t ce = nvfp4::launch_empty_scalars(o->amax, o->global_scale, s);
      if (ce != cudaSuccess) st = cuda_fail(ce, "empty-tensor scalars");
      continue;
    }
    nvfp4::QuantArgs& a = gp->a[n++];
    a = nvfp4::QuantArgs{};
    a.x = x[e];
    a.R_in = rows[e];
    a.C_in = cols[e];
    a.ld = ld[e];
    a.R = o->rows;
    a.K = o->cols;
    a.amax_in = o->amax;
    a.amax_out = o->amax;
    a.amax_accum = o->amax;
    a.g_out = o->global_scale;
    a.codes = o->codes;
    a.scales = o->scales;
    a.seed = cfg->seed;
    a.offset = cfg->offset + (uint64_t)e;
    a.err = nvfp4::device_error_word();  // bounded waits of the TMA-fed transposed encoder
    if (!a.err) {
      st = cuda_fail(cudaGetLastError(), "device error word (cudaGetSymbolAddress)");
      break;
    }
    if (n == nvfp4::kQuantGroups) st = flush();
  }
  if (st == NVFP4_OK) st = flush();
  return st;
}

nvfp4_status nvfp4_transpose_2d(const nvfp4_tensor* q, nvfp4_tensor* qt, void* stream) {
  nvfp4_status st = check_tensor_buffers(q, "q");
  if (st != NVFP4_OK) return st;
  st = check_tensor_buffers(qt, "qt");
  if (st != NVFP4_OK) return st;
  if (q->rows % 16 || q->cols % 16)
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "a 2D-block tensor has rows and cols that are multiples of 16");
  if (qt->rows != q->cols || qt->cols != q->rows) return fail(NVFP4_ERR_INVALID_ARG, "qt must be cols x rows of q");
  if (q->rows > 0 && q->cols > 0 && (q->codes == qt->codes || q->scales == qt->scales))
    return fail(NVFP4_ERR_INVALID_ARG, "qt must not share codes or scales with q");
  if (q->rows / 64 > 65535) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "rows too large for the launch grid");
  cudaError_t e = nvfp4::launch_transpose_2d(q->codes, q->scales, q->global_scale, q->amax, q->rows, q->cols,
                                             qt->codes, qt->scales, qt->global_scale, qt->amax,
                                             reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NVFP4_OK : cuda_fail(e, "transpose_2d launch");
}

nvfp4_status nvfp4_dequantize(const nvfp4_tensor* q, void* y, nvfp4_dtype yt, void* stream) {
  nvfp4_status st = check_tensor_buffers(q, "q");
  if (st != NVFP4_OK) return st;
  if (yt != NVFP4_F32 && yt != NVFP4_BF16) return fail(NVFP4_ERR_INVALID_ARG, "output dtype must be F32 or BF16");
  if (q->cols % 16) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "cols must be a multiple of 16");
  if (q->rows == 0 || q->cols == 0) return NVFP4_OK;
  if (!y) return fail(NVFP4_ERR_INVALID_ARG, "y is NULL");
  if (!aligned16(y)) return fail(NVFP4_ERR_MISALIGNED, "y must be 16-byte aligned");
  cudaError_t e = nvfp4::launch_dequantize(q->codes, q->scales, q->global_scale, q->rows, q->cols, y, yt == NVFP4_BF16,
                                           reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NVFP4_OK : cuda_fail(e, "dequantize launch");
}

nvfp4_status nvfp4_w4a16_gemm(const void* x, nvfp4_dtype xt, int64_t M, int64_t ldx, const nvfp4_tensor* W, void* y,
                              nvfp4_dtype yt, int64_t ldy, void* stream) {
  nvfp4_status st = check_tensor_buffers(W, "W");
  if (st != NVFP4_OK) return st;
  if (xt != NVFP4_BF16) return fail(NVFP4_ERR_INVALID_ARG, "x must be BF16");
  if (yt != NVFP4_F32 && yt != NVFP4_BF16) return fail(NVFP4_ERR_INVALID_ARG, "output dtype must be F32 or BF16");
  if (M < 0) return fail(NVFP4_ERR_INVALID_ARG, "negative M");
  const int64_t N = W->rows, K = W->cols;
  if (K % 16) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "K (W->cols) must be a multiple of 16");
  if (ldx < K) return fail(NVFP4_ERR_INVALID_ARG, "ldx < K");
  if (ldy < N) return fail(NVFP4_ERR_INVALID_ARG, "ldy < N");
  if (M == 0 || N == 0) return NVFP4_OK;
  if (!y) return fail(NVFP4_ERR_INVALID_ARG, "y is NULL");
  if (reinterpret_cast<uintptr_t>(y) % (yt == NVFP4_BF16 ? 2 : 4))
    return fail(NVFP4_ERR_MISALIGNED, "y must be aligned to its element");
  if (K > 0) {
    if (!x) return fail(NVFP4_ERR_INVALID_ARG, "x is NULL");
    if (!aligned16(x) || ldx % 8) return fail(NVFP4_ERR_MISALIGNED, "x must be 16-byte aligned with ldx % 8 == 0");
  }
  // the kernel's in-row offsets are 32-bit: scale bytes at (K/64) * 512 stay below 2^32 for K <= 2^28
  if (K > ((int64_t)1 << 28) || cdiv(N, 16) > ((int64_t)1 << 31) - 1)
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "tensor too large for one launch (K <= 2^28, N/16 < 2^31)");
  cudaError_t e = nvfp4::launch_w4a16(x, M, ldx, W->codes, W->scales, W->global_scale, N, K, y, yt == NVFP4_BF16, ldy,
                                      reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NVFP4_OK : cuda_fail(e, "w4a16 launch");
}

namespace {
nvfp4_status run_gemm(const nvfp4_tensor* A, const nvfp4_tensor* B, void* D, nvfp4_dtype dt, int64_t ldd,
                      float* amax_out, void* stream) {
  nvfp4_status st = check_gemm_operands(A, B);
  if (st != NVFP4_OK) return st;
  if (dt != NVFP4_F32 && dt != NVFP4_BF16) return fail(NVFP4_ERR_INVALID_ARG, "output dtype must be F32 or BF16");
  if (A->rows == 0 || B->rows == 0) return NVFP4_OK;
  if (!D) return fail(NVFP4_ERR_INVALID_ARG, "D is NULL");
  if (ldd < B->rows) return fail(NVFP4_ERR_INVALID_ARG, "ldd < N");
  const int64_t es = dt == NVFP4_BF16 ? 2 : 4;
  if (!aligned16(D) || (ldd * es) % 16) return fail(NVFP4_ERR_MISALIGNED, "D must be 16-byte aligned, ldd*elsize % 16 == 0");
  if (A->cols == 0) {  // an empty sum over k: D = 0 (and its amax 0, already zeroed by the caller)
    cudaError_t e = cudaMemset2DAsync(D, (size_t)(ldd * es), 0, (size_t)(B->rows * es), (size_t)A->rows,
                                      reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? NVFP4_OK : cuda_fail(e, "cudaMemset2DAsync(D)");
  }
  const char* why = "";
  cudaError_t e = nvfp4::launch_gemm(operand(A), operand(B), D, ldd, dt == NVFP4_BF16,
                                     reinterpret_cast<cudaStream_t>(stream), &why, amax_out);
  if (e != cudaSuccess) return cuda_fail(e, (std::string("gemm launch: ") + why).c_str());
  return NVFP4_OK;
}
}  // namespace

nvfp4_status nvfp4_gemm(const nvfp4_tensor* A, const nvfp4_tensor* B, void* D, nvfp4_dtype dt, int64_t ldd,
                        void* stream) {
  return run_gemm(A, B, D, dt, ldd, nullptr, stream);
}

nvfp4_status nvfp4_gemm_amax(const nvfp4_tensor* A, const nvfp4_tensor* B, void* D, nvfp4_dtype dt, int64_t ldd,
                             float* amax_out, void* stream) {
  if (!amax_out) return fail(NVFP4_ERR_INVALID_ARG, "amax_out is NULL");
  if (!A || !B) return fail(NVFP4_ERR_INVALID_ARG, "A or B is NULL");
  // arguments first (nothing launched on error), then zero the accumulator
  nvfp4_status st = check_gemm_operands(A, B);
  if (st != NVFP4_OK) return st;
  cudaError_t e = cudaMemsetAsync(amax_out, 0, sizeof(float), reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(amax_out)");
  return run_gemm(A, B, D, dt, ldd, amax_out, stream);
}

nvfp4_status nvfp4_gemm_quantize(const nvfp4_tensor* A, const nvfp4_tensor* B, const float* amax_in, void* D,
                                 int64_t ldd, float* amax_out, nvfp4_tensor* out, void* stream) {
  nvfp4_status st = check_gemm_operands(A, B);
  if (st != NVFP4_OK) return st;
  if (!amax_in) return fail(NVFP4_ERR_INVALID_ARG, "amax_in is NULL");
  st = check_tensor_buffers(out, "out");
  if (st != NVFP4_OK) return st;
  const int64_t M = A->rows, N = B->rows;
  if (out->rows != M || out->cols != N)
    return fail(NVFP4_ERR_INVALID_ARG, "out must be M x N (" + std::to_string(M) + " x " + std::to_string(N) + ")");
  if (N % 16) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "N (the encoded tensor's K) must be a multiple of 16");
  if (A->cols == 0) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "K must be positive");
  if (amax_out && (amax_out == amax_in || amax_out == out->amax))
    return fail(NVFP4_ERR_INVALID_ARG, "amax_out must not alias amax_in or out->amax");
  if (D) {
    if (ldd < N) return fail(NVFP4_ERR_INVALID_ARG, "ldd < N");
    if (!aligned16(D) || (ldd * 2) % 16) return fail(NVFP4_ERR_MISALIGNED, "D must be 16-byte aligned, ldd % 8 == 0");
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (amax_out) {
    cudaError_t e = cudaMemsetAsync(amax_out, 0, sizeof(float), s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(amax_out)");
  }
  if (M == 0 || N == 0) {
    cudaError_t e = nvfp4::launch_empty_scalars(out->amax, out->global_scale, s);
    return e == cudaSuccess ? NVFP4_OK : cuda_fail(e, "empty-tensor scalars");
  }
  nvfp4::GemmQuantOut q{out->codes, out->scales, out->global_scale, out->amax, amax_in, D ? 1 : 0};
  const char* why = "";
  cudaError_t e = nvfp4::launch_gemm(operand(A), operand(B), D, D ? ldd : N, true, s, &why, amax_out, &q);
  if (e != cudaSuccess) return cuda_fail(e, (std::string("gemm launch: ") + why).c_str());
  return NVFP4_OK;
}

nvfp4_status nvfp4_gemm_grouped(int count, const nvfp4_tensor* A, const nvfp4_tensor* B, void* const* D,
                                nvfp4_dtype dt, void* stream) {
  if (count < 0 || count > NVFP4_MAX_GROUPS) return fail(NVFP4_ERR_INVALID_ARG, "count out of range");
  if (count == 0) return NVFP4_OK;
  if (!A || !B || !D) return fail(NVFP4_ERR_INVALID_ARG, "A, B and D must not be NULL");
  if (dt != NVFP4_F32 && dt != NVFP4_BF16) return fail(NVFP4_ERR_INVALID_ARG, "output dtype must be F32 or BF16");
  const int64_t es = dt == NVFP4_BF16 ? 2 : 4;
  nvfp4::GemmOperand ga[NVFP4_MAX_GROUPS], gb[NVFP4_MAX_GROUPS];
  for (int e = 0; e < count; ++e) {
    nvfp4_status st = check_gemm_operands(&A[e], &B[e]);
    if (st != NVFP4_OK) return fail(st, "group " + std::to_string(e) + ": " + g_last_error);
    if (A[e].rows && B[e].rows && !D[e]) return fail(NVFP4_ERR_INVALID_ARG, "group " + std::to_string(e) + ": D is NULL");
    if (A[e].rows && B[e].rows && (!aligned16(D[e]) || (B[e].rows * es) % 16))
      return fail(NVFP4_ERR_MISALIGNED, "group " + std::to_string(e) + ": D must be 16-byte aligned with N*elsize % 16 == 0");
    if (A[e].cols == 0 && A[e].rows && B[e].rows)
      return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "group " + std::to_string(e) + ": K must be positive");
    ga[e] = operand(&A[e]);
    gb[e] = operand(&B[e]);
  }
  const char* why = "";
  cudaError_t e = nvfp4::launch_gemm_grouped(count, ga, gb, D, dt == NVFP4_BF16, reinterpret_cast<cudaStream_t>(stream), &why);
  if (e != cudaSuccess) return cuda_fail(e, (std::string("grouped gemm launch: ") + why).c_str());
  return NVFP4_OK;
}

nvfp4_status nvfp4_sync_check(void* stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "pending CUDA error");
  unsigned int v = 0;
  e = nvfp4::take_device_error(reinterpret_cast<cudaStream_t>(stream), &v);
  if (e != cudaSuccess) return cuda_fail(e, "read device error word");
  if (v) return fail(NVFP4_ERR_TIMEOUT, (v & 1u) ? "a GEMM pipeline wait exceeded its limit"
                                                  : "a transposed-encoder pipeline wait exceeded its limit");
  return NVFP4_OK;
}

nvfp4_status nvfp4_test_expire_next_wait(int op, uint64_t limit_ns) {
  if (op != 1 && op != 2) return fail(NVFP4_ERR_INVALID_ARG, "op must be 1 (GEMM) or 2 (transposed encoder)");
  if (limit_ns != 0 && (limit_ns < 1000000ull || limit_ns > 2000000000ull))
    return fail(NVFP4_ERR_INVALID_ARG, "limit_ns must be 0 or in [1e6, 2e9]");
  nvfp4::arm_wait_expiry(op, limit_ns);
  return NVFP4_OK;
}

const char* nvfp4_status_string(nvfp4_status s) {
  switch (s) {
    case NVFP4_OK: return "NVFP4_OK";
    case NVFP4_ERR_INVALID_ARG: return "NVFP4_ERR_INVALID_ARG";
    case NVFP4_ERR_UNSUPPORTED_SHAPE: return "NVFP4_ERR_UNSUPPORTED_SHAPE";
    case NVFP4_ERR_MISALIGNED: return "NVFP4_ERR_MISALIGNED";
    case NVFP4_ERR_CUDA: return "NVFP4_ERR_CUDA";
    case NVFP4_ERR_TIMEOUT: return "NVFP4_ERR_TIMEOUT";
  }
  return "NVFP4_ERR_UNKNOWN";
}

const char* nvfp4_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
