/*
 * nvfp4.h - C ABI of the B300 (sm_103a) NVFP4 quantizer, block-scaled GEMM
 * and weight-only (W4A16) GEMM.
 *
 * The format ("NVIDIA Introduces a 4-Bit Pretraining Methodology Using NVFP4",
 * section "Summary"): 16-element blocks of 4-bit E2M1 codes, one E4M3 scale per
 * block and one FP32 scale per tensor.  The recipe components ("Method" on the
 * same page; the hyper.ai story "NVIDIA présente NVFP4"): 2D 16x16 weight
 * blocks, a 16x16 Random Hadamard Transform on Wgrad inputs, stochastic
 * rounding on gradients.  Four-over-Six per-block scaling: the hyper.ai story
 * on the Nemotron 3 Ultra NVFP4 checkpoint.
 *
 * Arithmetic of the encoder (fl = one IEEE fp32 op, round to nearest even):
 *   amax = max |x| over the tensor (after the RHT when it is on)
 *   g    = fl(amax / 2688)   (2688 = 6 * 448; g = 1 when amax = 0)
 *   per block:  amax_b = max |x| over the block
 *               s_b = E4M3_rne_satfinite(fl(amax_b / fl(m * g))), m = 6
 *                     (Four-over-Six: also m = 4, keep the candidate whose
 *                      block squared error is strictly lower)
 *               S_b = fl(s_b * g);  r_b = S_b == 0 ? 0 : fl(1 / S_b)
 *   per element: code = E2M1(fl(x * r_b)), round to nearest even or stochastic,
 *               saturating at +-6, sign bit copied from the product
 *   decode:     y = fl(fl(value(code) * s_b) * g)
 *
 * Memory conventions (all functions):
 *  - Every pointer named "device" is CUDA device memory owned by the caller.
 *    The library never allocates device memory and never synchronises, except
 *    nvfp4_sync_check.  `stream` is a cudaStream_t (NULL = legacy default).
 *  - Arguments are validated on the host before any launch; a non-OK status
 *    means nothing was launched.  Asynchronous faults surface at the next CUDA
 *    call or in nvfp4_sync_check.
 *  - Supported range: finite inputs whose tensor amax is 0 or at least 2^-90
 *    (below that the block reciprocal may overflow).
 */
#ifndef NVFP4_H_
#define NVFP4_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  NVFP4_OK = 0,
  NVFP4_ERR_INVALID_ARG = 1,       /* null pointer, bad enum, negative size */
  NVFP4_ERR_UNSUPPORTED_SHAPE = 2, /* shape rule broken (see each function) */
  NVFP4_ERR_MISALIGNED = 3,        /* pointer or leading dimension not 16-byte aligned */
  NVFP4_ERR_CUDA = 4,              /* a CUDA runtime/driver call failed */
  NVFP4_ERR_TIMEOUT = 5            /* a pipeline wait (GEMM, transposed encoder) ran out; nvfp4_sync_check */
} nvfp4_status;

typedef enum { NVFP4_F32 = 0, NVFP4_BF16 = 1 } nvfp4_dtype;
typedef enum { NVFP4_BLOCK_1D = 0 /* 1 x 16 along K */, NVFP4_BLOCK_2D = 1 /* 16 x 16 */ } nvfp4_block;
typedef enum { NVFP4_ROUND_RNE = 0, NVFP4_ROUND_STOCHASTIC = 1 } nvfp4_round;
typedef enum { NVFP4_SCALE_MAX6 = 0, NVFP4_SCALE_FOUR_OVER_SIX = 1 } nvfp4_scaling;

/* A quantized tensor in its K-major orientation: `rows` x `cols`, K = cols.
 *   codes  device uint8 [rows][cols/2]; element 2j in the low nibble of byte j,
 *          2j+1 in the high nibble.  E2M1 code: bit 3 sign, bits 0-2 index
 *          into {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
 *   scales device uint8, nvfp4_scales_bytes(rows, cols) bytes: the E4M3 block
 *          scales in the tensor-core scale tile layout.  The logical matrix
 *          [rows][cols/16] is cut into 128-row x 4-column atoms of 512 bytes;
 *          atom (r/128, kb/4) starts at ((r/128) * ceil(cols/64) + kb/4) * 512
 *          and holds entry (r, kb) at (r%32)*16 + ((r%128)/32)*4 + kb%4.
 *          Padding entries are written as 0 by the quantizer.
 *   global_scale device float[1]: g.
 *   amax   device float[1]: the tensor amax the encoder used.
 * codes and scales may be NULL when rows or cols is 0. */
typedef struct {
  uint8_t* codes;
  uint8_t* scales;
  float* global_scale;
  float* amax;
  int64_t rows;
  int64_t cols;
} nvfp4_tensor;

/* Options of one quantize call.
 *   block      1D (activations, gradients) or 2D 16x16 (weights; W and W^T get
 *              the same codes, so a 2D-quantized weight serves both GEMMs).
 *   round      RNE, or stochastic from a Philox4x32-10 stream (gradients).
 *   scaling    max-6 or Four-over-Six.
 *   transpose  0: quantize x (K = cols of x); 1: quantize x^T (K = rows of x,
 *              the output has cols(x) rows) - the layout Wgrad operands need.
 *   seed, offset  the stochastic-rounding stream: element (r, k) of the output
 *              orientation, i = r*K + k, draws 16 bits: half (i & 1) (high for
 *              odd i) of word (i%8)/2 of Philox4x32-10(key = seed,
 *              counter = (i/8 low, i/8 high, offset low, offset high)); the
 *              element rounds up iff u16 < fl(frac * 65536). */
typedef struct {
  nvfp4_block block;
  nvfp4_round round;
  nvfp4_scaling scaling;
  int transpose;
  uint64_t seed;
  uint64_t offset;
} nvfp4_quant_config;

/* Largest `count` of the grouped calls. */
#define NVFP4_MAX_GROUPS 128

/* Byte sizes of the buffers of a rows x cols (K = cols) quantized tensor. */
size_t nvfp4_codes_bytes(int64_t rows, int64_t cols);
size_t nvfp4_scales_bytes(int64_t rows, int64_t cols); /* ceil(rows/128)*128 * ceil(cols/64)*4 */

/*
 * nvfp4_quantize - BF16/FP32 tensor -> NVFP4 (codes, block scales, g, amax).
 *   x        device, row-major [rows][ld] of dtype xt (only the first `cols`
 *            columns are read).  16-byte aligned; ld * sizeof(xt) % 16 == 0.
 *   cfg      host pointer, read during the call only.
 *   amax_in  device float[1] or NULL.  NULL: the library first reduces max|x|
 *            (one extra read of x).  Given: used as the tensor amax and copied
 *            to out->amax.
 *   out      host struct with device buffers sized for the OUTPUT orientation:
 *            out->rows = transpose ? cols : rows, out->cols = transpose ? rows : cols.
 * Shape rules: K (= out->cols) % 16 == 0; transpose = 1 needs cols % 16 == 0;
 * 2D blocks need out->rows % 16 == 0.  Empty tensors (rows or cols 0) return OK.
 */
nvfp4_status nvfp4_quantize(const void* x, nvfp4_dtype xt, int64_t rows, int64_t cols, int64_t ld,
                            const nvfp4_quant_config* cfg, const float* amax_in, nvfp4_tensor* out,
                            void* stream);

/*
 * nvfp4_amax - the tensor amax alone (step one of the encoder): max |x| over
 * the first `cols` columns of every row, written to the device float `amax`.
 * For a tensor sharded across processes the caller all-reduces (MAX) the
 * shards' amax and passes the result as amax_in to nvfp4_quantize, so every
 * shard encodes with the global g and the shards' codes and scales equal
 * the rows of the unsharded tensor's.  Empty tensors give 0.  x as in
 * nvfp4_quantize (16-byte aligned, ld*elsize % 16 == 0); cols*elsize % 16 == 0.
 */
nvfp4_status nvfp4_amax(const void* x, nvfp4_dtype xt, int64_t rows, int64_t cols, int64_t ld, float* amax,
                        void* stream);

/*
 * nvfp4_quantize_grouped - `count` tensors quantized with one configuration
 * in one amax launch and one encode launch (per 64 tensors): the per-expert
 * tensors of a Mixture-of-Experts layer, each its own tensor with its own
 * amax and g (the MoE workload of the recipe; Four-over-Six on expert
 * weights per the hyper.ai story on the Nemotron 3 Ultra NVFP4 checkpoint).
 *   x, rows, cols, ld, out: host arrays of `count` entries with the meaning
 *   they have in nvfp4_quantize; the tensor amax is always computed
 *   (amax_in = NULL).  Group e draws its stochastic-rounding bits with
 *   offset cfg->offset + e, so experts never share draws.  The result of
 *   group e equals nvfp4_quantize(x[e], ..., cfg with offset + e, NULL,
 *   &out[e]) bit for bit.  count <= NVFP4_MAX_GROUPS; every group follows
 *   the nvfp4_quantize shape rules; no RHT (use nvfp4_rht_quantize).
 */
nvfp4_status nvfp4_quantize_grouped(int count, const void* const* x, nvfp4_dtype xt, const int64_t* rows,
                                    const int64_t* cols, const int64_t* ld, const nvfp4_quant_config* cfg,
                                    nvfp4_tensor* out, void* stream);

/*
 * nvfp4_rht_quantize - the Wgrad operand path: 16x16 Random Hadamard Transform
 * along the contraction dimension, then quantization (1D blocks).
 *   Every 16-chunk of K of the output orientation is replaced by
 *   y = 1/4 * H16 * diag(sigma) * x, H16 the Sylvester Hadamard matrix
 *   (H[i][j] = (-1)^popcount(i&j)), sigma_i = -1 iff bit i of word 0 of
 *   Philox4x32-10(key = rht_seed, counter = (0, 0x80000000, 0, 0)).  One sign
 *   vector per seed: pass the same rht_seed for dY and X so that the transform
 *   cancels in dY^T X.  The amax and the scales are those of the transformed
 *   values.  cfg->block must be 1D; cfg->transpose selects K as for
 *   nvfp4_quantize (Wgrad operands use transpose = 1, K = tokens).
 *   transformed_debug  device fp32 [out->rows][out->cols] or NULL: receives
 *            the transformed values that were encoded (for tests).
 */
nvfp4_status nvfp4_rht_quantize(const void* x, nvfp4_dtype xt, int64_t rows, int64_t cols, int64_t ld,
                                const nvfp4_quant_config* cfg, uint64_t rht_seed, const float* amax_in,
                                nvfp4_tensor* out, float* transformed_debug, void* stream);

/*
 * nvfp4_dequantize - y = fl(fl(value(code) * s_b) * g), BF16 output rounded
 * from that fp32 value (nearest even).
 *   q  host struct with device buffers (codes, scales, global_scale read).
 *   y  device, row-major [q->rows][q->cols] of dtype yt, 16-byte aligned
 *      (32-byte aligned, each block's output leaves in one 256-bit store).
 */
nvfp4_status nvfp4_dequantize(const nvfp4_tensor* q, void* y, nvfp4_dtype yt, void* stream);

/*
 * nvfp4_w4a16_gemm - weight-only NVFP4 GEMM (W4A16) for BF16 activations:
 *   y[m][n] = sum_k x[m][k] * W_hat[n][k],  W_hat = BF16(fl(fl(value * s_b) * g)),
 * the weights dequantized exactly as nvfp4_dequantize with BF16 output, the
 * products and sums in FP32.  The serving variant for GPUs without FP4
 * tensor cores (the hyper.ai story on the Nemotron 3 Ultra NVFP4 checkpoint:
 * Blackwell computes W4A4, Hopper serving switches to W4A16; "BF16 vs NVFP4
 * with Nemotron 3.5 Lightning", "Key takeaways").  On this GPU it serves
 * decode-sized M, where it streams the 4.5-bit weights once.
 *   x    device BF16, row-major [M][ldx], ldx >= W->cols, 16-byte aligned,
 *        ldx % 8 == 0.  Only NVFP4_BF16 is accepted for xt.
 *   W    host struct with device buffers: N = W->rows output features,
 *        K = W->cols (% 16 == 0); codes, scales, global_scale read (1D or 2D
 *        blocks: the scale layout holds a byte per row and block either way).
 *   y    device, row-major [M][ldy] of dtype yt (F32 or BF16, rounded to
 *        nearest even), ldy >= N, aligned to its element.  Every element of
 *        the M x N result is written; the columns beyond N are not touched.
 *   M = 0 or N = 0 launches nothing.  K = 0 writes zeros.
 * Errors: NVFP4_ERR_INVALID_ARG (NULL buffer, bad dtype, ld too small),
 * NVFP4_ERR_UNSUPPORTED_SHAPE (K % 16, K > 2^28, ceil(N/16) >= 2^31),
 * NVFP4_ERR_MISALIGNED; nothing is launched on an argument error.
 */
nvfp4_status nvfp4_w4a16_gemm(const void* x, nvfp4_dtype xt, int64_t M, int64_t ldx, const nvfp4_tensor* W, void* y,
                              nvfp4_dtype yt, int64_t ldy, void* stream);

/*
 * nvfp4_transpose_2d - the NVFP4 tensor of x^T from that of x, for a tensor
 * quantized with 2D 16x16 blocks (the Dgrad operand W^T from the weight's
 * forward quantization; "NVIDIA Introduces a 4-Bit Pretraining Methodology
 * Using NVFP4", "Method": 16x16 weight blocks keep the forward and backward
 * quantization of W consistent).  A 16x16 block has one scale and its
 * elements keep their codes under transposition, so the result is a pure
 * repack: codes nibble-transposed, block scales re-laid out (padding 0),
 * global_scale and amax copied.  With RNE rounding it equals, bit for bit,
 * nvfp4_quantize of x^T with 2D blocks and the same scaling and amax; with
 * stochastic rounding it keeps the codes drawn for x (the draws depend on
 * the output orientation, so quantizing x^T would draw others): the same
 * quantized weight serves both passes.
 *   q   host struct with device buffers: rows x cols, quantized with
 *       NVFP4_BLOCK_2D (not checked: a 1D-block tensor gives the scales of
 *       every 16th row).  rows % 16 == 0, cols % 16 == 0.
 *   qt  host struct with device buffers sized for cols x rows; written.
 *       Must not share codes or scales with q.
 */
nvfp4_status nvfp4_transpose_2d(const nvfp4_tensor* q, nvfp4_tensor* qt, void* stream);

/*
 * nvfp4_gemm - D = g_A * g_B * sum_k (a_mk * s^A_{m,k/16}) * (b_nk * s^B_{n,k/16})
 * on the tensor cores (block-scaled FP4 x FP4, FP32 accumulation), W4A4 as the
 * Nemotron 3 Ultra story says Blackwell runs natively.
 *   A  M x K NVFP4 (A->rows = M, A->cols = K), B  N x K NVFP4: both K-major.
 *   D  device row-major [M][ldd] of dtype dt (FP32 or BF16 rounded to nearest
 *      even from the fp32 result); ldd >= N, ldd * sizeof(dt) % 16 == 0, D
 *      16-byte aligned.  Exactly the M x N outputs are written.
 * Shape rules: any M and N (up to 2^30), K % 64 == 0 (one tensor-core K-step);
 * codes and scales 16-byte aligned.  The operands' scale padding (rows up to
 * the next 128, blocks up to the next 4) must hold finite scales, as the
 * quantizer writes them (0).  M = 0 or N = 0 writes nothing; K = 0 writes
 * zeros.  The tile grid is 256 x 256 outputs per SM pair: shapes off that grid
 * compute the padded tile and store only the valid part.
 */
nvfp4_status nvfp4_gemm(const nvfp4_tensor* A, const nvfp4_tensor* B, void* D, nvfp4_dtype dt, int64_t ldd,
                        void* stream);

/*
 * nvfp4_gemm_amax - nvfp4_gemm that also reduces the tensor amax of its own
 * output in the epilogue: *amax_out = max |D| over the stored values (after
 * the BF16 rounding when dt = BF16).  The next layer's quantization of D then
 * takes amax_out as its amax_in and skips its own amax pass over D (one read
 * of D saved): nvfp4_quantize(D, ..., amax_in = amax_out) equals
 * nvfp4_quantize(D, ..., amax_in = NULL) bit for bit.  amax_out: device
 * float, zeroed and written by the call (on `stream`).  Other arguments and
 * rules as nvfp4_gemm.
 */
nvfp4_status nvfp4_gemm_amax(const nvfp4_tensor* A, const nvfp4_tensor* B, void* D, nvfp4_dtype dt, int64_t ldd,
                             float* amax_out, void* stream);

/*
 * nvfp4_gemm_quantize - the GEMM whose epilogue also emits the next layer's
 * NVFP4 input: D is rounded to BF16 exactly as nvfp4_gemm with dt = BF16
 * writes it, and that M x N BF16 matrix is quantized with 1D blocks of 16
 * along N, round to nearest even, max-6 scaling, using the tensor amax
 * *amax_in (the "producer amax" of "NVIDIA Introduces a 4-Bit Pretraining
 * Methodology Using NVFP4": typically the previous step's amax_out, or a
 * bound the caller holds).  `out` then equals
 *   nvfp4_quantize(D_bf16, BF16, M, N, N, {1D, RNE, max-6, transpose 0},
 *                  amax_in, out)
 * bit for bit, without D being written or read back.  D's codes and scales
 * are written for exactly the M x N outputs (scale padding as 0), and
 * out->global_scale and out->amax are set from *amax_in.  Values above
 * *amax_in saturate to the format's maximum, as in nvfp4_quantize.
 *   A, B     as nvfp4_gemm (K % 64 == 0, K > 0).
 *   amax_in  device float[1], read.
 *   D        device BF16 [M][ldd] or NULL (the BF16 output is then not
 *            stored); ldd >= N, ldd % 8 == 0, 16-byte aligned.
 *   amax_out device float[1] or NULL: as nvfp4_gemm_amax, max |D_bf16| over
 *            the outputs, for the next step's amax_in.  Must not alias
 *            amax_in or out->amax.
 *   out      host struct with device buffers for an M x N tensor (K = N);
 *            N % 16 == 0.
 */
nvfp4_status nvfp4_gemm_quantize(const nvfp4_tensor* A, const nvfp4_tensor* B, const float* amax_in, void* D,
                                 int64_t ldd, float* amax_out, nvfp4_tensor* out, void* stream);

/*
 * nvfp4_gemm_grouped - `count` independent GEMMs D[e] = A[e] * B[e]^T in one
 * launch (routed experts).  A, B: host arrays of `count` tensors; D: host
 * array of `count` device pointers, each row-major [M_e][N_e] (ldd = N_e, so
 * N_e * sizeof(dt) % 16 == 0).  Every group follows the nvfp4_gemm shape rules
 * (M_e may be any count of routed tokens, including 0: the group is skipped)
 * except that K_e must be positive; count <= NVFP4_MAX_GROUPS.
 */
nvfp4_status nvfp4_gemm_grouped(int count, const nvfp4_tensor* A, const nvfp4_tensor* B, void* const* D,
                                nvfp4_dtype dt, void* stream);

/* Synchronise `stream`, then report a pending CUDA error, or a pipeline
 * timeout recorded on the current device.  Every mbarrier wait of the GEMMs
 * and of the TMA-fed transposed encoder is bounded (2 s); on expiry the CTA
 * records it in a device word (bit 0: GEMM, bit 1: encoder), lets its copies
 * in flight land, frees its tensor memory and returns, leaving its outputs
 * undefined.  The word is one per device, shared by every kernel launched on
 * it from any stream or thread: it is read and cleared in one atomic exchange
 * ordered on `stream`, so a timeout is reported once, by the first
 * nvfp4_sync_check that follows it, and with kernels in flight on other
 * streams it may belong to one of those. */
nvfp4_status nvfp4_sync_check(void* stream);

/* Failure-detection test support; no operation of the method.  Arms the next
 * launch this process makes of
 *   op 1: the plain GEMM (nvfp4_gemm, nvfp4_gemm_amax), or
 *   op 2: the TMA-fed transposed encoder (the first kernel of a transposed
 *         nvfp4_quantize / nvfp4_rht_quantize that reads through its ring),
 * so that the first pipeline barrier of every CTA pair (op 1) or CTA (op 2)
 * waits for 16 bytes that no copy delivers.  The bounded wait on it runs out
 * after limit_ns and the kernel takes the timeout path above; the next
 * nvfp4_sync_check reports NVFP4_ERR_TIMEOUT and the device stays usable.
 * limit_ns in [1 ms, 2 s].  Arming is process-wide and consumed by the first
 * launch it matches; limit_ns = 0 disarms.  NVFP4_ERR_INVALID_ARG for another
 * op or limit. */
nvfp4_status nvfp4_test_expire_next_wait(int op, uint64_t limit_ns);

/* Human-readable status name (static string). */
const char* nvfp4_status_string(nvfp4_status s);

/* Text of the last error this thread's calls produced (static per thread). */
const char* nvfp4_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* NVFP4_H_ */
