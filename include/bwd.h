/*
 * bwd.h -- C ABI of the GB300 (sm_103a) 8-bit block-wise dynamic Adam library.
 *
 * The method: "8-BIT OPTIMIZERS VIA BLOCK-WISE QUANTIZATION", as summarised on
 * wiki.neutronadmin.com/news/16836.  Adam's two moments (section 一) are kept
 * as 8-bit codes; for the update they are dequantized to fp32, the update
 * runs, and they are quantized again (section 二, opening paragraph).  Codes
 * index a 256-entry dynamic-tree map (section 二 / 动态量化: sign, zero-run
 * exponent, indicator bit, linear fraction; the second moment uses the
 * unsigned variant whose sign bit is one more fraction bit), and every block
 * of 2048 elements carries one fp32 absmax (section 二 / 逐块量化).
 *
 * Conventions shared by every entry point
 *   - Pointers named "device" are CUDA device (or managed) memory of the
 *     CURRENT device; the caller owns them.  The library keeps only its own
 *     immutable code tables (about 26 KB per device, uploaded on first use)
 *     and one fault word (see bwd_check_device).
 *   - Every device operation is enqueued on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream) and returns without waiting for it.  Launch
 *     errors are reported as BWD_ERR_CUDA; faults inside a kernel surface on
 *     the caller's next synchronisation, as for any CUDA work.
 *   - Arguments are checked on the host before anything is enqueued; a
 *     rejected call has no effect.  n == 0 is a successful no-op.
 *   - Every pointer must be aligned to its element size (4 bytes for fp32,
 *     2 for bf16, 8 for int64; BWD_ERR_INVALID_ARG otherwise).  Beyond that
 *     any alignment is accepted: 16-byte aligned pointers (and, per tensor,
 *     full 2048-element blocks) take the vectorised path; other blocks take
 *     an element-wise path with identical results.
 *   - Input and output ranges must not overlap, except where an argument is
 *     documented as updated in place.
 *   - Non-finite inputs are outside the method; they never cause an
 *     out-of-bounds access but their codes are unspecified.
 *   - The first call on a device uploads the tables with a blocking copy, so
 *     it must not happen during CUDA stream capture; bwd_init() does it
 *     explicitly.
 *   - Entry points are thread-safe; bwd_last_error() is per thread.
 */
#ifndef BWD_H
#define BWD_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Elements per quantization block (section 二 / 逐块量化). */
#define BWD_BLOCK 2048

typedef enum {
  BWD_OK = 0,
  BWD_ERR_INVALID_ARG = 1,       /* null pointer, negative size, bad enum, ... */
  BWD_ERR_UNSUPPORTED_DTYPE = 2, /* gradient dtype not in bwd_dtype          */
  BWD_ERR_CUDA = 3               /* a CUDA runtime call or launch failed      */
} bwd_status;

/* Which dynamic-tree map (section 二 / 动态量化). */
typedef enum {
  BWD_MAP_SIGNED = 0,   /* sign + zero-run exponent + indicator + fraction  */
  BWD_MAP_UNSIGNED = 1  /* the sign bit reused as fraction (second moment)  */
} bwd_map_kind;

/* Element types of gradients and (for bwd_adam8bit_step_multi_ex) of
 * parameters: fp32, bf16, IEEE binary16.  16-bit values widen exactly; 16-bit
 * parameters are rounded back to nearest, ties to even. */
typedef enum { BWD_F32 = 0, BWD_BF16 = 1, BWD_F16 = 2 } bwd_dtype;

/* Adam hyper-parameters (section 一: first and second moment).  `step` is
 * the 1-based index t of the step being taken (bias corrections use it).
 * weight_decay >= 0 is decoupled weight decay (AdamW, an extension of the
 * method): p is first scaled by fp32(1 - lr * weight_decay); 0 gives Adam. */
typedef struct {
  float lr;
  float beta1;
  float beta2;
  float eps;
  float weight_decay;
  int64_t step;
} bwd_adam_hparams;

/* Number of 2048-element blocks of an n-element tensor: ceil(n / 2048).
 * Returns -1 for n < 0. */
int64_t bwd_num_blocks(int64_t n);

/* Host only.  Writes the 256-entry map of `kind` in ascending order (a code
 * is an index into it; the signed map holds -0.0 at 127 and +0.0 at 128) and
 * the 255 decision thresholds, threshold i being the binary32 value nearest
 * to the midpoint of entries i and i+1.  Magnitudes follow the dynamic-tree
 * layout of section 二 / 动态量化 with a decimal zero-run exponent and a
 * linear fraction grid on (0.1, 1] per decade.  Either output may be NULL. */
bwd_status bwd_build_map(bwd_map_kind kind, float* map_out /*[256]*/,
                         float* thresholds_out /*[255]*/);

/* Uploads the code tables to the current device if not done yet (blocking).
 * Optional: every entry point below does it on first use. */
bwd_status bwd_init(void);

/* Block-wise quantization (section 二 / 逐块量化 and 动态量化).
 *   x      : device, float[n], read only.
 *   codes  : device, uint8[n], written: index of the nearest map entry to
 *            x / absmax (binary32 IEEE division; a value exactly on a
 *            threshold takes the higher code; +-0 take the code of +0).
 *   absmax : device, float[ceil(n/2048)], written: max |x| of each block
 *            (the last block may be partial).  A block whose absmax is 0
 *            gets the code of +0.0 everywhere. */
bwd_status bwd_quantize_blockwise(const float* x, int64_t n, bwd_map_kind kind,
                                  uint8_t* codes, float* absmax, void* stream);

/* Block-wise dequantization (section 一: back from codes to values).
 *   codes  : device, uint8[n]; absmax: device, float[ceil(n/2048)].
 *   y      : device, float[n], written: map[code] * absmax[block] (one
 *            binary32 multiply). */
bwd_status bwd_dequantize_blockwise(const uint8_t* codes, const float* absmax,
                                    int64_t n, bwd_map_kind kind, float* y,
                                    void* stream);

/* State before the first step: m codes := code of +0.0 in the signed map,
 * v codes := code of 0 in the unsigned map, both absmax := 0.
 *   m_codes, v_codes : device uint8[n];  m_absmax, v_absmax : device
 *   float[ceil(n/2048)].  All written. */
bwd_status bwd_state_init(uint8_t* m_codes, float* m_absmax, uint8_t* v_codes,
                          float* v_absmax, int64_t n, void* stream);

/* One 8-bit Adam step on one flat tensor (section 二, opening paragraph):
 * dequantize m (signed map) and v (unsigned map), run Adam in fp32,
 *     m = b1 m + (1-b1) g;  v = b2 v + ((1-b2) g) g;
 *     p = p d - (s m) / (sqrt(v) / c + eps),
 * with s = fp32(lr / (1 - b1^t)), c = fp32(sqrt(1 - b2^t)) and the decay
 * factor d = fp32(1 - lr wd) formed in binary64 on the host; then requantize
 * m and v block by block with fresh absmax.  m and v take one binary32
 * rounding per operation in that order, so the new codes and absmax are
 * exactly those of IEEE arithmetic; the parameter update uses approximate
 * (sqrt / rcp) arithmetic and is within a few ulps of the update term.
 *   p                : device float[n], updated in place.
 *   g                : device, float[n], bf16[n] or fp16[n] per g_dtype, read
 *                      only.
 *   m_codes, v_codes : device uint8[n], updated in place.
 *   m_absmax,v_absmax: device float[ceil(n/2048)], updated in place.
 *   hp               : host pointer; hp->step >= 1, lr and eps finite,
 *                      eps >= 0, betas in [0, 1), weight_decay finite >= 0. */
bwd_status bwd_adam8bit_step(float* p, const void* g, bwd_dtype g_dtype,
                             uint8_t* m_codes, float* m_absmax,
                             uint8_t* v_codes, float* v_absmax, int64_t n,
                             const bwd_adam_hparams* hp, void* stream);

/* The same step over a list of tensors in as few launches as the kernel
 * parameter space allows (448 tensors per launch).  Blocks never span two
 * tensors.  All arrays are HOST arrays of length num_tensors holding device
 * pointers (or sizes); each tensor follows the single-tensor contract above.
 * Tensors with n == 0 are skipped; num_tensors == 0 is a no-op. */
bwd_status bwd_adam8bit_step_multi(int32_t num_tensors, float* const* p,
                                   const void* const* g, bwd_dtype g_dtype,
                                   uint8_t* const* m_codes,
                                   float* const* m_absmax,
                                   uint8_t* const* v_codes,
                                   float* const* v_absmax, const int64_t* n,
                                   const bwd_adam_hparams* hp, void* stream);

/* The multi-tensor step with the parameter type given: p_dtype BWD_F32
 * (as bwd_adam8bit_step_multi), BWD_BF16 or BWD_F16.  16-bit parameters are
 * widened to fp32 for the update and stored back rounded to nearest even
 * (the page's low-precision state with a high-precision update, section 二,
 * opening paragraph, which names FP16); codes and absmax are the same as
 * with fp32 parameters.
 *   p : HOST array of num_tensors device pointers to fp32[n], bf16[n] or
 *       fp16[n] parameters, updated in place.  Other arguments as above. */
bwd_status bwd_adam8bit_step_multi_ex(int32_t num_tensors, void* const* p,
                                      bwd_dtype p_dtype, const void* const* g,
                                      bwd_dtype g_dtype, uint8_t* const* m_codes,
                                      float* const* m_absmax,
                                      uint8_t* const* v_codes,
                                      float* const* v_absmax, const int64_t* n,
                                      const bwd_adam_hparams* hp, void* stream);

/* ------------------------------------------------------------------------
 * ZeRO-style sharding of the step over P processes ("Яндекс Публикует ЯЛМ
 * 100Б", section "ZeRO" under "Случай с несколькими графическими
 * процессорами": each process keeps the values and optimizer state of its own
 * group of parameters and alone updates them, so its step is O(N / P); the
 * gradients are reduced before the step and the parameters gathered after
 * it).  Blocks are independent (section 二 / 逐块量化 of the 8-bit optimizer
 * page), so the split follows block boundaries and a rank's step over its
 * pieces (bwd_adam8bit_step_multi / _ex, pointers offset by `offset`
 * elements) equals the unsharded step on those elements bit for bit.
 *
 * Layout: in a padded flat space tensor i occupies the blocks
 * [B_i, B_i + ceil(n_i / 2048)), B the prefix sums of the block counts and NB
 * their total; rank r owns the K = ceil(NB / world) blocks [r K, (r + 1) K)
 * clipped to NB (the last ranks may own fewer, or none), so padded buffers of
 * world * K * 2048 elements split into equal per-rank slices.
 *   n               : HOST int64[num_tensors], tensor sizes (0 allowed).
 *   world, rank     : 1 <= world, 0 <= rank < world.
 *   blocks_per_rank : HOST int64 out, K (may be NULL).
 *   num_pieces      : HOST int32 out, the tensors the rank's blocks touch.
 *   tensor, offset, count : HOST arrays of capacity num_tensors, written
 *            (each may be NULL): piece j is the elements
 *            [offset[j], offset[j] + count[j]) of tensor tensor[j]; offsets
 *            are multiples of 2048; pieces ascend in tensor order.
 * Host only (no device is touched).  BWD_ERR_INVALID_ARG for a negative size,
 * a NULL pointer, world < 1, rank outside [0, world) or a total that
 * overflows. */
bwd_status bwd_zero_shard(int32_t num_tensors, const int64_t* n, int32_t world,
                          int32_t rank, int64_t* blocks_per_rank,
                          int32_t* num_pieces, int32_t* tensor,
                          int64_t* offset, int64_t* count);

/* ------------------------------------------------------------------------
 * Stable embedding layer (section 二 / 稳定的词嵌入层): the embedding weight
 * is initialised Xavier-uniform and a layer normalisation follows the
 * lookup, so that the layer's output has variance close to 1.
 *   weight : device fp32[V * D], row-major (row v = embedding of token v).
 *   gamma, beta : device fp32[D], the normalisation's scale and shift.
 *   ids    : device int64[T] token ids.  An id outside [0, V) is outside
 *            the method: its output row is NaN (no access leaves the
 *            weight) and the backward pass skips it.
 * D a multiple of 4 and at most 4096 with 16-byte aligned weight, gamma,
 * beta / dy, y / dweight takes the vectorised path; any other shape takes an
 * element-wise path with the same arithmetic.  All fp32, eps as given.
 * Errors: BWD_ERR_INVALID_ARG for V < 1, D < 1, T < 0, V * D or T * D
 * overflowing int64, a NULL pointer, a non-finite or negative eps. */

/* Xavier-uniform initialisation from caller-supplied random words:
 * weight[i] = fp32((2 u_i - 1) * b), u_i = (words[i] >> 8) * 2^-24 and
 * b = fp32(sqrt(6 / (V + D))) (Glorot's bound for fan-in D and fan-out V;
 * 2 u - 1 is exact, so each weight takes one rounding).
 *   words  : device uint32[V * D], e.g. from any uniform 32-bit generator.
 *   weight : device fp32[V * D], written. */
bwd_status bwd_embedding_init(const uint32_t* words, int64_t num_embeddings,
                              int64_t dim, float* weight, void* stream);

/* Host only: the bound b above, or -1 for V < 1 or D < 1. */
float bwd_embedding_xavier_bound(int64_t num_embeddings, int64_t dim);

/* Forward: for each token t with x = weight[ids[t]],
 *   mean = sum(x) / D,  var = sum((x - mean)^2) / D,
 *   rstd = 1 / sqrt(var + eps),  y = (x - mean) * rstd * gamma + beta.
 *   y    : device fp32[T * D], written.
 *   mean, rstd : device fp32[T], written (the backward pass reads them);
 *          either may be NULL when no backward pass follows.
 * Row statistics are reduced in a fixed order: results are deterministic. */
bwd_status bwd_embedding_forward(const int64_t* ids, int64_t num_tokens,
                                 const float* weight, int64_t num_embeddings,
                                 int64_t dim, const float* gamma,
                                 const float* beta, float eps, float* y,
                                 float* mean, float* rstd, void* stream);

/* Backward: with xhat = (x - mean) * rstd (mean, rstd from the forward call)
 * and g = dy * gamma, per token
 *   dx = rstd * (g - mean(g) - xhat * mean(g * xhat)),
 * ACCUMULATED into the caller's buffers (zero them for a fresh gradient):
 *   dweight[ids[t]] += dx   (device fp32[V * D]; repeated ids add up),
 *   dgamma += sum_t dy * xhat,  dbeta += sum_t dy   (device fp32[D]).
 *   dy : device fp32[T * D].
 * The adds are atomic, so their order, and the last bits of dweight, dgamma
 * and dbeta, may differ between runs. */
bwd_status bwd_embedding_backward(const int64_t* ids, int64_t num_tokens,
                                  const float* weight, int64_t num_embeddings,
                                  int64_t dim, const float* gamma,
                                  const float* mean, const float* rstd,
                                  const float* dy, float* dweight,
                                  float* dgamma, float* dbeta, void* stream);

/* Waits for `stream` and reports whether a bounded wait inside one of the
 * library's kernels gave up since the last check (the staged embedding
 * backward waits for its own bulk copies; each wait gives up after about a
 * second, flags the device and lets the kernel return).  BWD_OK, or
 * BWD_ERR_CUDA with bwd_last_error() describing it; the flag is cleared.
 * Blocking; not callable during stream capture. */
bwd_status bwd_check_device(void* stream);

/* Self-test of the bounded waits: enqueues one kernel that waits for an
 * mbarrier phase nothing completes.  Its wait gives up after about a second,
 * sets the fault word and returns (no trap, the context stays usable); the
 * next bwd_check_device therefore returns BWD_ERR_CUDA and clears the word.
 * For tests and diagnostics; no counterpart in the method. */
bwd_status bwd_selftest_bounded_wait(void* stream);

/* Static description of a status code. */
const char* bwd_status_string(bwd_status status);

/* Detail of the last failed call on this thread ("" if none). */
const char* bwd_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* BWD_H */
