/*
 * rope_gb300.h -- C ABI of the GB300 (sm_103a) rotary position embedding library.
 *
 * Three operators, each an asynchronous call on a caller-given CUDA stream:
 *
 *   rope_inplace_partial          in-place partial-slice RoPE on a BSND tensor
 *                                 (interleave or half mode), and its backward
 *   rope_with_sin_cos_cache(_v2)  cos/sin-cache-indexed RoPE of query and key (rope /
 *                                 mrope, GPT-NeoX or GPT-J style; V2: interleaved mrope
 *                                 splice, strided inputs, separate outputs)
 *   rope_qkv_rmsnorm_rope_cache   fused QKV split + RMSNorm + RoPE + paged KV-cache write
 *
 * Sources (web pages, cited by title and section):
 *  [IPRM] "CANN ops-transformer 的 aclnnInplacePartialRotaryMul 算子：Inplace
 *         部分旋转位置编码接口详解与实现剖析"
 *  [RSCC] "CANN ops-transformer 旋转位置编码算子 RopeWithSinCosCache 深度解析：
 *         cache 化 RoPE 的计算原理与 aclnn 两段式调用实战"
 *  [QKV]  the "aclnnQkvRmsNormRopeCacheWithKScale" documentation page
 *
 * Memory and ownership.  Every tensor is described by a rope_tensor_t that the
 * caller owns; `data` is a DEVICE pointer to contiguous row-major storage,
 * borrowed for the duration of the call and of the work it enqueues.  All
 * tensors of a call live on the current device (cudaSetDevice), and `stream`
 * belongs to it: the launch goes to the current device.  The
 * library allocates nothing, needs no workspace, and never synchronises the
 * stream (except rope_get_device_error, which says so).  The two-phase
 * "GetWorkspaceSize, then execute" interface of the pages collapses to one call
 * because the workspace is always zero bytes.  (The fused op's kernel uses up to
 * 64 KB of on-chip shared memory per CTA; the first call that needs more than
 * 48 KB on a device raises the kernel's shared-memory limit there, once, with
 * cudaFuncSetAttribute.)
 *
 * Arithmetic.  Half-precision inputs are widened to binary32; each output is
 * a two-term dot product evaluated with Kahan's FMA-based difference of
 * products (relative error <= 2^-23, see Jeannerod, Louvet & Muller, Math. Comp.
 * 82 (2013)) and rounded once, to nearest even, to the output type.  Where
 * both products are exact in binary32 (query, key and the cache all binary16,
 * or all bfloat16, in the GPT-J and out-of-place cache kernels) it is one FMA
 * after an exact product: the correctly rounded binary32 value.  Results are
 * deterministic and do not depend on the launch shape.
 *
 * Errors.  Every argument check happens on the host before anything is
 * enqueued; a failed check returns a status and enqueues nothing.  A shape
 * whose element count (or a strided view's extent) overflows, or exceeds
 * INT64_MAX / 8, is ROPE_ERR_PARAM_INVALID.  So is a tensor the call rewrites
 * that shares memory with a tensor it reads or another one it writes (x with
 * cos or sin; in place, query with key, positions or the cache; an output of
 * the fused op with any other tensor of the call), whose result would depend
 * on the order in which threads run; query and key as disjoint column ranges
 * of one buffer, with one row stride, are accepted.  Status
 * values 161001 and 161002 are the ones [IPRM §返回值与错误码] lists
 * (ACLNN_ERR_PARAM_NULLPTR, ACLNN_ERR_PARAM_INVALID).  A CUDA launch error is
 * returned as ROPE_ERR_CUDA; errors that happen while the work runs surface at
 * the caller's next synchronisation, as with any CUDA launch.
 */
#ifndef ROPE_GB300_H_
#define ROPE_GB300_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ROPE_ABI_VERSION 4

typedef enum {
  ROPE_F32 = 0,  /* IEEE binary32 */
  ROPE_F16 = 1,  /* IEEE binary16 */
  ROPE_BF16 = 2, /* bfloat16 */
  ROPE_I64 = 3   /* int64 (positions only) */
} rope_dtype_t;

/* A borrowed, contiguous, row-major device tensor of 1 to 4 dimensions. */
typedef struct {
  void* data;       /* device pointer; may be NULL only if the tensor is empty */
  int32_t dtype;    /* a rope_dtype_t value */
  int32_t ndim;     /* 1..4 */
  int64_t shape[4]; /* shape[i] for i < ndim; entries past ndim are ignored */
} rope_tensor_t;

enum {
  ROPE_OK = 0,
  ROPE_ERR_PARAM_NULLPTR = 161001, /* a required tensor (or its data) is NULL */
  ROPE_ERR_PARAM_INVALID = 161002, /* dtype, shape, slice, mode or alignment not supported */
  ROPE_ERR_CUDA = 561000           /* the CUDA runtime refused a call (launch or query) */
};

/* Codes reported by rope_get_device_error. */
enum {
  ROPE_DEVICE_OK = 0,
  ROPE_DEVICE_POSITION_OUT_OF_RANGE = 1, /* some position was < 0 or >= maxSeqLen */
  ROPE_DEVICE_SLOT_OUT_OF_RANGE = 2,     /* some KV-cache slot was >= blocks * block size */
  ROPE_DEVICE_INDEX_OUT_OF_BOUNDS = 4    /* bounds-checking builds only: a kernel formed an address
                                            outside the tensor it addresses (the access was skipped) */
};

/*
 * In-place partial RoPE (interleave or half mode).
 * [IPRM §计算原理与公式, §partial_slice 局部旋转机制, §约束说明, §返回值与错误码]
 *
 * For every row r = (b, s, n) of x and every pair of the slice -- slot j and its
 * partner j', with j = start + 2p, j' = j + 1 in interleave mode (rotary_mode 1)
 * and j = start + i, j' = j + L/2 in half mode (rotary_mode 0) --
 *     x[r, j]  <- x[r, j]  * cos[r', j - start]  - x[r, j'] * sin[r', j - start]
 *     x[r, j'] <- x[r, j'] * cos[r', j' - start] + x[r, j]  * sin[r', j' - start]
 * (the page's  x = x*cos + x_rotate*sin  with x_rotate built from the negated
 * partners; interleave is the mode the page opens, half -- rotate_half over the
 * slice -- is the mode it declares), where r' is r broadcast into cos/sin's
 * [cB, cS, cN] dims.  Columns outside [start, end) are never read or written.
 *
 *   x            [B, S, N, D]; F32, F16 or BF16; D even, D <= 1024.  Rewritten in place.
 *   cos, sin     [cB, cS, cN, L] with L = end - start; each of cB, cS, cN is 1 or
 *                equal to x's B, S, N.  Same dtype as x, or F32 when x is F16/BF16
 *                (computed in binary32, the page's mixed-precision combination).
 *   rotary_mode  1 (interleave) or 0 (half); other values are rejected.
 *   start, end   the slice [start, end) of the D axis.  [0, 0] means the whole axis;
 *                any other start == end is a no-op that enqueues nothing.
 *                0 <= start <= end <= D, and end - start even.
 *   stream       a cudaStream_t (NULL: the legacy default stream).
 *
 * Returns ROPE_OK, ROPE_ERR_PARAM_NULLPTR, ROPE_ERR_PARAM_INVALID or ROPE_ERR_CUDA.
 * An empty x (some dim 0) is ROPE_OK and enqueues nothing.
 * Any element alignment is accepted.  Throughput: with 16-byte-aligned pointers
 * and a slice whose start and length are multiples of 16 bytes the kernel moves
 * 16-byte vectors; a slice that starts on a 128-byte boundary of the row touches
 * no more DRAM lines than it rotates, one that does not also fetches the line
 * holding its tail (about twice the DRAM reads for a 128-byte slice).
 */
int rope_inplace_partial(const rope_tensor_t* x, const rope_tensor_t* cos, const rope_tensor_t* sin,
                         int64_t rotary_mode, int64_t start, int64_t end, void* stream);

/*
 * Backward of rope_inplace_partial with respect to x, in place.
 * [IPRM §Python 接口与自动微分: the backward op computes the gradient of x only
 *  (cos/sin get none) and is a no-op for empty tensors and empty slices]
 *
 * `grad` holds dL/dy on entry and dL/dx on return.  Per pair (j, j') as above:
 *     grad[r, j]  <- grad[r, j]  * cos[r', j - start]  + grad[r, j'] * sin[r', j' - start]
 *     grad[r, j'] <- grad[r, j'] * cos[r', j' - start] - grad[r, j]  * sin[r', j - start]
 * i.e. the transpose of the forward map (for a true rotation, the inverse
 * rotation).  Arguments, checks and status values are those of
 * rope_inplace_partial, with `grad` in the place of x.
 */
int rope_inplace_partial_backward(const rope_tensor_t* grad, const rope_tensor_t* cos, const rope_tensor_t* sin,
                                  int64_t rotary_mode, int64_t start, int64_t end, void* stream);

/*
 * Cache-indexed RoPE of query and key, in place.
 * [RSCC §设计动机 (the three steps), §mrope 模式, §rope 模式, §rotate_half（GPT-NeoX style）,
 *  §rotate_interleaved（GPT-J style）, §约束说明, §入参校验逻辑]
 *
 * Per token t: gather cosSin = cache[positions[t]] (mrope: one row per positions
 * row), split it into cos = cosSin[:R/2] and sin = cosSin[R/2:] (mrope: index i
 * of cos and sin comes from the row of the section holding i), then rotate the
 * first R = rotary_dim columns of every head of query and key:
 *   NeoX (is_neox != 0), i < R/2:
 *     o[i] = x[i]*cos[i] - x[i+R/2]*sin[i];   o[i+R/2] = x[i+R/2]*cos[i] + x[i]*sin[i]
 *   GPT-J (is_neox == 0), i < R/2:
 *     o[2i] = x[2i]*cos[i] - x[2i+1]*sin[i];  o[2i+1] = x[2i+1]*cos[i] + x[2i]*sin[i]
 * Columns [R, head_size) of every head pass through: never read or written.
 *
 *   positions      I64; [numTokens] (rope) or [m, numTokens] (mrope, m = mrope_section_len).
 *                  8-byte aligned.
 *   query, key     2-D [numTokens, numQHeads*head_size] / [numTokens, numKHeads*head_size],
 *                  non-empty, same dtype (F32, F16 or BF16), 16-byte aligned.  Rewritten in
 *                  place (the page's queryOut/keyOut alias queryIn/keyIn).
 *   cos_sin_cache  2-D [maxSeqLen, R], same dtype as query, 16-byte aligned.
 *   head_size      a multiple of 32 (F16/BF16) or 16 (F32), dividing both row widths.
 *   rotary_dim     R; must equal cos_sin_cache.shape[1]; R <= head_size and a multiple of
 *                  32 (F16/BF16) or 16 (F32); at most 2048 (F16/BF16 NeoX), 1024 (F16/BF16
 *                  GPT-J, F32 NeoX) or 512 (F32 GPT-J).
 *   is_neox        nonzero: GPT-NeoX rotate_half; zero: GPT-J rotate_interleaved.
 *   mrope_section  HOST pointer to mrope_section_len int64 values, or NULL for rope mode.
 *                  mrope is on when the pointer is non-NULL and mrope_section[0] > 0;
 *                  then mrope_section_len is 3 or 4, every value >= 0, and
 *                  2 * sum == R.  A non-NULL section whose first value is 0 means rope.
 *   stream         a cudaStream_t (NULL: the legacy default stream).
 *
 * Positions outside [0, maxSeqLen) cannot be checked on the host: a token with such a
 * position is left untouched and ROPE_DEVICE_POSITION_OUT_OF_RANGE is recorded for
 * rope_get_device_error.
 *
 * Returns ROPE_OK, ROPE_ERR_PARAM_NULLPTR, ROPE_ERR_PARAM_INVALID or ROPE_ERR_CUDA.
 */
int rope_with_sin_cos_cache(const rope_tensor_t* positions, const rope_tensor_t* query,
                            const rope_tensor_t* key, const rope_tensor_t* cos_sin_cache,
                            int64_t head_size, int64_t rotary_dim, int32_t is_neox,
                            const int64_t* mrope_section, int64_t mrope_section_len, void* stream);

/*
 * Cache-indexed RoPE, V2 form: the V1 operation plus the interleaved mrope
 * splice, strided inputs and separate outputs.
 * [RSCC §V2 接口：cacheMode 扩展; §算子定义与属性 (qStride/kStride: row strides of
 *  query/key for non-contiguous inputs); §接口原型 (queryOut/keyOut)]
 *
 *   cache_mode        0: the sections are spliced in order, as in V1.
 *                     1: interleaved splice (three-section mrope only): cos and sin
 *                     start as the position row 0 values; indices i < 3*mrope_section[1]
 *                     with i % 3 == 1 take row 1, with i % 3 == 2 take row 2.
 *   query_row_stride  elements between the starts of consecutive query rows (0: the row
 *   key_row_stride    width, i.e. contiguous).  At least the row width, and a multiple of
 *                     16 bytes, so that query/key may be views into a fused QKV buffer.
 *   query_out,        NULL, NULL: rotate in place (only the first R columns of each head
 *   key_out           are written).  Otherwise contiguous [numTokens, ...] tensors of the
 *                     inputs' logical shape and dtype, 16-byte aligned, that receive the
 *                     whole rows: rotated columns and pass-through columns copied.  An
 *                     output equal to its input (same pointer, contiguous rows) means in
 *                     place; any other overlap of outputs with inputs is rejected.  Tokens
 *                     with an out-of-range position leave their output rows unwritten.
 *
 * Every other argument, check and status value is that of rope_with_sin_cos_cache.
 */
int rope_with_sin_cos_cache_v2(const rope_tensor_t* positions, const rope_tensor_t* query,
                               const rope_tensor_t* key, const rope_tensor_t* cos_sin_cache,
                               int64_t head_size, int64_t rotary_dim, int32_t is_neox,
                               const int64_t* mrope_section, int64_t mrope_section_len, int32_t cache_mode,
                               int64_t query_row_stride, int64_t key_row_stride, const rope_tensor_t* query_out,
                               const rope_tensor_t* key_out, void* stream);

/*
 * Fused QKV split + RMSNorm + RoPE + paged KV-cache write.
 * ["aclnnQkvRmsNormRopeCacheWithKScale" page, section 计算公式; its FP8
 *  quantisation and optional rotation matmul are not part of this call]
 *
 * Per token t of batch b (t in [query_start_loc[b], query_start_loc[b+1])):
 *   position = seq_lens[b] - (query_start_loc[b+1] - query_start_loc[b]) + (t - query_start_loc[b])
 *   cos, sin = the two halves of cos_sin_cache[position]
 *   for each of the Nq + Nk + Nv heads x of qkv[t] (D elements each):
 *     q and k heads:  y = x / sqrt(mean(x^2) + eps) * gamma   (q_gamma or k_gamma)
 *                     r = concat(y_lo*cos - y_hi*sin, y_hi*cos + y_lo*sin)
 *     q_out[t, h] = r;  k_cache[slot/BS, h, slot%BS, :] = r;  v_cache[slot/BS, h, slot%BS, :] = x (v heads)
 *   with slot = slot_mapping[t] and BS the cache block size.
 *
 *   qkv            [T, (Nq + Nk + Nv) * D]; F32, F16 or BF16; D a multiple of 32 (F16/BF16)
 *                  or 16 (F32), at most 512 (F16/BF16) or 256 (F32).
 *   q_gamma, k_gamma  [D], same dtype.      eps >= 0 (added to the mean of squares).
 *   cos_sin_cache  [maxSeq, D], same dtype: cos in the first half of a row, sin in the second.
 *   seq_lens       I64 [B]: tokens of each sequence including this call's; 1 <= B <= 2^30;
 *   query_start_loc I64 [B + 1]: first token of each batch in qkv, non-decreasing, from 0
 *                  to T (a batch may be empty).  Other values cannot make the kernel
 *                  access memory outside the tensors, but which batch a token is given
 *                  to is then unspecified;
 *   slot_mapping   I64 [T]: cache slot of each token; a negative slot writes no cache
 *                  (padding).
 *   q_out          [T, Nq * D] output; k_cache [NB, Nk, BS, D] and v_cache [NB, Nv, BS, D]
 *                  are updated in place at the tokens' slots only.  Nq + Nk + Nv and BS
 *                  are at most 2^30.
 * All float tensors 16-byte aligned, int64 tensors 8-byte aligned, all contiguous.
 * Computed in binary32 and rounded once per output element: the mean of squares, the
 * reciprocal square root, and the rotation with gamma folded into cos/sin,
 *   r_lo = (x_lo*(g_lo*cos) - x_hi*(g_hi*sin)) / rms,  r_hi = (x_hi*(g_hi*cos) + x_lo*(g_lo*sin)) / rms,
 * each a product, an FMA and the scaling (the terms already carry one rounding of
 * the normalisation, so the compensated difference of rope_with_sin_cos_cache would
 * not make the result more accurate).
 * A token whose position falls outside the table writes nothing and records
 * ROPE_DEVICE_POSITION_OUT_OF_RANGE; a slot at or past NB * BS writes no cache and
 * records ROPE_DEVICE_SLOT_OUT_OF_RANGE (q_out is still written).
 * Returns ROPE_OK, ROPE_ERR_PARAM_NULLPTR, ROPE_ERR_PARAM_INVALID or ROPE_ERR_CUDA.
 */
int rope_qkv_rmsnorm_rope_cache(const rope_tensor_t* qkv, int64_t num_q_heads, int64_t num_k_heads,
                                int64_t num_v_heads, const rope_tensor_t* q_gamma, const rope_tensor_t* k_gamma,
                                float eps, const rope_tensor_t* cos_sin_cache, const rope_tensor_t* seq_lens,
                                const rope_tensor_t* query_start_loc, const rope_tensor_t* slot_mapping,
                                const rope_tensor_t* q_out, const rope_tensor_t* k_cache,
                                const rope_tensor_t* v_cache, void* stream);

/*
 * Takes the device-side error word of the current device (an atomic exchange
 * with zero, enqueued on `stream`), then synchronises `stream`.  *code receives
 * ROPE_DEVICE_OK or a bitwise OR of the ROPE_DEVICE_* codes recorded since the
 * previous read.  The word is shared by every stream and every caller of this
 * process on that device: a read returns (and clears) bits that kernels on other
 * streams recorded too, and no bit is lost between two reads.  Enqueues one
 * one-thread kernel (counted by rope_launch_count).  Returns ROPE_OK,
 * ROPE_ERR_PARAM_NULLPTR (code is NULL) or ROPE_ERR_CUDA.
 */
int rope_get_device_error(void* stream, int32_t* code);

/* A static, human-readable name for a status value (never NULL). */
const char* rope_status_string(int status);

/* Number of kernels this library has launched in this process (all devices). */
uint64_t rope_launch_count(void);

/* ROPE_ABI_VERSION of the built library. */
int rope_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ROPE_GB300_H_ */
