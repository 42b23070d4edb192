// C ABI of the RoPE library: argument checks, dispatch, status strings.
//
// The checks follow the constraint and error-code lists of the two operator
// pages ("CANN ops-transformer 的 aclnnInplacePartialRotaryMul 算子…", sections
// 返回值与错误码 and 约束说明; "CANN ops-transformer 旋转位置编码算子
// RopeWithSinCosCache 深度解析…", sections 约束说明 and 入参校验逻辑).  Every check
// runs on the host before anything is enqueued, and no check touches the GPU,
// so a rejected call has no side effect at all.
#include <initializer_list>

#include "rope_gb300.h"
#include "rope_launch.h"


namespace {

using rope::kBF16;
using rope::kF16;
using rope::kF32;
using rope::kI64;

bool is_float(int32_t dt) { return dt == kF32 || dt == kF16 || dt == kBF16; }

// Largest element count accepted: the byte size of any tensor (8 bytes per
// element at most) and every element offset the kernels form stay in int64.
constexpr int64_t kMaxElements = INT64_MAX / 8;

// Product of the dims of a tensor that passed shape_ok().
int64_t numel(const rope_tensor_t* t) {
  int64_t n = 1;
  for (int i = 0; i < t->ndim; ++i) n *= t->shape[i];
  return n;
}

// 1 to 4 non-negative dims whose product (taken in order) stays within
// kMaxElements; a shape whose product overflows is rejected, not wrapped.
bool shape_ok(const rope_tensor_t* t) {
  if (t->ndim < 1 || t->ndim > 4) return false;
  int64_t n = 1;
  for (int i = 0; i < t->ndim; ++i) {
    if (t->shape[i] < 0) return false;
    if (__builtin_mul_overflow(n, t->shape[i], &n) || n > kMaxElements) return false;
  }
  return true;
}

// Elements spanned by `rows` rows of `width` elements, `stride` apart:
// (rows - 1) * stride + width, or -1 when that leaves kMaxElements.
int64_t strided_extent(int64_t rows, int64_t stride, int64_t width) {
  int64_t n = 0;
  if (rows <= 0) return 0;
  if (__builtin_mul_overflow(rows - 1, stride, &n) || __builtin_add_overflow(n, width, &n) || n > kMaxElements)
    return -1;
  return n;
}

bool aligned(const void* p, uintptr_t bytes) { return reinterpret_cast<uintptr_t>(p) % bytes == 0; }

int64_t elem_size(int32_t dt) { return dt == kF32 ? 4 : dt == kI64 ? 8 : 2; }

// Whether two sets of `rows` rows share a byte: set a starts at byte address
// a, its rows are aw bytes wide and as bytes apart (likewise b).  Sets whose
// byte ranges meet are treated as overlapping unless both have one stride s
// and their columns are disjoint modulo s (e.g. the q and k column ranges of
// one fused QKV buffer).  Empty sets overlap nothing.
bool rows_overlap(uintptr_t a, int64_t as, int64_t aw, uintptr_t b, int64_t bs, int64_t bw, int64_t rows) {
  if (rows <= 0 || aw <= 0 || bw <= 0) return false;
  const uintptr_t a_end = a + (uintptr_t)((rows - 1) * as + aw), b_end = b + (uintptr_t)((rows - 1) * bs + bw);
  if (a_end <= b || b_end <= a) return false;
  if (rows == 1 || as != bs || aw > as || bw > bs) return true;
  // a covers [0, aw) of every period of as bytes, b covers [r, r + bw)
  const int64_t d = (int64_t)(b - a);
  const int64_t r = ((d % as) + as) % as;
  return r < aw || r + bw > as;
}

// Whether the byte ranges [a, a + an) and [b, b + bn) share a byte.
bool ranges_overlap(uintptr_t a, int64_t an, uintptr_t b, int64_t bn) {
  return an > 0 && bn > 0 && a < b + (uintptr_t)bn && b < a + (uintptr_t)an;
}

// Whether two contiguous tensors (the byte ranges of their elements) overlap.
bool tensors_overlap(const rope_tensor_t* x, const rope_tensor_t* y) {
  return ranges_overlap(reinterpret_cast<uintptr_t>(x->data), numel(x) * elem_size(x->dtype),
                        reinterpret_cast<uintptr_t>(y->data), numel(y) * elem_size(y->dtype));
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? ROPE_OK : ROPE_ERR_CUDA; }

// Checks shared by the forward and backward in-place calls, then the launch.
int inplace_call(const rope_tensor_t* x, const rope_tensor_t* cos, const rope_tensor_t* sin, int64_t rotary_mode,
                 int64_t start, int64_t end, bool backward, void* stream) {
  if (!x || !cos || !sin) return ROPE_ERR_PARAM_NULLPTR;
  // dtypes: x in {F32, F16, BF16}; cos == sin; cos == x, or F32 with a half x
  if (!is_float(x->dtype) || !is_float(cos->dtype) || cos->dtype != sin->dtype) return ROPE_ERR_PARAM_INVALID;
  if (cos->dtype != x->dtype && !(cos->dtype == kF32 && x->dtype != kF32)) return ROPE_ERR_PARAM_INVALID;
  // modes: 1 interleave, 0 half; the other enum values have no formula
  if (rotary_mode != 1 && rotary_mode != 0) return ROPE_ERR_PARAM_INVALID;
  if (x->ndim != 4 || cos->ndim != 4 || sin->ndim != 4) return ROPE_ERR_PARAM_INVALID;
  if (!shape_ok(x) || !shape_ok(cos) || !shape_ok(sin)) return ROPE_ERR_PARAM_INVALID;
  for (int i = 0; i < 4; ++i)
    if (cos->shape[i] != sin->shape[i]) return ROPE_ERR_PARAM_INVALID;
  const int64_t D = x->shape[3];
  if (D > 1024 || D % 2) return ROPE_ERR_PARAM_INVALID;
  if (start < 0 || end < 0 || end > D || start > end) return ROPE_ERR_PARAM_INVALID;
  if (start == 0 && end == 0) end = D;  // no slice: the whole D axis
  const int64_t L = end - start;
  if (L % 2) return ROPE_ERR_PARAM_INVALID;
  if (L == 0) return ROPE_OK;  // empty slice: no-op, nothing enqueued
  if (cos->shape[3] != L) return ROPE_ERR_PARAM_INVALID;
  for (int i = 0; i < 3; ++i)
    if (cos->shape[i] != 1 && cos->shape[i] != x->shape[i]) return ROPE_ERR_PARAM_INVALID;
  if (numel(x) == 0) return ROPE_OK;
  if (!x->data || !cos->data || !sin->data) return ROPE_ERR_PARAM_NULLPTR;
  const uintptr_t xe = x->dtype == kF32 ? 4 : 2, ce = cos->dtype == kF32 ? 4 : 2;
  if (!aligned(x->data, xe) || !aligned(cos->data, ce) || !aligned(sin->data, ce)) return ROPE_ERR_PARAM_INVALID;
  // x is rewritten while cos/sin are read: they must not share memory
  if (tensors_overlap(x, cos) || tensors_overlap(x, sin)) return ROPE_ERR_PARAM_INVALID;

  rope::InplaceProblem p;
  p.mode = (int32_t)rotary_mode;
  p.backward = backward;
  p.x = x->data;
  p.cos = cos->data;
  p.sin = sin->data;
  p.x_dtype = x->dtype;
  p.cs_dtype = cos->dtype;
  p.B = x->shape[0];
  p.S = x->shape[1];
  p.N = x->shape[2];
  p.D = D;
  p.start = start;
  p.L = L;
  const int64_t cB = cos->shape[0], cS = cos->shape[1], cN = cos->shape[2];
  p.cs_n = cN == 1 ? 0 : 1;
  p.cs_s = cS == 1 ? 0 : cN;
  p.cs_b = cB == 1 ? 0 : cS * cN;
  p.cs_rows = cB * cS * cN;
  return cuda_status(rope::launch_inplace(p, static_cast<cudaStream_t>(stream)));
}

// Checks shared by the V1 and V2 cache calls, then the launch.
int cache_call(const rope_tensor_t* positions, const rope_tensor_t* query, const rope_tensor_t* key,
               const rope_tensor_t* cos_sin_cache, int64_t head_size, int64_t rotary_dim, int32_t is_neox,
               const int64_t* mrope_section, int64_t mrope_section_len, int32_t cache_mode, int64_t q_row_stride,
               int64_t k_row_stride, const rope_tensor_t* query_out, const rope_tensor_t* key_out, void* stream) {
  if (!positions || !query || !key || !cos_sin_cache) return ROPE_ERR_PARAM_NULLPTR;
  // dtypes: positions int64; query, key and cache the same floating type
  if (positions->dtype != kI64 || !is_float(query->dtype)) return ROPE_ERR_PARAM_INVALID;
  if (key->dtype != query->dtype || cos_sin_cache->dtype != query->dtype) return ROPE_ERR_PARAM_INVALID;
  // shapes: query, key, cache 2-D and non-empty; same token count
  if (query->ndim != 2 || key->ndim != 2 || cos_sin_cache->ndim != 2) return ROPE_ERR_PARAM_INVALID;
  if (!shape_ok(query) || !shape_ok(key) || !shape_ok(cos_sin_cache) || !shape_ok(positions))
    return ROPE_ERR_PARAM_INVALID;
  if (numel(query) == 0 || numel(key) == 0 || numel(cos_sin_cache) == 0) return ROPE_ERR_PARAM_INVALID;
  const int64_t T = query->shape[0];
  if (key->shape[0] != T) return ROPE_ERR_PARAM_INVALID;
  // head size and rotary dim: 64-byte multiples; R == cache width <= head size
  const int64_t mult = query->dtype == kF32 ? 16 : 32;
  if (head_size <= 0 || head_size % mult) return ROPE_ERR_PARAM_INVALID;
  if (query->shape[1] % head_size || key->shape[1] % head_size) return ROPE_ERR_PARAM_INVALID;
  if (rotary_dim != cos_sin_cache->shape[1]) return ROPE_ERR_PARAM_INVALID;
  if (rotary_dim <= 0 || rotary_dim % mult || rotary_dim > head_size) return ROPE_ERR_PARAM_INVALID;
  // mode and positions shape
  const bool mrope = mrope_section != nullptr && mrope_section_len > 0 && mrope_section[0] > 0;
  if (mrope_section != nullptr && mrope_section_len != 3 && mrope_section_len != 4) return ROPE_ERR_PARAM_INVALID;
  int32_t section_end[4] = {0, 0, 0, 0};
  if (mrope_section != nullptr) {
    int64_t sum = 0;
    for (int64_t i = 0; i < mrope_section_len; ++i) {
      if (mrope_section[i] < 0) return ROPE_ERR_PARAM_INVALID;
      sum += mrope_section[i];
      section_end[i] = (int32_t)sum;
    }
    if (mrope && 2 * sum != rotary_dim) return ROPE_ERR_PARAM_INVALID;
  }
  if (mrope) {
    if (positions->ndim != 2 || positions->shape[0] != mrope_section_len || positions->shape[1] != T)
      return ROPE_ERR_PARAM_INVALID;
  } else {
    if (positions->ndim != 1 || positions->shape[0] != T) return ROPE_ERR_PARAM_INVALID;
  }
  // V2: interleaved splice only for three-section mrope
  if (cache_mode != 0 && cache_mode != 1) return ROPE_ERR_PARAM_INVALID;
  if (cache_mode == 1 && !(mrope && mrope_section_len == 3)) return ROPE_ERR_PARAM_INVALID;
  // row strides (elements): 0 means contiguous rows
  const int64_t qw = query->shape[1], kw = key->shape[1];
  const int64_t qs = q_row_stride ? q_row_stride : qw, ks = k_row_stride ? k_row_stride : kw;
  const int64_t esz = query->dtype == kF32 ? 4 : 2;
  if (qs < qw || ks < kw || qs % (16 / esz) || ks % (16 / esz)) return ROPE_ERR_PARAM_INVALID;
  if (strided_extent(T, qs, qw) < 0 || strided_extent(T, ks, kw) < 0) return ROPE_ERR_PARAM_INVALID;
  // outputs: both or neither; contiguous, same shape and dtype as the inputs
  if ((query_out == nullptr) != (key_out == nullptr)) return ROPE_ERR_PARAM_NULLPTR;
  if (query_out) {
    if (query_out->dtype != query->dtype || key_out->dtype != key->dtype) return ROPE_ERR_PARAM_INVALID;
    if (query_out->ndim != 2 || key_out->ndim != 2 || query_out->shape[0] != T || query_out->shape[1] != qw ||
        key_out->shape[0] != T || key_out->shape[1] != kw)
      return ROPE_ERR_PARAM_INVALID;
    if (!query_out->data || !key_out->data) return ROPE_ERR_PARAM_NULLPTR;
    if (!aligned(query_out->data, 16) || !aligned(key_out->data, 16)) return ROPE_ERR_PARAM_INVALID;
  }
  if (!positions->data || !query->data || !key->data || !cos_sin_cache->data) return ROPE_ERR_PARAM_NULLPTR;
  if (!aligned(positions->data, 8) || !aligned(query->data, 16) || !aligned(key->data, 16) ||
      !aligned(cos_sin_cache->data, 16))
    return ROPE_ERR_PARAM_INVALID;
  // an output that is its input (same pointer, contiguous rows) means in place;
  // any other overlap between the outputs and the inputs is rejected
  bool in_place = query_out == nullptr;
  if (!in_place && query_out->data == query->data && key_out->data == key->data && qs == qw && ks == kw)
    in_place = true;
  {
    // rewritten rows must not share memory with each other or with the tables
    const uintptr_t qa = reinterpret_cast<uintptr_t>(query->data), ka = reinterpret_cast<uintptr_t>(key->data);
    const int64_t pb = numel(positions) * 8, cb = numel(cos_sin_cache) * esz;
    const uintptr_t pa = reinterpret_cast<uintptr_t>(positions->data),
                    ca = reinterpret_cast<uintptr_t>(cos_sin_cache->data);
    const int64_t qn = ((T - 1) * qs + qw) * esz, kn = ((T - 1) * ks + kw) * esz;
    if (in_place && (rows_overlap(qa, qs * esz, qw * esz, ka, ks * esz, kw * esz, T) ||
                     ranges_overlap(qa, qn, pa, pb) || ranges_overlap(qa, qn, ca, cb) ||
                     ranges_overlap(ka, kn, pa, pb) || ranges_overlap(ka, kn, ca, cb)))
      return ROPE_ERR_PARAM_INVALID;
  }
  if (!in_place) {
    const char* spans[4][2] = {
        {static_cast<const char*>(query->data), static_cast<const char*>(query->data) + ((T - 1) * qs + qw) * esz},
        {static_cast<const char*>(key->data), static_cast<const char*>(key->data) + ((T - 1) * ks + kw) * esz},
        {static_cast<const char*>(query_out->data), static_cast<const char*>(query_out->data) + T * qw * esz},
        {static_cast<const char*>(key_out->data), static_cast<const char*>(key_out->data) + T * kw * esz}};
    for (int o = 2; o < 4; ++o)
      for (int i = 0; i < 4; ++i)
        if (i != o && spans[o][0] < spans[i][1] && spans[i][0] < spans[o][1]) return ROPE_ERR_PARAM_INVALID;
  }

  rope::CacheProblem p;
  p.positions = static_cast<const int64_t*>(positions->data);
  p.query = query->data;
  p.key = key->data;
  p.cache = cos_sin_cache->data;
  p.dtype = query->dtype;
  p.T = T;
  p.hq = query->shape[1] / head_size;
  p.hk = key->shape[1] / head_size;
  p.head_size = head_size;
  p.rotary_dim = rotary_dim;
  p.max_seq = cos_sin_cache->shape[0];
  p.is_neox = is_neox != 0;
  p.mrope_rows = mrope ? (int32_t)mrope_section_len : 0;
  for (int i = 0; i < 4; ++i) p.section_end[i] = section_end[i];
  p.cache_mode = cache_mode;
  p.q_stride = qs;
  p.k_stride = ks;
  p.query_out = in_place ? nullptr : query_out->data;
  p.key_out = in_place ? nullptr : key_out->data;
  // one team of threads must fit one block of the cache kernel
  if (rope::cache_team_threads(p) > rope::cache_max_team_threads()) return ROPE_ERR_PARAM_INVALID;
  if (p.hq + p.hk > (int64_t)1 << 30 || head_size > (int64_t)1 << 30) return ROPE_ERR_PARAM_INVALID;
  return cuda_status(rope::launch_cache(p, static_cast<cudaStream_t>(stream)));
}

// Checks of the fused QKV call, then the launch.
int qkv_call(const rope_tensor_t* qkv, int64_t nq, int64_t nk, int64_t nv, const rope_tensor_t* q_gamma,
             const rope_tensor_t* k_gamma, float eps, const rope_tensor_t* cache, const rope_tensor_t* seq_lens,
             const rope_tensor_t* qsl, const rope_tensor_t* slot_mapping, const rope_tensor_t* q_out,
             const rope_tensor_t* k_cache, const rope_tensor_t* v_cache, void* stream) {
  const rope_tensor_t* all[] = {qkv, q_gamma, k_gamma, cache, seq_lens, qsl, slot_mapping, q_out, k_cache, v_cache};
  for (const rope_tensor_t* t : all)
    if (!t) return ROPE_ERR_PARAM_NULLPTR;
  for (const rope_tensor_t* t : all)
    if (!shape_ok(t)) return ROPE_ERR_PARAM_INVALID;
  // dtypes: one floating type for the data, int64 for the metadata
  const int32_t dt = qkv->dtype;
  if (!is_float(dt)) return ROPE_ERR_PARAM_INVALID;
  for (const rope_tensor_t* t : {q_gamma, k_gamma, cache, q_out, k_cache, v_cache})
    if (t->dtype != dt) return ROPE_ERR_PARAM_INVALID;
  for (const rope_tensor_t* t : {seq_lens, qsl, slot_mapping})
    if (t->dtype != kI64 || t->ndim != 1) return ROPE_ERR_PARAM_INVALID;
  // shapes
  if (nq < 0 || nk < 0 || nv < 0 || nq + nk + nv < 1) return ROPE_ERR_PARAM_INVALID;
  if (qkv->ndim != 2 || qkv->shape[0] < 1 || qkv->shape[1] % (nq + nk + nv)) return ROPE_ERR_PARAM_INVALID;
  const int64_t T = qkv->shape[0], D = qkv->shape[1] / (nq + nk + nv);
  const int64_t mult = dt == kF32 ? 16 : 32;
  const int64_t lanes = D / 2 / (dt == kF32 ? 4 : 8);  // threads per head row
  if (D < mult || D % mult || lanes > 32) return ROPE_ERR_PARAM_INVALID;
  if (q_gamma->ndim != 1 || q_gamma->shape[0] != D || k_gamma->ndim != 1 || k_gamma->shape[0] != D)
    return ROPE_ERR_PARAM_INVALID;
  if (cache->ndim != 2 || cache->shape[1] != D || cache->shape[0] < 1) return ROPE_ERR_PARAM_INVALID;
  const int64_t B = seq_lens->shape[0];
  if (B < 1 || B > (int64_t(1) << 30) || qsl->shape[0] != B + 1 || slot_mapping->shape[0] != T)
    return ROPE_ERR_PARAM_INVALID;
  if (q_out->ndim != 2 || q_out->shape[0] != T || q_out->shape[1] != nq * D) return ROPE_ERR_PARAM_INVALID;
  if (k_cache->ndim != 4 || v_cache->ndim != 4) return ROPE_ERR_PARAM_INVALID;
  const int64_t NB = k_cache->shape[0], BS = k_cache->shape[2];
  if (NB < 1 || BS < 1 || k_cache->shape[1] != nk || k_cache->shape[3] != D || v_cache->shape[0] != NB ||
      v_cache->shape[1] != nv || v_cache->shape[2] != BS || v_cache->shape[3] != D)
    return ROPE_ERR_PARAM_INVALID;
  int64_t slots = 0;  // NB * BS, also when a cache has no heads (and so no elements)
  if (__builtin_mul_overflow(NB, BS, &slots) || slots > kMaxElements) return ROPE_ERR_PARAM_INVALID;
  // head counts and the block size are kept in 32-bit fields by the kernel
  if (nq + nk + nv > (int64_t(1) << 30) || BS > (int64_t(1) << 30)) return ROPE_ERR_PARAM_INVALID;
  if (!(eps >= 0.0f) || !(eps < 1e30f)) return ROPE_ERR_PARAM_INVALID;
  for (const rope_tensor_t* t : all)
    if (!t->data && numel(t) > 0) return ROPE_ERR_PARAM_NULLPTR;
  // the outputs are written while every input is read: no output may share
  // memory with an input or with another output
  for (const rope_tensor_t* o : {q_out, k_cache, v_cache})
    for (const rope_tensor_t* t : all)
      if (t != o && tensors_overlap(o, t)) return ROPE_ERR_PARAM_INVALID;
  for (const rope_tensor_t* t : {qkv, q_gamma, k_gamma, cache, q_out, k_cache, v_cache})
    if (t->data && !aligned(t->data, 16)) return ROPE_ERR_PARAM_INVALID;
  for (const rope_tensor_t* t : {seq_lens, qsl, slot_mapping})
    if (!aligned(t->data, 8)) return ROPE_ERR_PARAM_INVALID;

  rope::QkvProblem p;
  p.qkv = qkv->data;
  p.q_gamma = q_gamma->data;
  p.k_gamma = k_gamma->data;
  p.cache = cache->data;
  p.seq_lens = static_cast<const int64_t*>(seq_lens->data);
  p.query_start_loc = static_cast<const int64_t*>(qsl->data);
  p.slot_mapping = static_cast<const int64_t*>(slot_mapping->data);
  p.q_out = q_out->data;
  p.k_cache = k_cache->data;
  p.v_cache = v_cache->data;
  p.dtype = dt;
  p.T = T;
  p.B = B;
  p.nq = nq;
  p.nk = nk;
  p.nv = nv;
  p.D = D;
  p.max_seq = cache->shape[0];
  p.num_blocks = NB;
  p.block_size = BS;
  p.eps = eps;
  return cuda_status(rope::launch_qkv(p, static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

int rope_inplace_partial(const rope_tensor_t* x, const rope_tensor_t* cos, const rope_tensor_t* sin,
                         int64_t rotary_mode, int64_t start, int64_t end, void* stream) {
  return inplace_call(x, cos, sin, rotary_mode, start, end, false, stream);
}

int rope_inplace_partial_backward(const rope_tensor_t* grad, const rope_tensor_t* cos, const rope_tensor_t* sin,
                                  int64_t rotary_mode, int64_t start, int64_t end, void* stream) {
  return inplace_call(grad, cos, sin, rotary_mode, start, end, true, stream);
}

int rope_with_sin_cos_cache(const rope_tensor_t* positions, const rope_tensor_t* query,
                            const rope_tensor_t* key, const rope_tensor_t* cos_sin_cache,
                            int64_t head_size, int64_t rotary_dim, int32_t is_neox,
                            const int64_t* mrope_section, int64_t mrope_section_len, void* stream) {
  return cache_call(positions, query, key, cos_sin_cache, head_size, rotary_dim, is_neox, mrope_section,
                    mrope_section_len, 0, 0, 0, nullptr, nullptr, stream);
}

int rope_with_sin_cos_cache_v2(const rope_tensor_t* positions, const rope_tensor_t* query,
                               const rope_tensor_t* key, const rope_tensor_t* cos_sin_cache,
                               int64_t head_size, int64_t rotary_dim, int32_t is_neox,
                               const int64_t* mrope_section, int64_t mrope_section_len, int32_t cache_mode,
                               int64_t query_row_stride, int64_t key_row_stride, const rope_tensor_t* query_out,
                               const rope_tensor_t* key_out, void* stream) {
  return cache_call(positions, query, key, cos_sin_cache, head_size, rotary_dim, is_neox, mrope_section,
                    mrope_section_len, cache_mode, query_row_stride, key_row_stride, query_out, key_out, stream);
}

int rope_qkv_rmsnorm_rope_cache(const rope_tensor_t* qkv, int64_t num_q_heads, int64_t num_k_heads,
                                int64_t num_v_heads, const rope_tensor_t* q_gamma, const rope_tensor_t* k_gamma,
                                float eps, const rope_tensor_t* cos_sin_cache, const rope_tensor_t* seq_lens,
                                const rope_tensor_t* query_start_loc, const rope_tensor_t* slot_mapping,
                                const rope_tensor_t* q_out, const rope_tensor_t* k_cache,
                                const rope_tensor_t* v_cache, void* stream) {
  return qkv_call(qkv, num_q_heads, num_k_heads, num_v_heads, q_gamma, k_gamma, eps, cos_sin_cache, seq_lens,
                  query_start_loc, slot_mapping, q_out, k_cache, v_cache, stream);
}

int rope_get_device_error(void* stream, int32_t* code) {
  if (!code) return ROPE_ERR_PARAM_NULLPTR;
  uint32_t c = 0;
  const cudaError_t e = rope::read_and_clear_device_error(static_cast<cudaStream_t>(stream), &c);
  *code = (int32_t)c;
  return cuda_status(e);
}

const char* rope_status_string(int status) {
  switch (status) {
    case ROPE_OK:
      return "ROPE_OK";
    case ROPE_ERR_PARAM_NULLPTR:
      return "ROPE_ERR_PARAM_NULLPTR: a required tensor or its data pointer is NULL";
    case ROPE_ERR_PARAM_INVALID:
      return "ROPE_ERR_PARAM_INVALID: unsupported dtype, shape, slice, mode, section or alignment";
    case ROPE_ERR_CUDA:
      return "ROPE_ERR_CUDA: the CUDA runtime rejected a launch or query";
    default:
      return "unknown status";
  }
}

uint64_t rope_launch_count(void) { return rope::launch_count(); }

int rope_abi_version(void) { return ROPE_ABI_VERSION; }

}  // extern "C"
