// Device-side building blocks shared by the RoPE kernels: element conversions,
// vector loads/stores with cache policies, and the accurate two-term dot product.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <float.h>
#include <stdint.h>

namespace rope {

// Wait until the grid this kernel depends on (the previous kernel of the
// stream, when launched with programmatic stream serialization) has completed
// and its memory is visible; returns at once otherwise.
__device__ __forceinline__ void wait_for_prior_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Element conversions: every storage type is widened exactly to binary32 and
// narrowed back with one round-to-nearest-even.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float widen(float v) { return v; }
__device__ __forceinline__ float widen(__half v) { return __half2float(v); }
__device__ __forceinline__ float widen(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ T narrow(float v);
template <>
__device__ __forceinline__ float narrow<float>(float v) { return v; }
template <>
__device__ __forceinline__ __half narrow<__half>(float v) { return __float2half_rn(v); }
template <>
__device__ __forceinline__ __nv_bfloat16 narrow<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// Adjacent element pairs <-> float2, for the packed binary32 instructions
// (__ffma2_rn, __fmul2_rn) that issue two lanes of arithmetic at once.
__device__ __forceinline__ float2 widen2(const float* p) { return make_float2(p[0], p[1]); }
__device__ __forceinline__ float2 widen2(const __half* p) {
  return __half22float2(*reinterpret_cast<const __half2*>(p));
}
__device__ __forceinline__ float2 widen2(const __nv_bfloat16* p) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}
__device__ __forceinline__ void narrow2(float* p, float2 v) {
  p[0] = v.x;
  p[1] = v.y;
}
__device__ __forceinline__ void narrow2(__half* p, float2 v) {
  *reinterpret_cast<__half2*>(p) = __floats2half2_rn(v.x, v.y);
}
__device__ __forceinline__ void narrow2(__nv_bfloat16* p, float2 v) {
  *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(v.x, v.y);
}

// ---------------------------------------------------------------------------
// Bounds checking (debug builds, -DROPE_DEBUG_BOUNDS).  Every global access of
// the kernels goes through access_ok() with the byte span of the tensor it
// addresses.  In a debug build an access that leaves its span is skipped (a
// skipped load yields zeros) and sets kIndexOutOfBounds in the device error
// word; nothing traps.  In a release build the spans are empty structs and
// access_ok() is the constant true, so the check costs nothing.
// ---------------------------------------------------------------------------
constexpr unsigned kIndexOutOfBounds = 4u;

struct Span {
#ifdef ROPE_DEBUG_BOUNDS
  const char* lo;
  const char* hi;  // one past the last byte
#endif
};

// The span [p, p + bytes) (host side).
inline Span make_span(const void* p, int64_t bytes) {
  Span s;
#ifdef ROPE_DEBUG_BOUNDS
  s.lo = static_cast<const char*>(p);
  s.hi = static_cast<const char*>(p) + (bytes > 0 ? bytes : 0);
#else
  (void)p;
  (void)bytes;
#endif
  return s;
}

__device__ __forceinline__ bool access_ok(const void* p, int bytes, const Span& s, unsigned int* err) {
#ifdef ROPE_DEBUG_BOUNDS
  const char* c = static_cast<const char*>(p);
  if (c >= s.lo && c + bytes <= s.hi) return true;
  atomicOr(err, kIndexOutOfBounds);
  return false;
#else
  (void)p;
  (void)bytes;
  (void)s;
  (void)err;
  return true;
#endif
}

// Quotient of a non-negative index by a positive divisor, in 32-bit
// arithmetic when the host has checked that both fit (much cheaper than the
// 64-bit division sequence).
__device__ __forceinline__ int64_t div_index(int64_t n, int64_t d, bool fits32) {
  return fits32 ? (int64_t)((uint32_t)n / (uint32_t)d) : n / d;
}

// ---------------------------------------------------------------------------
// a*b - c*d with relative error at most 2^-23 (Kahan's algorithm: the rounding
// error of c*d is recovered exactly by an FMA and added back; bound from
// Jeannerod, Louvet & Muller, "Further analysis of Kahan's algorithm for the
// accurate computation of 2x2 determinants", Math. Comp. 82 (2013)).  When c*d
// is not finite the error term is meaningless and the plain FMA result is the
// IEEE answer.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float diff_of_products(float a, float b, float c, float d) {
  const float w = __fmul_rn(c, d);
  const float e = __fmaf_rn(-c, d, w);  // w - c*d, exact
  const float f = __fmaf_rn(a, b, -w);  // a*b - w, one rounding
  const float r = __fadd_rn(f, e);
  return fabsf(e) <= FLT_MAX ? r : f;
}

// ---------------------------------------------------------------------------
// A register array of N elements, aligned so that it can be moved in 16-byte
// (or smaller power-of-two) pieces.
// ---------------------------------------------------------------------------
template <typename T, int N>
struct alignas((N * sizeof(T)) >= 16 ? 16 : (N * sizeof(T))) Vec {
  T e[N];
};

// Global -> registers.  STREAM: data touched once (evict-first in L1 and L2);
// otherwise read-only data that other threads reuse (non-coherent path).
template <bool STREAM, int BYTES>
__device__ __forceinline__ void gload(void* dst, const void* src) {
  if constexpr (BYTES >= 16) {
    static_assert(BYTES % 16 == 0, "vector size");
#pragma unroll
    for (int k = 0; k < BYTES / 16; ++k) {
      const uint4* s = static_cast<const uint4*>(src) + k;
      static_cast<uint4*>(dst)[k] = STREAM ? __ldcs(s) : __ldg(s);
    }
  } else if constexpr (BYTES == 8) {
    const uint2* s = static_cast<const uint2*>(src);
    *static_cast<uint2*>(dst) = STREAM ? __ldcs(s) : __ldg(s);
  } else if constexpr (BYTES == 4) {
    const unsigned int* s = static_cast<const unsigned int*>(src);
    *static_cast<unsigned int*>(dst) = STREAM ? __ldcs(s) : __ldg(s);
  } else {
    static_assert(BYTES == 2, "vector size");
    const unsigned short* s = static_cast<const unsigned short*>(src);
    *static_cast<unsigned short*>(dst) = STREAM ? __ldcs(s) : __ldg(s);
  }
}

// Registers -> global, streaming (evict-first).
template <int BYTES>
__device__ __forceinline__ void gstore(void* dst, const void* src) {
  if constexpr (BYTES >= 16) {
#pragma unroll
    for (int k = 0; k < BYTES / 16; ++k)
      __stcs(static_cast<uint4*>(dst) + k, static_cast<const uint4*>(src)[k]);
  } else if constexpr (BYTES == 8) {
    __stcs(static_cast<uint2*>(dst), *static_cast<const uint2*>(src));
  } else if constexpr (BYTES == 4) {
    __stcs(static_cast<unsigned int*>(dst), *static_cast<const unsigned int*>(src));
  } else {
    static_assert(BYTES == 2, "vector size");
    __stcs(static_cast<unsigned short*>(dst), *static_cast<const unsigned short*>(src));
  }
}

template <bool STREAM, typename T, int N>
__device__ __forceinline__ void load_vec(Vec<T, N>& v, const T* p) {
  gload<STREAM, N * sizeof(T)>(v.e, p);
}

template <typename T, int N>
__device__ __forceinline__ void store_vec(T* p, const Vec<T, N>& v) {
  gstore<N * sizeof(T)>(p, v.e);
}

// Read-only vector load widened to binary32.
template <typename T, int N>
__device__ __forceinline__ void load_f32(float (&out)[N], const T* p) {
  Vec<T, N> v;
  load_vec<false>(v, p);
#pragma unroll
  for (int i = 0; i < N; ++i) out[i] = widen(v.e[i]);
}

// The same accesses with the bounds check of access_ok() (a no-op in release
// builds; in debug builds a skipped load yields zeros).
template <bool STREAM, typename T, int N>
__device__ __forceinline__ void load_vec(Vec<T, N>& v, const T* p, const Span& s, unsigned int* err) {
  if (access_ok(p, N * sizeof(T), s, err)) {
    load_vec<STREAM>(v, p);
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) v.e[i] = T(0.0f);
  }
}

template <typename T, int N>
__device__ __forceinline__ void store_vec(T* p, const Vec<T, N>& v, const Span& s, unsigned int* err) {
  if (access_ok(p, N * sizeof(T), s, err)) store_vec(p, v);
}

template <typename T, int N>
__device__ __forceinline__ void load_f32(float (&out)[N], const T* p, const Span& s, unsigned int* err) {
  if (access_ok(p, N * sizeof(T), s, err)) {
    load_f32<T, N>(out, p);
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) out[i] = 0.0f;
  }
}

// ---------------------------------------------------------------------------
// Asynchronous 16-byte global -> shared copies (cp.async, cached in L2 only,
// evict-first there), completed in commit groups.  A thread that copies into
// a shared-memory slot and later reads that slot itself needs only
// cp_async_wait(), no barrier.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, uint64_t policy) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "l"(policy)
               : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// Wait until at most N of this thread's commit groups are still in flight.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// The copy with the bounds check of access_ok() (a skipped copy leaves zeros).
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, uint64_t policy, const Span& s,
                                           unsigned int* err) {
  if (access_ok(gmem, 16, s, err)) {
    cp_async16(smem, gmem, policy);
  } else {
    *static_cast<uint4*>(smem) = make_uint4(0u, 0u, 0u, 0u);
  }
}

// Scalar read-only load (zero when a debug build skips it).
template <typename T>
__device__ __forceinline__ T ldg(const T* p, const Span& s, unsigned int* err) {
  return access_ok(p, sizeof(T), s, err) ? __ldg(p) : T(0);
}

}  // namespace rope
