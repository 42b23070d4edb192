// Cache-indexed RoPE of query and key (rope and mrope modes, GPT-NeoX and GPT-J).
//
// Operator: "CANN ops-transformer 旋转位置编码算子 RopeWithSinCosCache 深度解析：
// cache 化 RoPE 的计算原理与 aclnn 两段式调用实战", sections 设计动机 (gather,
// chunk, rotate), mrope 模式, rope 模式, rotate_half（GPT-NeoX style） and
// rotate_interleaved（GPT-J style）.
//
// GB300 design.  The work is a stream of "head rows" (token t, head h) over
// the query heads then the key heads of each token, R rotated elements each,
// cut into items of U consecutive heads of one token.  A CTA's P row groups (C
// threads each) take P consecutive items and the persistent grid strides over
// the items, so at any moment the whole GPU works inside a window of a few MB
// of q/k: good DRAM row-buffer locality.  Thread c of a group owns one 16-byte
// chunk of a row (NeoX: the same chunk of both halves, GPT-J: VEC/2
// neighbouring pairs) and the matching cos/sin elements, gathered once per
// item (mrope: spliced from the section rows) and kept in registers for its U
// rows.  All U row loads are issued before the gather and any arithmetic, so
// each thread keeps U (NeoX: 2U) 16-byte streaming reads in flight; the
// in-place NeoX variants also load the next item's position rows early, so
// their gather leaves with the row loads.  q/k are read and written once with
// evict-first accesses; the cache goes through the read-only path and stays
// in L2.  Columns [R, head_size) of every head are never touched.
//
// cos/sin staging.  The gathered cos/sin values are staged per item (U heads)
// in registers, read through L2, not once per token in shared memory or by a
// bulk copy: a token's cos/sin row is a few hundred bytes that every item of
// the token finds in L2, and a shared-memory stage needs a team of threads per
// token (all of its heads) whose rows lie far apart.  Measured on GB300 over
// the whole hot-path step: a team per token reusing one staged row across all
// its heads 5.56 TB/s, items of 4 consecutive heads with per-item registers
// 6.07 TB/s (before the launch-overlap and CTA-size changes that followed).
//
// A position outside [0, maxSeqLen) leaves its token untouched and sets bit
// ROPE_DEVICE_POSITION_OUT_OF_RANGE of the device error word below.
#include <algorithm>
#include <mutex>

#include "rope_device.cuh"
#include "rope_launch.h"

namespace rope {

// Device-side error word (one per device context), read and cleared by
// read_and_clear_device_error().
__device__ unsigned int g_device_error;
// The value the last read-and-clear took from g_device_error.
__device__ unsigned int g_device_error_taken;

// Atomically takes the error word and leaves zero in it, so that a bit set by
// a kernel on another stream is either taken now or kept for the next read.
__global__ void take_device_error_kernel() { g_device_error_taken = atomicExch(&g_device_error, 0u); }

namespace {

// Compile-time launch parameters (the defaults are the measured best on GB300).
#ifndef ROPE_CACHE_ROWS_IN_FLIGHT
#define ROPE_CACHE_ROWS_IN_FLIGHT 4
#endif
#ifndef ROPE_CACHE_MIN_BLOCKS
#define ROPE_CACHE_MIN_BLOCKS 1
#endif
#ifndef ROPE_CACHE_THREADS
#define ROPE_CACHE_THREADS 128
#endif
#ifndef ROPE_CACHE_MIN_BLOCKS_GPTJ
#define ROPE_CACHE_MIN_BLOCKS_GPTJ 10
#endif
#ifndef ROPE_CACHE_ROWS_GPTJ
#define ROPE_CACHE_ROWS_GPTJ 4
#endif
#ifndef ROPE_CACHE_PREFETCH_GPTJ
#define ROPE_CACHE_PREFETCH_GPTJ 0
#endif
// 0: the grid is every CTA that fits at once; 1: the fewest CTAs that still
// take the same number of rounds of items (every row group gets an equal share)
#ifndef ROPE_CACHE_EVEN_ROUNDS
#define ROPE_CACHE_EVEN_ROUNDS 0
#endif
constexpr int kThreads = ROPE_CACHE_THREADS;
constexpr unsigned kPositionOutOfRange = 1u;

struct CacheArgs {
  int64_t T;
  int64_t max_seq;
  int64_t q_stride, k_stride;  // elements between consecutive input rows
  int64_t items;       // T * head_chunks
  int32_t head_chunks;  // ceil((hq + hk) / U): chunks of U consecutive heads per token
  int32_t hq, hk;
  int32_t head_size;
  int32_t R;
  int32_t chunks;  // threads per row (C)
  int32_t mrope_rows;
  int32_t section_end[4];
  int32_t cache_mode;      // 0 sectioned splice, 1 interleaved splice (V2)
  int32_t interleave_end;  // cache_mode 1: indices below 3 * mropeSection[1] interleave
  bool items32;            // items fit 32-bit index arithmetic
  // byte spans of the tensors (checked in debug builds)
  Span pos_span, q_span, k_span, cache_span, qo_span, ko_span;
};

// Section holding cos index i.  section_end[] holds cumulative ends and the
// last used end equals R/2, so each comparison adds one for every section that
// ends at or before i (empty sections included) without indexing an array.
__device__ __forceinline__ int section_of(int i, const CacheArgs& a) {
  return (i >= a.section_end[0]) + (i >= a.section_end[1]) + (i >= a.section_end[2]);
}

__device__ __forceinline__ int64_t select_row(int k, int64_t p0, int64_t p1, int64_t p2, int64_t p3) {
  return k == 0 ? p0 : k == 1 ? p1 : k == 2 ? p2 : p3;
}

// How the cos/sin chunk is assembled: plain rope, mrope with the sections
// spliced in order, mrope with the V2 interleaved splice.
enum Splice : int { kRope = 0, kSectioned = 1, kInterleaved = 2 };

// The in-place GPT-J rope kernel (one vector per row and thread, a quarter of
// each row touched) is latency-bound and has its own settings.
template <bool NEOX, bool OUT, int SPLICE>
__host__ __device__ constexpr bool gptj_rope() {
  return !NEOX && !OUT && SPLICE == kRope;
}

// CTAs per SM asked of the compiler: 10 for the GPT-J rope kernel (48
// registers, no spills; beats its uncapped 7); the other variants are best
// uncapped (a cap spills them).
template <bool NEOX, bool OUT, int SPLICE>
__host__ __device__ constexpr int min_blocks() {
  return gptj_rope<NEOX, OUT, SPLICE>() ? ROPE_CACHE_MIN_BLOCKS_GPTJ : ROPE_CACHE_MIN_BLOCKS;
}

// U: head rows per item, all loaded before any arithmetic.
template <bool NEOX, bool OUT, int SPLICE>
__host__ __device__ constexpr int rows_per_item() {
  return gptj_rope<NEOX, OUT, SPLICE>() ? ROPE_CACHE_ROWS_GPTJ : ROPE_CACHE_ROWS_IN_FLIGHT;
}

// Whether the next item's position rows are loaded while the current item is
// processed (so the cos/sin gather leaves with the row loads): measured faster
// for the in-place NeoX kernels; the out-of-place kernels lose an occupancy
// step to the extra registers and are faster without it.
template <bool NEOX, bool OUT, int SPLICE>
__host__ __device__ constexpr bool prefetch_positions() {
  return gptj_rope<NEOX, OUT, SPLICE>() ? ROPE_CACHE_PREFETCH_GPTJ != 0 : (NEOX && !OUT);
}

// The position rows of one token (rope: p[0] only; mrope: 3 or 4 rows).
struct TokenPos {
  int64_t p[4];
};

template <int SPLICE>
__device__ __forceinline__ TokenPos load_positions(const int64_t* __restrict__ pos, const CacheArgs& a, int64_t t) {
  TokenPos r;
  r.p[0] = ldg(pos + t, a.pos_span, &g_device_error);
  if constexpr (SPLICE == kRope) {
    r.p[1] = r.p[2] = r.p[3] = 0;
  } else {
    r.p[1] = ldg(pos + a.T + t, a.pos_span, &g_device_error);
    r.p[2] = ldg(pos + 2 * a.T + t, a.pos_span, &g_device_error);
    r.p[3] = a.mrope_rows > 3 ? ldg(pos + 3 * a.T + t, a.pos_span, &g_device_error) : 0;
  }
  return r;
}

// Steps 1-2 for one token: gather cosSin = cache[positions[t]] and split it
// into this thread's NC cos and NC sin values (first owned index i0).
// Returns false (nothing loaded) when a position is outside [0, maxSeqLen).
template <typename T, int NC, int SPLICE>
__device__ __forceinline__ bool gather_cos_sin(const TokenPos& tp, const T* __restrict__ cache, const CacheArgs& a,
                                               int i0, float (&cf)[NC], float (&sf)[NC]) {
  const int half = a.R / 2;
  if constexpr (SPLICE == kRope) {
    const int64_t p = tp.p[0];
    if (p < 0 || p >= a.max_seq) return false;
    const T* rowp = cache + p * a.R;
    load_f32<T, NC>(cf, rowp + i0, a.cache_span, &g_device_error);
    load_f32<T, NC>(sf, rowp + half + i0, a.cache_span, &g_device_error);
    return true;
  }
  const int64_t p0 = tp.p[0], p1 = tp.p[1], p2 = tp.p[2], p3 = tp.p[3];
  if (p0 < 0 || p0 >= a.max_seq || p1 < 0 || p1 >= a.max_seq || p2 < 0 || p2 >= a.max_seq || p3 < 0 ||
      p3 >= a.max_seq)
    return false;
  if constexpr (SPLICE == kInterleaved) {
    // V2 interleaved splice: row 0, except indices below interleave_end whose
    // remainder mod 3 is 1 (row 1) or 2 (row 2)
    if (i0 >= a.interleave_end) {
      const T* rowp = cache + p0 * a.R;
      load_f32<T, NC>(cf, rowp + i0, a.cache_span, &g_device_error);
      load_f32<T, NC>(sf, rowp + half + i0, a.cache_span, &g_device_error);
    } else {
#pragma unroll
      for (int e = 0; e < NC; ++e) {
        const int i = i0 + e;
        const T* rowp = cache + select_row(i < a.interleave_end ? i % 3 : 0, p0, p1, p2, p3) * a.R;
        cf[e] = widen(ldg(rowp + i, a.cache_span, &g_device_error));
        sf[e] = widen(ldg(rowp + half + i, a.cache_span, &g_device_error));
      }
    }
    return true;
  }
  const int k0 = section_of(i0, a);
  const int k1 = section_of(i0 + NC - 1, a);
  if (k0 == k1) {  // the whole chunk sits in one section: one vector per half
    const T* rowp = cache + select_row(k0, p0, p1, p2, p3) * a.R;
    load_f32<T, NC>(cf, rowp + i0, a.cache_span, &g_device_error);
    load_f32<T, NC>(sf, rowp + half + i0, a.cache_span, &g_device_error);
  } else {  // the chunk straddles a section boundary: per-element rows
#pragma unroll
    for (int e = 0; e < NC; ++e) {
      const T* rowp = cache + select_row(section_of(i0 + e, a), p0, p1, p2, p3) * a.R;
      cf[e] = widen(ldg(rowp + i0 + e, a.cache_span, &g_device_error));
      sf[e] = widen(ldg(rowp + half + i0 + e, a.cache_span, &g_device_error));
    }
  }
  return true;
}

// a*b - c*d is computed with one rounding, by fma(a, b, -(c*d)), when every
// product of two element values is exact in binary32: binary16 products have
// at most 22 significant bits and stay inside the normal binary32 range;
// bfloat16 products have at most 16, and leave the range only beyond 2^128 (an
// infinite c*d, where the compensated form also returns the plain FMA) or
// below 2^-126 (a rounding of at most 2^-150, far below a bfloat16 ulp of any
// result).  Binary32 operands keep the compensated form.
template <typename T>
__host__ __device__ constexpr bool exact_products() {
  return sizeof(T) == 2;
}

// Whether a kernel rotates with that one-FMA form: the GPT-J and out-of-place
// kernels, measured faster with it (the out-of-place NeoX kernels also drop
// under the register count of a fifth CTA per SM); the in-place NeoX kernels
// measured 0.2% faster with the compensated form at the same occupancy.
template <typename T, bool NEOX, bool OUT>
__host__ __device__ constexpr bool fma_rotation() {
  return exact_products<T>() && (!NEOX || OUT);
}

// OUT: results go to the contiguous outputs qo/ko (pass-through columns
// copied there); otherwise query/key are rewritten in place.
template <typename T, bool NEOX, bool OUT, int SPLICE, int VEC>
__global__ void __launch_bounds__(kThreads, min_blocks<NEOX, OUT, SPLICE>())
    cache_kernel(const int64_t* __restrict__ pos, T* __restrict__ q, T* __restrict__ k,
                 const T* __restrict__ cache, T* __restrict__ qo, T* __restrict__ ko, CacheArgs a) {
  constexpr int U = rows_per_item<NEOX, OUT, SPLICE>();
  constexpr int NC = NEOX ? VEC : VEC / 2;  // cos (and sin) indices owned per thread
  constexpr bool kExact = fma_rotation<T, NEOX, OUT>();
  const int C = a.chunks;
  const int P = blockDim.x / C;  // row groups per CTA
  const int g = threadIdx.x / C;
  if (g >= P) return;
  const int c = threadIdx.x - g * C;
  const int half = a.R / 2;
  const int i0 = c * NC;  // first owned cos index
  const int heads = a.hq + a.hk;
  wait_for_prior_grid();

  // item = (token t, head chunk j): heads [j*U, min(j*U + U, heads)) of token t.
  constexpr bool PREFETCH = prefetch_positions<NEOX, OUT, SPLICE>();
  const int64_t stride = (int64_t)gridDim.x * P;
  int64_t item = (int64_t)blockIdx.x * P + g;
  int64_t t = 0;
  TokenPos tp{};
  if constexpr (PREFETCH) {
    if (item < a.items) {
      t = div_index(item, a.head_chunks, a.items32);
      tp = load_positions<SPLICE>(pos, a, t);
    }
  }
  for (; item < a.items; item += stride) {
    if constexpr (!PREFETCH) t = div_index(item, a.head_chunks, a.items32);
    const int h0 = (int)(item - t * a.head_chunks) * U;
    const int n = min(U, heads - h0);
    // ---- issue the loads of the chunk's rows
    T* base[U];
    auto row_span = [&](int u) -> const Span& { return h0 + u < a.hq ? a.q_span : a.k_span; };
    Vec<T, VEC> x1[U], x2[U];  // GPT-J uses x1 only
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int h = h0 + (u < n ? u : 0);
      base[u] = h < a.hq ? q + t * a.q_stride + h * (int64_t)a.head_size
                         : k + t * a.k_stride + (h - a.hq) * (int64_t)a.head_size;
      if (u < n) {
        if constexpr (NEOX) {
          load_vec<true>(x1[u], base[u] + i0, row_span(u), &g_device_error);
          load_vec<true>(x2[u], base[u] + half + i0, row_span(u), &g_device_error);
        } else {
          load_vec<true>(x1[u], base[u] + 2 * i0, row_span(u), &g_device_error);
        }
      }
    }
    // ---- steps 1-2: the token's cos/sin chunk
    if constexpr (!PREFETCH) tp = load_positions<SPLICE>(pos, a, t);
    float cf[NC], sf[NC];
    const bool in_range = gather_cos_sin<T, NC, SPLICE>(tp, cache, a, i0, cf, sf);
    const int64_t tt = t;
    if constexpr (PREFETCH) {  // the next item's token and position rows
      const int64_t next = item + stride;
      if (next < a.items) {
        t = div_index(next, a.head_chunks, a.items32);
        tp = load_positions<SPLICE>(pos, a, t);
      }
    }
    if (!in_range) {
      // reported once per token, by thread 0 of the group holding head 0
      if (c == 0 && h0 == 0) atomicOr(&g_device_error, kPositionOutOfRange);
      continue;  // leave the token untouched
    }
    // ---- step 3: rotate and store
    // Coefficient pairs of the one-FMA form (two lanes per packed
    // instruction): NeoX (c[e], c[e+1]), (s[e], s[e+1]) and the negated sines;
    // GPT-J forms (c, c) and (-s, s) for each pair (a1, a2) where it is used.
    constexpr int NP = kExact && NEOX ? NC / 2 : 1;
    float2 c2[NP], s2[NP], ns2[NP];
    if constexpr (kExact && NEOX) {
#pragma unroll
      for (int j = 0; j < NP; ++j) {
        c2[j] = make_float2(cf[2 * j], cf[2 * j + 1]);
        s2[j] = make_float2(sf[2 * j], sf[2 * j + 1]);
        ns2[j] = make_float2(-sf[2 * j], -sf[2 * j + 1]);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (u >= n) break;
      T* const src = base[u];
      T* dst = src;
      const Span* dspan = &row_span(u);
      if constexpr (OUT) {
        const int h = h0 + u;
        dst = h < a.hq ? qo + (tt * a.hq + h) * (int64_t)a.head_size
                       : ko + (tt * a.hk + (h - a.hq)) * (int64_t)a.head_size;
        dspan = h < a.hq ? &a.qo_span : &a.ko_span;
      }
      if constexpr (NEOX) {
        if constexpr (kExact) {
#pragma unroll
          for (int e = 0; e < VEC; e += 2) {
            const float2 a1 = widen2(&x1[u].e[e]), a2 = widen2(&x2[u].e[e]);
            narrow2(&x1[u].e[e], __ffma2_rn(a1, c2[e / 2], __fmul2_rn(a2, ns2[e / 2])));  // a1*c - a2*s
            narrow2(&x2[u].e[e], __ffma2_rn(a2, c2[e / 2], __fmul2_rn(a1, s2[e / 2])));   // a2*c + a1*s
          }
        } else {
#pragma unroll
          for (int e = 0; e < VEC; ++e) {
            const float a1 = widen(x1[u].e[e]);
            const float a2 = widen(x2[u].e[e]);
            x1[u].e[e] = narrow<T>(diff_of_products(a1, cf[e], a2, sf[e]));
            x2[u].e[e] = narrow<T>(diff_of_products(a2, cf[e], -a1, sf[e]));
          }
        }
        store_vec(dst + i0, x1[u], *dspan, &g_device_error);
        store_vec(dst + half + i0, x2[u], *dspan, &g_device_error);
      } else {
        if constexpr (kExact) {
#pragma unroll
          for (int e = 0; e < NC; ++e) {
            const float2 v = widen2(&x1[u].e[2 * e]);  // (a1, a2) -> (a1*c - a2*s, a2*c + a1*s)
            const float2 w = __fmul2_rn(make_float2(v.y, v.x), make_float2(-sf[e], sf[e]));
            narrow2(&x1[u].e[2 * e], __ffma2_rn(v, make_float2(cf[e], cf[e]), w));
          }
        } else {
#pragma unroll
          for (int e = 0; e < NC; ++e) {
            const float a1 = widen(x1[u].e[2 * e]);
            const float a2 = widen(x1[u].e[2 * e + 1]);
            x1[u].e[2 * e] = narrow<T>(diff_of_products(a1, cf[e], a2, sf[e]));
            x1[u].e[2 * e + 1] = narrow<T>(diff_of_products(a2, cf[e], -a1, sf[e]));
          }
        }
        store_vec(dst + 2 * i0, x1[u], *dspan, &g_device_error);
      }
      if constexpr (OUT) {
        // pass-through columns [R, head_size) are copied to the output row
        for (int j = a.R + c * VEC; j < a.head_size; j += C * VEC) {
          Vec<T, VEC> v;
          load_vec<true>(v, src + j, row_span(u), &g_device_error);
          store_vec(dst + j, v, *dspan, &g_device_error);
        }
      }
    }
  }
}

template <typename T, bool NEOX, bool OUT, int SPLICE>
cudaError_t launch_typed(const CacheProblem& p, cudaStream_t stream) {
  constexpr int VEC = 16 / sizeof(T);
  constexpr int U = rows_per_item<NEOX, OUT, SPLICE>();
  CacheArgs a;
  a.T = p.T;
  a.max_seq = p.max_seq;
  a.q_stride = p.q_stride;
  a.k_stride = p.k_stride;
  a.hq = (int32_t)p.hq;
  a.hk = (int32_t)p.hk;
  a.head_size = (int32_t)p.head_size;
  a.R = (int32_t)p.rotary_dim;
  a.chunks = (int32_t)cache_team_threads(p);
  a.mrope_rows = p.mrope_rows;
  // ends past the used sections are R/2, so section_of() never counts them
  for (int i = 0; i < 4; ++i) a.section_end[i] = i < p.mrope_rows ? p.section_end[i] : (int32_t)(p.rotary_dim / 2);
  a.cache_mode = p.cache_mode;
  a.interleave_end = p.cache_mode == 1 ? 3 * (p.section_end[1] - p.section_end[0]) : 0;
  a.head_chunks = (int32_t)((p.hq + p.hk + U - 1) / U);
  a.items = p.T * a.head_chunks;
  a.items32 = a.items <= 0xffffffffLL;
  const int64_t e = sizeof(T), qw = p.hq * p.head_size, kw = p.hk * p.head_size;
  a.pos_span = make_span(p.positions, (p.mrope_rows ? p.mrope_rows : 1) * p.T * 8);
  a.q_span = make_span(p.query, ((p.T - 1) * p.q_stride + qw) * e);
  a.k_span = make_span(p.key, ((p.T - 1) * p.k_stride + kw) * e);
  a.cache_span = make_span(p.cache, p.max_seq * p.rotary_dim * e);
  a.qo_span = make_span(p.query_out, p.T * qw * e);
  a.ko_span = make_span(p.key_out, p.T * kw * e);
  const int threads = kThreads;
  const int64_t groups = threads / a.chunks;
  // Persistent grid: the CTAs that fit on the GPU at once stride over the items,
  // P consecutive items per CTA per step.
  auto kernel = cache_kernel<T, NEOX, OUT, SPLICE, VEC>;
  const int64_t resident = (int64_t)sm_count() * resident_blocks(reinterpret_cast<const void*>(kernel), threads);
  int64_t grid = std::max<int64_t>(1, std::min((a.items + groups - 1) / groups, resident));
  if (ROPE_CACHE_EVEN_ROUNDS) {
    const int64_t rounds = (a.items + grid * groups - 1) / (grid * groups);
    grid = std::max<int64_t>(1, (a.items + rounds * groups - 1) / (rounds * groups));
  }
  return launch_overlapped(kernel, (unsigned)grid, threads, stream, p.positions, static_cast<T*>(p.query),
                           static_cast<T*>(p.key), static_cast<const T*>(p.cache), static_cast<T*>(p.query_out),
                           static_cast<T*>(p.key_out), a);
}

template <typename T, bool NEOX, bool OUT>
cudaError_t launch_splice(const CacheProblem& p, cudaStream_t stream) {
  if (p.mrope_rows == 0) return launch_typed<T, NEOX, OUT, kRope>(p, stream);
  if (p.cache_mode == 1) return launch_typed<T, NEOX, OUT, kInterleaved>(p, stream);
  return launch_typed<T, NEOX, OUT, kSectioned>(p, stream);
}

template <typename T>
cudaError_t launch_style(const CacheProblem& p, cudaStream_t stream) {
  const bool out = p.query_out != nullptr;
  if (p.is_neox) return out ? launch_splice<T, true, true>(p, stream) : launch_splice<T, true, false>(p, stream);
  return out ? launch_splice<T, false, true>(p, stream) : launch_splice<T, false, false>(p, stream);
}

}  // namespace

int64_t cache_team_threads(const CacheProblem& p) {
  const int64_t vec = 16 / (p.dtype == kF32 ? 4 : 2);
  return p.is_neox ? (p.rotary_dim / 2) / vec : p.rotary_dim / vec;
}

int64_t cache_max_team_threads() { return kThreads; }

cudaError_t launch_cache(const CacheProblem& p, cudaStream_t stream) {
  switch (p.dtype) {
    case kF32:
      return launch_style<float>(p, stream);
    case kF16:
      return launch_style<__half>(p, stream);
    case kBF16:
      return launch_style<__nv_bfloat16>(p, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t device_error_address(unsigned int** out) {
  constexpr int kMaxDevices = 64;
  static unsigned int* addr[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaGetSymbolAddress(reinterpret_cast<void**>(out), g_device_error);
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&addr[dev]), g_device_error);
    if (e != cudaSuccess) return e;
  }
  *out = addr[dev];
  return cudaSuccess;
}

cudaError_t read_and_clear_device_error(cudaStream_t stream, uint32_t* code) {
  // one reader at a time: the taken value sits in one device word until copied out
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  unsigned int host = 0;
  take_device_error_kernel<<<1, 1, 0, stream>>>();
  count_launch();
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess)
    e = cudaMemcpyFromSymbolAsync(&host, g_device_error_taken, sizeof(host), 0, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  *code = host;
  return e;
}

}  // namespace rope
