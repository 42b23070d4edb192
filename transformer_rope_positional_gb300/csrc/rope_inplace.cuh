// In-place partial RoPE on a BSND tensor: kernels and launch logic, shared by
// the forward and backward translation units.
//
// Operator: "CANN ops-transformer 的 aclnnInplacePartialRotaryMul 算子：Inplace
// 部分旋转位置编码接口详解与实现剖析", sections 计算原理与公式, partial_slice
// 局部旋转机制 and Python 接口与自动微分.  Per row r = (b, s, n) the slice
// x[r, start:end] is rotated pair by pair with element-wise cos/sin broadcast
// from [cB, cS, cN, L].  A pair is (slot j, partner j'):
//   interleave (rotary_mode 1): j = 2p, j' = 2p + 1
//   half       (rotary_mode 0): j = i,  j' = i + L/2
// forward:  x[j]  <- x[j]  * cos[j]  - x[j'] * sin[j]
//           x[j'] <- x[j'] * cos[j'] + x[j]  * sin[j']
// backward (the transpose, applied to the incoming gradient in place):
//           g[j]  <- g[j]  * cos[j]  + g[j'] * sin[j']
//           g[j'] <- g[j'] * cos[j'] - g[j]  * sin[j]
//
// GB300 design.  The work is HBM-bound (a few flops per 4-8 bytes), so the
// kernel is organised around memory.  The rows (b, s, n) of x form one
// stream, cut into items of U consecutive heads of one token.  A CTA's P row
// groups (C threads each) take P consecutive items and the persistent grid
// strides over the items, so the whole GPU works inside a window of a few MB at
// any moment (good DRAM row-buffer locality).  Thread c of a group owns the
// c-th VEC-element chunk of the slice (half mode: the c-th chunk of each half),
// with 16-byte accesses when the slice is aligned.  When cos/sin are broadcast
// over N (the usual [B|1, S, 1, L] layout) the item's rows share one cos/sin
// chunk, loaded once into registers; otherwise every row loads its own chunk
// alongside x.  All U row loads are issued before any arithmetic.  x is read
// and written once with evict-first (streaming) accesses; cos/sin use the
// read-only path and stay in L2 for the other tokens that share them.  Columns
// outside the slice are never touched.  A slice whose pairs cannot be kept in
// aligned vectors (e.g. an odd start) takes a scalar pair-per-thread kernel.
#pragma once

#include <algorithm>

#include "rope_device.cuh"
#include "rope_launch.h"

namespace rope {
namespace inplace {

// Compile-time launch parameters (the defaults are the measured best on GB300).
#ifndef ROPE_INPLACE_ROWS_IN_FLIGHT
#define ROPE_INPLACE_ROWS_IN_FLIGHT 4
#endif
#ifndef ROPE_INPLACE_THREADS
#define ROPE_INPLACE_THREADS 128
#endif
#ifndef ROPE_INPLACE_MIN_BLOCKS
#define ROPE_INPLACE_MIN_BLOCKS 1
#endif
constexpr int kThreads = ROPE_INPLACE_THREADS;

// Rows per item (U): fewer when every row carries its own cos/sin chunk.
template <bool PER_HEAD_CS>
__host__ __device__ constexpr int rows_per_item() {
  return PER_HEAD_CS ? 2 : ROPE_INPLACE_ROWS_IN_FLIGHT;
}

struct InplaceArgs {
  int64_t S, N, D;
  int64_t start, L;
  int64_t cs_b, cs_s, cs_n;
  int64_t items;        // B * S * head_chunks
  int32_t head_chunks;  // ceil(N / U): chunks of U consecutive heads per token
  int32_t chunks;       // threads per row
  bool items32;         // items (and so tokens) fit 32-bit index arithmetic
  Span xs, coss, sins;  // byte spans of x, cos and sin (checked in debug builds)
  unsigned int* err;    // device error word (debug builds; NULL otherwise)
};

// One pair (a at slot j, b at its partner j') with element-wise cos/sin.
template <bool BWD>
__device__ __forceinline__ void rotate_pair(float& a, float& b, float ca, float sa, float cb, float sb) {
  float na, nb;
  if constexpr (!BWD) {
    na = diff_of_products(a, ca, b, sa);   // a*ca - b*sa
    nb = diff_of_products(b, cb, -a, sb);  // b*cb + a*sb
  } else {
    na = diff_of_products(a, ca, -b, sb);  // a*ca + b*sb
    nb = diff_of_products(b, cb, a, sa);   // b*cb - a*sa
  }
  a = na;
  b = nb;
}

// Rotate one row's chunk(s) held in xv with the cos/sin values of the same
// element positions (NV = 2 in half mode: [0] first half, [1] second half).
template <typename TX, int VEC, int NV, bool HALF, bool BWD>
__device__ __forceinline__ void rotate_chunk(Vec<TX, VEC> (&xv)[NV], const float (&c)[NV][VEC],
                                             const float (&s)[NV][VEC]) {
  if constexpr (HALF) {
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
      float a = widen(xv[0].e[e]), b = widen(xv[1].e[e]);
      rotate_pair<BWD>(a, b, c[0][e], s[0][e], c[NV - 1][e], s[NV - 1][e]);
      xv[0].e[e] = narrow<TX>(a);
      xv[NV - 1].e[e] = narrow<TX>(b);
    }
  } else {
#pragma unroll
    for (int q = 0; q < VEC / 2; ++q) {
      float a = widen(xv[0].e[2 * q]), b = widen(xv[0].e[2 * q + 1]);
      rotate_pair<BWD>(a, b, c[0][2 * q], s[0][2 * q], c[0][2 * q + 1], s[0][2 * q + 1]);
      xv[0].e[2 * q] = narrow<TX>(a);
      xv[0].e[2 * q + 1] = narrow<TX>(b);
    }
  }
}

// PER_HEAD_CS: cos/sin carry their own row for every head (cN == N); otherwise
// one cos/sin row serves all heads of the token.
template <typename TX, typename TC, int VEC, bool PER_HEAD_CS, bool HALF, bool BWD>
__global__ void __launch_bounds__(512, ROPE_INPLACE_MIN_BLOCKS)
    inplace_vec_kernel(TX* __restrict__ x, const TC* __restrict__ cosp, const TC* __restrict__ sinp,
                       InplaceArgs a) {
  constexpr int U = rows_per_item<PER_HEAD_CS>();
  constexpr int NV = HALF ? 2 : 1;  // vectors per row per thread
  const int C = a.chunks;
  const int P = blockDim.x / C;  // row groups per CTA
  const int g = threadIdx.x / C;
  if (g >= P) return;
  const int c = threadIdx.x - g * C;
  const int64_t half = a.L / 2;
  wait_for_prior_grid();

  // item = (token t, head chunk j): heads [j*U, min(j*U + U, N)) of token t
  for (int64_t item = (int64_t)blockIdx.x * P + g; item < a.items; item += (int64_t)gridDim.x * P) {
    const int64_t t = div_index(item, a.head_chunks, a.items32);
    const int h0 = (int)(item - t * a.head_chunks) * U;
    const int n = min(U, (int)a.N - h0);
    TX* xrow = x + (t * a.N + h0) * a.D + a.start + (int64_t)c * VEC;
    const int64_t b = div_index(t, a.S, a.items32);
    const int64_t coff = (b * a.cs_b + (t - b * a.S) * a.cs_s) * a.L + (int64_t)c * VEC;
    // ---- issue the loads of the item's rows (and, per head, of their cos/sin)
    Vec<TX, VEC> xv[U][NV];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (u < n) {
#pragma unroll
        for (int v = 0; v < NV; ++v) load_vec<true>(xv[u][v], xrow + u * a.D + v * half, a.xs, a.err);
      }
    if constexpr (PER_HEAD_CS) {
      Vec<TC, VEC> cv[U][NV], sv[U][NV];
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (u < n) {
          const int64_t o = coff + (int64_t)(h0 + u) * a.cs_n * a.L;
#pragma unroll
          for (int v = 0; v < NV; ++v) {
            load_vec<false>(cv[u][v], cosp + o + v * half, a.coss, a.err);
            load_vec<false>(sv[u][v], sinp + o + v * half, a.sins, a.err);
          }
        }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (u >= n) break;
        float cf[NV][VEC], sf[NV][VEC];
#pragma unroll
        for (int v = 0; v < NV; ++v)
#pragma unroll
          for (int i = 0; i < VEC; ++i) {
            cf[v][i] = widen(cv[u][v].e[i]);
            sf[v][i] = widen(sv[u][v].e[i]);
          }
        rotate_chunk<TX, VEC, NV, HALF, BWD>(xv[u], cf, sf);
#pragma unroll
        for (int v = 0; v < NV; ++v) store_vec(xrow + u * a.D + v * half, xv[u][v], a.xs, a.err);
      }
    } else {
      // one cos/sin chunk serves the item's heads
      float cf[NV][VEC], sf[NV][VEC];
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        load_f32<TC, VEC>(cf[v], cosp + coff + v * half, a.coss, a.err);
        load_f32<TC, VEC>(sf[v], sinp + coff + v * half, a.sins, a.err);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (u >= n) break;
        rotate_chunk<TX, VEC, NV, HALF, BWD>(xv[u], cf, sf);
#pragma unroll
        for (int v = 0; v < NV; ++v) store_vec(xrow + u * a.D + v * half, xv[u][v], a.xs, a.err);
      }
    }
  }
}

// Fallback for slices that cannot be vectorised: one thread per (row, pair),
// scalar accesses.
template <typename TX, typename TC, bool HALF, bool BWD>
__global__ void __launch_bounds__(256) inplace_pair_kernel(TX* __restrict__ x, const TC* __restrict__ cosp,
                                                           const TC* __restrict__ sinp, InplaceArgs a,
                                                           int64_t rows) {
  const int64_t pairs = a.L / 2;
  const int64_t total = rows * pairs;
  wait_for_prior_grid();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = div_index(i, pairs, a.items32);
    const int64_t q = i - r * pairs;
    const int64_t token = div_index(r, a.N, a.items32);
    const int64_t n = r - token * a.N;
    const int64_t b = div_index(token, a.S, a.items32);
    const int64_t s = token - b * a.S;
    const int64_t j = HALF ? q : 2 * q;           // slot
    const int64_t j2 = HALF ? q + pairs : 2 * q + 1;  // partner
    const int64_t co = (b * a.cs_b + s * a.cs_s + n * a.cs_n) * a.L;
    TX* p = x + r * a.D + a.start;
    const bool ok = access_ok(p + j, sizeof(TX), a.xs, a.err) && access_ok(p + j2, sizeof(TX), a.xs, a.err);
    float va = ok ? widen(p[j]) : 0.0f, vb = ok ? widen(p[j2]) : 0.0f;
    // cos/sin element e of this pair's row (zero where a debug build skips the load)
    auto cs = [&](const TC* base, const Span& span, int64_t e) -> float {
      return access_ok(base + co + e, sizeof(TC), span, a.err) ? widen(base[co + e]) : 0.0f;
    };
    rotate_pair<BWD>(va, vb, cs(cosp, a.coss, j), cs(sinp, a.sins, j), cs(cosp, a.coss, j2), cs(sinp, a.sins, j2));
    if (ok) {
      p[j] = narrow<TX>(va);
      p[j2] = narrow<TX>(vb);
    }
  }
}

inline bool aligned(const void* p, int64_t bytes) { return (reinterpret_cast<uintptr_t>(p) % bytes) == 0; }

inline InplaceArgs base_args(const InplaceProblem& p) {
  InplaceArgs a{};
  const int64_t xe = p.x_dtype == kF32 ? 4 : 2, ce = p.cs_dtype == kF32 ? 4 : 2;
  a.xs = make_span(p.x, p.B * p.S * p.N * p.D * xe);
  a.coss = make_span(p.cos, p.cs_rows * p.L * ce);
  a.sins = make_span(p.sin, p.cs_rows * p.L * ce);
  a.err = nullptr;
#ifdef ROPE_DEBUG_BOUNDS
  if (device_error_address(&a.err) != cudaSuccess) a.err = nullptr;
#endif
  a.S = p.S;
  a.N = p.N;
  a.D = p.D;
  a.start = p.start;
  a.L = p.L;
  a.cs_b = p.cs_b;
  a.cs_s = p.cs_s;
  a.cs_n = p.cs_n;
  return a;
}

template <typename TX, typename TC, int VEC, bool PER_HEAD_CS, bool HALF, bool BWD>
cudaError_t launch_vec_kernel(const InplaceProblem& p, cudaStream_t stream) {
  constexpr int U = rows_per_item<PER_HEAD_CS>();
  InplaceArgs a = base_args(p);
  a.chunks = (int32_t)((HALF ? p.L / 2 : p.L) / VEC);
  a.head_chunks = (int32_t)((p.N + U - 1) / U);
  a.items = p.B * p.S * a.head_chunks;
  a.items32 = a.items <= 0xffffffffLL;
  // a row group needs C threads: the block has at least kThreads and at least C
  const int threads = a.chunks > kThreads ? a.chunks : kThreads;
  const int64_t groups = threads / a.chunks;
  // Persistent grid: the CTAs that fit on the GPU at once stride over the items,
  // P consecutive items per CTA per step.
  auto kernel = inplace_vec_kernel<TX, TC, VEC, PER_HEAD_CS, HALF, BWD>;
  const int64_t resident = (int64_t)sm_count() * resident_blocks(reinterpret_cast<const void*>(kernel), threads);
  const int64_t grid = std::max<int64_t>(1, std::min((a.items + groups - 1) / groups, resident));
  return launch_overlapped(kernel, (unsigned)grid, threads, stream, static_cast<TX*>(p.x),
                           static_cast<const TC*>(p.cos), static_cast<const TC*>(p.sin), a);
}

template <typename TX, typename TC, int VEC, bool HALF, bool BWD>
cudaError_t launch_vec(const InplaceProblem& p, cudaStream_t stream) {
  return p.cs_n == 0 ? launch_vec_kernel<TX, TC, VEC, false, HALF, BWD>(p, stream)
                     : launch_vec_kernel<TX, TC, VEC, true, HALF, BWD>(p, stream);
}

template <typename TX, typename TC, bool HALF, bool BWD>
cudaError_t launch_pairs(const InplaceProblem& p, cudaStream_t stream) {
  InplaceArgs a = base_args(p);
  const int64_t rows = p.B * p.S * p.N;
  const int64_t total = rows * (p.L / 2);
  a.items32 = total <= 0xffffffffLL;  // pair indices (and so rows and tokens) fit 32 bits
  const int64_t blocks = std::min<int64_t>((total + 255) / 256, (int64_t)sm_count() * 8);
  return launch_overlapped(inplace_pair_kernel<TX, TC, HALF, BWD>, (unsigned)std::max<int64_t>(1, blocks), 256,
                           stream, static_cast<TX*>(p.x), static_cast<const TC*>(p.cos),
                           static_cast<const TC*>(p.sin), a, rows);
}

// Widest vector (in elements of TX) that the slice (half mode: each half), the
// row pitch and the base pointers all allow; 0 when pairs cannot be kept in
// aligned vectors.
template <typename TX, typename TC, bool HALF>
int pick_vec(const InplaceProblem& p) {
  const int max_vec = 16 / (int)sizeof(TX);
  const int64_t span = HALF ? p.L / 2 : p.L;
  for (int v = max_vec; v >= 2; v /= 2) {
    if (p.start % v || span % v || p.D % v) continue;
    if (!aligned(p.x, v * (int64_t)sizeof(TX))) continue;
    const int64_t cbytes = std::min<int64_t>(16, v * (int64_t)sizeof(TC));
    if (!aligned(p.cos, cbytes) || !aligned(p.sin, cbytes)) continue;
    return v;
  }
  return 0;
}

template <typename TX, typename TC, bool HALF, bool BWD>
cudaError_t dispatch(const InplaceProblem& p, cudaStream_t stream) {
  switch (pick_vec<TX, TC, HALF>(p)) {
    case 8:
      if constexpr (sizeof(TX) == 2) return launch_vec<TX, TC, 8, HALF, BWD>(p, stream);
      break;
    case 4:
      return launch_vec<TX, TC, 4, HALF, BWD>(p, stream);
    case 2:
      return launch_vec<TX, TC, 2, HALF, BWD>(p, stream);
    default:
      break;
  }
  return launch_pairs<TX, TC, HALF, BWD>(p, stream);
}

template <typename TX, typename TC, bool BWD>
cudaError_t dispatch_mode(const InplaceProblem& p, cudaStream_t stream) {
  return p.mode == 0 ? dispatch<TX, TC, true, BWD>(p, stream) : dispatch<TX, TC, false, BWD>(p, stream);
}

template <bool BWD>
cudaError_t launch_direction(const InplaceProblem& p, cudaStream_t stream) {
  const bool f32cs = p.cs_dtype == kF32;
  switch (p.x_dtype) {
    case kF32:
      return dispatch_mode<float, float, BWD>(p, stream);
    case kF16:
      return f32cs ? dispatch_mode<__half, float, BWD>(p, stream) : dispatch_mode<__half, __half, BWD>(p, stream);
    case kBF16:
      return f32cs ? dispatch_mode<__nv_bfloat16, float, BWD>(p, stream)
                   : dispatch_mode<__nv_bfloat16, __nv_bfloat16, BWD>(p, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace inplace
}  // namespace rope
