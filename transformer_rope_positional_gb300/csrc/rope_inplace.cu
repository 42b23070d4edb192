// In-place partial interleave RoPE on a BSND tensor.
//
// Operator: "CANN ops-transformer 的 aclnnInplacePartialRotaryMul 算子：Inplace
// 部分旋转位置编码接口详解与实现剖析", sections 计算原理与公式 and
// partial_slice 局部旋转机制.  For each row r = (b, s, n) and pair p of the
// slice (j = start + 2p), with cos/sin broadcast into r':
//   x[r, j]   <- x[r, j]   * cos[r', 2p]   - x[r, j+1] * sin[r', 2p]
//   x[r, j+1] <- x[r, j+1] * cos[r', 2p+1] + x[r, j]   * sin[r', 2p+1]
//
// GB300 design.  The work is HBM-bound (about 3 flops per 4-8 bytes), so the
// kernel is organised around memory.  The rows (b, s, n) of x form one
// stream, cut into items of U consecutive heads of one token.  A CTA's P row
// groups (C threads each) take P consecutive items and the persistent grid
// strides over the items, so the whole GPU works inside a window of a few MB at
// any moment (good DRAM row-buffer locality).  Thread c of a group owns the
// c-th VEC-element chunk of the slice (16-byte accesses when the slice is
// aligned).  When cos/sin are broadcast over N (the usual [B|1, S, 1, L]
// layout) the item's rows share one cos/sin chunk, loaded once into registers;
// otherwise every row loads its own chunk alongside x.  All U row loads are
// issued before any arithmetic.  x is read and written once with evict-first
// (streaming) accesses; cos/sin use the read-only path and stay in L2 for the
// other tokens that share them.  Columns outside the slice are never touched.
// A slice whose start is odd cannot be paired within an aligned vector and
// takes a scalar pair-per-thread kernel instead.
#include <algorithm>

#include "rope_device.cuh"
#include "rope_launch.h"

namespace rope {
namespace {

// Compile-time launch parameters (the defaults are the measured best on GB300).
#ifndef ROPE_INPLACE_ROWS_IN_FLIGHT
#define ROPE_INPLACE_ROWS_IN_FLIGHT 4
#endif
#ifndef ROPE_INPLACE_THREADS
#define ROPE_INPLACE_THREADS 256
#endif
#ifndef ROPE_INPLACE_MIN_BLOCKS
#define ROPE_INPLACE_MIN_BLOCKS 1
#endif
constexpr int kRowsInFlight = ROPE_INPLACE_ROWS_IN_FLIGHT;  // U: rows loaded before compute, per thread
constexpr int kThreads = ROPE_INPLACE_THREADS;

struct InplaceArgs {
  int64_t S, N, D;
  int64_t start, L;
  int64_t cs_b, cs_s, cs_n;
  int64_t items;        // B * S * head_chunks
  int32_t head_chunks;  // ceil(N / U): chunks of U consecutive heads per token
  int32_t chunks;       // threads per row = L / VEC
};

// Rotate VEC/2 interleaved pairs held in xv with per-element cos/sin.
template <typename TX, int VEC>
__device__ __forceinline__ void rotate_interleaved_pairs(Vec<TX, VEC>& xv, const float (&c)[VEC],
                                                         const float (&s)[VEC]) {
#pragma unroll
  for (int q = 0; q < VEC / 2; ++q) {
    const float x0 = widen(xv.e[2 * q]);
    const float x1 = widen(xv.e[2 * q + 1]);
    const float y0 = diff_of_products(x0, c[2 * q], x1, s[2 * q]);
    const float y1 = diff_of_products(x1, c[2 * q + 1], -x0, s[2 * q + 1]);
    xv.e[2 * q] = narrow<TX>(y0);
    xv.e[2 * q + 1] = narrow<TX>(y1);
  }
}

// PER_HEAD_CS: cos/sin carry their own row for every head (cN == N); otherwise
// one cos/sin row serves all heads of the token.
template <typename TX, typename TC, int VEC, bool PER_HEAD_CS>
__global__ void __launch_bounds__(512, ROPE_INPLACE_MIN_BLOCKS)
    inplace_vec_kernel(TX* __restrict__ x, const TC* __restrict__ cosp, const TC* __restrict__ sinp,
                       InplaceArgs a) {
  constexpr int U = kRowsInFlight;
  const int C = a.chunks;
  const int P = blockDim.x / C;  // row groups per CTA
  const int g = threadIdx.x / C;
  if (g >= P) return;
  const int c = threadIdx.x - g * C;
  wait_for_prior_grid();

  // item = (token t, head chunk j): heads [j*U, min(j*U + U, N)) of token t
  for (int64_t item = (int64_t)blockIdx.x * P + g; item < a.items; item += (int64_t)gridDim.x * P) {
    const int64_t t = item / a.head_chunks;
    const int h0 = (int)(item - t * a.head_chunks) * U;
    const int n = min(U, (int)a.N - h0);
    TX* xrow = x + (t * a.N + h0) * a.D + a.start + (int64_t)c * VEC;
    const int64_t b = t / a.S;
    const int64_t coff = (b * a.cs_b + (t - b * a.S) * a.cs_s) * a.L + (int64_t)c * VEC;
    // ---- issue the loads of the item's rows (and, per head, of their cos/sin)
    Vec<TX, VEC> xv[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (u < n) load_vec<true>(xv[u], xrow + u * a.D);
    if constexpr (PER_HEAD_CS) {
      Vec<TC, VEC> cv[U], sv[U];
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (u < n) {
          const int64_t o = coff + (int64_t)(h0 + u) * a.cs_n * a.L;
          load_vec<false>(cv[u], cosp + o);
          load_vec<false>(sv[u], sinp + o);
        }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (u >= n) break;
        float cf[VEC], sf[VEC];
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
          cf[i] = widen(cv[u].e[i]);
          sf[i] = widen(sv[u].e[i]);
        }
        rotate_interleaved_pairs<TX, VEC>(xv[u], cf, sf);
        store_vec(xrow + u * a.D, xv[u]);
      }
    } else {
      // one cos/sin chunk serves the item's heads
      float cf[VEC], sf[VEC];
      load_f32<TC, VEC>(cf, cosp + coff);
      load_f32<TC, VEC>(sf, sinp + coff);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (u >= n) break;
        rotate_interleaved_pairs<TX, VEC>(xv[u], cf, sf);
        store_vec(xrow + u * a.D, xv[u]);
      }
    }
  }
}

// Fallback for slices that cannot be vectorised (odd start or misaligned
// base): one thread per (row, pair), scalar accesses.
template <typename TX, typename TC>
__global__ void __launch_bounds__(256) inplace_pair_kernel(TX* __restrict__ x, const TC* __restrict__ cosp,
                                                           const TC* __restrict__ sinp, InplaceArgs a,
                                                           int64_t rows) {
  const int64_t pairs = a.L / 2;
  const int64_t total = rows * pairs;
  wait_for_prior_grid();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / pairs;
    const int64_t q = i - r * pairs;
    const int64_t n = r % a.N;
    const int64_t token = r / a.N;
    const int64_t b = token / a.S;
    const int64_t s = token - b * a.S;
    const int64_t co = (b * a.cs_b + s * a.cs_s + n * a.cs_n) * a.L + 2 * q;
    TX* p = x + r * a.D + a.start + 2 * q;
    const float x0 = widen(p[0]);
    const float x1 = widen(p[1]);
    const float c0 = widen(cosp[co]), c1 = widen(cosp[co + 1]);
    const float s0 = widen(sinp[co]), s1 = widen(sinp[co + 1]);
    p[0] = narrow<TX>(diff_of_products(x0, c0, x1, s0));
    p[1] = narrow<TX>(diff_of_products(x1, c1, -x0, s1));
  }
}

bool aligned(const void* p, int64_t bytes) { return (reinterpret_cast<uintptr_t>(p) % bytes) == 0; }

template <typename TX, typename TC, int VEC, bool PER_HEAD_CS>
cudaError_t launch_vec_kernel(const InplaceProblem& p, cudaStream_t stream) {
  InplaceArgs a;
  a.S = p.S;
  a.N = p.N;
  a.D = p.D;
  a.start = p.start;
  a.L = p.L;
  a.cs_b = p.cs_b;
  a.cs_s = p.cs_s;
  a.cs_n = p.cs_n;
  a.chunks = (int32_t)(p.L / VEC);
  a.head_chunks = (int32_t)((p.N + kRowsInFlight - 1) / kRowsInFlight);
  a.items = p.B * p.S * a.head_chunks;
  // a row group needs C threads: the block has at least kThreads and at least C
  const int threads = a.chunks > kThreads ? a.chunks : kThreads;
  const int64_t groups = threads / a.chunks;
  // Persistent grid: the CTAs that fit on the GPU at once stride over the items,
  // P consecutive items per CTA per step.
  auto kernel = inplace_vec_kernel<TX, TC, VEC, PER_HEAD_CS>;
  const int64_t resident = (int64_t)sm_count() * resident_blocks(reinterpret_cast<const void*>(kernel), threads);
  const int64_t grid = std::max<int64_t>(1, std::min((a.items + groups - 1) / groups, resident));
  return launch_overlapped(kernel, (unsigned)grid, threads, stream, static_cast<TX*>(p.x),
                           static_cast<const TC*>(p.cos), static_cast<const TC*>(p.sin), a);
}

template <typename TX, typename TC, int VEC>
cudaError_t launch_vec(const InplaceProblem& p, cudaStream_t stream) {
  return p.cs_n == 0 ? launch_vec_kernel<TX, TC, VEC, false>(p, stream)
                     : launch_vec_kernel<TX, TC, VEC, true>(p, stream);
}

template <typename TX, typename TC>
cudaError_t launch_pairs(const InplaceProblem& p, cudaStream_t stream) {
  InplaceArgs a{};
  a.S = p.S;
  a.N = p.N;
  a.D = p.D;
  a.start = p.start;
  a.L = p.L;
  a.cs_b = p.cs_b;
  a.cs_s = p.cs_s;
  a.cs_n = p.cs_n;
  const int64_t rows = p.B * p.S * p.N;
  const int64_t total = rows * (p.L / 2);
  const int64_t blocks = std::min<int64_t>((total + 255) / 256, (int64_t)sm_count() * 8);
  return launch_overlapped(inplace_pair_kernel<TX, TC>, (unsigned)std::max<int64_t>(1, blocks), 256, stream,
                           static_cast<TX*>(p.x), static_cast<const TC*>(p.cos), static_cast<const TC*>(p.sin), a,
                           rows);
}

// Widest vector (in elements of TX) that the slice, the row pitch and the
// base pointers all allow; 0 when pairs cannot be kept inside one vector.
template <typename TX, typename TC>
int pick_vec(const InplaceProblem& p) {
  const int max_vec = 16 / (int)sizeof(TX);
  for (int v = max_vec; v >= 2; v /= 2) {
    if (p.start % v || p.L % v || p.D % v) continue;
    if (!aligned(p.x, v * (int64_t)sizeof(TX))) continue;
    const int64_t cbytes = std::min<int64_t>(16, v * (int64_t)sizeof(TC));
    if (!aligned(p.cos, cbytes) || !aligned(p.sin, cbytes)) continue;
    return v;
  }
  return 0;
}

template <typename TX, typename TC>
cudaError_t dispatch(const InplaceProblem& p, cudaStream_t stream) {
  switch (pick_vec<TX, TC>(p)) {
    case 8:
      if constexpr (sizeof(TX) == 2) return launch_vec<TX, TC, 8>(p, stream);
      break;
    case 4:
      return launch_vec<TX, TC, 4>(p, stream);
    case 2:
      return launch_vec<TX, TC, 2>(p, stream);
    default:
      break;
  }
  return launch_pairs<TX, TC>(p, stream);
}

}  // namespace

cudaError_t launch_inplace(const InplaceProblem& p, cudaStream_t stream) {
  const bool f32cs = p.cs_dtype == kF32;
  switch (p.x_dtype) {
    case kF32:
      return dispatch<float, float>(p, stream);
    case kF16:
      return f32cs ? dispatch<__half, float>(p, stream) : dispatch<__half, __half>(p, stream);
    case kBF16:
      return f32cs ? dispatch<__nv_bfloat16, float>(p, stream)
                   : dispatch<__nv_bfloat16, __nv_bfloat16>(p, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace rope
