// Cache-indexed RoPE of query and key (rope and mrope modes, GPT-NeoX and GPT-J).
//
// Operator: "CANN ops-transformer 旋转位置编码算子 RopeWithSinCosCache 深度解析：
// cache 化 RoPE 的计算原理与 aclnn 两段式调用实战", sections 设计动机 (gather,
// chunk, rotate), mrope 模式, rope 模式, rotate_half（GPT-NeoX style） and
// rotate_interleaved（GPT-J style）.
//
// GB300 design.  Token-major teams, as in the in-place kernel: a team owns one
// token and a block of its heads (query heads first, then key heads); thread c
// owns one 16-byte chunk of cos and the matching chunk of sin.  The gather of
// the cache row (mrope: the section's row for each owned index) happens once
// per team, into registers, and serves every head of the block.  NeoX pairs
// element i with i + R/2, so a thread loads the same chunk of both halves;
// GPT-J pairs neighbours, so a thread loads one chunk holding VEC/2 pairs.
// query/key are read and written once (streaming); the cache goes through the
// read-only path and stays in L2 for later tokens at nearby positions.
// Columns [R, head_size) of every head are never touched.
//
// A position outside [0, maxSeqLen) leaves its token untouched and sets bit
// ROPE_DEVICE_POSITION_OUT_OF_RANGE of the device error word below.
#include <algorithm>

#include "rope_device.cuh"
#include "rope_launch.h"

namespace rope {

// Device-side error word (one per device context), read and cleared by
// read_and_clear_device_error().
__device__ unsigned int g_device_error;

namespace {

constexpr int kHeadsInFlight = 4;  // U: heads loaded before compute, per thread
constexpr unsigned kPositionOutOfRange = 1u;

struct CacheArgs {
  int64_t T;
  int64_t max_seq;
  int64_t items;  // T * head_blocks
  int32_t hq, hk;
  int32_t head_size;
  int32_t R;
  int32_t chunks;  // threads per team
  int32_t heads_per_item;
  int32_t head_blocks;
  int32_t mrope_rows;
  int32_t section_end[4];
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

template <typename T, bool NEOX, int VEC>
__global__ void __launch_bounds__(256) cache_kernel(const int64_t* __restrict__ pos, T* __restrict__ q,
                                                    T* __restrict__ k, const T* __restrict__ cache,
                                                    CacheArgs a) {
  constexpr int U = kHeadsInFlight;
  constexpr int NC = NEOX ? VEC : VEC / 2;  // cos (and sin) indices owned per thread
  const int team_size = a.chunks;
  const int teams = blockDim.x / team_size;
  const int team = threadIdx.x / team_size;
  if (team >= teams) return;
  const int c = threadIdx.x - team * team_size;
  const int half = a.R / 2;
  const int i0 = c * NC;  // first owned cos index
  const int64_t team_stride = (int64_t)gridDim.x * teams;

  for (int64_t item = (int64_t)blockIdx.x * teams + team; item < a.items; item += team_stride) {
    const int64_t t = item / a.head_blocks;
    const int hb = (int)(item - t * a.head_blocks);

    // ---- steps 1-2: gather cosSin = cache[positions] and split into cos / sin
    float cf[NC], sf[NC];
    bool ok = true;
    if (a.mrope_rows == 0) {
      const int64_t p = __ldg(pos + t);
      ok = p >= 0 && p < a.max_seq;
      if (ok) {
        const T* rowp = cache + p * a.R;
        load_f32<T, NC>(cf, rowp + i0);
        load_f32<T, NC>(sf, rowp + half + i0);
      }
    } else {
      const int64_t p0 = __ldg(pos + t);
      const int64_t p1 = __ldg(pos + a.T + t);
      const int64_t p2 = __ldg(pos + 2 * a.T + t);
      const int64_t p3 = a.mrope_rows > 3 ? __ldg(pos + 3 * a.T + t) : 0;
      ok = p0 >= 0 && p0 < a.max_seq && p1 >= 0 && p1 < a.max_seq && p2 >= 0 && p2 < a.max_seq &&
           p3 >= 0 && p3 < a.max_seq;
      if (ok) {
        const int k0 = section_of(i0, a);
        const int k1 = section_of(i0 + NC - 1, a);
        if (k0 == k1) {  // the whole chunk sits in one section: one vector per half
          const T* rowp = cache + select_row(k0, p0, p1, p2, p3) * a.R;
          load_f32<T, NC>(cf, rowp + i0);
          load_f32<T, NC>(sf, rowp + half + i0);
        } else {  // chunk straddles a section boundary: per-element rows
#pragma unroll
          for (int e = 0; e < NC; ++e) {
            const T* rowp = cache + select_row(section_of(i0 + e, a), p0, p1, p2, p3) * a.R;
            cf[e] = widen(__ldg(rowp + i0 + e));
            sf[e] = widen(__ldg(rowp + half + i0 + e));
          }
        }
      }
    }
    if (!ok) {
      if (c == 0 && hb == 0) atomicOr(&g_device_error, kPositionOutOfRange);
      continue;
    }

    // ---- step 3: rotate the first R columns of every head of the block
    const int h0 = hb * a.heads_per_item;
    const int h1 = min(h0 + a.heads_per_item, a.hq + a.hk);
    for (int h = h0; h < h1; h += U) {
      T* base[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int hh = h + u < h1 ? h + u : h;
        base[u] = hh < a.hq ? q + (t * a.hq + hh) * (int64_t)a.head_size
                            : k + (t * a.hk + (hh - a.hq)) * (int64_t)a.head_size;
      }
      if constexpr (NEOX) {
        Vec<T, VEC> x1[U], x2[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (h + u < h1) {
            load_vec<true>(x1[u], base[u] + i0);
            load_vec<true>(x2[u], base[u] + half + i0);
          }
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (h + u < h1) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
              const float a1 = widen(x1[u].e[e]);
              const float a2 = widen(x2[u].e[e]);
              x1[u].e[e] = narrow<T>(diff_of_products(a1, cf[e], a2, sf[e]));
              x2[u].e[e] = narrow<T>(diff_of_products(a2, cf[e], -a1, sf[e]));
            }
            store_vec(base[u] + i0, x1[u]);
            store_vec(base[u] + half + i0, x2[u]);
          }
      } else {
        Vec<T, VEC> xv[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (h + u < h1) load_vec<true>(xv[u], base[u] + 2 * i0);
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (h + u < h1) {
#pragma unroll
            for (int e = 0; e < NC; ++e) {
              const float a1 = widen(xv[u].e[2 * e]);
              const float a2 = widen(xv[u].e[2 * e + 1]);
              xv[u].e[2 * e] = narrow<T>(diff_of_products(a1, cf[e], a2, sf[e]));
              xv[u].e[2 * e + 1] = narrow<T>(diff_of_products(a2, cf[e], -a1, sf[e]));
            }
            store_vec(base[u] + 2 * i0, xv[u]);
          }
      }
    }
  }
}

template <typename T, bool NEOX>
cudaError_t launch_typed(const CacheProblem& p, cudaStream_t stream) {
  constexpr int VEC = 16 / sizeof(T);
  CacheArgs a;
  a.T = p.T;
  a.max_seq = p.max_seq;
  a.hq = (int32_t)p.hq;
  a.hk = (int32_t)p.hk;
  a.head_size = (int32_t)p.head_size;
  a.R = (int32_t)p.rotary_dim;
  a.chunks = (int32_t)cache_team_threads(p);
  a.mrope_rows = p.mrope_rows;
  // ends past the used sections are R/2, so section_of() never counts them
  for (int i = 0; i < 4; ++i) a.section_end[i] = i < p.mrope_rows ? p.section_end[i] : (int32_t)(p.rotary_dim / 2);
  const int threads = a.chunks > 256 ? a.chunks : 256;
  const int teams = threads / a.chunks;
  const int64_t heads = p.hq + p.hk;
  const int64_t sms = sm_count();
  const int64_t want_threads = sms * 1024;
  const int64_t base_threads = p.T * a.chunks;
  int64_t nb = (want_threads + base_threads - 1) / base_threads;
  nb = std::max<int64_t>(1, std::min<int64_t>(nb, heads));
  a.heads_per_item = (int32_t)((heads + nb - 1) / nb);
  a.head_blocks = (int32_t)((heads + a.heads_per_item - 1) / a.heads_per_item);
  a.items = p.T * a.head_blocks;
  const int64_t ctas_needed = (a.items + teams - 1) / teams;
  const int64_t ctas_resident = sms * std::max(1, 2048 / threads);
  const unsigned grid = (unsigned)std::max<int64_t>(1, std::min(ctas_needed, ctas_resident));
  cache_kernel<T, NEOX, VEC><<<grid, threads, 0, stream>>>(p.positions, static_cast<T*>(p.query),
                                                           static_cast<T*>(p.key),
                                                           static_cast<const T*>(p.cache), a);
  count_launch();
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_style(const CacheProblem& p, cudaStream_t stream) {
  return p.is_neox ? launch_typed<T, true>(p, stream) : launch_typed<T, false>(p, stream);
}

}  // namespace

int64_t cache_team_threads(const CacheProblem& p) {
  const int64_t vec = 16 / (p.dtype == kF32 ? 4 : 2);
  return p.is_neox ? (p.rotary_dim / 2) / vec : p.rotary_dim / vec;
}

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

cudaError_t read_and_clear_device_error(cudaStream_t stream, uint32_t* code) {
  unsigned int host = 0;
  const unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&host, g_device_error, sizeof(host), 0,
                                            cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess)
    e = cudaMemcpyToSymbolAsync(g_device_error, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  *code = host;
  return e;
}

}  // namespace rope
