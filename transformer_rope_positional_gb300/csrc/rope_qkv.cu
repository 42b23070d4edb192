// Fused QKV split + RMSNorm + RoPE + paged KV-cache write.
//
// Operator: the "aclnnQkvRmsNormRopeCacheWithKScale" page, section 计算公式,
// without its FP8 quantisation and its optional rotation matmul:
//   q, k, v = split(qkv, [Nq, Nk, Nv])                         (heads of D)
//   y = x / sqrt(mean(x^2) + eps) * gamma                      (q and k heads)
//   position = seqLens[b] - (qsl[b+1] - qsl[b]) + i            (token i of batch b)
//   y_rope = concat(y_low*cos - y_high*sin, y_high*cos + y_low*sin)
//   q_out[t, h] = y_rope;  kCache[slot/BS, h, slot%BS] = y_rope;  vCache[...] = v
// cos/sin are the halves of row `position` of a [maxSeq, D] cos||sin table.
//
// GB300 design.  Same streaming structure as the other kernels: items of U
// consecutive heads of one token, row groups of C threads (thread c owns the
// c-th 16-byte chunk of both halves of a head, the NeoX pairing), persistent
// grid striding over items.  The RMSNorm reduction is a sum of the thread's
// 2*VEC squares followed by a butterfly of warp shuffles inside the row group
// (groups are padded to a power of two lanes), so a head never leaves
// registers: one read of qkv, one write of q_out or of the cache slot.  The
// per-token metadata (batch by binary search over queryStartLoc, position,
// slot) is computed once per item, searching a shared-memory copy of
// queryStartLoc.  Positions outside the table and slots past
// the pool set bits of the device error word and skip the writes.
#include <algorithm>

#include "rope_device.cuh"
#include "rope_launch.h"

namespace rope {
namespace {

#ifndef ROPE_QKV_ROWS_IN_FLIGHT
#define ROPE_QKV_ROWS_IN_FLIGHT 4
#endif
#ifndef ROPE_QKV_THREADS
#define ROPE_QKV_THREADS 128
#endif
constexpr int kRowsInFlight = ROPE_QKV_ROWS_IN_FLIGHT;
constexpr int kThreads = ROPE_QKV_THREADS;
constexpr unsigned kPositionOutOfRange = 1u;
constexpr unsigned kSlotOutOfRange = 2u;
constexpr int64_t kSharedQsl = 4096;  // queryStartLoc entries kept in shared memory (32 KB)

struct QkvArgs {
  int64_t T, B;
  int64_t max_seq;
  int64_t W;          // qkv row width, (nq + nk + nv) * D
  int64_t num_slots;  // num_blocks * block_size
  int64_t items;      // T * head_chunks
  int32_t nq, nk, nv;
  int32_t D;
  int32_t block_size;
  int32_t chunks;       // C: active threads per head row
  int32_t group;        // C rounded up to a power of two (lanes per row group)
  int32_t head_chunks;  // ceil(H / U)
  float eps;
  float inv_d;
  bool items32;  // items and slots fit 32-bit index arithmetic
};

template <typename T, int VEC>
__global__ void __launch_bounds__(kThreads)
    qkv_kernel(const T* __restrict__ qkv, const T* __restrict__ q_gamma, const T* __restrict__ k_gamma,
               const T* __restrict__ cache, const int64_t* __restrict__ seq_lens, const int64_t* __restrict__ qsl,
               const int64_t* __restrict__ slot_mapping, T* __restrict__ q_out, T* __restrict__ k_cache,
               T* __restrict__ v_cache, unsigned int* __restrict__ err, QkvArgs a) {
  constexpr int U = kRowsInFlight;
  const int G = a.group;
  const int P = blockDim.x / G;  // row groups per CTA
  const int g = threadIdx.x / G;
  const int c = threadIdx.x - g * G;
  const bool active = c < a.chunks;  // padding lanes only join the reduction
  const int lane = threadIdx.x & 31;
  const unsigned gmask = (G >= 32 ? 0xffffffffu : ((1u << G) - 1u)) << (lane & ~(G - 1));
  const int half = a.D / 2;
  const int i0 = (active ? c : 0) * VEC;
  const int H = a.nq + a.nk + a.nv;
  wait_for_prior_grid();

  // queryStartLoc in shared memory for the batch lookup when it fits
  extern __shared__ int64_t s_qsl[];
  const bool qsl_shared = a.B + 1 <= kSharedQsl;
  if (qsl_shared) {
    for (int64_t i = threadIdx.x; i <= a.B; i += blockDim.x) s_qsl[i] = __ldg(qsl + i);
    __syncthreads();
  }

  for (int64_t item = (int64_t)blockIdx.x * P + g; item < a.items; item += (int64_t)gridDim.x * P) {
    const int64_t t = div_index(item, a.head_chunks, a.items32);
    const int h0 = (int)(item - t * a.head_chunks) * U;
    const int n = min(U, H - h0);
    // ---- issue the loads of the item's head rows
    Vec<T, VEC> x1[U], x2[U];
    const T* src = qkv + t * a.W + (int64_t)h0 * a.D;
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (u < n && active) {
        load_vec<true>(x1[u], src + u * a.D + i0);
        load_vec<true>(x2[u], src + u * a.D + half + i0);
      }
    // ---- token metadata: batch (largest b with qsl[b] <= t), position, slot
    int64_t lo = 0, hi = a.B - 1;
    while (lo < hi) {
      const int64_t mid = (lo + hi + 1) / 2;
      if ((qsl_shared ? s_qsl[mid] : __ldg(qsl + mid)) <= t) lo = mid; else hi = mid - 1;
    }
    const int64_t start = qsl_shared ? s_qsl[lo] : __ldg(qsl + lo);
    const int64_t qlen = (qsl_shared ? s_qsl[lo + 1] : __ldg(qsl + lo + 1)) - start;
    const int64_t position = __ldg(seq_lens + lo) - qlen + (t - start);
    const int64_t slot = __ldg(slot_mapping + t);
    const bool pos_ok = position >= 0 && position < a.max_seq;
    const bool cache_it = slot >= 0 && slot < a.num_slots;
    if (c == 0 && h0 == 0) {  // reported once per token
      if (!pos_ok) atomicOr(err, kPositionOutOfRange);
      else if (slot >= a.num_slots) atomicOr(err, kSlotOutOfRange);
    }
    if (!pos_ok) continue;  // nothing of this token is written
    Vec<T, VEC> cv, sv;  // kept in the storage type; widened at each use
    load_vec<false>(cv, cache + position * a.D + i0);
    load_vec<false>(sv, cache + position * a.D + half + i0);
    const int64_t blk = cache_it ? div_index(slot, a.block_size, a.items32) : 0;
    const int64_t off = cache_it ? slot - blk * a.block_size : 0;

    // ---- RMSNorm: squares of every q/k row of the item (independent chains),
    // then butterflies inside the row group, interleaved across the rows
    float ss[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float2 acc = make_float2(0.f, 0.f);
      if (u < n && h0 + u < a.nq + a.nk && active) {
#pragma unroll
        for (int j = 0; j < VEC; j += 2) {
          const float2 v1 = widen2(&x1[u].e[j]), v2 = widen2(&x2[u].e[j]);
          acc = __ffma2_rn(v1, v1, acc);
          acc = __ffma2_rn(v2, v2, acc);
        }
      }
      ss[u] = acc.x + acc.y;
    }
    for (int m = G / 2; m > 0; m /= 2)
#pragma unroll
      for (int u = 0; u < U; ++u) ss[u] += __shfl_xor_sync(gmask, ss[u], m, G);
    if (!active) continue;

#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (u >= n) break;
      const int h = h0 + u;
      if (h >= a.nq + a.nk) {  // V: stored as is
        if (cache_it) {
          T* dst = v_cache + ((blk * a.nv + (h - a.nq - a.nk)) * a.block_size + off) * a.D;
          store_vec(dst + i0, x1[u]);
          store_vec(dst + half + i0, x2[u]);
        }
        continue;
      }
      const bool is_q = h < a.nq;
      T* dst = is_q ? q_out + (t * a.nq + h) * (int64_t)a.D
                    : (cache_it ? k_cache + ((blk * a.nk + (h - a.nq)) * a.block_size + off) * a.D : nullptr);
      if (dst == nullptr) continue;
      const float inv = rsqrtf(__fmaf_rn(ss[u], a.inv_d, a.eps));
      const float2 inv2 = make_float2(inv, inv);
      // gamma of this thread's elements (L1-resident, reloaded per row to save registers)
      const T* gamma = is_q ? q_gamma : k_gamma;
      Vec<T, VEC> g1, g2;
      load_vec<false>(g1, gamma + i0);
      load_vec<false>(g2, gamma + half + i0);
#pragma unroll
      for (int j = 0; j < VEC; j += 2) {
        const float2 y1 = __fmul2_rn(__fmul2_rn(widen2(&x1[u].e[j]), inv2), widen2(&g1.e[j]));
        const float2 y2 = __fmul2_rn(__fmul2_rn(widen2(&x2[u].e[j]), inv2), widen2(&g2.e[j]));
        const float2 cs = widen2(&cv.e[j]), sn = widen2(&sv.e[j]);
        // y1, y2 already carry binary32 rounding from the normalisation, so a
        // plain FMA pair is as accurate here as the compensated form
        const float2 t2 = __fmul2_rn(y2, sn), t1 = __fmul2_rn(y1, sn);
        narrow2(&x1[u].e[j], __ffma2_rn(y1, cs, make_float2(-t2.x, -t2.y)));
        narrow2(&x2[u].e[j], __ffma2_rn(y2, cs, t1));
      }
      store_vec(dst + i0, x1[u]);
      store_vec(dst + half + i0, x2[u]);
    }
  }
}

template <typename T>
cudaError_t launch_typed(const QkvProblem& p, cudaStream_t stream) {
  constexpr int VEC = 16 / sizeof(T);
  QkvArgs a;
  a.T = p.T;
  a.B = p.B;
  a.max_seq = p.max_seq;
  a.nq = (int32_t)p.nq;
  a.nk = (int32_t)p.nk;
  a.nv = (int32_t)p.nv;
  a.D = (int32_t)p.D;
  a.W = (p.nq + p.nk + p.nv) * p.D;
  a.block_size = (int32_t)p.block_size;
  a.num_slots = p.num_blocks * p.block_size;
  a.chunks = (int32_t)(p.D / 2 / VEC);
  a.group = 1;
  while (a.group < a.chunks) a.group *= 2;
  a.head_chunks = (int32_t)((p.nq + p.nk + p.nv + kRowsInFlight - 1) / kRowsInFlight);
  a.items = p.T * a.head_chunks;
  a.eps = p.eps;
  a.inv_d = 1.0f / (float)p.D;
  a.items32 = a.items <= 0xffffffffLL && a.num_slots <= 0xffffffffLL;
  const int64_t groups = kThreads / a.group;
  auto kernel = qkv_kernel<T, VEC>;
  // occupancy with the largest shared-memory request the kernel can make
  const int64_t resident = (int64_t)sm_count() * resident_blocks(reinterpret_cast<const void*>(kernel), kThreads,
                                                                 kSharedQsl * sizeof(int64_t));
  const int64_t grid = std::max<int64_t>(1, std::min((a.items + groups - 1) / groups, resident));
  unsigned int* err = nullptr;
  const cudaError_t e = device_error_address(&err);
  if (e != cudaSuccess) return e;
  const size_t smem = p.B + 1 <= kSharedQsl ? (size_t)(p.B + 1) * sizeof(int64_t) : 0;
  return launch_overlapped_smem(kernel, (unsigned)grid, kThreads, smem, stream, static_cast<const T*>(p.qkv),
                           static_cast<const T*>(p.q_gamma), static_cast<const T*>(p.k_gamma),
                           static_cast<const T*>(p.cache), p.seq_lens, p.query_start_loc, p.slot_mapping,
                           static_cast<T*>(p.q_out), static_cast<T*>(p.k_cache), static_cast<T*>(p.v_cache), err,
                           a);
}

}  // namespace

cudaError_t launch_qkv(const QkvProblem& p, cudaStream_t stream) {
  switch (p.dtype) {
    case kF32:
      return launch_typed<float>(p, stream);
    case kF16:
      return launch_typed<__half>(p, stream);
    case kBF16:
      return launch_typed<__nv_bfloat16>(p, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace rope
