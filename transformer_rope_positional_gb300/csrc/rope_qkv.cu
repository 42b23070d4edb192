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
// GB300 design.  Same streaming structure as the other kernels: items of up
// to U consecutive heads of one token, row groups of C threads (thread c owns
// the c-th 16-byte chunk of both halves of a head, the NeoX pairing),
// persistent grid striding over items.  Items never mix q, k and v heads (a
// token has ceil(Nq/U) q items, then ceil(Nk/U) k items, then ceil(Nv/U) v
// items), so one item has one gamma and one destination layout.
//
//  * RMSNorm: each thread sums the squares of its 2*VEC elements, then a
//    butterfly of warp shuffles inside the row group (padded to a power of two
//    lanes) completes the head's sum.
//  * Head rows through shared memory: each thread copies its 16-byte chunks of
//    the NEXT item's rows into shared-memory slots of its own with cp.async
//    (cached in L2 only, evict-first) before it works on the current item,
//    whose rows arrived meanwhile, so a whole item of reads stays in flight
//    while the thread computes; no barrier is needed, since a thread reads
//    back only its own slots.  Two buffers measured best (35.9 -> 34.9 us on
//    the mixed prefill/decode batch); three or four buffers, reading the rows
//    from shared memory again for the rotation, and 5 CTAs per SM (which
//    spills) were slower.
//  * RoPE with the norm folded in: per item, thread c forms the products
//    gamma_low*cos, -gamma_high*sin, gamma_high*cos, gamma_low*sin of its
//    elements once, so each output element costs one product, one FMA and
//    the scaling by 1/rms:  out_low = (x_low*(g_low*cos) - x_high*(g_high*sin)) / rms.
//  * Token metadata (batch by search in queryStartLoc, position, slot) for
//    the NEXT item is computed while the current item's loads are in flight,
//    so the search and the dependent loads leave the critical path.  With few
//    enough sequences, queryStartLoc and seqLens[b] - queryStartLoc[b+1] sit in
//    shared memory (position = t + that difference), and the search starts
//    from the previous item's batch (a group's tokens only increase).
//
// Positions outside the table and slots past the pool set bits of the device
// error word and skip the writes.
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
// 4 CTAs per SM caps the kernel at 128 registers per thread without spills;
// measured faster than both the uncapped build (3 CTAs) and 5 CTAs with spills.
#ifndef ROPE_QKV_MIN_BLOCKS
#define ROPE_QKV_MIN_BLOCKS 4
#endif
// Row buffers per thread: the current item plus ROPE_QKV_STAGES - 1 items
// whose rows are being copied (2 measured best: 3 and 4 were slower).
#ifndef ROPE_QKV_STAGES
#define ROPE_QKV_STAGES 2
#endif
constexpr int kRowsInFlight = ROPE_QKV_ROWS_IN_FLIGHT;
constexpr int kStages = ROPE_QKV_STAGES;

static_assert(kStages >= 2, "at least one item in flight");
constexpr int kThreads = ROPE_QKV_THREADS;
constexpr unsigned kPositionOutOfRange = 1u;
constexpr unsigned kSlotOutOfRange = 2u;
constexpr int64_t kSharedTable = 4096;  // int64 entries of the shared batch tables (32 KB)
// Row stages: [kStages buffers][U rows][2 halves][kThreads] 16-byte slots.
constexpr size_t kStageBytes = size_t(kStages) * kRowsInFlight * 2 * kThreads * 16;

struct QkvArgs {
  int64_t T, B;
  int64_t max_seq;
  int64_t W;          // qkv row width, (nq + nk + nv) * D
  int64_t num_slots;  // num_blocks * block_size
  int64_t items;      // T * per_token
  int32_t nq, nk, nv;
  int32_t iq, ik;       // q items and k items per token
  int32_t per_token;    // items per token, iq + ik + ceil(nv / U)
  int32_t D;
  int32_t block_size;
  int32_t chunks;       // C: active threads per head row
  int32_t group;        // C rounded up to a power of two (lanes per row group)
  float eps;
  float inv_d;
  int64_t stride_t;     // a row group's step of grid * groups items: whole tokens
  int32_t stride_r;     // and items left over (< per_token)
  int32_t bs_shift;     // log2(block_size) when it is a power of two, else -1
  bool items32;  // items and slots fit 32-bit index arithmetic
  // byte spans of the tensors (checked in debug builds)
  Span qkv_span, qg_span, kg_span, cache_span, sl_span, qsl_span, slot_span, qo_span, kc_span, vc_span, tab_span;
};

// Token metadata of one item.
struct ItemMeta {
  int64_t t;         // token
  int64_t position;  // row of the cos/sin table
  int64_t slot;      // slot_mapping[t]
  int32_t r;         // item index within the token
  int32_t b;         // batch of the token
};

// Batch of token t: the largest b in [0, B) with queryStartLoc[b] <= t.  `lo`
// is a batch with queryStartLoc[lo] <= t (the previous answer for a smaller
// or equal token, or 0): the common case is one comparison.  `qsl` is the
// global tensor or its copy in shared memory, spanned by `span`.
__device__ __forceinline__ int find_batch(const int64_t* __restrict__ qsl, int B, int64_t t, int lo, const Span& span,
                                          unsigned int* err) {
  auto at = [&](int i) -> int64_t { return access_ok(qsl + i, 8, span, err) ? qsl[i] : 0; };
  if (lo + 1 < B && at(lo + 1) <= t) {
    int l = lo + 1, h = B - 1;
    while (l < h) {
      const int mid = (l + h + 1) >> 1;
      if (at(mid) <= t) l = mid; else h = mid - 1;
    }
    lo = l;
  }
  return lo;
}

// The heads of item index r within its token: kind 0 q, 1 k, 2 v; h0 the
// first head within the kind, n heads, hg the first head within the qkv row.
struct ItemHeads {
  int kind, h0, n, hg;
};

__device__ __forceinline__ ItemHeads item_heads(int r, const QkvArgs& a) {
  constexpr int U = kRowsInFlight;
  ItemHeads h;
  int nh;
  if (r < a.iq) {
    h.kind = 0, h.h0 = r * U, nh = a.nq, h.hg = h.h0;
  } else if (r < a.iq + a.ik) {
    h.kind = 1, h.h0 = (r - a.iq) * U, nh = a.nk, h.hg = a.nq + h.h0;
  } else {
    h.kind = 2, h.h0 = (r - a.iq - a.ik) * U, nh = a.nv, h.hg = a.nq + a.nk + h.h0;
  }
  h.n = min(U, nh - h.h0);
  return h;
}

// Item index as (token, item within the token), stepped by the grid stride
// without a division.
struct TokenItem {
  int64_t t;
  int32_t r;
};

__device__ __forceinline__ void advance(TokenItem& ti, const QkvArgs& a) {
  ti.t += a.stride_t;
  ti.r += a.stride_r;
  if (ti.r >= a.per_token) ti.r -= a.per_token, ++ti.t;
}

template <bool SHARED>
__device__ __forceinline__ ItemMeta item_meta(TokenItem ti, const QkvArgs& a, const int64_t* __restrict__ tab,
                                              const int64_t* __restrict__ qsl, const int64_t* __restrict__ seq_lens,
                                              const int64_t* __restrict__ slot_mapping, int cursor,
                                              unsigned int* err) {
  ItemMeta m;
  m.t = ti.t;
  m.r = ti.r;
  m.slot = ldg(slot_mapping + m.t, a.slot_span, err);
  if (SHARED) {
    m.b = find_batch(tab, (int)a.B, m.t, cursor, a.tab_span, err);
    const int64_t* d = tab + a.B + 1 + m.b;
    m.position = m.t + (access_ok(d, 8, a.tab_span, err) ? *d : 0);
  } else {
    m.b = find_batch(qsl, (int)a.B, m.t, cursor, a.qsl_span, err);
    m.position = ldg(seq_lens + m.b, a.sl_span, err) - ldg(qsl + m.b + 1, a.qsl_span, err) + m.t;
  }
  return m;
}

template <typename T, int VEC, bool SHARED>
__global__ void __launch_bounds__(kThreads, ROPE_QKV_MIN_BLOCKS)
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
  wait_for_prior_grid();

  extern __shared__ __align__(16) unsigned char s_raw[];
  // row stages, then [0, B]: queryStartLoc; [B + 1, 2B]: seqLens[b] - queryStartLoc[b + 1]
  uint4* const s_stage = reinterpret_cast<uint4*>(s_raw);
  int64_t* const s_tab = reinterpret_cast<int64_t*>(s_raw + kStageBytes);
  auto slot = [&](int buf, int u, int v) { return s_stage + ((buf * U + u) * 2 + v) * kThreads + threadIdx.x; };
  const uint64_t policy = l2_evict_first_policy();
  // copies of item `it`'s head rows into buffer `buf`, as one commit group
  auto copy_rows = [&](const TokenItem& it, int buf) {
    if (active) {
      const ItemHeads hd = item_heads(it.r, a);
      const T* src = qkv + it.t * a.W + (int64_t)hd.hg * a.D + i0;
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (u < hd.n) {
          cp_async16(slot(buf, u, 0), src + u * a.D, policy, a.qkv_span, err);
          cp_async16(slot(buf, u, 1), src + u * a.D + half, policy, a.qkv_span, err);
        }
    }
    cp_async_commit();
  };

  // items in token order: item i is (token i / per_token, item i % per_token
  // within it); a row group steps by the grid's groups, in (token, item) form
  const int64_t item0 = (int64_t)blockIdx.x * P + g;
  int buf = 0;  // buffer of the current item; the j-th item after it goes to (buf + j) % kStages
  TokenItem tc;  // the current item (tc.t < T while there is one)
  tc.t = div_index(item0, a.per_token, a.items32);
  tc.r = (int32_t)(item0 - tc.t * a.per_token);
  TokenItem ta = tc;  // the item whose rows are copied next
  // the first items' rows are copied before the tables are built: they need no metadata
#pragma unroll
  for (int j = 0; j < kStages - 1; ++j) {
    if (ta.t < a.T) copy_rows(ta, j);
    else cp_async_commit();
    advance(ta, a);
  }

#ifdef ROPE_DEBUG_BOUNDS
  a.tab_span.lo = reinterpret_cast<const char*>(s_tab);
  a.tab_span.hi = reinterpret_cast<const char*>(s_tab + (SHARED ? 2 * a.B + 1 : 0));
#endif
  if (SHARED) {
    for (int64_t i = threadIdx.x; i <= a.B; i += blockDim.x) s_tab[i] = ldg(qsl + i, a.qsl_span, err);
    for (int64_t i = threadIdx.x; i < a.B; i += blockDim.x)
      s_tab[a.B + 1 + i] = ldg(seq_lens + i, a.sl_span, err) - ldg(qsl + i + 1, a.qsl_span, err);
    __syncthreads();
  }

  if (tc.t >= a.T) return;
  ItemMeta m = item_meta<SHARED>(tc, a, s_tab, qsl, seq_lens, slot_mapping, 0, err);
  for (;;) {  // m: the current item's metadata, m.t < T
    TokenItem tn = {m.t, m.r};  // the next item
    advance(tn, a);
    {
      const int abuf = buf == 0 ? kStages - 1 : buf - 1;  // (buf + kStages - 1) % kStages
      if (kStages == 2) ta = tn;  // the item kStages - 1 ahead is the next one
      if (ta.t < a.T) copy_rows(ta, abuf);
      else cp_async_commit();  // one group per item keeps the wait count fixed
      if (kStages > 2) advance(ta, a);
    }
    // ---- this item's heads: kind 0 q, 1 k, 2 v; h0 within the kind
    const ItemHeads hd = item_heads(m.r, a);
    const int kind = hd.kind, h0 = hd.h0, n = hd.n;
    const bool pos_ok = m.position >= 0 && m.position < a.max_seq;
    const bool cache_it = m.slot >= 0 && m.slot < a.num_slots;
    const bool work = pos_ok && (kind == 0 || cache_it);  // uniform over the row group
    const bool rotate = kind < 2;
    // ---- issue the loads: head rows, then cos/sin and gamma
    Vec<T, VEC> x1[U], x2[U];
    Vec<T, VEC> cv, sv, g1, g2;
    if (work && active) {
      if (rotate) {
        const T* cs = cache + m.position * a.D + i0;
        load_vec<false>(cv, cs, a.cache_span, err);
        load_vec<false>(sv, cs + half, a.cache_span, err);
        const T* gamma = (kind == 0 ? q_gamma : k_gamma) + i0;
        const Span& gs = kind == 0 ? a.qg_span : a.kg_span;
        load_vec<false>(g1, gamma, gs, err);
        load_vec<false>(g2, gamma + half, gs, err);
      }
    }
    if (c == 0 && m.r == 0) {  // reported once per token
      if (!pos_ok) atomicOr(err, kPositionOutOfRange);
      else if (m.slot >= a.num_slots) atomicOr(err, kSlotOutOfRange);
    }
    // destination of head h0 and the distance between consecutive heads
    T* dst = nullptr;
    int64_t dstride = a.D;
    const Span* dspan = kind == 0 ? &a.qo_span : kind == 1 ? &a.kc_span : &a.vc_span;
    if (kind == 0) {
      dst = q_out + (m.t * a.nq + h0) * (int64_t)a.D;
    } else if (cache_it) {
      const int64_t blk = a.bs_shift >= 0 ? m.slot >> a.bs_shift : div_index(m.slot, a.block_size, a.items32);
      const int64_t off = m.slot - blk * a.block_size;
      dst = (kind == 1 ? k_cache + ((blk * a.nk + h0) * a.block_size + off) * a.D
                       : v_cache + ((blk * a.nv + h0) * a.block_size + off) * a.D);
      dstride = (int64_t)a.block_size * a.D;
    }
    // ---- next item's metadata while the loads are in flight
    const ItemMeta mn =
        tn.t < a.T ? item_meta<SHARED>(tn, a, s_tab, qsl, seq_lens, slot_mapping, m.b, err) : m;
    {  // this item's rows, copied kStages - 1 items ago
      cp_async_wait<kStages - 1>();
      if (work && active) {
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (u < n) {
            *reinterpret_cast<uint4*>(x1[u].e) = *slot(buf, u, 0);
            *reinterpret_cast<uint4*>(x2[u].e) = *slot(buf, u, 1);
          }
      }
      buf = buf + 1 == kStages ? 0 : buf + 1;
    }

    if (work && rotate) {
      // RMSNorm: squares of every row of the item (independent chains), then
      // butterflies inside the row group, interleaved across the rows
      float ss[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float2 acc = make_float2(0.f, 0.f);
        if (u < n && active) {
#pragma unroll
          for (int j = 0; j < VEC; j += 2) {
            const float2 v1 = widen2(&x1[u].e[j]), v2 = widen2(&x2[u].e[j]);
            acc = __ffma2_rn(v1, v1, acc);
            acc = __ffma2_rn(v2, v2, acc);
          }
        }
        ss[u] = acc.x + acc.y;
      }
      for (int sh = G / 2; sh > 0; sh /= 2)
#pragma unroll
        for (int u = 0; u < U; ++u) ss[u] += __shfl_xor_sync(gmask, ss[u], sh, G);
      if (active) {
        // gamma folded into cos/sin: ca = g_low*cos, cb = -g_high*sin,
        // cc = g_high*cos, cd = g_low*sin
        float2 ca[VEC / 2], cb[VEC / 2], cc[VEC / 2], cd[VEC / 2];
#pragma unroll
        for (int j = 0; j < VEC; j += 2) {
          const float2 gl = widen2(&g1.e[j]), gh = widen2(&g2.e[j]);
          const float2 co = widen2(&cv.e[j]), si = widen2(&sv.e[j]);
          ca[j / 2] = __fmul2_rn(gl, co);
          cb[j / 2] = __fmul2_rn(gh, make_float2(-si.x, -si.y));
          cc[j / 2] = __fmul2_rn(gh, co);
          cd[j / 2] = __fmul2_rn(gl, si);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          if (u >= n) break;
          const float inv = rsqrtf(__fmaf_rn(ss[u], a.inv_d, a.eps));
          const float2 inv2 = make_float2(inv, inv);
#pragma unroll
          for (int j = 0; j < VEC; j += 2) {
            const float2 xl = widen2(&x1[u].e[j]), xh = widen2(&x2[u].e[j]);
            // each product carries one binary32 rounding relative to the
            // normalised terms, so a plain product + FMA is as accurate here
            // as a compensated difference
            const float2 lo = __ffma2_rn(xl, ca[j / 2], __fmul2_rn(xh, cb[j / 2]));
            const float2 hi = __ffma2_rn(xh, cc[j / 2], __fmul2_rn(xl, cd[j / 2]));
            narrow2(&x1[u].e[j], __fmul2_rn(lo, inv2));
            narrow2(&x2[u].e[j], __fmul2_rn(hi, inv2));
          }
          store_vec(dst + u * dstride + i0, x1[u], *dspan, err);
          store_vec(dst + u * dstride + half + i0, x2[u], *dspan, err);
        }
      }
    } else if (work && active) {  // V: stored as is
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (u < n) {
          store_vec(dst + u * dstride + i0, x1[u], *dspan, err);
          store_vec(dst + u * dstride + half + i0, x2[u], *dspan, err);
        }
    }
    if (tn.t >= a.T) break;
    m = mn;
  }
}

template <typename T, bool SHARED>
cudaError_t launch_tables(const QkvProblem& p, const QkvArgs& a, cudaStream_t stream) {
  constexpr int VEC = 16 / sizeof(T);
  const int64_t groups = kThreads / a.group;
  auto kernel = qkv_kernel<T, VEC, SHARED>;
  // row stages, then the shared tables rounded up to 4 KB so that few distinct
  // sizes reach the occupancy cache
  const size_t tables = SHARED ? (size_t)((2 * p.B + 1) * sizeof(int64_t) + 4095) / 4096 * 4096 : 0;
  const size_t smem = kStageBytes + tables;
  if (smem > 48 * 1024) {
    const cudaError_t e = opt_in_shared(reinterpret_cast<const void*>(kernel), smem);
    if (e != cudaSuccess) return e;
  }
  const int64_t resident = (int64_t)sm_count() * resident_blocks(reinterpret_cast<const void*>(kernel), kThreads, smem);
  const int64_t grid = std::max<int64_t>(1, std::min((a.items + groups - 1) / groups, resident));
  QkvArgs args = a;
  args.stride_t = grid * groups / a.per_token;
  args.stride_r = (int32_t)(grid * groups % a.per_token);
  unsigned int* err = nullptr;
  const cudaError_t e = device_error_address(&err);
  if (e != cudaSuccess) return e;
  return launch_overlapped_smem(kernel, (unsigned)grid, kThreads, smem, stream, static_cast<const T*>(p.qkv),
                                static_cast<const T*>(p.q_gamma), static_cast<const T*>(p.k_gamma),
                                static_cast<const T*>(p.cache), p.seq_lens, p.query_start_loc, p.slot_mapping,
                                static_cast<T*>(p.q_out), static_cast<T*>(p.k_cache), static_cast<T*>(p.v_cache),
                                err, args);
}

template <typename T>
cudaError_t launch_typed(const QkvProblem& p, cudaStream_t stream) {
  constexpr int VEC = 16 / sizeof(T);
  constexpr int U = kRowsInFlight;
  QkvArgs a;
  a.T = p.T;
  a.B = p.B;
  a.max_seq = p.max_seq;
  a.nq = (int32_t)p.nq;
  a.nk = (int32_t)p.nk;
  a.nv = (int32_t)p.nv;
  a.iq = (int32_t)((p.nq + U - 1) / U);
  a.ik = (int32_t)((p.nk + U - 1) / U);
  a.per_token = a.iq + a.ik + (int32_t)((p.nv + U - 1) / U);
  a.D = (int32_t)p.D;
  a.W = (p.nq + p.nk + p.nv) * p.D;
  a.block_size = (int32_t)p.block_size;
  a.num_slots = p.num_blocks * p.block_size;
  a.chunks = (int32_t)(p.D / 2 / VEC);
  a.group = 1;
  while (a.group < a.chunks) a.group *= 2;
  a.items = p.T * a.per_token;
  a.eps = p.eps;
  a.inv_d = 1.0f / (float)p.D;
  a.items32 = a.items <= 0xffffffffLL && a.num_slots <= 0xffffffffLL;
  a.bs_shift = -1;
  for (int sh = 0; sh < 31; ++sh)
    if ((int64_t(1) << sh) == p.block_size) a.bs_shift = sh;
  a.stride_t = 0;  // set with the grid
  a.stride_r = 0;
  const int64_t e = sizeof(T);
  a.qkv_span = make_span(p.qkv, p.T * a.W * e);
  a.qg_span = make_span(p.q_gamma, p.D * e);
  a.kg_span = make_span(p.k_gamma, p.D * e);
  a.cache_span = make_span(p.cache, p.max_seq * p.D * e);
  a.sl_span = make_span(p.seq_lens, p.B * 8);
  a.qsl_span = make_span(p.query_start_loc, (p.B + 1) * 8);
  a.slot_span = make_span(p.slot_mapping, p.T * 8);
  a.qo_span = make_span(p.q_out, p.T * p.nq * p.D * e);
  a.kc_span = make_span(p.k_cache, p.num_blocks * p.nk * p.block_size * p.D * e);
  a.vc_span = make_span(p.v_cache, p.num_blocks * p.nv * p.block_size * p.D * e);
  a.tab_span = make_span(nullptr, 0);  // set in the kernel: the shared batch tables
  if (2 * p.B + 1 <= kSharedTable) return launch_tables<T, true>(p, a, stream);
  return launch_tables<T, false>(p, a, stream);
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
