// Host-side interface between the C ABI (rope_api.cu) and the kernel launchers.
// Arguments arrive here already validated.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace rope {

enum DType : int32_t { kF32 = 0, kF16 = 1, kBF16 = 2, kI64 = 3 };

// In-place partial RoPE on x[B, S, N, D], slice [start, start + L).
struct InplaceProblem {
  int32_t mode;   // 1 interleave, 0 half
  bool backward;  // apply the transpose (gradient) instead of the forward map
  void* x;
  const void* cos;
  const void* sin;
  int32_t x_dtype;
  int32_t cs_dtype;
  int64_t B, S, N, D;
  int64_t start, L;
  // cos/sin row strides (in rows of L elements) for b, s, n; 0 on broadcast dims
  int64_t cs_b, cs_s, cs_n;
  int64_t cs_rows;  // rows of L elements in cos (and sin): cB * cS * cN
};

// Cache-indexed RoPE of query[T, hq*hs] and key[T, hk*hs].
struct CacheProblem {
  const int64_t* positions;
  void* query;
  void* key;
  const void* cache;
  int32_t dtype;
  int64_t T;
  int64_t hq, hk;
  int64_t head_size;
  int64_t rotary_dim;
  int64_t max_seq;
  bool is_neox;
  int32_t mrope_rows;      // 0: rope; 3 or 4: mrope
  int32_t section_end[4];  // cumulative ends of the mrope sections (cos indices)
  int32_t cache_mode;      // 0: sections spliced in order; 1: interleaved splice
  int64_t q_stride;        // elements between consecutive query rows
  int64_t k_stride;        // elements between consecutive key rows
  void* query_out;         // contiguous outputs, or both NULL for in place
  void* key_out;
};

cudaError_t launch_inplace_forward(const InplaceProblem& p, cudaStream_t stream);
cudaError_t launch_inplace_backward(const InplaceProblem& p, cudaStream_t stream);
inline cudaError_t launch_inplace(const InplaceProblem& p, cudaStream_t stream) {
  return p.backward ? launch_inplace_backward(p, stream) : launch_inplace_forward(p, stream);
}
cudaError_t launch_cache(const CacheProblem& p, cudaStream_t stream);

// Fused QKV split + RMSNorm + RoPE + paged KV-cache write.
struct QkvProblem {
  const void* qkv;  // [T, (nq + nk + nv) * D]
  const void* q_gamma;
  const void* k_gamma;
  const void* cache;  // [max_seq, D] cos||sin
  const int64_t* seq_lens;         // [B]
  const int64_t* query_start_loc;  // [B + 1]
  const int64_t* slot_mapping;     // [T]
  void* q_out;                     // [T, nq * D]
  void* k_cache;                   // [num_blocks, nk, block_size, D]
  void* v_cache;                   // [num_blocks, nv, block_size, D]
  int32_t dtype;
  int64_t T, B;
  int64_t nq, nk, nv, D;
  int64_t max_seq;
  int64_t num_blocks, block_size;
  float eps;
};

cudaError_t launch_qkv(const QkvProblem& p, cudaStream_t stream);

// Threads that work on one head row in the cache kernel, and the most a CTA
// of that kernel holds.
int64_t cache_team_threads(const CacheProblem& p);
int64_t cache_max_team_threads();

// Device error word of the current device: read-and-clear, and its address
// for kernels of other translation units.
cudaError_t read_and_clear_device_error(cudaStream_t stream, uint32_t* code);
cudaError_t device_error_address(unsigned int** out);

// Launch bookkeeping.
void count_launch();
uint64_t launch_count();
int sm_count();
// CTAs of `kernel` (launched with `threads` threads and `smem` bytes of
// dynamic shared memory) that fit on one SM of the current device; cached, at
// least 1.
int resident_blocks(const void* kernel, int threads, size_t smem = 0);
// Let `kernel` launch with `smem` bytes of dynamic shared memory on the current
// device (needed above 48 KB); remembered per device and kernel.
cudaError_t opt_in_shared(const void* kernel, size_t smem);

// Launch `kernel` on `stream` with programmatic stream serialization allowed:
// the kernel may be scheduled while the previous kernel of the stream drains,
// and every kernel of this library executes wait_for_prior_grid() before its
// first global memory access, so stream order is unchanged; only the launch
// latency is overlapped with the previous kernel's tail.
template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped_smem(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                                   cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
  count_launch();
  return e == cudaSuccess ? cudaGetLastError() : e;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped(void (*kernel)(KArgs...), unsigned grid, unsigned block, cudaStream_t stream,
                              Args... args) {
  return launch_overlapped_smem(kernel, grid, block, 0, stream, args...);
}

}  // namespace rope
