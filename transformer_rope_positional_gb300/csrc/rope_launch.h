// Host-side interface between the C ABI (rope_api.cu) and the kernel launchers.
// Arguments arrive here already validated.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace rope {

enum DType : int32_t { kF32 = 0, kF16 = 1, kBF16 = 2, kI64 = 3 };

// In-place partial interleave RoPE on x[B, S, N, D], slice [start, start + L).
struct InplaceProblem {
  void* x;
  const void* cos;
  const void* sin;
  int32_t x_dtype;
  int32_t cs_dtype;
  int64_t B, S, N, D;
  int64_t start, L;
  // cos/sin row strides (in rows of L elements) for b, s, n; 0 on broadcast dims
  int64_t cs_b, cs_s, cs_n;
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
};

cudaError_t launch_inplace(const InplaceProblem& p, cudaStream_t stream);
cudaError_t launch_cache(const CacheProblem& p, cudaStream_t stream);

// Largest number of threads one team of the cache kernel may need.
int64_t cache_team_threads(const CacheProblem& p);

// Device error word of the current device.
cudaError_t read_and_clear_device_error(cudaStream_t stream, uint32_t* code);

// Launch bookkeeping.
void count_launch();
int sm_count();

}  // namespace rope
