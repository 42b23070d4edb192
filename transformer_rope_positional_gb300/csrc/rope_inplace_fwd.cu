// Forward in-place partial RoPE (interleave and half modes); see rope_inplace.cuh.
#include "rope_inplace.cuh"

namespace rope {

cudaError_t launch_inplace_forward(const InplaceProblem& p, cudaStream_t stream) {
  return inplace::launch_direction<false>(p, stream);
}

}  // namespace rope
