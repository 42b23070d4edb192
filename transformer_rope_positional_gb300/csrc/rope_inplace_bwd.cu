// Backward in-place partial RoPE: the transpose of the forward map applied to
// the incoming gradient in place (interleave and half modes); see rope_inplace.cuh.
#include "rope_inplace.cuh"

namespace rope {

cudaError_t launch_inplace_backward(const InplaceProblem& p, cudaStream_t stream) {
  return inplace::launch_direction<true>(p, stream);
}

}  // namespace rope
