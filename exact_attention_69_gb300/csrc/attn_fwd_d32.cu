// Instantiations of the sm_103a attention kernel for head dimension 32.
#include "attn_sm103.cuh"

namespace attn {
cudaError_t launch_d32(const KernelParams& p, int mask, int grid, cudaStream_t s) {
  return dev::launch_dim<32>(p, mask, grid, s);
}
}  // namespace attn
