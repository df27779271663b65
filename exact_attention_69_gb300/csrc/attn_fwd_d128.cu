// Instantiations of the sm_103a attention kernel for head dimension 128.
#include "attn_sm103.cuh"

namespace attn {
cudaError_t launch_d128(const KernelParams& p, int mask, int grid, cudaStream_t s) {
  return dev::launch_dim<128>(p, mask, grid, s);
}
}  // namespace attn
