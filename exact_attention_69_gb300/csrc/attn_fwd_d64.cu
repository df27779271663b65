// Instantiations of the sm_103a attention kernel for head dimension 64.
#include "attn_sm103.cuh"

namespace attn {
cudaError_t launch_d64(const KernelParams& p, int mask, int grid, cudaStream_t s) {
  return dev::launch_dim<64>(p, mask, grid, s);
}
// The twin decision depends on the tiles, not on the head dimension.
int twin_tasks(const KernelParams& p, int mask) { return dev::twin_dim(p, mask); }
}  // namespace attn
