// Instantiations of the sm_103a backward kernels (no mask and causal, d = 32 / 64 / 128).
#include "attn_bwd_sm103.cuh"

namespace attn {
cudaError_t launch_bwd(const BwdParams& p, int d, int mask, cudaStream_t s) {
  switch (d) {
    case 32: return dev::launch_bwd_dim<32>(p, mask, s);
    case 64: return dev::launch_bwd_dim<64>(p, mask, s);
    case 128: return dev::launch_bwd_dim<128>(p, mask, s);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace attn
