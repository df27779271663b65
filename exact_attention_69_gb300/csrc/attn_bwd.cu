// Instantiations of the sm_103a backward kernels (every mask, d = 32 / 64 / 128).
#include "attn_bwd_sm103.cuh"

namespace attn {
cudaError_t launch_bwd(const BwdParams& p, int d, int mask, cudaStream_t s, cudaStream_t aux,
                       cudaEvent_t fork, cudaEvent_t join) {
  const dev::BwdStreams st{s, aux, fork, join};
  switch (d) {
    case 32: return dev::launch_bwd_dim<32>(p, mask, st);
    case 64: return dev::launch_bwd_dim<64>(p, mask, st);
    case 128: return dev::launch_bwd_dim<128>(p, mask, st);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace attn
