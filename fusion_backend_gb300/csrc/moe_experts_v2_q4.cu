// Fast-path expert kernel, 4-bit weights: instantiations and launch.
#include "moe_experts_v2.cuh"

namespace moe {

cudaError_t launch_decode_v2_q4(const DecodeParams& p, cudaStream_t stream) {
  switch (tmax_for(p.T)) {
    case 1: return launch_v2_t<1, true, true>(p, stream);
    case 2: return launch_v2_t<2, true, false>(p, stream);
    case 4: return launch_v2_t<4, true, false>(p, stream);
    default: return launch_v2_t<8, true, false>(p, stream);
  }
}

}  // namespace moe
