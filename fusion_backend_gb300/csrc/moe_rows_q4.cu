// Row kernel instances: 4-bit weights on the tensor cores (codes decoded to
// exact bf16 fragments, block scales applied in fp32), H = 2048
// (T <= 1, 2, 4, 8).
#include "moe_rows.cuh"

namespace moe {

cudaError_t launch_rows_q4_fast(const LayerParams& p, cudaStream_t stream) {
  switch (tmax_for(p.T)) {
    case 1: return launch_rows_t<1, kWkQ4, true>(p, stream);
    case 2: return launch_rows_t<2, kWkQ4, true>(p, stream);
    case 4: return launch_rows_t<4, kWkQ4, true>(p, stream);
    default: return launch_rows_t<8, kWkQ4, true>(p, stream);
  }
}

}  // namespace moe
