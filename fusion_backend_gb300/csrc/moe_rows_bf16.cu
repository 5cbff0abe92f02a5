// Row kernel instances: bf16 weights, H = 2048 (T <= 1, 2, 4, 8).
#include "moe_rows.cuh"

namespace moe {

cudaError_t launch_rows_bf16_fast(const LayerParams& p, cudaStream_t stream) {
  switch (tmax_for(p.T)) {
    case 1: return launch_rows_t<1, kWkBf16, true>(p, stream);
    case 2: return launch_rows_t<2, kWkBf16, true>(p, stream);
    case 4: return launch_rows_t<4, kWkBf16, true>(p, stream);
    default: return launch_rows_t<8, kWkBf16, true>(p, stream);
  }
}

}  // namespace moe
