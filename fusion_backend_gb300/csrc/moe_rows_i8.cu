// Row kernel instances: int8 weights and activation on the tensor cores
// (codes as exact fp16 operands, integer dot products in fp32 accumulators),
// H = 2048 (T <= 1, 2, 4, 8).
#include "moe_rows.cuh"

namespace moe {

cudaError_t launch_rows_i8_fast(const LayerParams& p, cudaStream_t stream) {
  switch (tmax_for(p.T)) {
    case 1: return launch_rows_t<1, kWkI8, true>(p, stream);
    case 2: return launch_rows_t<2, kWkI8, true>(p, stream);
    case 4: return launch_rows_t<4, kWkI8, true>(p, stream);
    default: return launch_rows_t<8, kWkI8, true>(p, stream);
  }
}

}  // namespace moe
