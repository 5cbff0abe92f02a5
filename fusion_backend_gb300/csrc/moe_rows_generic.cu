// Row kernel instances for the other decode shapes: any H <= 4096 (bf16: a
// multiple of 8, 4-bit: of 256), E <= 1024, T <= 8, fp32 arithmetic; one or
// two 8-column chunks per thread (H <= 2048, H <= 4096).
#include "moe_rows.cuh"

namespace moe {

cudaError_t launch_rows_generic(const LayerParams& p, cudaStream_t stream) {
  if (p.H <= 2048)
    return p.wfmt == 1 ? launch_rows_t<8, true, false, 1>(p, stream) : launch_rows_t<8, false, false, 1>(p, stream);
  return p.wfmt == 1 ? launch_rows_t<8, true, false, 2>(p, stream) : launch_rows_t<8, false, false, 2>(p, stream);
}

}  // namespace moe
