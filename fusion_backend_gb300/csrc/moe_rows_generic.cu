// Row kernel instances for the other decode shapes: any H <= 4096 (bf16: a
// multiple of 8, 4-bit: of 256, int8: of 16), E <= 1024, T <= 8, fp32
// arithmetic (int8: int32 dot products); one or two 8-column chunks per
// thread (H <= 2048, H <= 4096).  Int8 weights with one token have their own
// instance (no registers or loop trips for absent tokens).
#include "moe_rows.cuh"

namespace moe {

cudaError_t launch_rows_generic(const LayerParams& p, cudaStream_t stream) {
  if (p.H <= 2048) {
    switch (p.wfmt) {
      case kWkQ4: return launch_rows_t<8, kWkQ4, false, 1>(p, stream);
      case kWkI8: return p.T == 1 ? launch_rows_t<1, kWkI8, false, 1>(p, stream)
                                  : launch_rows_t<8, kWkI8, false, 1>(p, stream);
      default: return launch_rows_t<8, kWkBf16, false, 1>(p, stream);
    }
  }
  switch (p.wfmt) {
    case kWkQ4: return launch_rows_t<8, kWkQ4, false, 2>(p, stream);
    case kWkI8: return launch_rows_t<8, kWkI8, false, 2>(p, stream);
    default: return launch_rows_t<8, kWkBf16, false, 2>(p, stream);
  }
}

}  // namespace moe
