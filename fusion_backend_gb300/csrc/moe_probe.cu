// The failure-path probe of the fused MoE FFN layer, sm_103a: one small
// kernel that runs the layer's kinds of bounded wait against conditions
// nothing ever satisfies, so that the give-up path (status word set to the
// timeout status, kernel returns, context usable) can be tested without a
// fault.
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_layer_common.cuh"

namespace moe {

// The waits of the layer's kernels, each on a condition nothing satisfies:
// the status word must end as the timeout status, and the kernel returns.
// which = 0: an mbarrier phase that never completes (the wait of a shared-
// memory copy that never lands); which = 1: the row kernel's grid-barrier
// wait on a flag slot that never receives the expected epoch; which = 2: the
// row kernel's poll of a tagged word (a partial output) that never carries
// the expected tag.  The slot is the control words 4..5; the value expected
// is one more than it holds.
__global__ void k_probe_timeout(uint32_t* ctrl, int which) {
  __shared__ uint64_t bar;
  const int lane = threadIdx.x & 31;
  bool ok = false;
  if (which == 0) {
    if (lane == 0) {
      ctrl[kCtrlStatus] = 0u;
      mbar_init(&bar, 1);
      mbar_fence_init();
      ok = mbar_wait(&bar, 0);  // nothing arrives: phase 0 never completes
    }
  } else {
    unsigned long long* slot = reinterpret_cast<unsigned long long*>(ctrl + kCtrlProbe + 2);
    const unsigned long long never = ld_relaxed_gpu_u64(slot) + 1ull;
    if (lane == 0) ctrl[kCtrlStatus] = 0u;
    __syncwarp();
    if (which == 1) {
      ok = grid_flags_wait(slot, 1, never);
    } else {
      float v;
      ok = poll_tagged<1>(slot, 0, 1, tag_of_word(ld_relaxed_gpu_u64(slot)) + 1u, &v);
      ok = __all_sync(0xffffffffu, ok);
    }
  }
  if (!ok && lane == 0) atomicExch(reinterpret_cast<int*>(&ctrl[kCtrlStatus]), kStatusTimeout);
}

cudaError_t launch_probe_timeout(uint32_t* ctrl, int which, cudaStream_t stream) {
  k_probe_timeout<<<1, 32, 0, stream>>>(ctrl, which);
  return cudaGetLastError();
}

}  // namespace moe
