// Router kernel of the fused MoE FFN layer (decode path), sm_103a.
//
// One block of 128 threads per router row (E rows, plus one for the
// shared-gate vector): logit[t,e] = sum_h W[e,h] x[t,h] accumulated
// error-free (TwoSum / TwoProduct with a compensation term), so the fp32
// logit is the exact dot product rounded once (up to a residual far below
// fp32 resolution) and the top-k decision does not depend on the summation
// order.  Block 0 also zeroes the control words that the row kernel of the
// same call counts on.
//
// The blocks are small (few registers, no dynamic shared memory) so that
// they fit on an SM beside a block of the previous call's row kernel: they
// start, pull their weight row into L2 and wait (griddepcontrol.wait) while
// that kernel finishes.
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_layer_common.cuh"

namespace moe {

template <int TMAX>
__global__ void __launch_bounds__(kRouteThreads) k_route(LayerParams P) {
  constexpr int kWarps = kRouteThreads / 32;
  __shared__ float red_s[kWarps][TMAX];
  __shared__ float red_c[kWarps][TMAX];
  __shared__ float s_inv[TMAX][2];
  __shared__ float s_red[kWarps * TMAX * 2];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x;
  const uint16_t* w = row < P.E ? P.router_w + (size_t)row * P.H : P.gate_w;
  // A prefetch only warms the coherent L2; every real access follows the wait.
  if (tid == 0) prefetch_l2(w, (uint32_t)P.H * 2);
  pdl_launch_dependents();
  pdl_wait();
  if (row == 0 && tid < kCtrlWords) P.ctrl[tid] = 0u;
  // this thread's weight chunks, loaded ahead of the norm factors (H <= 4096:
  // at most four 8-element chunks a thread)
  constexpr int kChunks = kMaxH / (kRouteThreads * 8);
  uint4 wreg[kChunks];
#pragma unroll
  for (int i = 0; i < kChunks; ++i) {
    const int c0 = tid * 8 + i * kRouteThreads * 8;
    wreg[i] = c0 < P.H ? *reinterpret_cast<const uint4*>(w + c0) : make_uint4(0u, 0u, 0u, 0u);
  }
  if (P.block_mode) block_norm_factors(static_cast<const float*>(P.x), P.T, P.H, P.eps, s_red, &s_inv[0][0], kWarps);
  float s[TMAX], c[TMAX];
#pragma unroll
  for (int t = 0; t < TMAX; ++t) s[t] = c[t] = 0.f;
  const bool exact_products = P.block_mode || P.act == 1;  // bf16 x bf16 is exact in fp32
#pragma unroll
  for (int i = 0; i < kChunks; ++i) {
    const int c0 = tid * 8 + i * kRouteThreads * 8;
    if (c0 >= P.H) break;
    const uint4 wv = wreg[i];
    const float wf[8] = {bf16_lo(wv.x), bf16_hi(wv.x), bf16_lo(wv.y), bf16_hi(wv.y),
                         bf16_lo(wv.z), bf16_hi(wv.z), bf16_lo(wv.w), bf16_hi(wv.w)};
#pragma unroll
    for (int t = 0; t < TMAX; ++t) {
      if (t >= P.T) break;
      float xf[8];
      load_x8(P, s_inv[t][0], s_inv[t][1], t, c0, xf);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float p, e1 = 0.f, tt, e2;
        if (exact_products)
          p = __fmul_rn(wf[j], xf[j]);
        else
          two_prod(wf[j], xf[j], p, e1);
        two_sum(s[t], p, tt, e2);
        s[t] = tt;
        c[t] = __fadd_rn(c[t], __fadd_rn(e1, e2));
      }
    }
  }
#pragma unroll
  for (int t = 0; t < TMAX; ++t) {
    warp_sum2(s[t], c[t]);
    if (lane == 0) {
      red_s[warp][t] = s[t];
      red_c[warp][t] = c[t];
    }
  }
  __syncthreads();
  if (tid < P.T) {
    float S = red_s[0][tid], C = red_c[0][tid];
    for (int wi = 1; wi < kWarps; ++wi) {
      float tt, e;
      two_sum(S, red_s[wi][tid], tt, e);
      S = tt;
      C = __fadd_rn(__fadd_rn(C, red_c[wi][tid]), e);
    }
    P.logits[(size_t)tid * P.ls + row] = __fadd_rn(S, C);
  }
}

template <int TMAX>
static cudaError_t launch_route_t(const LayerParams& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(p.E + 1);
  cfg.blockDim = dim3(kRouteThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_route<TMAX>, p);
}

// The waits of the layer's kernels, each on a condition nothing satisfies:
// the status word must end as the timeout status, and the kernel returns.
__global__ void k_probe_timeout(uint32_t* ctrl, int which) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  ctrl[kCtrlStatus] = 0u;
  ctrl[kCtrlProbe] = 0u;
  bool ok = false;
  if (which == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
    ok = mbar_wait(&bar, 0);  // nothing arrives: phase 0 never completes
  } else {
    for (uint32_t i = 0; i < kSpinLimit; ++i) {  // the grid barrier's spin; the target is never reached
      if (ld_acquire_gpu(&ctrl[kCtrlProbe]) >= 0xFFFFFFFFu) {
        ok = true;
        break;
      }
      if (i > 256) __nanosleep(32);
    }
  }
  if (!ok) atomicExch(reinterpret_cast<int*>(&ctrl[kCtrlStatus]), kStatusTimeout);
}

cudaError_t launch_probe_timeout(uint32_t* ctrl, int which, cudaStream_t stream) {
  k_probe_timeout<<<1, 32, 0, stream>>>(ctrl, which);
  return cudaGetLastError();
}

cudaError_t launch_route(const LayerParams& p, cudaStream_t stream) {
  switch (tmax_for(p.T)) {
    case 1: return launch_route_t<1>(p, stream);
    case 2: return launch_route_t<2>(p, stream);
    case 4: return launch_route_t<4>(p, stream);
    default: return launch_route_t<8>(p, stream);
  }
}

}  // namespace moe
