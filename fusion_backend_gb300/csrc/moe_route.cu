// Router kernel of the fused MoE FFN layer (decode path), sm_103a.
//
// One CTA of 256 threads per router row (E rows, plus one for the shared-gate
// vector): logit[t,e] = sum_h W[e,h] x[t,h] accumulated error-free (TwoSum /
// TwoProduct with a compensation term), so the fp32 logit is the correctly
// rounded exact dot product and the top-k decision does not depend on the
// summation order.  It also zeroes the control words of the expert kernel.
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_decode_common.cuh"

namespace moe {

template <int TMAX>
__global__ void __launch_bounds__(kRouteThreads) k_route(DecodeParams P) {
  __shared__ float red_s[kRouteThreads / 32][TMAX];
  __shared__ float red_c[kRouteThreads / 32][TMAX];
  __shared__ float s_inv[TMAX][2];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x;
  const uint16_t* w = row < P.E ? P.router_w + (size_t)row * P.H : P.gate_w;
  // When launched behind the previous layer (programmatic dependent launch),
  // pull this CTA's weight row into L2 while that layer finishes.  A prefetch
  // only warms the coherent L2; every real access comes after the wait.
  if (tid == 0) prefetch_l2(w, (uint32_t)P.H * 2);
  pdl_wait();
  pdl_launch_dependents();
  if (row == 0 && tid < kCtrlWords) P.ctrl[tid] = 0u;
  if (P.block_mode) {
    for (int t = warp; t < P.T; t += kRouteThreads / 32) {
      float hi, lo;
      warp_norm_factor(static_cast<const float*>(P.x) + (size_t)t * P.H, P.H, P.eps, hi, lo);
      if (lane == 0) {
        s_inv[t][0] = hi;
        s_inv[t][1] = lo;
      }
    }
    __syncthreads();
  }
  float s[TMAX], c[TMAX];
#pragma unroll
  for (int t = 0; t < TMAX; ++t) s[t] = c[t] = 0.f;
  const bool exact_products = P.block_mode || P.act == 1;  // bf16 x bf16 is exact in fp32
  for (int c0 = tid * 8; c0 < P.H; c0 += kRouteThreads * 8) {
    const uint4 wv = *reinterpret_cast<const uint4*>(w + c0);
    const float wf[8] = {bf16_lo(wv.x), bf16_hi(wv.x), bf16_lo(wv.y), bf16_hi(wv.y),
                         bf16_lo(wv.z), bf16_hi(wv.z), bf16_lo(wv.w), bf16_hi(wv.w)};
#pragma unroll
    for (int t = 0; t < TMAX; ++t) {
      if (t >= P.T) break;
      float xf[8];
      if (P.block_mode) {
        const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(P.x) + (size_t)t * P.H + c0);
        const float4 a = src[0], b = src[1];
        const float av[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) xf[j] = norm_apply(av[j], s_inv[t][0], s_inv[t][1]);
      } else if (P.act == 0) {
        const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(P.x) + (size_t)t * P.H + c0);
        const float4 a = src[0], b = src[1];
        xf[0] = a.x; xf[1] = a.y; xf[2] = a.z; xf[3] = a.w;
        xf[4] = b.x; xf[5] = b.y; xf[6] = b.z; xf[7] = b.w;
      } else {
        const uint4 v = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(P.x) + (size_t)t * P.H + c0);
        xf[0] = bf16_lo(v.x); xf[1] = bf16_hi(v.x); xf[2] = bf16_lo(v.y); xf[3] = bf16_hi(v.y);
        xf[4] = bf16_lo(v.z); xf[5] = bf16_hi(v.z); xf[6] = bf16_lo(v.w); xf[7] = bf16_hi(v.w);
      }
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
    for (int wi = 1; wi < kRouteThreads / 32; ++wi) {
      float tt, e;
      two_sum(S, red_s[wi][tid], tt, e);
      S = tt;
      C = __fadd_rn(__fadd_rn(C, red_c[wi][tid]), e);
    }
    P.logits[(size_t)tid * P.ls + row] = __fadd_rn(S, C);
  }
}

template <int TMAX>
static cudaError_t launch_route_t(const DecodeParams& p, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(p.E + 1);
  cfg.blockDim = dim3(kRouteThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_route<TMAX>, p);
}

cudaError_t launch_route(const DecodeParams& p, cudaStream_t stream, bool pdl) {
  switch (tmax_for(p.T)) {
    case 1: return launch_route_t<1>(p, stream, pdl);
    case 2: return launch_route_t<2>(p, stream, pdl);
    case 4: return launch_route_t<4>(p, stream, pdl);
    default: return launch_route_t<8>(p, stream, pdl);
  }
}

}  // namespace moe
