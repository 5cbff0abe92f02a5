// Device helpers shared by the kernels of the fused MoE FFN layer: warp
// reductions (plain and error-free), the pre-norm block factor and the
// 8-wide activation loads.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

static inline int tmax_for(int T) { return T <= 1 ? 1 : T <= 2 ? 2 : T <= 4 ? 4 : 8; }

// -------------------------------------------------------------- reductions
MOE_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Butterfly reduction of a (sum, compensation) pair; every lane ends with
// the same bits because TwoSum is symmetric in its operands.
MOE_DEV void warp_sum2(float& s, float& c) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float so = __shfl_xor_sync(0xffffffffu, s, o);
    const float co = __shfl_xor_sync(0xffffffffu, c, o);
    float t, e;
    two_sum(s, so, t, e);
    s = t;
    c = __fadd_rn(__fadd_rn(c, co), e);
  }
}

// RMSNorm factor of one fp32 row: inv = 1/sqrt(mean(x^2) + eps), computed
// from an error-free sum of squares and returned as hi + lo floats.  All
// lanes of the warp return the same value.
MOE_DEV void warp_norm_factor(const float* row, int H, float eps, float& hi, float& lo) {
  const int lane = threadIdx.x & 31;
  float s = 0.f, c = 0.f;
  for (int h = lane; h < H; h += 32) {
    const float v = row[h];
    float p, e1, t, e2;
    two_prod(v, v, p, e1);
    two_sum(s, p, t, e2);
    s = t;
    c = __fadd_rn(c, __fadd_rn(e1, e2));
  }
  warp_sum2(s, c);
  const double ss = (double)s + (double)c;
  const double inv = 1.0 / sqrt(ss / (double)H + (double)eps);
  hi = (float)inv;
  lo = (float)(inv - (double)hi);
}

// bf16(fp32(x * inv)) for the pre-norm block form, inv given as hi + lo.
MOE_DEV float norm_apply(float x, float hi, float lo) {
  float p, e;
  two_prod(x, hi, p, e);
  const float r = __fadd_rn(p, __fmaf_rn(x, lo, e));
  return bf16_to_float(float_to_bf16_rne(r));
}

// Eight activations of token t starting at column c0 (c0 % 8 == 0): fp32 x,
// bf16 x, or in the block form the normalised bf16 value of x_res (factor
// hi + lo of that token).
MOE_DEV void load_x8(const LayerParams& P, float hi, float lo, int t, int c0, float* xf) {
  if (P.block_mode) {
    const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(P.x) + (size_t)t * P.H + c0);
    const float4 a = src[0], b = src[1];
    xf[0] = norm_apply(a.x, hi, lo); xf[1] = norm_apply(a.y, hi, lo);
    xf[2] = norm_apply(a.z, hi, lo); xf[3] = norm_apply(a.w, hi, lo);
    xf[4] = norm_apply(b.x, hi, lo); xf[5] = norm_apply(b.y, hi, lo);
    xf[6] = norm_apply(b.z, hi, lo); xf[7] = norm_apply(b.w, hi, lo);
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
}

}  // namespace moe
