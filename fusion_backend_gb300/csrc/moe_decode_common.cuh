// Device helpers shared by the decode kernels of the fused MoE FFN layer:
// warp reductions (plain and error-free), the pre-norm block factor, 8-wide
// activation and weight loads, and the per-token top-k of one warp.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

static inline int tmax_for(int T) { return T <= 1 ? 1 : T <= 2 ? 2 : T <= 4 ? 4 : 8; }
static inline int align_up(int v, int a) { return (v + a - 1) / a * a; }

MOE_DEV int div_floor_ll(long long a, long long b) { return static_cast<int>(a / b); }

MOE_DEV void down_rows(const DecodeParams& P, int c, int& a, int& b) {
  a = div_floor_ll((long long)P.H * c, P.G);
  b = div_floor_ll((long long)P.H * (c + 1), P.G);
}

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

// Eight activations of token t starting at column c0 (c0 % 8 == 0).

// As load_x8, with the block-form factors given as an array inv[2t], inv[2t+1].
MOE_DEV void load_x8_any(const DecodeParams& P, const float* inv, int t, int c0, float* xf) {
  if (P.block_mode) {
    const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(P.x) + (size_t)t * P.H + c0);
    const float4 a = src[0], b = src[1];
    const float hi = inv[2 * t], lo = inv[2 * t + 1];
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

// Eight weights starting at column c0 of a stored row (bf16 or 4-bit).
MOE_DEV void load_w8(const uint8_t* row, int cols, int wfmt, int c0, float* w) {
  if (wfmt == 0) {
    const uint4 v = *reinterpret_cast<const uint4*>(row + (size_t)c0 * 2);
    w[0] = bf16_lo(v.x); w[1] = bf16_hi(v.x); w[2] = bf16_lo(v.y); w[3] = bf16_hi(v.y);
    w[4] = bf16_lo(v.z); w[5] = bf16_hi(v.z); w[6] = bf16_lo(v.w); w[7] = bf16_hi(v.w);
  } else {
    const uint32_t q = *reinterpret_cast<const uint32_t*>(row + c0 / 2);
    const float d = __half2float(*reinterpret_cast<const __half*>(row + cols / 2 + (c0 / 32) * 2));
#pragma unroll
    for (int j = 0; j < 8; ++j) w[j] = d * static_cast<float>(static_cast<int>((q >> (4 * j)) & 0xFu) - 8);
  }
}


MOE_DEV unsigned long long topk_key(float v, int e) {
  return (static_cast<unsigned long long>(float_order_key(v)) << 32) | (0xFFFFFFFFull - (unsigned)e);
}

// Top-k of one token's E logits by one warp: K rounds, each taking the warp
// maximum of the remaining values' order keys (hardware warp reduction) and,
// among the lanes holding that maximum, the lowest expert index -- so equal
// logits go to the lower index.  ids[0..K) in rank order; pout = softmax over
// the K chosen logits.  E <= 1024, K <= 32.
MOE_DEV void warp_topk(const float* lg, int E, int K, int32_t* ids, float* pout) {
  const int lane = threadIdx.x & 31;
  const int nk = (E - lane + 31) / 32;  // this lane's entries e = lane + 32 i
  uint32_t taken = 0u;
  int myid = 0;
  for (int j = 0; j < K; ++j) {
    uint32_t best = 0u;
    int bi = 0x7FFFFFFF;
    for (int i = 0; i < nk; ++i) {
      if (taken >> i & 1u) continue;
      const uint32_t k = float_order_key(lg[lane + 32 * i]);
      if (k > best) {
        best = k;
        bi = lane + 32 * i;
      }
    }
    const uint32_t m = __reduce_max_sync(0xffffffffu, best);
    const uint32_t win = __reduce_min_sync(0xffffffffu, best == m ? (uint32_t)bi : 0xFFFFFFFFu);
    if ((int)(win & 31u) == lane) taken |= 1u << (win >> 5);
    if (lane == j) myid = (int)win;
  }
  const float lj = lane < K ? lg[myid] : 0.f;
  const float l0 = __shfl_sync(0xffffffffu, lj, 0);
  const float z = lane < K ? expf(lj - l0) : 0.f;
  const float sum = warp_sum(z);
  if (lane < K) {
    ids[lane] = myid;
    pout[lane] = z / sum;
  }
  __syncwarp();
}

}  // namespace moe
