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

// Bounded wait of one thread until *word holds `epoch` (relaxed polls, then
// an acquire fence); false when the bound (about a second) ran out.
MOE_DEV bool word_wait(const unsigned long long* word, unsigned long long epoch) {
  unsigned long long t0 = 0;
  for (uint32_t it = 0;; ++it) {
    if (ld_relaxed_gpu_u64(word) == epoch) break;
    if (it == 16) t0 = global_ns();
    if (it >= kSpinLimit || (it > 16 && (it & 15) == 0 && global_ns() - t0 > kWaitLimitNs)) return false;
    if (it > 16) __nanosleep(64);
  }
  fence_acq_rel_gpu();
  return true;
}

// Bounded wait of one warp until every slot flags[0 .. G) holds `epoch`
// (the grid-wide barriers of the decode row kernel; see RowSync).  The
// lane's slots are polled with relaxed loads, all in flight together, and an
// acquire fence follows.  Gives up after about a second (the global timer,
// and an iteration cap in case it does not advance); returns false on every
// lane then.
MOE_DEV bool grid_flags_wait(const unsigned long long* flags, int G, unsigned long long epoch) {
  const int lane = threadIdx.x & 31;
  constexpr int kPer = (kMaxGrid + 31) / 32;
  uint32_t pending = 0u;
#pragma unroll
  for (int i = 0; i < kPer; ++i)
    if (lane + 32 * i < G) pending |= 1u << i;
  bool ok = true;
  unsigned long long t0 = 0;
  for (uint32_t it = 0; pending; ++it) {
    unsigned long long v[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) v[i] = (pending >> i & 1u) ? ld_relaxed_gpu_u64(flags + lane + 32 * i) : epoch;
#pragma unroll
    for (int i = 0; i < kPer; ++i)
      if (v[i] == epoch) pending &= ~(1u << i);
    if (!pending) break;
    if (it == 32) t0 = global_ns();
    if (it >= kSpinLimit || (it > 32 && (it & 15) == 0 && global_ns() - t0 > kWaitLimitNs)) {
      ok = false;
      break;
    }
    if (it > 32) __nanosleep(64);
  }
  fence_acq_rel_gpu();
  return __all_sync(0xffffffffu, ok);
}

// A grid-wide barrier of the decode row kernel (see RowSync), called by
// every thread of every block after the block's writes that the barrier
// publishes.  fast: each block adds one to *count (release) and waits until
// it reaches G.  Otherwise block c stores `epoch` into flags[c] (release);
// block 0's warp 0 waits for every slot and releases *go; every block waits
// for *go.  first: the call's first barrier -- block 0 then (after every
// block has arrived, hence has read RowSync's epoch and sig) clears the next
// call's counters and advances epoch and sig.  Returns false in every thread
// of the block when a wait gave up (bounded, about a second).
// NT: the threads of the block that take part (blk_sync).
template <int NT = 0>
MOE_DEV bool grid_barrier(RowSync* sy, int which, bool fast, int G, unsigned long long epoch, int cta, bool first) {
  const int tid = threadIdx.x, lane = tid & 31;
  blk_sync<NT>();
  bool ok = true;
  uint32_t* count = &sy->count[epoch & 1][which];
  if (tid == 0) {
    if (fast) {
      red_release_gpu_add(count, 1u);
      unsigned long long t0 = 0;
      for (uint32_t it = 0;; ++it) {
        if (ld_acquire_gpu(count) >= (uint32_t)G) break;
        if (it == 16) t0 = global_ns();
        if (it >= kSpinLimit || (it > 16 && (it & 15) == 0 && global_ns() - t0 > kWaitLimitNs)) {
          ok = false;
          break;
        }
        if (it > 16) __nanosleep(32);
      }
    } else {
      st_release_gpu_u64((which ? sy->partial_ready : sy->logits_ready) + cta, epoch);
    }
  }
  if (!fast && tid < 32) {
    if (cta == 0) {
      ok = grid_flags_wait(which ? sy->partial_ready : sy->logits_ready, G, epoch);
      if (ok && lane == 0) st_release_gpu_u64(&sy->go[which], epoch);
    }
    if (ok && lane == 0) ok = word_wait(&sy->go[which], epoch);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  }
  if (first && cta == 0 && tid == 0 && ok) {
    // every block has read epoch and sig: prepare the next call's fast path
    sy->count[(epoch + 1) & 1][0] = 0u;
    sy->count[(epoch + 1) & 1][1] = 0u;
    sy->epoch = epoch;
    __threadfence();
    sy->sig = ~epoch;
  }
  return !blk_sync_or<NT>(!ok);
}

// Bounded poll of one thread on n <= N tagged words p[i * stride] (see
// `tagged`): v[i] = the value of word i once its tag is `tag`.  The pending
// words are loaded together (relaxed loads), again and again until every
// tag matches.  Gives up after about a second (the global timer, and an
// iteration cap in case it does not advance) and returns false; a word never
// seen with the tag reads 0.
template <int N>
MOE_DEV bool poll_tagged(const unsigned long long* p, size_t stride, int n, uint32_t tag, float* v) {
  uint32_t pending = 0u;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    v[i] = 0.f;
    if (i < n) pending |= 1u << i;
  }
  unsigned long long t0 = 0;
  for (uint32_t it = 0; pending; ++it) {
    unsigned long long w[N];
#pragma unroll
    for (int i = 0; i < N; ++i) w[i] = (pending >> i & 1u) ? ld_relaxed_gpu_u64(p + (size_t)i * stride) : 0ull;
#pragma unroll
    for (int i = 0; i < N; ++i)
      if ((pending >> i & 1u) && tag_of_word(w[i]) == tag) {
        v[i] = value_of_word(w[i]);
        pending &= ~(1u << i);
      }
    if (!pending) break;
    if (it == 32) t0 = global_ns();
    if (it >= kSpinLimit || (it > 32 && (it & 15) == 0 && global_ns() - t0 > kWaitLimitNs)) return false;
    if (it > 32) __nanosleep(32);
  }
  return true;
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

// Error-free sum of squares of row[h] for h in [h_begin, h_end) (multiples
// of 4; the row 16-byte aligned) by one warp, as a (sum, compensation) pair
// held by every lane; eight float4 loads in flight per lane.
MOE_DEV void warp_sumsq(const float* row, int h_begin, int h_end, float& s, float& c) {
  const int lane = threadIdx.x & 31;
  s = 0.f;
  c = 0.f;
  for (int h0 = h_begin + 4 * lane; h0 < h_end; h0 += 128 * 8) {
    float4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int h = h0 + 128 * j;
      v[j] = h < h_end ? *reinterpret_cast<const float4*>(row + h) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float e4[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float p, e1, t, e2;
        two_prod(e4[q], e4[q], p, e1);
        two_sum(s, p, t, e2);
        s = t;
        c = __fadd_rn(c, __fadd_rn(e1, e2));
      }
    }
  }
  warp_sum2(s, c);
}

// inv = 1/sqrt((s + c)/H + eps) as hi + lo floats, in float-float
// arithmetic (no fp64): the mean as a float-float, an fp32 estimate y of the
// inverse square root and one Newton step y (1 + e/2), e = 1 - m y^2 formed
// from exact products (relative error about 2^-46).
MOE_DEV void norm_factor_ff(float s, float c, int H, float eps, float& hi, float& lo) {
  float mh, ml;
  {
    const float q = __fdiv_rn(s, (float)H);
    const float r = __fmaf_rn(-q, (float)H, s);  // s - q H, exact
    const float q2 = __fdiv_rn(__fadd_rn(r, c), (float)H);
    float th, tl;
    two_sum(q, q2, th, tl);
    two_sum(th, eps, mh, ml);
    ml = __fadd_rn(ml, tl);
  }
  const float y = __frsqrt_rn(mh);
  float y2h, y2l, ph, pl;
  two_prod(y, y, y2h, y2l);
  two_prod(mh, y2h, ph, pl);
  const float e = __fsub_rn(__fsub_rn(__fsub_rn(1.0f, ph), pl), __fmaf_rn(mh, y2l, __fmul_rn(ml, y2h)));
  const float corr = __fmul_rn(__fmul_rn(y, e), 0.5f);
  two_sum(y, corr, hi, lo);
}

// RMSNorm factors of T fp32 rows (row t at x + t H) by all W warps of the
// block: warp w sums squares over its H/W slice of every row, the W pairs
// of a row meet in shared memory (red[W][T][2]), and thread t < T combines
// them error-free in warp order and writes inv[2t], inv[2t+1].  Ends with a
// block barrier (of the NT threads that take part, blk_sync).
template <int NT = 0>
MOE_DEV void block_norm_factors(const float* x, int T, int H, float eps, float* red, float* inv, int W) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slice = (H / W + 3) & ~3;
  const int hb = min(H, warp * slice), he = min(H, hb + slice);
  for (int t = 0; t < T; ++t) {
    float s, c;
    warp_sumsq(x + (size_t)t * H, hb, he, s, c);
    if (lane == 0) {
      red[(warp * T + t) * 2] = s;
      red[(warp * T + t) * 2 + 1] = c;
    }
  }
  blk_sync<NT>();
  if ((int)threadIdx.x < T) {
    const int t = threadIdx.x;
    float S = red[t * 2], C = red[t * 2 + 1];
    for (int w = 1; w < W; ++w) {
      float tt, e;
      two_sum(S, red[(w * T + t) * 2], tt, e);
      S = tt;
      C = __fadd_rn(__fadd_rn(C, red[(w * T + t) * 2 + 1]), e);
    }
    float hi, lo;
    norm_factor_ff(S, C, H, eps, hi, lo);
    inv[2 * t] = hi;
    inv[2 * t + 1] = lo;
  }
  blk_sync<NT>();
}

// RMSNorm factor of one fp32 row by one warp (see block_norm_factors).
MOE_DEV void warp_norm_factor(const float* row, int H, float eps, float& hi, float& lo) {
  float s, c;
  warp_sumsq(row, 0, H, s, c);
  norm_factor_ff(s, c, H, eps, hi, lo);
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
