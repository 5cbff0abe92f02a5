// Batched path of the fused MoE FFN layer (T > 8 tokens), sm_103a: the
// router GEMV, top-k with the selection bitmap, the bucketing of the chosen
// (token, expert) pairs into an expert-sorted slot order with a gather of x,
// and the fixed-order combine.  The two grouped GEMMs between the gather and
// the combine are in moe_gemm.cu.
//
// Slot order (the rows of x_perm, h_ws and y_ws): the routed slots of expert
// e are rows offsets[e] .. offsets[e] + counts[e] - 1, its tokens ascending;
// the shared expert's slot for token t is row T K + t.  Every output is a
// pure function of the router's logits, so the layer is deterministic.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_layer_common.cuh"
#include "moe_rows.cuh"

namespace moe {

cudaError_t launch_gemm_gate_up(const BatchParams& p, cudaStream_t stream);
cudaError_t launch_gemm_down(const BatchParams& p, cudaStream_t stream);
cudaError_t launch_gemm_gate_up_q4(const BatchParams& p, cudaStream_t stream);
cudaError_t launch_gemm_down_q4(const BatchParams& p, cudaStream_t stream);

namespace {

constexpr int kRouteTokens = 8;   // tokens per router block
constexpr int kRouteRows = 4;     // router rows per block (1 per warp, 4 warps)
constexpr int kGatherSplit = 4;   // blocks per expert in the bucketing kernel

// Eight bf16 of x (elements 0..7) -> eight fp16 in the operand order of the
// 4-bit GEMMs, e0 e4 e1 e5 e2 e6 e3 e7 (the order their dequantisation
// gives the weights along K).
__device__ __forceinline__ uint4 x8_f16_order(uint4 v) {
  const uint32_t in[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t a = in[i >> 1], b = in[2 + (i >> 1)];  // (e 2(i/2), e 2(i/2)+1), (e 4+.., ..)
    const float lo = (i & 1) ? bf16_hi(a) : bf16_lo(a), hi = (i & 1) ? bf16_hi(b) : bf16_lo(b);
    const __half2 h = __floats2half2_rn(lo, hi);
    o[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// sqrt(H) 2^-75 rounded up: the most a norm can lose to squares that round
// in the subnormal range (see k_route_b).
__device__ __forceinline__ float norm_underflow_pad(int H) { return __fmul_ru(sqrtf((float)H) * 1.0001f, 0x1p-75f); }

// Router logits in two passes.  Pass 1 (this kernel): plain fp32 sums of
// the bf16 x bf16 products (fused multiply-adds: the product is exact inside
// each, only the sum rounds) -- each lane adds n = H/32 products and the warp
// tree adds 5 levels, so |l - exact| <= ((n + 5) u / (1 - (n + 5) u))
// sum|w x| + H 2^-150 (u = 2^-24; the second term is the rounding of partial
// sums in the subnormal range, at most 2^-150 per fused multiply-add, and the
// warp tree's additions there are exact) -- and the norms |w_r|_2, |x_t|_2,
// which bound sum|w x| from above (Cauchy-Schwarz).  The top-k kernel takes
// the bound (n + 8) 2^-22 |w|_2 |x|_2 + 2^-20 |l| + H 2^-149, about 4x the
// above (and it covers the final rounding of the exact value to fp32); the
// norms carry their own margin for squares lost to underflow, so the bound
// holds for every finite input.  Pass 2 (the top-k kernel)
// recomputes exactly every logit whose interval can reach the top-k.  Block
// (token group, row group): 4 warps x 1 row x 8 tokens, small blocks so that
// the whole grid is resident at once.  The first block also clears the
// control words and every block a share of the bitmap.
__global__ void __launch_bounds__(128, 7) k_route_b(const __grid_constant__ BatchParams P) {
  extern __shared__ __align__(128) uint8_t route_smem[];  // the block's x rows (kRouteTokens x H bf16)
  __shared__ uint64_t s_bar;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nblk = gridDim.x * gridDim.y, bid = blockIdx.y * gridDim.x + blockIdx.x;
  pdl_launch_dependents();
  pdl_wait();  // x and the workspace belong to the previous kernels of the stream until here
  for (int i = bid * 128 + tid; i < P.E * P.tw; i += nblk * 128) P.bitmap[i] = 0u;
  if (bid == 0 && tid < kCtrlWords) P.ctrl[tid] = 0u;
  const int t0 = blockIdx.x * kRouteTokens;
  const int nt = min(kRouteTokens, P.T - t0);
  if (tid == 0) {
    mbar_init(&s_bar, 1);
    mbar_fence_init();
    const uint32_t bytes = (uint32_t)nt * (uint32_t)P.H * 2u;
    mbar_arrive_expect_tx(&s_bar, bytes);
    bulk_g2s(route_smem, P.x + (size_t)t0 * P.H, bytes, &s_bar, policy_evict_last());
  }
  const int r = blockIdx.y * kRouteRows + warp;
  const uint16_t* w = r < P.E ? P.router_w + (size_t)r * P.H : P.gate_w;
  float s[kRouteTokens], wsq = 0.f;
#pragma unroll
  for (int t = 0; t < kRouteTokens; ++t) s[t] = 0.f;
  __syncthreads();  // the barrier is initialised before any thread waits on it
  const bool ok = mbar_wait(&s_bar, 0);
  if (!ok && lane == 0) atomicExch(reinterpret_cast<int*>(&P.ctrl[kCtrlStatus]), kStatusTimeout);
  if (r <= P.E && ok) {
    const uint16_t* xs = reinterpret_cast<const uint16_t*>(route_smem);
    // the router row in chunks of 8 x 8 elements per lane, loaded ahead of use
    for (int cb = 0; cb < P.H; cb += 8 * 256) {
      uint4 wv[8];
#pragma unroll
      for (int it = 0; it < 8; ++it) {
        const int c0 = cb + it * 256 + lane * 8;
        wv[it] = c0 < P.H ? *reinterpret_cast<const uint4*>(w + c0) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int it = 0; it < 8; ++it) {
        const int c0 = cb + it * 256 + lane * 8;
        if (c0 >= P.H) break;
        const uint4 v = wv[it];
        const float wf[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                             bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
#pragma unroll
        for (int e = 0; e < 8; ++e) wsq = fmaf(wf[e], wf[e], wsq);
#pragma unroll
        for (int t = 0; t < kRouteTokens; ++t) {
          if (t >= nt) break;
          const uint4 xv = *reinterpret_cast<const uint4*>(xs + (size_t)t * P.H + c0);
          const float xf[8] = {bf16_lo(xv.x), bf16_hi(xv.x), bf16_lo(xv.y), bf16_hi(xv.y),
                               bf16_lo(xv.z), bf16_hi(xv.z), bf16_lo(xv.w), bf16_hi(xv.w)};
#pragma unroll
          for (int e = 0; e < 8; ++e) s[t] = fmaf(wf[e], xf[e], s[t]);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kRouteTokens; ++t) {
      const float st = warp_sum(s[t]);
      if (lane == 0 && t < nt) P.logits[(size_t)(t0 + t) * P.ls + r] = st;
    }
    // |w_r|_2 (the first token group's blocks write it), rounded up by 2^-8:
    // the fp32 sum of squares and the square root are off by far less.  Squares
    // in the subnormal range lose at most 2^-150 each to rounding, so the exact
    // norm is below sqrt(sum + H 2^-150) <= sqrt(sum) + sqrt(H) 2^-75: that
    // term is added too.
    const float wn = __fadd_ru(__fmul_ru(sqrtf(warp_sum(wsq)), 1.0f + 0x1p-8f), norm_underflow_pad(P.H));
    if (lane == 0 && blockIdx.x == 0) P.lbound[r] = wn;
  }
  if (blockIdx.y == 0 && ok) {
    // |x_t|_2 of this block's tokens (16 threads a token), rounded up likewise
    const int t = tid >> 4, l16 = tid & 15;
    float q = 0.f;
    if (t < nt) {
      const uint16_t* xt = reinterpret_cast<const uint16_t*>(route_smem) + (size_t)t * P.H;
      for (int c0 = l16 * 8; c0 < P.H; c0 += 128) {
        const uint4 xv = *reinterpret_cast<const uint4*>(xt + c0);
        const float xf[8] = {bf16_lo(xv.x), bf16_hi(xv.x), bf16_lo(xv.y), bf16_hi(xv.y),
                             bf16_lo(xv.z), bf16_hi(xv.z), bf16_lo(xv.w), bf16_hi(xv.w)};
#pragma unroll
        for (int e = 0; e < 8; ++e) q = fmaf(xf[e], xf[e], q);
      }
    }
#pragma unroll
    for (int o = 8; o; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
    if (l16 == 0 && t < nt)
      P.lbound[P.ls + t0 + t] = __fadd_ru(__fmul_ru(sqrtf(q), 1.0f + 0x1p-8f), norm_underflow_pad(P.H));
  }
}

// Exact logit of router row r (r == E: the shared-gate vector) for token t
// by one warp: error-free sums as in the decode router; every lane returns it.
__device__ float exact_logit(const BatchParams& P, int t, int r) {
  const int lane = threadIdx.x & 31;
  const uint16_t* w = r < P.E ? P.router_w + (size_t)r * P.H : P.gate_w;
  const uint16_t* x = P.x + (size_t)t * P.H;
  float s0 = 0.f, c0 = 0.f, s1 = 0.f, c1 = 0.f;  // two independent error-free sums (even / odd elements)
  for (int cb = 0; cb < P.H; cb += 4 * 256) {
    uint4 wv[4], xv[4];
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      const int c = cb + it * 256 + lane * 8;
      wv[it] = c < P.H ? *reinterpret_cast<const uint4*>(w + c) : make_uint4(0u, 0u, 0u, 0u);
      xv[it] = c < P.H ? *reinterpret_cast<const uint4*>(x + c) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      const uint4 v = wv[it], u = xv[it];
      const float wf[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                           bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
      const float xf[8] = {bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y),
                           bf16_lo(u.z), bf16_hi(u.z), bf16_lo(u.w), bf16_hi(u.w)};
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        float tt, e2;
        two_sum(s0, __fmul_rn(wf[e], xf[e]), tt, e2);
        s0 = tt;
        c0 = __fadd_rn(c0, e2);
        two_sum(s1, __fmul_rn(wf[e + 1], xf[e + 1]), tt, e2);
        s1 = tt;
        c1 = __fadd_rn(c1, e2);
      }
    }
  }
  float s, e;
  two_sum(s0, s1, s, e);
  float c = __fadd_rn(__fadd_rn(c0, c1), e);
  warp_sum2(s, c);
  return __fadd_rn(s, c);
}

// Top-k of token t (block t, 8 warps).  L = the k-th largest
// lower end (l - b) of the logit intervals; the candidates are the experts
// whose upper end (l + b) reaches L -- at least k of them, and every expert
// of the exact top-k is among them (an expert outside has exact logit < L <=
// the k-th exact logit).  Every warp finds the same candidate list; the warps
// recompute the candidates' logits (and the shared-gate logit) exactly, in
// turn; warp 0 takes the top-k over them (the others at -inf), marks the
// selection bitmap and the token's shared-slot weight.
__global__ void __launch_bounds__(256) k_topk_b(const __grid_constant__ BatchParams P) {
  constexpr int EPL = kBatchMaxE / 32;
  __shared__ float s_ex[kBatchMaxE + 1];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, t = blockIdx.x;
  pdl_launch_dependents();
  pdl_wait();
  const int E = P.E, K = P.K;
  for (int e = tid; e <= E; e += 256) s_ex[e] = -INFINITY;
  // every warp derives the same candidate list (registers; no barrier)
  int cand_n = 0;
  uint32_t cmask[EPL];
  {
    const float* lg = P.logits + (size_t)t * P.ls;
    const float* wn = P.lbound;                                                   // |w_e|_2
    const float xb = __fmul_ru(__ldcg(P.lbound + P.ls + t), (float)(P.H / 32 + 8) * 0x1p-22f);  // (n + 8) 2^-22 |x_t|_2
    // rounding of partial sums in the subnormal range: at most 2^-150 per
    // fused multiply-add, H of them over the warp's lanes
    const float sub_floor = __fmul_ru((float)P.H, 0x1p-149f);
    float hi[EPL];
    uint32_t key[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      const float l = e < E ? __ldcg(lg + e) : 0.f;
      const float b =
          e < E ? __fadd_ru(__fadd_ru(__fmul_ru(__ldcg(wn + e), xb), __fmul_ru(fabsf(l), 0x1p-20f)), sub_floor) : 0.f;
      const float lo = __fsub_rd(l, b);
      hi[i] = __fadd_ru(l, b);
      key[i] = e < E ? float_order_key(lo != lo ? -INFINITY : lo) : 0u;
    }
    // the k-th largest lower end (order keys, one maximum removed per round)
    uint32_t kth = 0u;
    for (int j = 0; j < K; ++j) {
      uint32_t best = 0u, bi = 0xFFFFFFFFu;
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (key[i] > best) {
          best = key[i];
          bi = (uint32_t)(lane + 32 * i);
        }
      const uint32_t m = __reduce_max_sync(0xffffffffu, best);
      const uint32_t win = __reduce_min_sync(0xffffffffu, best == m ? bi : 0xFFFFFFFFu);
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if ((uint32_t)(lane + 32 * i) == win) key[i] = 0u;
      kth = m;
    }
    // candidates: upper end >= L (compared on order keys); ballot masks per slot
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      const bool c = e < E && float_order_key(hi[i] != hi[i] ? INFINITY : hi[i]) >= kth;
      cmask[i] = __ballot_sync(0xffffffffu, c);
      cand_n += __popc(cmask[i]);
    }
  }
  // candidate c (expert order), and c == cand_n the shared-gate logit, on warp c % 8
  for (int c = warp; c <= cand_n; c += 8) {
    int e = E;
    if (c < cand_n) {
      int rem = c;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const int pc = __popc(cmask[i]);
        if (rem >= 0 && rem < pc) {
          uint32_t m = cmask[i];
          for (int q = 0; q < rem; ++q) m &= m - 1u;
          e = 32 * i + __ffs((int)m) - 1;
        }
        rem -= pc;
      }
    }
    const float v = exact_logit(P, t, e);
    if (lane == 0) s_ex[e] = v;
  }
  __syncthreads();
  if (warp == 0) {
    warp_topk<EPL, true>(s_ex, E, K, P.ids + (size_t)t * K, P.p + (size_t)t * K);
    if (lane < K) {
      const int e = P.ids[(size_t)t * K + lane];
      atomicOr(&P.bitmap[(size_t)e * P.tw + (t >> 5)], 1u << (t & 31));
      if (P.topk_ids) P.topk_ids[(size_t)t * K + lane] = e;
      if (P.topk_w) P.topk_w[(size_t)t * K + lane] = P.p[(size_t)t * K + lane];
    }
    if (lane == 0) P.slot_w[(size_t)P.T * K + t] = 1.0f / (1.0f + expf(-s_ex[E]));
  }
  if (P.wfmt == 1) {
    // 4-bit weights: the shared slot's B row (x in fp16, operand order)
    const uint4* src = reinterpret_cast<const uint4*>(P.x + (size_t)t * P.H);
    uint4* dst = reinterpret_cast<uint4*>(P.x_perm + ((size_t)P.T * K + t) * P.H);
    for (int q = tid; q < P.H / 8; q += 256) dst[q] = x8_f16_order(src[q]);
  }
}

// Blocks (e, 0 .. kGatherSplit-1): the expert's count, offset (counts of the
// experts below) and active index; block (e, 0) writes them and the slots of
// its tokens (ascending), their weights and choice indices; every block
// gathers its share of the x rows into x_perm.
__global__ void __launch_bounds__(256) k_bucket_b(const __grid_constant__ BatchParams P) {
  __shared__ int s_red[3][8];
  __shared__ int16_t s_tok[kBatchMaxT];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, e = blockIdx.x, part = blockIdx.y;
  pdl_launch_dependents();
  pdl_wait();
  const uint32_t* row = P.bitmap + (size_t)e * P.tw;
  int cb = 0, nb = 0;
  for (int e2 = tid; e2 < e; e2 += 256) {
    int c = 0;
    for (int w = 0; w < P.tw; ++w) c += __popc(P.bitmap[(size_t)e2 * P.tw + w]);
    cb += c;
    nb += c > 0;
  }
  int mine = 0;
  for (int w = tid; w < P.tw; w += 256) mine += __popc(row[w]);
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    cb += __shfl_xor_sync(0xffffffffu, cb, o);
    nb += __shfl_xor_sync(0xffffffffu, nb, o);
    mine += __shfl_xor_sync(0xffffffffu, mine, o);
  }
  if (lane == 0) {
    s_red[0][warp] = cb;
    s_red[1][warp] = nb;
    s_red[2][warp] = mine;
  }
  __syncthreads();
  int off = 0, ub = 0, cnt = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    off += s_red[0][w];
    ub += s_red[1][w];
    cnt += s_red[2][w];
  }
  if (tid == 0 && part == 0) {
    P.r_counts[e] = cnt;
    P.r_offsets[e] = off;
    if (cnt > 0) P.r_active[ub] = e;
    if (e == P.E - 1) {
      P.r_offsets[P.E] = off + cnt;
      *P.r_nactive = ub + (cnt > 0);
    }
  }
  for (int t = tid; t < P.T; t += 256) {
    const uint32_t wd = row[t >> 5];
    if (wd >> (t & 31) & 1u) {
      int rank = __popc(wd & ((1u << (t & 31)) - 1u));
      for (int w = 0; w < (t >> 5); ++w) rank += __popc(row[w]);
      int k = 0;
      while (k < P.K - 1 && P.ids[(size_t)t * P.K + k] != e) ++k;
      const int slot = off + rank;
      if (part == 0) {
        P.slot_of[(size_t)t * P.K + k] = slot;
        P.slot_w[slot] = P.p[(size_t)t * P.K + k];
        P.r_perm[slot] = t * P.K + k;
      }
      s_tok[rank] = static_cast<int16_t>(t);
    }
  }
  __syncthreads();
  const int chunks = P.H / 8;  // 16-byte chunks of a row
  const int j0 = cnt * part / kGatherSplit, j1 = cnt * (part + 1) / kGatherSplit;
  for (int i = j0 * chunks + tid; i < j1 * chunks; i += 256) {
    const int j = i / chunks, q = i - j * chunks;
    const uint4 v = reinterpret_cast<const uint4*>(P.x + (size_t)s_tok[j] * P.H)[q];
    reinterpret_cast<uint4*>(P.x_perm + (size_t)(off + j) * P.H)[q] = P.wfmt == 1 ? x8_f16_order(v) : v;
  }
}

// out[t] = (sum over the token's choices in rank order of its slot's y) +
// y of its shared slot; 8 columns per thread.
__global__ void __launch_bounds__(256) k_combine_b(const __grid_constant__ BatchParams P) {
  const int t = blockIdx.x;
  pdl_launch_dependents();
  pdl_wait();
  for (int c = 8 * threadIdx.x; c < P.H; c += 8 * 256) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int k = 0; k <= P.K; ++k) {
      const int slot = k < P.K ? P.slot_of[(size_t)t * P.K + k] : P.T * P.K + t;
      const float4* src = reinterpret_cast<const float4*>(P.y_ws + (size_t)slot * P.H + c);
      const float4 a = src[0], b = src[1];
      acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
      acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
    }
    float4* dst = reinterpret_cast<float4*>(P.out + (size_t)t * P.H + c);
    dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

}  // namespace

// Launch behind the previous kernel of the stream with programmatic stream
// serialisation: every kernel of the batched path calls
// griddepcontrol.launch_dependents at entry and griddepcontrol.wait before
// its first access to memory, so only the launch latencies overlap.
template <typename Kern>
static cudaError_t launch_pdl(Kern kern, dim3 grid, int threads, size_t smem, cudaStream_t stream,
                              const BatchParams& p) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

cudaError_t launch_batch(const BatchParams& p, cudaStream_t stream) {
  const size_t route_smem = (size_t)kRouteTokens * p.H * 2;
  if (route_smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(k_route_b, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)route_smem);
    if (e != cudaSuccess) return e;
  }
  cudaError_t err = launch_pdl(k_route_b,
                               dim3((p.T + kRouteTokens - 1) / kRouteTokens, (p.E + 1 + kRouteRows - 1) / kRouteRows),
                               128, route_smem, stream, p);
  if (err == cudaSuccess) err = launch_pdl(k_topk_b, dim3(p.T), 256, 0, stream, p);
  if (err == cudaSuccess) err = launch_pdl(k_bucket_b, dim3(p.E, kGatherSplit), 256, 0, stream, p);
  if (err != cudaSuccess) return err;
  err = p.wfmt == 1 ? launch_gemm_gate_up_q4(p, stream) : launch_gemm_gate_up(p, stream);
  if (err != cudaSuccess) return err;
  err = p.wfmt == 1 ? launch_gemm_down_q4(p, stream) : launch_gemm_down(p, stream);
  if (err != cudaSuccess) return err;
  return launch_pdl(k_combine_b, dim3(p.T), 256, 0, stream, p);
}

}  // namespace moe
