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
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_layer_common.cuh"
#include "moe_rows.cuh"

namespace moe {

cudaError_t launch_gemm_gate_up(const BatchParams& p, cudaStream_t stream);
cudaError_t launch_gemm_down(const BatchParams& p, cudaStream_t stream);

namespace {

constexpr int kRouteTokens = 8;   // tokens per router block
constexpr int kRouteRows = 8;     // router rows per block (1 per warp)
constexpr int kGatherSplit = 4;   // blocks per expert in the bucketing kernel

// Router logits, error-free accumulated as in the decode router: the
// products of bf16 weights and bf16 activations are exact in fp32, their
// sum is kept as a (sum, compensation) pair and rounded once.  Block
// (token group, row group): 8 warps x 1 row x 8 tokens.  The first block
// also clears the control words and every block a share of the bitmap.
__global__ void __launch_bounds__(256) k_route_b(const __grid_constant__ BatchParams P) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nblk = gridDim.x * gridDim.y, bid = blockIdx.y * gridDim.x + blockIdx.x;
  for (int i = bid * 256 + tid; i < P.E * P.tw; i += nblk * 256) P.bitmap[i] = 0u;
  if (bid == 0 && tid < kCtrlWords) P.ctrl[tid] = 0u;
  const int t0 = blockIdx.x * kRouteTokens;
  constexpr int RPW = kRouteRows / 8;  // rows per warp
  const int r0 = blockIdx.y * kRouteRows + RPW * warp;
  const uint16_t* w[RPW];
#pragma unroll
  for (int j = 0; j < RPW; ++j) {
    const int r = r0 + j;
    w[j] = r < P.E ? P.router_w + (size_t)r * P.H : (r == P.E ? P.gate_w : nullptr);
  }
  float s[RPW][kRouteTokens], c[RPW][kRouteTokens];
#pragma unroll
  for (int j = 0; j < RPW; ++j)
#pragma unroll
    for (int t = 0; t < kRouteTokens; ++t) s[j][t] = c[j][t] = 0.f;
  for (int c0 = lane * 8; c0 < P.H; c0 += 256) {
    float wf[RPW][8];
#pragma unroll
    for (int j = 0; j < RPW; ++j) {
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (w[j]) v = *reinterpret_cast<const uint4*>(w[j] + c0);
      wf[j][0] = bf16_lo(v.x); wf[j][1] = bf16_hi(v.x); wf[j][2] = bf16_lo(v.y); wf[j][3] = bf16_hi(v.y);
      wf[j][4] = bf16_lo(v.z); wf[j][5] = bf16_hi(v.z); wf[j][6] = bf16_lo(v.w); wf[j][7] = bf16_hi(v.w);
    }
#pragma unroll
    for (int t = 0; t < kRouteTokens; ++t) {
      if (t0 + t >= P.T) break;
      const uint4 xv = *reinterpret_cast<const uint4*>(P.x + (size_t)(t0 + t) * P.H + c0);
      const float xf[8] = {bf16_lo(xv.x), bf16_hi(xv.x), bf16_lo(xv.y), bf16_hi(xv.y),
                           bf16_lo(xv.z), bf16_hi(xv.z), bf16_lo(xv.w), bf16_hi(xv.w)};
#pragma unroll
      for (int j = 0; j < RPW; ++j)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          float tt, e2;
          two_sum(s[j][t], __fmul_rn(wf[j][e], xf[e]), tt, e2);
          s[j][t] = tt;
          c[j][t] = __fadd_rn(c[j][t], e2);
        }
    }
  }
#pragma unroll
  for (int j = 0; j < RPW; ++j)
#pragma unroll
    for (int t = 0; t < kRouteTokens; ++t) {
      warp_sum2(s[j][t], c[j][t]);
      if (lane == 0 && w[j] && t0 + t < P.T) P.logits[(size_t)(t0 + t) * P.ls + r0 + j] = __fadd_rn(s[j][t], c[j][t]);
    }
}

// Top-k of token t on warp t % 8 of block t / 8; the chosen experts' bits in
// the selection bitmap and the shared-gate weight of the token's shared slot.
__global__ void __launch_bounds__(256) k_topk_b(const __grid_constant__ BatchParams P) {
  const int lane = threadIdx.x & 31, t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= P.T) return;
  const float* lg = P.logits + (size_t)t * P.ls;
  float sl = 0.f;
  if (lane == 0) sl = __ldcg(lg + P.E);
  warp_topk<kBatchMaxE / 32>(lg, P.E, P.K, P.ids + (size_t)t * P.K, P.p + (size_t)t * P.K);
  if (lane < P.K) {
    const int e = P.ids[(size_t)t * P.K + lane];
    atomicOr(&P.bitmap[(size_t)e * P.tw + (t >> 5)], 1u << (t & 31));
    if (P.topk_ids) P.topk_ids[(size_t)t * P.K + lane] = e;
    if (P.topk_w) P.topk_w[(size_t)t * P.K + lane] = P.p[(size_t)t * P.K + lane];
  }
  if (lane == 0) P.slot_w[(size_t)P.T * P.K + t] = 1.0f / (1.0f + expf(-sl));
}

// Blocks (e, 0 .. kGatherSplit-1): the expert's count, offset (counts of the
// experts below) and active index; block (e, 0) writes them and the slots of
// its tokens (ascending), their weights and choice indices; every block
// gathers its share of the x rows into x_perm.
__global__ void __launch_bounds__(256) k_bucket_b(const __grid_constant__ BatchParams P) {
  __shared__ int s_red[3][8];
  __shared__ int16_t s_tok[kBatchMaxT];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, e = blockIdx.x, part = blockIdx.y;
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
    reinterpret_cast<uint4*>(P.x_perm + (size_t)(off + j) * P.H)[q] =
        reinterpret_cast<const uint4*>(P.x + (size_t)s_tok[j] * P.H)[q];
  }
}

// out[t] = (sum over the token's choices in rank order of its slot's y) +
// y of its shared slot; 8 columns per thread.
__global__ void __launch_bounds__(256) k_combine_b(const __grid_constant__ BatchParams P) {
  const int t = blockIdx.x;
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

cudaError_t launch_batch(const BatchParams& p, cudaStream_t stream) {
  k_route_b<<<dim3((p.T + kRouteTokens - 1) / kRouteTokens, (p.E + 1 + kRouteRows - 1) / kRouteRows), 256, 0, stream>>>(p);
  k_topk_b<<<(p.T + 7) / 8, 256, 0, stream>>>(p);
  k_bucket_b<<<dim3(p.E, kGatherSplit), 256, 0, stream>>>(p);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  err = launch_gemm_gate_up(p, stream);
  if (err != cudaSuccess) return err;
  err = launch_gemm_down(p, stream);
  if (err != cudaSuccess) return err;
  k_combine_b<<<p.T, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
