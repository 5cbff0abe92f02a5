#pragma once
// Row kernel of the fused MoE FFN layer (decode path, T <= 8), sm_103a: the
// whole layer in one kernel per call.  Instantiated by the moe_rows_*.cu
// units.
//
// Work unit: one intermediate index i of one expert group (the shared expert,
// or a routed expert selected by some token).  Its weights are three
// contiguous stored rows of H elements -- gate row i, up row i and row i of
// the transposed down matrix -- and it contributes
//     y_t += w_t * silu(gate_i . x_t) * (up_i . x_t) * downT_i
// to every token t the group serves (w_t = the routing weight p, or the
// shared-expert gate s).  A block owns a contiguous run of units, so it needs
// nothing from other blocks but the routing until its partial y is complete.
//
// One persistent block of 8 warps (16 for the 4-bit and int8 tensor-core
// loops) per SM (G blocks).  Before the wait on the
// previous kernel (programmatic dependent launch; nothing produced by it is
// read), each block loads its router row and issues the shared expert's
// first stages -- weights are never written by a kernel that lets this one
// start early.  After the wait:
//   1. x (block form: x_res, and its RMSNorm factors) into shared memory;
//   2. router: block c computes the logits of router row c (row E: the
//      shared-gate vector) for all tokens with error-free sums, writes them
//      and announces them (first grid-wide barrier);
//   3. every block reads all logits, takes the top-k of each token (ties to
//      the lower index) and the softmax weights, builds the active-expert
//      tables, and issues its routed stages;
//   4. stages: weights stream through a ring of `ns` stages of `rs` units
//      (tensor copies issued by one thread on one mbarrier).  Per stage:
//        A  the gate and up dot products of the stage's rows for all tokens
//           (warp partials), then one block barrier;
//        A2 h_t = w_t silu(g_t) u_t of each row from the warp partials;
//        C  y[cols][tokens] += downT_r^T h over the stage's rows;
//   5. end: each block stores its partial y[T][H] (fp32) and announces it
//      (second grid-wide barrier; with one token the partials are words
//      tagged with the call instead, polled by their readers); then each block sums
//      the G partials of its own output columns in block order and writes
//      out (adding x_res in the block form).  All orders are fixed, so
//      results are bitwise repeatable.
// The grid-wide barriers use per-block flag slots tagged with the call's
// epoch (RowSync), so no workspace word has to be reset between calls.
//
// Tensor-core instances (H = 2048, bf16-exact activation): the stage loops
// run on mma.m16n8k16 over the swizzled tensor-copy boxes, one
// block barrier per stage.  With 4-bit weights each code becomes the exact
// bf16 (code - 8) in registers (the nibble OR-ed into the mantissa of bf16
// 128 reads 128 + n, minus 136), the products of a 32-element block are
// summed on the tensor cores and scaled by the block's fp16 scale in fp32, so
// no weight is rounded.  With int8 weights the activation is quantised per
// token and the codes of both operands enter fp16 products exactly, so the
// gate and up dot products are exact integers.  The 4-bit and int8 blocks
// have 16 warps: warps 0..7 run the whole path except the down projection
// of the stages, which warps 8..15 run beside them (rows_threads).  The
// general instance decodes every weight to fp32 and uses CUDA-core FMAs
// (int8: int32 dp4a).

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <cstddef>
#include <mutex>
#include <type_traits>

#include "moe_layer_common.cuh"

namespace moe {

enum : int { kXReg = 0, kXF32 = 1 };
constexpr int kMaxStagesRing = 8;
constexpr int kBarStage = 1;  // named barrier of the compute warps, once per stage
constexpr int kRsMaxB16 = 4;  // rows per stage, bf16 weights
constexpr int kRsMaxQ4 = 8;   // rows per stage, 4-bit and int8 weights
enum : int { kWkBf16 = 0, kWkQ4 = 1, kWkI8 = 2 };  // weight kinds (the plan's wfmt)

// Routing tables of one block, carved from shared memory with sizes of the
// plan (T tokens, K per token, E experts).
struct RowTab {
  int32_t* ids;      // [T*K] chosen experts, rank order
  float* p;          // [T*K] their weights
  float* s;          // [T] shared-expert gate sigmoid(g . x_t)
  float* inv;        // [2T] block form: RMSNorm factor hi, lo
  uint32_t* bitmap;  // [ceil(E/32)] selected experts
  int16_t* inv_u;    // [E] active index of a selected expert
  int32_t* active;   // [T*K] selected experts, ascending
  uint32_t* mask;    // [T*K] tokens of active expert u (bit t)
  float* wt;         // [T*K][T] weight of token t for active expert u (0 if not routed)
  int32_t* misc;     // [8] the number of active experts U; (split blocks) n_stages, first routed stage, call tag
  int32_t* qtab;     // [T*K - K + 1][4] per possible U: routed stages, first active expert, first group
  uint32_t* xmax;    // [T] int8 activation: bits of max |x| of token t
  float* xsc;        // [T] int8 activation: x_scale = max|x| / 127 of token t
};

__host__ __device__ inline int row_tab(uint8_t* base, int T, int K, int E, RowTab* v) {
  const int TK = T * K;
  const int sz[13] = {TK * 4, TK * 4, T * 4, 2 * T * 4, ((E + 31) / 32) * 4, E * 2, TK * 4, TK * 4, TK * T * 4, 8 * 4,
                      (TK - K + 1) * 16, T * 4, T * 4};
  int off = 0, o[13];
  for (int i = 0; i < 13; ++i) {
    o[i] = off;
    off += (sz[i] + 15) & ~15;
  }
  if (v && base) {
    v->ids = reinterpret_cast<int32_t*>(base + o[0]);
    v->p = reinterpret_cast<float*>(base + o[1]);
    v->s = reinterpret_cast<float*>(base + o[2]);
    v->inv = reinterpret_cast<float*>(base + o[3]);
    v->bitmap = reinterpret_cast<uint32_t*>(base + o[4]);
    v->inv_u = reinterpret_cast<int16_t*>(base + o[5]);
    v->active = reinterpret_cast<int32_t*>(base + o[6]);
    v->mask = reinterpret_cast<uint32_t*>(base + o[7]);
    v->wt = reinterpret_cast<float*>(base + o[8]);
    v->misc = reinterpret_cast<int32_t*>(base + o[9]);
    v->qtab = reinterpret_cast<int32_t*>(base + o[10]);
    v->xmax = reinterpret_cast<uint32_t*>(base + o[11]);
    v->xsc = reinterpret_cast<float*>(base + o[12]);
  }
  return off;
}

// ------------------------------------------------------------ 4-bit helpers
MOE_DEV uint32_t lop3_and_or(uint32_t a, uint32_t m, uint32_t c) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(m), "r"(c));
  return r;
}
// Code n of nibble j of a 32-bit word, as the float n - 8 (exact: the
// nibble OR-ed into the mantissa of 2^23 reads 2^23 + n).
MOE_DEV float nib_f32(uint32_t w, int j) {
  return __fsub_rn(__uint_as_float(0x4B000000u | ((w >> (4 * j)) & 0xFu)), 8388616.0f);
}
// Signed byte j of a 32-bit word as a float (exact: the byte with its sign
// bit flipped, c + 128 in 0..255, placed in the mantissa of 2^23 reads
// 2^23 + c + 128).
MOE_DEV float i8_f32(uint32_t w, int j) {
  return __fsub_rn(__uint_as_float(__byte_perm(w ^ 0x80808080u, 0x4B000000u, 0x7540u + j)), 8388736.0f);
}

// v[0..7] per lane -> the warp sum of v[(lane >> 2) & 7], in every lane of the
// group of four lanes 4i .. 4i+3 (9 shuffles, 5 levels).
MOE_DEV float warp_reduce8(const float* v) {
  const int l = threadIdx.x & 31;
  const bool b4 = l & 16, b3 = l & 8, b2 = l & 4;
  float n4[4], n2[2];
#pragma unroll
  for (int j = 0; j < 4; ++j) n4[j] = (b4 ? v[j + 4] : v[j]) + __shfl_xor_sync(0xffffffffu, b4 ? v[j] : v[j + 4], 16);
#pragma unroll
  for (int j = 0; j < 2; ++j) n2[j] = (b3 ? n4[j + 2] : n4[j]) + __shfl_xor_sync(0xffffffffu, b3 ? n4[j] : n4[j + 2], 8);
  float r = (b2 ? n2[1] : n2[0]) + __shfl_xor_sync(0xffffffffu, b2 ? n2[0] : n2[1], 4);
  r += __shfl_xor_sync(0xffffffffu, r, 2);
  r += __shfl_xor_sync(0xffffffffu, r, 1);
  return r;
}

// Top-k of one token's E logits by one warp.  Each lane holds the order keys
// of experts lane + 32 i (i < EPL); K rounds take the warp maximum (hardware
// reduction) and, among lanes holding it, the lowest expert index, so equal
// logits go to the lower index.  NaN ranks as -inf.  ids[0..K) in rank
// order; pout = softmax over the K chosen logits.  E <= 32 * EPL, K <= 32.
template <int EPL, bool SMEM = false>
MOE_DEV void warp_topk(const float* lg, int E, int K, int32_t* ids, float* pout) {
  const int lane = threadIdx.x & 31;
  uint32_t key[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    float v = e < E ? (SMEM ? lg[e] : __ldcg(lg + e)) : 0.f;
    v = v != v ? -INFINITY : v;
    key[i] = e < E ? float_order_key(v) : 0u;  // every real key is >= key(-inf) > 0
  }
  int myid = 0;
  uint32_t mykey = 0u;
  for (int j = 0; j < K; ++j) {
    uint32_t best = 0u;
    uint32_t bi = 0xFFFFFFFFu;
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
    if (lane == j) {
      myid = (int)win;
      mykey = m;
    }
  }
  // the chosen logit back from its order key (the key map is a bijection)
  const float lj = lane < K ? __uint_as_float((mykey & 0x80000000u) ? (mykey & 0x7FFFFFFFu) : ~mykey) : 0.f;
  const float l0 = __shfl_sync(0xffffffffu, lj, 0);
  const float z = lane < K ? expf(lj - l0) : 0.f;
  const float sum = warp_sum(z);
  if (lane < K) {
    ids[lane] = myid;
    pout[lane] = z / sum;
  }
}

// Eight activations of one row, columns c0 .. c0+7 (c0 % 8 == 0), from the
// shared-memory copy of x: fp32 rows (src4; in the block form the
// normalised bf16 value of x_res, factor hi + lo) or bf16 rows.
MOE_DEV void x8_from_smem(const uint8_t* row, int src4, int block_mode, float hi, float lo, int c0, float* xf) {
  if (src4) {
    const float4* p = reinterpret_cast<const float4*>(row + (size_t)c0 * 4);
    const float4 a = p[0], b = p[1];
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) xf[e] = block_mode ? norm_apply(v[e], hi, lo) : v[e];
  } else {
    const uint4 v = *reinterpret_cast<const uint4*>(row + (size_t)c0 * 2);
    xf[0] = bf16_lo(v.x); xf[1] = bf16_hi(v.x); xf[2] = bf16_lo(v.y); xf[3] = bf16_hi(v.y);
    xf[4] = bf16_lo(v.z); xf[5] = bf16_hi(v.z); xf[6] = bf16_lo(v.w); xf[7] = bf16_hi(v.w);
  }
}

// Two activations of one row, columns c0, c0+1 (c0 even), as x8_from_smem.
MOE_DEV void x2_from_smem(const uint8_t* row, int src4, int block_mode, float hi, float lo, int c0, float* xf) {
  if (src4) {
    const float2 a = *reinterpret_cast<const float2*>(row + (size_t)c0 * 4);
    xf[0] = block_mode ? norm_apply(a.x, hi, lo) : a.x;
    xf[1] = block_mode ? norm_apply(a.y, hi, lo) : a.y;
  } else {
    const uint32_t v = *reinterpret_cast<const uint32_t*>(row + (size_t)c0 * 2);
    xf[0] = bf16_lo(v);
    xf[1] = bf16_hi(v);
  }
}
// bf16 pair of two bf16-exact floats (their upper halves), a low.
MOE_DEV uint32_t bf16_pair_exact(float a, float b) { return (__float_as_uint(a) >> 16) | (__float_as_uint(b) & 0xFFFF0000u); }

// ------------------------------------------------------------ tensor cores
// D += A B, m16n8k16, bf16 operands, fp32 accumulators (A row-major 16x16,
// B column-major 16x8), fragments as in the PTX ISA for mma.m16n8k16.
MOE_DEV void mma_bf16(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Two 4-bit codes (bits 0-3 and 16-19 of v) -> the bf16 pair (code - 8):
// 0x4300 | n is the bf16 of 128 + n, and 128 + n - 136 is exact.
MOE_DEV uint32_t q4_pair_bf16(uint32_t v) {
  uint32_t r;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(lop3_and_or(v, 0x000F000Fu, 0x43004300u)), "r"(0x43084308u));
  return r;
}
// Scale k (0..7) of the 8 fp16 values in a 16-byte unit, as a float.
MOE_DEV float half_at(const uint4& v, int k) {
  const uint32_t w = k < 2 ? v.x : k < 4 ? v.y : k < 6 ? v.z : v.w;
  return __half2float(__ushort_as_half(static_cast<unsigned short>((k & 1) ? (w >> 16) : (w & 0xFFFFu))));
}
// Four 8x8 b16 matrices, transposed, from the shared-memory row address this
// lane supplies (lanes 8q .. 8q+7 give the 8 rows of matrix q).
MOE_DEV void ldmatrix_x4_trans(uint32_t* r, const void* row) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(row)));
}
// Four 8x8 b16 matrices from the shared-memory row address this lane
// supplies (lanes 8q .. 8q+7 give the 8 rows of matrix q): lane l gets
// 32-bit element (l / 4, l % 4) of each matrix.
MOE_DEV void ldmatrix_x4(uint32_t* r, const void* row) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(row)));
}
// D += A B, m16n8k16, fp16 operands, fp32 accumulators (fragments as for
// mma_bf16).
MOE_DEV void mma_f16(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Signed bytes 2j and 2j + 1 of a 32-bit word -> the fp16 pair of their
// values, exactly: the byte with its sign bit flipped, u = c + 128, as the
// low byte of fp16 0x6400 (1024) reads 1024 + u, and 1024 + u - 1152 = c.
MOE_DEV uint32_t i8_pair_f16(uint32_t w, int j) {
  const uint32_t v = __byte_perm(w ^ 0x80808080u, 0x64646464u, j ? 0x5342u : 0x5140u);
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(0x64806480u));
  return r;
}
// Byte offset of bf16 element k (even) of a row in a box stored as
// [H/64 chunks][rows][64 elements] with the 128-byte swizzle of the tensor
// copies: line L = chunk * rows + row, 16-byte unit (k / 8) % 8 at unit
// ((k / 8) % 8) ^ (L % 8).
MOE_DEV int swz_off(int line, int k) { return line * 128 + ((((k >> 3) & 7) ^ (line & 7)) << 4) + ((k & 7) << 1); }

// Two floats -> bf16 pair (round to nearest even), low element first.
MOE_DEV uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

MOE_DEV float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// floor(a * b / d) for the block partitions; 32-bit division when a * b fits.
MOE_DEV uint32_t muldiv(uint32_t a, uint32_t b, uint32_t d) {
  if (__umulhi(a, b) == 0u) return (a * b) / d;
  return (uint32_t)(((unsigned long long)a * b) / d);
}

// Walks the stages of a block in order without divisions.  Stage k < n_sh
// is shared group k (counted from the block's first); stage n_sh is routed
// group g0 of active expert u0, and later stages follow group by group
// (gI groups per expert).  slot / ph: the ring slot of the stage and the
// parity of its use of that slot.
struct StageCursor {
  int k, u, g, slot;
  uint32_t ph;
};
MOE_DEV void cursor_init(StageCursor& c, int ns) {
  c.k = -1;
  c.u = -1;
  c.g = 0;
  c.slot = ns - 1;
  c.ph = 1u;
}
MOE_DEV void cursor_next(StageCursor& c, int n_sh, int u0, int g0, int gI, int ns) {
  ++c.k;
  if (c.k < n_sh) {
    c.u = -1;
    c.g = c.k;
  } else if (c.k == n_sh) {
    c.u = u0;
    c.g = g0;
  } else if (++c.g == gI) {
    ++c.u;
    c.g = 0;
  }
  if (++c.slot == ns) {
    c.slot = 0;
    c.ph ^= 1u;
  }
}

// Threads of a row-kernel block.  The 4-bit and int8 tensor-core instances
// run 8 more warps that do only the stage loop's down projection (warps
// 8..15), so that it runs beside the gate/up products of the first 8 warps.
__host__ __device__ constexpr int rows_threads(int wk, bool fast) { return fast && wk != kWkBf16 ? 2 * kRowThreads : kRowThreads; }
constexpr int kBarSplit = 3;  // named barrier: main and down-projection warps meet (start and end of the stages)

// ------------------------------------------------------------------- kernel
// TMAX: token capacity (T <= TMAX).  WK: weight kind (kWkBf16, kWkQ4,
// kWkI8).  FAST: H = 2048, E <= 256 and a bf16-exact activation (the
// tensor-core loops; bf16 and 4-bit weights).
template <int TMAX, int WK, bool FAST, int NCH>
__global__ void __maxnreg__(rows_threads(WK, FAST) > kRowThreads ? 128 : 224) k_rows(const __grid_constant__ LayerParams Pk) {
  constexpr bool Q4 = WK == kWkQ4;
  constexpr bool I8 = WK == kWkI8;              // int8 weights and activation
  constexpr bool B16C = FAST && WK == kWkBf16;  // bf16 tensor-core loop
  constexpr bool MMA_C = B16C && TMAX >= 4;     // bf16: tensor-core down projection
  constexpr bool Q4C = FAST && Q4;              // 4-bit tensor-core loop
  constexpr bool I8C = FAST && I8;              // int8 tensor-core loop
  constexpr bool QMC = Q4C || I8C;              // the 8-row down projection (yc4 accumulators)
  // QMC: warps 8..15 do the down projection of every stage (see rows_threads)
  constexpr int NTB = rows_threads(WK, FAST);             // threads of the block
  constexpr int SYNC_NT = NTB > kRowThreads ? kRowThreads : 0;  // block barriers of warps 0..7 (blk_sync)
  // One token: the partial outputs are words tagged with the call, polled by
  // the column sums (no second grid-wide barrier; see RowSync)
  constexpr bool TAGGED = TMAX == 1;
  static_assert(NCH == 1 || (NCH == 2 && !FAST), "8-column chunks per thread: 1, or 2 for H > 2048");
  constexpr int EPL = FAST ? 8 : 32;         // top-k keys per lane
  extern __shared__ __align__(128) uint8_t sm[];
  // The parameter block is read in place (parameter space).  The set-up work
  // before the wait on the previous kernel is split over the warps so that
  // its pieces -- each short, and each first executed cold on every call --
  // run side by side rather than one after the other.
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cta = blockIdx.x;
  const LayerParams& P = Pk;
  const int T = P.T, K = P.K, TK = T * K;
  const int H = FAST ? 2048 : P.H;
  const int RS = P.rs, NS = P.ns;
  const long long rb = P.rb;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + P.off_bar);
  uint64_t* xbar = full + kMaxStagesRing;       // the activation copy
  uint64_t* fulld = full + kMaxStagesRing + 1;  // [nsd] tensor-core path: downT boxes
  int* scnt = reinterpret_cast<int*>(sm + P.off_bar + 160);  // [NS] warps that have read a stage's slot
  RowTab tb;
  row_tab(sm + P.off_tab, T, K, P.E, &tb);
  uint8_t* xs = sm + P.off_x;
  // The ring starts on a 1024-byte boundary of the shared window (the
  // 128-byte swizzle of the tensor copies follows absolute address bits);
  // the layout reserves the slack.
  const uint32_t ring_pad = (1024u - (smem_u32(sm + P.off_ring) & 1023u)) & 1023u;
  uint8_t* ring = sm + P.off_ring + ring_pad;
  uint8_t* dring = sm + P.off_dring + ring_pad;  // tensor-core path: downT boxes
  const uint64_t pol = policy_evict_first();

  // The next kernel of the stream (the next call's row kernel) may start its
  // blocks as soon as this kernel's blocks leave an SM.
  pdl_launch_dependents();

  // Units of this block: groups of RS consecutive rows of one expert (the
  // last group of an expert may be shorter).  Shared groups [gs0, gs1) are
  // known now; the routed groups are the run [q0, q1) of the flattened
  // (active expert u, group) order, known after the routing and sized so
  // that shared + routed groups (stages) are balanced over the blocks.
  const int gS = P.part == 1 ? 0 : (P.Is + RS - 1) / RS, gI = (P.I + RS - 1) / RS;
  const int gs0 = (int)muldiv(gS, cta, P.G), gs1 = (int)muldiv(gS, cta + 1, P.G);
  const int n_sh = gs1 - gs0;
  int n_stages = n_sh;
  int ur0 = 0, gr0 = 0;  // first routed stage: active expert, group in it

  const uint8_t* const r_expert_w = P.expert_w;
  const uint8_t* const r_shexp_w = P.shexp_w;
  const long long r_expert_bytes = P.expert_bytes;
  const long long r_mat = (long long)P.I * rb, r_smat = (long long)P.Is * rb;
  const int r_I = P.I, r_Is = P.Is, r_stage_bytes = P.stage_bytes;
  const long long rp = P.rp;
  // first row and row count of the stage a cursor stands on
  auto rows_of = [&](const StageCursor& c, int& i0, int& n) {
    if (c.u < 0) {
      i0 = (gs0 + c.g) * RS;
      n = min(RS, r_Is - i0);
    } else {
      i0 = c.g * RS;
      n = min(RS, r_I - i0);
    }
  };
  auto advance = [&](StageCursor& c, int ns) { cursor_next(c, n_sh, ur0, gr0, gI, ns); };
  // Tensor-core path: the downT box of a stage into its own ring (int8: the
  // codes, then the rows' scale records).
  auto issue_d = [&](const StageCursor& c) {
    int i0, n;
    rows_of(c, i0, n);
    const int e = c.u < 0 ? 0 : tb.active[c.u];
    const void* dm = c.u < 0 ? (const void*)&Pk.tm_d_s : (const void*)&Pk.tm_d_e;
    uint8_t* dst = dring + (size_t)c.slot * P.dstage_bytes;
    if constexpr (I8) {
      const void* dsc = c.u < 0 ? (const void*)&Pk.tm_dsc_s : (const void*)&Pk.tm_dsc_e;
      mbar_arrive_expect_tx(&fulld[c.slot], (uint32_t)(RS * H + RS * 16));
      tma_load_5d(dst, dm, 0, i0, 2, 0, e, &fulld[c.slot], pol);
      tma_load_5d(dst + (size_t)RS * H, dsc, 0, i0, 2, e, 0, &fulld[c.slot], pol);
    } else {
      mbar_arrive_expect_tx(&fulld[c.slot], (uint32_t)(RS * rb));
      tma_load_5d(dst, dm, 0, i0, 2, 0, e, &fulld[c.slot], pol);
    }
  };
  // One thread issues a stage.  Tensor-core path: one tiled tensor copy of
  // the stage's gate + up rows (a whole box; rows past the matrix are
  // zero-filled and unused).  Otherwise three bulk copies of the n rows of
  // each matrix.
  auto issue = [&](const StageCursor& c) {
    uint8_t* dst = ring + (size_t)c.slot * r_stage_bytes;
    uint64_t* bar = &full[c.slot];
    int i0, n;
    rows_of(c, i0, n);
    if constexpr (FAST) {
      const int e = c.u < 0 ? 0 : tb.active[c.u];
      const void* gu = c.u < 0 ? (const void*)&Pk.tm_gu_s : (const void*)&Pk.tm_gu_e;
      if constexpr (I8) {
        const void* gsc = c.u < 0 ? (const void*)&Pk.tm_gusc_s : (const void*)&Pk.tm_gusc_e;
        mbar_arrive_expect_tx(bar, (uint32_t)(2 * RS * H + 2 * RS * 16));
        tma_load_5d(dst, gu, 0, i0, 0, 0, e, bar, pol);
        tma_load_5d(dst + (size_t)2 * RS * H, gsc, 0, i0, 0, e, 0, bar, pol);
      } else {
        mbar_arrive_expect_tx(bar, (uint32_t)r_stage_bytes);
        tma_load_5d(dst, gu, 0, i0, 0, 0, e, bar, pol);
      }
    } else {
      const uint8_t* src;
      long long mat;
      if (c.u < 0) {
        src = r_shexp_w + (long long)i0 * rb;
        mat = r_smat;
      } else {
        src = r_expert_w + (long long)tb.active[c.u] * r_expert_bytes + (long long)i0 * rb;
        mat = r_mat;
      }
      const uint32_t bytes = (uint32_t)(n * rb);
      mbar_arrive_expect_tx(bar, 3 * bytes);
      bulk_g2s(dst, src, bytes, bar, pol);
      bulk_g2s(dst + (size_t)RS * rp, src + mat, bytes, bar, pol);
      bulk_g2s(dst + (size_t)2 * RS * rp, src + 2 * mat, bytes, bar, pol);
    }
  };
  // Issue cursors (main ring, downT ring): every thread advances them in
  // step so that any thread can issue.
  StageCursor ci, cd;
  cursor_init(ci, NS);
  cursor_init(cd, P.nsd > 0 ? P.nsd : 1);

  if constexpr (NTB > kRowThreads) {
    if (warp >= kRowWarps) {
      // ---- warps 8..15: the down projection of every stage.  Warp 8 + w
      // owns the 256-column slice [256w, 256w + 256) of H.  They wait at
      // kBarSplit until warps 0..7 have routed the call and issued the first
      // copies, then meet them at the stage barrier n_stages + 1 times: after
      // barrier s they refill the downT slot of stage s - 2 and project stage
      // s - 1 with the h that A2 formed for it (h by stage parity).  At the
      // end they store their partial y and meet warps 0..7 at kBarSplit once
      // more (the OR of every wait's time-out).
      const int w = warp - kRowWarps, gq = lane >> 2, qq = lane & 3;
      const float* hb = reinterpret_cast<const float*>(sm + P.off_h);  // [2][kRsMaxQ4][TMAX]
      bool h_timed_out = false;
      named_bar_sync(kBarSplit, NTB);
      n_stages = tb.misc[1];
      ur0 = tb.misc[2];
      gr0 = tb.misc[3];
      const uint32_t tag = static_cast<uint32_t>(tb.misc[4]);
      const uint64_t pol_keep = policy_evict_last();
      for (int k = 0; k < min(n_stages, P.nsd); ++k) advance(cd, P.nsd);  // the copies warps 0..7 issued
      StageCursor cc;  // the stage being projected
      cursor_init(cc, 1);
      int dslot = P.nsd - 1;  // its downT ring slot and phase parity
      uint32_t dph = 1u;
      float yc4[16][4];  // y of this warp's slice, D fragments (tiles 2b + i)
#pragma unroll
      for (int j = 0; j < 16; ++j) yc4[j][0] = yc4[j][1] = yc4[j][2] = yc4[j][3] = 0.f;
      for (int s = 0; s <= n_stages; ++s) {
        named_bar_sync(kBarStage, NTB);
        // C of stage s - 2 ended before this barrier: its downT slot is free
        if (s >= 2 && s - 2 + P.nsd < n_stages) {
          advance(cd, P.nsd);
          if (tid == NTB - 1) issue_d(cd);
        }
        if (s == 0) continue;
        advance(cc, 1);
        int i0c, n_prev;
        rows_of(cc, i0c, n_prev);
        if (++dslot == P.nsd) {
          dslot = 0;
          dph ^= 1u;
        }
        if (!mbar_wait(&fulld[dslot], dph)) h_timed_out = true;
        const uint8_t* dbox = dring + (size_t)dslot * P.dstage_bytes;
        const float* hp = hb + ((s - 1) & 1) * kRsMaxQ4 * TMAX;
        // B: h times the row's scale for rows 2q, 2q + 1 (k) and token lane/4
        // (n), as bf16 hi (k 0..7) + lo (k 8..15), so y keeps fp32 accuracy;
        // A: the codes of the same rows, exact in bf16.  Tile i of the
        // 32-column block b holds columns 32b + 4g + 2i (A rows g) and + 1
        // (rows g + 8) of the slice: this lane reads the 4 codes at 32b + 4g
        // of rows 2q and 2q + 1, two tiles' worth.
        const float h0 = (2 * qq < n_prev && gq < TMAX) ? hp[(2 * qq) * TMAX + gq] : 0.f;
        const float h1 = (2 * qq + 1 < n_prev && gq < TMAX) ? hp[(2 * qq + 1) * TMAX + gq] : 0.f;
        if constexpr (Q4) {
          // box lines: chunk * 8 + row; chunk 8 holds the rows' block scales
          const int l0 = 8 * kRsMaxQ4 + 2 * qq;
          const uint4 s0 = *reinterpret_cast<const uint4*>(dbox + l0 * 128 + ((w ^ (l0 & 7)) << 4));
          const uint4 s1 = *reinterpret_cast<const uint4*>(dbox + (l0 + 1) * 128 + ((w ^ ((l0 + 1) & 7)) << 4));
          const int lr = w * kRsMaxQ4 + 2 * qq;  // nibble chunk w, row 2q
          const uint8_t* r0p = dbox + lr * 128 + 2 * gq;
          const uint8_t* r1p = dbox + (lr + 1) * 128 + 2 * gq;
#pragma unroll
          for (int b = 0; b < 8; ++b) {
            const float v0 = h0 * half_at(s0, b), v1 = h1 * half_at(s1, b);
            const uint32_t bh = pack_bf16(v0, v1);
            const uint32_t bl = pack_bf16(v0 - bf16_lo(bh), v1 - bf16_hi(bh));
            // codes of rows 2q, 2q + 1 at columns 32b + 4g .. + 3 of the slice
            const uint32_t u0 = *reinterpret_cast<const uint16_t*>(r0p + ((b ^ (lr & 7)) << 4));
            const uint32_t u1 = *reinterpret_cast<const uint16_t*>(r1p + ((b ^ ((lr + 1) & 7)) << 4));
            const uint32_t X = u0 | (u1 << 16);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const uint32_t a0 = q4_pair_bf16(X >> (8 * i)), a1 = q4_pair_bf16(X >> (8 * i + 4));
              mma_bf16(yc4[2 * b + i], a0, a1, a0, a1, bh, bl);
            }
          }
        } else {
          // box lines: chunk * 8 + row (16 chunks of codes), then the rows'
          // 16-byte scale records
          const float v0 = h0 * *reinterpret_cast<const float*>(dbox + (size_t)RS * H + (size_t)(2 * qq) * 16);
          const float v1 = h1 * *reinterpret_cast<const float*>(dbox + (size_t)RS * H + (size_t)(2 * qq + 1) * 16);
          const uint32_t bh = pack_bf16(v0, v1);
          const uint32_t bl = pack_bf16(v0 - bf16_lo(bh), v1 - bf16_hi(bh));
#pragma unroll
          for (int b = 0; b < 8; ++b) {
            const int chunk = 2 * w + (b >> 2), unit = 2 * (b & 3) + (gq >> 2), off = 4 * (gq & 3);
            const int l0 = chunk * RS + 2 * qq;  // line & 7 = the row
            const uint32_t w0 = *reinterpret_cast<const uint32_t*>(dbox + (size_t)l0 * 128 + ((unit ^ (l0 & 7)) << 4) + off);
            const uint32_t w1 =
                *reinterpret_cast<const uint32_t*>(dbox + (size_t)(l0 + 1) * 128 + ((unit ^ ((l0 + 1) & 7)) << 4) + off);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              // (row 2q, row 2q + 1) of columns 2i and 2i + 1 of the four: bf16 of the exact float
              const uint32_t a0 = __byte_perm(__float_as_uint(i8_f32(w0, 2 * i)), __float_as_uint(i8_f32(w1, 2 * i)), 0x7632);
              const uint32_t a1 =
                  __byte_perm(__float_as_uint(i8_f32(w0, 2 * i + 1)), __float_as_uint(i8_f32(w1, 2 * i + 1)), 0x7632);
              mma_bf16(yc4[2 * b + i], a0, a1, a0, a1, bh, bl);
            }
          }
        }
      }
      // ---- partial y of this block, this warp's slice
      {
        // tiles 2b and 2b + 1: columns 256w + 32b + 4g .. + 3 (tile 2b + i holds
        // + 2i and + 2i + 1), tokens 2q and 2q + 1 -- four consecutive columns
        // of a token per lane and store
        const int g = lane >> 2, t0 = 2 * (lane & 3);
        unsigned long long* mine = reinterpret_cast<unsigned long long*>(P.partial) + (size_t)cta * T * H;
    #pragma unroll
        for (int b = 0; b < 8; ++b) {
          const int c = 256 * w + 32 * b + 4 * g;
    #pragma unroll
          for (int e = 0; e < 2; ++e) {
            if (t0 + e >= T) continue;
            if constexpr (TAGGED) {
              unsigned long long* dst = mine + (size_t)(t0 + e) * H + c;
              st_relaxed_gpu_v2_u64(dst, tagged(tag, yc4[2 * b][e]), tagged(tag, yc4[2 * b][2 + e]), pol_keep);
              st_relaxed_gpu_v2_u64(dst + 2, tagged(tag, yc4[2 * b + 1][e]), tagged(tag, yc4[2 * b + 1][2 + e]), pol_keep);
            } else {
              *reinterpret_cast<float4*>(P.partial + ((size_t)cta * T + t0 + e) * H + c) =
                  make_float4(yc4[2 * b][e], yc4[2 * b][2 + e], yc4[2 * b + 1][e], yc4[2 * b + 1][2 + e]);
            }
          }
        }
      }
      named_bar_or(kBarSplit, NTB, h_timed_out);
      return;
    }
  }

  // ---- before the wait (nothing the previous kernel writes is read), side
  // by side: warp 0 initialises the barriers and issues the shared expert's
  // first stages (their weights do not depend on the previous kernel), warp 1
  // clears the routing tables, warp 2 fills the per-U stage table, warp 3
  // fetches the tensor-map descriptors; every thread loads its part of the
  // block's router row.
  if (warp == 0) {
    if (lane == 0) {
      for (int i = 0; i < NS; ++i) {
        mbar_init(&full[i], 1);
        scnt[i] = 0;
      }
      for (int i = 0; i < P.nsd; ++i) mbar_init(&fulld[i], 1);
      mbar_init(xbar, 1);
      mbar_fence_init();
    }
  } else if (warp == 1) {
    for (int i = lane; i < (P.E + 31) / 32; i += 32) tb.bitmap[i] = 0u;
    for (int i = lane; i < TK; i += 32) tb.mask[i] = 0u;
    for (int i = lane; i < TK * T; i += 32) tb.wt[i] = 0.f;
    for (int i = lane; i < T; i += 32) tb.xmax[i] = 0u;
  } else if (warp == 2) {
    // the routed run of this block for every possible count U of active
    // experts (K <= U <= min(E, T K)): groups [q0, q1) of the flattened
    // (active expert, group) order, so that shared + routed groups are
    // balanced over the blocks
    for (int j = lane; j <= min(P.E, TK) - K; j += 32) {
      const uint32_t R = (uint32_t)(K + j) * (uint32_t)gI, G = P.G, cc = cta;
      uint32_t q0, q1;
      if (R >= G) {
        q0 = muldiv(R + gS, cc, G) - gs0;
        q1 = muldiv(R + gS, cc + 1, G) - gs1;
      } else {
        q0 = muldiv(R, cc, G);
        q1 = muldiv(R, cc + 1, G);
      }
      const uint32_t u0 = q0 / (uint32_t)gI;
      tb.qtab[4 * j] = (int)(q1 - q0);
      tb.qtab[4 * j + 1] = (int)u0;
      tb.qtab[4 * j + 2] = (int)(q0 - u0 * (uint32_t)gI);
    }
  } else if (warp == 3) {
    if constexpr (FAST) {
      // descriptors of the routed maps are first used after the routing,
      // under load: fetch all four now
      if (lane == 0) prefetch_tensormap(&Pk.tm_gu_e);
      if (lane == 1) prefetch_tensormap(&Pk.tm_d_e);
      if (lane == 2) prefetch_tensormap(&Pk.tm_gu_s);
      if (lane == 3) prefetch_tensormap(&Pk.tm_d_s);
      if constexpr (I8) {
        if (lane == 4) prefetch_tensormap(&Pk.tm_gusc_e);
        if (lane == 5) prefetch_tensormap(&Pk.tm_dsc_e);
        if (lane == 6) prefetch_tensormap(&Pk.tm_gusc_s);
        if (lane == 7) prefetch_tensormap(&Pk.tm_dsc_s);
      }
    }
  }
  // the shared stages (every thread advances the issue cursors in step; the
  // thread that initialised the barriers issues)
  for (int k = 0; k < min(n_sh, NS); ++k) {
    advance(ci, NS);
    if (tid == 0) issue(ci);
  }
  if constexpr (FAST)
    for (int k = 0; k < min(n_sh, P.nsd); ++k) {
      advance(cd, P.nsd);
      if (tid == 0) issue_d(cd);
    }

  // Router row of this block (row cta of router_w; row E is the shared-gate
  // vector), read before the wait: the weights are never written by a kernel
  // that lets this one start early (only this kernel does, and it writes no
  // weights; any other predecessor has completed before this kernel starts).
  constexpr int kRC = kMaxH / (kRowThreads * 8);  // 8-element chunks of a row per thread
  uint4 wr[kRC];
  // the shared-expert part needs only the shared-gate row (block 0)
  const int r_first = P.part == 2 ? (cta == 0 ? P.E : P.E + 1) : cta;
  const int r_step = P.part == 2 ? P.E + 1 : P.G;
  {
    const uint16_t* w = r_first < P.E ? P.router_w + (size_t)r_first * H : P.gate_w;
#pragma unroll
    for (int q = 0; q < kRC; ++q) {
      const int c0 = 8 * tid + kRowThreads * 8 * q;
      wr[q] = (r_first <= P.E && c0 < H) ? *reinterpret_cast<const uint4*>(w + c0) : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  blk_sync<SYNC_NT>();  // barriers initialised, tables cleared

  // ---- the activation (block form: x_res) and the workspace belong to this
  // kernel from here on
  pdl_wait();
  // The activation (or x_res) of all tokens: one bulk copy per block into
  // shared memory -- every block needs all of it, and one read per block
  // keeps the L2 lines of x from being hammered by every warp of the grid.
  // Issued first: nothing before it depends on it, and its latency covers
  // the reads of the call's epoch.
  const int src4 = P.act == 0 || P.block_mode;  // fp32 source rows
  if (tid == 0) {
    const uint32_t bytes = (uint32_t)(T * H * (src4 ? 4 : 2));
    mbar_arrive_expect_tx(xbar, bytes);
    bulk_g2s(xs, P.x, bytes, xbar, policy_evict_last());
  }
  RowSync* const sync = P.sync;
  const unsigned long long prev_epoch = __ldcg(&sync->epoch);
  const unsigned long long epoch = prev_epoch + 1ull;
  const bool fast_sync = __ldcg(&sync->sig) == ~prev_epoch;
  const uint32_t tag = (uint32_t)epoch;
  // tagged partials: kept in L2 (evict-last; rewritten every call, read
  // within microseconds)
  const uint64_t pol_keep = policy_evict_last();
  if (cta == 0) {
    if (tid == 0) P.ctrl[kCtrlStatus] = 0u;  // a status left by the failure-path probe
    for (int c = P.G + tid; c < kMaxGrid; c += kRowThreads) sync->status[c] = 0;
  }
  bool timed_out = false;
  if (!mbar_wait(xbar, 0)) timed_out = true;
  // block form: RMSNorm factors of the fp32 rows, all warps (scratch: the
  // partials region, unused before the stage loop; ends with a barrier)
  if (P.block_mode)
    block_norm_factors<SYNC_NT>(reinterpret_cast<const float*>(xs), T, H, P.eps, reinterpret_cast<float*>(sm + P.off_part),
                       tb.inv, kRowWarps);
  // ---- router logits of this block's rows r = cta, cta + G, ... (<= E):
  // logit[t][r] = sum_h W[r,h] x_t[h], accumulated error-free (TwoSum of the
  // exact bf16 x bf16 products, TwoProduct for fp32 x) so that the fp32 logit
  // is the exact dot product rounded once (up to a residual far below fp32
  // resolution) and the top-k decision does not depend on any summation
  // order.  The block's 8 warps reduce in warp order.
  {
    float* red = reinterpret_cast<float*>(sm + P.off_part);  // [kRowWarps][TMAX][2]
    const bool exact_products = P.block_mode || P.act == 1;   // bf16 x bf16 is exact in fp32
    for (int r = r_first, j = 0; r <= P.E; r += r_step, ++j) {
      if (j > 0) {
        const uint16_t* w = r < P.E ? P.router_w + (size_t)r * H : P.gate_w;
#pragma unroll
        for (int q = 0; q < kRC; ++q) {
          const int c0 = 8 * tid + kRowThreads * 8 * q;
          wr[q] = c0 < H ? *reinterpret_cast<const uint4*>(w + c0) : make_uint4(0u, 0u, 0u, 0u);
        }
      }
      float sa[TMAX], ca[TMAX];
#pragma unroll
      for (int t = 0; t < TMAX; ++t) sa[t] = ca[t] = 0.f;
#pragma unroll
      for (int q = 0; q < kRC; ++q) {
        const int c0 = 8 * tid + kRowThreads * 8 * q;
        if (c0 >= H) break;
        const uint4 wv = wr[q];
        const float wf[8] = {bf16_lo(wv.x), bf16_hi(wv.x), bf16_lo(wv.y), bf16_hi(wv.y),
                             bf16_lo(wv.z), bf16_hi(wv.z), bf16_lo(wv.w), bf16_hi(wv.w)};
#pragma unroll
        for (int t = 0; t < TMAX; ++t) {
          if (t >= T) break;
          float xf[8];
          x8_from_smem(xs + (size_t)t * H * (src4 ? 4 : 2), src4, P.block_mode, P.block_mode ? tb.inv[2 * t] : 0.f,
                       P.block_mode ? tb.inv[2 * t + 1] : 0.f, c0, xf);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            float pr, e1 = 0.f, tt, e2;
            if (exact_products)
              pr = __fmul_rn(wf[e], xf[e]);
            else
              two_prod(wf[e], xf[e], pr, e1);
            two_sum(sa[t], pr, tt, e2);
            sa[t] = tt;
            ca[t] = __fadd_rn(ca[t], __fadd_rn(e1, e2));
          }
        }
      }
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
        warp_sum2(sa[t], ca[t]);
        if (lane == 0) {
          red[(warp * TMAX + t) * 2] = sa[t];
          red[(warp * TMAX + t) * 2 + 1] = ca[t];
        }
      }
      blk_sync<SYNC_NT>();
      if (tid < T) {
        float S = red[tid * 2], C = red[tid * 2 + 1];
        for (int w = 1; w < kRowWarps; ++w) {
          float tt, e;
          two_sum(S, red[(w * TMAX + tid) * 2], tt, e);
          S = tt;
          C = __fadd_rn(__fadd_rn(C, red[(w * TMAX + tid) * 2 + 1]), e);
        }
        __stcg(P.logits + (size_t)tid * P.ls + r, __fadd_rn(S, C));
      }
      blk_sync<SYNC_NT>();
    }
  }
  // tagged partials: this block's words first get a tag that is not the
  // call's -- the grid-wide barrier below publishes that before any reader
  // polls them
  if constexpr (TAGGED) {
    const unsigned long long stale = tagged(~tag, 0.f);
    unsigned long long* mine = reinterpret_cast<unsigned long long*>(P.partial) + (size_t)cta * T * H;
    for (int i = 2 * tid; i < T * H; i += 2 * kRowThreads) st_relaxed_gpu_v2_u64(mine + i, stale, stale, pol_keep);
  }
  // activation in its compute form, in place, while the other blocks finish
  // their logits.  Fast shapes: the bf16 fragments of the tensor-core loops
  // (A operand of the bf16 loop, B operand of the 4-bit loop; the same
  // registers per lane), token t's row at t * kXPitch, 16 bytes per (warp slice w, 32-column
  // block kp, lane quad q) -- unit tid = (8w + kp) * 4 + q, the fragments of
  // steps 2kp and 2kp + 1.  Other shapes: fp32 rows.  All reads of the source
  // precede the barrier, all writes follow it.
  if constexpr (I8C) {
    // int8 loop: each token quantised as in the general loop (x_scale =
    // max|x| / 127 in fp32, codes round-half-away(x / x_scale) clamped to
    // +-127), the codes as exact fp16 B fragments.  Unit U = (4w + b) * 4 + q
    // of token t's row (32 bytes at 32 U) holds, for the 16-column steps i of
    // the 64-column block b of warp slice w, the pairs (x[c], x[c + 1]) and
    // (x[c + 2], x[c + 3]), c = 256w + 64b + 16i + 4q, i = 0..3; thread tid
    // stages half hh = tid & 1 (i = 2hh, 2hh + 1) of unit tid / 2.  Odd
    // tokens store the two halves swapped, so a quarter warp's 16-byte reads
    // of tokens 2k and 2k + 1 fall in different banks.
    const int U = tid >> 1, hh = tid & 1;
    const int c_base = 256 * (U >> 4) + 64 * ((U >> 2) & 3) + 4 * (U & 3) + 32 * hh;
    float v[TMAX][8];
#pragma unroll
    for (int t = 0; t < TMAX; ++t) {
      float m = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) v[t][e] = 0.f;
      if (t < T) {
        const uint8_t* row = xs + (size_t)t * H * (src4 ? 4 : 2);
        const float hi = P.block_mode ? tb.inv[2 * t] : 0.f, lo = P.block_mode ? tb.inv[2 * t + 1] : 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) x2_from_smem(row, src4, P.block_mode, hi, lo, c_base + 16 * (j >> 1) + 2 * (j & 1), v[t] + 2 * j);
#pragma unroll
        for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(v[t][e]));
      }
      // max |x| of token t over the warp, then over the block (non-negative
      // floats order as their bit patterns)
      const uint32_t mw = __reduce_max_sync(0xffffffffu, __float_as_uint(m));
      if (lane == 0 && t < T) atomicMax(&tb.xmax[t], mw);
    }
    blk_sync<SYNC_NT>();
#pragma unroll
    for (int t = 0; t < TMAX; ++t) {
      if (t < T) {
        const float sc = __fdiv_rn(__uint_as_float(tb.xmax[t]), 127.0f);
        uint32_t f[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          int c[2];
#pragma unroll
          for (int e = 0; e < 2; ++e)
            c[e] = sc != 0.f ? max(-127, min(127, (int)roundf(__fdiv_rn(v[t][2 * j + e], sc)))) : 0;
          f[j] = (uint32_t)__half_as_ushort(__int2half_rn(c[0])) | ((uint32_t)__half_as_ushort(__int2half_rn(c[1])) << 16);
        }
        *reinterpret_cast<uint4*>(xs + (size_t)t * kXPitch + 32 * U + 16 * (hh ^ (t & 1))) = make_uint4(f[0], f[1], f[2], f[3]);
      }
    }
    if (tid < T) tb.xsc[tid] = __fdiv_rn(__uint_as_float(tb.xmax[tid]), 127.0f);
  } else if constexpr (FAST) {
    uint32_t fr[TMAX][4];
    const int w = tid >> 5, kp = (tid >> 2) & 7, q = tid & 3;
#pragma unroll
    for (int t = 0; t < TMAX; ++t) {
      fr[t][0] = fr[t][1] = fr[t][2] = fr[t][3] = 0u;
      if (t < T) {
        const uint8_t* row = xs + (size_t)t * H * (src4 ? 4 : 2);
        const float hi = P.block_mode ? tb.inv[2 * t] : 0.f, lo = P.block_mode ? tb.inv[2 * t + 1] : 0.f;
        if constexpr (Q4) {
          // 4-bit loop: step 2kp + h, pair e = (x[c + 2h + e], x[c + 2h + e + 4]), c = 256w + 32kp + 8q
          float v[8];
          x8_from_smem(row, src4, P.block_mode, hi, lo, 256 * w + 32 * kp + 8 * q, v);
#pragma unroll
          for (int j = 0; j < 4; ++j) fr[t][j] = bf16_pair_exact(v[j], v[j + 4]);
        } else {
          // bf16 loop: step 2kp + h, pair e = x[k0 + 8e], x[k0 + 8e + 1], k0 = 256w + 32kp + 16h + 2q
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float v[2];
            x2_from_smem(row, src4, P.block_mode, hi, lo, 256 * w + 32 * kp + 16 * (j >> 1) + 8 * (j & 1) + 2 * q, v);
            fr[t][j] = bf16_pair_exact(v[0], v[1]);
          }
        }
      }
    }
    blk_sync<SYNC_NT>();
#pragma unroll
    for (int t = 0; t < TMAX; ++t)
      if (t < T) *reinterpret_cast<uint4*>(xs + (size_t)t * kXPitch + 16 * tid) = make_uint4(fr[t][0], fr[t][1], fr[t][2], fr[t][3]);
  } else {
    constexpr int kMaxGroups = kDecodeMaxT * kMaxH / 8 / kRowThreads;  // 8-value groups per compute thread
    const int groups = T * (H / 8);
    float v[kMaxGroups][8];
#pragma unroll
    for (int k = 0; k < kMaxGroups; ++k) {
      const int gi = tid + kRowThreads * k;
      if (gi < groups) {
        const int t = gi / (H / 8), q = gi % (H / 8);
        x8_from_smem(xs + (size_t)t * H * (src4 ? 4 : 2), src4, P.block_mode, P.block_mode ? tb.inv[2 * t] : 0.f,
                     P.block_mode ? tb.inv[2 * t + 1] : 0.f, 8 * q, v[k]);
      }
    }
    if constexpr (I8) {
      // int8 activation: max |x| of every token (non-negative floats order
      // as their bit patterns)
#pragma unroll
      for (int k = 0; k < kMaxGroups; ++k) {
        const int gi = tid + kRowThreads * k;
        if (gi < groups) {
          float m = 0.f;
#pragma unroll
          for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(v[k][e]));
          atomicMax(&tb.xmax[gi / (H / 8)], __float_as_uint(m));
        }
      }
    }
    blk_sync<SYNC_NT>();
    if constexpr (I8) {
      // token t's codes at xs + t H (bytes), its scale x_scale = max|x| / 127
      // in the routing tables: q = round-half-away(x / x_scale) clamped to
      // +-127, all in fp32 (x_scale = 0: q = 0)
#pragma unroll
      for (int k = 0; k < kMaxGroups; ++k) {
        const int gi = tid + kRowThreads * k;
        if (gi < groups) {
          const int t = gi / (H / 8), q = gi % (H / 8);
          const float sc = __fdiv_rn(__uint_as_float(tb.xmax[t]), 127.0f);
          uint32_t w[2] = {0u, 0u};
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            int c = 0;
            if (sc != 0.f) c = max(-127, min(127, (int)roundf(__fdiv_rn(v[k][e], sc))));
            w[e >> 2] |= (uint32_t)(c & 0xFF) << (8 * (e & 3));
          }
          *reinterpret_cast<uint2*>(xs + (size_t)t * H + 8 * q) = make_uint2(w[0], w[1]);
        }
      }
      if (tid < T) tb.xsc[tid] = __fdiv_rn(__uint_as_float(tb.xmax[tid]), 127.0f);
    } else {
#pragma unroll
      for (int k = 0; k < kMaxGroups; ++k) {
        const int gi = tid + kRowThreads * k;
        if (gi < groups) {
          const int t = gi / (H / 8), q = gi % (H / 8);
          float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(xs) + (size_t)t * H + 8 * q);
          dst[0] = make_float4(v[k][0], v[k][1], v[k][2], v[k][3]);
          dst[1] = make_float4(v[k][4], v[k][5], v[k][6], v[k][7]);
        }
      }
    }
  }
  // ---- every block's logits (first barrier; see RowSync)
  if (!grid_barrier<SYNC_NT>(sync, 0, fast_sync, P.G, epoch, cta, true)) timed_out = true;
  // routing, every block from all logits: top-k of token t on warp 7 - t
  // (the chosen experts, their softmax weights and their bits in the
  // selection bitmap) and the shared gate sigmoid(logit_E)
  if (P.part == 2) {
    // shared-expert part: only the gate s of every token
    if (tid < T) tb.s[tid] = 1.0f / (1.0f + expf(-__ldcg(P.logits + (size_t)tid * P.ls + P.E)));
  } else {
    const int t = kRowWarps - 1 - warp;
    if (t < T) {
      float sl = 0.f;
      if (lane == 0) sl = __ldcg(P.logits + (size_t)t * P.ls + P.E);
      warp_topk<EPL>(P.logits + (size_t)t * P.ls, P.E, K, tb.ids + t * K, tb.p + t * K);
      if (lane < K) {
        const int e = tb.ids[t * K + lane];
        atomicOr(&tb.bitmap[e >> 5], 1u << (e & 31));
      }
      if (lane == 0) tb.s[t] = 1.0f / (1.0f + expf(-sl));
      if constexpr (TMAX == 1) {
        // one token: its k distinct experts are the active list; expert j's
        // active index is its rank among them (ascending)
        __syncwarp();
        const int e = lane < K ? tb.ids[lane] : 0x7FFFFFFF;
        int rank = 0;
        for (int j = 0; j < K; ++j) rank += __shfl_sync(0xffffffffu, e, j) < e;
        if (lane < K) {
          tb.active[rank] = e;
          tb.inv_u[e] = static_cast<int16_t>(rank);
          tb.mask[rank] = 1u;
          tb.wt[rank] = tb.p[lane];
        }
        if (lane == 0) tb.misc[0] = K;
      }
    }
  }
  blk_sync<SYNC_NT>();
  if (TMAX > 1 && warp == 0 && P.part != 2) {
    // active experts in ascending order (active index u): bitmap word l on
    // lane l, an exclusive scan of the word counts
    const int nw = (P.E + 31) / 32;
    const uint32_t w = lane < nw ? tb.bitmap[lane] : 0u;
    const int c = __popc(w);
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const int U = __shfl_sync(0xffffffffu, incl, 31);
    int u = incl - c;
    for (uint32_t m = w; m; m &= m - 1u, ++u) {
      const int e = 32 * lane + __ffs((int)m) - 1;
      tb.active[u] = e;
      tb.inv_u[e] = static_cast<int16_t>(u);
    }
    __syncwarp();
    // tokens of every active expert and their weights
    for (int t = 0; t < T; ++t)
      for (int k = lane; k < K; k += 32) {
        const int ts = t * K + k;
        const int ua = tb.inv_u[tb.ids[ts]];
        atomicOr(&tb.mask[ua], 1u << t);
        tb.wt[ua * T + t] = tb.p[ts];
      }
    if (lane == 0) tb.misc[0] = U;
  }
  if (TMAX > 1 && P.part != 2) blk_sync<SYNC_NT>();
  const int U = P.part == 2 ? 0 : tb.misc[0];
  if (P.part != 2) {
    const int32_t* q = tb.qtab + 4 * (U - K);
    n_stages = n_sh + q[0];
    ur0 = q[1];
    gr0 = q[2];
  }
  // the first routed stages of the rings, issued by the warps in turn
  {
    int j = 0;
    while (ci.k + 1 < min(n_stages, NS)) {
      advance(ci, NS);
      if (tid == 32 * (j++ & (kRowWarps - 1))) issue(ci);
    }
    if constexpr (FAST)
      while (cd.k + 1 < min(n_stages, P.nsd)) {
        advance(cd, P.nsd);
        if (tid == 32 * (j++ & (kRowWarps - 1))) issue_d(cd);
      }
  }
  if constexpr (NTB > kRowThreads) {
    // warps 8..15 take the stage count, the first routed stage and the
    // call's tag from here (they wait at kBarSplit since their start)
    if (tid == 0) {
      tb.misc[1] = n_stages;
      tb.misc[2] = ur0;
      tb.misc[3] = gr0;
      tb.misc[4] = static_cast<int32_t>(tag);
    }
    named_bar_sync(kBarSplit, NTB);
  }
  if (cta == 0 && warp == kRowWarps - 1 && P.part != 2) {
    // routing outputs for the caller and the test readers: counts, offsets
    // (a scan over the experts) and the stable token-major permutation
    int base = 0;
    for (int e0 = 0; e0 < P.E; e0 += 32) {
      const int e = e0 + lane;
      int cnt = 0;
      if (e < P.E && (tb.bitmap[e >> 5] >> (e & 31) & 1u)) cnt = __popc(tb.mask[tb.inv_u[e]]);
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (e < P.E) {
        P.r_counts[e] = cnt;
        P.r_offsets[e] = base + incl - cnt;
      }
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      P.r_offsets[P.E] = base;
      *P.r_nactive = U;
    }
    __syncwarp();
    for (int ts = lane; ts < TK; ts += 32) {
      if (P.topk_ids) P.topk_ids[ts] = tb.ids[ts];
      if (P.topk_w) P.topk_w[ts] = tb.p[ts];
      const int t = ts / K, e = tb.ids[ts];
      P.r_perm[P.r_offsets[e] + __popc(tb.mask[tb.inv_u[e]] & ((1u << t) - 1u))] = ts;
    }
    for (int u = lane; u < U; u += 32) P.r_active[u] = tb.active[u];
  }
  const uint32_t all_tokens = (1u << T) - 1u;

  // ---- stages
  // Thread j owns the 8-column chunks ch = j + 256 k
  // (k < NCH) of H: it forms the partial gate/up dot products of every row
  // of a stage over its chunks (A), and accumulates y over the same chunks
  // (C).  Each thread first copies its chunks of the stage into registers;
  // the last warp to do so refills the slot at once, so the copies in flight
  // never wait on arithmetic.  The 8 warps' partials meet in shared memory:
  // after the stage barrier a few threads (spread over the warps) form
  // h = w silu(g) u (A2), which C uses one stage later -- one block barrier
  // per stage, and C of stage s overlaps A2 of stage s + 1.
  constexpr int RSM = Q4 || I8 ? kRsMaxQ4 : kRsMaxB16;
  constexpr int NV = 2 * RSM * TMAX;  // dot values per warp per stage: (row, gate|up, token)
  float* part = reinterpret_cast<float*>(sm + P.off_part);  // [2][kRowWarps][NV]
  float* hb = reinterpret_cast<float*>(sm + P.off_h);       // [2][RSM][TMAX]
  float y[TMAX][NCH][8];
#pragma unroll
  for (int t = 0; t < TMAX; ++t)
#pragma unroll
    for (int k = 0; k < NCH; ++k)
#pragma unroll
      for (int e = 0; e < 8; ++e) y[t][k][e] = 0.f;
  float yc[MMA_C ? 16 : 1][4];  // tensor-core down projection: y of this warp's slice, D fragments
#pragma unroll
  for (int j = 0; j < (MMA_C ? 16 : 1); ++j) yc[j][0] = yc[j][1] = yc[j][2] = yc[j][3] = 0.f;
  float yc4[QMC ? 16 : 1][4];  // 4-bit / int8 tensor-core down projection: y of this warp's slice, D fragments
#pragma unroll
  for (int j = 0; j < (QMC ? 16 : 1); ++j) yc4[j][0] = yc4[j][1] = yc4[j][2] = yc4[j][3] = 0.f;

  if constexpr (B16C) {
    // ---- tensor-core stage loop (bf16 weights, H = 2048, 4 rows a stage).
    // Warp w owns the 256-column slice [256w, 256w + 256) of H.
    //   A: D[token][stage row] = x . W over the slice, m16n8k16 with the
    //      tokens as the 16 A rows (8 real) and the stage's 8 gate/up rows
    //      as the 8 B columns; 16 k-steps, B read straight from the slot.
    //   A2: h = w silu(g) u from the 8 warps' partials (after a barrier).
    //   C: y[16 cols][8 tokens] += downT^T h, one k-step of 16 rows per
    //      16-column tile (the stage's 4 downT rows; the other 12 are other
    //      rows of the slot, times h = 0); h enters as two bf16 terms
    //      (hi + lo), so y keeps fp32 accuracy.
    // x: the A fragments of token lane/4 (rows 8..15 zero) from the
    // fragment rows in shared memory, 16 bytes per 32-column block.
    const uint8_t* xrow = xs + (size_t)(lane >> 2) * kXPitch + (size_t)(32 * warp + (lane & 3)) * 16;
    const bool xon = (lane >> 2) < T;
    // One block barrier per stage: after the barrier of stage s, A2 of stage
    // s and C of stage s - 1 run together (partials and h by stage parity),
    // so a downT slot is refilled one stage later than its gate + up slot.
    StageCursor cs;
    cursor_init(cs, NS);
    int dslot = P.nsd - 1;  // downT ring slot and phase parity of the stage C works on
    uint32_t dph = 1u;
    int n_prev = 0;
    for (int s = 0; s <= n_stages; ++s) {
      const int par = s & 1;
      int n = 0, su = -1;
      if (s < n_stages) {
        advance(cs, NS);
        if (!mbar_wait(&full[cs.slot], cs.ph)) timed_out = true;
        su = cs.u;
        int si0;
        rows_of(cs, si0, n);
        const uint8_t* sl = ring + (size_t)cs.slot * P.stage_bytes;
        // -- A (four accumulators, so the tensor-core steps do not chain).  B
        // column n = lane / 4 is row n of the gate + up box (lines chunk * 8 + n).
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        {
          const int nrow = lane >> 2;
          float dq[4][4];
#pragma unroll
          for (int q = 0; q < 4; ++q) dq[q][0] = dq[q][1] = dq[q][2] = dq[q][3] = 0.f;
#pragma unroll
          for (int kp2 = 0; kp2 < 8; kp2 += 2) {
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
              const int kp = kp2 + e2;
              const uint4 xv = xon ? *reinterpret_cast<const uint4*>(xrow + 64 * kp) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int k0 = 256 * warp + 32 * kp + 16 * h + 2 * (lane & 3);
                const int line = (k0 >> 6) * (2 * kRsMaxB16) + nrow;
                const uint32_t b0 = *reinterpret_cast<const uint32_t*>(sl + swz_off(line, k0));
                const uint32_t b1 = *reinterpret_cast<const uint32_t*>(sl + swz_off(line, k0 + 8));
                mma_bf16(dq[2 * e2 + h], h ? xv.z : xv.x, 0u, h ? xv.w : xv.y, 0u, b0, b1);
              }
            }
          }
#pragma unroll
          for (int e = 0; e < 2; ++e) d[e] = (dq[0][e] + dq[1][e]) + (dq[2][e] + dq[3][e]);
        }
        // this lane: token lane/4, stage rows 2(lane & 3) and +1 (0..3 gate, 4..7 up)
        const int t = lane >> 2;
        if (t < TMAX) {
          float* pw = part + (size_t)(par * kRowWarps + warp) * NV;
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int nr = 2 * (lane & 3) + q, gu = nr >> 2, r = nr & 3;
            pw[(gu * RSM + r) * TMAX + t] = d[q];
          }
        }
      }
      named_bar_sync(kBarStage, kRowThreads);
      // every warp is done with this stage's gate + up box and (C of stage
      // s - 2 ended before this barrier) with the downT box of stage s - 2
      if (s + NS < n_stages) {
        advance(ci, NS);
        if (tid == kRowThreads - 1) issue(ci);
      }
      if (s >= 2 && s - 2 + P.nsd < n_stages) {
        advance(cd, P.nsd);
        if (tid == kRowThreads - 1) issue_d(cd);
      }
      // -- A2 of stage s: value j = (row, token) = r * TMAX + t on thread j
      {
        const int j = tid;
        if (s < n_stages && j < n * TMAX) {
          const int t = j % TMAX;
          const float* pp = part + (size_t)par * kRowWarps * NV;
          float g = 0.f, u = 0.f;
#pragma unroll
          for (int w = 0; w < kRowWarps; ++w) {
            g += pp[w * NV + j];
            u += pp[w * NV + RSM * TMAX + j];
          }
          float h = 0.f;
          if (su < 0)
            h = t < T ? tb.s[t] * silu_mul(g, u) : 0.f;
          else
            h = (tb.mask[su] >> t & 1u) ? tb.wt[su * T + t] * silu_mul(g, u) : 0.f;
          hb[par * RSM * TMAX + j] = h;
        }
      }
      // -- C of stage s - 1
      if (s >= 1) {
        if (++dslot == P.nsd) {
          dslot = 0;
          dph ^= 1u;
        }
        if (!mbar_wait(&fulld[dslot], dph)) timed_out = true;
        const uint8_t* dbox = dring + (size_t)dslot * kRsMaxB16 * rb;
        const float* hp = hb + (par ^ 1) * RSM * TMAX;
        if constexpr (!MMA_C) {
          // CUDA cores (one or two tokens): chunk tid of every downT row
          const int k = 8 * tid;
#pragma unroll
          for (int r = 0; r < kRsMaxB16; ++r) {
            if (r < n_prev) {
              const uint4 v = *reinterpret_cast<const uint4*>(dbox + swz_off((k >> 6) * kRsMaxB16 + r, k));
              const float w[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                                  bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
#pragma unroll
              for (int t = 0; t < TMAX; ++t) {
                const float hv = hp[r * TMAX + t];
#pragma unroll
                for (int e = 0; e < 8; ++e) y[t][0][e] = fmaf(hv, w[e], y[t][0][e]);
              }
            }
          }
        } else {
          const int t = lane >> 2, k0 = 2 * (lane & 3);
          const float h0 = (k0 < n_prev && t < TMAX) ? hp[k0 * TMAX + t] : 0.f;
          const float h1 = (k0 + 1 < n_prev && t < TMAX) ? hp[(k0 + 1) * TMAX + t] : 0.f;
          const uint32_t bh = pack_bf16(h0, h1);
          const uint32_t bl = pack_bf16(h0 - bf16_lo(bh), h1 - bf16_hi(bh));
          // matrix q = lane / 8 of the 16x16 A tile: stored rows k = (q / 2) * 8
          // + lane % 8 at columns (q % 2) * 8 ..; row k is downT row k % 4 of
          // the stage (k >= 4 repeat them, times h = 0)
          const int q = lane >> 3, r = lane & 3;
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t at[8][4];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int m0 = 256 * warp + 16 * (8 * half + j) + (q & 1) * 8;
              ldmatrix_x4_trans(at[j], dbox + swz_off((m0 >> 6) * kRsMaxB16 + r, m0));
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) mma_bf16(yc[8 * half + j], at[j][0], at[j][1], at[j][2], at[j][3], bh, 0u);
#pragma unroll
            for (int j = 0; j < 8; ++j) mma_bf16(yc[8 * half + j], at[j][0], at[j][1], at[j][2], at[j][3], bl, 0u);
          }
        }
      }
      n_prev = n;
    }
  } else if constexpr (Q4C) {
    // ---- tensor-core stage loop (4-bit weights, H = 2048, 8 rows a stage).
    // A stored row is 9 chunks of 128 bytes: chunks 0..7 the nibbles, chunk
    // 8 the 64 fp16 block scales.  Warp w owns the 256-column slice
    // [256w, 256w + 256) of H: nibble chunk w of every row, and the 8 block
    // scales in 16-byte unit w of chunk 8.
    //   A: per 32-column block kp, D[row][token] = Q . x over the block
    //      (two m16n8k16 steps; Q = code - 8 is exact in bf16), then times
    //      the row's block scale into fp32 accumulators; the 16 A rows are
    //      the 8 gate rows and the 8 up rows, the B columns the tokens.  The
    //      k order inside a block follows the nibble order of a 32-bit word,
    //      and the x fragments follow it.
    //   A2: h = w silu(g) u from the 8 warps' partials.
    //   C (warps 8..15, q4_down_stage): the down projection.
    const int gq = lane >> 2, qq = lane & 3;
    // x: the B fragments of token lane/4 from the fragment rows in shared
    // memory (nibble order), 16 bytes per block.
    const uint8_t* xrow = xs + (size_t)gq * kXPitch + (size_t)(32 * warp + qq) * 16;
    const bool xon = gq < T;
    // One barrier of all 16 warps per stage: after the barrier of stage s,
    // A2 of stage s runs here and C of stage s - 1 on warps 8..15 (partials
    // and h by stage parity).  n_stages + 1 barriers, as warps 8..15 make.
    StageCursor cs;
    cursor_init(cs, NS);
    for (int s = 0; s <= n_stages; ++s) {
      const int par = s & 1;
      int n = 0, su = -1;
      if (s < n_stages) {
        advance(cs, NS);
        if (!mbar_wait(&full[cs.slot], cs.ph)) timed_out = true;
        su = cs.u;
        int si0;
        rows_of(cs, si0, n);
        const uint8_t* sl = ring + (size_t)cs.slot * P.stage_bytes;
        // -- A.  Box lines: (chunk * 2 + matrix) * 8 + row.  The 16 A rows
        // are the stage's 8 gate rows and its 8 up rows, the 8 B columns the
        // tokens, so one m16n8k16 step covers both tiles.
        float acc[4] = {0.f, 0.f, 0.f, 0.f};  // D fragment: gate row g, tokens 2q, 2q + 1; up row g, the same tokens
        const int lg = 16 * kRsMaxQ4 + gq, lu = 17 * kRsMaxQ4 + gq;  // scale lines of row g (line & 7 == g)
        const uint4 sg = *reinterpret_cast<const uint4*>(sl + lg * 128 + ((warp ^ gq) << 4));
        const uint4 su4 = *reinterpret_cast<const uint4*>(sl + lu * 128 + ((warp ^ gq) << 4));
        const uint8_t* wgp = sl + (2 * warp * kRsMaxQ4 + gq) * 128 + 4 * qq;        // nibble chunk w, gate row g
        const uint8_t* wup = sl + ((2 * warp + 1) * kRsMaxQ4 + gq) * 128 + 4 * qq;  // nibble chunk w, up row g
        // blocks in two halves of four (the scale words of a half picked once)
#pragma unroll
        for (int kh = 0; kh < 2; ++kh) {
          const uint32_t g01 = kh ? sg.z : sg.x, g23 = kh ? sg.w : sg.y;
          const uint32_t u01 = kh ? su4.z : su4.x, u23 = kh ? su4.w : su4.y;
#pragma unroll
          for (int e4 = 0; e4 < 4; ++e4) {
            const int kp = 4 * kh + e4;
            const uint4 xv = xon ? *reinterpret_cast<const uint4*>(xrow + 64 * kp) : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t wg = *reinterpret_cast<const uint32_t*>(wgp + ((kp ^ gq) << 4));
            const uint32_t wu = *reinterpret_cast<const uint32_t*>(wup + ((kp ^ gq) << 4));
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            mma_bf16(d, q4_pair_bf16(wg), q4_pair_bf16(wu), q4_pair_bf16(wg >> 4), q4_pair_bf16(wu >> 4), xv.x, xv.y);
            mma_bf16(d, q4_pair_bf16(wg >> 8), q4_pair_bf16(wu >> 8), q4_pair_bf16(wg >> 12), q4_pair_bf16(wu >> 12),
                     xv.z, xv.w);
            const uint32_t gw = (e4 >> 1) ? g23 : g01, uw = (e4 >> 1) ? u23 : u01;
            const float s_g = __half2float(__ushort_as_half(static_cast<unsigned short>((e4 & 1) ? (gw >> 16) : (gw & 0xFFFFu))));
            const float s_u = __half2float(__ushort_as_half(static_cast<unsigned short>((e4 & 1) ? (uw >> 16) : (uw & 0xFFFFu))));
            acc[0] = fmaf(s_g, d[0], acc[0]);
            acc[1] = fmaf(s_g, d[1], acc[1]);
            acc[2] = fmaf(s_u, d[2], acc[2]);
            acc[3] = fmaf(s_u, d[3], acc[3]);
          }
        }
        {
          float* pw = part + (size_t)(par * kRowWarps + warp) * NV;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int t = 2 * qq + e;
            if (t < TMAX) {
              pw[gq * TMAX + t] = acc[e];
              pw[(RSM + gq) * TMAX + t] = acc[2 + e];
            }
          }
        }
      }
      named_bar_sync(kBarStage, NTB);
      // warps 0..7 are done with this stage's gate + up box
      if (s + NS < n_stages) {
        advance(ci, NS);
        if (tid == kRowThreads - 1) issue(ci);
      }
      // -- A2 of stage s: value j = (row, token) = r * TMAX + t on thread j
      {
        const int j = tid;
        if (s < n_stages && j < n * TMAX) {
          const int t = j % TMAX;
          const float* pp = part + (size_t)par * kRowWarps * NV;
          float g = 0.f, u = 0.f;
#pragma unroll
          for (int w = 0; w < kRowWarps; ++w) {
            g += pp[w * NV + j];
            u += pp[w * NV + RSM * TMAX + j];
          }
          float h = 0.f;
          if (su < 0)
            h = t < T ? tb.s[t] * silu_mul(g, u) : 0.f;
          else
            h = (tb.mask[su] >> t & 1u) ? tb.wt[su * T + t] * silu_mul(g, u) : 0.f;
          hb[par * RSM * TMAX + j] = h;
        }
      }
    }
  } else if constexpr (I8C) {
    // ---- tensor-core stage loop (int8 weights and activation, H = 2048, 8
    // rows a stage).  A stored row is H codes, then a 16-byte record whose
    // first word is the row's fp32 scale; the boxes hold the codes (128-byte
    // chunks, swizzled) and, after them, the stage rows' records.  Warp w
    // owns the 256-column slice [256w, 256w + 256) of H: code chunks 2w and
    // 2w + 1 of every row.
    //   A: D[row][token] = q . qx over the slice, m16n8k16 on fp16 operands
    //      (codes are exact in fp16; each product is exact in fp32, and every
    //      partial sum is an integer below 256 * 127^2 < 2^22, so the fp32
    //      accumulators hold the int32 dot product exactly); per 64-column
    //      block, one ldmatrix brings 4 codes of each stage row per lane for
    //      each of the block's four 16-column steps, and the x fragments use
    //      the same column order.  The 16 A rows are the 8 gate rows and the
    //      8 up rows, the B columns the tokens.
    //   A2: g = float(sum of the 8 warps' integer partials) * x_scale * s in
    //      fp32 (the up rows alike), h = w silu(g) u.
    //   C (warps 8..15, i8_down_stage): y[col][token] += Q^T (h s_down) on
    //      the tensor cores (as the 4-bit loop).
    // One barrier of all 16 warps per stage (as the 4-bit loop).
    const int gq = lane >> 2, qq = lane & 3;
    const uint8_t* xrow = xs + (size_t)gq * kXPitch + (size_t)(512 * warp + 32 * qq);
    const int xh0 = 16 * (gq & 1), xh1 = 16 * ((gq & 1) ^ 1);  // the two halves of a unit (odd tokens swapped)
    const bool xon = gq < T;
    const int rr = lane & 7, mi = lane >> 3;  // ldmatrix: the row and the matrix (16-byte unit) this lane addresses
    StageCursor cs;
    cursor_init(cs, NS);
    for (int s = 0; s <= n_stages; ++s) {
      const int par = s & 1;
      int n = 0, su = -1;
      const int j = tid;  // A2 value j = (row, token) = r * TMAX + t
      float s_gate = 0.f, s_up = 0.f;
      if (s < n_stages) {
        advance(cs, NS);
        if (!mbar_wait(&full[cs.slot], cs.ph)) timed_out = true;
        su = cs.u;
        int si0;
        rows_of(cs, si0, n);
        const uint8_t* sl = ring + (size_t)cs.slot * P.stage_bytes;
        // -- A.  Box lines: (chunk * 2 + matrix) * 8 + row.
        // The 16 A rows are the stage's 8 gate rows and its 8 up rows, the 8
        // B columns the tokens, so one m16n8k16 step covers both tiles.
        float acc[4][4];  // [step i of a block][D: gate row g, tokens 2q, 2q + 1; up row g, the same tokens]
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const uint4 xa = xon ? *reinterpret_cast<const uint4*>(xrow + 128 * b + xh0) : make_uint4(0u, 0u, 0u, 0u);
          const uint4 xb = xon ? *reinterpret_cast<const uint4*>(xrow + 128 * b + xh1) : make_uint4(0u, 0u, 0u, 0u);
          const int chunk = 2 * warp + (b >> 1);
          const int unit = (((b & 1) * 4 + mi) ^ rr) << 4;
          uint32_t wg[4], wu[4];
          ldmatrix_x4(wg, sl + (size_t)((chunk * 2) * 8 + rr) * 128 + unit);
          ldmatrix_x4(wu, sl + (size_t)((chunk * 2 + 1) * 8 + rr) * 128 + unit);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint4& xv = i < 2 ? xa : xb;
            const uint32_t b0 = (i & 1) ? xv.z : xv.x, b1 = (i & 1) ? xv.w : xv.y;
            mma_f16(acc[i], i8_pair_f16(wg[i], 0), i8_pair_f16(wu[i], 0), i8_pair_f16(wg[i], 1), i8_pair_f16(wu[i], 1),
                    b0, b1);
          }
        }
        {
          float* pw = part + (size_t)(par * kRowWarps + warp) * NV;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int t = 2 * qq + e;
            if (t < TMAX) {
              pw[gq * TMAX + t] = (acc[0][e] + acc[1][e]) + (acc[2][e] + acc[3][e]);
              pw[(RSM + gq) * TMAX + t] = (acc[0][2 + e] + acc[1][2 + e]) + (acc[2][2 + e] + acc[3][2 + e]);
            }
          }
        }
        // the row scales of A2's value j, read before the slot is released
        if (j < n * TMAX) {
          const int r = j / TMAX;
          s_gate = *reinterpret_cast<const float*>(sl + (size_t)2 * RS * H + (size_t)r * 16);
          s_up = *reinterpret_cast<const float*>(sl + (size_t)2 * RS * H + (size_t)(RS + r) * 16);
        }
      }
      named_bar_sync(kBarStage, NTB);
      // warps 0..7 are done with this stage's gate + up box
      if (s + NS < n_stages) {
        advance(ci, NS);
        if (tid == kRowThreads - 1) issue(ci);
      }
      // -- A2 of stage s
      if (s < n_stages && j < n * TMAX) {
        const int t = j % TMAX;
        const float* pp = part + (size_t)par * kRowWarps * NV;
        int gi = 0, ui = 0;
#pragma unroll
        for (int w = 0; w < kRowWarps; ++w) {
          gi += __float2int_rn(pp[w * NV + j]);
          ui += __float2int_rn(pp[w * NV + RSM * TMAX + j]);
        }
        const float xsc_t = t < T ? tb.xsc[t] : 0.f;
        const float g = __fmul_rn(__fmul_rn(__int2float_rn(gi), xsc_t), s_gate);
        const float u = __fmul_rn(__fmul_rn(__int2float_rn(ui), xsc_t), s_up);
        float h = 0.f;
        if (su < 0)
          h = t < T ? tb.s[t] * silu_mul(g, u) : 0.f;
        else
          h = (tb.mask[su] >> t & 1u) ? tb.wt[su * T + t] * silu_mul(g, u) : 0.f;
        hb[par * RSM * TMAX + j] = h;
      }
    }
  } else {

    // downT chunks of this thread, by stage parity
    constexpr bool B16 = !Q4 && !I8;
    uint4 dwb[2][B16 ? RSM : 1][NCH];
    uint32_t dwq[2][Q4 ? RSM : 1][NCH];
    uint16_t dsc[2][Q4 ? RSM : 1][NCH];
    uint2 dwi[2][I8 ? RSM : 1][NCH];
    // int8: the stage's row scales (gate, up, downT) by stage parity, and
    // the activation scales
    float* wsc = hb + 2 * RSM * TMAX;  // [2][3][RSM]
    const float* xsc = tb.xsc;
    int n_prev = 0;
    uint32_t m_prev = 0u;
    StageCursor cs;
    cursor_init(cs, NS);

    auto step = [&](auto parc, int s) {
      constexpr int par = decltype(parc)::value;
      uint32_t m = 0u;
      int n = 0, su = -1, si0 = 0;
      if (s < n_stages) {
        advance(cs, NS);
        const int slot = cs.slot;
        if (!mbar_wait(&full[slot], cs.ph)) timed_out = true;
        su = cs.u;
        rows_of(cs, si0, n);
        const uint8_t* sl = ring + (size_t)slot * P.stage_bytes;
        // this thread's chunks of every row of the stage, into registers
        uint4 wgb[B16 ? RSM : 1][NCH], wub[B16 ? RSM : 1][NCH];
        uint32_t wgq[Q4 ? RSM : 1][NCH], wuq[Q4 ? RSM : 1][NCH];
        uint16_t sgq[Q4 ? RSM : 1][NCH], suq[Q4 ? RSM : 1][NCH];
        uint2 wgi[I8 ? RSM : 1][NCH], wui[I8 ? RSM : 1][NCH];
        (void)wgb, (void)wub, (void)wgq, (void)wuq, (void)sgq, (void)suq, (void)wgi, (void)wui;  // one kind is used
        if constexpr (I8) {
          // the scale after each row's H codes
          if (warp == 0 && lane < 3 * RSM) {
            const int m = lane / RSM, r = lane % RSM;
            if (r < n) wsc[(par * 3 + m) * RSM + r] = *reinterpret_cast<const float*>(sl + (size_t)(m * RS + r) * rp + H);
          }
        }
#pragma unroll
        for (int r = 0; r < RSM; ++r) {
          if (r < n) {
            const uint8_t* rg = sl + (size_t)r * rp;
            const uint8_t* ru = sl + (size_t)(RS + r) * rp;
            const uint8_t* rd = sl + (size_t)(2 * RS + r) * rp;
#pragma unroll
            for (int k = 0; k < NCH; ++k) {
              const int ch = tid + kRowThreads * k;
              if (FAST || ch < H / 8) {
                if constexpr (I8) {
                  wgi[I8 ? r : 0][k] = *reinterpret_cast<const uint2*>(rg + (size_t)ch * 8);
                  wui[I8 ? r : 0][k] = *reinterpret_cast<const uint2*>(ru + (size_t)ch * 8);
                  dwi[par][I8 ? r : 0][k] = *reinterpret_cast<const uint2*>(rd + (size_t)ch * 8);
                } else if constexpr (B16) {
                  wgb[B16 ? r : 0][k] = *reinterpret_cast<const uint4*>(rg + (size_t)ch * 16);
                  wub[B16 ? r : 0][k] = *reinterpret_cast<const uint4*>(ru + (size_t)ch * 16);
                  dwb[par][B16 ? r : 0][k] = *reinterpret_cast<const uint4*>(rd + (size_t)ch * 16);
                } else {
                  const int so = H / 2 + 2 * (ch >> 2);
                  wgq[Q4 ? r : 0][k] = *reinterpret_cast<const uint32_t*>(rg + (size_t)ch * 4);
                  wuq[Q4 ? r : 0][k] = *reinterpret_cast<const uint32_t*>(ru + (size_t)ch * 4);
                  dwq[par][Q4 ? r : 0][k] = *reinterpret_cast<const uint32_t*>(rd + (size_t)ch * 4);
                  sgq[Q4 ? r : 0][k] = *reinterpret_cast<const uint16_t*>(rg + so);
                  suq[Q4 ? r : 0][k] = *reinterpret_cast<const uint16_t*>(ru + so);
                  dsc[par][Q4 ? r : 0][k] = *reinterpret_cast<const uint16_t*>(rd + so);
                }
              }
            }
          }
        }
        // release the slot: the warp's loads are ordered before its arrival
        // (warp barrier, then a CTA-scope fence), and the last warp to
        // arrive refills the slot at once
        const bool refill = s + NS < n_stages;
        if (refill) advance(ci, NS);
        __syncwarp();
        if (lane == 0) {
          __threadfence_block();
          if (atomicAdd(&scnt[slot], 1) == kRowWarps - 1) {
            scnt[slot] = 0;
            if (refill) issue(ci);
          }
        }
        // tokens of the stage's group (every row of a stage has the same one)
        m = su < 0 ? all_tokens : tb.mask[su];
        uint32_t mrow[RSM];
#pragma unroll
        for (int r = 0; r < RSM; ++r) mrow[r] = r < n ? m : 0u;
        // -- A: partial dots of every row over this thread's chunks; packed
        // in eights, reduced across the warp, one partial per warp
        float* pw = part + (size_t)(par * kRowWarps + warp) * NV;
        float pend[8];
#pragma unroll
        for (int r = 0; r < RSM; ++r) {
          float ga[TMAX], ua[TMAX];
#pragma unroll
          for (int t = 0; t < TMAX; ++t) ga[t] = ua[t] = 0.f;
          if (r < n) {
#pragma unroll
            for (int k = 0; k < NCH; ++k) {
              const int ch = tid + kRowThreads * k;
              if (!FAST && ch >= H / 8) break;
              if constexpr (I8) {
                // exact int32 dot products of the codes (each thread's part
                // stays below 2^24, so the fp32 warp sums are exact too)
                const uint2 vg = wgi[I8 ? r : 0][k], vu = wui[I8 ? r : 0][k];
#pragma unroll
                for (int t = 0; t < TMAX; ++t) {
                  if (!(mrow[r] >> t & 1u)) continue;
                  const uint2 xq = *reinterpret_cast<const uint2*>(xs + (size_t)t * H + 8 * ch);
                  const int gd = __dp4a((int)vg.y, (int)xq.y, __dp4a((int)vg.x, (int)xq.x, 0));
                  const int ud = __dp4a((int)vu.y, (int)xq.y, __dp4a((int)vu.x, (int)xq.x, 0));
                  ga[t] += (float)gd;
                  ua[t] += (float)ud;
                }
              } else if constexpr (B16) {
                const uint4 vg = wgb[B16 ? r : 0][k], vu = wub[B16 ? r : 0][k];
                const float gf[8] = {bf16_lo(vg.x), bf16_hi(vg.x), bf16_lo(vg.y), bf16_hi(vg.y),
                                     bf16_lo(vg.z), bf16_hi(vg.z), bf16_lo(vg.w), bf16_hi(vg.w)};
                const float uf[8] = {bf16_lo(vu.x), bf16_hi(vu.x), bf16_lo(vu.y), bf16_hi(vu.y),
                                     bf16_lo(vu.z), bf16_hi(vu.z), bf16_lo(vu.w), bf16_hi(vu.w)};
#pragma unroll
                for (int t = 0; t < TMAX; ++t) {
                  if (!(mrow[r] >> t & 1u)) continue;
                  const float4* xp =
                      reinterpret_cast<const float4*>(reinterpret_cast<const float*>(xs) + (size_t)t * H + 8 * ch);
                  const float4 a = xp[0], b = xp[1];
                  const float xv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
                  float g0 = 0.f, g1 = 0.f, u0 = 0.f, u1 = 0.f;
#pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    g0 = fmaf(gf[e], xv[e], g0);
                    g1 = fmaf(gf[e + 4], xv[e + 4], g1);
                    u0 = fmaf(uf[e], xv[e], u0);
                    u1 = fmaf(uf[e + 4], xv[e + 4], u1);
                  }
                  ga[t] += g0 + g1;
                  ua[t] += u0 + u1;
                }
              } else {
                const uint32_t qg = wgq[Q4 ? r : 0][k], qu = wuq[Q4 ? r : 0][k];
                const float dg = __half2float(__ushort_as_half(sgq[Q4 ? r : 0][k]));
                const float du = __half2float(__ushort_as_half(suq[Q4 ? r : 0][k]));
#pragma unroll
                for (int t = 0; t < TMAX; ++t) {
                  if (!(mrow[r] >> t & 1u)) continue;
                  const float4* xp =
                      reinterpret_cast<const float4*>(reinterpret_cast<const float*>(xs) + (size_t)t * H + 8 * ch);
                  const float4 a = xp[0], b = xp[1];
                  const float xv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
                  float sg = 0.f, su = 0.f;
#pragma unroll
                  for (int e = 0; e < 8; ++e) {
                    sg = fmaf(nib_f32(qg, e), xv[e], sg);
                    su = fmaf(nib_f32(qu, e), xv[e], su);
                  }
                  ga[t] = fmaf(dg, sg, ga[t]);
                  ua[t] = fmaf(du, su, ua[t]);
                }
              }
            }
          }
          // values (r, gate|up, t) at v = (2r + gu) * TMAX + t, reduced in eights
#pragma unroll
          for (int gu = 0; gu < 2; ++gu)
#pragma unroll
            for (int t = 0; t < TMAX; ++t) {
              const int v = (2 * r + gu) * TMAX + t;
              pend[v & 7] = gu ? ua[t] : ga[t];
              if ((v & 7) == 7 && 8 * (v >> 3) < 2 * n * TMAX) {
                const float red = warp_reduce8(pend);
                if ((lane & 3) == 0) pw[(v & ~7) + (lane >> 2)] = red;
              }
            }
        }
      }
      named_bar_sync(kBarStage, kRowThreads);
      if (s < n_stages) {
        // -- A2: h of (row, token) from the warp partials in order; value j
        // goes to thread (j % 8) * 32 + j / 8, spreading the work over warps
        const int j = (tid & 31) * kRowWarps + (tid >> 5);
        if (j < n * TMAX) {
          const int r = j / TMAX, t = j % TMAX;
          const float* pp = part + (size_t)par * kRowWarps * NV;
          float g = 0.f, u = 0.f;
          if constexpr (I8) {
            // int32 sums of the exact warp partials; then
            // g = float(dot) * x_scale * s_gate in fp32, in that order (u alike)
            int gi = 0, ui = 0;
#pragma unroll
            for (int w = 0; w < kRowWarps; ++w) {
              gi += __float2int_rn(pp[w * NV + (2 * r) * TMAX + t]);
              ui += __float2int_rn(pp[w * NV + (2 * r + 1) * TMAX + t]);
            }
            const float xsc_t = t < T ? xsc[t] : 0.f;
            g = __fmul_rn(__fmul_rn(__int2float_rn(gi), xsc_t), wsc[(par * 3 + 0) * RSM + r]);
            u = __fmul_rn(__fmul_rn(__int2float_rn(ui), xsc_t), wsc[(par * 3 + 1) * RSM + r]);
          } else {
#pragma unroll
            for (int w = 0; w < kRowWarps; ++w) {
              g += pp[w * NV + (2 * r) * TMAX + t];
              u += pp[w * NV + (2 * r + 1) * TMAX + t];
            }
          }
          float h = 0.f;
          if (su < 0)
            h = t < T ? tb.s[t] * silu_mul(g, u) : 0.f;
          else
            h = (tb.mask[su] >> t & 1u) ? tb.wt[su * T + t] * silu_mul(g, u) : 0.f;
          // int8: the downT row's scale goes with h (y += (h s) q)
          if constexpr (I8) h *= wsc[(par * 3 + 2) * RSM + r];
          hb[par * RSM * TMAX + j] = h;
        }
      }
      // -- C of the previous stage: y += h_r * downT_r, this thread's chunks
      if (s >= 1) {
        constexpr int pp = 1 - par;
        const float* hp = hb + pp * RSM * TMAX;
#pragma unroll
        for (int r = 0; r < RSM; ++r) {
          if (r < n_prev) {
            float hv[TMAX];
#pragma unroll
            for (int t = 0; t < TMAX; ++t) hv[t] = hp[r * TMAX + t];
#pragma unroll
            for (int k = 0; k < NCH; ++k) {
              const int ch = tid + kRowThreads * k;
              if (!FAST && ch >= H / 8) break;
              float w[8];
              float sc = 1.f;  // 4-bit: the block scale d, applied to h
              if constexpr (I8) {
                const uint2 v = dwi[pp][I8 ? r : 0][k];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  w[e] = i8_f32(v.x, e);
                  w[e + 4] = i8_f32(v.y, e);
                }
              } else if constexpr (B16) {
                const uint4 v = dwb[pp][B16 ? r : 0][k];
                w[0] = bf16_lo(v.x); w[1] = bf16_hi(v.x); w[2] = bf16_lo(v.y); w[3] = bf16_hi(v.y);
                w[4] = bf16_lo(v.z); w[5] = bf16_hi(v.z); w[6] = bf16_lo(v.w); w[7] = bf16_hi(v.w);
              } else {
                const uint32_t qw = dwq[pp][Q4 ? r : 0][k];
                sc = __half2float(__ushort_as_half(dsc[pp][Q4 ? r : 0][k]));
#pragma unroll
                for (int e = 0; e < 8; ++e) w[e] = nib_f32(qw, e);
              }
#pragma unroll
              for (int t = 0; t < TMAX; ++t) {
                if (!(m_prev >> t & 1u)) continue;
                const float c = Q4 ? hv[t] * sc : hv[t];
#pragma unroll
                for (int e = 0; e < 8; ++e) y[t][k][e] = fmaf(c, w[e], y[t][k][e]);
              }
            }
          }
        }
      }
      n_prev = n;
      m_prev = m;
    };
    for (int s = 0; s <= n_stages; s += 2) {
      step(std::integral_constant<int, 0>(), s);
      if (s + 1 <= n_stages) step(std::integral_constant<int, 1>(), s + 1);
    }
  }
  // every issued copy has been waited on (or timed out); QMC: the down-projection
  // warps meet the others here once more, after storing their partial y
  bool block_timed_out;
  if constexpr (NTB > kRowThreads)
    block_timed_out = named_bar_or(kBarSplit, NTB, timed_out);
  else
    block_timed_out = __syncthreads_or(timed_out) != 0;
  if (block_timed_out && tid == 0) {
    // leave no copy in flight into this block's shared memory: wait (bounded)
    // once more for the last stages issued
    for (int s = max(0, n_stages - NS); s < n_stages; ++s) mbar_wait(&full[s % NS], (uint32_t)(s / NS) & 1u);
    for (int s = max(0, n_stages - P.nsd); s < n_stages; ++s) mbar_wait(&fulld[s % P.nsd], (uint32_t)(s / P.nsd) & 1u);
  }

  // ---- partial y of this block
  if constexpr (MMA_C) {
    // D fragment j: columns 256w + 16j + lane/4 (and + 8), tokens 2(lane & 3) (and + 1)
    const int t0 = 2 * (lane & 3);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int c = 256 * warp + 16 * j + (lane >> 2);
      if (t0 < T) {
        P.partial[((size_t)cta * T + t0) * H + c] = yc[j][0];
        P.partial[((size_t)cta * T + t0) * H + c + 8] = yc[j][2];
      }
      if (t0 + 1 < T) {
        P.partial[((size_t)cta * T + t0 + 1) * H + c] = yc[j][1];
        P.partial[((size_t)cta * T + t0 + 1) * H + c + 8] = yc[j][3];
      }
    }
  } else if constexpr (QMC) {
    // stored by warps 8..15 (qmc_store_partial)
  } else {
    unsigned long long* mine = reinterpret_cast<unsigned long long*>(P.partial) + (size_t)cta * T * H;
#pragma unroll
    for (int t = 0; t < TMAX; ++t) {
      if (t >= T) break;
#pragma unroll
      for (int k = 0; k < NCH; ++k) {
        const int ch = tid + kRowThreads * k;
        if (!FAST && ch >= H / 8) break;
        if constexpr (TAGGED) {
          unsigned long long* dst = mine + (size_t)t * H + 8 * ch;
#pragma unroll
          for (int e = 0; e < 8; e += 2)
            st_relaxed_gpu_v2_u64(dst + e, tagged(tag, y[t][k][e]), tagged(tag, y[t][k][e + 1]), pol_keep);
        } else {
          float4* dst = reinterpret_cast<float4*>(P.partial + ((size_t)cta * T + t) * H + 8 * ch);
          dst[0] = make_float4(y[t][k][0], y[t][k][1], y[t][k][2], y[t][k][3]);
          dst[1] = make_float4(y[t][k][4], y[t][k][5], y[t][k][6], y[t][k][7]);
        }
      }
    }
  }
  // every block's partial, then the sum of this block's columns.  fp32
  // partials: the second grid-wide barrier orders all blocks' stores before
  // the reads (the block barrier orders all threads' stores before thread
  // 0's cumulative release, warp 0's acquire orders every other block's
  // stores before this block's reads).  Tagged partials (one token): each read
  // polls its word until it carries the call's tag; the first barrier
  // already ordered every block's reads of x before any block writes out.
  // This block's output columns [da, db) for all tokens (O values).  In the
  // block form the residual x_res of those columns is read now: no other
  // block writes them, and every block read all of x at its start.
  const int da = (int)muldiv(H, cta, P.G), db = (int)muldiv(H, cta + 1, P.G);
  const int nD = db - da, O = T * nD;
  float resid = 0.f;
  if (P.block_mode && tid < O) resid = __ldcg(P.out + (size_t)(tid / nD) * H + da + tid % nD);
  bool tail_timed_out = false;
  if constexpr (!TAGGED) tail_timed_out = !grid_barrier<SYNC_NT>(sync, 1, fast_sync, P.G, epoch, cta, false);
  // The O sums of G partials.  Thread (sp, o) adds partials sp, sp + S, ...
  // in order, up to 16 loads in flight together; the S part sums are then
  // added in order.
  bool sums_timed_out = false;
  const int S = O >= kRowThreads ? 1 : kRowThreads / max(O, 1);
  // The ring is idle now (every issued stage was waited on); reuse it.
  float* red = reinterpret_cast<float*>(ring);  // [S][O]
  for (int idx = tid; idx < S * O; idx += kRowThreads) {
    const int o = idx % O, sp = idx / O;
    const int t = o / nD, col = da + o % nD;
    const size_t stride = (size_t)T * H;
    float acc = 0.f;
    for (int c0 = sp; c0 < P.G; c0 += 16 * S) {
      float v[16];
      if constexpr (TAGGED) {
        const unsigned long long* src = reinterpret_cast<const unsigned long long*>(P.partial) + (size_t)t * H + col;
        const int n = min(16, (P.G - 1 - c0) / S + 1);
        if (!poll_tagged<16>(src + (size_t)c0 * stride, (size_t)S * stride, n, tag, v)) sums_timed_out = true;
      } else {
        const float* src = P.partial + (size_t)t * H + col;
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const int c = c0 + q * S;
          v[q] = c < P.G ? __ldcg(src + (size_t)c * stride) : 0.f;
        }
      }
#pragma unroll
      for (int q = 0; q < 16; ++q)
        if (c0 + q * S < P.G) acc += v[q];
    }
    red[sp * O + o] = acc;
  }
  if (blk_sync_or<SYNC_NT>(sums_timed_out)) tail_timed_out = true;
  for (int oo = tid; oo < O; oo += kRowThreads) {
    float acc = red[oo];
    for (int q = 1; q < S; ++q) acc += red[q * O + oo];
    const int t = oo / nD, col = da + oo % nD;
    float* dst = P.out + (size_t)t * H + col;
    *dst = P.block_mode ? __fadd_rn(oo < kRowThreads ? resid : *dst, acc) : acc;
  }
  if (tid == 0) sync->status[cta] = tail_timed_out || block_timed_out ? kStatusTimeout : 0;
}

// Per device, once per instance and shared-memory size: the kernel's dynamic
// shared-memory limit, and a check that one block fits on an SM next to
// nothing else of this kernel -- the combine's grid barrier needs all G
// blocks (G <= the SM count) resident at once.  A launch whose blocks could
// not all be resident is refused (cudaErrorCooperativeLaunchTooLarge) instead
// of ending in a timed-out barrier.
template <int TMAX, int WK, bool FAST, int NCH>
inline cudaError_t rows_configure(int smem, int G) {
  // one record per instance (the statics of each template instantiation)
  auto* const kern = k_rows<TMAX, WK, FAST, NCH>;
  constexpr int kDevs = 64;
  static std::atomic<int> done_smem[kDevs];
  static std::mutex mu;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kDevs) return cudaErrorInvalidDevice;
  if (done_smem[dev].load(std::memory_order_acquire) >= smem) return cudaSuccess;
  std::lock_guard<std::mutex> lock(mu);
  if (done_smem[dev].load(std::memory_order_relaxed) >= smem) return cudaSuccess;
  err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  int per_sm = 0, sms = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, rows_threads(WK, FAST), smem);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  if ((long long)per_sm * sms < G) return cudaErrorCooperativeLaunchTooLarge;
  done_smem[dev].store(smem, std::memory_order_release);
  return cudaSuccess;
}

template <int TMAX, int WK, bool FAST, int NCH = 1>
inline cudaError_t launch_rows_t(const LayerParams& p, cudaStream_t stream) {
  cudaError_t err = rows_configure<TMAX, WK, FAST, NCH>(p.smem, p.G);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(p.G);
  cfg.blockDim = dim3(rows_threads(WK, FAST));
  cfg.dynamicSmemBytes = p.smem;
  return cudaLaunchKernelEx(&cfg, k_rows<TMAX, WK, FAST, NCH>, p);
}

}  // namespace moe
