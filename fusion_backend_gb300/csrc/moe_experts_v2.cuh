#pragma once
// Per-warp-ring expert kernel: the decode fast path of the fused MoE FFN
// layer, sm_103a.  Instantiated by moe_experts_v2_bf16.cu and
// moe_experts_v2_q4.cu.
//
// One persistent CTA per SM with `nw` warps.
// Every consumer warp owns a private ring of shared-memory slots that its
// lane 0 fills with bulk copies (TMA engine) ahead of use and processes whole
// weight rows, so dot-product reductions stay inside the warp and no
// CTA-wide barrier is taken per item.  Work per warp, in order:
//   S  its share of the shared expert's gate/up row pairs
//   R  its share of the routed experts' gate/up row pairs: h = silu(g) * u
//   D  its share of the (down group, output row) pairs of this CTA, where the
//      groups are the shared expert and every selected expert
// The routing is computed first (the shared-expert rows stream meanwhile).
// Down-matrix rows stream into the rings while every CTA of the grid
// publishes its h (a counter that thread 0 waits on, bounded); then
// the staged h of all groups is read from shared memory and the CTA combines
// out = sum_j p_j y_j + s y_sh for its rows in a fixed order.
//
// With one token, partial dot products of several rows are kept per lane and
// reduced together (9 shuffles for 8 values), which hides the shuffle
// latency; several tokens use one butterfly per (row, token).
//
// 4-bit weights are decoded with the fp16 exponent trick: a nibble n OR-ed
// into the mantissa of the fp16 constant 1024 reads as 1024 + n, so
// (1024 + n) - 1032 = n - 8 exactly; products n*x and their block sums are
// formed with packed half2 FMAs and scaled by the block's d in fp32.

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "moe_decode_common.cuh"

namespace moe {

constexpr int kV2MaxWarps = 8;
constexpr int kBarV2Cons = 3;  // all warps of the CTA
constexpr int kV2MaxCols = 1024;  // I and Is of the fast path
constexpr int kV2H = 2048;        // H of the fast path

enum : int { kXReg = 0, kXF32 = 1, kXH2 = 2 };
enum : int { kHF32 = 0, kHBF16 = 1, kHH2 = 2 };

struct V2Tab {
  int32_t* ids;
  float* p;
  float* s;
  float* inv;
  int32_t* counts;
  int32_t* offsets;
  int16_t* inv_u;
  int32_t* active;
  uint32_t* mask;
  int32_t* pre;    // tokens of the active experts before u (exclusive prefix)
  int32_t* goff;   // element offset of each down group's h in shared memory
  int32_t* hsrc;   // per staged h row: >= 0 routed (t,slot) row, < 0: -(1+t) shared row t
  int32_t* hdst;   // per staged h row: element offset in shared memory
  int16_t* tsmap;  // [U][T] flat (t*K + j) of token t for active expert u
  int32_t* misc;   // [0] U
  float* ys;       // [T*K + T][rows_cta] down outputs of this CTA's rows
};

__host__ __device__ inline int v2_tab(uint8_t* base, int T, int K, int E, int rows_cta, V2Tab* v) {
  const int TK = T * K;
  const int sz[16] = {TK * 4, TK * 4, T * 4, T * 8, E * 4, (E + 1) * 4, E * 2, TK * 4,
                      TK * 4, TK * 4, (TK + 2) * 4, (TK + T) * 4, (TK + T) * 4, TK * T * 2, 16 * 4,
                      (TK + T) * rows_cta * 4};
  int off = 0, o[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    o[i] = off;
    off += (sz[i] + 15) & ~15;
  }
  if (v && base) {
    v->ids = reinterpret_cast<int32_t*>(base + o[0]);
    v->p = reinterpret_cast<float*>(base + o[1]);
    v->s = reinterpret_cast<float*>(base + o[2]);
    v->inv = reinterpret_cast<float*>(base + o[3]);
    v->counts = reinterpret_cast<int32_t*>(base + o[4]);
    v->offsets = reinterpret_cast<int32_t*>(base + o[5]);
    v->inv_u = reinterpret_cast<int16_t*>(base + o[6]);
    v->active = reinterpret_cast<int32_t*>(base + o[7]);
    v->mask = reinterpret_cast<uint32_t*>(base + o[8]);
    v->pre = reinterpret_cast<int32_t*>(base + o[9]);
    v->goff = reinterpret_cast<int32_t*>(base + o[10]);
    v->hsrc = reinterpret_cast<int32_t*>(base + o[11]);
    v->hdst = reinterpret_cast<int32_t*>(base + o[12]);
    v->tsmap = reinterpret_cast<int16_t*>(base + o[13]);
    v->misc = reinterpret_cast<int32_t*>(base + o[14]);
    v->ys = reinterpret_cast<float*>(base + o[15]);
  }
  return off;
}

struct V2Ctx {
  int sa, sb;        // shared gate/up row pairs of this warp
  long long fa, fb;  // routed (active expert, row) pairs of this warp, flattened
  int fa_u, fa_i;    // fa as (active index, row)
  int da, nD;        // this CTA's output rows [da, da + nD)
  int dfa, dfb;      // this warp's (group, row) pairs, flattened group-major
  int dfa_g, dfa_r;  // dfa as (group, row offset)
  int U;
  bool routed;
};

struct V2Unit {
  int kind;  // 0 shared gate/up, 1 routed gate/up, 2 down rows of one group
  int a;     // S: first row; R: active index; D: group (0 shared, 1 + u routed)
  int b;     // R: first row; D: first output row (absolute)
  int n;     // row pairs (S, R) or rows (D)
};

struct V2It {
  int phase;
  long long pos;
  int ua, i;
};

MOE_DEV int v2_rb_group(const DecodeParams& P, int g) { return g == 0 ? P.rbIs : P.rbI; }

MOE_DEV bool v2_next(V2It& it, const V2Ctx& c, const DecodeParams& P, V2Unit& u) {
  if (it.phase == 0) {
    if (it.pos < c.sb) {
      const int n = min(P.v2_cap_gu, c.sb - (int)it.pos);
      u = V2Unit{0, (int)it.pos, 0, n};
      it.pos += n;
      return true;
    }
    if (!c.routed) return false;
    it.phase = 1;
    it.pos = c.fa;
    it.ua = c.fa_u;
    it.i = c.fa_i;
  }
  if (it.phase == 1) {
    if (it.pos < c.fb) {
      const int n = (int)min((long long)min(P.v2_cap_gu, P.I - it.i), c.fb - it.pos);
      u = V2Unit{1, it.ua, it.i, n};
      it.pos += n;
      it.i += n;
      if (it.i >= P.I) {
        it.i = 0;
        ++it.ua;
      }
      return true;
    }
    it.phase = 2;
    it.pos = c.dfa;
    it.ua = c.dfa_g;
    it.i = c.dfa_r;
  }
  if (it.phase == 2) {
    if (it.pos < c.dfb) {
      const int cap = min(P.v2_slot / v2_rb_group(P, it.ua), P.wfmt == 1 ? 8 : 2);
      const int n = (int)min((long long)min(cap, c.nD - it.i), (long long)c.dfb - it.pos);
      u = V2Unit{2, it.ua, c.da + it.i, n};
      it.pos += n;
      it.i += n;
      if (it.i >= c.nD) {
        it.i = 0;
        ++it.ua;
      }
      return true;
    }
    it.phase = 3;
  }
  return false;
}

MOE_DEV void v2_issue(const DecodeParams& P, const V2Tab& tb, const V2Unit& u, uint8_t* slot, uint64_t* bar,
                      uint64_t pol) {
  if (u.kind <= 1) {
    const uint8_t* base;
    long long mat;
    int row0;
    if (u.kind == 0) {
      base = P.shexp_w;
      mat = P.sgu_bytes;
      row0 = u.a;
    } else {
      base = P.expert_w + (size_t)tb.active[u.a] * P.expert_bytes;
      mat = P.gu_bytes;
      row0 = u.b;
    }
    const uint32_t bytes = (uint32_t)u.n * P.rbH;
    mbar_arrive_expect_tx(bar, 2 * bytes);
    bulk_g2s(slot, base + (size_t)row0 * P.rbH, bytes, bar, pol);
    bulk_g2s(slot + bytes, base + mat + (size_t)row0 * P.rbH, bytes, bar, pol);
  } else {
    const int rb = v2_rb_group(P, u.a);
    const uint8_t* src = u.a == 0 ? P.shexp_w + 2 * P.sgu_bytes
                                  : P.expert_w + (size_t)tb.active[u.a - 1] * P.expert_bytes + 2 * P.gu_bytes;
    const uint32_t bytes = (uint32_t)(u.n * rb);
    mbar_arrive_expect_tx(bar, bytes);
    bulk_g2s(slot, src + (size_t)u.b * rb, bytes, bar, pol);
  }
}

// One entry of a warp's unit list (built once; the copy issue and the
// consumer loop then only index it).
struct V2U {
  const uint8_t* src;  // first copy source
  int info;            // kind (bits 0-1) | n (bits 2-9) | group or active index (bits 10..)
  int row0;            // first row
};
constexpr int kV2ListLen = 96;

MOE_DEV int v2_build_s(const DecodeParams& P, const V2Ctx& c, V2U* L) {
  int k = 0;
  for (int i = c.sa; i < c.sb; i += P.v2_cap_gu) {
    const int n = min(P.v2_cap_gu, c.sb - i);
    L[k++] = V2U{P.shexp_w + (size_t)i * P.rbH, 0 | (n << 2), i};
  }
  return k;
}

MOE_DEV int v2_build_rd(const DecodeParams& P, const V2Tab& tb, const V2Ctx& c, V2U* L, int k) {
  long long pos = c.fa;
  int ua = c.fa_u, i = c.fa_i;
  while (pos < c.fb) {
    const int n = (int)min((long long)min(P.v2_cap_gu, P.I - i), c.fb - pos);
    L[k++] = V2U{P.expert_w + (size_t)tb.active[ua] * P.expert_bytes + (size_t)i * P.rbH, 1 | (n << 2) | (ua << 10), i};
    pos += n;
    i += n;
    if (i >= P.I) {
      i = 0;
      ++ua;
    }
  }
  int dpos = c.dfa, g = c.dfa_g, r = c.dfa_r;
  while (dpos < c.dfb) {
    const int rb = v2_rb_group(P, g);
    const int cap = min(P.v2_slot / rb, P.wfmt == 1 ? 8 : 2);
    const int n = min(min(cap, c.nD - r), c.dfb - dpos);
    const uint8_t* base = g == 0 ? P.shexp_w + 2 * P.sgu_bytes
                                 : P.expert_w + (size_t)tb.active[g - 1] * P.expert_bytes + 2 * P.gu_bytes;
    L[k++] = V2U{base + (size_t)(c.da + r) * rb, 2 | (n << 2) | (g << 10), c.da + r};
    dpos += n;
    r += n;
    if (r >= c.nD) {
      r = 0;
      ++g;
    }
  }
  return k;
}

// ------------------------------------------------------------ 4-bit helpers
MOE_DEV uint32_t lop3_and_or(uint32_t a, uint32_t m, uint32_t c) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(m), "r"(c));
  return r;
}
MOE_DEV uint32_t h2_sub(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
MOE_DEV uint32_t h2_fma(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}
MOE_DEV float h2_sum(uint32_t a) {
  const __half2 h = *reinterpret_cast<const __half2*>(&a);
  const float2 f = __half22float2(h);
  return f.x + f.y;
}
MOE_DEV uint32_t pack_h2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// 32 codes of one block (16 bytes, element 2j in the low nibble of byte j)
// -> 16 half2 of (n - 8), ordered per 8-column quarter k as
// (c0,c4) (c1,c5) (c2,c6) (c3,c7) with c = 8k + i.
MOE_DEV void dequant_block(const uint4 q, uint32_t* o) {
  const uint32_t words[4] = {q.x, q.y, q.z, q.w};
  constexpr uint32_t kMagic = 0x64006400u;  // fp16 1024 in both halves
  constexpr uint32_t kSub = 0x64086408u;    // fp16 1032
  constexpr uint32_t kSixteenth = 0x2C002C00u;  // fp16 1/16
  constexpr uint32_t kMinus72 = 0xD480D480u;    // fp16 -72
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t w = words[k];
    const uint32_t w8 = w >> 8;
    o[4 * k + 0] = h2_sub(lop3_and_or(w, 0x000F000Fu, kMagic), kSub);
    o[4 * k + 1] = h2_fma(lop3_and_or(w, 0x00F000F0u, kMagic), kSixteenth, kMinus72);
    o[4 * k + 2] = h2_sub(lop3_and_or(w8, 0x000F000Fu, kMagic), kSub);
    o[4 * k + 3] = h2_fma(lop3_and_or(w8, 0x00F000F0u, kMagic), kSixteenth, kMinus72);
  }
}

// Byte offset of quarter k of block b in the swizzled fp16 block layout
// (64 bytes per block; rotating the quarters by (b >> 1) keeps the 16-byte
// reads of consecutive lanes on distinct banks).
MOE_DEV int h2_quarter_off(int b, int k) { return b * 64 + 16 * ((k + (b >> 1)) & 3); }

// Eight consecutive values c = 8q .. 8q+7 of a row -> the uint4 of quarter q%4.
MOE_DEV uint4 pack_quarter(const float* v) {
  return make_uint4(pack_h2(v[0], v[4]), pack_h2(v[1], v[5]), pack_h2(v[2], v[6]), pack_h2(v[3], v[7]));
}


// Address of element `col` of an h row (row base `row`) in the staged format.
MOE_DEV uint8_t* h_elem_addr(uint8_t* row, int col, int hmode) {
  if (hmode == kHF32) return row + (size_t)col * 4;
  if (hmode == kHBF16) return row + (size_t)col * 2;
  const int b = col / 32, w = col % 32, k = w / 8, e = w % 8;
  return row + h2_quarter_off(b, k) + 4 * (e % 4) + 2 * (e / 4);
}
MOE_DEV void h_store(uint8_t* p, float v, int hmode) {
  if (hmode == kHF32)
    *reinterpret_cast<float*>(p) = v;
  else if (hmode == kHBF16)
    *reinterpret_cast<uint16_t*>(p) = float_to_bf16_rne(v);
  else
    *reinterpret_cast<__half*>(p) = __float2half_rn(v);
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

// Rows of one group's y whose lane partials wait for a batched reduction
// (one token): up to 8 (row, value) entries.
struct PendY {
  float v[8];
  int dst[8];  // index into ys
  int n;
  MOE_DEV void clear() {
#pragma unroll
    for (int q = 0; q < 8; ++q) v[q] = 0.f;
    n = 0;
  }
  MOE_DEV void push(float x, int d) {
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (q == n) {
        v[q] = x;
        dst[q] = d;
      }
    ++n;
  }
  MOE_DEV void flush(float* ys) {
    if (n == 0) return;
    const float r = warp_reduce8(v);
    const int lane = threadIdx.x & 31, q = lane >> 2;
    if ((lane & 3) == 0 && q < n) {
      int d = dst[0];
#pragma unroll
      for (int k = 1; k < 8; ++k)
        if (k == q) d = dst[k];
      ys[d] = r;
    }
    clear();
  }
};

// Gate/up row pairs waiting for a batched reduction (one token): up to 4.
struct PendH {
  float v[8];  // (g, u) of row q in v[2q], v[2q+1]
  uint8_t* dst[4];
  int n;
  MOE_DEV void clear() {
#pragma unroll
    for (int q = 0; q < 8; ++q) v[q] = 0.f;
    n = 0;
  }
  MOE_DEV void push(float g, float u, uint8_t* d) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (q == n) {
        v[2 * q] = g;
        v[2 * q + 1] = u;
        dst[q] = d;
      }
    ++n;
  }
  MOE_DEV void flush(int hmode) {
    if (n == 0) return;
    const float r = warp_reduce8(v);
    const float u = __shfl_down_sync(0xffffffffu, r, 4);
    const int lane = threadIdx.x & 31, q = lane >> 3;
    if ((lane & 7) == 0 && q < n) {
      uint8_t* d = dst[0];
#pragma unroll
      for (int k = 1; k < 4; ++k)
        if (k == q) d = dst[k];
      h_store(d, r / (1.0f + expf(-r)) * u, hmode);
    }
    clear();
  }
};


// ------------------------------------------------------------------- kernel
template <int TMAX, bool Q4, bool XREG>
__global__ void __launch_bounds__(kV2MaxWarps * 32, 1) k_experts_v2(DecodeParams P) {
  extern __shared__ __align__(1024) uint8_t sm[];
  const int nw = P.v2_nw;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cta = blockIdx.x;
  const int T = P.T, K = P.K, TK = P.T * P.K;
  const int nslots = P.v2_nslots;
  const int hmode = P.v2_hmode;
  const int hel = hmode == kHF32 ? 4 : 2;  // bytes per staged h element
  uint64_t* fbar = reinterpret_cast<uint64_t*>(sm + P.v2_off_bar);
  uint64_t* aux_bar = fbar + kV2MaxWarps * 4;      // router logits copy
  uint64_t* hst_bar = fbar + kV2MaxWarps * 4 + 1;  // h staging copies
  uint8_t* ring = sm + P.v2_off_ring;
  uint8_t* uni = sm + P.v2_off_union;
  int da, db;
  down_rows(P, cta, da, db);
  const int nD = db - da;
  V2Tab tb;
  v2_tab(sm + P.v2_off_tab, T, K, P.E, P.v2_rows_w, &tb);
  const int xsz = XREG ? 0 : (Q4 ? T * P.H * 2 : T * P.H * 4);
  float* lgs = reinterpret_cast<float*>(uni + xsz);

  // Let the next call's router kernel start and prefetch its weights.
  pdl_launch_dependents();

  if (tid == 0) {
    for (int i = 0; i < nw * nslots; ++i) mbar_init(&fbar[i], 1);
    mbar_init(aux_bar, 1);
    mbar_init(hst_bar, 1);
    mbar_fence_init();
  }
  if (P.block_mode) {
    for (int t = warp; t < T; t += nw) {
      float hi, lo;
      warp_norm_factor(static_cast<const float*>(P.x) + (size_t)t * P.H, P.H, P.eps, hi, lo);
      if (lane == 0) {
        tb.inv[2 * t] = hi;
        tb.inv[2 * t + 1] = lo;
      }
    }
  }
  __syncthreads();
  if (!XREG) {
    // x of all tokens into shared memory: fp32 rows, or the fp16 block layout.
    const int groups = T * (P.H / 8);
    for (int gi = tid; gi < groups; gi += blockDim.x) {
      const int t = gi / (P.H / 8), q = gi % (P.H / 8);
      float v[8];
      load_x8_any(P, tb.inv, t, 8 * q, v);
      if (Q4) {
        *reinterpret_cast<uint4*>(uni + (size_t)t * P.H * 2 + h2_quarter_off(q / 4, q % 4)) = pack_quarter(v);
      } else {
        float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(uni) + (size_t)t * P.H + 8 * q);
        dst[0] = make_float4(v[0], v[1], v[2], v[3]);
        dst[1] = make_float4(v[4], v[5], v[6], v[7]);
      }
    }
    __syncthreads();
  }

  // ==================================================== consumer warps
  const uint32_t all_tokens = (1u << T) - 1u;
  V2Ctx c;
  {
    const int a = div_floor_ll((long long)P.Is * cta, P.G), b = div_floor_ll((long long)P.Is * (cta + 1), P.G);
    c.sa = a + (b - a) * warp / nw;
    c.sb = a + (b - a) * (warp + 1) / nw;
    c.da = da;
    c.nD = nD;
    c.fa = c.fb = 0;
    c.fa_u = c.fa_i = 0;
    c.dfa = c.dfb = c.dfa_g = c.dfa_r = 0;
    c.U = 0;
    c.routed = false;
  }
  uint8_t* my_ring = ring + (size_t)warp * nslots * P.v2_slot;
  uint64_t* my_bar = fbar + warp * nslots;
  const uint64_t pol = policy_evict_first();
  const uint64_t pol_keep = policy_evict_last();

  // x of token 0 in registers (one token): bf16 path 8 columns per 256-column
  // chunk, 4-bit path the 16 half2 of each of the lane's 32-column blocks.
  float xr[XREG && !Q4 ? 8 : 1][8];
  uint32_t xh[XREG && Q4 ? 2 : 1][16];
  if (XREG) {
    if (!Q4) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int c0 = 256 * j + 8 * lane;
        if (c0 < P.H) load_x8_any(P, tb.inv, 0, c0, xr[j]);
      }
    } else {
#pragma unroll
      for (int jb = 0; jb < 2; ++jb) {
        const int b = lane + 32 * jb;
        if (b < P.H / 32) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            float v[8];
            load_x8_any(P, tb.inv, 0, 32 * b + 8 * k, v);
            const uint4 qv = pack_quarter(v);
            xh[jb][4 * k + 0] = qv.x;
            xh[jb][4 * k + 1] = qv.y;
            xh[jb][4 * k + 2] = qv.z;
            xh[jb][4 * k + 3] = qv.w;
          }
        }
      }
    }
  }

  // This warp's unit list: the shared-expert units now, the routed and down
  // units once the routing is known.  `k_iss` copies into the ring up to
  // nslots units ahead of `k_con`, which consumes.
  V2U* L = reinterpret_cast<V2U*>(sm + P.v2_off_list) + (size_t)warp * kV2ListLen;
  int n_units = 0, n_gu = 0;
  if (lane == 0) n_units = v2_build_s(P, c, L);
  n_units = __shfl_sync(0xffffffffu, n_units, 0);
  __syncwarp();
  int k_iss = 0, k_con = 0;
  auto pump = [&]() {
    while (k_iss < k_con + nslots && k_iss < n_units) {
      const V2U d = L[k_iss];
      const int sl = k_iss % nslots;
      uint8_t* dst = my_ring + (size_t)sl * P.v2_slot;
      uint64_t* bar = &my_bar[sl];
      const int kind = d.info & 3, n = (d.info >> 2) & 255;
      if (kind <= 1) {
        const uint32_t bytes = (uint32_t)n * P.rbH;
        mbar_arrive_expect_tx(bar, 2 * bytes);
        bulk_g2s(dst, d.src, bytes, bar, pol);
        bulk_g2s(dst + bytes, d.src + (kind == 0 ? P.sgu_bytes : P.gu_bytes), bytes, bar, pol);
      } else {
        const uint32_t bytes = (uint32_t)(n * v2_rb_group(P, d.info >> 10));
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s(dst, d.src, bytes, bar, pol);
      }
      ++k_iss;
    }
  };
  if (lane == 0) pump();

  PendH pend_h;
  pend_h.clear();
  PendY pend_y;
  pend_y.clear();

  // A unit's weights are copied from its ring slot into registers first; the
  // slot is then released (and refilled) before any arithmetic, so the ring
  // keeps nslots copies in flight whatever the compute latency.
  auto release = [&]() {
    __syncwarp();
    ++k_con;
    if (lane == 0) pump();
  };

  // ---- gate/up row pairs: h = silu(gate x) * (up x), written to global h in
  // the format the down phase stages (fp32, bf16 or the fp16 block layout).
  // The fast path has H = 2048: 8 chunks of 8 bf16 columns per lane, or 2
  // blocks of 32 4-bit columns per lane.
  auto do_gu = [&](const V2Unit& u, const uint8_t* slot) {
    const uint32_t m = u.kind == 0 ? all_tokens : tb.mask[u.a];
    const int cols = u.kind == 0 ? P.Is : P.I;
    uint8_t* hbase = reinterpret_cast<uint8_t*>(u.kind == 0 ? P.hsh : P.h);
    const int row0 = u.kind == 0 ? u.a : u.b;
    constexpr int RU = Q4 ? 3 : 1;  // row pairs per unit
    float gsum[RU][TMAX], usum[RU][TMAX];
#pragma unroll
    for (int rr = 0; rr < RU; ++rr)
#pragma unroll
      for (int t = 0; t < TMAX; ++t) gsum[rr][t] = usum[rr][t] = 0.f;
    if (!Q4) {
      uint4 wg[8], wu[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        wg[j] = *reinterpret_cast<const uint4*>(slot + (size_t)(256 * j + 8 * lane) * 2);
        wu[j] = *reinterpret_cast<const uint4*>(slot + kV2H * 2 + (size_t)(256 * j + 8 * lane) * 2);
      }
      release();
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
        if (!(m >> t & 1u)) continue;
        float g4[4] = {0.f, 0.f, 0.f, 0.f}, u4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float xv[8];
          if (XREG) {
#pragma unroll
            for (int e = 0; e < 8; ++e) xv[e] = xr[XREG && !Q4 ? j : 0][e];
          } else {
            const float4* xp =
                reinterpret_cast<const float4*>(reinterpret_cast<const float*>(uni) + (size_t)t * kV2H + 256 * j + 8 * lane);
            const float4 a = xp[0], b = xp[1];
            xv[0] = a.x; xv[1] = a.y; xv[2] = a.z; xv[3] = a.w;
            xv[4] = b.x; xv[5] = b.y; xv[6] = b.z; xv[7] = b.w;
          }
          const uint32_t gw[4] = {wg[j].x, wg[j].y, wg[j].z, wg[j].w};
          const uint32_t uw[4] = {wu[j].x, wu[j].y, wu[j].z, wu[j].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            g4[j & 3] = fmaf(bf16_lo(gw[e]), xv[2 * e], g4[j & 3]);
            g4[j & 3] = fmaf(bf16_hi(gw[e]), xv[2 * e + 1], g4[j & 3]);
            u4[j & 3] = fmaf(bf16_lo(uw[e]), xv[2 * e], u4[j & 3]);
            u4[j & 3] = fmaf(bf16_hi(uw[e]), xv[2 * e + 1], u4[j & 3]);
          }
        }
        gsum[0][t] = (g4[0] + g4[1]) + (g4[2] + g4[3]);
        usum[0][t] = (u4[0] + u4[1]) + (u4[2] + u4[3]);
      }
    } else {
      uint4 qg[RU][2], qu[RU][2];
      uint32_t dd[RU][2];  // fp16 bits: d of gate (low) and up (high)
#pragma unroll
      for (int rr = 0; rr < RU; ++rr) {
        if (rr >= u.n) break;
        const uint8_t* rg = slot + (size_t)rr * P.rbH;
        const uint8_t* ru = slot + (size_t)(u.n + rr) * P.rbH;
#pragma unroll
        for (int jb = 0; jb < 2; ++jb) {
          const int b = lane + 32 * jb;
          qg[rr][jb] = *reinterpret_cast<const uint4*>(rg + 16 * b);
          qu[rr][jb] = *reinterpret_cast<const uint4*>(ru + 16 * b);
          dd[rr][jb] = (uint32_t)*reinterpret_cast<const uint16_t*>(rg + kV2H / 2 + 2 * b) |
                       ((uint32_t)*reinterpret_cast<const uint16_t*>(ru + kV2H / 2 + 2 * b) << 16);
        }
      }
      release();
#pragma unroll
      for (int rr = 0; rr < RU; ++rr) {
        if (rr >= u.n) break;
#pragma unroll
        for (int jb = 0; jb < 2; ++jb) {
          const int b = lane + 32 * jb;
          uint32_t q1[16], q2[16];
          dequant_block(qg[rr][jb], q1);
          dequant_block(qu[rr][jb], q2);
          const __half2 dh = *reinterpret_cast<const __half2*>(&dd[rr][jb]);
          const float dg = __low2float(dh), du = __high2float(dh);
#pragma unroll
          for (int t = 0; t < TMAX; ++t) {
            if (!(m >> t & 1u)) continue;
            uint32_t xv[16];
            if (XREG) {
#pragma unroll
              for (int i = 0; i < 16; ++i) xv[i] = xh[XREG && Q4 ? jb : 0][i];
            } else {
              const uint8_t* xb = uni + (size_t)t * kV2H * 2;
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const uint4 v = *reinterpret_cast<const uint4*>(xb + h2_quarter_off(b, k));
                xv[4 * k] = v.x; xv[4 * k + 1] = v.y; xv[4 * k + 2] = v.z; xv[4 * k + 3] = v.w;
              }
            }
            uint32_t g0 = 0u, g1 = 0u, u0 = 0u, u1 = 0u;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              g0 = h2_fma(q1[2 * i], xv[2 * i], g0);
              g1 = h2_fma(q1[2 * i + 1], xv[2 * i + 1], g1);
              u0 = h2_fma(q2[2 * i], xv[2 * i], u0);
              u1 = h2_fma(q2[2 * i + 1], xv[2 * i + 1], u1);
            }
            gsum[rr][t] = fmaf(dg, h2_sum(g0) + h2_sum(g1), gsum[rr][t]);
            usum[rr][t] = fmaf(du, h2_sum(u0) + h2_sum(u1), usum[rr][t]);
          }
        }
      }
    }
    if (TMAX == 1) {
      // one token: defer the reductions, four row pairs at a time
#pragma unroll
      for (int rr = 0; rr < RU; ++rr) {
        if (rr >= u.n) break;
        const size_t hrow = u.kind == 0 ? 0 : (size_t)tb.tsmap[u.a * T];
        pend_h.push(gsum[rr][0], usum[rr][0], h_elem_addr(hbase + hrow * cols * hel, row0 + rr, hmode));
        if (pend_h.n == 4) pend_h.flush(hmode);
      }
    } else {
#pragma unroll
      for (int o = 16; o; o >>= 1) {
#pragma unroll
        for (int rr = 0; rr < RU; ++rr)
#pragma unroll
          for (int t = 0; t < TMAX; ++t) {
            if ((m >> t & 1u) && rr < u.n) {
              gsum[rr][t] += __shfl_xor_sync(0xffffffffu, gsum[rr][t], o);
              usum[rr][t] += __shfl_xor_sync(0xffffffffu, usum[rr][t], o);
            }
          }
      }
#pragma unroll
      for (int rr = 0; rr < RU; ++rr) {
        if (rr >= u.n) break;
        float hsel = 0.f;
#pragma unroll
        for (int t = 0; t < TMAX; ++t)
          if (lane == t) hsel = gsum[rr][t] / (1.0f + expf(-gsum[rr][t])) * usum[rr][t];
        if (lane < TMAX && (m >> lane & 1u)) {
          const size_t hrow = u.kind == 0 ? (size_t)lane : (size_t)tb.tsmap[u.a * T + lane];
          h_store(h_elem_addr(hbase + hrow * cols * hel, row0 + rr, hmode), hsel, hmode);
        }
      }
    }
  };

  // ---- down rows of one group: y[ts][row] into ys (this CTA's rows).
  // Up to kV2DownRows rows per unit: bf16 4 chunks of 8 columns per lane
  // (cols <= 1024), 4-bit one 32-column block per lane.
  int hg_cur = -1;
  float hreg[XREG && !Q4 ? 4 : 1][8];  // one token, bf16 path: h of the current group
  uint32_t hq[XREG && Q4 ? 16 : 1];     // one token, 4-bit path
  auto do_down = [&](const V2Unit& u, const uint8_t* slot) {
    const int g = u.a;
    const bool shared = g == 0;
    const int cols = shared ? P.Is : P.I;
    const int rb = shared ? P.rbIs : P.rbI;
    const uint32_t m = shared ? all_tokens : tb.mask[g - 1];
    const int ntok = __popc(m);
    const uint8_t* hg = uni + (size_t)tb.goff[g] * hel;
    constexpr int RD = Q4 ? 8 : 2;
    float acc[RD][TMAX];
#pragma unroll
    for (int rr = 0; rr < RD; ++rr)
#pragma unroll
      for (int t = 0; t < TMAX; ++t) acc[rr][t] = 0.f;
    if (!Q4) {
      uint4 w[RD][4];
#pragma unroll
      for (int rr = 0; rr < RD; ++rr) {
        if (rr >= u.n) break;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int c0 = 256 * j + 8 * lane;
          if (c0 < cols) w[rr][j] = *reinterpret_cast<const uint4*>(slot + (size_t)rr * rb + (size_t)c0 * 2);
        }
      }
      release();
      if (TMAX == 1 && hg_cur != g) {
        hg_cur = g;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int c0 = 256 * j + 8 * lane;
          if (c0 < cols) {
            if (hmode == kHF32) {
              const float4* hp = reinterpret_cast<const float4*>(hg + (size_t)c0 * 4);
              const float4 a = hp[0], b = hp[1];
              const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
              for (int e = 0; e < 8; ++e) hreg[XREG && !Q4 ? j : 0][e] = v[e];
            } else {
              const uint4 hb = *reinterpret_cast<const uint4*>(hg + (size_t)c0 * 2);
              const uint32_t w4[4] = {hb.x, hb.y, hb.z, hb.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                hreg[XREG && !Q4 ? j : 0][2 * e] = bf16_lo(w4[e]);
                hreg[XREG && !Q4 ? j : 0][2 * e + 1] = bf16_hi(w4[e]);
              }
            }
          }
        }
      }
#pragma unroll
      for (int rr = 0; rr < RD; ++rr) {
        if (rr >= u.n) break;
#pragma unroll
        for (int t = 0; t < TMAX; ++t) {
          if (t >= ntok) continue;
          float a2[2] = {0.f, 0.f};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int c0 = 256 * j + 8 * lane;
            if (c0 < cols) {
              float hv[8];
              if (TMAX == 1) {
#pragma unroll
                for (int e = 0; e < 8; ++e) hv[e] = hreg[XREG && !Q4 ? j : 0][e];
              } else if (hmode == kHF32) {
                const float4* hp = reinterpret_cast<const float4*>(hg + ((size_t)t * cols + c0) * 4);
                const float4 a = hp[0], b = hp[1];
                hv[0] = a.x; hv[1] = a.y; hv[2] = a.z; hv[3] = a.w;
                hv[4] = b.x; hv[5] = b.y; hv[6] = b.z; hv[7] = b.w;
              } else {
                const uint4 hb = *reinterpret_cast<const uint4*>(hg + ((size_t)t * cols + c0) * 2);
                hv[0] = bf16_lo(hb.x); hv[1] = bf16_hi(hb.x); hv[2] = bf16_lo(hb.y); hv[3] = bf16_hi(hb.y);
                hv[4] = bf16_lo(hb.z); hv[5] = bf16_hi(hb.z); hv[6] = bf16_lo(hb.w); hv[7] = bf16_hi(hb.w);
              }
              const uint32_t ww[4] = {w[rr][j].x, w[rr][j].y, w[rr][j].z, w[rr][j].w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                a2[j & 1] = fmaf(bf16_lo(ww[e]), hv[2 * e], a2[j & 1]);
                a2[j & 1] = fmaf(bf16_hi(ww[e]), hv[2 * e + 1], a2[j & 1]);
              }
            }
          }
          acc[rr][t] = a2[0] + a2[1];
        }
      }
    } else {
      uint4 qv[RD];
      uint16_t dv[RD];
      const bool act = lane < cols / 32;
#pragma unroll
      for (int rr = 0; rr < RD; ++rr) {
        if (rr >= u.n) break;
        if (act) {
          qv[rr] = *reinterpret_cast<const uint4*>(slot + (size_t)rr * rb + 16 * lane);
          dv[rr] = *reinterpret_cast<const uint16_t*>(slot + (size_t)rr * rb + cols / 2 + 2 * lane);
        }
      }
      release();
      if (TMAX == 1 && hg_cur != g) {
        hg_cur = g;
        if (act) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint4 v = *reinterpret_cast<const uint4*>(hg + h2_quarter_off(lane, k));
            hq[XREG && Q4 ? 4 * k : 0] = v.x;
            hq[XREG && Q4 ? 4 * k + 1 : 0] = v.y;
            hq[XREG && Q4 ? 4 * k + 2 : 0] = v.z;
            hq[XREG && Q4 ? 4 * k + 3 : 0] = v.w;
          }
        }
      }
      if (act) {
#pragma unroll
        for (int rr = 0; rr < RD; ++rr) {
          if (rr >= u.n) break;
          uint32_t q[16];
          dequant_block(qv[rr], q);
          const float d = __half2float(*reinterpret_cast<const __half*>(&dv[rr]));
#pragma unroll
          for (int t = 0; t < TMAX; ++t) {
            if (t >= ntok) continue;
            uint32_t hv[16];
            if (TMAX == 1) {
#pragma unroll
              for (int i = 0; i < 16; ++i) hv[i] = hq[XREG && Q4 ? i : 0];
            } else {
              const uint8_t* hb = hg + (size_t)t * cols * 2;
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const uint4 v = *reinterpret_cast<const uint4*>(hb + h2_quarter_off(lane, k));
                hv[4 * k] = v.x; hv[4 * k + 1] = v.y; hv[4 * k + 2] = v.z; hv[4 * k + 3] = v.w;
              }
            }
            uint32_t s0 = 0u, s1 = 0u;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              s0 = h2_fma(q[2 * i], hv[2 * i], s0);
              s1 = h2_fma(q[2 * i + 1], hv[2 * i + 1], s1);
            }
            acc[rr][t] = d * (h2_sum(s0) + h2_sum(s1));
          }
        }
      }
    }
    if (TMAX == 1) {
      const int ysrow = shared ? TK : tb.tsmap[(g - 1) * T];
#pragma unroll
      for (int rr = 0; rr < RD; ++rr) {
        if (rr >= u.n) break;
        pend_y.push(acc[rr][0], ysrow * P.v2_rows_w + (u.b + rr - c.da));
        if (pend_y.n == 8) pend_y.flush(tb.ys);
      }
      return;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
#pragma unroll
      for (int rr = 0; rr < RD; ++rr)
#pragma unroll
        for (int t = 0; t < TMAX; ++t)
          if (t < ntok && rr < u.n) acc[rr][t] += __shfl_xor_sync(0xffffffffu, acc[rr][t], o);
    }
    if (lane < ntok) {
      int ysrow;
      if (shared) {
        ysrow = TK + lane;
      } else {
        int cnt = 0, tsel = 0;
        for (int t = 0; t < T; ++t)
          if (m >> t & 1u) {
            if (cnt == lane) tsel = t;
            ++cnt;
          }
        ysrow = tb.tsmap[(g - 1) * T + tsel];
      }
#pragma unroll
      for (int rr = 0; rr < RD; ++rr) {
        if (rr >= u.n) break;
        float v = 0.f;
#pragma unroll
        for (int t = 0; t < TMAX; ++t)
          if (lane == t) v = acc[rr][t];
        tb.ys[(size_t)ysrow * P.v2_rows_w + (u.b + rr - c.da)] = v;
      }
    }
  };

  auto routing = [&]() {
    const int nct = nw * 32;
    pdl_wait();
    // the router's logits (all tokens) in one bulk copy
    if (tid == 0) {
      const uint32_t bytes = (uint32_t)T * P.ls * 4;
      mbar_arrive_expect_tx(aux_bar, bytes);
      bulk_g2s(lgs, P.logits, bytes, aux_bar, pol_keep);
    }
    for (int i = tid; i < (P.E + 31) / 32; i += nct) tb.counts[i] = 0;  // expert bitmap
    for (int i = tid; i < TK; i += nct) tb.mask[i] = 0u;
    if (!mbar_wait(aux_bar, 0)) atomicExch(reinterpret_cast<int*>(&P.ctrl[kCtrlStatus]), -6);
    // rank of every logit among its token's E logits (larger value first,
    // then lower index; NaN counts as -inf); ranks < K give the top-k in
    // order.  Threads split each comparison run in S parts.
    {
      const int pairs = T * P.E;
      int S = 1;
      while (S < 32 && pairs * S * 2 <= nct) S *= 2;
      for (int base = 0; base < pairs * S; base += nct) {
        const int q = base + tid;
        const int pi = q / S, sub = q % S;
        int rank = 0;
        int t = 0, i = 0;
        if (pi < pairs) {
          t = pi / P.E;
          i = pi % P.E;
          const float* lg = lgs + (size_t)t * P.ls;
          float li = lg[i];
          li = li != li ? -INFINITY : li;
          const int j0 = (P.E * sub) / S, j1 = (P.E * (sub + 1)) / S;
          for (int j = j0; j < j1; ++j) {
            float lj = lg[j];
            lj = lj != lj ? -INFINITY : lj;
            rank += (lj > li || (lj == li && j < i)) ? 1 : 0;
          }
        }
        for (int o = 1; o < S; o <<= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
        if (pi < pairs && sub == 0 && rank < K) tb.ids[t * K + rank] = i;
      }
    }
    named_bar_sync(kBarV2Cons, nct);
    // softmax of the chosen logits and the shared gate (warp t: token t);
    // all threads: the set of selected experts as a bitmap
    for (int t = warp; t < T; t += nw) {
      const float* lg = lgs + (size_t)t * P.ls;
      const float lj = lane < K ? lg[tb.ids[t * K + lane]] : 0.f;
      const float l0 = __shfl_sync(0xffffffffu, lj, 0);
      const float z = lane < K ? expf(lj - l0) : 0.f;
      const float sum = warp_sum(z);
      if (lane < K) tb.p[t * K + lane] = z / sum;
      if (lane == 0) tb.s[t] = 1.0f / (1.0f + expf(-lg[P.E]));
    }
    for (int ts = tid; ts < TK; ts += nct) {
      const int e = tb.ids[ts];
      atomicOr(reinterpret_cast<uint32_t*>(&tb.counts[e >> 5]), 1u << (e & 31));
    }
    named_bar_sync(kBarV2Cons, nct);
    // active index of an expert = selected experts below it (bitmap popcount)
    for (int ts = tid; ts < TK; ts += nct) {
      const int e = tb.ids[ts], t = ts / K;
      int u = __popc((uint32_t)tb.counts[e >> 5] & ((1u << (e & 31)) - 1u));
      for (int w = 0; w < (e >> 5); ++w) u += __popc((uint32_t)tb.counts[w]);
      tb.active[u] = e;
      tb.inv_u[e] = static_cast<int16_t>(u);
      atomicOr(&tb.mask[u], 1u << t);
      tb.tsmap[u * T + t] = static_cast<int16_t>(ts);
    }
    if (tid == 0) {
      int U = 0;
      for (int w = 0; w < (P.E + 31) / 32; ++w) U += __popc((uint32_t)tb.counts[w]);
      tb.misc[0] = U;
    }
    named_bar_sync(kBarV2Cons, nct);
    const int U = tb.misc[0];
    if (warp == 0) {
      // tokens of the active experts before u, and where each group's h goes
      int run = 0;
      for (int u0 = 0; u0 < U; u0 += 32) {
        const int u = u0 + lane;
        const int n = u < U ? __popc(tb.mask[u]) : 0;
        int incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += v;
        }
        if (u < U) {
          tb.pre[u] = run + incl - n;
          tb.goff[u + 1] = T * P.Is + (run + incl - n) * P.I;
        }
        run += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) {
        tb.goff[0] = 0;
        tb.goff[U + 1] = T * P.Is + TK * P.I;
      }
      for (int t = lane; t < T; t += 32) {
        tb.hsrc[t] = -(1 + t);
        tb.hdst[t] = t * P.Is;
      }
      __syncwarp();
      for (int ts = lane; ts < TK; ts += 32) {
        const int t = ts / K;
        const int u = tb.inv_u[tb.ids[ts]];
        const int rank = __popc(tb.mask[u] & ((1u << t) - 1u));
        const int rowi = T + tb.pre[u] + rank;
        tb.hsrc[rowi] = ts;
        tb.hdst[rowi] = tb.goff[u + 1] + rank * P.I;
      }
    }
    named_bar_sync(kBarV2Cons, nct);
    if (cta == 0 && warp == nw - 1) {
      // routing outputs for the caller and the test readers: counts, offsets
      // (a scan over the experts) and the stable token-major permutation
      int base = 0;
      for (int e0 = 0; e0 < P.E; e0 += 32) {
        const int e = e0 + lane;
        int cnt = 0;
        if (e < P.E && tb.inv_u[e] >= 0 && (uint32_t)tb.counts[e >> 5] >> (e & 31) & 1u)
          cnt = __popc(tb.mask[tb.inv_u[e]]);
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
        const int u = tb.inv_u[e];
        P.r_perm[P.r_offsets[e] + __popc(tb.mask[u] & ((1u << t) - 1u))] = ts;
      }
      for (int u = lane; u < U; u += 32) P.r_active[u] = tb.active[u];
    }
    c.U = U;
    const long long tot = (long long)c.U * P.I;
    const long long a = tot * cta / P.G, b = tot * (cta + 1) / P.G;
    c.fa = a + (b - a) * warp / nw;
    c.fb = a + (b - a) * (warp + 1) / nw;
    c.fa_u = (int)(c.fa / P.I);
    c.fa_i = (int)(c.fa % P.I);
    const int W = (c.U + 1) * c.nD;
    c.dfa = (int)((long long)W * warp / nw);
    c.dfb = (int)((long long)W * (warp + 1) / nw);
    c.dfa_g = c.nD > 0 ? c.dfa / c.nD : 0;
    c.dfa_r = c.nD > 0 ? c.dfa % c.nD : 0;
    c.routed = true;
    const int n_s = n_units;
    int cnt = 0;
    if (lane == 0) cnt = v2_build_rd(P, tb, c, L, n_s);
    n_units = __shfl_sync(0xffffffffu, cnt, 0);
    __syncwarp();
    // gate/up units = shared + routed ones (the down units follow)
    n_gu = n_s;
    for (int k = n_s; k < n_units; ++k)
      if ((L[k].info & 3) == 1) ++n_gu;
  };

  auto h_sync = [&]() {
    if (TMAX == 1) pend_h.flush(hmode);
    // every thread's h stores, then one release for the CTA; thread 0 then
    // waits (bounded) until every CTA of the grid has released
    __threadfence();
    named_bar_sync(kBarV2Cons, nw * 32);
    if (tid == 0) {
      red_release_gpu_add(&P.ctrl[kCtrlHDone], 1u);
      if (nD > 0) {
        bool ok = false;
        for (uint32_t i = 0; i < kSpinLimit; ++i) {
          if (ld_acquire_gpu(&P.ctrl[kCtrlHDone]) >= (uint32_t)P.G) {
            ok = true;
            break;
          }
          __nanosleep(32);
        }
        if (!ok) atomicExch(reinterpret_cast<int*>(&P.ctrl[kCtrlStatus]), -6);
      }
    }
    named_bar_sync(kBarV2Cons, nw * 32);
    if (nD > 0) {
      // every down group's h rows (already in the staged format), one batch of
      // bulk copies on one barrier
      if (tid == 0) {
        fence_proxy_async();
        const int nrows = T + TK;
        uint32_t total = 0;
        for (int rowi = 0; rowi < nrows; ++rowi) total += (tb.hsrc[rowi] < 0 ? P.Is : P.I) * hel;
        mbar_arrive_expect_tx(hst_bar, total);
        for (int rowi = 0; rowi < nrows; ++rowi) {
          const int src = tb.hsrc[rowi];
          const bool shared = src < 0;
          const int cols = shared ? P.Is : P.I;
          const uint8_t* sp = shared ? reinterpret_cast<const uint8_t*>(P.hsh) + (size_t)(-src - 1) * P.Is * hel
                                     : reinterpret_cast<const uint8_t*>(P.h) + (size_t)src * P.I * hel;
          bulk_g2s(uni + (size_t)tb.hdst[rowi] * hel, sp, (uint32_t)(cols * hel), hst_bar, pol_keep);
        }
      }
      if (!mbar_wait(hst_bar, 0)) atomicExch(reinterpret_cast<int*>(&P.ctrl[kCtrlStatus]), -6);
    }
  };

  // route first: the shared-expert copies issued above land meanwhile
  routing();
  if (lane == 0) pump();

  // gate/up units (S then R)
  while (k_con < n_gu) {
    const V2U d = L[k_con];
    const int kind = d.info & 3, n = (d.info >> 2) & 255;
    const V2Unit u{kind, kind == 0 ? d.row0 : (d.info >> 10), d.row0, n};
    const int sl = k_con % nslots;
    if (!mbar_wait(&my_bar[sl], (uint32_t)(k_con / nslots) & 1u))
      atomicExch(reinterpret_cast<int*>(&P.ctrl[kCtrlStatus]), -6);
    do_gu(u, my_ring + (size_t)sl * P.v2_slot);  // releases the slot itself
  }
  // publish h and wait for every CTA's (down rows keep streaming into the ring)
  h_sync();
  // down units
  while (k_con < n_units) {
    const V2U d = L[k_con];
    const V2Unit u{2, d.info >> 10, d.row0, (d.info >> 2) & 255};
    const int sl = k_con % nslots;
    if (!mbar_wait(&my_bar[sl], (uint32_t)(k_con / nslots) & 1u))
      atomicExch(reinterpret_cast<int*>(&P.ctrl[kCtrlStatus]), -6);
    do_down(u, my_ring + (size_t)sl * P.v2_slot);  // releases the slot itself
  }
  if (TMAX == 1) pend_y.flush(tb.ys);

  // ---- combine this CTA's rows: out = sum_j p_j y_j + s y_sh (+ residual)
  named_bar_sync(kBarV2Cons, nw * 32);
  for (int i = tid; i < T * nD; i += nw * 32) {
    const int t = i / nD, r = i % nD;
    float o = 0.f;
    for (int j = 0; j < K; ++j) o = fmaf(tb.p[t * K + j], tb.ys[(size_t)(t * K + j) * P.v2_rows_w + r], o);
    o = fmaf(tb.s[t], tb.ys[(size_t)(TK + t) * P.v2_rows_w + r], o);
    float* dst = P.out + (size_t)t * P.H + da + r;
    if (P.block_mode)
      *dst = __fadd_rn(*dst, o);
    else
      *dst = o;
  }
}

template <int TMAX, bool Q4, bool XREG>
inline cudaError_t launch_v2_t(const DecodeParams& p, cudaStream_t stream) {
  cudaError_t err =
      cudaFuncSetAttribute(k_experts_v2<TMAX, Q4, XREG>, cudaFuncAttributeMaxDynamicSharedMemorySize, p.v2_smem);
  if (err != cudaSuccess) return err;
  err = launch_route(p, stream, true);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(p.G);
  cfg.blockDim = dim3(p.v2_nw * 32);
  cfg.dynamicSmemBytes = p.v2_smem;
  return cudaLaunchKernelEx(&cfg, k_experts_v2<TMAX, Q4, XREG>, p);
}


}  // namespace moe
