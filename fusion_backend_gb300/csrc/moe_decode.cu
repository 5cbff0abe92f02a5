// Decode path of the fused MoE FFN layer (T <= 8 tokens), sm_103a.
//
// Two kernels per call, chained with programmatic dependent launch:
//
//  k_route   one CTA per router row (E rows + the shared-gate vector):
//            logit[t,e] = sum_h W[e,h] x[t,h] with an error-free (TwoSum /
//            TwoProduct) accumulation, so the fp32 logit is the correctly
//            rounded exact dot product and the top-k decision does not depend
//            on the summation order.  Also zeroes the control words of the
//            expert kernel.
//
//  k_experts one persistent CTA per SM.  Weight bytes are streamed once
//            through a ring of shared-memory stages filled by the bulk-copy
//            (TMA) engine from one producer warp; eight consumer warps do the
//            arithmetic.  Phases per CTA:
//              S  its slice of the shared expert's gate/up rows
//                 (routing-independent, overlaps k_route: the in-kernel form
//                 of the shared-expert / routed-expert overlap)
//              -  wait for k_route, top-k + softmax + bucketing (redundantly
//                 in every CTA, so no second grid-wide exchange is needed)
//              R  its slice of the routed experts' gate/up rows:
//                 h = silu(gate x) * (up x) -> workspace
//              D  after every CTA has published its h (bounded spin on a
//                 counter), its block of output rows of every selected
//                 expert's down matrix and of the shared down matrix, then
//                 the fixed-order combine out = sum_j p_j y_j + s y_sh.
//            The down weights are prefetched into the ring while the counter
//            wait runs; h rows come in through a second small ring.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "moe_decode_common.cuh"

namespace moe {

namespace {
constexpr int kBarCons = 1;   // named barrier: the 256 consumer threads
constexpr int kBarRoute = 2;  // named barrier: all threads of the CTA
constexpr int kConsThreads = kNumConsumerWarps * 32;
constexpr int kMaxBarriers = 64;

struct Tabs {
  int32_t ids[kDecodeMaxT * kMaxTopK];
  float p[kDecodeMaxT * kMaxTopK];
  float s[kDecodeMaxT];
  float inv[kDecodeMaxT][2];
  int32_t counts[kMaxExperts];
  int32_t offsets[kMaxExperts + 1];
  int16_t inv_u[kMaxExperts];
  int32_t active[kDecodeMaxT * kMaxTopK];
  uint32_t mask[kDecodeMaxT * kMaxTopK];
  int16_t tsmap[kDecodeMaxT * kMaxTopK][kDecodeMaxT];
  int U;
  int abort;
};

struct Item {
  int kind;  // 0 shared gate/up, 1 routed gate/up, 2 shared down, 3 routed down
  int u;     // active-expert index (kinds 1, 3)
  int row0;  // first row
  int n;     // rows (row pairs for gate/up)
  int group; // down: 0 = shared, 1 + u = routed
  bool first, last;  // first / last item of its down group
};


MOE_DEV int cap_gu(const DecodeParams& P) { return min(kMaxGuRows, kStageBytes / (2 * P.rbH)); }
MOE_DEV int cap_dn(int rb) { return min(kMaxDownRows, kStageBytes / rb); }

template <class F>
MOE_DEV void walk_shared_gu(const DecodeParams& P, int c, F&& f) {
  const int a = div_floor_ll((long long)P.Is * c, P.G), b = div_floor_ll((long long)P.Is * (c + 1), P.G);
  const int cap = cap_gu(P);
  for (int i = a; i < b; i += cap) f(Item{0, -1, i, min(cap, b - i), -1, false, false});
}

template <class F>
MOE_DEV void walk_routed_gu(const DecodeParams& P, int c, int U, F&& f) {
  const long long tot = (long long)U * P.I;
  const long long a = tot * c / P.G, b = tot * (c + 1) / P.G;
  const int cap = cap_gu(P);
  for (long long fp = a; fp < b;) {
    const int u = static_cast<int>(fp / P.I), i = static_cast<int>(fp % P.I);
    const int n = static_cast<int>(min((long long)min(cap, P.I - i), b - fp));
    f(Item{1, u, i, n, -1, false, false});
    fp += n;
  }
}


template <class F>
MOE_DEV void walk_down(const DecodeParams& P, int c, int U, F&& f) {
  int a, b;
  down_rows(P, c, a, b);
  if (a >= b) return;
  const int cs = cap_dn(P.rbIs), cr = cap_dn(P.rbI);
  for (int r = a; r < b; r += cs) f(Item{2, -1, r, min(cs, b - r), 0, r == a, r + cs >= b});
  for (int u = 0; u < U; ++u)
    for (int r = a; r < b; r += cr) f(Item{3, u, r, min(cr, b - r), 1 + u, r == a, r + cr >= b});
}

}  // namespace

// ============================================================ expert kernel
namespace {
struct Smem {
  uint8_t* stage;
  uint8_t* hslot;
  float* red;
  float* ys;
  float* logits;
  unsigned long long* cand;
  uint64_t* bar;  // full[nst], empty[nst], hfull[nhs], hempty[nhs]
  Tabs* tb;
};

MOE_DEV Smem smem_views(const DecodeParams& P, uint8_t* base) {
  Smem s;
  s.stage = base + P.off_stage;
  s.hslot = base + P.off_hslot;
  s.red = reinterpret_cast<float*>(base + P.off_red);
  s.ys = reinterpret_cast<float*>(base + P.off_ys);
  s.logits = reinterpret_cast<float*>(base + P.off_logits);
  s.cand = reinterpret_cast<unsigned long long*>(base + P.off_logits + ((size_t)P.T * (P.E + 1) * 4 + 15) / 16 * 16);
  s.bar = reinterpret_cast<uint64_t*>(base + P.off_bar);
  s.tb = reinterpret_cast<Tabs*>(base + P.off_tab);
  return s;
}

}  // namespace

template <int TMAX>
__global__ void __launch_bounds__(kDecodeThreads, 1) k_experts(DecodeParams P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Smem S = smem_views(P, smem_raw);
  Tabs& tb = *S.tb;
  uint64_t* full = S.bar;
  uint64_t* empty = S.bar + P.nst;
  uint64_t* hfull = S.bar + 2 * P.nst;
  uint64_t* hempty = S.bar + 2 * P.nst + P.nhs;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cta = blockIdx.x;
  const int T = P.T, K = P.K;

  if (tid == 0) {
    for (int i = 0; i < P.nst; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kNumConsumerWarps);
    }
    for (int i = 0; i < P.nhs; ++i) {
      mbar_init(&hfull[i], 1);
      mbar_init(&hempty[i], kNumConsumerWarps);
    }
    tb.abort = 0;
    mbar_fence_init();
  }
  if (P.block_mode && warp < T) {
    float hi, lo;
    warp_norm_factor(static_cast<const float*>(P.x) + (size_t)warp * P.H, P.H, P.eps, hi, lo);
    if (lane == 0) {
      tb.inv[warp][0] = hi;
      tb.inv[warp][1] = lo;
    }
  }
  __syncthreads();

  if (warp == kNumConsumerWarps) {
    // ------------------------------------------------ weight producer warp
    const uint64_t pol = policy_evict_first();
    int it = 0;
    auto issue = [&](const Item& item) {
      const int st = it % P.nst, use = it / P.nst;
      if (use > 0 && !mbar_wait(&empty[st], (use - 1) & 1)) {
        atomicExch(reinterpret_cast<int*>(&P.ctrl[kCtrlStatus]), -6);
      }
      uint8_t* dst = S.stage + (size_t)st * kStageBytes;
      if (item.kind == 0 || item.kind == 1) {
        const uint8_t* base;
        long long mat;
        if (item.kind == 0) {
          base = P.shexp_w;
          mat = P.sgu_bytes;
        } else {
          base = P.expert_w + (size_t)tb.active[item.u] * P.expert_bytes;
          mat = P.gu_bytes;
        }
        const uint32_t bytes = (uint32_t)item.n * P.rbH;
        mbar_arrive_expect_tx(&full[st], 2 * bytes);
        bulk_g2s(dst, base + (size_t)item.row0 * P.rbH, bytes, &full[st], pol);
        bulk_g2s(dst + bytes, base + mat + (size_t)item.row0 * P.rbH, bytes, &full[st], pol);
      } else {
        const uint8_t* src;
        int rb;
        if (item.kind == 2) {
          rb = P.rbIs;
          src = P.shexp_w + 2 * P.sgu_bytes + (size_t)item.row0 * rb;
        } else {
          rb = P.rbI;
          src = P.expert_w + (size_t)tb.active[item.u] * P.expert_bytes + 2 * P.gu_bytes + (size_t)item.row0 * rb;
        }
        const uint32_t bytes = (uint32_t)item.n * rb;
        mbar_arrive_expect_tx(&full[st], bytes);
        bulk_g2s(dst, src, bytes, &full[st], pol);
      }
      ++it;
    };
    if (lane == 0) walk_shared_gu(P, cta, issue);
    __syncwarp();
    pdl_wait();
    named_bar_sync(kBarRoute, kDecodeThreads);
    if (lane == 0) {
      const int U = tb.U;
      walk_routed_gu(P, cta, U, issue);
      walk_down(P, cta, U, issue);
    }
    return;
  }

  if (warp == kNumConsumerWarps + 1) {
    // ------------------------------------------------ h producer warp
    pdl_wait();
    named_bar_sync(kBarRoute, kDecodeThreads);
    if (lane == 0) {
      int a, b;
      down_rows(P, cta, a, b);
      if (a < b) {
        bool ok = false;
        for (uint32_t i = 0; i < kSpinLimit; ++i) {
          if (ld_acquire_gpu(&P.ctrl[kCtrlHDone]) >= (uint32_t)P.G) {
            ok = true;
            break;
          }
          __nanosleep(64);
        }
        if (!ok) atomicExch(reinterpret_cast<int*>(&P.ctrl[kCtrlStatus]), -6);
        fence_proxy_async_global();
        const uint64_t pol = policy_evict_last();
        const int U = tb.U;
        for (int g = 0; g <= U; ++g) {
          const int sl = g % P.nhs, use = g / P.nhs;
          if (use > 0 && !mbar_wait(&hempty[sl], (use - 1) & 1))
            atomicExch(reinterpret_cast<int*>(&P.ctrl[kCtrlStatus]), -6);
          uint8_t* dst = S.hslot + (size_t)sl * P.hslot_bytes;
          if (g == 0) {
            const uint32_t bytes = (uint32_t)T * P.Is * 4;
            mbar_arrive_expect_tx(&hfull[sl], bytes);
            bulk_g2s(dst, P.hsh, bytes, &hfull[sl], pol);
          } else {
            const int u = g - 1;
            const uint32_t m = tb.mask[u];
            const uint32_t rowb = (uint32_t)P.I * 4;
            mbar_arrive_expect_tx(&hfull[sl], rowb * __popc(m));
            int j = 0;
            for (int t = 0; t < T; ++t)
              if (m >> t & 1u) {
                bulk_g2s(dst + (size_t)j * rowb, P.h + (size_t)tb.tsmap[u][t] * P.I, rowb, &hfull[sl], pol);
                ++j;
              }
          }
        }
      }
    }
    return;
  }

  // ==================================================== consumer warps
  const int ctid = tid;  // 0 .. 255
  const uint32_t all_tokens = (T >= 32) ? 0xFFFFFFFFu : ((1u << T) - 1u);
  float xs[TMAX][8];
  int xseg = -1;
  int it = 0;
  int da, db;
  down_rows(P, cta, da, db);
  const int nrowsD = db - da;
  const int nsegH = (P.H + kSegCols - 1) / kSegCols;

  // Gate/up item: h = silu(gate x) * (up x) for the item's rows.
  auto consume_gu = [&](const Item& item) {
    const int st = it % P.nst, use = it / P.nst;
    float* red = S.red + (size_t)(it & 1) * P.red_floats;
    if (!mbar_wait(&full[st], use & 1)) {
      atomicExch(reinterpret_cast<int*>(&P.ctrl[kCtrlStatus]), -6);
    }
    const uint32_t m = item.kind == 0 ? all_tokens : tb.mask[item.u];
    const uint8_t* sg = S.stage + (size_t)st * kStageBytes;
    const uint8_t* su = sg + (size_t)item.n * P.rbH;
    const int nunits = item.n * nsegH;
    for (int q = warp; q < nunits; q += kNumConsumerWarps) {
      const int r = q / nsegH, sgi = q % nsegH;
      const int c0 = sgi * kSegCols + lane * 8;
      const bool valid = c0 < P.H;
      if (sgi != xseg) {
        xseg = sgi;
#pragma unroll
        for (int t = 0; t < TMAX; ++t)
          if (t < T && valid) load_x8_any(P, &tb.inv[0][0], t, c0, xs[t]);
      }
      float ag[TMAX], au[TMAX];
#pragma unroll
      for (int t = 0; t < TMAX; ++t) ag[t] = au[t] = 0.f;
      if (valid) {
        float wg[8], wu[8];
        load_w8(sg + (size_t)r * P.rbH, P.H, P.wfmt, c0, wg);
        load_w8(su + (size_t)r * P.rbH, P.H, P.wfmt, c0, wu);
#pragma unroll
        for (int t = 0; t < TMAX; ++t) {
          if (m >> t & 1u) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              ag[t] = fmaf(wg[j], xs[t][j], ag[t]);
              au[t] = fmaf(wu[j], xs[t][j], au[t]);
            }
          }
        }
      }
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
        if (m >> t & 1u) {
          const float g = warp_sum(ag[t]);
          const float u = warp_sum(au[t]);
          if (lane == 0) {
            red[((size_t)q * TMAX + t) * 2] = g;
            red[((size_t)q * TMAX + t) * 2 + 1] = u;
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
    named_bar_sync(kBarCons, kConsThreads);
    for (int pidx = ctid; pidx < item.n * TMAX; pidx += kConsThreads) {
      const int r = pidx / TMAX, t = pidx % TMAX;
      if (!(m >> t & 1u)) continue;
      float g = 0.f, u = 0.f;
      for (int sgi = 0; sgi < nsegH; ++sgi) {
        g += red[(((size_t)r * nsegH + sgi) * TMAX + t) * 2];
        u += red[(((size_t)r * nsegH + sgi) * TMAX + t) * 2 + 1];
      }
      const float hv = g / (1.0f + expf(-g)) * u;
      if (item.kind == 0)
        P.hsh[(size_t)t * P.Is + item.row0 + r] = hv;
      else
        P.h[(size_t)tb.tsmap[item.u][t] * P.I + item.row0 + r] = hv;
    }
    ++it;
  };

  auto consume_down = [&](const Item& item) {
    const int st = it % P.nst, use = it / P.nst;
    float* red = S.red + (size_t)(it & 1) * P.red_floats;
    const int sl = item.group % P.nhs, huse = item.group / P.nhs;
    if (item.first) {
      if (!mbar_wait(&hfull[sl], huse & 1)) atomicExch(reinterpret_cast<int*>(&P.ctrl[kCtrlStatus]), -6);
    }
    if (!mbar_wait(&full[st], use & 1)) atomicExch(reinterpret_cast<int*>(&P.ctrl[kCtrlStatus]), -6);
    const bool shared = item.kind == 2;
    const int cols = shared ? P.Is : P.I;
    const int rb = shared ? P.rbIs : P.rbI;
    const uint32_t m = shared ? all_tokens : tb.mask[item.u];
    const int ntok = __popc(m);
    const int nseg = (cols + kSegCols - 1) / kSegCols;
    const uint8_t* sw = S.stage + (size_t)st * kStageBytes;
    const float* hs = reinterpret_cast<const float*>(S.hslot + (size_t)sl * P.hslot_bytes);
    const int nunits = item.n * nseg;
    for (int q = warp; q < nunits; q += kNumConsumerWarps) {
      const int r = q / nseg, sgi = q % nseg;
      const int c0 = sgi * kSegCols + lane * 8;
      float acc[TMAX];
#pragma unroll
      for (int j = 0; j < TMAX; ++j) acc[j] = 0.f;
      if (c0 < cols) {
        float w[8];
        load_w8(sw + (size_t)r * rb, cols, P.wfmt, c0, w);
#pragma unroll
        for (int j = 0; j < TMAX; ++j) {
          if (j < ntok) {
            const float4* hp = reinterpret_cast<const float4*>(hs + (size_t)j * cols + c0);
            const float4 a = hp[0], b = hp[1];
            acc[j] = fmaf(w[0], a.x, acc[j]); acc[j] = fmaf(w[1], a.y, acc[j]);
            acc[j] = fmaf(w[2], a.z, acc[j]); acc[j] = fmaf(w[3], a.w, acc[j]);
            acc[j] = fmaf(w[4], b.x, acc[j]); acc[j] = fmaf(w[5], b.y, acc[j]);
            acc[j] = fmaf(w[6], b.z, acc[j]); acc[j] = fmaf(w[7], b.w, acc[j]);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < TMAX; ++j) {
        if (j < ntok) {
          const float v = warp_sum(acc[j]);
          if (lane == 0) red[(size_t)q * TMAX + j] = v;
        }
      }
    }
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&empty[st]);
      if (item.last) mbar_arrive(&hempty[sl]);
    }
    named_bar_sync(kBarCons, kConsThreads);
    for (int pidx = ctid; pidx < item.n * TMAX; pidx += kConsThreads) {
      const int r = pidx / TMAX, j = pidx % TMAX;
      if (j >= ntok) continue;
      float y = 0.f;
      for (int sgi = 0; sgi < nseg; ++sgi) y += red[((size_t)r * nseg + sgi) * TMAX + j];
      int ysrow;
      if (shared) {
        ysrow = T * K + j;
      } else {
        int cnt = 0, tsel = 0;
        for (int t = 0; t < T; ++t)
          if (m >> t & 1u) {
            if (cnt == j) tsel = t;
            ++cnt;
          }
        ysrow = tb.tsmap[item.u][tsel];
      }
      S.ys[(size_t)ysrow * P.ys_rows_max + (item.row0 + r - da)] = y;
    }
    ++it;
  };

  // ---- phase S: shared expert gate/up (does not need the routing)
  walk_shared_gu(P, cta, consume_gu);

  // ---- routing: wait for the router kernel, then top-k and bucketing
  pdl_wait();
  for (int t = warp; t < T; t += kNumConsumerWarps) {
    float* lg = S.logits + (size_t)t * (P.E + 1);
    for (int e = lane; e <= P.E; e += 32) lg[e] = P.logits[(size_t)t * P.ls + e];
    __syncwarp();
    warp_topk(lg, P.E, K, &tb.ids[t * K], &tb.p[t * K]);
    if (lane == 0) tb.s[t] = 1.0f / (1.0f + expf(-lg[P.E]));
  }
  for (int e = ctid; e < P.E; e += kConsThreads) {
    tb.counts[e] = 0;
    tb.inv_u[e] = -1;
  }
  for (int u = ctid; u < T * K; u += kConsThreads) tb.mask[u] = 0u;
  named_bar_sync(kBarCons, kConsThreads);
  for (int ts = ctid; ts < T * K; ts += kConsThreads) atomicAdd(&tb.counts[tb.ids[ts]], 1);
  named_bar_sync(kBarCons, kConsThreads);
  if (warp == 0) {
    int base = 0, nact = 0;
    for (int e0 = 0; e0 < P.E; e0 += 32) {
      const int e = e0 + lane;
      const int cnt = e < P.E ? tb.counts[e] : 0;
      // inclusive scan of counts across the warp
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (e < P.E) tb.offsets[e] = base + incl - cnt;
      const unsigned bb = __ballot_sync(0xffffffffu, cnt > 0);
      if (cnt > 0) {
        const int pos = nact + __popc(bb & ((1u << lane) - 1u));
        tb.active[pos] = e;
        tb.inv_u[e] = static_cast<int16_t>(pos);
      }
      nact += __popc(bb);
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      tb.offsets[P.E] = base;
      tb.U = nact;
    }
  }
  named_bar_sync(kBarCons, kConsThreads);
  for (int ts = ctid; ts < T * K; ts += kConsThreads) {
    const int t = ts / K;
    const int u = tb.inv_u[tb.ids[ts]];
    atomicOr(&tb.mask[u], 1u << t);
    tb.tsmap[u][t] = static_cast<int16_t>(ts);
  }
  named_bar_sync(kBarRoute, kDecodeThreads);
  const int U = tb.U;

  if (cta == 0) {
    for (int ts = ctid; ts < T * K; ts += kConsThreads) {
      if (P.topk_ids) P.topk_ids[ts] = tb.ids[ts];
      if (P.topk_w) P.topk_w[ts] = tb.p[ts];
      const int t = ts / K, e = tb.ids[ts];
      const int u = tb.inv_u[e];
      const int pos = tb.offsets[e] + __popc(tb.mask[u] & ((1u << t) - 1u));
      P.r_perm[pos] = ts;
    }
    for (int e = ctid; e < P.E; e += kConsThreads) {
      P.r_counts[e] = tb.counts[e];
      P.r_offsets[e] = tb.offsets[e];
    }
    for (int u = ctid; u < U; u += kConsThreads) P.r_active[u] = tb.active[u];
    if (ctid == 0) {
      P.r_offsets[P.E] = tb.offsets[P.E];
      *P.r_nactive = U;
    }
  }

  // ---- phase R: routed gate/up
  walk_routed_gu(P, cta, U, consume_gu);
  __threadfence();
  named_bar_sync(kBarCons, kConsThreads);
  if (ctid == 0) red_release_gpu_add(&P.ctrl[kCtrlHDone], 1u);

  // ---- phase D: down rows of every selected expert and of the shared expert
  walk_down(P, cta, U, consume_down);
  if (nrowsD <= 0) return;
  named_bar_sync(kBarCons, kConsThreads);
  for (int pidx = ctid; pidx < T * nrowsD; pidx += kConsThreads) {
    const int t = pidx / nrowsD, rr = pidx % nrowsD;
    float o = 0.f;
    for (int j = 0; j < K; ++j) o = fmaf(tb.p[t * K + j], S.ys[(size_t)(t * K + j) * P.ys_rows_max + rr], o);
    o = fmaf(tb.s[t], S.ys[(size_t)(T * K + t) * P.ys_rows_max + rr], o);
    float* dst = P.out + (size_t)t * P.H + da + rr;
    if (P.block_mode)
      *dst = __fadd_rn(*dst, o);
    else
      *dst = o;
  }
}

// ============================================================ host side

int decode_kernel_count() { return 2; }


int decode_smem_layout(DecodeParams& p, int smem_limit) {
  const int TM = tmax_for(p.T);
  const int nsegH = (p.H + kSegCols - 1) / kSegCols;
  const int nsegI = (p.I + kSegCols - 1) / kSegCols;
  const int nsegIs = (p.Is + kSegCols - 1) / kSegCols;
  const int capgu = std::min(kMaxGuRows, kStageBytes / (2 * p.rbH));
  const int capdi = std::min(kMaxDownRows, kStageBytes / p.rbI);
  const int capds = std::min(kMaxDownRows, kStageBytes / p.rbIs);
  if (capgu < 1 || capdi < 1 || capds < 1) return -1;
  p.red_floats = std::max(capgu * nsegH * TM * 2, std::max(capdi * nsegI * TM, capds * nsegIs * TM));
  p.ys_rows_max = (p.H + p.G - 1) / p.G;
  p.hslot_bytes = align_up(p.T * std::max(p.I, p.Is) * 4, 128);
  p.nhs = 2;
  int off = 0;
  p.off_bar = off;
  off += kMaxBarriers * 8;
  off = align_up(off, 128);
  p.off_tab = off;
  off += align_up((int)sizeof(Tabs), 128);
  p.off_logits = off;
  off += align_up(p.T * (p.E + 1) * 4, 16) + p.T * p.E * 8;
  off = align_up(off, 128);
  p.off_red = off;
  off += 2 * p.red_floats * 4;
  off = align_up(off, 128);
  p.off_ys = off;
  off += (p.T * p.K + p.T) * p.ys_rows_max * 4;
  off = align_up(off, 128);
  p.off_hslot = off;
  off += p.nhs * p.hslot_bytes;
  off = align_up(off, 1024);
  p.off_stage = off;
  const int room = smem_limit - off;
  int nst = room / kStageBytes;
  if (nst > 8) nst = 8;
  if (nst < 2) return -1;
  if (2 * nst + 2 * p.nhs > kMaxBarriers) return -1;
  p.nst = nst;
  p.smem_bytes = off + nst * kStageBytes;
  return p.smem_bytes;
}

template <int TMAX>
static cudaError_t launch_t(const DecodeParams& p, cudaStream_t stream, bool use_pdl) {
  static_assert(TMAX <= kDecodeMaxT, "TMAX");
  cudaError_t err = cudaFuncSetAttribute(k_experts<TMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize, p.smem_bytes);
  if (err != cudaSuccess) return err;
  err = launch_route(p, stream, false);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.stream = stream;
  cfg.gridDim = dim3(p.G);
  cfg.blockDim = dim3(kDecodeThreads);
  cfg.dynamicSmemBytes = p.smem_bytes;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = use_pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_experts<TMAX>, p);
}

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream, bool use_pdl) {
  switch (tmax_for(p.T)) {
    case 1: return launch_t<1>(p, stream, use_pdl);
    case 2: return launch_t<2>(p, stream, use_pdl);
    case 4: return launch_t<4>(p, stream, use_pdl);
    default: return launch_t<8>(p, stream, use_pdl);
  }
}

}  // namespace moe
