// Grouped GEMMs of the batched MoE FFN layer for 4-bit weights (blocks of 32
// along each stored row, one fp16 scale d per block, weight d (code - 8)),
// on the tcgen05 tensor cores, sm_103a.  Same groups, units and epilogues as
// the bf16 kernels (moe_gemm.cu); the weights reach the tensor cores through
// eight dequantising warps, and the MMAs are kind::f16 with fp16 A and B (x
// and h are carried in fp16 on this path).
//
// Each weight is fp16(d (code - 8)), rounded once: (0x6400 | code) is the
// fp16 of 1024 + code, minus 1032 is code - 8 exactly, times d rounds once.
// Eight codes of a 32-bit word give four half2 (e0,e4) (e1,e5) (e2,e6)
// (e3,e7): in every group of eight the operands are stored in the order
// e0 e4 e1 e5 e2 e6 e3 e7.  gate / up take that order along K, so x_perm
// holds x in the same order (k_bucket_b).
//
// gate / up (PHASE 0): a raw stage is 64 gate + 64 up rows x 256 K of codes
// and scales (one TMA transaction); the slots' B rows come in a ring of their
// own.  The dequant warps write A straight into tensor memory (tcgen05.st,
// one row per lane), and the MMA reads A from there (the [a] operand form)
// and B from shared memory.
// down (PHASE 1): the raw stage is 64 downT rows (K) x 256 columns (M); the
// codes run along M, so each dequant thread transposes an 8 x 8 block of
// codes in registers and writes K-major fp16 tiles (128-byte swizzle) to
// shared memory (an MN-major A operand costs the tensor core about twice
// the time per MMA); within each group of 8 the K order is rotated by the
// group index and interleaved as above, and the gate / up epilogue writes h
// in that order.
//
// Block roles (15 warps): warp 0 lane 0 streams the raw and B stages; lane 0
// of warps 1 and 14 issue the MMAs, each into its own accumulator (gate / up:
// the two 128-K halves of every raw stage; down: alternate raw stages), and
// the epilogue adds the two in a fixed order (one thread issues a
// tcgen05.mma every ~85 cycles and spends ~500 more per stage on waits and
// commits; two overlap); warp 1 also owns the tensor memory; warps 2..9
// dequantise in two groups that take alternate raw stages; warps 10..13 are
// the epilogue, on two accumulator buffers.  A warp reaches tensor-memory
// lanes 32 (w % 4) .. + 31.  Every wait is bounded; on a timeout the roles
// leave their loops and the status word records it.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "moe_tc.cuh"

namespace moe {

namespace {

using namespace tc;

struct UnitQ {
  int shared, e, slot0, n, tile;
};

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// D (tensor memory) += A (tensor memory, 128 lanes x 8 columns of fp16
// pairs) x B (shared-memory descriptor)
__device__ __forceinline__ void umma_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 lanes x 16 columns of 32 bits into this warp's lane quarter
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Eight codes (element j in bits 4j..4j+3 of w) with the block scale pair dd
// -> four half2 (e0,e4) (e1,e5) (e2,e6) (e3,e7) of fp16(d (code - 8)).
__device__ __forceinline__ void dequant8(uint32_t w, __half2 dd, uint32_t* o) {
  const __half2 k1032 = __half2half2(__ushort_as_half((unsigned short)0x6408u));  // 1032.0
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t q = ((w >> (4 * i)) & 0x000F000Fu) | 0x64006400u;  // 1024 + code, two at a time
    const __half2 c = __hsub2(*reinterpret_cast<const __half2*>(&q), k1032);  // code - 8, exact
    const __half2 r = __hmul2(c, dd);
    o[i] = *reinterpret_cast<const uint32_t*>(&r);
  }
}

// Same with one scale pair per half2: o[q] = (code q, code q + 4) times dd[q].
__device__ __forceinline__ void dequant8s(uint32_t w, const __half2* dd, uint32_t* o) {
  const __half2 k1032 = __half2half2(__ushort_as_half((unsigned short)0x6408u));  // 1032.0
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t q = ((w >> (4 * i)) & 0x000F000Fu) | 0x64006400u;
    const __half2 c = __hsub2(*reinterpret_cast<const __half2*>(&q), k1032);
    const __half2 r = __hmul2(c, dd[i]);
    o[i] = *reinterpret_cast<const uint32_t*>(&r);
  }
}

// 8 x 8 transpose of 4-bit codes: r[s] holds row s (code j in bits 4j ..),
// c[j] gets column j (row s in bits 4s ..).  Two byte-permute stages swap
// 16-bit and 8-bit blocks, a mask stage swaps single codes.
__device__ __forceinline__ void transpose8x8_nibbles(const uint32_t* r, uint32_t* c) {
  uint32_t a[8], b[8];
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    a[s] = __byte_perm(r[s], r[s + 4], 0x5410);      // columns 0-3 of rows s, s + 4
    a[s + 4] = __byte_perm(r[s], r[s + 4], 0x7632);  // columns 4-7 of rows s, s + 4
  }
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const int i = 4 * h + s;
      b[i] = __byte_perm(a[i], a[i + 2], 0x6240);      // 2 columns, rows s, s + 2, s + 4, s + 6
      b[i + 2] = __byte_perm(a[i], a[i + 2], 0x7351);  // the next 2 columns, same rows
    }
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const uint32_t e = b[2 * t], o = b[2 * t + 1];  // even rows, odd rows of columns 2t, 2t + 1
    c[2 * t] = (e & 0x0F0F0F0Fu) | ((o & 0x0F0F0F0Fu) << 4);
    c[2 * t + 1] = ((e >> 4) & 0x0F0F0F0Fu) | (o & 0xF0F0F0F0u);
  }
}

// Bounded wait that sleeps between polls: for the epilogue warps, which wait
// a whole unit for their accumulator and would otherwise take issue slots
// from the dequant warps.
__device__ __forceinline__ bool mbar_wait_idle(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t i = 1; i < kSpinLimit; ++i) {
    __nanosleep(256);
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 15) == 0 && global_ns() - t0 > kWaitLimitNs) return false;
  }
  return false;
}

// fp16 scale of a raw stage (little-endian, 2-byte aligned) as a half2 pair
__device__ __forceinline__ __half2 scale2(const uint8_t* p) {
  return __half2half2(*reinterpret_cast<const __half*>(p));
}

}  // namespace

template <int PHASE>
__global__ void __launch_bounds__(kQ4Threads, 1) k_gemm_q4(const __grid_constant__ BatchParams P) {
  constexpr int kRS = PHASE == 0 ? kQ4RawStages0 : kQ4RawStages1;
  constexpr int kRB = PHASE == 0 ? kQ4Raw0 : kQ4Raw1;
  constexpr int kBS = PHASE == 0 ? kQ4BStages0 : kQ4BStages1;
  constexpr int kBB = PHASE == 0 ? kQ4B0 : kQ4B1;
  constexpr int kTS = PHASE == 0 ? kQ4AStages0 : kQ4TileStages1;  // A stages (tensor memory / shared)
  constexpr int kAPer = PHASE == 0 ? 2 : 1;                         // A stages per raw stage
  constexpr int kSubs = PHASE == 0 ? 4 : 1;                         // 64-wide K sub-chunks of B per raw stage
  constexpr uint32_t kCols = PHASE == 0 ? kQ4TmemCols0 : kQ4TmemCols1;
  // one accumulator buffer (of two): one accumulator per MMA issuer (gate /
  // up: 64 columns; down: two 64-column halves of the output tile)
  constexpr uint32_t kParCols = PHASE == 0 ? kGemmNC : 2 * kGemmNC;
  constexpr uint32_t kAccCols = 2 * kParCols;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* tiles = sm;                                             // down: kTS x kQ4Tile1
  uint8_t* bst = sm + (PHASE == 0 ? 0 : kTS * kQ4Tile1);           // kBS x kBB
  uint8_t* raws = bst + kBS * kBB;                                 // kRS x kRB
  float* exch = reinterpret_cast<float*>(raws + kRS * kRB);        // gate / up: [NC][64]
  uint64_t* bars = reinterpret_cast<uint64_t*>(raws + kRS * kRB + (PHASE == 0 ? kGemmExch : 0));
  uint64_t* raw_full = bars;
  uint64_t* raw_empty = raw_full + kRS;
  uint64_t* b_full = raw_empty + kRS;
  uint64_t* b_empty = b_full + kBS;
  uint64_t* a_full = b_empty + kBS;
  uint64_t* a_empty = a_full + kTS;
  uint64_t* acc_full = a_empty + kTS;  // [2]
  uint64_t* acc_empty = acc_full + 2;  // [2]
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_cum[kBatchMaxE + 2];
  __shared__ int s_grp[kBatchMaxE + 1][3];
  __shared__ float s_sw[kGemmNC];  // gate / up epilogue: the unit's slot weights

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = P.T, K = P.K;
  const int MT = PHASE == 0 ? P.I / 64 : P.H / 256;
  const int MT_s = PHASE == 0 ? P.Is / 64 : P.H / 256;

  pdl_launch_dependents();
  if (tid == 64) {
    for (int i = 0; i < kRS; ++i) {
      mbar_init(&raw_full[i], 1);
      mbar_init(&raw_empty[i], kQ4Dequant);
    }
    for (int i = 0; i < kBS; ++i) {
      mbar_init(&b_full[i], 1);
      mbar_init(&b_empty[i], PHASE == 0 ? 2 : 1);  // gate / up: both issuers read every B stage
    }
    for (int i = 0; i < kTS; ++i) {
      mbar_init(&a_full[i], kQ4Dequant);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 2);
      mbar_init(&acc_empty[i], 128);
    }
    s_abort = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                 "r"(kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  pdl_wait();
  if (warp == 0) {
    // groups (active experts ascending, then the shared expert) and the
    // prefix sums of their units
    const int U = *P.r_nactive;
    int sum = 0;
    int cnt[9];
#pragma unroll
    for (int q = 0; q < 9; ++q) {
      const int g = 9 * lane + q;
      cnt[q] = 0;
      if (g < U) {
        const int e = P.r_active[g];
        const int c = P.r_counts[e];
        s_grp[g][0] = e;
        s_grp[g][1] = P.r_offsets[e];
        s_grp[g][2] = c;
        cnt[q] = (c + kGemmNC - 1) / kGemmNC * MT;
      } else if (g == U) {
        s_grp[g][0] = -1;
        s_grp[g][1] = T * K;
        s_grp[g][2] = T;
        cnt[q] = (T + kGemmNC - 1) / kGemmNC * MT_s;
      }
      sum += cnt[q];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - sum;
#pragma unroll
    for (int q = 0; q < 9; ++q) {
      const int g = 9 * lane + q;
      if (g <= U + 1 && g < kBatchMaxE + 2) s_cum[g] = run;
      run += cnt[q];
    }
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const int U = *P.r_nactive;
  const int n_units = s_cum[U + 1];

  int gscan = 0;
  auto unit_of = [&](int u, UnitQ& w) {
    while (gscan < U && s_cum[gscan + 1] <= u) ++gscan;
    const int local = u - s_cum[gscan];
    const int mt = s_grp[gscan][0] < 0 ? MT_s : MT;
    const int chunk = local / mt;
    w.tile = local - chunk * mt;
    w.shared = s_grp[gscan][0] < 0;
    w.e = w.shared ? 0 : s_grp[gscan][0];
    w.slot0 = s_grp[gscan][1] + chunk * kGemmNC;  // shared slots: T K + token, in x_perm too
    w.n = min(kGemmNC, s_grp[gscan][2] - chunk * kGemmNC);
  };
  // raw stages of a unit: gate / up K = H in chunks of 256; down K = I (Is) in chunks of 64
  auto raw_chunks = [&](const UnitQ& w) { return PHASE == 0 ? P.H / 256 : (w.shared ? P.Is : P.I) / 64; };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // per K chunk: the raw stage (weights), then the B stage (slot rows);
    // the B ring is shallower, the raw ring runs ahead of it
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      int rs = 0, bs = 0;
      uint32_t rph = 0, bph = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok && !aborted(&s_abort); u += gridDim.x) {
        UnitQ w;
        unit_of(u, w);
        const CUtensorMap* mn = w.shared ? &P.tm_qn_s : &P.tm_qn_e;
        const CUtensorMap* ms = w.shared ? &P.tm_qs_s : &P.tm_qs_e;
        const int I = w.shared ? P.Is : P.I;
        const int npad = (w.n + 15) & ~15;
        const int nrc = raw_chunks(w);
        for (int rc = 0; rc < nrc; ++rc) {
          if (!mbar_wait(&raw_empty[rs], rph ^ 1u)) {
            ok = false;
            break;
          }
          uint8_t* dst = raws + (size_t)rs * kRB;
          mbar_arrive_expect_tx(&raw_full[rs], (uint32_t)kRB);
          if (PHASE == 0) {
            const int rg = w.e * 3 * I + w.tile * 64;  // gate rows; the up rows follow I rows later
            tma_load_2d(dst, mn, rc * 128, rg, &raw_full[rs], pol_w);
            tma_load_2d(dst + 8192, mn, rc * 128, rg + I, &raw_full[rs], pol_w);
            tma_load_2d(dst + 16384, ms, P.H / 2 + rc * 16, rg, &raw_full[rs], pol_w);
            tma_load_2d(dst + 16384 + 1024, ms, P.H / 2 + rc * 16, rg + I, &raw_full[rs], pol_w);
          } else {
            const int r = (w.e * 3 + 2) * I + rc * 64;  // downT rows (K); columns tile * 256 .. (M)
            tma_load_2d(dst, mn, w.tile * 128, r, &raw_full[rs], pol_w);
            tma_load_2d(dst + 8192, ms, P.H / 2 + w.tile * 16, r, &raw_full[rs], pol_w);
          }
          if (++rs == kRS) {
            rs = 0;
            rph ^= 1u;
          }
          if (!mbar_wait(&b_empty[bs], bph ^ 1u)) {
            ok = false;
            break;
          }
          uint8_t* bd = bst + (size_t)bs * kBB;
          mbar_arrive_expect_tx(&b_full[bs], (uint32_t)(kSubs * npad * 128));
          if (PHASE == 0) {
#pragma unroll
            for (int sc = 0; sc < 4; ++sc)
              for (int j = 0; j < npad; j += 16)
                tma_load_2d(bd + sc * (kGemmNC * 128) + j * 128, &P.tm_xp, (rc * 4 + sc) * 64, w.slot0 + j,
                            &b_full[bs], pol_x);
          } else {
            for (int j = 0; j < npad; j += 16)
              tma_load_2d(bd + j * 128, &P.tm_h, rc * 64, w.slot0 + j, &b_full[bs], pol_x);
          }
          if (++bs == kBS) {
            bs = 0;
            bph ^= 1u;
          }
        }
      }
      if (!ok) set_abort(&s_abort);
      // wind down: every issued copy has landed before the block exits
      for (int i = 0; i < kRS; ++i) mbar_wait(&raw_full[i], i < rs ? rph : rph ^ 1u);
      for (int i = 0; i < kBS; ++i) mbar_wait(&b_full[i], i < bs ? bph : bph ^ 1u);
    }
  } else if (warp == 1 || warp == 14) {
    // ---------------------------------------------------------- MMA issuers
    // Two issuers, each into its own accumulator (the epilogue adds the two
    // in a fixed order), so that one issuer's waits and commits overlap the
    // other's MMAs.  gate / up: warp 1 the first 128 K of every raw stage,
    // warp 14 the second; down: warp 1 the even raw stages of a unit, warp
    // 14 the odd ones.
    const int par = warp == 14 ? 1 : 0;
    if (lane == 0) {
      int bs = 0, ts = 0, nu = 0;
      uint32_t bph = 0, tph = 0;
      bool pending = false;
      for (int u = blockIdx.x; u < n_units && !aborted(&s_abort); u += gridDim.x, ++nu) {
        UnitQ w;
        unit_of(u, w);
        const int nrc = raw_chunks(w);
        const int npad = (w.n + 15) & ~15;
        const uint32_t idesc = instr_desc(128, npad, 0, true);  // A and B K-major
        const int ab = nu & 1;
        const uint32_t acc_ph = (uint32_t)(nu >> 1) & 1u;
        const uint32_t dacc = tmem + (uint32_t)ab * kAccCols + (uint32_t)par * kParCols;
        if (!mbar_wait(&acc_empty[ab], acc_ph ^ 1u)) {
          set_abort(&s_abort);
          break;
        }
        tc_fence_after();
        bool ok = true;
        for (int rc = 0; rc < nrc; ++rc) {
          if (PHASE == 1 && (rc & 1) != par) {  // the other issuer's stage
            if (++ts == kTS) {
              ts = 0;
              tph ^= 1u;
            }
            if (++bs == kBS) {
              bs = 0;
              bph ^= 1u;
            }
            continue;
          }
          const int ta = PHASE == 0 ? ts + par : ts;  // gate / up: this issuer's A stage of the pair
          ok = mbar_wait(&b_full[bs], bph) && mbar_wait(&a_full[ta], tph);
          if (!ok) break;
          tc_fence_after();
          const uint32_t sb = smem_u32(bst + (size_t)bs * kBB);
          if (PHASE == 0) {
            // 128 K: A columns kQ4ACol0 + 64 ta + 8 ks, B sub-chunks 2 par, 2 par + 1
            const uint64_t bdsc = smem_desc(sb + par * (2 * kGemmNC * 128), 16, 1024);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
              umma_ts(dacc, tmem + (uint32_t)(kQ4ACol0 + 64 * ta + 8 * ks),
                      bdsc + (uint64_t)((ks >> 2) * (kGemmNC * 128 / 16) + (ks & 3) * 2), idesc,
                      (rc > 0 || ks > 0) ? 1u : 0u);
          } else {
            const uint64_t adsc = smem_desc(smem_u32(tiles + (size_t)ts * kQ4Tile1), 16, 1024);
            const uint64_t bdsc = smem_desc(sb, 16, 1024);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {  // +32 bytes of K per step: +2 in the address field
              const uint32_t acc = (rc >= 2 || ks > 0) ? 1u : 0u;  // this issuer's first stage starts the sum
              umma(dacc, adsc + 2 * ks, bdsc + 2 * ks, idesc, acc);
              umma(dacc + kGemmNC, adsc + 1024 + 2 * ks, bdsc + 2 * ks, idesc, acc);  // +16 KB: second half
            }
          }
          umma_commit(&a_empty[ta]);
          umma_commit(&b_empty[bs]);
          pending = true;
          if ((ts += kAPer) == kTS) {
            ts = 0;
            tph ^= 1u;
          }
          if (++bs == kBS) {
            bs = 0;
            bph ^= 1u;
          }
        }
        if (!ok) {
          set_abort(&s_abort);
          // left with MMAs in flight: they complete before the block frees its tensor memory
          if (pending) {
            umma_commit(&acc_full[ab]);
            mbar_wait(&acc_full[ab], acc_ph);
          }
          pending = false;
          break;
        }
        umma_commit(&acc_full[ab]);
        pending = false;
      }
    }
  } else if (warp >= 2 && warp < 10) {
    // ------------------------------------------------------------ dequant
    // Two groups of four warps (warps 2-5, 6-9; each covers the four lane
    // quarters) take alternate raw stages, so two stages are in flight.
    // Each warp runs on its own: the waits are per thread, the exit test
    // warp-uniform (tcgen05.st is warp-collective).
    const int grp = (warp - 2) >> 2;
    const int dt = (warp & 3) * 32 + lane;  // 0 .. 127 within the group
    int rs = 0, ts = 0, cc = 0;
    uint32_t rph = 0, tph = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      UnitQ w;
      unit_of(u, w);
      const int nrc = raw_chunks(w);
      for (int rc = 0; rc < nrc; ++rc, ++cc) {
        if ((cc & 1) == grp) {
          ok = __all_sync(0xffffffffu, mbar_wait(&raw_full[rs], rph) && mbar_wait(&a_empty[ts], tph ^ 1u) &&
                                           (kAPer == 1 || mbar_wait(&a_empty[ts + kAPer - 1], tph ^ 1u)) &&
                                           !aborted(&s_abort));
          if (!ok) break;
          const uint8_t* raw = raws + (size_t)rs * kRB;
          if (PHASE == 0) {
            // this thread: A row m (tensor-memory lane; 64 gate rows over 64
            // up rows), the stage's 256 K: 16-byte units 0..7 of the row,
            // one scale block each; units 0-3 go to A stage ts, 4-7 to ts + 1
            const int q = warp & 3;
            const int m = 32 * q + lane, rr = m & 63;
            const uint8_t* nib = raw + (m >> 6) * 8192 + rr * 128;
            const uint8_t* scl = raw + 16384 + (m >> 6) * 1024 + rr * 16;
            uint4 wq[8];
            __half2 dd[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              wq[j] = *reinterpret_cast<const uint4*>(nib + ((j ^ (rr & 7)) << 4));
              dd[j] = scale2(scl + j * 2);
            }
            mbar_arrive(&raw_empty[rs]);  // this thread's reads of the raw stage are done
            const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(kQ4ACol0 + 64 * ts);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              uint32_t v[16];
              dequant8(wq[j].x, dd[j], v);
              dequant8(wq[j].y, dd[j], v + 4);
              dequant8(wq[j].z, dd[j], v + 8);
              dequant8(wq[j].w, dd[j], v + 12);
              tmem_st16(ta + 16 * j, v);  // columns 64 ts + 16 j: stage ts + j / 4
            }
            tmem_wait_st();
            tc_fence_before();
          } else {
            // 64 rows (K) x 256 columns (M) -> two K-major 128-row tiles.
            // Item (k8, g): rows 8 k8 .. + 7, columns 8 g .. + 7; this thread
            // takes g and g + 16.  The rows are read rotated by k8 (register s
            // holds row (s + k8) % 8, which keeps the reads conflict-free),
            // transposed to one code word per column, and stored as one
            // 16-byte unit per column: position p holds row
            // (p / 2 + 4 (p % 2) + k8) % 8 of the group, the order in which
            // the gate / up epilogue writes h.
            uint8_t* tile = tiles + (size_t)ts * kQ4Tile1;
            const int k8 = dt & 7;
            uint32_t rw[2][8];
            __half dsc[2][8];
#pragma unroll
            for (int it = 0; it < 2; ++it) {
              const int g = (dt >> 3) + 16 * it;
#pragma unroll
              for (int s2 = 0; s2 < 8; ++s2) {
                const int i = 8 * k8 + ((s2 + k8) & 7);
                rw[it][s2] =
                    *reinterpret_cast<const uint32_t*>(raw + i * 128 + (((g >> 2) ^ (i & 7)) << 4) + (g & 3) * 4);
                dsc[it][s2] = *reinterpret_cast<const __half*>(raw + 8192 + i * 16 + (g >> 2) * 2);
              }
            }
            mbar_arrive(&raw_empty[rs]);
#pragma unroll
            for (int it = 0; it < 2; ++it) {
              const int g = (dt >> 3) + 16 * it;
              __half2 dd[4];
#pragma unroll
              for (int q2 = 0; q2 < 4; ++q2) dd[q2] = __halves2half2(dsc[it][q2], dsc[it][q2 + 4]);
              uint32_t cw[8];
              transpose8x8_nibbles(rw[it], cw);
              uint8_t* dst = tile + (g >> 4) * 16384 + (g & 15) * 1024;
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                uint32_t v[4];
                dequant8s(cw[j], dd, v);
                *reinterpret_cast<uint4*>(dst + j * 128 + ((k8 ^ j) << 4)) = make_uint4(v[0], v[1], v[2], v[3]);
              }
            }
            fence_async_smem();  // the tile's generic writes, visible to the tensor cores
          }
          mbar_arrive(&a_full[ts]);
          if (kAPer == 2) mbar_arrive(&a_full[ts + 1]);
        }
        if ((ts += kAPer) == kTS) {
          ts = 0;
          tph ^= 1u;
        }
        if (++rs == kRS) {
          rs = 0;
          rph ^= 1u;
        }
      }
    }
    if (!ok) set_abort(&s_abort);
  } else if (warp < 14) {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;
    const int m = 32 * q + lane;
    const uint32_t lane_addr = (uint32_t)(32 * q) << 16;
    uint16_t* h_ws = P.h_ws;
    int nu = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++nu) {
      UnitQ w;
      unit_of(u, w);
      const int ab = nu & 1;
      const uint32_t acc = tmem + lane_addr + (uint32_t)ab * kAccCols;
      const bool ok = mbar_wait_idle(&acc_full[ab], (uint32_t)(nu >> 1) & 1u) && !aborted(&s_abort);
      if (!epilogue_all(ok)) {
        set_abort(&s_abort);
        break;
      }
      tc_fence_after();
      if (PHASE == 0) {
        // lanes 0..63 gate, 64..127 up of the same rows tile * 64 ..
        const int r = m & 63;
        if (q < 2) {
          if (r < w.n) s_sw[r] = P.slot_w[w.slot0 + r];
          for (int j0 = 0; j0 < w.n; j0 += 16) {
            uint32_t v[16], v2[16];
            tmem_ld16(acc + (uint32_t)j0, v);
            tmem_ld16(acc + kParCols + (uint32_t)j0, v2);  // the second K half
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) exch[(j0 + jj) * 64 + r] = __uint_as_float(v[jj]) + __uint_as_float(v2[jj]);
          }
        }
        epilogue_sync();
        if (q >= 2) {
          // h row i of the slot goes to position 8 G + p of group G = i / 8,
          // where (p / 2 + 4 (p % 2) + G) % 8 = i % 8: the K order of the
          // down kernel's A tiles
          const int i = w.tile * 64 + r;
          const int xr = ((i & 7) - (i >> 3)) & 7;
          const int ip = (i & ~7) + 2 * (xr & 3) + (xr >> 2);
          for (int j0 = 0; j0 < w.n; j0 += 16) {
            uint32_t v[16], v2[16];
            tmem_ld16(acc + (uint32_t)j0, v);
            tmem_ld16(acc + kParCols + (uint32_t)j0, v2);
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int j = j0 + jj;
              if (j < w.n) {
                const int slot = w.slot0 + j;
                const float g = exch[j * 64 + r], up = __uint_as_float(v[jj]) + __uint_as_float(v2[jj]);
                const float h = __fdividef(g, 1.0f + __expf(-g)) * up * s_sw[j];
                h_ws[(size_t)slot * (size_t)P.hw + ip] = __half_as_ushort(__float2half_rn(h));
              }
            }
          }
        }
        tc_fence_before();
        epilogue_sync();
      } else {
        // accumulator row 128 half + m holds output column tile * 256 + 128 half + m
        const int c0 = w.tile * 256 + m;
        // the even-stage accumulator plus the odd-stage one
        for (int j0 = 0; j0 < w.n; j0 += 16) {
          uint32_t r0[16], r1[16], s0[16], s1[16];
          tmem_ld16(acc + (uint32_t)j0, r0);
          tmem_ld16(acc + (uint32_t)kGemmNC + (uint32_t)j0, r1);
          tmem_ld16(acc + (uint32_t)(2 * kGemmNC) + (uint32_t)j0, s0);
          tmem_ld16(acc + (uint32_t)(3 * kGemmNC) + (uint32_t)j0, s1);
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const int j = j0 + jj;
            if (j < w.n) {
              float* dst = P.y_ws + (size_t)(w.slot0 + j) * P.H + c0;
              dst[0] = __uint_as_float(r0[jj]) + __uint_as_float(s0[jj]);
              dst[128] = __uint_as_float(r1[jj]) + __uint_as_float(s1[jj]);
            }
          }
        }
        tc_fence_before();
      }
      mbar_arrive(&acc_empty[ab]);
    }
  }
  __syncthreads();
  if (aborted(&s_abort) && tid == 0) atomicExch(reinterpret_cast<int*>(&P.ctrl[kCtrlStatus]), kStatusTimeout);
  tc_fence_before();
  __syncthreads();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols) : "memory");
}

template <int PHASE>
static cudaError_t launch_q4(const BatchParams& p, cudaStream_t stream) {
  constexpr int smem = PHASE == 0 ? kQ4Smem0 : kQ4Smem1;
  cudaError_t err = cudaFuncSetAttribute(k_gemm_q4<PHASE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(p.G);
  cfg.blockDim = dim3(kQ4Threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_gemm_q4<PHASE>, p);
}

cudaError_t launch_gemm_gate_up_q4(const BatchParams& p, cudaStream_t stream) { return launch_q4<0>(p, stream); }
cudaError_t launch_gemm_down_q4(const BatchParams& p, cudaStream_t stream) { return launch_q4<1>(p, stream); }

}  // namespace moe
