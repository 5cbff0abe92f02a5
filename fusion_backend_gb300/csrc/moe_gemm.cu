// Grouped GEMMs of the batched MoE FFN layer on the 5th-generation tensor
// cores (tcgen05), sm_103a.
//
// A group is one active expert (its slots offsets[e] .. + counts[e], x rows
// gathered in x_perm) or the shared expert (slot T K + t for every token t,
// x itself).  Groups are cut into units of at most kGemmNC slots (the MMA N)
// and a tile of the weights; the persistent blocks take units round robin.
//
//   gate / up (PHASE 0):  [G; U] = [W_g; W_u] X^T over K = H: 64 rows of I
//     of the gate matrix over the same 64 rows of the up matrix form one
//     128-row A tile, so one accumulator holds both; h = silu(G) * U *
//     w(slot), stored as two bf16 parts, hi = bf16(h) and lo = bf16(h - hi),
//     in the rows h_ws[slot][2 hw] (hi in [0, hw), lo in [hw, 2 hw)).
//   down (PHASE 1):  Y^T = downT^T (H_hi + H_lo)^T over K = I (Is for the
//     shared expert), 256 output columns per unit (two 128-column
//     accumulators); the downT tile is the MN-major A operand, straight from
//     its [I][H] rows, and every K step runs once with each part of h, so h
//     enters the products with about 16 significant bits instead of bf16's
//     8; y_ws[slot][H] in fp32.
//
// Block roles: warp 0 lane 0 moves tiles with TMA into a ring of stages
// (one or two 128 x 64 A tiles + an NC x 64 B tile, 128-byte swizzled);
// warp 1 owns the tensor memory (two fp32 accumulators of up to kGemmNC
// columns) and lane 0 issues the MMAs (M = 128,
// N = slots rounded up to 16, K = 16), committing each ring slot back to the
// producer and each finished unit to the epilogue; warps 2..5 read the
// accumulators (warp w reads lanes 32 (w % 4) ..) and write the unit's rows.
// Every wait is bounded; a wait that gives up sets the status word and the
// block winds down without leaving copies or tensor-core work in flight.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "moe_tc.cuh"

namespace moe {

namespace {

using namespace tc;

// One unit of work.
struct Unit {
  int shared;  // the shared expert
  int e;       // expert (routed)
  int slot0;   // first slot (row of h_ws / y_ws; of x_perm for routed gate / up)
  int brow0;   // first row of the B operand
  int n;       // slots (1 .. kGemmNC)
  int tile;    // row tile (gate / up: 128 rows of I) or column tile (down: 256 columns of H)
};

}  // namespace

template <int PHASE>
__global__ void __launch_bounds__(kGemmThreads, 1) k_gemm(const __grid_constant__ BatchParams P) {
  constexpr int kS = PHASE == 0 ? kGemmStages0 : kGemmStages1;
  constexpr int kSB = PHASE == 0 ? kGemmStageBytes0 : kGemmStageBytes1;
  constexpr int kA = PHASE == 0 ? 128 * 128 : 2 * 128 * 128;  // A bytes of a 64-wide K sub-chunk; its B tile follows
  constexpr int kKSub = PHASE == 0 ? kGemmKSub0 : 1;            // K sub-chunks per stage
  constexpr int kSub = kA + kGemmNC * 128;                       // bytes of one sub-chunk
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* ring = sm;  // kS x kSB, 1024-byte aligned slots
  float* exch = reinterpret_cast<float*>(sm + kS * kSB);  // gate / up: [NC][64] gate values
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + kS * kSB + (PHASE == 0 ? kGemmExch : 0));
  uint64_t* empty = full + kS;
  uint64_t* acc_full = empty + kS;
  uint64_t* acc_empty = acc_full + 1;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_cum[kBatchMaxE + 2];     // units before group g
  __shared__ int s_grp[kBatchMaxE + 1][3];  // group g: expert (-1 shared), first slot, slots

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = P.T, K = P.K;
  // weight tiles per slot chunk: gate / up 64 rows of I (Is), down 256 columns of H
  const int MT = PHASE == 0 ? P.I / 64 : P.H / 256;
  const int MT_s = PHASE == 0 ? P.Is / 64 : P.H / 256;

  pdl_launch_dependents();
  // ---- barriers (thread 64) and tensor memory (warp 1) before the wait on
  // the previous kernel; then the groups and their unit counts (warp 0)
  if (tid == 64) {
    for (int i = 0; i < kS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 128);
    s_abort = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                 "r"(2 * kGemmNC)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  pdl_wait();
  if (warp == 0) {
    const int U = *P.r_nactive;
    // lane l sums groups [9l, 9l + 9) (U + 1 <= 257 groups)
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

  // unit u -> its group and tile, scanning forward from the last group
  int gscan = 0;
  auto unit_of = [&](int u, Unit& w) {
    while (gscan < U && s_cum[gscan + 1] <= u) ++gscan;
    const int local = u - s_cum[gscan];
    const int mt = s_grp[gscan][0] < 0 ? MT_s : MT;
    const int chunk = local / mt;
    w.tile = local - chunk * mt;
    w.shared = s_grp[gscan][0] < 0;
    w.e = w.shared ? 0 : s_grp[gscan][0];
    w.slot0 = s_grp[gscan][1] + chunk * kGemmNC;
    w.n = min(kGemmNC, s_grp[gscan][2] - chunk * kGemmNC);
    // B rows: gate / up read x_perm (routed) or x (shared, row = token);
    // down reads h_ws at the slot rows
    w.brow0 = (PHASE == 0 && w.shared) ? chunk * kGemmNC : w.slot0;
  };
  // stages per unit (K / (64 kKSub))
  const int nk_r = PHASE == 0 ? P.H / (64 * kKSub) : P.I / 64;
  const int nk_s = PHASE == 0 ? P.H / (64 * kKSub) : P.Is / 64;

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      int stage = 0;
      uint32_t ph = 0;
      for (int u = blockIdx.x; u < n_units && !aborted(&s_abort); u += gridDim.x) {
        Unit w;
        unit_of(u, w);
        const int nk = w.shared ? nk_s : nk_r;
        const int npad = (w.n + 15) & ~15;
        const uint32_t bytes = kKSub * (kA + (PHASE == 0 ? 1u : 2u) * (uint32_t)npad * 128);
        const CUtensorMap* m = w.shared ? &P.tm_w64_s : &P.tm_w64_e;
        const int I = w.shared ? P.Is : P.I;
        for (int kc = 0; kc < nk; ++kc) {
          if (!mbar_wait(&empty[stage], ph ^ 1u)) {
            set_abort(&s_abort);
            break;
          }
          uint8_t* slot = ring + (size_t)stage * kSB;
          mbar_arrive_expect_tx(&full[stage], bytes);
          if (PHASE == 0) {
            // per sub-chunk: 64 gate rows over the same 64 up rows (one
            // 128-row A tile) and the B rows, k columns (kKSub kc + sc) * 64 ..
            const int rb = w.e * 3 * I + w.tile * 64;
            const CUtensorMap* bm = w.shared ? &P.tm_x : &P.tm_xp;
#pragma unroll
            for (int sc = 0; sc < kKSub; ++sc) {
              const int k0 = (kc * kKSub + sc) * 64;
              uint8_t* sub = slot + sc * kSub;
              tma_load_2d(sub, m, k0, rb, &full[stage], pol_w);
              tma_load_2d(sub + 8192, m, k0, rb + I, &full[stage], pol_w);
              for (int j = 0; j < npad; j += 16)
                tma_load_2d(sub + kA + j * 128, bm, k0, w.brow0 + j, &full[stage], pol_x);
            }
          } else {
            // downT rows kc*64 .. (k) x columns tile*256 .. (m), four 64-column boxes
            const int r = (w.e * 3 + 2) * I + kc * 64;
#pragma unroll
            for (int q = 0; q < 4; ++q) tma_load_2d(slot + q * 8192, m, w.tile * 256 + 64 * q, r, &full[stage], pol_w);
            for (int j = 0; j < npad; j += 16) {
              tma_load_2d(slot + kA + j * 128, &P.tm_h, kc * 64, w.brow0 + j, &full[stage], pol_x);
              tma_load_2d(slot + kA + kGemmNC * 128 + j * 128, &P.tm_h, P.hw + kc * 64, w.brow0 + j, &full[stage],
                          pol_x);
            }
          }
          if (++stage == kS) {
            stage = 0;
            ph ^= 1u;
          }
        }
      }
      // wind down: every issued copy has landed before the block exits
      for (int i = 0; i < kS; ++i) {
        // slot i was last filled in the phase before (stage, ph), the next fill
        const uint32_t last = i < stage ? ph : ph ^ 1u;
        mbar_wait(&full[i], last);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t ph = 0, acc_ph = 0;
      bool pending = false;  // MMAs issued for a unit whose accumulator is not committed
      for (int u = blockIdx.x; u < n_units && !aborted(&s_abort); u += gridDim.x) {
        Unit w;
        unit_of(u, w);
        const int nk = w.shared ? nk_s : nk_r;
        const int npad = (w.n + 15) & ~15;
        const uint32_t idesc = instr_desc(128, npad, PHASE);
        if (!mbar_wait(acc_empty, acc_ph ^ 1u)) {
          set_abort(&s_abort);
          break;
        }
        tc_fence_after();
        for (int kc = 0; kc < nk; ++kc) {
          if (!mbar_wait(&full[stage], ph)) {
            set_abort(&s_abort);
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(ring + (size_t)stage * kSB);
#pragma unroll
          for (int ks = 0; ks < 4 * kKSub; ++ks) {
            const uint32_t sub = sa + (ks >> 2) * kSub;  // sub-chunk base
            const uint64_t bd = smem_desc(sub + kA + (ks & 3) * 32, 16, 1024);
            const uint32_t acc = (kc > 0 || ks > 0) ? 1u : 0u;
            if (PHASE == 0) {
              umma(tmem, smem_desc(sub + (ks & 3) * 32, 16, 1024), bd, idesc, acc);
            } else {
              // h hi, then h lo, into each of the two column halves
              const uint64_t bl = smem_desc(sub + kA + kGemmNC * 128 + (ks & 3) * 32, 16, 1024);
              const uint64_t a0 = smem_desc(sa + ks * 2048, 8192, 1024), a1 = smem_desc(sa + 16384 + ks * 2048, 8192, 1024);
              umma(tmem, a0, bd, idesc, acc);
              umma(tmem, a0, bl, idesc, 1u);
              umma(tmem + kGemmNC, a1, bd, idesc, acc);
              umma(tmem + kGemmNC, a1, bl, idesc, 1u);
            }
          }
          umma_commit(&empty[stage]);
          pending = true;
          if (++stage == kS) {
            stage = 0;
            ph ^= 1u;
          }
        }
        if (aborted(&s_abort)) break;
        umma_commit(acc_full);
        pending = false;
        acc_ph ^= 1u;
      }
      // after a wait that gave up: the tensor cores finish the MMAs in
      // flight before the tensor memory is released
      if (pending) {
        umma_commit(acc_full);
        mbar_wait(acc_full, acc_ph);
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;  // lane quarter of the accumulator this warp reads
    const int m = 32 * q + lane;
    const uint32_t lane_addr = (uint32_t)(32 * q) << 16;
    uint32_t acc_ph = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      Unit w;
      unit_of(u, w);
      const bool ok = mbar_wait(acc_full, acc_ph) && !aborted(&s_abort);
      if (!epilogue_all(ok)) {
        set_abort(&s_abort);
        break;
      }
      tc_fence_after();
      if (PHASE == 0) {
        // rows 0..63 of the accumulator are gate rows, 64..127 the same up
        // rows: the gate half goes through shared memory to the up half
        const int r = m & 63;
        if (q < 2) {
          for (int j0 = 0; j0 < w.n; j0 += 16) {
            uint32_t v[16];
            tmem_ld16(tmem + lane_addr + (uint32_t)j0, v);
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) exch[(j0 + jj) * 64 + r] = __uint_as_float(v[jj]);
          }
        }
        epilogue_sync();
        if (q >= 2) {
          const int i = w.tile * 64 + r;
          for (int j0 = 0; j0 < w.n; j0 += 16) {
            uint32_t v[16];
            tmem_ld16(tmem + lane_addr + (uint32_t)j0, v);
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int j = j0 + jj;
              if (j < w.n) {
                const int slot = w.slot0 + j;
                const float g = exch[j * 64 + r], up = __uint_as_float(v[jj]);
                const float h = g / (1.0f + expf(-g)) * up * P.slot_w[slot];
                const uint16_t hi = float_to_bf16_rne(h);
                uint16_t* row = P.h_ws + (size_t)slot * (size_t)(2 * P.hw);
                row[i] = hi;
                row[P.hw + i] = float_to_bf16_rne(h - bf16_to_float(hi));
              }
            }
          }
        }
        epilogue_sync();  // the exchange buffer is free for the next unit
      } else {
        const int c = w.tile * 256 + m;
        for (int j0 = 0; j0 < w.n; j0 += 16) {
          uint32_t r0[16], r1[16];
          tmem_ld16(tmem + lane_addr + (uint32_t)j0, r0);
          tmem_ld16(tmem + lane_addr + (uint32_t)kGemmNC + (uint32_t)j0, r1);
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const int j = j0 + jj;
            if (j < w.n) {
              float* dst = P.y_ws + (size_t)(w.slot0 + j) * P.H + c;
              dst[0] = __uint_as_float(r0[jj]);
              dst[128] = __uint_as_float(r1[jj]);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(acc_empty);
      acc_ph ^= 1u;
    }
  }
  __syncthreads();
  if (aborted(&s_abort) && tid == 0) atomicExch(reinterpret_cast<int*>(&P.ctrl[kCtrlStatus]), kStatusTimeout);
  tc_fence_before();
  __syncthreads();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * kGemmNC) : "memory");
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 gemm_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    tried = true;
  }
  return fn;
}

// 2-D bf16 view [rows][cols] (row pitch cols * 2 bytes) with a box of
// bcols x brows, 128-byte swizzled in shared memory.
bool encode_2d(PFN_cuTensorMapEncodeTiled_v12000 fn, CUtensorMap* m, const void* base, long long rows, int cols,
               int bcols, int brows) {
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)bcols, (cuuint32_t)brows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D byte view [rows][row_bytes] of stored 4-bit weight rows with a box of
// bbytes x 64 rows: 128-byte swizzled (codes) or plain (scales).
bool encode_q4(PFN_cuTensorMapEncodeTiled_v12000 fn, CUtensorMap* m, const void* base, long long rows,
               long long row_bytes, int bbytes, bool swizzle) {
  const cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  const cuuint32_t box[2] = {(cuuint32_t)bbytes, 64u};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t batch_tensor_maps(BatchParams& p) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = gemm_encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const long long er = (long long)p.E * 3 * p.I, sr = 3LL * p.Is, TK = (long long)p.T * p.K;
  if (p.wfmt == 1) {
    // 4-bit rows: codes and scales of the expert and shared blocks; B rows
    // in fp16: x_perm (routed slots, then the shared slots T K + t) and h_ws
    if (!encode_q4(fn, &p.tm_qn_e, p.expert_w, er, p.rb, 128, true) ||
        !encode_q4(fn, &p.tm_qs_e, p.expert_w, er, p.rb, 16, false) ||
        !encode_q4(fn, &p.tm_qn_s, p.shexp_w, sr, p.rb, 128, true) ||
        !encode_q4(fn, &p.tm_qs_s, p.shexp_w, sr, p.rb, 16, false) ||
        !encode_2d(fn, &p.tm_xp, p.x_perm, TK + p.T, p.H, 64, 16) ||
        !encode_2d(fn, &p.tm_h, p.h_ws, TK + p.T, p.hw, 64, 16))
      return cudaErrorInvalidValue;
    return cudaSuccess;
  }
  if (!encode_2d(fn, &p.tm_w64_e, p.expert_w, er, p.H, 64, 64) ||
      !encode_2d(fn, &p.tm_w64_s, p.shexp_w, sr, p.H, 64, 64) ||
      !encode_2d(fn, &p.tm_xp, p.x_perm, TK, p.H, 64, 16) || !encode_2d(fn, &p.tm_x, p.x, p.T, p.H, 64, 16) ||
      !encode_2d(fn, &p.tm_h, p.h_ws, TK + p.T, 2 * p.hw, 64, 16))
    return cudaErrorInvalidValue;
  return cudaSuccess;
}

template <int PHASE>
static cudaError_t launch_gemm(const BatchParams& p, cudaStream_t stream) {
  constexpr int smem = PHASE == 0 ? kGemmSmem0 : kGemmSmem1;
  cudaError_t err = cudaFuncSetAttribute(k_gemm<PHASE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  // behind the previous kernel with programmatic stream serialisation (the
  // kernel waits on it after its set-up)
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(p.G);
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_gemm<PHASE>, p);
}

cudaError_t launch_gemm_gate_up(const BatchParams& p, cudaStream_t stream) { return launch_gemm<0>(p, stream); }
cudaError_t launch_gemm_down(const BatchParams& p, cudaStream_t stream) { return launch_gemm<1>(p, stream); }

}  // namespace moe
