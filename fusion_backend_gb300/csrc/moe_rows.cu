// Row kernel: choice of instance and shared-memory layout (host side).
#include <cudaTypedefs.h>

#include <algorithm>

#include "moe_ffn.h"
#include "moe_rows.cuh"

namespace moe {

static_assert(int(kWkBf16) == int(MOE_FFN_W_BF16) && int(kWkQ4) == int(MOE_FFN_W_Q4B32) && int(kWkI8) == int(MOE_FFN_W_I8),
              "weight kinds follow the public weight formats");

cudaError_t launch_rows_bf16_fast(const LayerParams& p, cudaStream_t stream);
cudaError_t launch_rows_q4_fast(const LayerParams& p, cudaStream_t stream);
cudaError_t launch_rows_i8_fast(const LayerParams& p, cudaStream_t stream);
cudaError_t launch_rows_generic(const LayerParams& p, cudaStream_t stream);

namespace {

// The fast (tensor-core) instances: H = 2048, E <= 256, and an activation
// that bf16 holds exactly -- bf16 x, or the block form whose normalised
// input is bf16 -- so that it enters the bf16 products unchanged (int8
// weights quantise it, which needs no more).
bool rows_fast(const LayerParams& p) { return p.H == 2048 && p.E <= 256 && (p.act == 1 || p.block_mode); }

// Rows per stage at most, by weight format.
int rows_rsm(int wfmt) { return wfmt == kWkBf16 ? kRsMaxB16 : kRsMaxQ4; }

int align128(int v) { return (v + 127) & ~127; }

}  // namespace

// Layout with `rs` rows per stage; false when fewer than 3 stages fit.
static bool rows_layout_rs(LayerParams& p, int rs, int xbytes, int tab, int tmax) {
  p.rs = rs;
  p.rp = (int)p.rb;
  p.stage_bytes = 3 * rs * p.rp;
  p.off_bar = 0;
  p.off_tab = 256;
  const int rsm = rows_rsm(p.wfmt);
  p.off_h = align128(p.off_tab + tab);
  // h by stage parity, then (int8) the stage's row scales by parity
  p.off_part = align128(p.off_h + 2 * rsm * tmax * 4 + 2 * 3 * kRsMaxQ4 * 4);
  p.off_x = align128(p.off_part + 2 * kRowWarps * 2 * rsm * tmax * 4);
  p.off_ring = (p.off_x + xbytes + 1023) & ~1023;  // 128-byte-swizzled tensor copies want 1024-byte alignment
  if (p.off_ring >= kSmemBudget) return false;
  // the end-of-kernel column sums reuse the ring: max(threads, T x columns) floats
  const int red_bytes = std::max(kRowThreads, p.T * ((p.H + p.G - 1) / p.G)) * 4;
  const int avail = kSmemBudget - 1024 - p.off_ring;  // 1024: slack to align the ring in the shared window
  if (rows_fast(p)) {
    // tensor-core path: a ring of gate + up boxes (2 rs rows) and a ring of
    // downT boxes (rs rows) with one slot more.  Int8: the boxes hold the H
    // codes of each row, then (1 KB further, keeping slots 1 KB aligned) the
    // rows' 16-byte scale records.
    const bool i8 = p.wfmt == kWkI8;
    p.stage_bytes = i8 ? 2 * rs * p.H + 1024 : 2 * rs * p.rp;
    const int dbytes = i8 ? rs * p.H + 1024 : rs * p.rp;
    p.dstage_bytes = dbytes;
    p.ns = std::min(kMaxStagesRing - 1, (avail - dbytes) / (p.stage_bytes + dbytes));
    p.nsd = p.ns + 1;
    if (p.ns < 2 || red_bytes > p.ns * p.stage_bytes) return false;
    p.off_dring = p.off_ring + p.ns * p.stage_bytes;
    p.smem = p.off_dring + p.nsd * dbytes + 1024;
    return true;
  }
  p.nsd = 0;
  p.ns = std::min(kMaxStagesRing, avail / p.stage_bytes);
  if (p.ns < 3 || red_bytes > p.ns * p.stage_bytes) return false;
  p.off_dring = p.off_ring;
  p.smem = p.off_ring + p.ns * p.stage_bytes + 1024;
  return true;
}

int rows_layout(LayerParams& p) {
  if (p.T < 1 || p.T > kDecodeMaxT || p.H < 8 || p.H > kMaxH || p.G < 1 || p.G > kMaxGrid) return -1;
  if (p.wfmt < kWkBf16 || p.wfmt > kWkI8) return -1;
  if (p.H % (p.wfmt == kWkQ4 ? 256 : p.wfmt == kWkI8 ? 16 : 8)) return -1;
  const bool fast = rows_fast(p);
  const int tmax = fast ? tmax_for(p.T) : 8;
  p.rb = p.wfmt == kWkQ4 ? (long long)p.H * 9 / 16 : p.wfmt == kWkI8 ? (long long)p.H + 16 : (long long)p.H * 2;
  p.expert_bytes = 3LL * p.I * p.rb;
  p.xmode = fast ? kXReg : kXF32;
  // x region: the bulk copy of the source rows (fp32 for fp32 x and the block
  // form, else bf16), rewritten in place into the compute form
  const bool src4 = p.act == 0 || p.block_mode;
  int xbytes = p.T * p.H * (p.xmode == kXF32 || src4 ? 4 : 2);
  if (fast) xbytes = std::max(xbytes, p.T * kXPitch);  // rewritten in place as A fragments
  const int tab = row_tab(nullptr, p.T, p.K, p.E, nullptr);
  // Rows per stage: the choice that keeps the most bytes in flight (all ns
  // stages), with at least 3 stages in the ring; ties go to larger stages.
  const int rs_list[4] = {8, 4, 2, 1};
  int best_rs = 0;
  long long best_flight = -1;
  for (int r = 0; r < 4; ++r) {
    if (rs_list[r] > rows_rsm(p.wfmt)) continue;
    if (fast && rs_list[r] != rows_rsm(p.wfmt)) continue;  // tensor-core stages: fixed rows
    LayerParams t = p;
    if (!rows_layout_rs(t, rs_list[r], xbytes, tab, tmax)) continue;
    const long long flight = (long long)t.ns * t.stage_bytes + (long long)t.nsd * t.rs * t.rp;
    if (flight > best_flight) {
      best_flight = flight;
      best_rs = rs_list[r];
    }
  }
  if (best_rs == 0) return -1;
  rows_layout_rs(p, best_rs, xbytes, tab, tmax);
  return p.smem;
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// 5-D byte view of an expert block sequence [E][3 matrices][I rows][rb bytes]
// (a bf16 row, a 4-bit row of nibbles + scales, or the codes of an int8 row):
// (128 bytes, row, matrix, 128-byte chunk, expert), and a box of `rows` rows
// x `mats` matrices x `chunks` chunks of one expert, stored in shared memory
// as [chunk][matrix][row][128 bytes] with the 128-byte swizzle.
bool encode_rows(PFN_cuTensorMapEncodeTiled_v12000 fn, CUtensorMap* m, const void* base, int rb, int chunks, int I,
                 int E, int rows, int mats) {
  if (rb % 16 || chunks * 128 > rb) return false;
  const cuuint64_t dims[5] = {128, (cuuint64_t)I, 3, (cuuint64_t)chunks, (cuuint64_t)E};
  const cuuint64_t strides[4] = {(cuuint64_t)rb, (cuuint64_t)I * rb, 128, (cuuint64_t)3 * I * rb};
  const cuuint32_t box[5] = {128, (cuuint32_t)rows, (cuuint32_t)mats, (cuuint32_t)chunks, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The 16-byte scale records of int8 rows (at byte H of each row): (16 bytes,
// row, matrix, expert, 1), a box of `rows` rows x `mats` matrices stored as
// [matrix][row][16 bytes], unswizzled.
bool encode_scales(PFN_cuTensorMapEncodeTiled_v12000 fn, CUtensorMap* m, const uint8_t* base, int H, int rb, int I,
                   int E, int rows, int mats) {
  const cuuint64_t dims[5] = {16, (cuuint64_t)I, 3, (cuuint64_t)E, 1};
  const cuuint64_t strides[4] = {(cuuint64_t)rb, (cuuint64_t)I * rb, (cuuint64_t)3 * I * rb,
                                 (cuuint64_t)3 * I * rb * E};
  const cuuint32_t box[5] = {16, (cuuint32_t)rows, (cuuint32_t)mats, 1, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<uint8_t*>(base + H), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t rows_tensor_maps(LayerParams& p) {
  if (!rows_fast(p)) return cudaSuccess;
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const int rs = rows_rsm(p.wfmt);
  const int rb = (int)p.rb;
  const int chunks = p.wfmt == kWkI8 ? p.H / 128 : rb / 128;
  if (!encode_rows(fn, &p.tm_gu_e, p.expert_w, rb, chunks, p.I, p.E, rs, 2) ||
      !encode_rows(fn, &p.tm_d_e, p.expert_w, rb, chunks, p.I, p.E, rs, 1) ||
      !encode_rows(fn, &p.tm_gu_s, p.shexp_w, rb, chunks, p.Is, 1, rs, 2) ||
      !encode_rows(fn, &p.tm_d_s, p.shexp_w, rb, chunks, p.Is, 1, rs, 1))
    return cudaErrorInvalidValue;
  if (p.wfmt == kWkI8 &&
      (!encode_scales(fn, &p.tm_gusc_e, p.expert_w, p.H, rb, p.I, p.E, rs, 2) ||
       !encode_scales(fn, &p.tm_dsc_e, p.expert_w, p.H, rb, p.I, p.E, rs, 1) ||
       !encode_scales(fn, &p.tm_gusc_s, p.shexp_w, p.H, rb, p.Is, 1, rs, 2) ||
       !encode_scales(fn, &p.tm_dsc_s, p.shexp_w, p.H, rb, p.Is, 1, rs, 1)))
    return cudaErrorInvalidValue;
  return cudaSuccess;
}

namespace {

__global__ void __launch_bounds__(256) k_join_add(const float* __restrict__ a, const float* __restrict__ b,
                                                  float* __restrict__ out, int n) {
  const int i = blockIdx.x * 256 + threadIdx.x;
  if (i < n) out[i] = __fadd_rn(a[i], b[i]);
}

}  // namespace

cudaError_t launch_join_add(const float* a, const float* b, float* out, int n, cudaStream_t stream) {
  k_join_add<<<(n + 255) / 256, 256, 0, stream>>>(a, b, out, n);
  return cudaGetLastError();
}

cudaError_t launch_rows(const LayerParams& p, cudaStream_t stream) {
  if (!rows_fast(p)) return launch_rows_generic(p, stream);
  switch (p.wfmt) {
    case kWkQ4: return launch_rows_q4_fast(p, stream);
    case kWkI8: return launch_rows_i8_fast(p, stream);
    default: return launch_rows_bf16_fast(p, stream);
  }
}

}  // namespace moe
