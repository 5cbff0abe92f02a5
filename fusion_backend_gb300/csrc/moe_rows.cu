// Row kernel: choice of instance and shared-memory layout (host side).
#include <algorithm>

#include "moe_rows.cuh"

namespace moe {

cudaError_t launch_rows_bf16_fast(const LayerParams& p, cudaStream_t stream);
cudaError_t launch_rows_q4_fast(const LayerParams& p, cudaStream_t stream);
cudaError_t launch_rows_generic(const LayerParams& p, cudaStream_t stream);

namespace {

// The fast instances: H = 2048, E <= 256, and an activation that bf16 (and
// so fp16) holds exactly -- bf16 x, or the block form whose normalised input
// is bf16 -- kept packed in registers; 4-bit weights form fp16 products.
bool rows_fast(const LayerParams& p) { return p.H == 2048 && p.E <= 256 && (p.act == 1 || p.block_mode); }

int align128(int v) { return (v + 127) & ~127; }

}  // namespace

// Layout with `rs` rows per stage; false when fewer than 3 stages fit.
static bool rows_layout_rs(LayerParams& p, int rs, int xbytes, int tab, int tmax) {
  p.rs = rs;
  p.stage_bytes = (int)(3 * rs * p.rb);
  p.off_bar = 0;
  p.off_tab = 128;
  const int rsm = p.wfmt == 1 ? kRsMaxQ4 : kRsMaxB16;
  p.off_h = align128(p.off_tab + tab);
  p.off_part = align128(p.off_h + 2 * rsm * tmax * 4);
  p.off_x = align128(p.off_part + 2 * kRowWarps * 2 * rsm * tmax * 4);
  p.off_ring = align128(p.off_x + xbytes);
  if (p.off_ring >= kSmemBudget) return false;
  p.ns = std::min(kMaxStagesRing, (kSmemBudget - p.off_ring) / p.stage_bytes);
  // the end-of-kernel column sums reuse the ring: max(threads, T x columns) floats
  const int red_bytes = std::max(kRowThreads, p.T * ((p.H + p.G - 1) / p.G)) * 4;
  if (p.ns < 3 || red_bytes > p.ns * p.stage_bytes) return false;
  p.smem = p.off_ring + p.ns * p.stage_bytes;
  return true;
}

int rows_layout(LayerParams& p) {
  if (p.T < 1 || p.T > kDecodeMaxT || p.H < 8 || p.H > kMaxH || p.G < 1 || p.G > kMaxGrid) return -1;
  const bool q4 = p.wfmt == 1;
  if (q4 ? (p.H % 256) : (p.H % 8)) return -1;
  const bool fast = rows_fast(p);
  const int tmax = fast ? tmax_for(p.T) : 8;
  p.rb = q4 ? (long long)p.H * 9 / 16 : (long long)p.H * 2;
  p.expert_bytes = 3LL * p.I * p.rb;
  p.xmode = fast ? kXReg : kXF32;
  // x region: the bulk copy of the source rows (fp32 for fp32 x and the block
  // form, else bf16), rewritten in place into the compute form
  const bool src4 = p.act == 0 || p.block_mode;
  const int xbytes = p.T * p.H * (p.xmode == kXF32 || src4 ? 4 : 2);
  const int tab = row_tab(nullptr, p.T, p.K, p.E, nullptr);
  // Rows per stage: the choice that keeps the most bytes in flight (all ns
  // stages), with at least 3 stages in the ring; ties go to larger stages.
  const int rs_list[4] = {8, 4, 2, 1};
  int best_rs = 0;
  long long best_flight = -1;
  for (int r = 0; r < 4; ++r) {
    if (rs_list[r] > (q4 ? kRsMaxQ4 : kRsMaxB16)) continue;
    LayerParams t = p;
    if (!rows_layout_rs(t, rs_list[r], xbytes, tab, tmax)) continue;
    const long long flight = (long long)t.ns * t.stage_bytes;
    if (flight > best_flight) {
      best_flight = flight;
      best_rs = rs_list[r];
    }
  }
  if (best_rs == 0) return -1;
  rows_layout_rs(p, best_rs, xbytes, tab, tmax);
  return p.smem;
}

cudaError_t launch_rows(const LayerParams& p, cudaStream_t stream) {
  if (!rows_fast(p)) return launch_rows_generic(p, stream);
  return p.wfmt == 1 ? launch_rows_q4_fast(p, stream) : launch_rows_bf16_fast(p, stream);
}

}  // namespace moe
