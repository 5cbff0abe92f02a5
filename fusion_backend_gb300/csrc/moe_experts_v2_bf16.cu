// Fast-path expert kernel, bf16 weights: instantiations, launch and layout.
#include "moe_experts_v2.cuh"

namespace moe {

int decode_v2_layout(DecodeParams& p, int smem_limit) {
  p.v2 = 0;
  if (p.T > kDecodeMaxT) return -1;
  if (p.H != kV2H) return -1;  // the fast path is specialised for H = 2048
  if (p.I > kV2MaxCols || p.Is > kV2MaxCols) return -1;
  const bool q4 = p.wfmt == 1;
  const bool xreg = p.T == 1;
  const int TK = p.T * p.K;
  const int slot = align_up(std::max(2 * p.rbH, q4 ? 6912 : 8192), 128);
  const int cap_gu = std::min(kMaxGuRows, slot / (2 * p.rbH));
  const int rows_cta = (p.H + p.G - 1) / p.G;
  const int hmodes_bf16[2] = {kHF32, kHBF16};
  const int umax = std::min(p.E, TK);
  for (int nw : {8, 6}) {
    // upper bound of one warp's units (shared, routed, down), which must fit its list
    const long long s_rows = ((p.Is + p.G - 1) / p.G + nw - 1) / nw + 1;
    const long long r_rows = ((long long)umax * p.I / p.G + 2) / nw + 2;
    const long long d_pairs = ((long long)(umax + 1) * rows_cta) / nw + 2;
    const int cap_d = std::max(1, std::min(slot / std::max(p.rbI, p.rbIs), q4 ? 8 : 2));
    const long long bound = s_rows / cap_gu + 1 + r_rows / cap_gu + r_rows / p.I + 2 + d_pairs / cap_d +
                            d_pairs / std::max(1, rows_cta) + 2;
    if (bound > kV2ListLen) continue;
    for (int hi = 0; hi < (q4 ? 1 : 2); ++hi) {
      const int hmode = q4 ? kHH2 : hmodes_bf16[hi];
      const int hel = hmode == kHF32 ? 4 : 2;
      const int xsz = xreg ? 0 : (q4 ? p.T * p.H * 2 : p.T * p.H * 4);
      const int lsz = p.T * p.ls * 4;
      const int hsz = (p.T * p.Is + TK * p.I) * hel;
      const int uni = align_up(std::max(xsz + lsz, hsz), 128);
      const int tab = align_up(v2_tab(nullptr, p.T, p.K, p.E, rows_cta, nullptr), 128);
      int off = 0;
      const int off_bar = off;
      off += align_up((kV2MaxWarps * 4 + 2) * 8, 128);
      const int off_tab = off;
      off += tab;
      const int off_uni = off;
      off += uni;
      const int off_list = align_up(off, 16);
      off = off_list + nw * kV2ListLen * (int)sizeof(V2U);
      off = align_up(off, 1024);
      const int room = smem_limit - off;
      int nslots = room / (nw * slot);
      if (nslots > 4) nslots = 4;
      if (nslots < 2) continue;
      p.v2 = 1;
      p.v2_nw = nw;
      p.v2_nslots = nslots;
      p.v2_slot = slot;
      p.v2_xmode = xreg ? kXReg : (q4 ? kXH2 : kXF32);
      p.v2_hmode = hmode;
      p.v2_rows_w = rows_cta;
      p.v2_cap_gu = cap_gu;
      p.v2_off_bar = off_bar;
      p.v2_off_tab = off_tab;
      p.v2_off_union = off_uni;
      p.v2_union_bytes = uni;
      p.v2_off_list = off_list;
      p.v2_off_ring = off;
      p.v2_smem = off + nslots * nw * slot;
      return p.v2_smem;
    }
  }
  return -1;
}

cudaError_t launch_decode_v2_bf16(const DecodeParams& p, cudaStream_t stream) {
  switch (tmax_for(p.T)) {
    case 1: return launch_v2_t<1, false, true>(p, stream);
    case 2: return launch_v2_t<2, false, false>(p, stream);
    case 4: return launch_v2_t<4, false, false>(p, stream);
    default: return launch_v2_t<8, false, false>(p, stream);
  }
}

cudaError_t launch_decode_v2_q4(const DecodeParams& p, cudaStream_t stream);

cudaError_t launch_decode_v2(const DecodeParams& p, cudaStream_t stream) {
  return p.wfmt == 1 ? launch_decode_v2_q4(p, stream) : launch_decode_v2_bf16(p, stream);
}

}  // namespace moe
