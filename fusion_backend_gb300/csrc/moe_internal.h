// Internal host/device interface between the C ABI (moe_api.cu) and the
// kernels.  Not installed; the public interface is include/moe_ffn.h.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

constexpr int kNumConsumerWarps = 8;                         // compute warps per CTA
constexpr int kDecodeThreads = (kNumConsumerWarps + 2) * 32;  // + weight producer + h producer
constexpr int kSegCols = 256;                                // columns per warp unit (32 lanes x 8)
constexpr int kStageBytes = 32 * 1024;                       // weight ring stage
constexpr int kMaxGuRows = 16;                               // gate/up row pairs per ring item
constexpr int kMaxDownRows = 32;                             // down rows per ring item
constexpr int kDecodeMaxT = 8;                               // decode path: T <= 8
constexpr int kMaxTopK = 32;
constexpr int kMaxExperts = 1024;
constexpr int kRouteThreads = 256;

// Control words at the start of the workspace.
enum : int { kCtrlStatus = 0, kCtrlHDone = 1, kCtrlWords = 64 };

struct DecodeParams {
  // shapes
  int T, H, E, K, I, Is;
  int act;   // 0 fp32 x, 1 bf16 x
  int wfmt;  // 0 bf16 weights, 1 4-bit blocks
  int block_mode;
  float eps;
  int G;  // grid of the expert kernel

  // caller tensors
  const void* x;  // [T,H] (block mode: fp32 x_res)
  const uint16_t* router_w;
  const uint16_t* gate_w;
  const uint8_t* expert_w;
  const uint8_t* shexp_w;
  float* out;
  int32_t* topk_ids;  // optional
  float* topk_w;      // optional

  // workspace
  uint32_t* ctrl;
  float* logits;  // [T][ls], columns 0..E-1 router logits, column E the shared-gate logit
  int ls;         // logits row stride in floats: E + 1 rounded up to a multiple of 4
  float* h;       // [T*K][I]
  float* hsh;     // [T][Is]
  int32_t* r_counts;
  int32_t* r_offsets;
  int32_t* r_perm;
  int32_t* r_active;
  int32_t* r_nactive;

  // weight layout (bytes)
  long long expert_bytes;  // one routed expert block
  long long gu_bytes;      // one routed gate (or up) matrix [I,H]
  long long sgu_bytes;     // shared gate (or up) matrix [Is,H]
  int rbH, rbI, rbIs;      // bytes of one row with H / I / Is columns

  // shared-memory layout of the general expert kernel (bytes from the dynamic base)
  int nst, nhs, hslot_bytes;
  int off_stage, off_hslot, off_red, red_floats, off_ys, ys_rows_max, off_logits, off_tab, off_bar;
  int smem_bytes;

  // layout of the per-warp-ring expert kernel (fast path)
  int v2;           // 1 when the fast path is launched
  int v2_nw;        // consumer warps
  int v2_nslots;    // ring slots per warp
  int v2_slot;      // bytes per slot
  int v2_xmode;     // 0 x in registers (T=1), 1 x fp32 in smem, 2 x fp16 (4-bit layout) in smem
  int v2_hmode;     // 0 h fp32 in smem, 1 h bf16, 2 h fp16 (4-bit layout)
  int v2_rows_w;    // max output rows per CTA (stride of the down outputs)
  int v2_cap_gu;    // gate/up row pairs per slot
  int v2_off_bar, v2_off_ring, v2_off_tab, v2_off_union, v2_union_bytes, v2_off_list, v2_smem;
};

// Router kernel (moe_route.cu); pdl = launch behind the previous kernel with
// programmatic stream serialisation.
cudaError_t launch_route(const DecodeParams& p, cudaStream_t stream, bool pdl);

// Launchers (moe_decode.cu).  Return cudaSuccess or the launch error.
cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream, bool use_pdl);
// Shared-memory bytes the expert kernel needs for these shapes; fills the
// layout fields of p.  Returns -1 when the shapes do not fit.
int decode_smem_layout(DecodeParams& p, int smem_optin_limit);
int decode_kernel_count();

// Per-warp-ring fast path (moe_decode_v2.cu): fills the v2 layout fields and
// returns the shared-memory bytes, or -1 when these shapes need the general
// kernel.
int decode_v2_layout(DecodeParams& p, int smem_optin_limit);
cudaError_t launch_decode_v2(const DecodeParams& p, cudaStream_t stream);

}  // namespace moe
