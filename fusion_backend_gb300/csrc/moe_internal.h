// Internal host/device interface between the C ABI (moe_api.cu) and the
// kernels.  Not installed; the public interface is include/moe_ffn.h.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

constexpr int kDecodeMaxT = 8;    // tokens of the decode path
constexpr int kMaxTopK = 32;
constexpr int kMaxExperts = 1024;
constexpr int kRowWarps = 8;      // warps of the row kernel
constexpr int kRowThreads = kRowWarps * 32;
constexpr int kRouteThreads = 128;
constexpr int kMaxH = 4096;       // H of the decode path (bf16: multiple of 8, 4-bit: of 256)
constexpr int kSmemBudget = 220 * 1024;  // row kernel: leaves room for a router block on the SM
constexpr int kMaxGrid = 192;            // row kernel blocks (one per SM, at most this many)
constexpr int kStatusTimeout = -6;       // device status word: a bounded wait gave up
constexpr int kXPitch = 4160;            // tensor-core loops: bytes per token row of x fragments (4 KB + 64)

// Control words at the start of the workspace.  The batched path's router
// kernel zeroes them on each call before its later kernels use them; the
// decode row kernel clears the status word on each call.
enum : int { kCtrlStatus = 0, kCtrlProbe = 2, kCtrlWords = 64 };

// Decode row kernel: its grid-wide synchronisation words (in the workspace,
// after the control words).  The call's epoch e is one more than the value in
// `epoch`, which every block reads after the wait on the previous kernel.  A
// barrier: block c stores e into its own slot of a flag array (release);
// block 0 waits until every slot holds e, then stores e into the barrier's
// `go` word (release); every block waits until `go` holds e.  Nothing has to
// be reset between calls: each call overwrites every word it waits on with a
// value no earlier call stored (the previous call stored e - 1).  Block 0
// advances `epoch` once all blocks have read it (in the first barrier, after
// it has seen every slot).  Each block also writes its own status slot (0 or
// the timeout status) on every call.
//
// Fast path: once a call has run to its first barrier on this workspace, the
// two arrival counters of the next call (count[e + 1 parity]) are zero --
// block 0 clears them after that barrier, when no block of this call can
// touch them -- and `sig` holds ~e.  A call that finds sig == ~epoch uses the
// counters (each block adds one; a barrier is complete at G), one hop through
// L2 instead of two; any other state (a workspace that another user
// overwrote, or never initialised) takes the flag barrier, which needs no
// prior state.  Both decisions are the same in every block: they read
// `epoch` and `sig` before any block can change them.
//
// With one token the second barrier is not used: each partial output is a word
// tagged with the call (the low half of e above the fp32 value).  Each block
// first marks its own partial words with another tag, before the first
// barrier, which publishes the marks; a reader then polls the words it needs
// until each carries the call's tag -- it can see only the mark or the value.
struct RowSync {
  unsigned long long epoch;
  unsigned long long sig;
  unsigned long long go[2];  // the two barriers' release words
  uint32_t count[2][2];      // [call parity][barrier] arrival counters of the fast path
  unsigned long long pad[10];
  unsigned long long logits_ready[kMaxGrid];   // first barrier: the block's router logits are written
  unsigned long long partial_ready[kMaxGrid];  // second barrier: the block's partial output is written
  int32_t status[kMaxGrid];
};

struct LayerParams {
  // shapes
  int T, H, E, K, I, Is;
  int act;   // 0 fp32 x, 1 bf16 x
  int wfmt;  // 0 bf16 weights, 1 4-bit blocks, 2 int8 rows (int8 activation)
  int block_mode;
  float eps;
  int G;  // grid of the row kernel
  // 0: the whole layer; 1: the routed experts only, out = sum_j p_j FFN_j(x)
  // (ffn_moe_out); 2: the gated shared expert only, out = s FFN_shared(x)
  // (ffn_shexp).  Parts 1 and 2 are the two branches of the two-stream form.
  int part;

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
  RowSync* sync;
  float* logits;   // [T][ls]: columns 0..E-1 router logits, column E the shared-gate logit
  int ls;          // logits row stride in floats: E + 1 rounded up to a multiple of 4
  float* partial;  // [G][T][H] per-block partial outputs: fp32, or (T = 1) 8-byte tagged words
  int32_t* r_counts;
  int32_t* r_offsets;
  int32_t* r_perm;
  int32_t* r_active;
  int32_t* r_nactive;

  // weight layout (bytes)
  long long rb;            // one stored row (H elements)
  long long expert_bytes;  // one routed expert block: 3 * I * rb

  // shared-memory layout of the row kernel (bytes from the dynamic base)
  int rs;           // rows per stage
  int ns;           // stages in the ring (tensor-core path: gate + up boxes)
  int nsd;          // tensor-core path: downT boxes in their own ring
  int rp;           // row pitch in a ring slot (rb)
  int stage_bytes;  // 3 * rs * rb (tensor-core path: one gate + up slot)
  int dstage_bytes; // tensor-core path: one downT slot
  int xmode;        // 0 x in registers (each thread its 8 columns), 1 fp32 rows in shared memory
  int off_bar, off_x, off_tab, off_h, off_part, off_ring, off_dring, smem;

  // Tensor maps of the tensor-core path (H = 2048): boxes of one stage's
  // gate + up rows (gu) and downT rows (d) of the routed experts (e) and of
  // the shared expert (s), 128-byte swizzled in shared memory.  Int8
  // weights: the boxes hold the codes, and the sc maps the rows' 16-byte
  // scale records.
  CUtensorMap tm_gu_e;
  CUtensorMap tm_d_e;
  CUtensorMap tm_gu_s;
  CUtensorMap tm_d_s;
  CUtensorMap tm_gusc_e;
  CUtensorMap tm_dsc_e;
  CUtensorMap tm_gusc_s;
  CUtensorMap tm_dsc_s;
};

// ---- batched path (T > kDecodeMaxT): routing, a gather of x by expert, two
// grouped GEMMs on the tcgen05 tensor cores and a fixed-order combine.
constexpr int kBatchMaxT = 1024;
constexpr int kBatchMaxE = 256;
constexpr int kGemmNC = 64;       // slots (tokens) per GEMM unit: the MMA N, at most
constexpr int kGemmThreads = 192; // warp 0 TMA producer, warp 1 MMA issuer, warps 2..5 epilogue

struct BatchParams {
  int T, H, E, K, I, Is, G;
  const uint16_t* x;         // [T][H] bf16
  const uint16_t* router_w;  // [E][H]
  const uint16_t* gate_w;    // [H] shared-expert gate vector
  const uint8_t* expert_w;   // E x (gate[I][H] | up[I][H] | downT[I][H]) bf16
  const uint8_t* shexp_w;    // gate[Is][H] | up[Is][H] | downT[Is][H] bf16
  float* out;                // [T][H]
  int32_t* topk_ids;         // optional [T][K]
  float* topk_w;             // optional [T][K]
  // workspace
  uint32_t* ctrl;
  float* logits;  // [T][ls] fp32 logits (plain sums)
  float* lbound;  // norms for the logit error bound: [0, ls) router rows' |w|_2, [ls, ls + T) tokens' |x|_2 (rounded up)
  int ls;
  int32_t* ids;       // [T][K] chosen experts, rank order
  float* p;           // [T][K] their weights
  uint32_t* bitmap;   // [E][tw] tokens of each expert
  int tw;             // bitmap words per expert: ceil(T / 32)
  int32_t* slot_of;   // [T][K] slot (row of the expert-sorted order) of each choice
  float* slot_w;      // [T K + T] weight of each slot (routed p, then the shared gate per token)
  uint16_t* x_perm;   // [T K][H] bf16, x of each routed slot (4-bit weights: [T K + T][H] fp16)
  uint16_t* h_ws;     // h of each slot (weight applied): bf16 weights [T K + T][2 hw], the bf16 hi part in
                      // columns [0, hw) and the bf16 lo part (h - hi) in [hw, 2 hw); 4-bit [T K + T][hw] fp16
  int hw;             // h values per slot: max(I, Is)
  float* y_ws;        // [T K + T][H] fp32, expert output of each slot
  int32_t* r_counts;  // [E]
  int32_t* r_offsets; // [E + 1]
  int32_t* r_perm;    // [T K] token-major choice index of each slot
  int32_t* r_active;  // [E] active experts ascending
  int32_t* r_nactive; // [1]
  int wfmt;           // 0 bf16 weights, 1 4-bit blocks (then x_perm, h_ws hold fp16)
  long long rb;       // bytes of one stored weight row (2H, or 9H/16)
  // 4-bit weights: byte views [rows][rb] of the expert and shared blocks with
  // boxes of 128 nibble bytes x 64 rows (128-byte swizzle) and 16 scale bytes
  // x 64 rows
  CUtensorMap tm_qn_e;
  CUtensorMap tm_qs_e;
  CUtensorMap tm_qn_s;
  CUtensorMap tm_qs_s;
  // Tensor maps (bf16, 128-byte swizzle): weight rows of the expert blocks
  // and of the shared block with boxes of 64 x 64 (gate / up half tiles and
  // downT tiles), and the B operands: x_perm, x, h_ws rows with boxes of
  // 64 x 16.
  CUtensorMap tm_w64_e;
  CUtensorMap tm_w64_s;
  CUtensorMap tm_xp;
  CUtensorMap tm_x;
  CUtensorMap tm_h;
};
// Encodes the tensor maps; cudaSuccess or an error.
cudaError_t batch_tensor_maps(BatchParams& p);
// Enqueues the whole batched layer (kBatchLaunches kernels).
cudaError_t launch_batch(const BatchParams& p, cudaStream_t stream);
constexpr int kBatchLaunches = 6;
// Ring depth and stage bytes of the GEMM kernels: gate / up stages hold
// kGemmKSub0 pairs of a 128 x 64 A tile (64 gate rows over 64 up rows) and
// an NC x 64 B tile;
// down stages two 128 x 64 A tiles (MN-major) and two NC x 64 B tiles (the
// bf16 hi and lo parts of h).
constexpr int kGemmKSub0 = 2;  // gate / up: 64-wide K sub-chunks per stage (256 bytes of each weight row)
constexpr int kGemmStages0 = 4, kGemmStageBytes0 = kGemmKSub0 * (128 * 128 + kGemmNC * 128);
constexpr int kGemmStages1 = 4, kGemmStageBytes1 = 2 * 128 * 128 + 2 * kGemmNC * 128;
constexpr int kGemmExch = 64 * kGemmNC * 4;  // gate / up epilogue: the gate half of the accumulator
constexpr int kGemmSmem0 = kGemmStages0 * kGemmStageBytes0 + kGemmExch + 1024 + 256;
constexpr int kGemmSmem1 = kGemmStages1 * kGemmStageBytes1 + 1024 + 256;
// 4-bit grouped GEMMs (moe_gemm_q4.cu).  Three rings: raw stages (codes
// with the 128-byte swizzle + scales, from TMA), B stages (the slots' fp16
// rows, from TMA) and A stages (dequantised weights).
// gate / up: raw stage = 64 gate + 64 up rows x 256 K (codes 2 x 8 KB,
// scales 2 x 1 KB); B stage = four 64-wide K sub-chunks (4 x NC x 128
// bytes); A stages in tensor memory (128 K, 64 columns each, two per raw
// stage) behind the accumulators: 2 buffers x 2 K-half parities x 64 columns.  down: raw stage = 64 downT rows x 256 columns
// (8 KB + 1 KB); B stage = NC x 128 bytes; A stages in shared memory (64 K x
// 256 M fp16, K-major); accumulators: 2 buffers x 2 K-stage parities x 128
// columns.
constexpr int kQ4Threads = 480;  // producer, 2 MMA issuers (warps 1, 14), 8 dequant warps, 4 epilogue warps
constexpr int kQ4Dequant = 128;  // dequant threads per stage (two groups of four warps take alternate stages)
constexpr int kQ4Raw0 = 2 * 64 * 128 + 2 * 64 * 16, kQ4RawStages0 = 6;  // 18432
constexpr int kQ4B0 = 4 * kGemmNC * 128, kQ4BStages0 = 3;
constexpr int kQ4AStages0 = 4, kQ4ACol0 = 256, kQ4TmemCols0 = 512;
constexpr int kQ4Raw1 = 64 * 128 + 64 * 16, kQ4RawStages1 = 8;  // 9216
constexpr int kQ4B1 = kGemmNC * 128, kQ4BStages1 = 6;
constexpr int kQ4Tile1 = 64 * 256 * 2, kQ4TileStages1 = 3, kQ4TmemCols1 = 512;
constexpr int kQ4Smem0 = kQ4BStages0 * kQ4B0 + kQ4RawStages0 * kQ4Raw0 + kGemmExch + 1024 + 512;
constexpr int kQ4Smem1 = kQ4TileStages1 * kQ4Tile1 + kQ4BStages1 * kQ4B1 + kQ4RawStages1 * kQ4Raw1 + 1024 + 512;
static_assert(kQ4ACol0 + 64 * kQ4AStages0 <= kQ4TmemCols0 && 4 * kGemmNC <= kQ4ACol0 && kQ4AStages0 % 2 == 0,
              "tensor memory, gate / up");
static_assert(kQ4Smem0 + 4608 <= 232448 && kQ4Smem1 + 4608 <= 232448, "shared memory of the 4-bit GEMMs");
static_assert(kQ4Raw0 % 1024 == 0 && kQ4B0 % 1024 == 0 && kQ4Raw1 % 1024 == 0 && kQ4B1 % 1024 == 0,
              "swizzled stage alignment");

// The failure-path probe (moe_probe.cu): one warp waits, bounded, on an
// mbarrier phase that never completes (which = 0) or on a grid-barrier flag
// slot that never receives its epoch (which = 1), then records the timeout.
cudaError_t launch_probe_timeout(uint32_t* ctrl, int which, cudaStream_t stream);

// Row kernel (moe_rows_*.cu).  rows_layout fills the layout fields and
// returns the dynamic shared-memory bytes, or -1 when the shapes do not fit.
int rows_layout(LayerParams& p);
// Encodes the tensor maps when the launch takes the tensor-core path;
// cudaSuccess or an error.
cudaError_t rows_tensor_maps(LayerParams& p);
cudaError_t launch_rows(const LayerParams& p, cudaStream_t stream);
constexpr int kLaunchesPerExecute = 1;
// out[i] = a[i] + b[i], i < n: the join add(ffn_moe_out, ffn_shexp) of the
// two-stream form (moe_rows.cu).
cudaError_t launch_join_add(const float* a, const float* b, float* out, int n, cudaStream_t stream);

}  // namespace moe
