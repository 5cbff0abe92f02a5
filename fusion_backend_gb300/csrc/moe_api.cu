// C ABI of the fused MoE FFN layer: plan, validation, workspace layout and
// launches.  See include/moe_ffn.h for the contract.
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <new>

#include "moe_ffn.h"
#include "moe_internal.h"

using namespace moe;

namespace {

constexpr uint32_t kPlanMagic = 0x4D6F4546u;  // "MoEF"
constexpr int kMaxDevices = 64;

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

struct WsLayout {
  size_t ctrl, sync, logits, partial, counts, offsets, perm, active, nactive, total;
  // batched path
  size_t ids, p, bitmap, slot_of, slot_w, x_perm, h_ws, y_ws, lbound;
};

}  // namespace

struct moe_ffn_plan {
  uint32_t magic;
  moe_ffn_shapes s;
  int act, wfmt;
  int path;  // 0 decode (row kernel), 1 batched (grouped GEMMs)
  WsLayout ws;
};

namespace {

struct DeviceInfo {
  std::atomic<int> ready{0};
  int sm_count = 0;
  int smem_optin = 0;
  int major = 0, minor = 0;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

// Device properties are read once per device, lazily on the first execute
// (prepare never touches the device).
int device_info(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_FFN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_FFN_ERR_DEVICE;
  DeviceInfo& d = g_dev[dev];
  if (!d.ready.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(g_dev_mu);
    if (!d.ready.load(std::memory_order_relaxed)) {
      if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return MOE_FFN_ERR_CUDA;
      d.ready.store(1, std::memory_order_release);
    }
  }
  if (d.major != 10 || d.minor != 3) return MOE_FFN_ERR_DEVICE;
  *out = &d;
  return MOE_FFN_OK;
}

thread_local char t_last_cuda_error[256];

// MOE_FFN_OK, or MOE_FFN_ERR_CUDA with the runtime's text kept for
// moe_ffn_last_cuda_error.
int cuda_status(cudaError_t err) {
  if (err == cudaSuccess) return MOE_FFN_OK;
  snprintf(t_last_cuda_error, sizeof(t_last_cuda_error), "%s: %s", cudaGetErrorName(err), cudaGetErrorString(err));
  return MOE_FFN_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool valid_plan(const moe_ffn_plan* p) { return p && p->magic == kPlanMagic; }

void fill_params(const moe_ffn_plan* plan, LayerParams& P, void* ws) {
  memset(&P, 0, sizeof(P));
  const moe_ffn_shapes& s = plan->s;
  P.T = s.T;
  P.H = s.H;
  P.E = s.E;
  P.K = s.top_k;
  P.I = s.I;
  P.Is = s.Is;
  P.act = plan->act;
  P.wfmt = plan->wfmt;
  uint8_t* w = static_cast<uint8_t*>(ws);
  P.ctrl = reinterpret_cast<uint32_t*>(w + plan->ws.ctrl);
  P.sync = reinterpret_cast<RowSync*>(w + plan->ws.sync);
  P.logits = reinterpret_cast<float*>(w + plan->ws.logits);
  P.ls = (s.E + 1 + 3) / 4 * 4;
  P.partial = reinterpret_cast<float*>(w + plan->ws.partial);
  P.r_counts = reinterpret_cast<int32_t*>(w + plan->ws.counts);
  P.r_offsets = reinterpret_cast<int32_t*>(w + plan->ws.offsets);
  P.r_perm = reinterpret_cast<int32_t*>(w + plan->ws.perm);
  P.r_active = reinterpret_cast<int32_t*>(w + plan->ws.active);
  P.r_nactive = reinterpret_cast<int32_t*>(w + plan->ws.nactive);
}

int run(moe_ffn_plan_t plan, moe_ffn_stream_t stream, void* workspace, size_t workspace_bytes, const void* x,
        const void* router_w, const void* expert_w, const void* shexp_w, const void* shexp_gate_w, float* out,
        int32_t* topk_ids, float* topk_w, int block_mode, float eps) {
  if (!valid_plan(plan)) return MOE_FFN_ERR_INVALID_ARG;
  if (!workspace || !x || !router_w || !expert_w || !shexp_w || !shexp_gate_w || !out)
    return MOE_FFN_ERR_INVALID_ARG;
  if (workspace_bytes < plan->ws.total) return MOE_FFN_ERR_WORKSPACE;
  if (!aligned(workspace, 256) || !aligned(x, 16) || !aligned(router_w, 16) || !aligned(expert_w, 16) ||
      !aligned(shexp_w, 16) || !aligned(shexp_gate_w, 16) || !aligned(out, 16) || !aligned(topk_ids, 4) ||
      !aligned(topk_w, 4))
    return MOE_FFN_ERR_MISALIGNED;
  if (block_mode && (plan->act != MOE_FFN_ACT_BF16 || plan->path != 0)) return MOE_FFN_ERR_UNSUPPORTED;
  DeviceInfo* dev = nullptr;
  int rc = device_info(&dev);
  if (rc != MOE_FFN_OK) return rc;

  if (plan->path == 1) {
    const moe_ffn_shapes& s = plan->s;
    uint8_t* w = static_cast<uint8_t*>(workspace);
    const WsLayout& L = plan->ws;
    BatchParams B;
    memset(&B, 0, sizeof(B));
    B.T = s.T;
    B.H = s.H;
    B.E = s.E;
    B.K = s.top_k;
    B.I = s.I;
    B.Is = s.Is;
    B.G = dev->sm_count < kMaxGrid ? dev->sm_count : kMaxGrid;
    B.x = static_cast<const uint16_t*>(x);
    B.router_w = static_cast<const uint16_t*>(router_w);
    B.gate_w = static_cast<const uint16_t*>(shexp_gate_w);
    B.expert_w = static_cast<const uint8_t*>(expert_w);
    B.shexp_w = static_cast<const uint8_t*>(shexp_w);
    B.out = out;
    B.topk_ids = topk_ids;
    B.topk_w = topk_w;
    B.ctrl = reinterpret_cast<uint32_t*>(w + L.ctrl);
    B.logits = reinterpret_cast<float*>(w + L.logits);
    B.ls = (s.E + 1 + 3) / 4 * 4;
    B.lbound = reinterpret_cast<float*>(w + L.lbound);
    B.ids = reinterpret_cast<int32_t*>(w + L.ids);
    B.p = reinterpret_cast<float*>(w + L.p);
    B.bitmap = reinterpret_cast<uint32_t*>(w + L.bitmap);
    B.tw = (s.T + 31) / 32;
    B.slot_of = reinterpret_cast<int32_t*>(w + L.slot_of);
    B.slot_w = reinterpret_cast<float*>(w + L.slot_w);
    B.x_perm = reinterpret_cast<uint16_t*>(w + L.x_perm);
    B.h_ws = reinterpret_cast<uint16_t*>(w + L.h_ws);
    B.hw = s.I > s.Is ? s.I : s.Is;
    B.wfmt = plan->wfmt;
    B.rb = plan->wfmt == MOE_FFN_W_Q4B32 ? (long long)s.H / 2 + s.H / 16 : 2LL * s.H;
    B.y_ws = reinterpret_cast<float*>(w + L.y_ws);
    B.r_counts = reinterpret_cast<int32_t*>(w + L.counts);
    B.r_offsets = reinterpret_cast<int32_t*>(w + L.offsets);
    B.r_perm = reinterpret_cast<int32_t*>(w + L.perm);
    B.r_active = reinterpret_cast<int32_t*>(w + L.active);
    B.r_nactive = reinterpret_cast<int32_t*>(w + L.nactive);
    const int smem0 = B.wfmt == 1 ? kQ4Smem0 : kGemmSmem0, smem1 = B.wfmt == 1 ? kQ4Smem1 : kGemmSmem1;
    if (smem0 + 4608 > dev->smem_optin || smem1 + 4608 > dev->smem_optin) return MOE_FFN_ERR_UNSUPPORTED;
    cudaError_t err = batch_tensor_maps(B);
    if (err != cudaSuccess) return cuda_status(err);
    return cuda_status(launch_batch(B, reinterpret_cast<cudaStream_t>(stream)));
  }

  LayerParams P;
  fill_params(plan, P, workspace);
  P.x = x;
  P.router_w = static_cast<const uint16_t*>(router_w);
  P.gate_w = static_cast<const uint16_t*>(shexp_gate_w);
  P.expert_w = static_cast<const uint8_t*>(expert_w);
  P.shexp_w = static_cast<const uint8_t*>(shexp_w);
  P.out = out;
  P.topk_ids = topk_ids;
  P.topk_w = topk_w;
  P.block_mode = block_mode;
  P.eps = eps;
  P.G = dev->sm_count < kMaxGrid ? dev->sm_count : kMaxGrid;
  if (rows_layout(P) < 0 || P.smem > dev->smem_optin) return MOE_FFN_ERR_UNSUPPORTED;
  cudaError_t err = rows_tensor_maps(P);
  if (err != cudaSuccess) return cuda_status(err);
  err = launch_rows(P, reinterpret_cast<cudaStream_t>(stream));
  return cuda_status(err);
}

// Workspace of the two-stream form: the routed part's and the shared part's
// own workspaces, then their outputs y_r and y_s ([T][H] fp32 each).
size_t two_stream_bytes(const moe_ffn_plan* plan) {
  const size_t y = align256((size_t)plan->s.T * plan->s.H * 4);
  return 2 * plan->ws.total + 2 * y;
}

int run_two_stream(moe_ffn_plan_t plan, cudaStream_t stream, cudaStream_t aux, cudaEvent_t fork, cudaEvent_t join,
                   void* workspace, size_t workspace_bytes, const void* x, const void* router_w,
                   const void* expert_w, const void* shexp_w, const void* shexp_gate_w, float* out) {
  if (!valid_plan(plan)) return MOE_FFN_ERR_INVALID_ARG;
  if (plan->path != 0) return MOE_FFN_ERR_UNSUPPORTED;
  if (!workspace || !x || !router_w || !expert_w || !shexp_w || !shexp_gate_w || !out) return MOE_FFN_ERR_INVALID_ARG;
  if (workspace_bytes < two_stream_bytes(plan)) return MOE_FFN_ERR_WORKSPACE;
  if (!aligned(workspace, 256) || !aligned(x, 16) || !aligned(router_w, 16) || !aligned(expert_w, 16) ||
      !aligned(shexp_w, 16) || !aligned(shexp_gate_w, 16) || !aligned(out, 16))
    return MOE_FFN_ERR_MISALIGNED;
  DeviceInfo* dev = nullptr;
  int rc = device_info(&dev);
  if (rc != MOE_FFN_OK) return rc;
  const moe_ffn_shapes& s = plan->s;
  const int G = dev->sm_count < kMaxGrid ? dev->sm_count : kMaxGrid;
  if (G < 2) return MOE_FFN_ERR_UNSUPPORTED;
  // SMs split by the bytes each branch streams (the routed branch at its
  // largest number of distinct experts), so that both grids are resident at
  // once: every grid waits at grid-wide barriers for all of its blocks.
  const double eb = 3.0 * (plan->wfmt == MOE_FFN_W_Q4B32 ? 9.0 / 16.0 * s.H
                                : plan->wfmt == MOE_FFN_W_I8  ? s.H + 16.0
                                                              : 2.0 * s.H);
  const double b_sh = eb * s.Is, b_r = eb * s.I * (double)(s.E < s.T * s.top_k ? s.E : s.T * s.top_k);
  int Gs = (int)(G * b_sh / (b_sh + b_r) + 0.5);
  Gs = Gs < 1 ? 1 : (Gs > G - 1 ? G - 1 : Gs);
  uint8_t* w = static_cast<uint8_t*>(workspace);
  const size_t y = align256((size_t)s.T * s.H * 4);
  float* y_r = reinterpret_cast<float*>(w + 2 * plan->ws.total);
  float* y_s = reinterpret_cast<float*>(w + 2 * plan->ws.total + y);
  LayerParams P[2];
  for (int part = 1; part <= 2; ++part) {
    LayerParams& L = P[part - 1];
    fill_params(plan, L, w + (part - 1) * plan->ws.total);
    L.x = x;
    L.router_w = static_cast<const uint16_t*>(router_w);
    L.gate_w = static_cast<const uint16_t*>(shexp_gate_w);
    L.expert_w = static_cast<const uint8_t*>(expert_w);
    L.shexp_w = static_cast<const uint8_t*>(shexp_w);
    L.out = part == 1 ? y_r : y_s;
    L.part = part;
    L.G = part == 1 ? G - Gs : Gs;
    if (rows_layout(L) < 0 || L.smem > dev->smem_optin) return MOE_FFN_ERR_UNSUPPORTED;
    cudaError_t err = rows_tensor_maps(L);
    if (err != cudaSuccess) return cuda_status(err);
  }
  const bool two = aux && fork && join && aux != stream;
  cudaError_t err = cudaSuccess;
  if (two) {
    // fork: the shared branch on the aux stream after everything before
    // this call on the main stream; join: the add after both branches
    err = cudaEventRecord(fork, stream);
    if (err == cudaSuccess) err = cudaStreamWaitEvent(aux, fork, 0);
    if (err == cudaSuccess) err = launch_rows(P[0], stream);
    if (err == cudaSuccess) err = launch_rows(P[1], aux);
    if (err == cudaSuccess) err = cudaEventRecord(join, aux);
    if (err == cudaSuccess) err = cudaStreamWaitEvent(stream, join, 0);
  } else {
    err = launch_rows(P[0], stream);
    if (err == cudaSuccess) err = launch_rows(P[1], stream);
  }
  if (err == cudaSuccess) err = launch_join_add(y_r, y_s, out, s.T * s.H, stream);
  return cuda_status(err);
}

}  // namespace

extern "C" {

int moe_ffn_prepare(const moe_ffn_shapes* shapes, moe_ffn_dtype dtype, moe_ffn_plan_t* plan,
                    size_t* workspace_bytes) {
  if (!shapes || !plan || !workspace_bytes) return MOE_FFN_ERR_INVALID_ARG;
  *plan = nullptr;
  const moe_ffn_shapes s = *shapes;
  if (dtype.act != MOE_FFN_ACT_F32 && dtype.act != MOE_FFN_ACT_BF16) return MOE_FFN_ERR_INVALID_ARG;
  if (dtype.wfmt != MOE_FFN_W_BF16 && dtype.wfmt != MOE_FFN_W_Q4B32 && dtype.wfmt != MOE_FFN_W_I8)
    return MOE_FFN_ERR_INVALID_ARG;
  if (s.T < 1 || s.T > kBatchMaxT || s.E < 1 || s.E > kMaxExperts || s.top_k < 1 || s.top_k > s.E ||
      s.top_k > kMaxTopK || s.H < 1 || s.I < 1 || s.Is < 1)
    return MOE_FFN_ERR_UNSUPPORTED;
  if (s.I > (1 << 20) || s.Is > (1 << 20)) return MOE_FFN_ERR_UNSUPPORTED;
  const int path = s.T > kDecodeMaxT ? 1 : 0;
  if (path == 0) {
    // Decode path: T <= 8; stored rows of H elements (bf16: H a multiple of
    // 8, 4-bit: of 256, int8: of 16, so that rows are 16-byte multiples);
    // H <= 4096.
    if (s.H > kMaxH) return MOE_FFN_ERR_UNSUPPORTED;
    if (s.H % (dtype.wfmt == MOE_FFN_W_BF16 ? 8 : dtype.wfmt == MOE_FFN_W_I8 ? 16 : 256))
      return MOE_FFN_ERR_UNSUPPORTED;
  } else {
    // Batched path (grouped GEMMs): bf16 or 4-bit weights, bf16 activation, E <= 256,
    // tiles of 256 columns of H and 128 rows of I and Is.
    if (dtype.act != MOE_FFN_ACT_BF16 || dtype.wfmt == MOE_FFN_W_I8) return MOE_FFN_ERR_UNSUPPORTED;
    if (s.E > kBatchMaxE || s.H % 256 || s.I % 128 || s.Is % 128) return MOE_FFN_ERR_UNSUPPORTED;
    if ((long long)s.E * 3 * s.I >= (1LL << 31) || 3LL * s.Is >= (1LL << 31)) return MOE_FFN_ERR_UNSUPPORTED;
  }

  moe_ffn_plan* p = new (std::nothrow) moe_ffn_plan();
  if (!p) return MOE_FFN_ERR_INVALID_ARG;
  p->magic = kPlanMagic;
  p->s = s;
  p->act = dtype.act;
  p->wfmt = dtype.wfmt;
  p->path = path;
  size_t off = 0;
  WsLayout& L = p->ws;
  const size_t T = s.T, E = s.E, K = s.top_k;
  L.ctrl = off;
  off = align256(off + kCtrlWords * 4);
  L.sync = off;
  if (path == 0) off = align256(off + sizeof(RowSync));
  L.logits = off;
  off = align256(off + T * ((E + 1 + 3) / 4 * 4) * 4);
  L.partial = off;
  // per-block partial outputs: fp32, or (T = 1) 8-byte tagged words
  if (path == 0) off = align256(off + (size_t)kMaxGrid * T * (size_t)s.H * (T == 1 ? 8 : 4));
  if (path == 1) {
    const size_t TK = T * K, H = s.H, hw = s.I > s.Is ? s.I : s.Is;
    L.lbound = off;
    off = align256(off + T * ((E + 1 + 3) / 4 * 4) * 4);
    L.ids = off;
    off = align256(off + TK * 4);
    L.p = off;
    off = align256(off + TK * 4);
    L.bitmap = off;
    off = align256(off + E * ((T + 31) / 32) * 4);
    L.slot_of = off;
    off = align256(off + TK * 4);
    L.slot_w = off;
    off = align256(off + (TK + T) * 4);
    L.x_perm = off;
    off = align256(off + (dtype.wfmt == MOE_FFN_W_Q4B32 ? TK + T : TK) * H * 2);
    L.h_ws = off;
    off = align256(off + (TK + T) * hw * 2 * (dtype.wfmt == MOE_FFN_W_Q4B32 ? 1 : 2));
    L.y_ws = off;
    off = align256(off + (TK + T) * H * 4);
  }
  L.counts = off;
  off = align256(off + E * 4);
  L.offsets = off;
  off = align256(off + (E + 1) * 4);
  L.perm = off;
  off = align256(off + T * K * 4);
  L.active = off;
  off = align256(off + E * 4);
  L.nactive = off;
  off = align256(off + 4);
  L.total = off;
  *plan = p;
  *workspace_bytes = off;
  return MOE_FFN_OK;
}

int moe_ffn_execute(moe_ffn_plan_t plan, moe_ffn_stream_t stream, void* workspace, size_t workspace_bytes,
                    const void* x, const void* router_w, const void* expert_w, const void* shexp_w,
                    const void* shexp_gate_w, float* out) {
  return run(plan, stream, workspace, workspace_bytes, x, router_w, expert_w, shexp_w, shexp_gate_w, out, nullptr,
             nullptr, 0, 0.f);
}

int moe_ffn_execute_ex(moe_ffn_plan_t plan, moe_ffn_stream_t stream, void* workspace, size_t workspace_bytes,
                       const void* x, const void* router_w, const void* expert_w, const void* shexp_w,
                       const void* shexp_gate_w, float* out, int32_t* topk_ids, float* topk_w) {
  return run(plan, stream, workspace, workspace_bytes, x, router_w, expert_w, shexp_w, shexp_gate_w, out, topk_ids,
             topk_w, 0, 0.f);
}

int moe_ffn_execute_block(moe_ffn_plan_t plan, moe_ffn_stream_t stream, void* workspace, size_t workspace_bytes,
                          float* x_res, const void* router_w, const void* expert_w, const void* shexp_w,
                          const void* shexp_gate_w, float eps, int32_t* topk_ids, float* topk_w) {
  if (!(eps >= 0.f)) return MOE_FFN_ERR_INVALID_ARG;
  return run(plan, stream, workspace, workspace_bytes, x_res, router_w, expert_w, shexp_w, shexp_gate_w, x_res,
             topk_ids, topk_w, 1, eps);
}

int moe_ffn_read_status(moe_ffn_plan_t plan, const void* workspace, moe_ffn_stream_t stream,
                        int32_t* device_status) {
  if (!valid_plan(plan) || !workspace || !device_status) return MOE_FFN_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_FFN_ERR_CUDA;
  const uint8_t* w = static_cast<const uint8_t*>(workspace);
  int32_t status = 0;
  if (cudaMemcpy(&status, w + plan->ws.ctrl + kCtrlStatus * 4, 4, cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_FFN_ERR_CUDA;
  if (status == 0 && plan->path == 0) {
    // decode path: each block of the row kernel writes its own status slot
    int32_t slots[kMaxGrid];
    if (cudaMemcpy(slots, w + plan->ws.sync + offsetof(RowSync, status), sizeof(slots), cudaMemcpyDeviceToHost) !=
        cudaSuccess)
      return MOE_FFN_ERR_CUDA;
    for (int i = 0; i < kMaxGrid && status == 0; ++i) status = slots[i];
  }
  *device_status = status;
  return MOE_FFN_OK;
}

int moe_ffn_read_routing(moe_ffn_plan_t plan, const void* workspace, moe_ffn_stream_t stream, int32_t* counts,
                         int32_t* offsets, int32_t* perm, int32_t* active, int32_t* num_active) {
  if (!valid_plan(plan) || !workspace || !counts || !offsets || !perm || !active || !num_active)
    return MOE_FFN_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_FFN_ERR_CUDA;
  const uint8_t* w = static_cast<const uint8_t*>(workspace);
  const size_t E = plan->s.E, TK = (size_t)plan->s.T * plan->s.top_k;
  int32_t n = 0;
  if (cudaMemcpy(&n, w + plan->ws.nactive, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_FFN_ERR_CUDA;
  if (n < 0 || (size_t)n > E) n = 0;
  if (cudaMemcpy(counts, w + plan->ws.counts, E * 4, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(offsets, w + plan->ws.offsets, (E + 1) * 4, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(perm, w + plan->ws.perm, TK * 4, cudaMemcpyDeviceToHost) != cudaSuccess ||
      (n > 0 && cudaMemcpy(active, w + plan->ws.active, (size_t)n * 4, cudaMemcpyDeviceToHost) != cudaSuccess))
    return MOE_FFN_ERR_CUDA;
  *num_active = n;
  return MOE_FFN_OK;
}

int moe_ffn_probe_timeout(moe_ffn_plan_t plan, moe_ffn_stream_t stream, void* workspace, size_t workspace_bytes,
                          int32_t which) {
  if (!valid_plan(plan) || !workspace || which < 0 || which > 2) return MOE_FFN_ERR_INVALID_ARG;
  if (workspace_bytes < plan->ws.total) return MOE_FFN_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return MOE_FFN_ERR_MISALIGNED;
  DeviceInfo* dev = nullptr;
  const int rc = device_info(&dev);
  if (rc != MOE_FFN_OK) return rc;
  uint32_t* ctrl = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(workspace) + plan->ws.ctrl);
  return cuda_status(launch_probe_timeout(ctrl, which, reinterpret_cast<cudaStream_t>(stream)));
}

int moe_ffn_query(moe_ffn_plan_t plan, int32_t what, int64_t* value) {
  if (!valid_plan(plan) || !value) return MOE_FFN_ERR_INVALID_ARG;
  switch (what) {
    case MOE_FFN_QUERY_PATH:
      *value = plan->path;
      return MOE_FFN_OK;
    case MOE_FFN_QUERY_LAUNCHES_PER_EXECUTE:
      *value = plan->path == 1 ? kBatchLaunches : kLaunchesPerExecute;
      return MOE_FFN_OK;
    case MOE_FFN_QUERY_TWO_STREAM_WORKSPACE:
      if (plan->path != 0) return MOE_FFN_ERR_UNSUPPORTED;
      *value = (int64_t)two_stream_bytes(plan);
      return MOE_FFN_OK;
    default:
      return MOE_FFN_ERR_INVALID_ARG;
  }
}

int moe_ffn_execute_two_stream(moe_ffn_plan_t plan, moe_ffn_stream_t stream, moe_ffn_stream_t aux_stream,
                               moe_ffn_event_t fork_event, moe_ffn_event_t join_event, void* workspace,
                               size_t workspace_bytes, const void* x, const void* router_w, const void* expert_w,
                               const void* shexp_w, const void* shexp_gate_w, float* out) {
  return run_two_stream(plan, reinterpret_cast<cudaStream_t>(stream), reinterpret_cast<cudaStream_t>(aux_stream),
                        reinterpret_cast<cudaEvent_t>(fork_event), reinterpret_cast<cudaEvent_t>(join_event),
                        workspace, workspace_bytes, x, router_w, expert_w, shexp_w, shexp_gate_w, out);
}

void moe_ffn_destroy(moe_ffn_plan_t plan) {
  if (!valid_plan(plan)) return;
  plan->magic = 0;
  delete plan;
}

const char* moe_ffn_last_cuda_error(void) { return t_last_cuda_error; }

const char* moe_ffn_strerror(int status) {
  switch (status) {
    case MOE_FFN_OK: return "ok";
    case MOE_FFN_ERR_INVALID_ARG: return "invalid argument";
    case MOE_FFN_ERR_UNSUPPORTED: return "unsupported shapes or dtype";
    case MOE_FFN_ERR_WORKSPACE: return "workspace too small";
    case MOE_FFN_ERR_MISALIGNED: return "misaligned pointer";
    case MOE_FFN_ERR_CUDA: return "CUDA error";
    case MOE_FFN_ERR_TIMEOUT: return "in-kernel wait timed out";
    case MOE_FFN_ERR_DEVICE: return "unsupported device (needs sm_103)";
    default: return "unknown status";
  }
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free entry point: the scratch lives in a file-scope device array
// instead of a caller-provided workspace (see moe_ffn.h).
namespace {

// Scratch of moe_ffn_execute_static_scratch, shared by every call on a device.
// Every GPU that loads this library holds these bytes until the process exits.
__device__ __align__(256) uint8_t g_static_scratch[MOE_FFN_STATIC_SCRATCH_BYTES];

std::atomic<void*> g_static_scratch_addr[kMaxDevices];
std::mutex g_static_scratch_mu;

// Device address of g_static_scratch on the current device, looked up once per
// device with that device current (the host-side symbol is only a stand-in for
// it).  Later calls read the cached address without taking the lock.
int static_scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_FFN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_FFN_ERR_DEVICE;
  void* p = g_static_scratch_addr[dev].load(std::memory_order_acquire);
  if (!p) {
    std::lock_guard<std::mutex> lock(g_static_scratch_mu);
    p = g_static_scratch_addr[dev].load(std::memory_order_relaxed);
    if (!p) {
      cudaError_t err = cudaGetSymbolAddress(&p, g_static_scratch);
      if (err != cudaSuccess || !p) return cuda_status(err != cudaSuccess ? err : cudaErrorInvalidSymbol);
      g_static_scratch_addr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return MOE_FFN_OK;
}

}  // namespace

extern "C" int moe_ffn_execute_static_scratch(moe_ffn_plan_t plan, moe_ffn_stream_t stream, const void* x,
                                              const void* router_w, const void* expert_w, const void* shexp_w,
                                              const void* shexp_gate_w, float* out) {
  if (!valid_plan(plan)) return MOE_FFN_ERR_INVALID_ARG;
  if (plan->ws.total > (size_t)MOE_FFN_STATIC_SCRATCH_BYTES) return MOE_FFN_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int rc = static_scratch_address(&scratch);
  if (rc != MOE_FFN_OK) return rc;
  // The kernels initialise on each call every word of the workspace that they
  // count on (see RowSync and the batched path's router kernel), so no part
  // of the (shared, reused) array has to be cleared here.
  return run(plan, stream, scratch, MOE_FFN_STATIC_SCRATCH_BYTES, x, router_w, expert_w, shexp_w, shexp_gate_w, out,
             nullptr, nullptr, 0, 0.f);
}
