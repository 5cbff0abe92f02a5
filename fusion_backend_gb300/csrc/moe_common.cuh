// Device helpers shared by the kernels of the fused MoE FFN layer (sm_103a).
// Inline PTX for mbarriers, bulk async copies (TMA engine, 1-D form),
// programmatic dependent launch and scoped atomics.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#define MOE_DEV __device__ __forceinline__

namespace moe {

// Bound for every spin-wait in these kernels: iterations of a polling loop
// that sleeps between polls.  Far above any legitimate wait (~0.5 s).
constexpr uint32_t kSpinLimit = 1u << 22;
// mbarrier waits: a wall-clock bound (the global nanosecond timer), since one
// try_wait may itself suspend the thread for microseconds; plus an iteration
// cap in case the timer did not advance.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

MOE_DEV unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t)::"memory");
  return t;
}

MOE_DEV uint32_t smem_u32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

// ---------------------------------------------------------------- mbarrier
MOE_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
MOE_DEV void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
MOE_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
MOE_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
MOE_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase with the given parity to complete.  Returns
// false when the bound ran out (the caller records an error and carries on
// without blocking again).
MOE_DEV bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t i = 1; i < kSpinLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 31) == 0 && global_ns() - t0 > kWaitLimitNs) return false;
    if (i > 64) __nanosleep(32);
  }
  return false;
}

// ------------------------------------------------------- bulk async copies
// Global -> this CTA's shared memory, completion counted on `bar` in bytes.
// dst, src 16-byte aligned; bytes a multiple of 16.
MOE_DEV void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
// Tiled tensor copy (TMA engine) of one box of the 5-D tensor map `tmap`
// (a __grid_constant__ kernel parameter) at coordinates c0..c4 into this
// CTA's shared memory, completion counted on `bar` in bytes.
MOE_DEV void tma_load_5d(void* dst, const void* tmap, int c0, int c1, int c2, int c3, int c4, uint64_t* bar,
                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(smem_u32(bar)),
      "l"(policy)
      : "memory");
}
// Pulls a tensor map (a kernel parameter) into the descriptor cache ahead of
// its first tensor copy.
MOE_DEV void prefetch_tensormap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}
// Bulk prefetch of [src, src + bytes) into L2 (hint only; src 16-byte aligned,
// bytes a multiple of 16).
MOE_DEV void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
MOE_DEV uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
MOE_DEV uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// Order this thread's earlier generic-proxy global accesses (and the ones it
// acquired) before its later async-proxy (bulk copy) accesses.
MOE_DEV void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
// The same for all state spaces (global and shared).
MOE_DEV void fence_proxy_async() { asm volatile("fence.proxy.async;" ::: "memory"); }

// -------------------------------------------- programmatic dependent launch
MOE_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
MOE_DEV void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------- scoped atomics
MOE_DEV uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
MOE_DEV void red_release_gpu_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
MOE_DEV unsigned long long ld_relaxed_gpu_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
MOE_DEV void st_release_gpu_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
// Two consecutive 8-byte words (16-byte aligned) with an L2 policy
// (createpolicy); each word is written whole, the pair is not one access.
MOE_DEV void st_relaxed_gpu_v2_u64(unsigned long long* p, unsigned long long a, unsigned long long b, uint64_t pol) {
  asm volatile("st.relaxed.gpu.global.L2::cache_hint.v2.u64 [%0], {%1, %2}, %3;" ::"l"(p), "l"(a), "l"(b), "l"(pol)
               : "memory");
}

// ------------------------------------------------------- tagged words
// A value published to other blocks together with the call that wrote it:
// the upper half of a 64-bit word is the call's tag, the lower half the
// fp32 value.  A reader polls the word until the tag is its own call's, so
// the value arrives with its own "ready" flag (one trip through L2 instead
// of a barrier and then the data).
MOE_DEV unsigned long long tagged(uint32_t tag, float v) {
  return ((unsigned long long)tag << 32) | __float_as_uint(v);
}
MOE_DEV uint32_t tag_of_word(unsigned long long w) { return (uint32_t)(w >> 32); }
MOE_DEV float value_of_word(unsigned long long w) { return __uint_as_float((uint32_t)w); }
// With relaxed loads that observed other threads' release stores before it,
// this fence makes the loads an acquire: later accesses see what those
// threads wrote before their releases.
MOE_DEV void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// ------------------------------------------------------- named barriers
MOE_DEV void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// OR of v over the nthreads threads that meet at barrier id (all of them
// execute this call).
MOE_DEV bool named_bar_or(uint32_t id, uint32_t nthreads, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(v ? 1u : 0u), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}
// Block-level barrier of the threads that run a kernel's whole path: every
// thread of the block (NT == 0: barrier 0), or the first NT threads on
// barrier kBarMain when the block has more threads with a role of their own.
constexpr uint32_t kBarMain = 2;
template <int NT>
MOE_DEV void blk_sync() {
  if constexpr (NT == 0)
    __syncthreads();
  else
    named_bar_sync(kBarMain, NT);
}
template <int NT>
MOE_DEV bool blk_sync_or(bool v) {
  if constexpr (NT == 0)
    return __syncthreads_or(v) != 0;
  else
    return named_bar_or(kBarMain, NT, v);
}

// ------------------------------------------------------- conversions
MOE_DEV float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
MOE_DEV float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
MOE_DEV float bf16_to_float(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }

// Float -> bf16 bits, round to nearest even (finite inputs; NaN stays NaN).
MOE_DEV uint16_t float_to_bf16_rne(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return static_cast<uint16_t>((u >> 16) | 0x40u);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

// Monotone map float -> uint32 (larger float -> larger key).  -0 is folded
// into +0 first so the two compare equal, as they do as floats.
MOE_DEV uint32_t float_order_key(float v) {
  uint32_t u = __float_as_uint(v + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ------------------------------------------------------- error-free sums
// TwoSum (Knuth): s + e == a + b exactly, s = fl(a + b).
MOE_DEV void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}
// TwoProduct via fused multiply-add: p + e == a * b exactly.
MOE_DEV void two_prod(float a, float b, float& p, float& e) {
  p = __fmul_rn(a, b);
  e = __fmaf_rn(a, b, -p);
}

}  // namespace moe
