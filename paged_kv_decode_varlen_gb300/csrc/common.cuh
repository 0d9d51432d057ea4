// Device helpers shared by the libpa kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

constexpr int kHeadDim = PA_HEAD_DIM;      // D
constexpr int kPage = PA_BLOCK_SIZE;       // tokens per page
constexpr int kGroup = PA_GQA_GROUP;       // q heads per kv head
constexpr int kSlabBytes = kPage * kHeadDim * 2;  // one (page, kv head) of K or V: 4 KiB
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// Upper bound on any in-kernel wait (nanoseconds of %globaltimer).
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// Record the first device-side error in the error word (first writer wins).
__device__ __forceinline__ void record_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Two bf16 packed in a 32-bit word -> two fp32 (exact: bf16 is the high half
// of a binary32).  lo = element 0 (lower address), hi = element 1.
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // round to nearest even
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` to complete, giving up after limit_ns
// (kWaitLimitNs unless a diagnostic kernel shortens it).  Returns false on
// timeout (the caller records it).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0 && globaltimer() - t0 > limit_ns) return false;
  }
}

// 1-D bulk copy global -> shared (TMA engine), completing on `bar` with a
// transaction count of `bytes`.  Both addresses 16-byte aligned, bytes a
// multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Bulk prefetch of global memory into L2 (no shared memory, no completion).
__device__ __forceinline__ void bulk_prefetch_l2(const void* src_gmem, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src_gmem), "r"(bytes) : "memory");
}

// ------------------------------------------------------------- cp.async (16 B)
__device__ __forceinline__ void cp_async16(void* dst_smem, const void* src_gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst_smem)), "l"(src_gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// 2^x with the MUFU unit (ex2.approx.ftz: relative error ~2^-22; -inf -> 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Orders this thread's earlier generic-proxy shared-memory accesses (and
// those made visible to it) before its later async-proxy (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Orders this thread's earlier generic-proxy global writes before async-
// proxy (bulk copy) accesses that follow a barrier.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// mbarrier arrive without a transaction count (consumer release).
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// atomicAdd with acquire-release semantics at GPU scope: writes this thread
// has made (or observed, e.g. through a CTA barrier) before it are visible to
// a thread that reads the counter's result after it, and the reads that
// follow it see what the earlier adders published.
__device__ __forceinline__ int atom_add_acq_rel_gpu(int* addr, int v) {
  int old;
  asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v) : "memory");
  return old;
}

// Acquire load at GPU scope (pairs with a release by another CTA).
__device__ __forceinline__ int ld_acquire_gpu(const int* addr) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
  return v;
}

// Relaxed load at GPU scope: with fence_acq_rel_gpu() after it, an acquire
// (the load can be issued early and its latency hidden behind other loads).
__device__ __forceinline__ int ld_relaxed_gpu(const int* addr) {
  int v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// Release add at GPU scope: this thread's earlier writes (and those it has
// observed, e.g. through a CTA barrier) are visible to a thread that
// acquires the new value.
__device__ __forceinline__ void red_add_release_gpu(int* addr, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(addr), "r"(v) : "memory");
}

// ------------------------------------------- programmatic dependent launch
// Kernels are launched with programmatic stream serialization: each CTA of
// the short kernels lets the next kernel of the stream be scheduled as soon
// as it starts, and every kernel waits for the previous one to complete
// (memory visible) before it touches any input, so only launch latency and
// CTA dispatch overlap.  Both return at once for a kernel launched without
// the attribute.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launch `kernel` on `stream`, with programmatic stream serialization when
// `overlap` is set (else in plain stream order).
template <class... Exp, class... Act>
cudaError_t launch_maybe_pdl(bool overlap, void (*kernel)(Exp...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Act&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = overlap ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Act&&>(args)...);
}

// Launch `kernel` on `stream` with programmatic stream serialization.
template <class... Exp, class... Act>
cudaError_t launch_pdl(void (*kernel)(Exp...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Act&&... args) {
  return launch_maybe_pdl(true, kernel, grid, block, smem, stream, static_cast<Act&&>(args)...);
}

// bf16 pair -> float2 (element 0 in .x)
__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t w) { return make_float2(bf16lo(w), bf16hi(w)); }

// Log-sum-exp merge of two normalised partials over disjoint key sets with
// log2-domain lse a and b: the merged partial is wa * o_a + wb * o_b and the
// merged lse is returned (both empty: weights 0, lse -inf).
__device__ __forceinline__ float merge2_weights(float a, float b, float& wa, float& wb) {
  const float M = fmaxf(a, b);
  if (M == -INFINITY) {
    wa = wb = 0.f;
    return -INFINITY;
  }
  const float ea = exp2f(a - M), eb = exp2f(b - M);  // an empty side gives exp2(-inf) = 0
  const float inv = 1.f / (ea + eb);
  wa = ea * inv;
  wb = eb * inv;
  return M + log2f(ea + eb);
}

}  // namespace pa
