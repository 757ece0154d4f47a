// common.cuh -- device helpers shared by the libbonsai kernels (sm_103a).
//
// Inline PTX for the Blackwell asynchronous machinery: mbarrier phases with
// bounded waits, 1-D bulk copies global->shared (TMA engine), programmatic
// dependent launch, and the legacy warp-level mma.sync used as a wide FP32
// accumulator by the streaming decode kernels.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/bonsai.h"

namespace bonsai {

// Each translation unit has its own status word; the host reads and clears
// all of them in bonsai_check_async. First error wins.
#define BONSAI_DEFINE_STATUS(name)                                          \
  static __device__ unsigned int name;                                      \
  [[maybe_unused]] static __device__ __forceinline__ void set_status(      \
      unsigned int code) {                                                  \
    atomicCAS(&name, 0u, code);                                             \
  }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------- mbarrier ----------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Default bound of a device-side wait: 2 seconds of wall-clock time.
constexpr uint64_t kWaitNs = 2000000000ull;

// Waits until the phase with the given parity has completed. Returns false
// if `limit_ns` of wall-clock time ran out (the caller records a timeout and
// stops waiting instead of hanging the GPU).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          uint64_t limit_ns = kWaitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

// ---------------- bulk copy (TMA engine, no tensor map) ----------------
// dst, src 16-byte aligned, bytes a multiple of 16. Completion is signalled
// as transaction bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// 16-byte asynchronous copy global -> shared through L2 (bypassing L1), and
// the mbarrier arrival that fires once this thread's prior copies landed.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst),
               "l"(src), "l"(policy)
               : "memory");
}
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 2-D TMA tile load into shared memory, completion as transaction bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

// ---------------- gated feed-forward epilogue ----------------
// silu(g) = g * sigmoid(g) = g / (1 + e^-g), in FP32 (expf, IEEE divide):
// e^-g overflows to +inf below g ~ -88 and the quotient is then -0.
__device__ __forceinline__ float silu(float g) { return g / (1.f + expf(-g)); }

// ---------------- programmatic dependent launch ----------------
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------- named barriers ----------------
__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---------------- warp MMA: D = A(16x16 f16) * B(16x8 f16) + C (f32) --------
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                          uint32_t a2, uint32_t a3, uint32_t b0,
                                          uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_half2(__half lo, __half hi) {
  return static_cast<uint32_t>(__half_as_ushort(lo)) |
         (static_cast<uint32_t>(__half_as_ushort(hi)) << 16);
}

}  // namespace bonsai

// ---------------- host helpers ----------------
namespace bonsai {

inline bonsai_status cuda_status(cudaError_t e) {
  return e == cudaSuccess ? BONSAI_OK : BONSAI_ERR_CUDA;
}

int device_sm_count();
int device_max_smem_optin();
// Raises a kernel's dynamic shared-memory limit on the current device once
// (later calls with the same or a smaller size touch no CUDA API, so launches
// can be captured into a CUDA graph after a first eager call).
cudaError_t ensure_dynamic_smem(const void* kernel, int bytes);
// 2-D tiled tensor map (no swizzle unless given), out-of-range elements
// read as zero. Returns false if the driver rejects it.
bool encode_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType type, void* base,
                          uint64_t dim0, uint64_t dim1, uint64_t stride1_bytes, uint32_t box0,
                          uint32_t box1, CUtensorMapSwizzle swizzle);

}  // namespace bonsai
