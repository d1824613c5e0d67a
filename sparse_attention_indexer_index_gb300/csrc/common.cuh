// common.cuh -- shared device helpers of the QSA indexer kernels (sm_103a).
//
// Fixed problem sizes of the QSA indexer (Qwen3.8-Flash-Next day-0 write-up,
// theainews.cc, section "Qwen sparse attention (QSA)"): 4 index query heads
// of 128 dims, one shared 128-dim key head, 4 raw keys per compressed block.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace qsa {

constexpr int kDim = 128;          // index head dim
constexpr int kHeads = 4;          // index query heads
constexpr int kBlock = 4;          // raw keys per compressed block (c4)
constexpr int kMaxK = 2048;        // largest k a selection supports
constexpr int kMaxShareExtra = 1 << 16;  // drafted columns a reused row may reserve
// 1/sqrt(128) rounded to FP32.
constexpr float kScoreScale = 0.08838834764831845f;

// Device fault word bits (reported by qsa_device_status()).
constexpr unsigned kFaultIndex = 1u;      // row / page index out of range
constexpr unsigned kFaultPool = 2u;       // pool row out of range
constexpr unsigned kFaultWait = 4u;       // a bounded wait expired
constexpr unsigned kFaultGrouping = 8u;   // inconsistent row grouping / lengths
constexpr unsigned kFaultCapacity = 16u;  // an output row too narrow for its entries

// Device fault word of this translation unit (internal linkage: every
// translation unit that launches kernels has its own and exposes a host
// reader; qsa_device_status() combines them).
static __device__ unsigned g_fault_word = 0u;

__device__ __forceinline__ void raise_fault(unsigned bits) { atomicOr(&g_fault_word, bits); }

// ---------------------------------------------------------------------------
// Order-preserving map FP32 -> u32 used by the radix selection: larger float
// -> larger key; -0 and +0 map to the same key; NaN maps to 0, below -inf.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0u;  // NaN
  if (u == 0x80000000u) u = 0u;                      // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ---------------------------------------------------------------------------
// Thread-block cluster helpers (distributed shared memory).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// Full cluster barrier with release/acquire semantics on shared::cluster.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// Address of the same shared variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_shared_rank(const void* smem_ptr, uint32_t rank) {
  uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(smem_ptr));
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}
// Load from distributed shared memory.  volatile keeps it after the cluster
// barrier that precedes it (the barrier is a volatile asm with a memory
// clobber); without its own clobber, several of these loads can be in flight
// at once when their results are consumed later.
__device__ __forceinline__ uint32_t ld_dsmem_u32(uint32_t cluster_addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(cluster_addr));
  return v;
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch: the primary grid lets the dependent grid be
// scheduled early; the dependent grid waits for the primary's memory.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---------------------------------------------------------------------------
// mbarrier + bulk asynchronous copy (TMA engine, no tensor map) helpers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Arrive on the barrier and announce `bytes` of incoming asynchronous copies.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait for a barrier phase: gives up after `limit_ns` of wall time
// (returns false; the caller latches kFaultWait and leaves cleanly).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns = 200000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
  return true;
}
// Global -> shared bulk copy of `bytes` (multiple of 16, both addresses
// 16-byte aligned), completing on `bar` with a transaction count.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Read-only 16-byte load that does not allocate in L1 (streamed once).
__device__ __forceinline__ uint4 ld_stream_16(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// BF16 pair (packed in one u32, low half first) -> two floats.
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t u) {
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

// Request of row t: the r with req_row_start[r] <= t < req_row_start[r+1]
// (rows grouped by request, starts non-decreasing).  Binary search.
__device__ __forceinline__ int row_request(const int32_t* __restrict__ req_row_start, int n_req,
                                           int t) {
  int lo = 0, hi = n_req - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(req_row_start + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

}  // namespace qsa
