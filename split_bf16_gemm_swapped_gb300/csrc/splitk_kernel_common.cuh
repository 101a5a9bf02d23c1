// Device-side helpers shared by the split-K kernels (the per-tile kernel in
// splitk_kernel.cu and the persistent one in splitk_persistent.cu): the
// bounded mbarrier waits and their fault record, the drain after a failure,
// timeline stamps, clipped stores and accumulator reads from tensor memory.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "splitk.h"
#include "splitk_device.cuh"
#include "splitk_internal.h"

namespace splitk {

// First timeout since the last read of the kernels of the translation unit
// that includes this header (each kernel file has its own record; the host
// reads them all): code, role, index, parity, blockIdx.{x,y,z}, cluster rank.
static __device__ int g_fault[kFaultWords];

namespace {

// Records the first timeout of the device (out of line: cold path).
__device__ __noinline__ void record_fault(int role, int index, uint32_t parity) {
  if (atomicCAS(&g_fault[0], 0, (int)SPLITK_ERR_TIMEOUT) == 0) {
    g_fault[1] = role;
    g_fault[2] = index;
    g_fault[3] = (int)parity;
    g_fault[4] = (int)blockIdx.x;
    g_fault[5] = (int)blockIdx.y;
    g_fault[6] = (int)blockIdx.z;
    g_fault[7] = (int)dev::cluster_ctarank();
    __threadfence();
  }
}

template <bool kClusterScope>
__device__ __forceinline__ bool poll_phase(uint32_t bar, uint32_t parity) {
  return kClusterScope ? dev::mbar_try_wait_cluster(bar, parity, kWaitHintNs)
                       : dev::mbar_try_wait(bar, parity, kWaitHintNs);
}

// The bounded part of a wait (out of line: reached only when the first
// try_wait gave up).  Returns false if the limit ran out (recording it) or
// another wait of the CTA already failed.
template <bool kClusterScope>
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, uint32_t abort_flag,
                                       unsigned long long limit_ns, int role, int index) {
  const uint64_t t0 = dev::globaltimer_ns();
  while (true) {
    if (poll_phase<kClusterScope>(bar, parity)) return true;
    if (dev::ld_shared_u32(abort_flag) != 0u) return false;
    if (dev::globaltimer_ns() - t0 > limit_ns) {
      dev::st_shared_u32(abort_flag, 1u);
      record_fault(role, index, parity);
      return false;
    }
  }
}

// After a failure: waits, bounded by `limit_ns` and regardless of the CTA's
// failure flag, for the phase of `bar` with `parity` -- the landing of copies
// this CTA issued into its own shared memory -- so that it does not leave
// with a copy still writing there.  Returns whether the phase completed.
__device__ __noinline__ bool drain_wait(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
  const uint64_t t0 = dev::globaltimer_ns();
  while (!dev::mbar_try_wait(bar, parity, 10000u)) {
    if (dev::globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// A position in a ring of n entries after `count` uses: the entry
// count % n and the parity of count / n, kept by additions.  (An integer
// division by a runtime value is a long dependent instruction sequence; in a
// per-tile loop it sits on the critical path.)
struct RingPos {
  int index;
  uint32_t phase;
  __device__ __forceinline__ static RingPos at(int count, int n) {
    return RingPos{count % n, (uint32_t)((count / n) & 1)};
  }
  // `by` more uses, 1 <= by <= n
  __device__ __forceinline__ void advance(int by, int n) {
    index += by;
    if (index >= n) {
      index -= n;
      phase ^= 1u;
    }
  }
};

struct Waiter {
  uint32_t abort_flag;            // shared-memory u32, sticky per CTA
  unsigned long long limit_ns;

  // Waits for the phase of `bar` with `parity` to complete (bounded).
  // `spans` > 1 for waits that legitimately cover other bounded waits of the
  // CTA (the TMEM release covers the whole epilogue), so those report first.
  template <bool kClusterScope>
  __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity, int role, int index,
                                       unsigned spans = 1) const {
    if (poll_phase<kClusterScope>(bar, parity)) return true;
    return wait_slow<kClusterScope>(bar, parity, abort_flag, limit_ns * spans, role, index);
  }
};

__device__ __forceinline__ uint32_t smid() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
  return r;
}

// One %globaltimer stamp into this CTA's trace record (tracing on only).
__device__ __forceinline__ void stamp(const KernelParams& p, int slot) {
  if (p.trace != nullptr) {
    const uint32_t cta = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
    if (cta < p.trace_ctas) p.trace[(size_t)cta * kTraceSlots + slot] = dev::globaltimer_ns();
  }
}

// Element stores of up to 8 bf16 of one C row, clipped at N (cold path:
// N not a multiple of 8, C not 16-byte aligned, or the row's last vector).
__device__ __noinline__ void store8_clipped(uint16_t* dst, int n, int N, uint32_t q0, uint32_t q1,
                                            uint32_t q2, uint32_t q3) {
  const uint32_t q[4] = {q0, q1, q2, q3};
  for (int e = 0; e < 8 && n + e < N; ++e) {
    dst[e] = (uint16_t)((e & 1) ? (q[e >> 1] >> 16) : (q[e >> 1] & 0xFFFFu));
  }
}

// Accumulator columns [col, col + 16) (or + 4) of this thread's TMEM lane:
// with two MMA issuers, the sum of both accumulators (`second` columns
// apart), accumulator 0 first.
__device__ __forceinline__ void load_acc16(uint32_t taddr, uint32_t second, bool two, uint32_t (&v)[16]) {
  dev::tmem_ld_x16(taddr, v);
  if (two) {
    uint32_t w[16];
    dev::tmem_ld_x16(taddr + second, w);
    dev::tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) + __uint_as_float(w[e]));
  } else {
    dev::tmem_wait_ld();
  }
}

__device__ __forceinline__ void load_acc4(uint32_t taddr, uint32_t second, bool two, uint32_t (&v)[4]) {
  dev::tmem_ld_x4(taddr, v[0], v[1], v[2], v[3]);
  if (two) {
    uint32_t w[4];
    dev::tmem_ld_x4(taddr + second, w[0], w[1], w[2], w[3]);
    dev::tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) + __uint_as_float(w[e]));
  } else {
    dev::tmem_wait_ld();
  }
}

}  // namespace

}  // namespace splitk
