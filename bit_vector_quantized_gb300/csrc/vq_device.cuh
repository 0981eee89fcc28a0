// vq_device.cuh -- device-side building blocks for the sm_103a VQ attention kernels.
//
// Inline-PTX wrappers (mbarrier, bulk asynchronous copy, warp-level mma,
// movmatrix, fences) and the warp-shuffle fast Walsh-Hadamard transform that the
// encode kernel and the query transform share.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace vqk {

constexpr int kHeadDim = 128;
constexpr int kChunk = 16;  // tokens per mma row block

enum DeviceStatus : int32_t {
  kDevOk = 0, kDevBadPage = 1, kDevBadSlot = 2, kDevTimeout = 3, kDevBadConfig = 4
};

__device__ __forceinline__ void report(int32_t* status, int32_t code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------- programmatic dependent launch ---
// A kernel launched with programmatic stream serialization may be scheduled
// while the previous kernel in the stream still runs, once that kernel
// signals pdl_trigger.  The library launches only the second and later
// kernels of one call that way, and the first kernel of a call starts after
// all earlier stream work has completed; so before pdl_wait a kernel reads
// only its call's inputs that the previous kernel of the same call does not
// write (codebooks, lambda, queries, new keys/values, page tables, lengths,
// slots) and writes nothing.  pdl_wait blocks until the previous kernel has
// completed and its memory is visible.  Without the launch attribute both
// are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- mbarrier ---

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// One bounded wait for phase `parity` of `bar`: the warp may be suspended by
// the hardware until the phase completes or about `suspend_ns` nanoseconds
// pass, whichever comes first; true when the phase completed.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity,
                                              uint32_t suspend_ns = 0x10000u) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(suspend_ns)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits for phase `parity` of `bar` to complete, giving up after `timeout_ns`
// nanoseconds (or soon after *abort is set by another warp).  Each try may
// park the warp for up to ~65 us, so a waiting warp costs almost no issue
// slots.  Returns false when it gave up; the caller then treats the stage as
// empty.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort, uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > timeout_ns) return false;
  }
}

// ------------------------------------------------------- bulk async copy ---

// One contiguous global -> shared copy completing on `bar` (TMA bulk engine).
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Orders this thread's earlier generic-proxy global-memory accesses before
// later async-proxy (bulk copy) accesses, once a release / acquire pair has
// carried them to the issuing thread.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ------------------------------------------------------------ warp mma ---

// D (16x8 fp32) += A (16x16 fp16, row) * B (16x8 fp16, col).
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 b16 matrix held one row pair per thread (row lane/4,
// columns 2*(lane%4) and 2*(lane%4)+1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_half2(__half lo, __half hi) {
  return static_cast<uint32_t>(__half_as_ushort(lo)) |
         (static_cast<uint32_t>(__half_as_ushort(hi)) << 16);
}

// fp32 pair -> (hi, lo) fp16 pairs with hi + lo == x to about 2^-22 relative.
__device__ __forceinline__ void split_half2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
  const __half l0 = __float2half_rn(x0 - __half2float(h0));
  const __half l1 = __float2half_rn(x1 - __half2float(h1));
  hi = pack_half2(h0, h1);
  lo = pack_half2(l0, l1);
}

// -------------------------------------------------- fast Walsh-Hadamard ---

// Unnormalised Walsh-Hadamard transform (Sylvester / natural order) of a
// 128-vector spread over a warp: lane l holds elements 4l .. 4l+3.  Butterflies
// (a, b) -> (a + b, a - b) at strides 1 and 2 in registers, 4 .. 64 across
// lanes.  Multiply by 1/sqrt(128) for the orthonormal H_128.
// 2^x with the hardware approximation (ex2.approx.ftz); 2^-inf = 0.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void fwht128_warp(float (&x)[4], int lane) {
  {
    const float a0 = x[0] + x[1], a1 = x[0] - x[1];
    const float a2 = x[2] + x[3], a3 = x[2] - x[3];
    x[0] = a0 + a2;
    x[2] = a0 - a2;
    x[1] = a1 + a3;
    x[3] = a1 - a3;
  }
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float y = __shfl_xor_sync(0xffffffffu, x[e], m);
      x[e] = upper ? (y - x[e]) : (x[e] + y);
    }
  }
}

}  // namespace vqk
