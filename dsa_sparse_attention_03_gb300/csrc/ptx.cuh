// Device helpers shared by the kernels: PTX wrappers for warp-level MMA,
// ldmatrix, bulk copies and mbarriers, and the two bounded waits (an mbarrier
// phase, a grid barrier), each of which gives up after a limit in nanoseconds
// and raises DSA_DEVICE_TIMEOUT instead of waiting forever.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "barrier_protocol.h"
#include "common.cuh"

namespace dsa {

__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Device operations of the barrier protocol (barrier_protocol.h) on one
// global counter.
struct GridOps {
  uint32_t* c;
  uint32_t* status;
  __device__ void fence() { __threadfence(); }
  __device__ void arrive() { atomicAdd(c, 1u); }
  __device__ uint32_t count() { return ld_acquire(c); }
  __device__ uint64_t now() { return gtimer(); }
  __device__ void timeout() { raise_status(status, DSA_DEVICE_TIMEOUT); }
};

// Barrier over the whole grid (co-resident by the cooperative launch): the
// CTA's writes are published before it arrives at counter c, and every later
// read sees the other CTAs' writes.  Bounded: after limit_ns the CTA raises
// DSA_DEVICE_TIMEOUT and returns false (the caller then exits).
static __device__ __noinline__ bool grid_barrier(uint32_t* c, uint32_t* status, uint64_t limit_ns) {
  __shared__ int ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    GridOps ops{c, status};
    ok = barrier_arrive_and_wait(ops, gridDim.x, limit_ns) ? 1 : 0;
  }
  __syncthreads();
  return ok != 0;
}

// The same protocol among `n` CTAs that share the counter c (all of them
// co-resident): every thread of each CTA takes part.
static __device__ __noinline__ bool group_barrier(uint32_t* c, uint32_t n, uint32_t* status, uint64_t limit_ns) {
  __shared__ int ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    GridOps ops{c, status};
    ok = barrier_arrive_and_wait(ops, n, limit_ns) ? 1 : 0;
  }
  __syncthreads();
  return ok != 0;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// One contiguous row (16-byte aligned, size a multiple of 16) by the bulk-copy engine.
__device__ __forceinline__ void bulk_row(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}
// One non-blocking test of the phase of parity `parity`.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}
// Bounded wait for the phase of parity `parity`: false (and DSA_DEVICE_TIMEOUT
// raised, if `status`) once `limit_ns` have passed.  A phase that has already
// completed returns at once, without reading the clock.
static __device__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t* status, uint64_t limit_ns) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = gtimer();
  for (;;) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    if (ok) return true;
    if (gtimer() - t0 > limit_ns) {
      raise_status(status, DSA_DEVICE_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Sixteen e4m3 codes to sixteen bf16 values (eight packed pairs), exactly:
// e4m3 -> f16 by the hardware conversion, f16 -> f32 -> bf16 lossless for
// these values (at most 4 significant bits, exponents within both ranges).
__device__ __forceinline__ void e4m3x16_to_bf16(const uint4 v, uint4& lo, uint4& hi) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int hpair = 0; hpair < 2; ++hpair) {
      const __nv_fp8x2_storage_t b = static_cast<__nv_fp8x2_storage_t>(w[i] >> (16 * hpair));
      const __half2 h = __half2(__nv_cvt_fp8x2_to_halfraw2(b, __NV_E4M3));
      const float2 f = __half22float2(h);
      o[2 * i + hpair] = pack_bf16(f.x, f.y);
    }
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

}  // namespace dsa
