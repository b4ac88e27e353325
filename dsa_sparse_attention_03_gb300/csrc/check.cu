// Device check of the declared operand bounds (dsa_check_bounds): every byte
// of the int8 operands against qk_abs_max, every head weight against
// w_abs_max.  Streams the operands once with 16-byte loads; a warp that finds
// a violation raises DSA_DEVICE_RANGE once.
#include "common.cuh"

namespace dsa {
namespace {

// Largest |byte| of a word of four int8 values (|-128| = 128, no saturation).
__device__ __forceinline__ uint32_t max_abs_bytes(uint32_t w) {
  const uint32_t a = __vabs4(w);   // per byte, modulo 256: 0x80 stays 0x80 = 128
  return max(max(a & 0xFFu, (a >> 8) & 0xFFu), max((a >> 16) & 0xFFu, a >> 24));
}

__global__ void check_bounds_kernel(const int8_t* k, size_t k_chunks, const int8_t* q, size_t q_chunks,
                                    const int32_t* w, size_t nw, uint32_t qk, int64_t wmax, uint32_t* status) {
  bool bad = false;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  const size_t i0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (qk < 128u) {
    for (size_t i = i0; i < k_chunks; i += stride) {
      const int4 v = __ldg(reinterpret_cast<const int4*>(k) + i);
      const uint32_t m = max(max(max_abs_bytes(v.x), max_abs_bytes(v.y)), max(max_abs_bytes(v.z), max_abs_bytes(v.w)));
      bad |= m > qk;
    }
    for (size_t i = i0; i < q_chunks; i += stride) {
      const int4 v = __ldg(reinterpret_cast<const int4*>(q) + i);
      const uint32_t m = max(max(max_abs_bytes(v.x), max_abs_bytes(v.y)), max(max_abs_bytes(v.z), max_abs_bytes(v.w)));
      bad |= m > qk;
    }
  }
  for (size_t i = i0; i < nw; i += stride) {
    const int64_t v = w[i];
    bad |= (v < 0 ? -v : v) > wmax;
  }
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(status, DSA_DEVICE_RANGE);
}

}  // namespace

cudaError_t launch_check_bounds(const int8_t* k, size_t k_bytes, const int8_t* q, size_t q_bytes,
                                const int32_t* w, size_t nw, int qk, int wmax, uint32_t* status,
                                cudaStream_t st) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const size_t work = (k_bytes + q_bytes) / 16 + nw;
  size_t blocks = (work + 255) / 256;
  const size_t cap = (size_t)(sms > 0 ? sms : 1) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  check_bounds_kernel<<<(unsigned)blocks, 256, 0, st>>>(k, k_bytes / 16, q, q_bytes / 16, w, nw,
                                                         (uint32_t)qk, (int64_t)wmax, status);
  return cudaGetLastError();
}

}  // namespace dsa
