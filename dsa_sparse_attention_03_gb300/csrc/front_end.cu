// Indexer front end: the integer indexer query q_idx and head weights w_idx of
// each query row, projected from the row's hidden vector by weights stored as
// 8-bit affine group-quantised codes ("GLM-5.3-Flash-Alis-MLX-4bit", page 3:
// the DSA indexer projections at 8 bits in groups of 64, MLX affine form), then
// quantised to the operand bounds the indexer declares.
//
// One kernel, HBM-bound at one query row: the weights are the traffic (one
// byte per weight plus 4 bytes of scale and bias per 64), read once per pass of
// up to RB query rows.
//
//   * Output rows (H_i * D_i query rows, then H_i head-weight rows) are split
//     into contiguous, equal ranges, one per CTA (one CTA per SM).
//   * A producer warp streams the CTA's rows with bulk copies into a ring of
//     shared-memory stages of 4 rows (codes, scales, biases; about 26 KB at
//     d = 6144): few, large copies, since the copy engine's cost is per request.
//   * Sixteen consumer warps take items of one stage x 512 inputs: each lane
//     takes the same 16 inputs (a quarter of one 64-input group) of the 4 rows
//     and reads those inputs from shared memory once per query row for all 4
//     (the hidden rows are stored lane-interleaved, so the reads are
//     conflict-free).  Per row it forms sum_k code_k * x_k in fp32 (codes
//     widened exactly through the 2^23 float trick, each product exact),
//     scales it by the group's scale and, in the group's first lane, adds
//     bias * (sum of the group's inputs); a fixed exchange tree reduces the 4
//     rows over the warp.
//   * Partials go to shared memory by (row, item) and are summed in item
//     order: the result does not depend on timing.
//   * Per-head max |qf| is merged with atomicMax on the float bits (|y| >= 0).
//   * The last CTA to finish a pass (an arrival ticket per pass) quantises that
//     pass's rows: sigma_h = max|qf_h| / q_max, q = rint(qf / sigma_h),
//     u_h = wf_h * sigma_h, tau = max|u| / w_max, w = rint(u / tau), each
//     clamped, in fp32 with IEEE division and round-half-to-even.
//
// The projection is fp32 (the exact products summed in a fixed tree), so the
// projected values differ from the exact real ones by at most about 2^-17 of
// the sum of the magnitudes of their terms; codes whose exact ratio lies that
// close to a rounding midpoint may come out one step away from the
// exact-arithmetic code.
#include "common.cuh"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kFeConsumerWarps = 16;
constexpr int kFeConsumers = kFeConsumerWarps * 32;
constexpr int kFeThreads = kFeConsumers + 32;   // + one producer warp
constexpr int kFeSeg = 512;                     // inputs per warp item (16 per lane)
constexpr int kFeMaxStages = 8;
constexpr int kFeMinStages = 3;

// Byte k of w as a float, exactly: 0x4B0000cc is 2^23 + c.
__device__ __forceinline__ float code_at(uint32_t w, int k) {
  return __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7440 + k)) - 8388608.f;
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ void mbar_arrive1(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// The consumer warps' own barrier (the producer warp does not take part).
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kFeConsumers) : "memory");
}
// The same barrier, returning whether any consumer thread passed p (the same
// answer in every thread).
__device__ __forceinline__ bool consumers_any(bool p) {
  uint32_t r;
  asm volatile("{\n.reg .pred pi, po;\nsetp.ne.u32 pi, %1, 0;\nbar.red.or.pred po, 1, %2, pi;\n"
               "selp.u32 %0, 1, 0, po;\n}\n"
               : "=r"(r) : "r"((uint32_t)p), "n"(kFeConsumers) : "memory");
  return r != 0;
}

// Shared-memory map (bytes from the 128-byte-aligned base).
struct FeSmem {
  uint32_t stage_bytes, off_x, off_sx, off_part, off_sig, off_list, off_bar, total;
};
__host__ __device__ inline FeSmem fe_smem_map(int RB, int S, int d, int rows_max, int H_i) {
  FeSmem m;
  const int G = d / 64, nseg = d / kFeSeg;
  m.stage_bytes = 4u * ((uint32_t)d + (uint32_t)d / 16);   // 4 rows: codes, scales, biases
  uint32_t off = (uint32_t)S * m.stage_bytes;
  m.off_x = off; off += (uint32_t)RB * d * 4;
  m.off_sx = off; off += (uint32_t)RB * G * 4;
  m.off_part = off; off += (uint32_t)RB * rows_max * nseg * 4;
  m.off_sig = off; off += (uint32_t)H_i * 4;
  m.off_list = off; off += (32 + 4 * 16) * 4;   // head list [32], per-head maxima [4][16]
  off = (off + 7) & ~7u;
  m.off_bar = off; off += (uint32_t)S * 16;
  m.total = off;
  return m;
}

template <int RB>
__global__ void __launch_bounds__(kFeThreads, 1) front_end_kernel(const __grid_constant__ FrontArgs a) {
  extern __shared__ float4 fe_smem4[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(fe_smem4);
  const int d = a.d, G = d / 64, nseg = d / kFeSeg, S = a.stages;
  const int O = a.Oq + a.H_i;
  const int o0 = (int)(((int64_t)blockIdx.x * O) / gridDim.x);
  const int o1 = (int)(((int64_t)(blockIdx.x + 1) * O) / gridDim.x);
  const int nrows = o1 - o0;
  const int npass = (a.R + RB - 1) / RB;
  const FeSmem m = fe_smem_map(RB, S, d, a.rows_max, a.H_i);
  float* xs = reinterpret_cast<float*>(smem + m.off_x);         // [RB][d], lane-interleaved (below)
  float* sx = reinterpret_cast<float*>(smem + m.off_sx);        // [RB][G]
  float* part = reinterpret_cast<float*>(smem + m.off_part);    // [RB][rows_max][nseg]
  float* sig = reinterpret_cast<float*>(smem + m.off_sig);      // [H_i]
  int* list = reinterpret_cast<int*>(smem + m.off_list);        // [0] count, [1..30] heads, [31] last
  const uint32_t bar_full = smem_u32(smem + m.off_bar);         // S barriers, then S "empty"
  const uint32_t bar_empty = bar_full + 8 * S;
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, nseg);   // one arrival per warp item of the row group
    }
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  if (warp == kFeConsumerWarps) {
    // ------------------------------------------------------------ producer
    // Streams the CTA's weights, one stage per group of 4 output rows (their
    // codes, scales and biases: consecutive rows of one matrix are contiguous,
    // so a group is one copy of each, or two where it crosses from the query
    // rows to the head-weight rows), for every pass.  The weights are inputs no
    // kernel of the step writes, so the first stages go out before the wait on
    // the previous kernel.
    if (lane == 0) {
      const int ngrp = (nrows + 3) / 4, total = npass * ngrp;
      const uint32_t cb = 4u * (uint32_t)d, sbb = 4u * (uint32_t)G * 2u;   // codes / scales bytes of a stage
      int i = 0;
      for (; i < total; ++i) {
        const int s = i % S, n = i / S;
        if (n > 0 && !mbar_wait(bar_empty + 8 * s, (n - 1) & 1, a.status, a.wait_ns)) {
          abort_flag = 1;
          break;
        }
        if (*reinterpret_cast<volatile int*>(&abort_flag)) break;
        const int g0 = o0 + (i % ngrp) * 4, nr = min(4, o1 - g0);
        const uint32_t dst = smem_u32(smem + (size_t)s * m.stage_bytes);
        mbar_expect_tx(bar_full + 8 * s, (uint32_t)nr * ((uint32_t)d + (uint32_t)G * 4u));
        for (int j = 0; j < nr;) {   // runs of rows within one matrix
          const int o = g0 + j;
          const bool q = o < a.Oq;
          const int run = q ? min(nr - j, a.Oq - o) : nr - j;
          const size_t orow = (size_t)(q ? o : o - a.Oq);
          bulk_row(dst + j * d, (q ? a.wq : a.ww) + orow * d, (uint32_t)(run * d), bar_full + 8 * s);
          bulk_row(dst + cb + j * G * 2, (q ? a.sq : a.sw) + orow * G, (uint32_t)(run * G * 2), bar_full + 8 * s);
          bulk_row(dst + cb + sbb + j * G * 2, (q ? a.bq : a.bw) + orow * G, (uint32_t)(run * G * 2),
                   bar_full + 8 * s);
          j += run;
        }
      }
      // No copy may be in flight when the CTA exits (bounded).
      for (int k = max(0, i - S); k < i; ++k) mbar_wait(bar_full + 8 * (k % S), (k / S) & 1, a.status, a.wait_ns);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  pdl_wait();   // the hidden rows may come from the previous kernel
  pdl_trigger();
  const int ngrp = (nrows + 3) / 4, nitems = ngrp * nseg;
  for (int pass = 0; pass < npass; ++pass) {
    const int r0 = pass * RB, rb = min(RB, a.R - r0);
    consumers_sync();   // the previous pass is done with xs, sx, part and sig
    // This pass's hidden rows, widened to fp32.  Input i = 512 s + 16 l + k (lane
    // l of item segment s) is stored at 512 s + 128 (k / 4) + 4 l + k % 4, so the
    // lanes of a warp read their 16 inputs as four conflict-free 16-byte loads.
    for (int i = tid; i < rb * d / 4; i += kFeConsumers) {
      const int r = i / (d / 4), e = (i % (d / 4)) * 4;
      const uint2 v = *reinterpret_cast<const uint2*>(a.x + (size_t)(r0 + r) * d + e);
      const int sg = e / kFeSeg, l = (e % kFeSeg) / 16, k = e % 16;
      *reinterpret_cast<float4*>(xs + r * d + sg * kFeSeg + (k / 4) * 128 + l * 4) =
          make_float4(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y));
    }
    for (int i = tid; i < rb * G; i += kFeConsumers) {   // each group's input sum, in input order
      const uint4* p = reinterpret_cast<const uint4*>(a.x + (size_t)(r0 + i / G) * d + (i % G) * 64);
      float s = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint4 v = p[j];
        s += bf16_lo(v.x); s += bf16_hi(v.x); s += bf16_lo(v.y); s += bf16_hi(v.y);
        s += bf16_lo(v.z); s += bf16_hi(v.z); s += bf16_lo(v.w); s += bf16_hi(v.w);
      }
      sx[i] = s;
    }
    consumers_sync();

    // Warp items: 4 output rows x one 512-input segment.  Lane l takes inputs
    // 512 s + 16 l .. + 15 of the 4 rows' stages and reads those inputs once
    // per query row for all 4.
    for (int it = warp; it < nitems; it += kFeConsumerWarps) {
      const int og = it / nseg, seg = it % nseg, i0 = seg * kFeSeg + lane * 16, g = i0 / 64;
      const int nr = min(4, nrows - og * 4);
      uint4 cw[4];
      uint32_t sb[4];
      const int gi = pass * ngrp + og, st = gi % S;
      // Lane 0 polls the stage's barrier (512 polling threads would crowd the
      // barrier the copies complete on); then every lane observes the
      // completed phase itself, which makes the copied bytes visible to it.
      int okw = !*reinterpret_cast<volatile int*>(&abort_flag);
      if (lane == 0 && okw && !mbar_wait(bar_full + 8 * st, (gi / S) & 1, a.status, a.wait_ns)) {
        okw = 0;
        abort_flag = 1;
      }
      bool ok = __shfl_sync(0xffffffffu, okw, 0) != 0;
      if (ok) mbar_wait(bar_full + 8 * st, (gi / S) & 1, a.status, a.wait_ns);   // already complete
      const unsigned char* sp = smem + (size_t)st * m.stage_bytes;
      const uint16_t* ssc = reinterpret_cast<const uint16_t*>(sp + 4 * d);
      const uint16_t* sbi = ssc + 4 * G;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        cw[j] = make_uint4(0, 0, 0, 0);
        sb[j] = 0;
        if (j < nr && ok) {
          cw[j] = *reinterpret_cast<const uint4*>(sp + j * d + i0);
          sb[j] = (uint32_t)ssc[j * G + g] | ((uint32_t)sbi[j * G + g] << 16);
        }
      }
      __syncwarp();
      if (lane == 0 && ok) mbar_arrive1(bar_empty + 8 * st);
      if (!__all_sync(0xffffffffu, ok)) continue;
#pragma unroll
      for (int r = 0; r < RB; ++r) {
        if (r >= rb) break;
        float xv[16];
        const float4* xp = reinterpret_cast<const float4*>(xs + r * d + seg * kFeSeg + lane * 4);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 t = xp[q * 32];
          xv[4 * q + 0] = t.x; xv[4 * q + 1] = t.y; xv[4 * q + 2] = t.z; xv[4 * q + 3] = t.w;
        }
        const float gs = sx[r * G + g];
        float v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t w4[4] = {cw[j].x, cw[j].y, cw[j].z, cw[j].w};
          float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
          for (int k = 0; k < 16; k += 2) {
            acc0 = fmaf(code_at(w4[k / 4], k % 4), xv[k], acc0);
            acc1 = fmaf(code_at(w4[k / 4], k % 4 + 1), xv[k + 1], acc1);
          }
          v[j] = bf16_lo(sb[j]) * (acc0 + acc1);
          if ((lane & 3) == 0) v[j] = fmaf(bf16_hi(sb[j]), gs, v[j]);
        }
        // Reduce the four rows' values over the warp in six exchanges: lanes
        // with bit 4 set keep rows 2-3, then bit 3 picks one row, then sum.
        const bool h4 = lane & 16, h3 = lane & 8;
        const float a0 = (h4 ? v[2] : v[0]) + __shfl_xor_sync(0xffffffffu, h4 ? v[0] : v[2], 16);
        const float a1 = (h4 ? v[3] : v[1]) + __shfl_xor_sync(0xffffffffu, h4 ? v[1] : v[3], 16);
        float b = (h3 ? a1 : a0) + __shfl_xor_sync(0xffffffffu, h3 ? a0 : a1, 8);
        b += __shfl_xor_sync(0xffffffffu, b, 4);
        b += __shfl_xor_sync(0xffffffffu, b, 2);
        b += __shfl_xor_sync(0xffffffffu, b, 1);
        const int rl = og * 4 + (lane >> 3);
        if ((lane & 7) == 0 && (lane >> 3) < nr) part[(r * a.rows_max + rl) * nseg + seg] = b;
      }
    }
    if (consumers_any(*reinterpret_cast<volatile int*>(&abort_flag) != 0)) return;   // a wait ran out
    // Query heads this CTA touches: h0 .. h0 + nh - 1 (at most 10: rows_max <= 8 D_i).
    const int q1 = min(o1, a.Oq);
    const int h0 = o0 / a.D_i, nh = o0 < q1 ? (q1 - 1) / a.D_i - h0 + 1 : 0;
    uint32_t* hmax = reinterpret_cast<uint32_t*>(list + 32);   // [RB][16]
    if (tid < RB * 16) hmax[tid] = 0;
    if (tid == 0) list[0] = 0;
    consumers_sync();
    for (int i = tid; i < rb * nrows; i += kFeConsumers) {
      const int r = i / nrows, row = i % nrows, o = o0 + row;
      const float* p = part + (r * a.rows_max + row) * nseg;
      float y = 0.f;
      for (int j = 0; j < nseg; ++j) y += p[j];
      a.y[(size_t)(r0 + r) * a.y_stride + o] = y;
      if (a.proj) a.proj[(size_t)(r0 + r) * O + o] = y;
      if (o < a.Oq) atomicMax(hmax + r * 16 + (o / a.D_i - h0), __float_as_uint(fabsf(y)));
    }
    consumers_sync();
    if (tid < rb * nh) {   // one global merge per (query row, head) of this CTA
      const int r = tid / nh, hl = tid % nh;
      atomicMax(a.amax + (size_t)(r0 + r) * a.H_i + h0 + hl, hmax[r * 16 + hl]);
    }
    __threadfence();   // this CTA's projections and maxima before its arrivals
    consumers_sync();
    // Count this CTA's rows into each query head it touches (one thread per
    // head); the CTA that completes a head quantises it.  The last CTA of the
    // pass has every head's maximum and weight projection, and quantises the
    // head weights.
    if (tid < nh) {
      const int h = h0 + tid;
      const uint32_t c = (uint32_t)(min(q1, (h + 1) * a.D_i) - max(o0, h * a.D_i));
      if (atomicAdd(a.cnt + (size_t)pass * a.H_i + h, c) + c == (uint32_t)a.D_i) list[1 + atomicAdd(list, 1)] = h;
      __threadfence();
    }
    if (tid == 32) {
      list[31] = atomicAdd(a.ticket + pass, 1u) == gridDim.x - 1;
      __threadfence();
    }
    consumers_sync();
    const float qm = (float)a.q_max, wm = (float)a.w_max;
    for (int e = 0; e < list[0]; ++e) {
      const int h = list[1 + e];
      const int per_row = a.D_i / 4;
      for (int i = tid; i < rb * per_row; i += kFeConsumers) {
        const int r = r0 + i / per_row, j = (i % per_row) * 4;
        const float am = __uint_as_float(__ldcg(a.amax + (size_t)r * a.H_i + h));
        const float sg = __fdiv_rn(am, qm);
        const float4 y4 = __ldcg(reinterpret_cast<const float4*>(a.y + (size_t)r * a.y_stride + h * a.D_i + j));
        char4 c = make_char4(0, 0, 0, 0);
        if (sg > 0.f) {
          c.x = (signed char)fminf(fmaxf(rintf(__fdiv_rn(y4.x, sg)), -qm), qm);
          c.y = (signed char)fminf(fmaxf(rintf(__fdiv_rn(y4.y, sg)), -qm), qm);
          c.z = (signed char)fminf(fmaxf(rintf(__fdiv_rn(y4.z, sg)), -qm), qm);
          c.w = (signed char)fminf(fmaxf(rintf(__fdiv_rn(y4.w, sg)), -qm), qm);
        }
        *reinterpret_cast<char4*>(a.q_idx + (size_t)r * a.Oq + h * a.D_i + j) = c;
        if (j == 0 && a.q_scale) a.q_scale[(size_t)r * a.H_i + h] = sg;
      }
    }
    if (list[31] && warp == 0) {
      // Head weights of the pass's rows: u_h = wf_h * sigma_h, tau = max |u| / w_max.
      for (int r = r0; r < r0 + rb; ++r) {
        const float* yr = a.y + (size_t)r * a.y_stride;
        float um = 0.f;
        for (int h = lane; h < a.H_i; h += 32) {
          const float sg = __fdiv_rn(__uint_as_float(__ldcg(a.amax + (size_t)r * a.H_i + h)), qm);
          sig[h] = __ldcg(yr + a.Oq + h) * sg;
          um = fmaxf(um, fabsf(sig[h]));
        }
#pragma unroll
        for (int k = 16; k >= 1; k >>= 1) um = fmaxf(um, __shfl_xor_sync(0xffffffffu, um, k));
        const float tau = __fdiv_rn(um, wm);
        for (int h = lane; h < a.H_i; h += 32)
          a.w_idx[(size_t)r * a.H_i + h] = tau > 0.f ? (int32_t)fminf(fmaxf(rintf(__fdiv_rn(sig[h], tau)), -wm), wm) : 0;
        if (lane == 0 && a.w_scale) a.w_scale[r] = tau;
        __syncwarp();
      }
    }
  }
}

template <int RB>
cudaError_t launch_rb(const FrontArgs& a, int grid, size_t smem, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(front_end_kernel<RB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(front_end_kernel<RB>, dim3(grid), dim3(kFeThreads), smem, st, a);
}

constexpr uint32_t kFeSmemBudget = 227u * 1024u - 128u;

// Rows per pass and weight stages: the most rows (at most 4, at most R) that
// leave room for at least 8 stages; then as many stages as fit (at most 24).
bool fe_config(int R, int d, int H_i, int rows_max, int* RB, int* S) {
  for (int rb = 4; rb >= 1; rb >>= 1) {
    if (rb > R && rb > 1) continue;
    const FeSmem m0 = fe_smem_map(rb, 0, d, rows_max, H_i);
    const uint32_t per = fe_smem_map(rb, 1, d, rows_max, H_i).total - m0.total;
    if (m0.total + kFeMinStages * per > kFeSmemBudget) continue;
    int s = (int)((kFeSmemBudget - m0.total) / per);
    *RB = rb;
    *S = s > kFeMaxStages ? kFeMaxStages : s;
    return true;
  }
  return false;
}

}  // namespace

cudaError_t launch_front_end(FrontArgs a, cudaStream_t st) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int O = a.Oq + a.H_i;
  // One CTA per SM (at most one per output row), and enough CTAs that none
  // spans more than 8 D_i rows (so at most 10 query heads).
  int grid = sms < O ? sms : O;
  const int g_min = (O + 8 * a.D_i - 1) / (8 * a.D_i);
  if (grid < g_min) grid = g_min;
  a.rows_max = (O + grid - 1) / grid;
  int RB = 0, S = 0;
  if (!fe_config(a.R, a.d, a.H_i, a.rows_max, &RB, &S)) return cudaErrorInvalidConfiguration;
  a.stages = S;
  const size_t smem = fe_smem_map(RB, S, a.d, a.rows_max, a.H_i).total;
  switch (RB) {
    case 4: return launch_rb<4>(a, grid, smem, st);
    case 2: return launch_rb<2>(a, grid, smem, st);
    default: return launch_rb<1>(a, grid, smem, st);
  }
}

}  // namespace dsa
