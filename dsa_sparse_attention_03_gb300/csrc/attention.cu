// Sparse MLA attention over the selected latent rows, split along the selected
// positions, then a fixed-order log-sum-exp merge of the splits.
//
// For query row r and head h ("ds4 glm53-m3ultra", page 1: attention over the
// ~2048 selected positions only; latent cache of "glm53-tensorfold-spark",
// page 4: key = the whole D_k-wide latent row, value = its first D_v columns):
//   z_j = scale * q[r,h,:] . kv[idx_j, :],  o[h,:] = sum_j softmax(z)_j kv[idx_j, :D_v]
//
// attn_split_kernel  grid (split, head group of 16, row), 4 warps.  Per tile of
//   64 selected positions: gather the rows (16-byte cp.async, whole rows, as the
//   front-axis gather of "GLM-5.3-Flash-Alis-MLX-4bit", page 3), S = Q K^T and
//   O += P V with bf16 mma.sync (fp32 accumulation), online softmax in fp32
//   (log2 domain).  Writes unnormalised O, the running max m and sum l.
// attn_combine_kernel  grid (head, row): merges the splits in split order and
//   rounds to bf16 (nearest even).
#include "common.cuh"

#include <cuda_bf16.h>
#include <math_constants.h>

namespace dsa {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kPStride = kAttnRows + 8;  // bf16 elements per P row in shared memory

struct AttnArgs {
  const uint16_t* q;
  const uint16_t* kv;
  const int32_t* offsets;
  const int32_t* row_offsets;
  const int32_t* row_len;
  const int32_t* idx;
  const int32_t* nsel;
  float* part;        // [R, nsplit, H_q, D_v]
  float* ml;          // [R, nsplit, H_q, 2]
  uint16_t* out;      // [R, H_q, D_v]
  float* lse;         // [R, H_q] or null
  uint32_t* status;
  int B, H_q, D_k, D_v, k, nsplit, tiles_per_split;
  int qs, ks;         // shared-memory row strides (elements)
  float scale_log2;
};

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

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src));
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;\n" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ int row_request(const int32_t* row_offsets, int B, int r) {
  int lo = 0, hi = B - 1;  // largest b with row_offsets[b] <= r
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (row_offsets[mid] <= r) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// NT: output n-tiles (of 8 columns) per warp; the 4 warps cover 32*NT >= D_v columns.
template <int NT>
__global__ void __launch_bounds__(kThreads) attn_split_kernel(AttnArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  uint16_t* Qs = reinterpret_cast<uint16_t*>(smem);                          // [16][qs]
  uint16_t* Ks = Qs + kAttnHeads * a.qs;                                    // [64][ks]
  uint16_t* Ps = Ks + kAttnRows * a.ks;                                     // [16][kPStride]
  float* red = reinterpret_cast<float*>(Ps + kAttnHeads * kPStride);        // [2][4][16]
  int* idx_s = reinterpret_cast<int*>(red + 2 * kWarps * kAttnHeads);       // [64]
  __shared__ int req_s;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int r = blockIdx.z, h0 = blockIdx.y * kAttnHeads, split = blockIdx.x;

  pdl_wait();
  pdl_trigger();
  if (tid == 0) req_s = row_request(a.row_offsets, a.B, r);
  __syncthreads();
  const int b = req_s;
  const int64_t base = a.offsets[b];
  const int L_b = a.offsets[b + 1] - a.offsets[b];
  int n = a.nsel ? a.nsel[r] : min(a.k, a.row_len[r]);
  n = max(0, min(n, a.k));
  const int ntiles = (n + kAttnRows - 1) / kAttnRows;
  const int t_begin = split * a.tiles_per_split;
  const int t_end = min(t_begin + a.tiles_per_split, ntiles);

  // Queries of this head group (zero rows past H_q).
  const int qchunks = a.D_k / 8;
  for (int i = tid; i < kAttnHeads * qchunks; i += kThreads) {
    const int hh = i / qchunks, c8 = i % qchunks;
    uint16_t* dst = Qs + hh * a.qs + c8 * 8;
    if (h0 + hh < a.H_q)
      cp_async16(smem_u32(dst), a.q + ((int64_t)r * a.H_q + h0 + hh) * a.D_k + c8 * 8);
    else
      *reinterpret_cast<int4*>(dst) = make_int4(0, 0, 0, 0);
  }

  float acc[NT][4];
#pragma unroll
  for (int i = 0; i < NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  float m_run[2] = {-CUDART_INF_F, -CUDART_INF_F};
  float l_run[2] = {0.f, 0.f};
  const int32_t* idx_row = a.idx + (int64_t)r * a.k;

  for (int tile = t_begin; tile < t_end; ++tile) {
    const int pos0 = tile * kAttnRows;
    if (tid < kAttnRows) {
      const int p = pos0 + tid;
      int t = -1;
      if (p < n) {
        t = idx_row[p];
        if (t < 0 || t >= L_b) {
          raise_status(a.status, DSA_DEVICE_BAD_INDEX);
          t = -1;
        }
      }
      idx_s[tid] = t;
    }
    __syncthreads();
    for (int i = tid; i < kAttnRows * qchunks; i += kThreads) {
      const int j = i / qchunks, c8 = i % qchunks;
      uint16_t* dst = Ks + j * a.ks + c8 * 8;
      const int t = idx_s[j];
      if (t >= 0)
        cp_async16(smem_u32(dst), a.kv + (base + t) * a.D_k + c8 * 8);
      else
        *reinterpret_cast<int4*>(dst) = make_int4(0, 0, 0, 0);
    }
    cp_async_wait_all();
    __syncthreads();

    // S = Q K^T for kv rows [warp*16, warp*16+16).
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
      const int arow = (lane & 7) + ((lane >> 3) & 1) * 8, acol = (lane >> 4) * 8;
      const int brow = warp * 16 + (lane & 7) + (lane >> 4) * 8, bcol = ((lane >> 3) & 1) * 8;
      const uint32_t aaddr = smem_u32(Qs + arow * a.qs + acol);
      const uint32_t baddr = smem_u32(Ks + brow * a.ks + bcol);
      for (int kk = 0; kk < a.D_k / 16; ++kk) {
        uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
        ldsm_x4(aaddr + kk * 32, a0, a1, a2, a3);
        ldsm_x4(baddr + kk * 32, b0, b1, b2, b3);
        mma16816(s[0], a0, a1, a2, a3, b0, b1);
        mma16816(s[1], a0, a1, a2, a3, b2, b3);
      }
    }
    // Online softmax (rows g and g+8 of the head group; columns of this warp).
    float x[2][4];
    float mx[2] = {-CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int col = warp * 16 + nt * 8 + 2 * c + (e & 1);
        const float v = idx_s[col] >= 0 ? s[nt][e] * a.scale_log2 : -CUDART_INF_F;
        x[nt][e] = v;
        mx[e >> 1] = fmaxf(mx[e >> 1], v);
      }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 1));
      mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 2));
    }
    float* red_max = red;
    float* red_sum = red + kWarps * kAttnHeads;
    if (c == 0) {
      red_max[warp * kAttnHeads + g] = mx[0];
      red_max[warp * kAttnHeads + g + 8] = mx[1];
    }
    __syncthreads();
    float m_new[2], alpha[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      float tm = -CUDART_INF_F;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) tm = fmaxf(tm, red_max[w * kAttnHeads + g + 8 * i]);
      m_new[i] = fmaxf(m_run[i], tm);
      alpha[i] = m_new[i] == -CUDART_INF_F ? 1.f : exp2f(m_run[i] - m_new[i]);
    }
    float ps[2] = {0.f, 0.f};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      float p[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float mm = m_new[e >> 1];
        p[e] = (x[nt][e] == -CUDART_INF_F) ? 0.f : exp2f(x[nt][e] - mm);
        ps[e >> 1] += p[e];
      }
      const int col = warp * 16 + nt * 8 + 2 * c;
      *reinterpret_cast<uint32_t*>(Ps + g * kPStride + col) = pack_bf16(p[0], p[1]);
      *reinterpret_cast<uint32_t*>(Ps + (g + 8) * kPStride + col) = pack_bf16(p[2], p[3]);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      ps[i] += __shfl_xor_sync(0xffffffffu, ps[i], 1);
      ps[i] += __shfl_xor_sync(0xffffffffu, ps[i], 2);
    }
    if (c == 0) {
      red_sum[warp * kAttnHeads + g] = ps[0];
      red_sum[warp * kAttnHeads + g + 8] = ps[1];
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      float ts = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) ts += red_sum[w * kAttnHeads + g + 8 * i];
      l_run[i] = l_run[i] * alpha[i] + ts;
      m_run[i] = m_new[i];
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      acc[nt][0] *= alpha[0]; acc[nt][1] *= alpha[0];
      acc[nt][2] *= alpha[1]; acc[nt][3] *= alpha[1];
    }
    // O += P V for output columns [warp*8*NT, (warp+1)*8*NT).
    {
      const int arow = (lane & 7) + ((lane >> 3) & 1) * 8, acol = (lane >> 4) * 8;
      const uint32_t paddr = smem_u32(Ps + arow * kPStride + acol);
      const int vrow = (lane & 7) + ((lane >> 3) & 1) * 8, vcol = warp * 8 * NT + (lane >> 4) * 8;
      const uint32_t vaddr = smem_u32(Ks + vrow * a.ks + vcol);
#pragma unroll
      for (int ks = 0; ks < kAttnRows / 16; ++ks) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(paddr + ks * 32, a0, a1, a2, a3);
#pragma unroll
        for (int n2 = 0; n2 < NT / 2; ++n2) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vaddr + (ks * 16 * a.ks + n2 * 16) * 2, b0, b1, b2, b3);
          mma16816(acc[2 * n2], a0, a1, a2, a3, b0, b1);
          mma16816(acc[2 * n2 + 1], a0, a1, a2, a3, b2, b3);
        }
      }
    }
    __syncthreads();  // Ks / Ps / idx_s are rewritten by the next tile
  }

  cp_async_wait_all();  // an empty split still issued its query copies
  // Unnormalised partial output of this split.
  const int64_t prow = ((int64_t)r * a.nsplit + split) * a.H_q;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int h = h0 + g + 8 * i;
    if (h >= a.H_q) continue;
    float* dst = a.part + (prow + h) * a.D_v;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int col = warp * 8 * NT + nt * 8 + 2 * c;
      if (col < a.D_v)
        *reinterpret_cast<float2*>(dst + col) = make_float2(acc[nt][2 * i], acc[nt][2 * i + 1]);
    }
    if (warp == 0 && c == 0)
      *reinterpret_cast<float2*>(a.ml + (prow + h) * 2) = make_float2(m_run[i], l_run[i]);
  }
}

// One CTA per (head, row): warp 0 derives the split weights exp2(m_s - M) and
// 1/L in parallel; then every thread merges 4 columns over the splits, in
// split order, and rounds to bf16.
__global__ void __launch_bounds__(128) attn_combine_kernel(AttnArgs a) {
  pdl_wait();
  pdl_trigger();
  const int h = blockIdx.x, r = blockIdx.y;
  extern __shared__ float wts[];  // [nsplit]
  __shared__ float inv_l_s;
  const int lane = threadIdx.x & 31;
  const float2* ml = reinterpret_cast<const float2*>(a.ml) + ((int64_t)r * a.nsplit) * a.H_q + h;
  if (threadIdx.x < 32) {
    float M = -CUDART_INF_F;
    for (int s = lane; s < a.nsplit; s += 32) {
      const float2 v = ml[(int64_t)s * a.H_q];
      if (v.y > 0.f) M = fmaxf(M, v.x);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = 0.f;
    for (int s = lane; s < a.nsplit; s += 32) {
      const float2 v = ml[(int64_t)s * a.H_q];
      const float w = v.y > 0.f ? exp2f(v.x - M) : 0.f;
      wts[s] = w;
      L += w * v.y;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    if (lane == 0) {
      inv_l_s = L > 0.f ? 1.f / L : 0.f;
      if (a.lse) a.lse[(int64_t)r * a.H_q + h] = L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -CUDART_INF_F;
    }
  }
  __syncthreads();
  const float inv_l = inv_l_s;
  uint16_t* o = a.out + ((int64_t)r * a.H_q + h) * a.D_v;
  const float* part = a.part + (((int64_t)r * a.nsplit) * a.H_q + h) * a.D_v;
  const int64_t sstride = (int64_t)a.H_q * a.D_v;
  for (int col = threadIdx.x * 4; col < a.D_v; col += blockDim.x * 4) {
    // Every split wrote its partial (zeros when it saw no position), so the
    // loads are unconditional and eight of them are kept in flight.
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    int s = 0;
    for (; s + 8 <= a.nsplit; s += 8) {
      float4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = *reinterpret_cast<const float4*>(part + (s + j) * sstride + col);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float w = wts[s + j];
        x.x += w * v[j].x; x.y += w * v[j].y; x.z += w * v[j].z; x.w += w * v[j].w;
      }
    }
    for (; s < a.nsplit; ++s) {
      const float w = wts[s];
      const float4 v = *reinterpret_cast<const float4*>(part + s * sstride + col);
      x.x += w * v.x; x.y += w * v.y; x.z += w * v.z; x.w += w * v.w;
    }
    uint2 pk;
    pk.x = pack_bf16(x.x * inv_l, x.y * inv_l);
    pk.y = pack_bf16(x.z * inv_l, x.w * inv_l);
    *reinterpret_cast<uint2*>(o + col) = pk;
  }
}

template <int NT>
cudaError_t launch_split(const AttnArgs& a, dim3 grid, size_t smem, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(attn_split_kernel<NT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_split_kernel<NT>, grid, dim3(kThreads), smem, st, a);
}

}  // namespace

cudaError_t launch_attention(const dsa_problem& p, const Plan& pl, const int32_t* idx,
                             const int32_t* nsel, uint16_t* out, float* lse, char* ws,
                             cudaStream_t st) {
  AttnArgs a;
  a.q = p.q; a.kv = p.kv; a.offsets = p.offsets; a.row_offsets = p.row_offsets;
  a.row_len = p.row_len; a.idx = idx; a.nsel = nsel;
  a.part = reinterpret_cast<float*>(ws + pl.off_part);
  a.ml = reinterpret_cast<float*>(ws + pl.off_ml);
  a.out = out; a.lse = lse;
  a.status = reinterpret_cast<uint32_t*>(ws + pl.off_status);
  a.B = p.B; a.H_q = p.H_q; a.D_k = p.D_k; a.D_v = p.D_v; a.k = p.k;
  a.nsplit = pl.nsplit;
  const int tiles = (p.k + kAttnRows - 1) / kAttnRows;
  a.tiles_per_split = (tiles + pl.nsplit - 1) / pl.nsplit;
  a.scale_log2 = p.softmax_scale * 1.4426950408889634f;

  int NT = 2;
  while (NT * 32 < p.D_v) NT *= 2;            // 2, 4, 8 or 16
  const int cols = NT * 32;
  a.qs = p.D_k + 8;
  a.ks = (p.D_k > cols ? p.D_k : cols) + 8;
  const size_t smem = (size_t)kAttnHeads * a.qs * 2 + (size_t)kAttnRows * a.ks * 2 +
                      (size_t)kAttnHeads * kPStride * 2 + 2 * kWarps * kAttnHeads * 4 +
                      kAttnRows * 4;
  const dim3 grid(pl.nsplit, (p.H_q + kAttnHeads - 1) / kAttnHeads, p.R);
  cudaError_t e;
  switch (NT) {
    case 2: e = launch_split<2>(a, grid, smem, st); break;
    case 4: e = launch_split<4>(a, grid, smem, st); break;
    case 8: e = launch_split<8>(a, grid, smem, st); break;
    default: e = launch_split<16>(a, grid, smem, st); break;
  }
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_combine_kernel, dim3(p.H_q, p.R), dim3(128), (size_t)pl.nsplit * 4, st, a);
}

}  // namespace dsa
