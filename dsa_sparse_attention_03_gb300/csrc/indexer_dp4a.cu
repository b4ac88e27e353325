// Lightning indexer on CUDA cores: int8 dot products with dp4a.
//
// s[r, t] = sum_h w[r, h] * max(0, q_idx[r, h, :] . k_idx[offsets[b] + t, :])
// ("ds4 glm53-m3ultra", page 1: every cached position is scored against the
// current query).  Exact in int32 (the host bounds the value ranges).
//
// Work: tiles of 128*KPT consecutive positions inside one request.  A thread
// keeps KPT keys in registers (16-byte non-coherent loads) and reuses them for
// every row of the request; the row's queries sit in shared memory and are read
// as 16-byte broadcasts, one per four dp4a.
#include "common.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 128;

struct IdxArgs {
  const int8_t* q_idx;
  const int32_t* w_idx;
  const int8_t* k_idx;
  const int32_t* offsets;
  const int32_t* row_offsets;
  const int32_t* row_len;
  int32_t* scores;
  int64_t L_max;
  int B, H_i;
  int relu;
  int total_tiles_bound;
  uint4* zero;          // workspace words to clear (status + top-k state)
  int n_zero;
  RowState* rows;       // per-row key range for the top-k
};

// Exclusive prefix of per-request tile counts into tile_start[0..B], by one block.
__device__ void tile_prefix(const int32_t* offsets, int B, int tile, int* tile_start) {
  __shared__ int warp_sums[kThreads / 32];
  const int per = (B + kThreads - 1) / kThreads;
  const int lo = threadIdx.x * per;
  int local = 0;
  for (int b = lo; b < lo + per && b < B; ++b) {
    const int len = offsets[b + 1] - offsets[b];
    local += (len + tile - 1) / tile;
  }
  // inclusive scan over threads
  int v = local;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_sums[wid] = v;
  __syncthreads();
  int base = 0;
  for (int w = 0; w < wid; ++w) base += warp_sums[w];
  int run = base + v - local;  // exclusive start of this thread's range
  for (int b = lo; b < lo + per && b < B; ++b) {
    tile_start[b] = run;
    const int len = offsets[b + 1] - offsets[b];
    run += (len + tile - 1) / tile;
  }
  if (threadIdx.x == kThreads - 1) tile_start[B] = run;
  __syncthreads();
}

__device__ __forceinline__ int find_request(const int* tile_start, int B, int g) {
  int lo = 0, hi = B - 1;  // largest b with tile_start[b] <= g
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tile_start[mid] <= g) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <int D_I, int KPT>
__global__ void __launch_bounds__(kThreads) indexer_dp4a_kernel(IdxArgs a) {
  constexpr int W = D_I / 4;          // 32-bit words per key
  constexpr int TILE = kThreads * KPT;
  extern __shared__ __align__(16) unsigned char smem[];
  int* tile_start = reinterpret_cast<int*>(smem);                       // [B+1]
  const size_t ts_bytes = ((size_t)(a.B + 1) * 4 + 15) / 16 * 16;
  int4* q_s = reinterpret_cast<int4*>(smem + ts_bytes);                  // [H_i * D_I / 16]
  int* w_s = reinterpret_cast<int*>(smem + ts_bytes + (size_t)a.H_i * D_I);

  pdl_wait();
  for (int i = blockIdx.x * kThreads + threadIdx.x; i < a.n_zero; i += gridDim.x * kThreads)
    a.zero[i] = make_uint4(0, 0, 0, 0);
  tile_prefix(a.offsets, a.B, TILE, tile_start);
  const int total = tile_start[a.B];
  int cached_row = -1;  // row whose q/w are in shared memory

  for (int g = blockIdx.x; g < total; g += gridDim.x) {
    const int b = find_request(tile_start, a.B, g);
    const int t0 = (g - tile_start[b]) * TILE;
    const int64_t base = a.offsets[b];
    const int L_b = a.offsets[b + 1] - a.offsets[b];
    const int r0 = a.row_offsets[b], r1 = a.row_offsets[b + 1];

    // Keys of this thread, kept for all rows of the request.
    int key[KPT][W];
#pragma unroll
    for (int kk = 0; kk < KPT; ++kk) {
      const int t = t0 + kk * kThreads + threadIdx.x;
      if (t < L_b) {
        const int4* src = reinterpret_cast<const int4*>(a.k_idx + (base + t) * D_I);
#pragma unroll
        for (int j = 0; j < W / 4; ++j) {
          const int4 v = __ldg(src + j);
          key[kk][4 * j + 0] = v.x; key[kk][4 * j + 1] = v.y;
          key[kk][4 * j + 2] = v.z; key[kk][4 * j + 3] = v.w;
        }
      } else {
#pragma unroll
        for (int j = 0; j < W; ++j) key[kk][j] = 0;
      }
    }

    for (int r = r0; r < r1; ++r) {
      const int len = a.row_len[r];
      if (t0 >= len) continue;
      if (r != cached_row) {
        __syncthreads();  // previous row's q_s / w_s no longer in use
        const int4* qsrc = reinterpret_cast<const int4*>(a.q_idx + (size_t)r * a.H_i * D_I);
        for (int i = threadIdx.x; i < a.H_i * D_I / 16; i += kThreads) q_s[i] = qsrc[i];
        for (int i = threadIdx.x; i < a.H_i; i += kThreads) w_s[i] = a.w_idx[(size_t)r * a.H_i + i];
        __syncthreads();
        cached_row = r;
      }

      int acc[KPT];
#pragma unroll
      for (int kk = 0; kk < KPT; ++kk) acc[kk] = 0;
      for (int h = 0; h < a.H_i; ++h) {
        const int4* qh = q_s + h * (D_I / 16);
        int d[KPT];
#pragma unroll
        for (int kk = 0; kk < KPT; ++kk) d[kk] = 0;
#pragma unroll
        for (int j = 0; j < W / 4; ++j) {
          const int4 qv = qh[j];
#pragma unroll
          for (int kk = 0; kk < KPT; ++kk) {
            d[kk] = __dp4a(key[kk][4 * j + 0], qv.x, d[kk]);
            d[kk] = __dp4a(key[kk][4 * j + 1], qv.y, d[kk]);
            d[kk] = __dp4a(key[kk][4 * j + 2], qv.z, d[kk]);
            d[kk] = __dp4a(key[kk][4 * j + 3], qv.w, d[kk]);
          }
        }
        const int wh = w_s[h];
#pragma unroll
        for (int kk = 0; kk < KPT; ++kk) acc[kk] += wh * (a.relu ? max(d[kk], 0) : d[kk]);
      }
      int32_t* out = a.scores + (int64_t)r * a.L_max;
      uint32_t umax = 0, uminv = 0;
#pragma unroll
      for (int kk = 0; kk < KPT; ++kk) {
        const int t = t0 + kk * kThreads + threadIdx.x;
        if (t < len) {
          out[t] = acc[kk];
          const uint32_t u = ordered_key(acc[kk]);
          umax = max(umax, u);
          uminv = max(uminv, ~u);
        }
      }
      row_minmax_flush(a.rows + r, umax, uminv);
    }
  }
  pdl_trigger();
}

template <int D_I, int KPT>
cudaError_t launch(const dsa_problem& p, const Plan& pl, int32_t* scores, char* ws, cudaStream_t st) {
  constexpr int TILE = kThreads * KPT;
  IdxArgs a;
  a.q_idx = p.q_idx; a.w_idx = p.w_idx; a.k_idx = p.k_idx;
  a.offsets = p.offsets; a.row_offsets = p.row_offsets; a.row_len = p.row_len;
  a.scores = scores; a.L_max = p.L_max; a.B = p.B; a.H_i = p.H_i;
  a.relu = (p.flags & DSA_FLAG_NO_RELU) ? 0 : 1;
  a.zero = reinterpret_cast<uint4*>(ws);
  a.n_zero = pl.fused_row ? (int)(pl.zero_end / 16) : 0;   // else cleared before the launch
  a.rows = reinterpret_cast<RowState*>(ws + pl.off_state);
  const int64_t bound = p.L_total / TILE + p.B;
  a.total_tiles_bound = (int)bound;
  const size_t ts_bytes = ((size_t)(p.B + 1) * 4 + 15) / 16 * 16;
  const size_t smem = ts_bytes + (size_t)p.H_i * D_I + (size_t)p.H_i * 4;
  cudaError_t e = cudaFuncSetAttribute(indexer_dp4a_kernel<D_I, KPT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t grid = bound < int64_t(sms) * 16 ? bound : int64_t(sms) * 16;
  if (grid < 1) grid = 1;
  return launch_pdl(indexer_dp4a_kernel<D_I, KPT>, dim3((unsigned)grid), dim3(kThreads), smem, st, a);
}

}  // namespace

cudaError_t launch_indexer_dp4a(const dsa_problem& p, const Plan& pl, int32_t* scores, char* ws,
                                cudaStream_t st) {
  switch (p.D_i) {
    case 32: return launch<32, 2>(p, pl, scores, ws, st);
    case 64: return launch<64, 2>(p, pl, scores, ws, st);
    case 128: return launch<128, 2>(p, pl, scores, ws, st);
    default: return launch<256, 1>(p, pl, scores, ws, st);
  }
}

}  // namespace dsa
