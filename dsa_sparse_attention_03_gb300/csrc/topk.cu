// Exact ordered top-k of the indexer scores, per query row.
//
// "ds4 glm53-m3ultra" (page 1) replaced a selection that sorted and merged
// ever larger candidate lists with parallel scans that narrow the candidates,
// a sort of the small surviving list, and the original exact algorithm for the
// ambiguous cases -- keeping the same positions in the same order.  Here:
//
//   minmax   the range [umin, umax] of the row's order-preserving keys
//            u = s ^ 0x80000000 (merged by the indexer's epilogue in a decode
//            step; a separate scan for dsa_topk); the bits above the highest
//            bit where umin and umax differ are common to every key, so only
//            D = bitlen(umin ^ umax) bits remain to be searched.
//   pass x3  radix search for the k-th largest key T, 11 bits per pass, over
//            the positions still in the candidate bin (shared-memory histogram,
//            global merge, the row's last CTA picks the bin).  Rows finish in
//            ceil(D / 11) passes; the remaining launches return at once.
//   compact  every u > T is selected (unordered slots); positions with u == T
//            are counted per chunk.
//   ties     the r = k - #{u > T} lowest-index positions with u == T: each
//            chunk takes its share from the exclusive prefix of the counts and
//            writes its ties in index order (the exact fallback: it never
//            depends on how many positions tie).
//   rank     the <= k survivors are ordered by (score desc, position asc): the
//            rank of a survivor is the number of survivors whose 64-bit key
//            (u << 32 | ~position) is larger; keys are unique, so ranks are a
//            permutation and the order is exact.
// A row with row_len <= k selects every position; an empty row selects none.
// Nothing here waits on another CTA: cross-CTA steps use the last-arriving
// CTA of a row (fence + counter), and kernel boundaries.
#include "common.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 256;
constexpr int kRankPerBlock = 32;                    // survivors ranked per CTA
constexpr int kRankLanes = kThreads / kRankPerBlock; // threads per survivor

struct TopkArgs {
  const int32_t* scores;
  const int32_t* row_len;
  int32_t* idx;
  int32_t* nsel;
  RowState* state;
  uint32_t* hist;      // [R, kHistBins]
  uint32_t* tiecnt;    // [R, nchunk]
  uint64_t* sel;       // [R, k]
  int64_t L_max;
  int k, chunk;
};

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__device__ __forceinline__ uint64_t sel_key(uint32_t u, int t) {
  return (static_cast<uint64_t>(u) << 32) | static_cast<uint32_t>(0xFFFFFFFFu - (uint32_t)t);
}

template <typename T>
__device__ __forceinline__ T ld_volatile(const T* p) {
  return *reinterpret_cast<const volatile T*>(p);
}

// Block-wide max of two values (all threads get the result).
__device__ void block_max2(uint32_t& a, uint32_t& b) {
  __shared__ uint32_t sa[kThreads / 32], sb[kThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a = max(a, __shfl_xor_sync(0xffffffffu, a, o));
    b = max(b, __shfl_xor_sync(0xffffffffu, b, o));
  }
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (lane == 0) { sa[w] = a; sb[w] = b; }
  __syncthreads();
  a = 0; b = 0;
  for (int i = 0; i < kThreads / 32; ++i) { a = max(a, sa[i]); b = max(b, sb[i]); }
  __syncthreads();
}

__device__ uint32_t block_sum(uint32_t v) {
  __shared__ uint32_t s[kThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (lane == 0) s[w] = v;
  __syncthreads();
  uint32_t t = 0;
  for (int i = 0; i < kThreads / 32; ++i) t += s[i];
  __syncthreads();
  return t;
}

// True in every thread of the CTA that arrives last at counter `c`.
__device__ bool last_arrival(uint32_t* c, uint32_t expected) {
  __shared__ int is_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = (atomicAdd(c, 1u) == expected - 1);
  __syncthreads();
  if (is_last) __threadfence();
  return is_last != 0;
}

__global__ void __launch_bounds__(kThreads) topk_minmax_kernel(TopkArgs a) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.y;
  const int len = a.row_len[r];
  const int start = blockIdx.x * a.chunk;
  const int end = min(start + a.chunk, len);
  const int32_t* s = a.scores + (int64_t)r * a.L_max;
  uint32_t umax = 0, uminv = 0;
  for (int t = start + threadIdx.x; t < end; t += kThreads) {
    const uint32_t u = ordered_key(s[t]);
    umax = max(umax, u);
    uminv = max(uminv, ~u);
  }
  row_minmax_flush(a.state + r, umax, uminv);
}

__global__ void __launch_bounds__(kThreads) topk_pass_kernel(TopkArgs a, int phase) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.y;
  RowState* st = a.state + r;
  const int len = a.row_len[r];
  uint32_t mode, shift, prefix, k_rem;
  if (phase == kPhasePass0) {
    // Initial state from the row's key range; every CTA derives the same.
    mode = len <= 0 ? 2u : (len <= a.k ? 1u : 0u);
    const uint32_t hi = st->umax, lo = ~st->uminv;
    const uint32_t diff = hi ^ lo;
    shift = (mode == 0 && diff) ? 32u - __clz(diff) : 0u;
    prefix = shift >= 32 ? 0u : (hi >> shift);
    k_rem = (uint32_t)a.k;
    if (mode != 0 || shift == 0) {
      // Nothing to search: the last CTA records the state for the next kernels.
      if (!last_arrival(&st->arrive[phase], gridDim.x) || threadIdx.x != 0) return;
      st->mode = mode;
      st->shift = 0;
      st->prefix = prefix;
      st->k_rem = k_rem;
      st->n_take = (uint32_t)min(a.k, max(len, 0));
      return;
    }
  } else {
    mode = st->mode;
    if (mode != 0) return;
    shift = st->shift;
    if (shift == 0) return;                     // threshold already exact
    prefix = st->prefix;
    k_rem = st->k_rem;                          // read before the last CTA rewrites it
  }
  const uint32_t bits = min(shift, (uint32_t)kHistBits);
  const uint32_t ns = shift - bits;
  const uint32_t mask = (1u << bits) - 1u;
  const int nbins = 1 << bits;

  __shared__ uint32_t h[kHistBins];
  for (int i = threadIdx.x; i < nbins; i += kThreads) h[i] = 0;
  __syncthreads();

  const int start = blockIdx.x * a.chunk;
  const int end = min(start + a.chunk, len);
  const int32_t* s = a.scores + (int64_t)r * a.L_max;
  for (int t = start + threadIdx.x; t < end; t += kThreads) {
    const uint32_t u = ordered_key(s[t]);
    if ((static_cast<uint64_t>(u) >> shift) == prefix) atomicAdd(&h[(u >> ns) & mask], 1u);
  }
  __syncthreads();
  uint32_t* gh = a.hist + (size_t)r * kHistBins;
  for (int i = threadIdx.x; i < nbins; i += kThreads)
    if (h[i]) atomicAdd(&gh[i], h[i]);

  if (!last_arrival(&st->arrive[phase], gridDim.x)) return;

  // Last CTA of the row: find the bin holding the k_rem-th largest candidate.
  // Thread i owns bins [i*per, (i+1)*per) counted from the top.
  constexpr int per = kHistBins / kThreads;
  uint32_t local[per];
  uint32_t sum = 0;
#pragma unroll
  for (int j = 0; j < per; ++j) {
    const int bin = nbins - 1 - (threadIdx.x * per + j);
    local[j] = bin >= 0 ? ld_volatile(&gh[bin]) : 0u;
    sum += local[j];
  }
  // exclusive scan of `sum` over threads (top bins first)
  __shared__ uint32_t wsum[kThreads / 32];
  uint32_t v = sum;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) wsum[w] = v;
  __syncthreads();
  uint32_t above = v - sum;
  for (int i = 0; i < w; ++i) above += wsum[i];
  if (above < k_rem && above + sum >= k_rem) {
    uint32_t acc = above;
#pragma unroll
    for (int j = 0; j < per; ++j) {
      const int bin = nbins - 1 - (threadIdx.x * per + j);
      if (acc + local[j] >= k_rem) {
        st->k_rem = k_rem - acc;
        st->prefix = (prefix << bits) | (uint32_t)bin;
        st->shift = ns;
        if (phase == kPhasePass0) {
          st->mode = 0;
          st->n_take = (uint32_t)a.k;
        }
        break;
      }
      acc += local[j];
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < nbins; i += kThreads) gh[i] = 0;  // ready for the next pass
}

__global__ void __launch_bounds__(kThreads) topk_compact_kernel(TopkArgs a) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.y;
  RowState* st = a.state + r;
  const uint32_t mode = st->mode;
  if (mode == 2) return;
  const uint32_t T = st->prefix;       // exact threshold key (shift is 0 here)
  const int len = a.row_len[r];
  const int start = blockIdx.x * a.chunk;
  const int end = min(start + a.chunk, len);
  const int32_t* s = a.scores + (int64_t)r * a.L_max;
  uint64_t* sel = a.sel + (size_t)r * a.k;
  const int lane = threadIdx.x & 31;
  uint32_t ties = 0;
  for (int base = start; base < end; base += kThreads) {
    const int t = base + threadIdx.x;
    uint32_t u = 0;
    bool take = false;
    if (t < end) {
      u = ordered_key(s[t]);
      if (mode == 1 || u > T) take = true;
      else if (u == T) ++ties;
    }
    const uint32_t m = __ballot_sync(0xffffffffu, take);
    if (m) {
      uint32_t slot = 0;
      if (lane == 0) slot = atomicAdd(&st->n_gt, (uint32_t)__popc(m));
      slot = __shfl_sync(0xffffffffu, slot, 0);
      if (take) sel[slot + __popc(m & lanemask_lt())] = sel_key(u, t);
    }
  }
  if (mode == 0) {
    const uint32_t tot = block_sum(ties);
    if (threadIdx.x == 0) a.tiecnt[(size_t)r * gridDim.x + blockIdx.x] = tot;
  }
}

__global__ void __launch_bounds__(kThreads) topk_ties_kernel(TopkArgs a) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.y;
  RowState* st = a.state + r;
  if (st->mode != 0) return;
  const uint32_t k_rem = st->k_rem;
  const uint32_t* cnt = a.tiecnt + (size_t)r * gridDim.x;
  if (k_rem == 0 || cnt[blockIdx.x] == 0) return;
  uint32_t mine = 0;
  for (int c = threadIdx.x; c < (int)blockIdx.x; c += kThreads) mine += cnt[c];
  const uint32_t before = block_sum(mine);
  if (before >= k_rem) return;
  const uint32_t take = min(k_rem - before, cnt[blockIdx.x]);
  const uint32_t T = st->prefix;
  const int len = a.row_len[r];
  const int start = blockIdx.x * a.chunk;
  const int end = min(start + a.chunk, len);
  const int32_t* s = a.scores + (int64_t)r * a.L_max;
  uint64_t* out = a.sel + (size_t)r * a.k + (a.k - k_rem) + before;

  __shared__ uint32_t wcnt[kThreads / 32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  uint32_t done = 0;
  for (int base = start; base < end && done < take; base += kThreads) {
    const int t = base + threadIdx.x;
    const bool tie = t < end && ordered_key(s[t]) == T;
    const uint32_t m = __ballot_sync(0xffffffffu, tie);
    if (lane == 0) wcnt[w] = __popc(m);
    __syncthreads();
    uint32_t pos = done + __popc(m & lanemask_lt());
    uint32_t total = 0;
    for (int i = 0; i < kThreads / 32; ++i) {
      if (i < w) pos += wcnt[i];
      total += wcnt[i];
    }
    if (tie && pos < take) out[pos] = sel_key(T, t);
    done += total;
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kThreads) topk_rank_kernel(TopkArgs a) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.y;
  RowState* st = a.state + r;
  const int n = st->mode == 2 ? 0 : (int)st->n_take;
  extern __shared__ uint64_t keys[];
  const uint64_t* sel = a.sel + (size_t)r * a.k;
  for (int i = threadIdx.x; i < n; i += kThreads) keys[i] = sel[i];
  __syncthreads();
  int32_t* idx = a.idx + (size_t)r * a.k;
  const int e = blockIdx.x * kRankPerBlock + threadIdx.x / kRankLanes;
  const int part = threadIdx.x % kRankLanes;
  const uint64_t key = e < n ? keys[e] : 0;
  uint32_t rank = 0;
  if (e < n)
    for (int j = part; j < n; j += kRankLanes) rank += keys[j] > key;
#pragma unroll
  for (int o = kRankLanes / 2; o > 0; o >>= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
  if (e < n && part == 0) idx[rank] = (int32_t)(0xFFFFFFFFu - (uint32_t)key);
  if (threadIdx.x < kRankPerBlock) {
    const int p = blockIdx.x * kRankPerBlock + threadIdx.x;
    if (p >= n && p < a.k) idx[p] = -1;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0 && a.nsel) a.nsel[r] = n;
}

}  // namespace

cudaError_t launch_topk(const dsa_problem& p, const Plan& pl, const int32_t* scores,
                        int32_t* idx, int32_t* nsel, char* ws, cudaStream_t st, bool minmax_done) {
  TopkArgs a;
  a.scores = scores;
  a.row_len = p.row_len;
  a.idx = idx;
  a.nsel = nsel;
  a.state = reinterpret_cast<RowState*>(ws + pl.off_state);
  a.hist = reinterpret_cast<uint32_t*>(ws + pl.off_hist);
  a.tiecnt = reinterpret_cast<uint32_t*>(ws + pl.off_tiecnt);
  a.sel = reinterpret_cast<uint64_t*>(ws + pl.off_sel);
  a.L_max = pl.L_max;
  a.k = pl.k;
  a.chunk = pl.chunk;
  const dim3 grid(pl.nchunk, pl.R), block(kThreads);
  cudaError_t e;
  if (!minmax_done && (e = launch_pdl(topk_minmax_kernel, grid, block, 0, st, a)) != cudaSuccess) return e;
  if ((e = launch_pdl(topk_pass_kernel, grid, block, 0, st, a, (int)kPhasePass0)) != cudaSuccess) return e;
  if ((e = launch_pdl(topk_pass_kernel, grid, block, 0, st, a, (int)kPhasePass1)) != cudaSuccess) return e;
  if ((e = launch_pdl(topk_pass_kernel, grid, block, 0, st, a, (int)kPhasePass2)) != cudaSuccess) return e;
  if ((e = launch_pdl(topk_compact_kernel, grid, block, 0, st, a)) != cudaSuccess) return e;
  if ((e = launch_pdl(topk_ties_kernel, grid, block, 0, st, a)) != cudaSuccess) return e;
  const size_t smem = (size_t)pl.k * 8;
  e = cudaFuncSetAttribute(topk_rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const dim3 rgrid((pl.k + kRankPerBlock - 1) / kRankPerBlock, pl.R);
  return launch_pdl(topk_rank_kernel, rgrid, block, smem, st, a);
}

}  // namespace dsa
