// Exact ordered top-k of the indexer scores, per query row.
//
// "ds4 glm53-m3ultra" (page 1) replaced a selection that sorted and merged
// ever larger candidate lists with parallel scans that narrow the candidates,
// a sort of the small surviving list, and the original exact algorithm for the
// ambiguous cases -- keeping the same positions in the same order.  Here, with
// u = s ^ 0x80000000 the order-preserving unsigned key of a score s, one
// persistent kernel over a co-resident (cooperatively launched) grid runs the
// phases, separated by bounded grid barriers:
//
//   range   (standalone calls only) the row's key range [umin, umax]; a
//           decode step has it already, merged by the indexer's epilogue.
//   hist    a histogram of 2048 equal-width bins over [umin, umax]:
//           bin(u) = (u - umin) >> shift with the smallest shift that fits.
//           Each chunk of a row is binned in shared memory and added into
//           one of the row's hist_rep global copies.
//   select  each CTA sums the copies of the rows it serves and finds the
//           threshold bin b*: fewer than k positions lie above it, at least
//           k at or above it.  Every position whose bin is >= b* joins the
//           row's survivor list (unordered slots): the n_above sure winners
//           plus the bin's candidates, a few thousand at long context.
//   rank    each survivor's rank is the number of survivors with a larger
//           64-bit key (u << 32 | ~position).  Keys are unique, so the ranks
//           are a permutation and sort by (score desc, position asc); a
//           survivor with rank < k is written at idx[rank].  This spreads one
//           row's O(U^2) comparisons over many CTAs; once the rows alone fill
//           the grid (R >= kSortRows) each CTA instead sorts whole rows'
//           survivor keys (bitonic, O(U log^2 U)) and writes the first k.
//   exact fallback  when the survivor list would exceed kCapFast (heavy ties
//           at the threshold), one CTA resolves the row exactly: the
//           candidates' key range, radix passes to the exact k-th key T,
//           every key > T plus the lowest-index positions with key == T in
//           index order, then a bitonic sort.
// A row with row_len <= k selects every position; an empty row selects none.
#include "common.cuh"
#include "ptx.cuh"
#include "select.cuh"

namespace dsa {
namespace {

using namespace sel;

constexpr int kThreads = 512;
constexpr int kRankSlice = 16;                             // survivors ranked per work unit
constexpr int kRankLanes = kThreads / kRankSlice;          // threads per survivor
constexpr int kRankSlices = kCapFast / kRankSlice;         // units per row (also covers idx[0, k))
static_assert(kRankSlices * kRankSlice >= kMaxK, "rank units must cover idx");
constexpr int kSortRows = kTopkSortRows;                   // rank by per-row sort from this many rows

enum Mode : uint32_t { kFast = 0, kAll = 1, kEmpty = 2, kExact = 3 };

struct TopkArgs {
  const int32_t* scores;
  const int32_t* row_len;
  int32_t* idx;
  int32_t* nsel;
  RowState* state;
  uint32_t* hist;      // [R, hist_rep, kBuckets]
  uint64_t* surv;      // [R, kCapFast] survivor keys
  uint32_t* status;    // device status word
  uint32_t* bar;       // grid barrier counters (zeroed with the status block)
  int64_t L_max;
  int R, k, chunk, nchunk, hist_rep, range;
  uint64_t wait_ns;    // grid barrier limit
  int skip_cta;        // test hook: this CTA returns before its first grid barrier (-1: none)
  unsigned char* pair_x;   // [R][pair_x_bytes(k)] exchange buffers of the two-CTA exact fallback, or null
  uint32_t* pair_c;        // [R][kPairPhases] its barrier counters (zeroed with the status block)
};

// Equal-width bins over the row's key range: bin(u) = (u - umin) >> shift,
// monotone in u and below kBuckets.
struct Bins {
  uint32_t umin, shift;
  __device__ __forceinline__ explicit Bins(const RowState* st) {
    const uint32_t hi = st->umax, lo = ~st->uminv;
    const uint32_t range = hi >= lo ? hi - lo : 0u;
    const int bl = range ? 32 - __clz(range) : 0;
    umin = lo;
    shift = (uint32_t)max(0, bl - kBucketBits);
  }
  // (The clamps only guard memory and keep the bins monotone: every key of the
  // row lies in [umin, umax].)
  __device__ __forceinline__ uint32_t operator()(uint32_t u) const {
    return u < umin ? 0u : min((u - umin) >> shift, (uint32_t)(kBuckets - 1));
  }
};


// ------------------------------------------------------------------ exact fallback

// One CTA (or, with part >= 0, part `part` of a pair of CTAs) resolves a row
// exactly: the candidates are the positions in bucket b*; k - n_above of them
// are taken.  Part 0 (or the single CTA) writes idx.
__device__ void exact_row(const TopkArgs& a, RowState* st, int r, uint64_t* keys, int part = -1) {
  const int len = a.row_len[r];
  const int32_t* s = a.scores + (int64_t)r * a.L_max;
  const uint32_t bstar = st->bstar;
  const Bins bin(st);
  PairX px;
  if (part >= 0) {
    px.part = part;
    px.xb = a.pair_x + (size_t)r * pair_x_bytes(a.k);
    px.xc = a.pair_c + (size_t)r * kPairPhases;
    px.wait_ns = a.wait_ns;
  }
  exact_row_keys<kThreads>(s, len, a.k, (uint32_t)a.k - st->n_above,
                           [&](uint32_t u) { return bin(u) == bstar; }, keys, a.status, part >= 0 ? &px : nullptr);
  if (part > 0) return;
  int32_t* idx = a.idx + (size_t)r * a.k;
  for (int j = threadIdx.x; j < a.k; j += kThreads) idx[j] = key_pos(keys[j]);
}

// ------------------------------------------------------------------ the kernel

// The selection parameters of row r, from its merged histogram (every thread
// gets the same values).  h: kBuckets words of shared memory.
struct RowPick {
  uint32_t mode, bstar, above, cand, n_take;
};
__device__ RowPick row_pick(const TopkArgs& a, int r, uint32_t* h, uint32_t* res) {
  RowPick p;
  const int len = a.row_len[r];
  if (len <= a.k) {
    p.mode = len <= 0 ? kEmpty : kAll;
    p.n_take = (uint32_t)max(len, 0);
    p.bstar = p.above = p.cand = 0;
    return p;
  }
  const uint32_t* gh = a.hist + (size_t)r * a.hist_rep * kBuckets;
  __syncthreads();   // h may still be read by the previous pick
  for (int i = threadIdx.x; i < kBuckets; i += kThreads) {
    uint32_t c = 0;
    for (int j = 0; j < a.hist_rep; ++j) c += gh[(size_t)j * kBuckets + i];
    h[i] = c;
  }
  __syncthreads();
  find_crossing<kThreads>(h, kBuckets, (uint32_t)a.k, res);
  p.bstar = res[0];
  p.above = res[1];
  p.cand = h[p.bstar];
  p.n_take = (uint32_t)a.k;
  p.mode = (p.above + p.cand <= (uint32_t)kCapFast) ? kFast : kExact;
  return p;
}

__global__ void __launch_bounds__(kThreads, 1) topk_kernel(TopkArgs a) {
  extern __shared__ uint64_t keys[];   // [max(kCapFast, pow2 >= k)]: ranks / exact fallback
  __shared__ uint32_t h[kBuckets];
  __shared__ uint32_t res[2];
  __shared__ uint32_t wt[2 * kThreads / 32];
  __shared__ uint32_t slot0;
  pdl_wait();
  pdl_trigger();
  const int nunits = a.R * a.nchunk;
  int nb = 0;
  if ((int)blockIdx.x == a.skip_cta) return;   // test hook: an arrival that never comes

  // ---- range (standalone call): the row's max key and max complemented key.
  if (a.range) {
    for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
      const int r = u / a.nchunk, c = u % a.nchunk;
      const int len = a.row_len[r];
      const int start = c * a.chunk, end = min(start + a.chunk, len);
      uint32_t umax = 0, uminv = 0;
      scan_row<kThreads>(a.scores + (int64_t)r * a.L_max, start, end, [&](int32_t v, int) {
        const uint32_t x = ordered_key(v);
        umax = max(umax, x);
        uminv = max(uminv, ~x);
      });
      block_reduce_max2<kThreads>(umax, uminv, wt);
      if (threadIdx.x == 0) {
        if (umax) atomicMax(&a.state[r].umax, umax);
        if (uminv) atomicMax(&a.state[r].uminv, uminv);
      }
    }
    if (!grid_barrier(a.bar + nb++, a.status, a.wait_ns)) return;
  }

  // ---- hist
  for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
    const int r = u / a.nchunk, c = u % a.nchunk;
    const int len = a.row_len[r];
    const int start = c * a.chunk, end = min(start + a.chunk, len);
    if (len <= a.k || start >= end) continue;
    for (int i = threadIdx.x; i < kBuckets; i += kThreads) h[i] = 0;
    __syncthreads();
    const Bins bin(a.state + r);
    scan_row<kThreads>(a.scores + (int64_t)r * a.L_max, start, end,
                       [&](int32_t v, int) { atomicAdd(&h[bin(ordered_key(v))], 1u); });
    __syncthreads();
    uint32_t* mine = a.hist + ((size_t)r * a.hist_rep + (size_t)(c % a.hist_rep)) * kBuckets;
    for (int i = threadIdx.x; i < kBuckets; i += kThreads)
      if (h[i]) atomicAdd(&mine[i], h[i]);
    __syncthreads();
  }
  if (!grid_barrier(a.bar + nb++, a.status, a.wait_ns)) return;

  // ---- select
  {
    int cur = -1;
    RowPick pk;
    pk.mode = kEmpty;
    pk.bstar = 0;
    constexpr int U = 4;
    for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
      const int r = u / a.nchunk, c = u % a.nchunk;
      RowState* st = a.state + r;
      const int len = a.row_len[r];
      const int start = c * a.chunk, end = min(start + a.chunk, len);
      const int32_t* s = a.scores + (int64_t)r * a.L_max;
      const Bins bin(st);
      // The first sweep's scores are loaded before the threshold is known.
      int32_t v[U];
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const int t = start + j * kThreads + (int)threadIdx.x;
        v[j] = t < end ? s[t] : 0;
      }
      if (r != cur) {
        pk = row_pick(a, r, h, res);
        cur = r;
      }
      if (c == 0 && threadIdx.x == 0) {
        st->mode = pk.mode;
        st->bstar = pk.bstar;
        st->n_above = pk.above;
        st->cand = pk.cand;
        st->n_take = pk.n_take;
      }
      if (pk.mode != kFast && pk.mode != kAll) continue;
      uint64_t* surv = a.surv + (size_t)r * kCapFast;
      // U positions per thread per sweep; the CTA claims its slots with one
      // atomic (per-warp atomics on n_union would serialise).
      for (int base = start; base < end; base += U * kThreads) {
        uint32_t take = 0;
#pragma unroll
        for (int j = 0; j < U; ++j) {
          const int t = base + j * kThreads + (int)threadIdx.x;
          if (base != start) v[j] = t < end ? s[t] : 0;
          if (t < end && (pk.mode == kAll || bin(ordered_key(v[j])) >= pk.bstar)) take |= 1u << j;
        }
        const uint32_t cnt = (uint32_t)__popc(take);
        const uint32_t incl = block_scan_incl<kThreads>(cnt, wt);
        if (threadIdx.x == kThreads - 1) slot0 = incl ? atomicAdd(&st->n_union, incl) : 0u;
        __syncthreads();
        uint32_t slot = slot0 + incl - cnt;
#pragma unroll
        for (int j = 0; j < U; ++j)
          if (take & (1u << j))
            surv[slot++] = surv_key(ordered_key(v[j]), base + j * kThreads + (int)threadIdx.x);
        __syncthreads();
      }
    }
  }
  if (!grid_barrier(a.bar + nb++, a.status, a.wait_ns)) return;

  // ---- rank by sort: whole rows per CTA (many rows).
  if (a.R >= kSortRows) {
    // With two CTAs per row, CTA R + r is the second part of row r's exact
    // fallback (and idle otherwise).
    const bool pairs = a.pair_x != nullptr && 2 * a.R <= (int)gridDim.x;
    if (pairs && (int)blockIdx.x >= a.R) {
      const int r = (int)blockIdx.x - a.R;
      if (r < a.R && a.state[r].mode == kExact) exact_row(a, a.state + r, r, keys, 1);
      return;
    }
    for (int r = blockIdx.x; r < a.R; r += gridDim.x) {
      RowState* st = a.state + r;
      const uint32_t mode = st->mode;
      const int n_take = mode == kEmpty ? 0 : (int)st->n_take;
      int32_t* idx = a.idx + (size_t)r * a.k;
      if (threadIdx.x == 0 && a.nsel) a.nsel[r] = n_take;
      if (mode == kExact) {
        exact_row(a, st, r, keys, pairs ? 0 : -1);
        __syncthreads();
        continue;
      }
      const int U = mode == kEmpty ? 0 : (int)min(st->n_union, (uint32_t)kCapFast);
      const uint64_t* surv = a.surv + (size_t)r * kCapFast;
      __syncthreads();   // keys may still be read by the previous row
      for (int i = threadIdx.x; i < U; i += kThreads) keys[i] = surv[i];
      __syncthreads();
      if (U > 1) sort_desc<kThreads>(keys, U);
      for (int j = threadIdx.x; j < a.k; j += kThreads) idx[j] = j < n_take && j < U ? key_pos(keys[j]) : -1;
    }
    return;
  }

  // ---- rank: units (row, slice of kRankSlice survivors), one warp per
  // survivor.  Units go out in runs of `run` consecutive units, run c to CTA
  // c % grid: with one row the few active slices land on different CTAs; with
  // many rows a CTA's runs stay within a row, which it loads once per run.
  const int nr = a.R * kRankSlices;
  const int run = max(1, nr / (4 * (int)gridDim.x));
  int loaded = -1;
  for (int c = (int)blockIdx.x; (int64_t)c * run < nr; c += (int)gridDim.x)
  for (int u = c * run; u < min(nr, (c + 1) * run); ++u) {
    const int r = u / kRankSlices, sl = u % kRankSlices;
    RowState* st = a.state + r;
    const uint32_t mode = st->mode;
    const int n_take = mode == kEmpty ? 0 : (int)st->n_take;
    int32_t* idx = a.idx + (size_t)r * a.k;
    if (sl == 0 && threadIdx.x == 0 && a.nsel) a.nsel[r] = n_take;
    if (mode == kExact) {
      if (sl == 0) {
        exact_row(a, st, r, keys);
        loaded = -1;
      }
      continue;
    }
    if (threadIdx.x < kRankSlice) {
      const int p = sl * kRankSlice + threadIdx.x;
      if (p >= n_take && p < a.k) idx[p] = -1;
    }
    if (mode == kEmpty) continue;
    const int U = (int)st->n_union;
    if (sl * kRankSlice >= U) continue;
    if (loaded != r) {
      __syncthreads();
      const uint64_t* surv = a.surv + (size_t)r * kCapFast;
      for (int i = threadIdx.x; i < U; i += kThreads) keys[i] = surv[i];
      __syncthreads();
      loaded = r;
    }
    const int e = sl * kRankSlice + (int)threadIdx.x / kRankLanes;
    const int part = (int)threadIdx.x % kRankLanes;
    const uint64_t key = e < U ? keys[e] : ~0ull;
    uint32_t rank = 0;
    if (e < U)
      for (int j = part; j < U; j += kRankLanes) rank += keys[j] > key;
#pragma unroll
    for (int o = kRankLanes / 2; o > 0; o >>= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
    if (e < U && part == 0 && rank < (uint32_t)n_take) idx[rank] = key_pos(key);
  }
}

}  // namespace

cudaError_t launch_topk(const dsa_problem& p, const Plan& pl, const int32_t* scores,
                        int32_t* idx, int32_t* nsel, char* ws, cudaStream_t st, bool minmax_done,
                        const TestHooks* hooks) {
  TopkArgs a;
  const TestHooks none;
  if (!hooks) hooks = &none;
  a.wait_ns = hooks->wait_ns;
  a.skip_cta = hooks->topk_skip_cta;
  a.scores = scores;
  a.row_len = p.row_len;
  a.idx = idx;
  a.nsel = nsel;
  a.state = reinterpret_cast<RowState*>(ws + pl.off_state);
  a.hist = reinterpret_cast<uint32_t*>(ws + pl.off_hist);
  a.surv = reinterpret_cast<uint64_t*>(ws + pl.off_surv);
  a.status = reinterpret_cast<uint32_t*>(ws + pl.off_status);
  a.bar = a.status + kBarrierWord;
  a.pair_x = pl.off_pairx ? reinterpret_cast<unsigned char*>(ws + pl.off_pairx) : nullptr;
  a.pair_c = reinterpret_cast<uint32_t*>(ws + pl.off_pairc);
  a.L_max = pl.L_max;
  a.R = pl.R;
  a.k = pl.k;
  a.chunk = pl.chunk;
  a.nchunk = pl.nchunk;
  a.hist_rep = pl.hist_rep;
  a.range = minmax_done ? 0 : 1;
  int n = 1;
  while (n < pl.k) n <<= 1;
  const size_t smem = (size_t)(n > kCapFast ? n : kCapFast) * 8;
  cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0, per_sm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, topk_kernel, kThreads, smem)) != cudaSuccess)
    return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  // One CTA per SM: enough for every phase, and always co-resident.
  int grid = sms;
  const int most = pl.R * (pl.nchunk > kRankSlices ? pl.nchunk : kRankSlices);
  if (grid > most) grid = most;
  return launch_coop(topk_kernel, dim3(grid), dim3(kThreads), smem, st, a);
}

}  // namespace dsa
