// Block-level building blocks of the exact ordered top-k, shared by the top-k
// kernel and the single-row decode kernel.  Keys: u = s ^ 0x80000000 is the
// order-preserving unsigned key of an int32 score s; a survivor's 64-bit key
// (u << 32 | ~position) orders by (score desc, position asc) when sorted
// descending, and is never zero.
#pragma once

#include "common.cuh"
#include "ptx.cuh"

namespace dsa {
namespace sel {

constexpr int kRadixBits = 11;

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Visits s[t] for t in [begin, end) with `t += NT` striding, eight loads in
// flight per thread; f(value, t) is called in increasing t for each thread.
template <int NT, typename F>
__device__ __forceinline__ void scan_row(const int32_t* s, int begin, int end, F f) {
  constexpr int U = 8;
  for (int base = begin + (int)threadIdx.x; base < end; base += U * NT) {
    int32_t v[U];
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const int t = base + j * NT;
      v[j] = t < end ? s[t] : 0;
    }
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const int t = base + j * NT;
      if (t < end) f(v[j], t);
    }
  }
}

// The same visit with 16-byte loads (U = 8 in flight per thread): a scalar
// head up to the first 16-byte boundary, aligned chunks of four, a scalar
// tail.  f(value, t) sees every t in [begin, end) once, in no fixed order.
template <int NT, typename F>
__device__ __forceinline__ void scan_row_v(const int32_t* s, int begin, int end, F f) {
  constexpr int U = 8;
  const int mis = (int)((reinterpret_cast<uintptr_t>(s + begin) >> 2) & 3);
  const int a0 = min(end, begin + ((4 - mis) & 3));
  for (int t = begin + (int)threadIdx.x; t < a0; t += NT) f(s[t], t);
  const int nch = (end - a0) >> 2;
  const int4* c4 = reinterpret_cast<const int4*>(s + a0);
  for (int cb = (int)threadIdx.x; cb < nch; cb += U * NT) {
    int4 v[U];
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const int c = cb + j * NT;
      v[j] = c < nch ? c4[c] : make_int4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const int c = cb + j * NT;
      if (c < nch) {
        const int t = a0 + 4 * c;
        f(v[j].x, t);
        f(v[j].y, t + 1);
        f(v[j].z, t + 2);
        f(v[j].w, t + 3);
      }
    }
  }
  for (int t = a0 + 4 * nch + (int)threadIdx.x; t < end; t += NT) f(s[t], t);
}

__device__ __forceinline__ uint64_t surv_key(uint32_t u, int t) {
  return (static_cast<uint64_t>(u) << 32) | static_cast<uint32_t>(0xFFFFFFFFu - (uint32_t)t);
}
__device__ __forceinline__ int key_pos(uint64_t key) {
  return (int)(0xFFFFFFFFu - (uint32_t)key);
}

// Block-wide inclusive scan in thread order (NT threads).
template <int NT>
__device__ uint32_t block_scan_incl(uint32_t v, uint32_t* warp_tot) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_tot[w] = v;
  __syncthreads();
  uint32_t base = lane < w ? warp_tot[lane] : 0u;   // the totals of the warps before this one
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) base += __shfl_xor_sync(0xffffffffu, base, o);
  __syncthreads();
  return base + v;
}

// Block-wide maxima of two values at once (NT threads); tmp holds 2 NT / 32
// words.
template <int NT>
__device__ void block_reduce_max2(uint32_t& a, uint32_t& b, uint32_t* tmp) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a = max(a, __shfl_xor_sync(0xffffffffu, a, o));
    b = max(b, __shfl_xor_sync(0xffffffffu, b, o));
  }
  if (lane == 0) {
    tmp[w] = a;
    tmp[NW + w] = b;
  }
  __syncthreads();
  a = lane < NW ? tmp[lane] : 0u;
  b = lane < NW ? tmp[NW + lane] : 0u;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a = max(a, __shfl_xor_sync(0xffffffffu, a, o));
    b = max(b, __shfl_xor_sync(0xffffffffu, b, o));
  }
  __syncthreads();
}

// Finds, in a histogram of `nbins` counts held in shared memory, the bin b
// (counting from the top) with above(b) < need <= above(b) + h[b].  Writes
// (b, above) to out[0..1].  Every thread of the NT-thread block takes part.
template <int NT>
__device__ void find_crossing(const uint32_t* h, int nbins, uint32_t need, uint32_t* out) {
  __shared__ uint32_t wt[NT / 32];
  const int per = (nbins + NT - 1) / NT;
  const int top = nbins - 1 - threadIdx.x * per;   // this thread owns bins top, top-1, ...
  uint32_t sum = 0;
  for (int j = 0; j < per; ++j)
    if (top - j >= 0) sum += h[top - j];
  const uint32_t incl = block_scan_incl<NT>(sum, wt);
  uint32_t above = incl - sum;
  if (above < need && incl >= need) {
    for (int j = 0; j < per; ++j) {
      const uint32_t c = h[top - j];
      if (above + c >= need) {
        out[0] = (uint32_t)(top - j);
        out[1] = above;
        break;
      }
      above += c;
    }
  }
  __syncthreads();
}

// Bitonic sort, descending, of keys[0, n) in shared memory (zero keys pad to a
// power of two; every real key is nonzero).  All threads of the CTA; ends
// with a barrier.
template <int NT>
__device__ void sort_desc(uint64_t* keys, int n0) {
  int n = 1;
  while (n < n0) n <<= 1;
  for (int i = n0 + threadIdx.x; i < n; i += NT) keys[i] = 0;
  __syncthreads();
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < (n >> 1); i += NT) {
        const int lo = ((i & ~(stride - 1)) << 1) | (i & (stride - 1)), hi = lo + stride;   // stride: a power of two
        const uint64_t x = keys[lo], y = keys[hi];
        const bool desc = (lo & size) == 0;
        if (desc ? (x < y) : (x > y)) {
          keys[lo] = y;
          keys[hi] = x;
        }
      }
      __syncthreads();
    }
  }
}

// One CTA resolves a row exactly.  The candidates are the positions whose
// ordered key u satisfies in_cand(u) (one histogram bin); every position with
// a key above the candidates' is taken, plus the k_rem largest candidates, the
// lowest positions first among equal keys.  Radix passes over the candidates'
// key range find the exact k_rem-th largest candidate key T.  The ties at T
// are counted per block of positions; the block where the count reaches k_rem
// is numbered in position order to find the last tie taken; one more pass
// writes the winners (keys above T, ties up to that position), which are
// sorted into keys[0, k) by (score desc, position asc).  keys holds at least
// the next power of two >= k entries.  The count of keys above the candidates
// comes from the caller's histogram; a key beyond k (a histogram that does not
// match the scores) is not written and raises DSA_DEVICE_CAPACITY in *status.
// All NT threads of the CTA take part; ends with a barrier.
//
// With a pair (px != nullptr), two co-resident CTAs resolve the row together:
// part 0 takes the tie blocks [0, ceil(nblk / 2)), part 1 the rest, for every
// pass over the row, and they exchange their partial results through a global
// buffer at each step (key range, radix histograms, tie counts per block, the
// last tie taken, part 1's winners), each exchange behind a two-CTA barrier.
// Part 0 ends with the sorted keys; part 1's keys are not meaningful.  A
// barrier that runs out raises DSA_DEVICE_TIMEOUT and both parts return early
// (the result is then unspecified).
constexpr int kTieBlocks = 32;
struct PairX {
  int part;                // 0 or 1
  unsigned char* xb;       // kPairXBytes of global memory for this row
  uint32_t* xc;            // kPairPhases barrier counters for this row, zero at the start
  uint64_t wait_ns;
};
static_assert((1 << kRadixBits) == 2048 && kTieBlocks == 32, "the pair exchange layout (common.cuh)");

template <int NT, class InCand>
__device__ __noinline__ void exact_row_keys(const int32_t* s, int len, int k, uint32_t k_rem, InCand in_cand,
                                            uint64_t* keys, uint32_t* status, const PairX* px = nullptr) {
  __shared__ uint32_t h[1 << kRadixBits];
  __shared__ uint32_t tmp[2 * NT / 32];
  __shared__ uint32_t res[2];
  __shared__ uint32_t n_list;
  __shared__ uint32_t tie8[8 * (NT / 32)];
  __shared__ uint32_t wcnt[NT / 32][kTieBlocks];
  __shared__ uint32_t cut[2];
  __shared__ int pstar;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  // Tie blocks of 2^lb positions (at most kTieBlocks); a pair splits the row
  // at a block boundary.
  int lb = 12;
  while ((int64_t(1) << lb) * kTieBlocks < (int64_t)len) ++lb;
  const int nblk = (int)((len + (int64_t(1) << lb) - 1) >> lb);
  const int mid = (int)min((int64_t)len, (int64_t)((nblk + 1) / 2) << lb);
  const int r0 = px ? (px->part ? mid : 0) : 0, r1 = px ? (px->part ? len : mid) : len;
  int phase = 0;
  auto exchange = [&]() { return group_barrier(px->xc + phase++, 2u, status, px->wait_ns); };
  uint32_t* xw = px ? reinterpret_cast<uint32_t*>(px->xb) : nullptr;

  // Key range of the candidates.
  uint32_t umax = 0, uminv = 0;
  scan_row_v<NT>(s, r0, r1, [&](int32_t v, int) {
    const uint32_t u = ordered_key(v);
    if (in_cand(u)) {
      umax = max(umax, u);
      uminv = max(uminv, ~u);
    }
  });
  block_reduce_max2<NT>(umax, uminv, tmp);
  if (px) {
    if (threadIdx.x == 0) {
      __stcg(xw + 2 * px->part, umax);
      __stcg(xw + 2 * px->part + 1, uminv);
    }
    if (!exchange()) return;
    umax = max(__ldcg(xw), __ldcg(xw + 2));
    uminv = max(__ldcg(xw + 1), __ldcg(xw + 3));
  }
  const uint32_t diff = umax ^ ~uminv;
  uint32_t shift = diff ? 32u - __clz(diff) : 0u;
  uint32_t prefix = shift >= 32 ? 0u : (umax >> shift);

  // Radix passes down to the exact k_rem-th largest candidate key T.
  while (shift > 0) {
    const uint32_t bits = min(shift, (uint32_t)kRadixBits);
    const uint32_t ns = shift - bits;
    const int nb = 1 << bits;
    for (int i = threadIdx.x; i < nb; i += NT) h[i] = 0;
    __syncthreads();
    scan_row_v<NT>(s, r0, r1, [&](int32_t v, int) {
      const uint32_t u = ordered_key(v);
      if (in_cand(u) && (static_cast<uint64_t>(u) >> shift) == prefix)
        atomicAdd(&h[(u >> ns) & (uint32_t)(nb - 1)], 1u);
    });
    __syncthreads();
    if (px) {   // buffer (pass mod 2): the other part has read the older one
      uint32_t* hx = reinterpret_cast<uint32_t*>(px->xb + kPairHistOff) + (size_t)((phase & 1) * 2) * (1 << kRadixBits);
      for (int i = threadIdx.x; i < nb; i += NT) __stcg(hx + (size_t)px->part * (1 << kRadixBits) + i, h[i]);
      if (!exchange()) return;
      for (int i = threadIdx.x; i < nb; i += NT) h[i] = __ldcg(hx + i) + __ldcg(hx + (1 << kRadixBits) + i);
      __syncthreads();
    }
    find_crossing<NT>(h, nb, k_rem, res);
    k_rem -= res[1];
    prefix = (prefix << bits) | res[0];
    shift = ns;
    __syncthreads();
  }
  const uint32_t T = prefix;

  // Ties at T per block of 2^lb positions; each thread visits its positions
  // in increasing order and adds its count when it moves to another block
  // (into its warp's own counters).
  for (int i = threadIdx.x; i < (NT / 32) * kTieBlocks; i += NT) (&wcnt[0][0])[i] = 0;
  if (threadIdx.x == 0) {
    n_list = 0;
    pstar = -1;
  }
  __syncthreads();
  if (k_rem > 0) {
    int cb = -1;
    uint32_t cnt = 0;
    scan_row_v<NT>(s, r0, r1, [&](int32_t v, int t) {
      if (ordered_key(v) == T) {
        const int b = t >> lb;
        if (b != cb) {
          if (cnt) atomicAdd(&wcnt[w][cb], cnt);
          cb = b;
          cnt = 0;
        }
        ++cnt;
      }
    });
    if (cnt) atomicAdd(&wcnt[w][cb], cnt);
  }
  __syncthreads();
  if (px) {   // per-block totals of both parts (each block is counted by one part)
    uint32_t* tx = reinterpret_cast<uint32_t*>(px->xb + kPairTieOff);
    if (threadIdx.x < kTieBlocks) {
      uint32_t tb = 0;
      for (int ww = 0; ww < NT / 32; ++ww) tb += wcnt[ww][threadIdx.x];
      __stcg(tx + px->part * kTieBlocks + threadIdx.x, tb);
    }
    if (!exchange()) return;
    if (threadIdx.x < kTieBlocks) {
      wcnt[0][threadIdx.x] = __ldcg(tx + threadIdx.x) + __ldcg(tx + kTieBlocks + threadIdx.x);
      for (int ww = 1; ww < NT / 32; ++ww) wcnt[ww][threadIdx.x] = 0;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {   // the block holding the k_rem-th tie, and the ties before it
    uint32_t run = 0;
    int cbk = nblk;
    for (int b = 0; b < nblk && k_rem > 0; ++b) {
      uint32_t tb = 0;
      for (int ww = 0; ww < NT / 32; ++ww) tb += wcnt[ww][b];
      if (run + tb >= k_rem) {
        cbk = b;
        break;
      }
      run += tb;
    }
    cut[0] = (uint32_t)cbk;
    cut[1] = run;
  }
  __syncthreads();
  const int cbk = (int)cut[0];
  if (cbk < nblk && (!px || ((cbk << lb) >= mid) == (px->part == 1))) {   // (a pair: the block's owner)
    // Number the ties of that block in position order: position t = base0 +
    // j * NT + thread, so (j, warp, lane) order; the need-th one is the last
    // tie taken.
    const int lo = cbk << lb, hi = (int)min((int64_t)len, (int64_t)(cbk + 1) << lb);
    const uint32_t need = k_rem - cut[1];
    uint32_t before = 0;
    for (int base0 = lo; base0 < hi; base0 += 8 * NT) {
      uint32_t tm[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int t = base0 + j * NT + threadIdx.x;
        const bool tie = t < hi && ordered_key(s[t]) == T;
        tm[j] = __ballot_sync(0xffffffffu, tie);
        if (lane == 0) tie8[j * (NT / 32) + w] = __popc(tm[j]);
      }
      __syncthreads();
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t tot = 0, mine = 0;
        for (int i = 0; i < NT / 32; ++i) {
          const uint32_t c = tie8[j * (NT / 32) + i];
          if (i < w) mine += c;
          tot += c;
        }
        if (tm[j] & (1u << lane)) {
          const uint32_t pos = before + mine + __popc(tm[j] & lanemask_lt());
          if (pos + 1 == need) pstar = base0 + j * NT + threadIdx.x;
        }
        before += tot;
      }
      __syncthreads();   // tie8 is rewritten next
    }
  }
  __syncthreads();
  if (px && cbk < nblk) {   // the block's owner passes on the last tie taken
    const bool owner = ((cbk << lb) >= mid) == (px->part == 1);
    if (owner && threadIdx.x == 0) __stcg(reinterpret_cast<int*>(xw) + 4, pstar);
    if (!exchange()) return;
    if (threadIdx.x == 0) pstar = __ldcg(reinterpret_cast<const int*>(xw) + 4);
    __syncthreads();
  }
  const int ps = pstar;

  // Winners: every key above T, and the ties at or before position ps; slots
  // are reserved once per group of lanes that found one.
  const uint32_t lt = lanemask_lt();
  scan_row_v<NT>(s, r0, r1, [&](int32_t v, int t) {
    const uint32_t u = ordered_key(v);
    if (u > T || (u == T && t <= ps)) {
      const uint32_t m = __activemask();
      const int leader = __ffs(m) - 1;
      uint32_t base = 0;
      if (lane == leader) base = atomicAdd(&n_list, (uint32_t)__popc(m));
      base = __shfl_sync(m, base, leader);
      const uint32_t slot = base + __popc(m & lt);
      if (slot < (uint32_t)k) keys[slot] = surv_key(u, t);
      else raise_status(status, DSA_DEVICE_CAPACITY);
    }
  });
  __syncthreads();
  if (px) {   // part 1's winners join part 0's
    uint64_t* wx = reinterpret_cast<uint64_t*>(px->xb + kPairWinOff);
    const uint32_t mine = min(n_list, (uint32_t)k);
    if (px->part == 1) {
      for (uint32_t i = threadIdx.x; i < mine; i += NT) __stcg(wx + i, keys[i]);
      if (threadIdx.x == 0) __stcg(xw + 5, mine);
    }
    if (!exchange()) return;
    if (px->part == 1) return;
    const uint32_t other = __ldcg(xw + 5);
    for (uint32_t i = threadIdx.x; i < other; i += NT) {
      if (mine + i < (uint32_t)k) keys[mine + i] = __ldcg(wx + i);
      else raise_status(status, DSA_DEVICE_CAPACITY);
    }
    __syncthreads();
  }
  sort_desc<NT>(keys, k);
}

}  // namespace sel
}  // namespace dsa
