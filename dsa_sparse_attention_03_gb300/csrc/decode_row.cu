// The decode step of one query row after its indexer scores: the exact ordered
// top-k and the sparse attention over the selected latent rows, in one
// cooperative kernel (one CTA per SM; one grid barrier, before the merge).
//
// "ds4 glm53-m3ultra" (page 1): parallel scans narrow the candidates, a small
// surviving list is sorted, the original exact algorithm settles ambiguous
// ties, and attention runs over the ~2048 selected positions only.  Here:
//
//   (indexer) its epilogue counts the row's scores into 8192 log-spaced bins
//      (score_bin: 128 per octave of |score|, monotone, independent of the
//      data) and adds them into one of eight copies of the row's histogram,
//      with their sums over coarse bins of 128.
//   P  every CTA sums the copies: warp 0 adds the coarse sums, which give
//      the coarse bin C* holding the k-th largest score; the fine bins of C*
//      and above (only the coarse bins that hold positions) are summed one
//      per thread and scanned one coarse bin per warp: E(b) = positions in
//      bins above b, and the bin b* of the k-th largest.  The histogram is
//      checked (its total is the row length, each coarse sum the sum of its
//      bins); if the indexer could not complete it, the CTAs rebuild it from
//      the scores (H).
//   S  if the bins >= b* hold at most 4096 positions, each CTA scatters its
//      positions in bins >= b* into bin order: position t of bin b goes to
//      slot E(b) + (arrival order within the bin).  No barrier follows: a
//      unit waits (bounded) for the slots of its own bins, and a survivor's
//      key is never 0.
//   R  attention unit u takes ranks [uP, uP + P) of the selection.  Its CTA
//      loads the slots of the bins holding those ranks and ranks the members
//      by their 64-bit keys (score desc, position asc): up to 64 members by
//      one warp's comparisons; more by a histogram of their exact scores
//      (the members above each score), equal scores ordered by position
//      within their group.  It writes idx[rank] for its ranks, and
//   A  gathers its P latent rows once (one bulk copy per row) for all 64
//      heads -- the queries arrived by tensor-map copies at the start -- :
//      S = Q K^T and O = P V on bf16 mma.sync with an fp32 softmax.  The
//      unit's O / l goes to the workspace as fp16 scaled by a power of two
//      (from its rows' largest value), in the accumulators' chunk order, with
//      the max m and sum l per head.                               barrier
//   M  CTA c merges output slices (a head, 256 columns) over the units:
//      weights exp2(m_u - M) l_u, divided by their sum, bf16; every sum in a
//      fixed order.
// When the bins >= b* hold more than 4096 positions (heavy ties at the
// threshold), CTA 0 selects the row exactly (radix passes to the k-th key,
// ties by position) into idx, and after one more barrier the units read their
// positions from idx.  The units partition the selection by rank, so the
// output is the same on every run.
//
// State kept across steps (Plan::off_lkeep): the indexer's clearing counter,
// reset here for the next step.  The bin cursors and survivor slots of S are
// cleared with the rest of the workspace's zero range by the indexer at the
// start of every step.
#include "common.cuh"
#include "ptx.cuh"
#include "select.cuh"

#include <cuda_fp16.h>

#include <cstring>
#include <math_constants.h>

namespace dsa {
namespace {

using namespace sel;

constexpr int kRowThreads = 512;
constexpr int kRowWarps = kRowThreads / 32;
constexpr int kRowHeads = 64;            // query heads: four groups of 16, one per four warps
constexpr int kCoarse = kLogCoarse;
constexpr int kMergeCols = 256;          // output columns per merge slice
constexpr int kRegScores = 4;            // scores per thread kept in registers (2048 per CTA)
constexpr int kSubRange = 2048;          // exact-score histogram of a unit's bins, at most
constexpr int kWindowList = 256;         // members whose rank may fall in a unit's window
static_assert(kLogBins == kRowThreads * 16, "P phase: 16 bins per thread");
static_assert(kCoarse == 64, "P phase: two coarse bins per lane of one warp");

enum RowMode : uint32_t { kRowEmpty = 0, kRowFast = 1, kRowExact = 2 };

__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
// A survivor slot, once its scatterer has written it (keys are never 0).
// Bounded: 0 and DSA_DEVICE_TIMEOUT once limit_ns have passed.
__device__ uint64_t wait_key(const uint64_t* p, uint32_t* status, uint64_t limit_ns) {
  uint64_t v = ld_relaxed_u64(p);
  if (v) return v;
  const uint64_t t0 = gtimer();
  while ((v = ld_relaxed_u64(p)) == 0) {
    if (gtimer() - t0 > limit_ns) {
      raise_status(status, DSA_DEVICE_TIMEOUT);
      return 0;
    }
  }
  return v;
}

struct RowArgs {
  const int32_t* scores;   // [L] the row's indexer scores
  const int32_t* row_len;  // [1]
  const uint16_t* q;       // bf16 [64, D_k]
  const uint16_t* kv;      // bf16 [L_total, D_k]; with f8, e4m3 bytes [L_total, D_k]
  const float* kv_scale;   // f8: per-row scales, or null (= 1)
  int f8;                  // the cache holds e4m3 codes with per-row scales (the kernel's F8)
  int32_t* idx;            // [k]
  int32_t* nsel;           // [1] or null
  uint16_t* out;           // bf16 [64, D_v]
  float* lse;              // [64] or null
  uint32_t* status;
  uint32_t* bar;           // grid barrier counters (zeroed by the indexer)
  uint32_t* hist;          // [kRowHistCopies][kRowHistWords]: the row's histogram, as partial
                           // copies filled by the indexer's epilogue, then kCoarse sums over 128 bins
  uint32_t* zcount;        // the indexer's clearing counter, reset here for the next step
  uint32_t* cnt;           // [kLogBins] bin cursors of S (cleared by the indexer)
  uint64_t* surv;          // [kCapFast] survivor keys in bin order
  __half* po;              // [units][64][32 NT] the unit's O / l of each head, times psc[u]
  float* pml;              // [units][64][2] the unit's max m and sum l of each head
  float* psc;              // [units] a power of two that puts the unit's values near 2^14
  int L1;                  // the request's length (L_total)
  int k, D_k, D_v, qs, ks;
  float scale_log2;
  uint64_t wait_ns;
  CUtensorMap qmap;        // q as [64 rows][D_k] bf16, boxes of 64 x 64 with the 128-byte swizzle
};

// Shared-memory layout (bytes), for P positions per unit.
struct RowSmem {
  uint32_t q, kb, hs, keys, sub, ss, pb, mls, wm, pos, f8s, scs, total;
  __host__ __device__ RowSmem(int P, int qs, int ks, bool f8) {
    q = 0;                                 // [D_k / 64][64 rows][128 B], 128-byte swizzled
    kb = q + kRowHeads * qs * 2;
    hs = kb + P * ks * 2;
    keys = hs + (kLogBins + kLogBins / 16) * 4;
    sub = keys + kCapFast * 8;
    ss = sub + (kSubRange + 4) * 4;
    pb = ss + 2 * kRowHeads * P * 4;
    mls = pb + kRowHeads * (P + 8) * 2;
    wm = mls + kRowHeads * 2 * 4;
    pos = wm + 2 * 256 * 4;
    f8s = (pos + (P + kWindowList + kCoarse) * 4 + 15) / 16 * 16;   // FP8 cache: [P][D_k] staged codes
    scs = f8s + P * qs;                                            // FP8 cache: [P] row scales
    total = f8 ? scs + P * 4 : f8s;
  }
};

// NT: output n-tiles of 8 columns per warp (four warps per head group cover
// 32 NT >= D_v columns; NT >= 4).  P: selected positions per attention unit
// (16 or 32).
//
// A unit's partial holds 32 NT columns per head (the columns from D_v on are
// padding), in chunks of 16 bytes: chunk c = (wq NG + ng) 4 + cq of a head
// holds columns wq 8 NT + (4 ng + t) 8 + 2 cq + {0, 1}, t = 0..3 (NG = NT / 4),
// the four n-tiles of one accumulator thread.  Each thread then stores 16
// bytes at a time and a warp's store fills whole 32-byte sectors.
template <int NT, int P, bool F8>
__global__ void __launch_bounds__(kRowThreads, 1) decode_row_kernel(const __grid_constant__ RowArgs a) {
  static_assert(NT >= 4 && NT % 4 == 0, "four n-tiles per partial chunk");
  constexpr int NG = NT / 4;
  constexpr int Dvp = 32 * NT;             // partial columns per head
  constexpr int NTILES = P / 8;            // n-tiles of S per head group
  constexpr int KP = 4 / NTILES;           // K parts of S per n-tile (4 warps per head group)
  static_assert(NTILES * KP == 4, "four warps per head group");
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem =   // the swizzled query boxes want 1024-byte alignment
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const RowSmem L(P, a.qs, a.ks, F8);
  uint16_t* Qs = reinterpret_cast<uint16_t*>(smem + L.q);      // [64][qs]
  uint16_t* Ks = reinterpret_cast<uint16_t*>(smem + L.kb);     // [P][ks]
  // hs: [kLogBins] counts, then E(b), one pad word after every 16 bins so that
  // a thread's 16 consecutive bins fall in distinct banks from its neighbours'.
  uint32_t* hs_raw = reinterpret_cast<uint32_t*>(smem + L.hs);
  auto HS = [&](int b) -> uint32_t& { return hs_raw[b + (b >> 4)]; };
  uint64_t* keys = reinterpret_cast<uint64_t*>(smem + L.keys); // [kCapFast]
  float* Ss = reinterpret_cast<float*>(smem + L.ss);           // [KP][64][P] parts of S
  uint16_t* Pb = reinterpret_cast<uint16_t*>(smem + L.pb);     // [64][P + 8] bf16 weights
  float* mls = reinterpret_cast<float*>(smem + L.mls);         // [64][2] m, l
  float* wm = reinterpret_cast<float*>(smem + L.wm);           // merge: weights / partial sums
  uint32_t* sub = reinterpret_cast<uint32_t*>(smem + L.sub);   // [kSubRange] exact-score counts
  int* pos_s = reinterpret_cast<int*>(smem + L.pos);           // [P]
  uint8_t* F8s = smem + L.f8s;                                  // FP8 cache: [P][D_k] staged codes
  float* scs = reinterpret_cast<float*>(smem + L.scs);          // FP8 cache: [P] row scales
  int* wlist = pos_s + P;                                       // [kWindowList] member indices
  uint32_t* coarse_s = reinterpret_cast<uint32_t*>(wlist + kWindowList);   // [kCoarse]
  uint32_t* cab = sub + kRowThreads;                            // [kCoarse] positions above each coarse bin
  __shared__ __align__(8) uint64_t bars[2];                     // queries, latent rows
  __shared__ uint32_t sh[8];                                    // b*, E(b*), |b*|, mode, C*, total, ...
  __shared__ uint32_t wt[2 * kRowWarps];
  __shared__ float red[kRowWarps];
  __shared__ int key_lost;                                      // a survivor slot's wait ran out

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = (int)gridDim.x, cta = (int)blockIdx.x;
  const uint32_t bar_q = smem_u32(&bars[0]), bar_k = smem_u32(&bars[1]);
  const uint32_t qrow = (uint32_t)a.D_k * 2;

  if (tid == 0) {
    key_lost = 0;
    mbar_init(bar_q, 1);
    mbar_init(bar_k, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // The queries are an input of the step that none of its kernels writes, so
  // their copy (D_k / 64 tensor-map boxes of 64 x 64) starts before the wait
  // for the indexer.
  if (tid == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&a.qmap)) : "memory");
    mbar_expect_tx(bar_q, kRowHeads * qrow);
    for (int bx = 0; bx < a.D_k / 64; ++bx)
      asm volatile(
          "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
          ::"r"(smem_u32(Qs) + bx * 8192u), "l"(reinterpret_cast<uint64_t>(&a.qmap)), "r"(bx * 64), "r"(0),
            "r"(bar_q)
          : "memory");
  }
  bool q_done = false;
  // Leaves the kernel after a wait ran out: the copies still in flight land
  // first (bounded), and the next step rebuilds nothing from this one.
  auto bail = [&]() {
    if (tid == 0 && !q_done) mbar_wait(bar_q, 0, nullptr, a.wait_ns);
    __syncthreads();
  };

  // Parameters read right after the wait, fetched into the constant cache
  // while the previous kernel finishes (each asm forces the read here).
  asm volatile("" ::"l"(a.scores), "l"(a.row_len), "l"(a.kv), "l"(a.idx), "l"(a.hist), "l"(a.cnt),
               "l"(a.surv), "l"(a.po), "l"(a.pml), "r"(a.L1), "r"(a.k), "r"(a.D_k), "r"(a.ks), "l"(a.wait_ns));
  pdl_wait();
  pdl_trigger();
  const int len = max(0, min(a.row_len[0], a.L1));
  const int n_take = min(a.k, len);
  int chunk = (len + G - 1) / G;
  chunk = (chunk + 3) & ~3;
  const int c0 = min(len, cta * chunk), c1 = min(len, c0 + chunk);

  // This CTA's scores stay in registers from here to S (the first
  // kRegScores * 512; the rest are re-read).
  int32_t sreg[kRegScores];
#pragma unroll
  for (int j = 0; j < kRegScores; ++j) {
    const int t = c0 + j * kRowThreads + tid;
    sreg[j] = t < c1 ? a.scores[t] : 0;
  }
  const int c_reg = min(c1, c0 + kRegScores * kRowThreads);
  if (cta == 0 && tid == 0) *a.zcount = 0;   // the next step's indexer counts from zero

  // ---- P: the coarse bin C* holding the n_take-th largest score (one warp),
  // then E(b) = positions in bins above b for every bin of C* and above --
  // only the coarse bins that hold positions are read -- and b* within C*.
  // The histogram is checked (its total is the row length, each coarse sum
  // the sum of its bins); if the indexer could not complete it, it is rebuilt
  // here from the scores (H) and read again.
  uint32_t bstar = 0, n_above = 0, mode = kRowEmpty;
  for (int attempt = 0;; ++attempt) {
    if (warp == 0) {   // the coarse sums of all copies, loaded and summed by one warp
      if (lane < 8) sh[lane] = 0;
      const int ch = kCoarse - 1 - 2 * lane;   // this lane's coarse bins ch, ch - 1 (top down)
      uint32_t vh[kRowHistCopies], vl[kRowHistCopies];
#pragma unroll
      for (int cp = 0; cp < kRowHistCopies; ++cp) {
        vh[cp] = __ldcg(a.hist + (size_t)cp * kRowHistWords + kLogBins + ch);
        vl[cp] = __ldcg(a.hist + (size_t)cp * kRowHistWords + kLogBins + ch - 1);
      }
      uint32_t n_hi = 0, n_lo = 0;
#pragma unroll
      for (int cp = 0; cp < kRowHistCopies; ++cp) {
        n_hi += vh[cp];
        n_lo += vl[cp];
      }
      __syncwarp();   // sh is cleared before any lane sets it
      coarse_s[ch] = n_hi;
      coarse_s[ch - 1] = n_lo;
      uint32_t incl = n_hi + n_lo;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const uint32_t above = incl - n_hi - n_lo;
      cab[ch] = above;   // positions in the coarse bins above ch
      cab[ch - 1] = above + n_hi;
      if (above < (uint32_t)n_take && above + n_hi >= (uint32_t)n_take) sh[4] = (uint32_t)ch;
      else if (above + n_hi < (uint32_t)n_take && incl >= (uint32_t)n_take) sh[4] = (uint32_t)(ch - 1);
      if (lane == 31) sh[5] = incl;   // all positions counted
      // The nonempty coarse bins at or above C*, top down, for the fine loads.
      const int cstar = n_take > 0 ? (int)sh[4] : kCoarse;
      const uint32_t m_hi = __ballot_sync(0xffffffffu, n_hi != 0 && ch >= cstar);
      const uint32_t m_lo = __ballot_sync(0xffffffffu, n_lo != 0 && ch - 1 >= cstar);
      // order: lane 0 hi, lane 0 lo, lane 1 hi, ...
      const uint32_t before = __popc(m_hi & ((1u << lane) - 1)) + __popc(m_lo & ((1u << lane) - 1));
      if (n_hi != 0 && ch >= cstar) wlist[before] = ch;
      if (n_lo != 0 && ch - 1 >= cstar) wlist[before + (n_hi != 0 && ch >= cstar)] = ch - 1;
      if (lane == 0) sh[6] = __popc(m_hi) + __popc(m_lo);
    }
    __syncthreads();
    const int fb_lo = n_take > 0 ? (int)(sh[4] << 7) : kLogBins;   // lowest bin read
    {   // fine bins of those coarse bins: each thread sums one bin over the copies
      const int nb = (int)sh[6] * 128;
      for (int i = tid; i < nb; i += kRowThreads) {
        const int b = wlist[i >> 7] * 128 + (i & 127);
        uint32_t v[kRowHistCopies];
#pragma unroll
        for (int cp = 0; cp < kRowHistCopies; ++cp) v[cp] = __ldcg(a.hist + (size_t)cp * kRowHistWords + b);
        uint32_t sum = 0;
#pragma unroll
        for (int cp = 0; cp < kRowHistCopies; ++cp) sum += v[cp];
        HS(b) = sum;
      }
    }
    __syncthreads();
    {
      // E(b) for every bin of the coarse bins C* and above: the positions in
      // the coarse bins above b's plus those in the bins above b within it.
      // One warp per coarse bin, four bins per lane (top down); each coarse
      // bin's fine counts must add up to its coarse sum.
      const int cstar = fb_lo >> 7;
      for (int c = kCoarse - 1 - warp; c >= cstar; c -= kRowWarps) {
        const int b0 = c * 128 + 127 - 4 * lane;   // this lane's bins b0, ..., b0 - 3
        uint32_t v[4] = {0u, 0u, 0u, 0u};
        const uint32_t cs = coarse_s[c];
        if (cs != 0) {
#pragma unroll
          for (int j = 0; j < 4; ++j) v[j] = HS(b0 - j);
        }
        const uint32_t s4 = (v[0] + v[1]) + (v[2] + v[3]);
        uint32_t incl = s4;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t n = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += n;
        }
        if (lane == 31 && incl != cs) sh[7] = 1;
        uint32_t above = cab[c] + incl - s4;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          HS(b0 - j) = above;
          if (above < (uint32_t)n_take && above + v[j] >= (uint32_t)n_take) {
            sh[0] = (uint32_t)(b0 - j);
            sh[1] = above;
            sh[2] = v[j];
            sh[3] = above + v[j] <= (uint32_t)kCapFast ? kRowFast : kRowExact;
          }
          above += v[j];
        }
      }
      if (tid == 0 && cstar > 0 && cstar < kCoarse) HS(fb_lo - 1) = cab[cstar] + coarse_s[cstar];   // all bins read
    }
    __syncthreads();
    if (sh[5] == (uint32_t)len && sh[7] == 0) {
      bstar = sh[0];
      n_above = sh[1];
      mode = n_take == 0 ? kRowEmpty : sh[3];
      break;
    }
    if (attempt > 0) {   // a histogram built here must add up
      if (tid == 0) raise_status(a.status, DSA_DEVICE_CAPACITY);
      return bail();
    }
    // ---- H: clear the histogram, then each CTA adds its scores' counts.
    for (int i = cta * kRowThreads + tid; i < (int)(kRowHistCopies * kRowHistWords); i += G * kRowThreads)
      a.hist[i] = 0;
    if (!grid_barrier(a.bar + 3, a.status, a.wait_ns)) return bail();
    for (int i = tid; i < kLogBins; i += kRowThreads) HS(i) = 0;
    if (tid < kCoarse) coarse_s[tid] = 0;
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kRegScores; ++j)
      if (c0 + j * kRowThreads + tid < c1) atomicAdd(&HS(score_bin(sreg[j])), 1u);
    scan_row<kRowThreads>(a.scores, c_reg, c1, [&](int32_t v, int) { atomicAdd(&HS(score_bin(v)), 1u); });
    __syncthreads();
    for (int i = tid; i < kLogBins; i += kRowThreads) {   // a warp covers 32 bins of one coarse bin
      const uint32_t n = HS(i);
      if (n) atomicAdd(a.hist + i, n);
      const uint32_t cs = __reduce_add_sync(0xffffffffu, n);
      if (lane == 0 && cs) atomicAdd(&coarse_s[i >> 7], cs);
    }
    __syncthreads();
    if (tid < kCoarse && coarse_s[tid]) atomicAdd(a.hist + kLogBins + tid, coarse_s[tid]);
    if (!grid_barrier(a.bar + 4, a.status, a.wait_ns)) return bail();
  }
  // E(b - 1) - E(b) = positions in bin b (bins >= b*).
  auto E = [&](int b) -> uint32_t { return b >= kLogBins ? 0u : HS(b); };

  // ---- S: this CTA's survivors into bin order: position t of bin b goes to
  // slot E(b) + its arrival order in the bin (a cursor per bin; cursors and
  // slots were cleared by the indexer).  No barrier follows: an attention unit
  // reads only the slots of its own bins and waits for each to be written
  // (a survivor's key is never 0).
  if (mode == kRowFast) {
    auto put = [&](int32_t v, int t) {
      const uint32_t b = score_bin(v);
      if (b >= bstar) {
        const uint32_t i = atomicAdd(a.cnt + b, 1u);
        if (i < E((int)b - 1) - E((int)b)) st_relaxed_u64(a.surv + HS(b) + i, surv_key(ordered_key(v), t));
        else raise_status(a.status, DSA_DEVICE_CAPACITY);   // cannot happen: the bins were counted
      }
    };
#pragma unroll
    for (int j = 0; j < kRegScores; ++j) {
      const int t = c0 + j * kRowThreads + tid;
      if (t < c1) put(sreg[j], t);
    }
    scan_row<kRowThreads>(a.scores, c_reg, c1, put);
  }

  if (mode == kRowExact) {
    if (cta == 0) {
      exact_row_keys<kRowThreads>(a.scores, len, a.k, (uint32_t)a.k - n_above,
                                  [&](uint32_t u) { return score_bin((int32_t)(u ^ 0x80000000u)) == bstar; },
                                  keys, a.status);
      for (int j = tid; j < a.k; j += kRowThreads) a.idx[j] = key_pos(keys[j]);
    }
    if (!grid_barrier(a.bar + 1, a.status, a.wait_ns)) return bail();
  }
  // Entries past the selection, and its size.
  for (int j = n_take + cta * kRowThreads + tid; j < a.k; j += G * kRowThreads) a.idx[j] = -1;
  if (cta == 0 && tid == 0 && a.nsel) a.nsel[0] = n_take;

  // ---- R + A: attention units.
  const int units = (n_take + P - 1) / P;
  const int g = lane >> 2, cq = lane & 3;
  const int hg = warp >> 2, wq = warp & 3;
  int it = 0;
  for (int u = cta; u < units; u += G, ++it) {
    const int r0 = u * P, r1 = min(r0 + P, n_take), np = r1 - r0;
    if (mode == kRowExact) {
      if (tid < np) {
        const int t = __ldcg(a.idx + r0 + tid);
        pos_s[tid] = t;
      }
    } else {
      // Bins holding ranks r0 and r1 - 1: the smallest b with E(b) <= r.
      auto bin_of_rank = [&](uint32_t r) {
        int lo = (int)bstar, hi = kLogBins - 1;
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (E(mid) <= r) hi = mid; else lo = mid + 1;
        }
        return lo;
      };
      const int b_top = bin_of_rank((uint32_t)r0), b_bot = bin_of_rank((uint32_t)(r1 - 1));
      const uint32_t s0 = E(b_top), s1 = E(b_bot - 1);   // slots of bins b_top .. b_bot
      const int M = (int)(s1 - s0);
      if (M <= 64) {
        // Few members (the usual case: a unit's ranks span a few fine bins):
        // warp 0 ranks them by comparison.  Keys are unique, so a member's
        // rank is s0 + the number of members with a larger key.
        if (warp == 0) {
          const uint64_t k0 = lane < M ? wait_key(a.surv + s0 + lane, a.status, a.wait_ns) : 0ull;
          const uint64_t k1 = lane + 32 < M ? wait_key(a.surv + s0 + lane + 32, a.status, a.wait_ns) : 0ull;
          if ((lane < M && k0 == 0) || (lane + 32 < M && k1 == 0)) key_lost = 1;   // a wait ran out
          uint32_t n0 = 0, n1 = 0;
          for (int j = 0; j < 32; ++j) {
            const uint64_t o0 = __shfl_sync(0xffffffffu, k0, j);
            const uint64_t o1 = __shfl_sync(0xffffffffu, k1, j);
            const bool v0 = j < M, v1 = j + 32 < M;
            n0 += (uint32_t)(v0 && o0 > k0) + (uint32_t)(v1 && o1 > k0);
            n1 += (uint32_t)(v0 && o0 > k1) + (uint32_t)(v1 && o1 > k1);
          }
          const uint32_t ra = s0 + n0, rb = s0 + n1;
          if (lane < M && ra >= (uint32_t)r0 && ra < (uint32_t)r1) {
            const int t = key_pos(k0);
            pos_s[ra - r0] = t;
            a.idx[ra] = t;
          }
          if (lane + 32 < M && rb >= (uint32_t)r0 && rb < (uint32_t)r1) {
            const int t = key_pos(k1);
            pos_s[rb - r0] = t;
            a.idx[rb] = t;
          }
        }
      } else {
      uint32_t umax = 0, uminv = 0;
      for (int i0 = tid; i0 < M; i0 += 8 * kRowThreads) {   // eight slot loads in flight per thread
        uint64_t v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int i = i0 + j * kRowThreads;
          v[j] = i < M ? ld_relaxed_u64(a.surv + s0 + i) : 0ull;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int i = i0 + j * kRowThreads;
          if (i >= M) break;
          const uint64_t key = v[j] ? v[j] : wait_key(a.surv + s0 + i, a.status, a.wait_ns);
          if (key == 0) key_lost = 1;   // a wait ran out
          keys[i] = key;
          const uint32_t u = (uint32_t)(key >> 32);
          umax = max(umax, u);
          uminv = max(uminv, ~u);
        }
      }
      block_reduce_max2<kRowThreads>(umax, uminv, wt);
      // Rank of a member = E(b_top) + (members with a larger score) + (members
      // with its score and a lower position).  The first count comes from a
      // histogram of the members' exact scores; the second only matters for
      // members whose rank range meets the window, and is counted for those.
      const uint32_t range = umax - ~uminv + 1u;   // distinct scores spanned (>= 1)
      bool sorted_path = M > 0 && range > (uint32_t)kSubRange;
      if (!sorted_path && M > 0) {
        for (int i = tid; i <= (int)range; i += kRowThreads) sub[i] = 0;
        if (tid == 0) sh[6] = 0;
        if (tid == 1) sh[7] = 0;
        __syncthreads();
        for (int i = tid; i < M; i += kRowThreads) atomicAdd(&sub[umax - (uint32_t)(keys[i] >> 32)], 1u);
        __syncthreads();
        {   // exclusive prefix over the scores from the top: sub[d] = members above score umax - d
          const int base = tid * 4;
          uint32_t c[4], tsum = 0;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            c[j] = base + j < (int)range ? sub[base + j] : 0u;
            tsum += c[j];
          }
          const uint32_t incl = block_scan_incl<kRowThreads>(tsum, wt);
          uint32_t run = incl - tsum;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (base + j < (int)range) sub[base + j] = run;
            run += c[j];
          }
          if (tid == 0) sub[range] = (uint32_t)M;
        }
        __syncthreads();
        for (int i = tid; i < M; i += kRowThreads) {
          const uint64_t key = keys[i];
          const uint32_t d = umax - (uint32_t)(key >> 32);
          const uint32_t lo_r = s0 + sub[d], n_eq = sub[d + 1] - sub[d];
          if (lo_r >= (uint32_t)r1 || lo_r + n_eq <= (uint32_t)r0) continue;
          if (n_eq == 1) {
            const int t = key_pos(key);
            pos_s[lo_r - r0] = t;
            a.idx[lo_r] = t;
          } else {
            const uint32_t slot = atomicAdd(&sh[6], 1u);
            if (slot < (uint32_t)kWindowList) wlist[slot] = i; else sh[7] = 1;
          }
        }
        __syncthreads();
        sorted_path = sh[7] != 0;
        if (!sorted_path) {
          const int nl = (int)sh[6];
          for (int j = warp; j < nl; j += kRowWarps) {   // one warp per tied member
            const uint64_t key = keys[wlist[j]];
            const uint32_t u = (uint32_t)(key >> 32);
            uint32_t before = 0;
            // Every member of a score group that meets the window is in
            // wlist, so the group's larger keys are counted there.
            for (int m = lane; m < nl; m += 32) {
              const uint64_t o = keys[wlist[m]];
              before += ((uint32_t)(o >> 32) == u) & (o > key);
            }
            before = __reduce_add_sync(0xffffffffu, before);
            const uint32_t rank = s0 + sub[umax - u] + before;
            if (lane == 0 && rank >= (uint32_t)r0 && rank < (uint32_t)r1) {
              const int t = key_pos(key);
              pos_s[rank - r0] = t;
              a.idx[rank] = t;
            }
          }
        }
        __syncthreads();
      }
      if (sorted_path) {   // wide or heavily tied bins: sort the members
        sort_desc<kRowThreads>(keys, M);
        for (int i = tid; i < M; i += kRowThreads) {
          const uint32_t rank = s0 + (uint32_t)i;
          if (rank >= (uint32_t)r0 && rank < (uint32_t)r1) {
            const int t = key_pos(keys[i]);
            pos_s[rank - r0] = t;
            a.idx[rank] = t;
          }
        }
      }
      }
    }
    __syncthreads();   // pos_s final; the previous unit's reads of Ks, Pb, Ss are done
    if (key_lost) return bail();

    // Gather: one bulk copy per selected latent row (an FP8 cache's code rows
    // land in a staging buffer); rows past np are zero.
    if (warp == 0) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      const uint32_t rowb = F8 ? (uint32_t)a.D_k : qrow;
      if (lane == 0) mbar_expect_tx(bar_k, (uint32_t)np * rowb);
      __syncwarp();
      for (int j = lane; j < P; j += 32) {
        if (j < np) {
          if (F8)
            bulk_row(smem_u32(F8s + j * a.D_k), reinterpret_cast<const uint8_t*>(a.kv) + (size_t)pos_s[j] * a.D_k,
                     rowb, bar_k);
          else
            bulk_row(smem_u32(Ks + j * a.ks), a.kv + (size_t)pos_s[j] * a.D_k, rowb, bar_k);
        } else {
          for (int c8 = 0; c8 < a.ks / 8; ++c8) *reinterpret_cast<int4*>(Ks + j * a.ks + c8 * 8) = make_int4(0, 0, 0, 0);
        }
      }
    }
    if (F8 && warp == 1 && lane < P)   // the rows' scales, while the copies fly
      scs[lane] = lane < np ? (a.kv_scale ? __ldg(a.kv_scale + pos_s[lane]) : 1.f) : 0.f;
    bool ok = true;
    if (!q_done) ok = mbar_wait(bar_q, 0, a.status, a.wait_ns);
    ok = ok && mbar_wait(bar_k, (uint32_t)it & 1u, a.status, a.wait_ns);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) mbar_wait(bar_k, (uint32_t)it & 1u, nullptr, a.wait_ns);
      return bail();
    }
    q_done = true;
    if (F8) {   // widen the codes to bf16 in the K buffer (exact)
      const int chunks = a.D_k / 16;
      for (int e = tid; e < np * chunks; e += kRowThreads) {
        const int row = e / chunks, ch = e - row * chunks;
        uint4 lo, hi;
        e4m3x16_to_bf16(*reinterpret_cast<const uint4*>(F8s + row * a.D_k + ch * 16), lo, hi);
        *reinterpret_cast<uint4*>(Ks + row * a.ks + ch * 16) = lo;
        *reinterpret_cast<uint4*>(Ks + row * a.ks + ch * 16 + 8) = hi;
      }
      __syncthreads();
    }

    // S = Q K^T: warp (hg, wq) takes n-tile wq % NTILES of head group hg over
    // K part wq / NTILES.
    {
      const int nt = wq % NTILES, kp = wq / NTILES;
      const int nks = a.D_k / 16, kb = kp * (nks / KP), ke = kb + nks / KP;
      // Query row hg * 16 + arow, 16-byte chunk c of box bx at chunk c ^ (row mod 8).
      const int arow = (lane & 7) + ((lane >> 3) & 1) * 8, a8 = lane >> 4;
      const uint32_t qrow_addr = smem_u32(Qs) + (uint32_t)(hg * 16 + arow) * 128u;
      const int sw = lane & 7;
      auto qaddr = [&](int kk) {
        return qrow_addr + (uint32_t)(kk >> 2) * 8192u + ((uint32_t)((((kk & 3) << 1) + a8) ^ sw) << 4);
      };
      const uint32_t baddr = smem_u32(Ks + (nt * 8 + (lane & 7)) * a.ks + (lane >> 3) * 8);
      float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
      for (int kk = kb; kk < ke; kk += 2) {   // two k-steps per B load (ke - kb is even)
        uint32_t a0, a1, a2, a3, e0, e1, e2, e3, b0, b1, b2, b3;
        ldsm_x4(qaddr(kk), a0, a1, a2, a3);
        ldsm_x4(qaddr(kk + 1), e0, e1, e2, e3);
        ldsm_x4(baddr + kk * 32, b0, b1, b2, b3);
        mma16816(s0, a0, a1, a2, a3, b0, b1);
        mma16816(s1, e0, e1, e2, e3, b2, b3);
      }
      float* dst = Ss + kp * kRowHeads * P;
      const int h0 = hg * 16 + g, p0 = nt * 8 + 2 * cq;
      dst[h0 * P + p0] = s0[0] + s1[0];
      dst[h0 * P + p0 + 1] = s0[1] + s1[1];
      dst[(h0 + 8) * P + p0] = s0[2] + s1[2];
      dst[(h0 + 8) * P + p0 + 1] = s0[3] + s1[3];
    }
    __syncthreads();

    // Softmax over the unit's positions (log2 domain): eight threads per head.
    {
      const int h = tid >> 3, sub = tid & 7;
      float v[P / 8];
      float m = -CUDART_INF_F;
#pragma unroll
      for (int j = 0; j < P / 8; ++j) {
        const int p = sub + 8 * j;
        float x = Ss[h * P + p];
        if (KP == 2) x += Ss[kRowHeads * P + h * P + p];
        v[j] = p < np ? x * a.scale_log2 * (F8 ? scs[p] : 1.f) : -CUDART_INF_F;
        m = fmaxf(m, v[j]);
      }
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      float l = 0.f;
#pragma unroll
      for (int j = 0; j < P / 8; ++j) {
        const float e = v[j] == -CUDART_INF_F ? 0.f : exp2f(v[j] - m);
        l += e;   // an FP8 row's scale weights its values, not the softmax sum
        const float pw = F8 ? e * scs[sub + 8 * j] : e;
        Pb[h * (P + 8) + sub + 8 * j] = __bfloat16_as_ushort(__float2bfloat16_rn(pw));
      }
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
      if (sub == 0) {
        mls[h * 2] = m;
        mls[h * 2 + 1] = l;
      }
      // Largest |value| among the gathered rows (an FP8 row's codes times its
      // scale), as float bits (monotone for values >= 0).
      uint32_t vb = 0;
      const int cpr = a.D_v / 8;   // 16-byte chunks of a value row
      if (F8) {
        float vf = 0.f;
        for (int e = tid; e < np * cpr; e += kRowThreads) {
          const uint4 w4 = *reinterpret_cast<const uint4*>(Ks + (e / cpr) * a.ks + (e % cpr) * 8);
          const uint32_t ws4[4] = {w4.x, w4.y, w4.z, w4.w};
          uint32_t cm = 0;
#pragma unroll
          for (int i = 0; i < 4; ++i) cm = max(cm, max(ws4[i] & 0x7FFFu, (ws4[i] >> 16) & 0x7FFFu));
          vf = fmaxf(vf, __uint_as_float(cm << 16) * scs[e / cpr]);
        }
        vb = __float_as_uint(vf);
      } else {
        for (int e = tid; e < np * cpr; e += kRowThreads) {
          const uint4 w4 = *reinterpret_cast<const uint4*>(Ks + (e / cpr) * a.ks + (e % cpr) * 8);
          const uint32_t ws4[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) vb = max(vb, max(ws4[i] & 0x7FFFu, (ws4[i] >> 16) & 0x7FFFu));
        }
        vb <<= 16;   // bf16 bits -> float bits
      }
      vb = __reduce_max_sync(0xffffffffu, vb);
      if (lane == 0) wt[warp] = vb;
    }
    __syncthreads();
    // psc: 2^(141 - E) for the largest value's exponent E (clamped), so the
    // stored O / l (a convex combination of these rows) stays below 2^15.
    float sc;
    {
      const uint32_t vb = __reduce_max_sync(0xffffffffu, lane < kRowWarps ? wt[lane] : 0u);
      const int E = min(254, max(20, (int)(vb >> 23)));
      sc = __int_as_float((127 + 141 - E) << 23);
    }

    // O = P V for head group hg, columns [wq 8 NT, (wq + 1) 8 NT).
    float acc[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    {
      const int arow = (lane & 7) + ((lane >> 3) & 1) * 8, acol = (lane >> 4) * 8;
      const uint32_t paddr = smem_u32(Pb + (hg * 16 + arow) * (P + 8) + acol);
      const int vrow = (lane & 7) + ((lane >> 3) & 1) * 8, vcol = wq * 8 * NT + (lane >> 4) * 8;
      const uint32_t vaddr = smem_u32(Ks + vrow * a.ks + vcol);
#pragma unroll
      for (int kq = 0; kq < P / 16; ++kq) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(paddr + kq * 32, a0, a1, a2, a3);
#pragma unroll
        for (int n2 = 0; n2 < NT / 2; ++n2) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vaddr + (kq * 16 * a.ks + n2 * 16) * 2, b0, b1, b2, b3);
          mma16816(acc[2 * n2], a0, a1, a2, a3, b0, b1);
          mma16816(acc[2 * n2 + 1], a0, a1, a2, a3, b2, b3);
        }
      }
    }
    // The unit's partial: O / l of each head as fp16 (times sc), and (m, l).
    __half* po_u = a.po + (size_t)u * kRowHeads * Dvp;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int h = hg * 16 + g + 8 * j;
      const float lh = mls[h * 2 + 1];
      const float inv = lh > 0.f ? sc / lh : 0.f;
#pragma unroll
      for (int ng = 0; ng < NG; ++ng) {
        uint32_t w4[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const __half2 hv = __floats2half2_rn(acc[4 * ng + t][2 * j] * inv, acc[4 * ng + t][2 * j + 1] * inv);
          w4[t] = *reinterpret_cast<const uint32_t*>(&hv);
        }
        __stcg(reinterpret_cast<uint4*>(po_u + (size_t)h * Dvp + ((wq * NG + ng) * 4 + cq) * 8),
               make_uint4(w4[0], w4[1], w4[2], w4[3]));
      }
    }
    if (tid < 2 * kRowHeads) __stcg(a.pml + (size_t)u * 2 * kRowHeads + tid, mls[tid]);
    if (tid == 0) __stcg(a.psc + u, sc);
  }
  if (!q_done && tid == 0) mbar_wait(bar_q, 0, nullptr, a.wait_ns);   // a CTA without a unit
  if (!grid_barrier(a.bar + 2, a.status, a.wait_ns)) return;

  // ---- M: output slices (head h, partial chunks [c0, c0 + 32)).  Thread
  // (v, j) sums chunk c0 + v (eight columns, one 16-byte load) over the units
  // j, j + 16, ...: all its loads are issued before the sums; then the sixteen
  // groups are added in order.
  const int nhalf = (Dvp + kMergeCols - 1) / kMergeCols;
  float* wgt = wm;                                     // [256] weight of each unit's values
  float* gsum = reinterpret_cast<float*>(keys);        // [16][256] group sums
  constexpr int kVec = kMergeCols / 8;                 // 32 threads cover a slice's columns
  constexpr int kGroups = kRowThreads / kVec;          // 16
  constexpr int kBatch = 8;                            // loads in flight per thread
  for (int sl = cta; sl < kRowHeads * nhalf; sl += G) {
    const int h = sl / nhalf, cb = (sl % nhalf) * kMergeCols;
    const int width = min(kMergeCols, Dvp - cb);
    const int v = tid % kVec, grp = tid / kVec;
    const bool live = 8 * v < width;
    const int c = cb / 8 + v;                          // partial chunk
    const __half* base = a.po + (size_t)h * Dvp + 8 * c;
    // The first batch of values is loaded with the units' (m, l, scale).
    uint4 x[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int uu = grp + kGroups * j;
      x[j] = live && uu < units ? __ldcg(reinterpret_cast<const uint4*>(base + (size_t)uu * kRowHeads * Dvp))
                                : make_uint4(0u, 0u, 0u, 0u);
    }
    float m = -CUDART_INF_F, l = 0.f, scu = 1.f;
    if (tid < units) {
      const float* ml = a.pml + ((size_t)tid * kRowHeads + h) * 2;
      m = __ldcg(ml);
      l = __ldcg(ml + 1);
      scu = __ldcg(a.psc + tid);
    }
    float M = l > 0.f ? m : -CUDART_INF_F;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if (lane == 0) red[warp] = M;
    __syncthreads();
    M = lane < kRowWarps ? red[lane] : -CUDART_INF_F;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float w = (tid < units && l > 0.f) ? exp2f(m - M) : 0.f;
    float Lw = w * l;
    __syncthreads();   // red is rewritten
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Lw += __shfl_xor_sync(0xffffffffu, Lw, o);
    if (lane == 0) red[warp] = Lw;
    if (tid < 256) wgt[tid] = w * l / scu;
    __syncthreads();
    float Lsum = lane < kRowWarps ? red[lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Lsum += __shfl_xor_sync(0xffffffffu, Lsum, o);
    float o8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int u0 = grp;; u0 += kGroups * kBatch) {
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int uu = u0 + kGroups * j;
        const float wu = uu < units ? wgt[uu] : 0.f;
        const uint32_t xs[4] = {x[j].x, x[j].y, x[j].z, x[j].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&xs[i]));
          o8[2 * i] += wu * f.x;
          o8[2 * i + 1] += wu * f.y;
        }
      }
      const int nx = u0 + kGroups * kBatch;
      if (nx >= units) break;
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int uu = nx + kGroups * j;
        x[j] = live && uu < units ? __ldcg(reinterpret_cast<const uint4*>(base + (size_t)uu * kRowHeads * Dvp))
                                  : make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) gsum[grp * kMergeCols + 8 * v + i] = o8[i];
    __syncthreads();
    {   // the sixteen group sums of each column, in two steps over all threads:
        // thread (pair p, quarter r) adds groups 4r .. 4r + 3 of columns 2p, 2p + 1
      float2* part = reinterpret_cast<float2*>(gsum + kGroups * kMergeCols);   // [4][128]
      const int pp = tid & (kMergeCols / 2 - 1), r = tid / (kMergeCols / 2);
      float2 t = reinterpret_cast<const float2*>(gsum + 4 * r * kMergeCols)[pp];
#pragma unroll
      for (int j = 1; j < 4; ++j) {
        const float2 g = reinterpret_cast<const float2*>(gsum + (4 * r + j) * kMergeCols)[pp];
        t.x += g.x;
        t.y += g.y;
      }
      part[r * (kMergeCols / 2) + pp] = t;
      __syncthreads();
      if (tid < kMergeCols / 2 && 8 * (tid / 4) < width) {   // pair tid of the slice: chunk tid / 4
        float2 u = part[tid];
#pragma unroll
        for (int q = 1; q < 4; ++q) {
          const float2 g = part[q * (kMergeCols / 2) + tid];
          u.x += g.x;
          u.y += g.y;
        }
        const float il = Lsum > 0.f ? 1.f / Lsum : 0.f;
        const int cc2 = cb / 8 + tid / 4, q = tid % 4;   // partial chunk, and its n-tile
        const int cw = cc2 / (4 * NG), cg = (cc2 / 4) % NG, cc = cc2 % 4;
        const int col = cw * 8 * NT + (4 * cg + q) * 8 + 2 * cc;
        if (col < a.D_v)   // D_v is even: a pair is in or out whole
          *reinterpret_cast<uint32_t*>(a.out + (size_t)h * a.D_v + col) = pack_bf16(u.x * il, u.y * il);
      }
    }
    if (tid == 0 && cb == 0 && a.lse)
      a.lse[h] = Lsum > 0.f ? (M + log2f(Lsum)) * 0.69314718055994531f : -CUDART_INF_F;
    __syncthreads();   // wgt, gsum and red are rewritten by the next slice
  }
}

template <int NT, int P, bool F8>
cudaError_t launch_row(const RowArgs& a, cudaStream_t st) {
  const RowSmem L(P, a.qs, a.ks, F8);
  const size_t smem = L.total + 1024;   // alignment slack
  cudaError_t e = cudaFuncSetAttribute(decode_row_kernel<NT, P, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0, per_sm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_row_kernel<NT, P, F8>, kRowThreads,
                                                         smem)) != cudaSuccess)
    return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  return launch_coop(decode_row_kernel<NT, P, F8>, dim3(sms), dim3(kRowThreads), smem, st, a);
}

}  // namespace

constexpr int kRowUnitRows = 16;   // selected positions per attention unit

bool decode_row_supported(const dsa_problem& p) {
  return p.R == 1 && p.B == 1 && p.H_q == kRowHeads && p.D_k % 64 == 0 && p.D_k <= 576 && p.D_v <= 512 && p.k <= kCapFast;
}

// Partials of the attention units: fp16 O / l [units][64][32 NT] (columns in
// the kernel's chunk order), fp32 (m, l) [units][64][2], fp32 scale [units],
// each region 256-byte aligned.
static size_t row_units(const dsa_problem& p) { return (size_t)(p.k + kRowUnitRows - 1) / kRowUnitRows; }
// Output n-tiles per warp: the smallest of 4, 8, 16 with 32 NT >= D_v.
static int row_nt(int D_v) {
  int NT = 4;
  while (NT * 32 < D_v) NT *= 2;
  return NT;
}
static size_t align256(size_t x) { return (x + 255) / 256 * 256; }

size_t decode_row_partials_bytes(const dsa_problem& p) {
  const size_t u = row_units(p);
  return align256(u * kRowHeads * 32 * row_nt(p.D_v) * 2) + align256(u * kRowHeads * 2 * 4) + align256(u * 4);
}

cudaError_t launch_decode_row(const dsa_problem& p, const Plan& pl, const int32_t* scores, int32_t* idx,
                              int32_t* nsel, uint16_t* out, char* ws, cudaStream_t st) {
  RowArgs a;
  std::memset(&a, 0, sizeof a);
  a.scores = scores;
  a.row_len = p.row_len;
  a.q = p.q;
  a.kv = p.kv;
  a.f8 = (p.flags & DSA_FLAG_KV_FP8) ? 1 : 0;
  a.kv_scale = a.f8 ? p.kv_scale : nullptr;
  a.idx = idx;
  a.nsel = nsel;
  a.out = out;
  a.lse = nullptr;
  a.status = reinterpret_cast<uint32_t*>(ws + pl.off_status);
  a.bar = a.status + kBarrierWord;
  a.hist = reinterpret_cast<uint32_t*>(ws + pl.off_lhist);
  a.zcount = reinterpret_cast<uint32_t*>(ws + pl.off_lkeep);
  a.cnt = reinterpret_cast<uint32_t*>(ws + pl.off_lcur);
  a.surv = reinterpret_cast<uint64_t*>(ws + pl.off_lsurv);
  const size_t u = row_units(p);
  char* pp = ws + pl.off_rpart;
  a.po = reinterpret_cast<__half*>(pp);
  a.pml = reinterpret_cast<float*>(pp + align256(u * kRowHeads * 32 * row_nt(p.D_v) * 2));
  a.psc = reinterpret_cast<float*>(pp + align256(u * kRowHeads * 32 * row_nt(p.D_v) * 2) + align256(u * kRowHeads * 2 * 4));
  a.L1 = (int)p.L_total;
  a.k = p.k;
  a.D_k = p.D_k;
  a.D_v = p.D_v;
  a.scale_log2 = p.softmax_scale * 1.4426950408889634f;
  a.wait_ns = kDefaultWaitNs;
  const int NT = row_nt(p.D_v);
  a.qs = p.D_k;   // the swizzled query boxes need no padding
  a.ks = (p.D_k > NT * 32 ? p.D_k : NT * 32) + 8;
  EncodeTiledFn encode = encode_tiled_fn();
  if (!encode) return cudaErrorNotSupported;
  {
    const cuuint64_t gdim[2] = {(cuuint64_t)p.D_k, (cuuint64_t)kRowHeads};
    const cuuint64_t gstride[1] = {(cuuint64_t)p.D_k * 2};
    const cuuint32_t box[2] = {64u, 64u};
    const cuuint32_t estride[2] = {1u, 1u};
    if (encode(&a.qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(p.q), gdim, gstride, box,
               estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  if (a.f8) {
    switch (NT) {
      case 4: return launch_row<4, kRowUnitRows, true>(a, st);
      case 8: return launch_row<8, kRowUnitRows, true>(a, st);
      default: return launch_row<16, kRowUnitRows, true>(a, st);
    }
  }
  switch (NT) {
    case 4: return launch_row<4, kRowUnitRows, false>(a, st);
    case 8: return launch_row<8, kRowUnitRows, false>(a, st);
    default: return launch_row<16, kRowUnitRows, false>(a, st);
  }
}

}  // namespace dsa
