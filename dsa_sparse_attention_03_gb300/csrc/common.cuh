// Internal definitions shared by the libdsa translation units (not installed).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stddef.h>

#include "dsa.h"
#include "dsa_testing.h"
#include "dsa_front_end.h"

namespace dsa {

constexpr int kBucketBits = 11;               // linear bins over the row's key range
constexpr int kBuckets = 1 << kBucketBits;
constexpr int kCapFast = 4096;                // survivors ranked directly (else exact fallback)
constexpr int kAttnRows = 64;                 // selected positions per attention tile
constexpr int kAttnHeads = 16;                // query heads per attention CTA (mma M)
constexpr int kMaxB = 4096;
constexpr int kMaxK = 4096;

// Per-row state of the top-k, in the workspace.  Zeroed (with the histograms)
// by the indexer of a decode step, or by dsa_topk before its first kernel.
struct RowState {
  uint32_t umax;       // max ordered key of the row (merged by the indexer)
  uint32_t uminv;      // max of ~key, i.e. ~min
  uint32_t bstar;      // threshold bucket
  uint32_t n_above;    // positions in buckets above it (all selected)
  uint32_t cand;       // positions in the threshold bucket
  uint32_t n_union;    // survivor slot counter
  uint32_t mode;       // fast / take all / empty / exact fallback
  uint32_t n_take;     // min(k, row_len)
  uint32_t spare[8];
};
static_assert(sizeof(RowState) == 64, "RowState is 64 bytes");

// Everything the launchers need: validated sizes and the workspace map.
struct Plan {
  int R, B, H_i, D_i, H_q, D_k, D_v, k, L_max;
  int flags;
  int chunk, nchunk;       // top-k: positions per CTA, CTAs per row
  int hist_rep;            // top-k: copies of each row's global histogram
  int attn_kc_max;          // attention: clusters per (row, head group), at most
  int fused_row;            // dsa_decode_step runs the single-row kernel (decode_row.cu)
  size_t off_status, off_state, off_hist, off_acnt, off_lhist, zero_end;
  size_t off_lcur, off_lsurv;   // single-row step: bin cursors and survivor slots (cleared)
  size_t off_lkeep;         // single-row step: words the indexer must not clear (see decode_row.cu)
  size_t off_surv, off_scores, off_apart, off_rpart, total;
  size_t off_pairc, off_pairx;  // top-k, exact fallback by CTA pairs: counters (cleared), buffers (0: none)
};

// Top-k: from kTopkSortRows rows on, each CTA sorts whole rows; up to
// kPairRows rows, a row in the exact fallback is resolved by two CTAs when
// the grid holds two per row.  Per row the pair has kPairPhases barrier
// counters (cleared with the status block) and an exchange buffer:
// [0, 256) scalars, then two radix histograms per part (alternate passes),
// the per-block tie counts of both parts, and part 1's winners.
constexpr int kTopkSortRows = 8;
constexpr int kPairRows = 80;
constexpr int kPairPhases = 8;
constexpr size_t kPairHistOff = 256;
constexpr size_t kPairTieOff = kPairHistOff + 4 * 2048 * 4;
constexpr size_t kPairWinOff = kPairTieOff + 2 * 32 * 4 + 256;
__host__ __device__ constexpr size_t pair_x_bytes(int k) { return kPairWinOff + size_t(k) * 8; }

// Attention cluster size for k selected positions: one 64-position tile per
// CTA, clusters of 4 (one CTA per SM) up to 32 tiles, else of 8, so that at
// most 8 clusters share a (row, head group).
__host__ __device__ inline int attn_cluster_size(int k) {
  const int tiles = (k + kAttnRows - 1) / kAttnRows;
  const int cmax = tiles <= 32 ? 4 : 8;
  int c = 1;
  while (c < tiles && c < cmax) c <<= 1;
  return c;
}

// Clusters per (row, head group) for R rows, hgroups head groups and top-k k:
// enough for one 64-position tile per CTA, halved while the grid exceeds about
// 600 CTAs (a few waves), so that many rows make each CTA loop over several
// tiles instead of paying each CTA's fixed latency in dozens of waves.
inline int attn_clusters(int R, int hgroups, int k) {
  const int tiles = (k + kAttnRows - 1) / kAttnRows;
  const int C = attn_cluster_size(k);
  int kc = (tiles + C - 1) / C;
  const int64_t per_kc = (int64_t)R * hgroups * C;
  while (kc > 1 && per_kc * kc > 600) kc = (kc + 1) / 2;
  return kc;
}

// Log-spaced score bins of the single-row step, shared by the indexer's
// epilogue (which counts its scores into them) and decode_row.cu.  A score's
// bin is its magnitude |s| (or -1 - s when negative) as a float with 7 mantissa
// bits -- exact below 128, then 128 bins per octave -- above 4096 for s >= 0
// and mirrored below it for s < 0: monotone in s, independent of the data.
constexpr int kLogMant = 7;
constexpr int kLogBins = 8192;
constexpr int kLogCoarse = kLogBins / 128;   // coarse bins of 128 log bins (one octave)
__device__ __forceinline__ uint32_t score_bin(int32_t s) {
  const uint32_t a = s >= 0 ? (uint32_t)s : (uint32_t)(-1 - s);
  uint32_t g = a;
  if (a >= (1u << kLogMant)) {
    const int e = 31 - __clz(a);   // floor(log2 a) >= 7
    g = ((uint32_t)(e - kLogMant + 1) << kLogMant) + ((a >> (e - kLogMant)) & ((1u << kLogMant) - 1));
  }
  return s >= 0 ? (kLogBins / 2) + g : (kLogBins / 2 - 1) - g;
}

// Order-preserving map of int32 onto uint32.
__host__ __device__ __forceinline__ uint32_t ordered_key(int32_t s) {
  return static_cast<uint32_t>(s) ^ 0x80000000u;
}

__device__ __forceinline__ void raise_status(uint32_t* status, uint32_t bit) {
  if (status) atomicOr(status, bit);
}

// Programmatic dependent launch: every kernel waits for its predecessor in the
// stream to complete (and flush) before touching global memory, and lets its
// successor be scheduled early.  Both are no-ops without the launch attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch with the programmatic-stream-serialization attribute (captured into
// CUDA graphs as a programmatic edge).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// The same with the cooperative attribute as well: every CTA of the grid is
// resident at once (the launch fails otherwise), so CTAs may wait on one
// another at grid barriers.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_coop(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                               cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Words of the 256-byte status block: [0] device status bits; from
// kBarrierWord on, grid barrier counters (zeroed with the block).
constexpr int kBarrierWord = 16;

// Per-row running max of the ordered keys and of their complements (= ~min),
// merged into RowState.umax / uminv by the indexers' epilogues (one warp).
__device__ __forceinline__ void row_minmax_flush(RowState* st, uint32_t umax, uint32_t uminv) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    umax = max(umax, __shfl_xor_sync(0xffffffffu, umax, o));
    uminv = max(uminv, __shfl_xor_sync(0xffffffffu, uminv, o));
  }
  if ((threadIdx.x & 31) == 0) {
    if (umax) atomicMax(&st->umax, umax);
    if (uminv) atomicMax(&st->uminv, uminv);
  }
}

// Limit of every bounded device wait in normal operation.
constexpr uint64_t kDefaultWaitNs = 2000000000ull;

// Fault injection for the tests of the bounded waits (include/dsa_testing.h):
// each hook makes one wait run out on purpose, with no copy in flight when it
// does.  Normal calls pass none (nullptr).
struct TestHooks {
  uint64_t wait_ns = kDefaultWaitNs;   // limit of every bounded wait
  int topk_skip_cta = -1;              // this top-k CTA returns before its first grid barrier
  int attn_no_gather = 0;              // attention CTAs arm their first gather, issue no copy
  int indexer_no_load = 0;             // indexer CTAs arm their first key tile, issue no copy
};

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
// (null if the driver lacks it).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();

// Launchers (one per translation unit).  Each returns the launch error.
// For the single-row step (Plan::fused_row) both indexers also clear the
// workspace's range [0, Plan::zero_end) (status word, histograms, cursors), so
// that step needs no separate memset; other callers clear it before the launch.
cudaError_t launch_indexer_dp4a(const dsa_problem& p, const Plan& pl, int32_t* scores, char* ws,
                                cudaStream_t st);
cudaError_t launch_indexer_tc(const dsa_problem& p, const Plan& pl, int32_t* scores, char* ws,
                              cudaStream_t st, const TestHooks* hooks = nullptr);
bool indexer_tc_supported(const dsa_problem& p);
// The tensor-core indexer keeps its A operand in tensor memory (D_i = 128, at
// most 128 accumulator columns per tile, at least one full key tile).
bool indexer_tc_tmem_operand(const dsa_problem& p);
// minmax_done: the indexer already merged each row's key range into RowState.
cudaError_t launch_topk(const dsa_problem& p, const Plan& pl, const int32_t* scores,
                        int32_t* idx, int32_t* nsel, char* ws, cudaStream_t st, bool minmax_done,
                        const TestHooks* hooks = nullptr);
cudaError_t launch_attention(const dsa_problem& p, const Plan& pl, const int32_t* idx,
                             const int32_t* nsel, uint16_t* out, float* lse, char* ws,
                             cudaStream_t st, const TestHooks* hooks = nullptr);
// Single-row decode step after the indexer: selection and attention in one
// cooperative kernel (decode_row.cu).
bool decode_row_supported(const dsa_problem& p);
size_t decode_row_partials_bytes(const dsa_problem& p);
constexpr int kRowHistCopies = 8;   // CTA c of the indexer adds into copy c % 8 (spreads the atomics)
constexpr size_t kRowHistWords = 8192 + 64;             // one copy: log-bin histogram and its coarse sums
constexpr size_t kRowHistBytes = kRowHistCopies * kRowHistWords * 4;
constexpr size_t kRowCursorBytes = 8192 * 4;          // bin cursors of the scatter (cleared each step)
constexpr size_t kRowSurvBytes = 4096 * 8;             // survivor slots (cleared each step: 0 = not yet written)
constexpr size_t kRowKeepBytes = 256;                  // arrival counter of the indexer's CTAs (not cleared)
cudaError_t launch_decode_row(const dsa_problem& p, const Plan& pl, const int32_t* scores, int32_t* idx,
                              int32_t* nsel, uint16_t* out, char* ws, cudaStream_t st);

// Indexer front end (front_end.cu): affine 8-bit projections of the hidden rows
// and their quantisation to q_idx / w_idx.
struct FrontArgs {
  const uint8_t* wq;          // [Oq, d] codes
  const uint16_t* sq;         // [Oq, d / 64] bf16 scales
  const uint16_t* bq;         // [Oq, d / 64] bf16 biases
  const uint8_t* ww;          // [H_i, d]
  const uint16_t* sw;
  const uint16_t* bw;
  const uint16_t* x;          // [R, d] bf16
  int R, d, H_i, D_i, Oq;     // Oq = H_i * D_i
  int q_max, w_max;
  int rows_max;               // set by the launcher: output rows per CTA, at most
  int stages;                 // set by the launcher: weight rows in flight per CTA
  int y_stride;               // floats per row of y (a multiple of 4)
  float* y;                   // [R, y_stride] workspace: the projections
  float* proj;                // [R, Oq + H_i] or null
  uint32_t* amax;             // [R, H_i] workspace, zeroed: max |qf| per head (float bits)
  uint32_t* ticket;           // [passes] workspace, zeroed: CTAs done with each pass
  uint32_t* cnt;              // [passes, H_i] workspace, zeroed: rows done of each query head
  uint32_t* status;           // the workspace's status word
  uint64_t wait_ns;           // limit of every bounded wait
  int8_t* q_idx;
  int32_t* w_idx;
  float* q_scale;             // or null
  float* w_scale;             // or null
};
cudaError_t launch_front_end(FrontArgs a, cudaStream_t st);

// Declared-bound check (check.cu): int8 bytes of k and q (16-byte multiples)
// against qk (>= 128: not checked), head weights against wmax.
cudaError_t launch_check_bounds(const int8_t* k, size_t k_bytes, const int8_t* q, size_t q_bytes,
                                const int32_t* w, size_t nw, int qk, int wmax, uint32_t* status,
                                cudaStream_t st);

}  // namespace dsa
