// libdsa C ABI: argument validation, workspace map and the launch sequence of
// each entry point.  All compute lives in the kernels of the other units.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include "common.cuh"

namespace dsa {
namespace {

thread_local std::string g_err;

dsa_status fail(dsa_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
dsa_status fail(dsa_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

dsa_status cuda_fail(cudaError_t e, const char* what) {
  return fail(DSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline bool aligned(const void* ptr, size_t a) {
  return (reinterpret_cast<uintptr_t>(ptr) % a) == 0;
}

enum Need { kNeedIndexer = 1, kNeedTopk = 2, kNeedAttn = 4 };

// Validates the fields an entry point reads and builds the workspace map.
dsa_status make_plan(const dsa_problem* p, int need, Plan* pl) {
  if (!p) return fail(DSA_ERR_INVALID_ARG, "problem is NULL");
  if (p->R < 0 || p->R > 65535) return fail(DSA_ERR_INVALID_ARG, "R=%d outside [0,65535]", p->R);
  if (p->B < 1 || p->B > kMaxB) return fail(DSA_ERR_UNSUPPORTED, "B=%d outside [1,%d]", p->B, kMaxB);
  if (p->L_max < 0) return fail(DSA_ERR_INVALID_ARG, "L_max=%d < 0", p->L_max);
  if (p->L_total < 0 || p->L_total >= (int64_t(1) << 31))
    return fail(DSA_ERR_UNSUPPORTED, "L_total=%lld outside [0,2^31)", (long long)p->L_total);
  if (p->k < 1 || p->k > kMaxK) return fail(DSA_ERR_UNSUPPORTED, "k=%d outside [1,%d]", p->k, kMaxK);
  if (p->flags & ~(DSA_INDEXER_MASK | DSA_FLAG_NO_RELU | DSA_FLAG_KV_FP8))
    return fail(DSA_ERR_INVALID_ARG, "unknown flag bits 0x%x", p->flags);
  if (need && p->R > 0 && (!p->offsets || !p->row_offsets || !p->row_len))
    return fail(DSA_ERR_INVALID_ARG, "offsets/row_offsets/row_len must be set");

  if (need & kNeedIndexer) {
    if (p->H_i < 1 || p->H_i > 128) return fail(DSA_ERR_UNSUPPORTED, "H_i=%d outside [1,128]", p->H_i);
    if (p->D_i != 32 && p->D_i != 64 && p->D_i != 128 && p->D_i != 256)
      return fail(DSA_ERR_UNSUPPORTED, "D_i=%d not in {32,64,128,256}", p->D_i);
    if (p->R > 0 && (!p->q_idx || !p->w_idx || (p->L_total > 0 && !p->k_idx)))
      return fail(DSA_ERR_INVALID_ARG, "q_idx/w_idx/k_idx must be set");
    if (!aligned(p->k_idx, 16) || !aligned(p->q_idx, 16) || !aligned(p->w_idx, 4))
      return fail(DSA_ERR_INVALID_ARG, "k_idx/q_idx must be 16-byte aligned, w_idx 4-byte");
    const int64_t qk = p->qk_abs_max > 0 ? p->qk_abs_max : 128;
    const int64_t wm = p->w_abs_max > 0 ? p->w_abs_max : 4;
    if (qk > 128) return fail(DSA_ERR_INVALID_ARG, "qk_abs_max=%d > 128", p->qk_abs_max);
    const double bound = double(p->H_i) * double(wm) * double(p->D_i) * double(qk * qk);
    if (bound >= 2147483648.0)
      return fail(DSA_ERR_OVERFLOW_RISK,
                  "H_i*w_abs_max*D_i*qk_abs_max^2 = %.0f reaches 2^31 (int32 scores)", bound);
    const int ix = p->flags & DSA_INDEXER_MASK;
    if (ix != DSA_INDEXER_AUTO && ix != DSA_INDEXER_DP4A && ix != DSA_INDEXER_TC)
      return fail(DSA_ERR_INVALID_ARG, "unknown indexer selector %d", ix);
    if (ix == DSA_INDEXER_TC && !indexer_tc_supported(*p))
      return fail(DSA_ERR_UNSUPPORTED, "tensor-core indexer does not support this shape");
  }
  if (need & kNeedAttn) {
    if (p->H_q < 1 || p->H_q > 128) return fail(DSA_ERR_UNSUPPORTED, "H_q=%d outside [1,128]", p->H_q);
    if (p->D_k < 16 || p->D_k > 576 || p->D_k % 16)
      return fail(DSA_ERR_UNSUPPORTED, "D_k=%d: need a multiple of 16 in [16,576]", p->D_k);
    if (p->D_v < 32 || p->D_v > 512 || p->D_v % 32 || p->D_v > p->D_k)
      return fail(DSA_ERR_UNSUPPORTED, "D_v=%d: need a multiple of 32, <= 512 and <= D_k", p->D_v);
    if (p->R > 0 && (!p->q || (p->L_total > 0 && !p->kv)))
      return fail(DSA_ERR_INVALID_ARG, "q/kv must be set");
    if (!aligned(p->q, 16) || !aligned(p->kv, 16))
      return fail(DSA_ERR_INVALID_ARG, "q/kv must be 16-byte aligned");
    if ((p->flags & DSA_FLAG_KV_FP8) && !aligned(p->kv_scale, 4))
      return fail(DSA_ERR_INVALID_ARG, "kv_scale must be 4-byte aligned");
    if (!(p->softmax_scale == p->softmax_scale) || p->softmax_scale <= 0.f)
      return fail(DSA_ERR_INVALID_ARG, "softmax_scale must be positive");
  }

  Plan& P = *pl;
  std::memset(&P, 0, sizeof P);
  P.R = p->R; P.B = p->B; P.H_i = p->H_i; P.D_i = p->D_i; P.H_q = p->H_q;
  P.D_k = p->D_k; P.D_v = p->D_v; P.k = p->k; P.L_max = p->L_max; P.flags = p->flags;

  // Top-k: about one chunk of 1K..64K positions per CTA of the persistent grid.
  const int64_t work = int64_t(p->L_max) * (p->R > 0 ? p->R : 1);
  int chunk = 1024;
  while (chunk < 65536 && int64_t(chunk) * 160 < work) chunk <<= 1;
  P.chunk = chunk;
  P.nchunk = p->L_max > 0 ? (p->L_max + chunk - 1) / chunk : 1;
  // Many chunks adding into one row's 2048 bins would serialise on the hot
  // bins' L2 lines; chunk c adds into copy c % hist_rep instead.
  P.hist_rep = P.nchunk >= 256 ? 8 : (P.nchunk >= 64 ? 4 : 1);

  const size_t R = size_t(p->R);
  size_t off = 0;
  P.off_status = off; off += 256;
  P.off_state = off; off = align_up(off + R * sizeof(RowState), 256);
  P.off_hist = off; off = align_up(off + R * size_t(P.hist_rep) * kBuckets * 4, 256);
  // Attention: clusters of 4 or 8 CTAs take one 64-position tile per CTA; a
  // (row, head group) with more tiles uses several clusters (at most 8),
  // merged through per-slice partials and arrival counters.
  const int hgroups = p->H_q > 0 ? (p->H_q + kAttnHeads - 1) / kAttnHeads : 0;
  P.attn_kc_max = attn_clusters(p->R, hgroups, p->k);
  P.off_acnt = off; off = align_up(off + R * size_t(hgroups) * 16 * 4, 256);
  const bool pairs = p->R >= kTopkSortRows && p->R <= kPairRows;
  P.off_pairc = off;
  if (pairs) off = align_up(off + R * kPairPhases * 4, 256);
  // Single-row decode step (one layout for every entry point): its histogram,
  // bin cursors and survivor slots start at zero.
  P.fused_row = decode_row_supported(*p) ? 1 : 0;
  P.off_lhist = off;
  if (P.fused_row) off = align_up(off + kRowHistBytes, 256);
  P.off_lcur = off;
  if (P.fused_row) off = align_up(off + kRowCursorBytes, 256);
  P.off_lsurv = off;
  if (P.fused_row) off = align_up(off + kRowSurvBytes, 256);
  P.zero_end = off;
  P.off_lkeep = off;
  if (P.fused_row) off = align_up(off + kRowKeepBytes, 256);
  P.off_surv = off; off = align_up(off + R * size_t(kCapFast) * 8, 256);
  P.off_scores = off; off = align_up(off + R * size_t(p->L_max) * 4, 256);
  const size_t dv = p->D_v > 0 ? size_t(p->D_v) : 0;
  P.off_apart = off;
  if (P.attn_kc_max > 1)
    off = align_up(off + R * size_t(hgroups) * P.attn_kc_max * (16 * dv + 32 * 16) * 4, 256);
  P.off_rpart = off;
  if (P.fused_row) off = align_up(off + decode_row_partials_bytes(*p), 256);
  P.off_pairx = 0;
  if (pairs) {
    P.off_pairx = off;
    off = align_up(off + R * pair_x_bytes(p->k), 256);
  }
  P.total = off;
  return DSA_OK;
}

dsa_status check_ws(const Plan& pl, void* ws, size_t ws_bytes) {
  if (!ws) return fail(DSA_ERR_INVALID_ARG, "workspace is NULL");
  if (!aligned(ws, 256)) return fail(DSA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (ws_bytes < pl.total)
    return fail(DSA_ERR_INVALID_ARG, "workspace %zu bytes < required %zu", ws_bytes, pl.total);
  return DSA_OK;
}

dsa_status run_indexer(const dsa_problem& p, const Plan& pl, int32_t* scores, char* ws,
                       cudaStream_t st) {
  if (p.R == 0) return DSA_OK;
  const int ix = p.flags & DSA_INDEXER_MASK;
  const bool tc = ix == DSA_INDEXER_TC || (ix == DSA_INDEXER_AUTO && indexer_tc_supported(p));
  // The indexer merges each row's key range into the row state as its CTAs
  // finish row groups, so the range must be zero before any CTA starts: a
  // memset here, except for the single-row step, whose indexer clears the
  // range itself (its row state is unused; its histogram has its own
  // clearing counter).
  if (!pl.fused_row) {
    cudaError_t z = cudaMemsetAsync(ws, 0, pl.zero_end, st);
    if (z != cudaSuccess) return cuda_fail(z, "clear workspace");
  }
  cudaError_t e = tc ? launch_indexer_tc(p, pl, scores, ws, st)
                     : launch_indexer_dp4a(p, pl, scores, ws, st);
  if (e != cudaSuccess) return cuda_fail(e, tc ? "indexer (tensor core)" : "indexer (dp4a)");
  return DSA_OK;
}

// Scratch of dsa_topk_static: the top-k's status block, row state, histograms
// and survivor lists, for problems whose top-k scratch fits in 4 MiB.
constexpr size_t kStaticScratchBytes = size_t(4) << 20;

}  // namespace

__device__ __align__(256) unsigned char g_topk_scratch[kStaticScratchBytes];

}  // namespace dsa

using namespace dsa;

extern "C" {

int dsa_version(void) { return 101; }

const char* dsa_last_error_string(void) { return g_err.c_str(); }

int dsa_indexer_kind(const dsa_problem* p) {
  Plan pl;
  if (make_plan(p, 0, &pl) != DSA_OK) return -1;
  const int ix = p->flags & DSA_INDEXER_MASK;
  const bool tc = ix == DSA_INDEXER_TC || (ix == DSA_INDEXER_AUTO && indexer_tc_supported(*p));
  return tc ? DSA_INDEXER_TC : DSA_INDEXER_DP4A;
}

int dsa_decode_step_kernels(const dsa_problem* p) {
  Plan pl;
  if (make_plan(p, 0, &pl) != DSA_OK) return -1;
  if (p->R == 0) return 0;
  return pl.fused_row ? 2 : 3;
}

size_t dsa_workspace_size(const dsa_problem* p) {
  Plan pl;
  if (make_plan(p, 0, &pl) != DSA_OK) return 0;
  return pl.total;
}

dsa_status dsa_index_scores(const dsa_problem* p, int32_t* scores, void* ws, size_t ws_bytes,
                            void* stream) {
  g_err.clear();
  Plan pl;
  dsa_status s = make_plan(p, kNeedIndexer, &pl);
  if (s != DSA_OK) return s;
  if ((s = check_ws(pl, ws, ws_bytes)) != DSA_OK) return s;
  if (p->R > 0 && p->L_max > 0 && !scores) return fail(DSA_ERR_INVALID_ARG, "scores is NULL");
  if (!aligned(scores, 16)) return fail(DSA_ERR_INVALID_ARG, "scores must be 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (p->R == 0) {  // nothing to score; still honour "clears the status word"
    cudaError_t e = cudaMemsetAsync(ws, 0, 256, st);
    if (e != cudaSuccess) return cuda_fail(e, "clear status");
    return DSA_OK;
  }
  return run_indexer(*p, pl, scores, static_cast<char*>(ws), st);
}

dsa_status dsa_topk(const dsa_problem* p, const int32_t* scores, int32_t* idx, int32_t* nsel,
                    void* ws, size_t ws_bytes, void* stream) {
  g_err.clear();
  Plan pl;
  dsa_status s = make_plan(p, kNeedTopk, &pl);
  if (s != DSA_OK) return s;
  if ((s = check_ws(pl, ws, ws_bytes)) != DSA_OK) return s;
  if (p->R > 0 && (!idx || (p->L_max > 0 && !scores)))
    return fail(DSA_ERR_INVALID_ARG, "scores/idx is NULL");
  if (!aligned(scores, 16)) return fail(DSA_ERR_INVALID_ARG, "scores must be 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(ws, 0, pl.zero_end, st);
  if (e != cudaSuccess) return cuda_fail(e, "clear workspace");
  if (p->R == 0) return DSA_OK;
  e = launch_topk(*p, pl, scores, idx, nsel, static_cast<char*>(ws), st, false);
  if (e != cudaSuccess) return cuda_fail(e, "top-k");
  return DSA_OK;
}

dsa_status dsa_topk_static(const dsa_problem* p, const int32_t* scores, int32_t* idx,
                           int32_t* nsel, void* stream) {
  g_err.clear();
  Plan pl;
  dsa_status s = make_plan(p, kNeedTopk, &pl);
  if (s != DSA_OK) return s;
  const size_t need = pl.off_scores;   // status block, row state, histograms, survivors
  if (need > kStaticScratchBytes)
    return fail(DSA_ERR_UNSUPPORTED,
                "dsa_topk_static: this problem needs %zu bytes of scratch; the static scratch "
                "holds %zu (use dsa_topk with a workspace)",
                need, kStaticScratchBytes);
  if (p->R > 0 && (!idx || (p->L_max > 0 && !scores)))
    return fail(DSA_ERR_INVALID_ARG, "scores/idx is NULL");
  if (!aligned(scores, 16)) return fail(DSA_ERR_INVALID_ARG, "scores must be 16-byte aligned");
  // The array's device address in the current device's context, looked up on
  // every call (it allocates nothing), so no stale address survives a device
  // reset or a change of context.
  void* base = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&base, g_topk_scratch);
  if (e != cudaSuccess) return cuda_fail(e, "static scratch address");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The status block, row state and histograms must start at zero; the exact
  // fallback runs on single CTAs (its pair buffers lie past the scratch).
  pl.off_pairx = 0;
  e = cudaMemsetAsync(base, 0, pl.zero_end, st);
  if (e != cudaSuccess) return cuda_fail(e, "clear static scratch");
  if (p->R == 0) return DSA_OK;
  e = launch_topk(*p, pl, scores, idx, nsel, static_cast<char*>(base), st, false);
  if (e != cudaSuccess) return cuda_fail(e, "top-k");
  return DSA_OK;
}

dsa_status dsa_sparse_attn(const dsa_problem* p, const int32_t* idx, const int32_t* nsel,
                           uint16_t* out, float* lse, void* ws, size_t ws_bytes, void* stream) {
  g_err.clear();
  Plan pl;
  dsa_status s = make_plan(p, kNeedAttn, &pl);
  if (s != DSA_OK) return s;
  if ((s = check_ws(pl, ws, ws_bytes)) != DSA_OK) return s;
  if (p->R > 0 && (!idx || !out)) return fail(DSA_ERR_INVALID_ARG, "idx/out is NULL");
  if (!aligned(out, 8)) return fail(DSA_ERR_INVALID_ARG, "out must be 8-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(ws, 0, pl.zero_end, st);   // status word and merge counters
  if (e != cudaSuccess) return cuda_fail(e, "clear workspace");
  if (p->R == 0) return DSA_OK;
  e = launch_attention(*p, pl, idx, nsel, out, lse, static_cast<char*>(ws), st);
  if (e != cudaSuccess) return cuda_fail(e, "sparse attention");
  return DSA_OK;
}

dsa_status dsa_decode_step(const dsa_problem* p, int32_t* idx, int32_t* nsel, uint16_t* out,
                           void* ws, size_t ws_bytes, void* stream) {
  g_err.clear();
  Plan pl;
  dsa_status s = make_plan(p, kNeedIndexer | kNeedTopk | kNeedAttn, &pl);
  if (s != DSA_OK) return s;
  if ((s = check_ws(pl, ws, ws_bytes)) != DSA_OK) return s;
  if (p->R > 0 && (!idx || !out)) return fail(DSA_ERR_INVALID_ARG, "idx/out is NULL");
  if (!aligned(out, 8)) return fail(DSA_ERR_INVALID_ARG, "out must be 8-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  cudaError_t e;
  if (p->R == 0) {
    e = cudaMemsetAsync(ws, 0, 256, st);
    if (e != cudaSuccess) return cuda_fail(e, "clear status");
    return DSA_OK;
  }
  int32_t* scores = reinterpret_cast<int32_t*>(w + pl.off_scores);
  if ((s = run_indexer(*p, pl, scores, w, st)) != DSA_OK) return s;
  if (pl.fused_row) {
    e = launch_decode_row(*p, pl, scores, idx, nsel, out, w, st);
    if (e != cudaSuccess) return cuda_fail(e, "selection and attention (one row)");
    return DSA_OK;
  }
  e = launch_topk(*p, pl, scores, idx, nsel, w, st, true);
  if (e != cudaSuccess) return cuda_fail(e, "top-k");
  e = launch_attention(*p, pl, idx, nsel, out, nullptr, w, st);
  if (e != cudaSuccess) return cuda_fail(e, "sparse attention");
  return DSA_OK;
}

// ------------------------------------------------------------------ front end

namespace {

// Workspace of the front end: status word, one arrival ticket per pass (at most
// R passes), per-pass head counters and the per-head maxima, all zeroed before
// the kernel; then the projections, rows padded to a multiple of 4 floats.
struct FrontPlan {
  int q_max, w_max, y_stride;
  size_t off_ticket, off_cnt, off_amax, zero_end, off_y, total;
};

dsa_status front_plan(const dsa_problem* p, int32_t d, FrontPlan* fp) {
  if (!p) return fail(DSA_ERR_INVALID_ARG, "problem is NULL");
  if (p->R < 0 || p->R > 65535) return fail(DSA_ERR_INVALID_ARG, "R=%d outside [0,65535]", p->R);
  if (p->H_i < 1 || p->H_i > 128) return fail(DSA_ERR_UNSUPPORTED, "H_i=%d outside [1,128]", p->H_i);
  if (p->D_i != 32 && p->D_i != 64 && p->D_i != 128 && p->D_i != 256)
    return fail(DSA_ERR_UNSUPPORTED, "D_i=%d not in {32,64,128,256}", p->D_i);
  if (d < 512 || d > 8192 || d % 512)
    return fail(DSA_ERR_UNSUPPORTED, "d=%d is not a multiple of 512 in [512,8192]", d);
  if (p->qk_abs_max < 0 || p->qk_abs_max > 128)
    return fail(DSA_ERR_INVALID_ARG, "qk_abs_max=%d outside [0,128]", p->qk_abs_max);
  if (p->w_abs_max < 0 || p->w_abs_max > (1 << 24))
    return fail(DSA_ERR_INVALID_ARG, "w_abs_max=%d outside [0,2^24]", p->w_abs_max);
  fp->q_max = (p->qk_abs_max == 0 || p->qk_abs_max == 128) ? 127 : p->qk_abs_max;
  fp->w_max = p->w_abs_max > 0 ? p->w_abs_max : 4;
  const size_t R = size_t(p->R);
  const int O = p->H_i * p->D_i + p->H_i;
  fp->y_stride = (O + 3) / 4 * 4;
  size_t off = 256;
  fp->off_ticket = off; off = align_up(off + R * 4, 256);
  fp->off_cnt = off; off = align_up(off + R * size_t(p->H_i) * 4, 256);
  fp->off_amax = off; off = align_up(off + R * size_t(p->H_i) * 4, 256);
  fp->zero_end = off;
  fp->off_y = off; off = align_up(off + R * size_t(fp->y_stride) * 4, 256);
  fp->total = off;
  return DSA_OK;
}

dsa_status check_affine(const dsa_affine_weights* w, const char* name) {
  if (!w || !w->codes || !w->scales || !w->biases)
    return fail(DSA_ERR_INVALID_ARG, "%s: codes, scales and biases must be set", name);
  if (!aligned(w->codes, 16) || !aligned(w->scales, 16) || !aligned(w->biases, 16))
    return fail(DSA_ERR_INVALID_ARG, "%s: codes, scales and biases must be 16-byte aligned", name);
  return DSA_OK;
}

}  // namespace

size_t dsa_front_end_workspace_size(const dsa_problem* p, int32_t d) {
  g_err.clear();
  FrontPlan fp;
  if (front_plan(p, d, &fp) != DSA_OK) return 0;
  return fp.total;
}

dsa_status dsa_indexer_front_end(const dsa_problem* p, int32_t d, const uint16_t* x,
                                 const dsa_affine_weights* wq, const dsa_affine_weights* ww,
                                 int8_t* q_idx, int32_t* w_idx, float* q_scale, float* w_scale,
                                 float* proj, void* ws, size_t ws_bytes, void* stream) {
  g_err.clear();
  FrontPlan fp;
  dsa_status s = front_plan(p, d, &fp);
  if (s != DSA_OK) return s;
  if (p->R == 0) return DSA_OK;
  if ((s = check_affine(wq, "wq")) != DSA_OK) return s;
  if ((s = check_affine(ww, "ww")) != DSA_OK) return s;
  if (!x || !q_idx || !w_idx) return fail(DSA_ERR_INVALID_ARG, "x, q_idx and w_idx must be set");
  if (!aligned(x, 16) || !aligned(q_idx, 16) || !aligned(w_idx, 4))
    return fail(DSA_ERR_INVALID_ARG, "x and q_idx must be 16-byte aligned, w_idx 4-byte");
  if (!aligned(q_scale, 4) || !aligned(w_scale, 4) || !aligned(proj, 4))
    return fail(DSA_ERR_INVALID_ARG, "q_scale, w_scale and proj must be 4-byte aligned");
  if (!ws || !aligned(ws, 256)) return fail(DSA_ERR_INVALID_ARG, "ws must be set and 256-byte aligned");
  if (ws_bytes < fp.total)
    return fail(DSA_ERR_INVALID_ARG, "ws_bytes=%zu below the required %zu", ws_bytes, fp.total);
  char* w = static_cast<char*>(ws);
  FrontArgs a;
  std::memset(&a, 0, sizeof a);
  a.wq = wq->codes; a.sq = wq->scales; a.bq = wq->biases;
  a.ww = ww->codes; a.sw = ww->scales; a.bw = ww->biases;
  a.x = x;
  a.R = p->R; a.d = d; a.H_i = p->H_i; a.D_i = p->D_i; a.Oq = p->H_i * p->D_i;
  a.q_max = fp.q_max; a.w_max = fp.w_max;
  a.y_stride = fp.y_stride;
  a.y = reinterpret_cast<float*>(w + fp.off_y);
  a.proj = proj;
  a.amax = reinterpret_cast<uint32_t*>(w + fp.off_amax);
  a.ticket = reinterpret_cast<uint32_t*>(w + fp.off_ticket);
  a.cnt = reinterpret_cast<uint32_t*>(w + fp.off_cnt);
  a.status = reinterpret_cast<uint32_t*>(w);
  a.wait_ns = kDefaultWaitNs;
  a.q_idx = q_idx; a.w_idx = w_idx; a.q_scale = q_scale; a.w_scale = w_scale;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(ws, 0, fp.zero_end, st);
  if (e != cudaSuccess) return cuda_fail(e, "clear workspace");
  e = launch_front_end(a, st);
  if (e != cudaSuccess) return cuda_fail(e, "indexer front end");
  return DSA_OK;
}

// ------------------------------------------------------------------ test hooks

static dsa_status check_limit(int64_t limit_ns, TestHooks* h) {
  if (limit_ns <= 0 || limit_ns > 10000000000ll)
    return fail(DSA_ERR_INVALID_ARG, "limit_ns=%lld outside (0, 1e10]", (long long)limit_ns);
  h->wait_ns = (uint64_t)limit_ns;
  return DSA_OK;
}

dsa_status dsa_test_topk_missing_arrival(const dsa_problem* p, const int32_t* scores, int32_t* idx,
                                         int32_t* nsel, void* ws, size_t ws_bytes, int skip_cta,
                                         int64_t limit_ns, void* stream) {
  g_err.clear();
  TestHooks h;
  dsa_status s = check_limit(limit_ns, &h);
  if (s != DSA_OK) return s;
  Plan pl;
  if ((s = make_plan(p, kNeedTopk, &pl)) != DSA_OK) return s;
  if ((s = check_ws(pl, ws, ws_bytes)) != DSA_OK) return s;
  if (p->R < 1 || !idx || !scores) return fail(DSA_ERR_INVALID_ARG, "need R >= 1, scores and idx");
  if (skip_cta < 0) return fail(DSA_ERR_INVALID_ARG, "skip_cta=%d < 0", skip_cta);
  h.topk_skip_cta = skip_cta;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(ws, 0, pl.zero_end, st);
  if (e != cudaSuccess) return cuda_fail(e, "clear workspace");
  e = launch_topk(*p, pl, scores, idx, nsel, static_cast<char*>(ws), st, false, &h);
  if (e != cudaSuccess) return cuda_fail(e, "top-k");
  return DSA_OK;
}

dsa_status dsa_test_attn_missing_gather(const dsa_problem* p, const int32_t* idx, const int32_t* nsel,
                                        uint16_t* out, float* lse, void* ws, size_t ws_bytes,
                                        int64_t limit_ns, void* stream) {
  g_err.clear();
  TestHooks h;
  dsa_status s = check_limit(limit_ns, &h);
  if (s != DSA_OK) return s;
  Plan pl;
  if ((s = make_plan(p, kNeedAttn, &pl)) != DSA_OK) return s;
  if ((s = check_ws(pl, ws, ws_bytes)) != DSA_OK) return s;
  if (p->R < 1 || !idx || !out) return fail(DSA_ERR_INVALID_ARG, "need R >= 1, idx and out");
  if (!aligned(out, 8)) return fail(DSA_ERR_INVALID_ARG, "out must be 8-byte aligned");
  h.attn_no_gather = 1;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(ws, 0, pl.zero_end, st);
  if (e != cudaSuccess) return cuda_fail(e, "clear workspace");
  e = launch_attention(*p, pl, idx, nsel, out, lse, static_cast<char*>(ws), st, &h);
  if (e != cudaSuccess) return cuda_fail(e, "sparse attention");
  return DSA_OK;
}

dsa_status dsa_test_indexer_missing_tile(const dsa_problem* p, int32_t* scores, void* ws,
                                         size_t ws_bytes, int64_t limit_ns, void* stream) {
  g_err.clear();
  TestHooks h;
  dsa_status s = check_limit(limit_ns, &h);
  if (s != DSA_OK) return s;
  Plan pl;
  if ((s = make_plan(p, kNeedIndexer, &pl)) != DSA_OK) return s;
  if ((s = check_ws(pl, ws, ws_bytes)) != DSA_OK) return s;
  if (p->R < 1 || !scores) return fail(DSA_ERR_INVALID_ARG, "need R >= 1 and scores");
  if (!aligned(scores, 16)) return fail(DSA_ERR_INVALID_ARG, "scores must be 16-byte aligned");
  const int ix = p->flags & DSA_INDEXER_MASK;
  if (ix == DSA_INDEXER_DP4A || !indexer_tc_tmem_operand(*p))
    return fail(DSA_ERR_UNSUPPORTED, "the hook needs the tensor-memory-operand indexer");
  h.indexer_no_load = 1;
  if (!pl.fused_row) {
    cudaError_t z = cudaMemsetAsync(ws, 0, pl.zero_end, static_cast<cudaStream_t>(stream));
    if (z != cudaSuccess) return cuda_fail(z, "clear workspace");
  }
  cudaError_t e = launch_indexer_tc(*p, pl, scores, static_cast<char*>(ws),
                                    static_cast<cudaStream_t>(stream), &h);
  if (e != cudaSuccess) return cuda_fail(e, "indexer (tensor core)");
  return DSA_OK;
}

dsa_status dsa_check_bounds(const dsa_problem* p, int64_t key_row0, int64_t key_rows, void* ws,
                            size_t ws_bytes, void* stream) {
  g_err.clear();
  if (!p) return fail(DSA_ERR_INVALID_ARG, "problem is NULL");
  if (!ws || !aligned(ws, 256) || ws_bytes < 256)
    return fail(DSA_ERR_INVALID_ARG, "ws must be set, 256-byte aligned and at least 256 bytes");
  if (p->R < 0 || p->H_i < 1 || p->H_i > 128 || p->D_i < 16 || p->D_i % 16)
    return fail(DSA_ERR_INVALID_ARG, "R=%d, H_i=%d, D_i=%d out of range", p->R, p->H_i, p->D_i);
  if (p->qk_abs_max < 0 || p->qk_abs_max > 128 || p->w_abs_max < 0)
    return fail(DSA_ERR_INVALID_ARG, "declared bounds out of range");
  if (key_row0 < 0 || key_rows < 0 || key_row0 + key_rows > p->L_total)
    return fail(DSA_ERR_INVALID_ARG, "key rows [%lld, %lld) outside [0, L_total=%lld)", (long long)key_row0,
                (long long)(key_row0 + key_rows), (long long)p->L_total);
  if ((key_rows > 0 && !p->k_idx) || (p->R > 0 && (!p->q_idx || !p->w_idx)))
    return fail(DSA_ERR_INVALID_ARG, "k_idx/q_idx/w_idx must be set");
  if (!aligned(p->k_idx, 16) || !aligned(p->q_idx, 16) || !aligned(p->w_idx, 4))
    return fail(DSA_ERR_INVALID_ARG, "k_idx/q_idx must be 16-byte aligned, w_idx 4-byte");
  const int qk = p->qk_abs_max > 0 ? p->qk_abs_max : 128;
  const int wm = p->w_abs_max > 0 ? p->w_abs_max : 4;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(ws, 0, 256, st);
  if (e != cudaSuccess) return cuda_fail(e, "clear status");
  const size_t D = size_t(p->D_i), R = size_t(p->R), H = size_t(p->H_i);
  e = launch_check_bounds(p->k_idx ? p->k_idx + size_t(key_row0) * D : nullptr, size_t(key_rows) * D, p->q_idx,
                          R * H * D, p->w_idx, R * H, qk, wm, static_cast<uint32_t*>(ws), st);
  if (e != cudaSuccess) return cuda_fail(e, "bound check");
  return DSA_OK;
}

dsa_status dsa_get_device_status(void* ws, void* stream) {
  int32_t bits = 0;
  return dsa_read_device_status(ws, stream, &bits);
}

dsa_status dsa_read_device_status(void* ws, void* stream, int32_t* bits) {
  g_err.clear();
  if (!ws || !bits) return fail(DSA_ERR_INVALID_ARG, "ws/bits is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  uint32_t v = 0;
  e = cudaMemcpy(&v, ws, sizeof v, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read status");
  *bits = static_cast<int32_t>(v);
  if (v & DSA_DEVICE_TIMEOUT) return fail(DSA_ERR_TIMEOUT, "a bounded device wait ran out");
  if (v & DSA_DEVICE_BAD_INDEX) return fail(DSA_ERR_DEVICE_INDEX, "an out-of-range index was skipped");
  if (v & DSA_DEVICE_RANGE) return fail(DSA_ERR_RANGE, "an operand exceeds its declared bound");
  return DSA_OK;
}

}  // extern "C"
