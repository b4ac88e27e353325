/*
 * libdsa -- the decode step of a DSA (DeepSeek-style sparse attention) layer,
 * written for NVIDIA GB300 (sm_103a).
 *
 * One decode step of a DSA layer ("ds4 glm53-m3ultra", page 1: the model's
 * attention works over roughly 2,048 selected positions at 62k and at 300k
 * context; what grows with context is finding them):
 *
 *   1. indexer scores   s[r,t] = sum_h w[r,h] * max(0, q_idx[r,h,:] . k_idx[t,:])
 *                       for every visible cached position t of query row r;
 *   2. ordered top-k    the min(k, len) best positions, ordered by score
 *                       descending, then position ascending ("same positions
 *                       selected, same order");
 *   3. sparse attention softmax attention of every query head over the selected
 *                       latent rows only; key = all D_k columns of the row, value
 *                       = its first D_v columns (the latent, absorbed-MLA cache
 *                       of "glm53-tensorfold-spark", page 4).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensor pointers are DEVICE pointers owned by the caller; the library
 *   never allocates or frees memory.  Scratch memory is the caller's workspace
 *   (`ws`, at least dsa_workspace_size() bytes, 256-byte aligned), which matches
 *   the pre-grown selection scratch of "glm53-tensorfold-spark" (page 4).
 * - Every call is asynchronous on `stream` (a cudaStream_t passed as void*,
 *   NULL = the legacy default stream) and enqueues no host synchronisation, so
 *   it may be captured in a CUDA graph.  Calls are reentrant; the only global
 *   state is the thread-local error string.
 * - Host-side validation failures return a non-zero dsa_status and enqueue
 *   nothing; dsa_last_error_string() then says why.  Problems found on the device
 *   (an out-of-range index handed to dsa_sparse_attn, a bounded wait that ran
 *   out) never trap: the kernel skips the access, sets a bit in the workspace's
 *   status word, and carries on; read it with dsa_read_device_status().
 * - Each entry point clears the status word before its own kernels run.
 * - dsa_topk and dsa_decode_step launch one cooperative kernel (at most one CTA
 *   per SM, all resident at once); dsa_sparse_attn and dsa_decode_step launch
 *   thread-block clusters of up to 8 CTAs.  A launch the device cannot place
 *   returns DSA_ERR_CUDA and enqueues nothing further.
 *
 * Layouts (row-major, no padding unless stated)
 * ---------------------------------------------
 *   q_idx   int8  [R, H_i, D_i]   indexer query of each row, one vector per head
 *   w_idx   int32 [R, H_i]        indexer head weights of each row
 *   k_idx   int8  [L_total, D_i]  indexer key of each cached position, shared by
 *                                 all indexer heads; 16-byte aligned base
 *   q       bf16  [R, H_q, D_k]   attention queries (uint16 bit patterns)
 *   kv      bf16  [L_total, D_k]  latent cache rows; 16-byte aligned base.  With
 *                                 DSA_FLAG_KV_FP8: e4m3 bytes [L_total, D_k]
 *   kv_scale fp32 [L_total]       DSA_FLAG_KV_FP8 only: row j of the cache holds
 *                                 kv_scale[j] * e4m3(kv[j, :]); NULL = all 1
 *   offsets     int32 [B+1]  cache rows of request b: offsets[b] .. offsets[b+1]-1;
 *                            offsets[0] = 0 and offsets[B] = L_total
 *   row_offsets int32 [B+1]  query rows of request b: row_offsets[b] .. row_offsets[b+1]-1;
 *                            row_offsets[0] = 0 and row_offsets[B] = R
 *   row_len     int32 [R]    row r sees request-local positions 0 .. row_len[r]-1
 *                            (row_len[r] <= its request's length).  Validity comes
 *                            from each row's own length, never from padding
 *                            ("GLM-5.3-Flash-Alis-MLX-4bit", page 3, indexer
 *                            padding fix).
 *   scores  int32 [R, L_max]      entry (r, t) for t < row_len[r]; others untouched
 *   idx     int32 [R, k]          request-local positions; entries past nsel[r] = -1
 *   nsel    int32 [R]             min(k, row_len[r])
 *   out     bf16  [R, H_q, D_v]   round-to-nearest-even; 8-byte aligned base
 *   lse     fp32  [R, H_q]        natural-log log-sum-exp of the scaled logits
 */
#ifndef DSA_H
#define DSA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DSA_API __attribute__((visibility("default")))
#else
#define DSA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dsa_status {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1,     /* null/misaligned pointer, bad size            */
  DSA_ERR_UNSUPPORTED = 2,     /* valid but outside the library's shape limits */
  DSA_ERR_OVERFLOW_RISK = 3,   /* declared value ranges could overflow int32   */
  DSA_ERR_CUDA = 4,            /* a CUDA runtime call failed                    */
  DSA_ERR_TIMEOUT = 5,         /* device: a bounded wait ran out (status bit)   */
  DSA_ERR_DEVICE_INDEX = 6,    /* device: out-of-range index skipped (status)   */
  DSA_ERR_RANGE = 7            /* device: an operand outside its declared bound */
} dsa_status;

/* Device status bits, as returned by dsa_read_device_status(). */
#define DSA_DEVICE_TIMEOUT      0x1
#define DSA_DEVICE_BAD_INDEX    0x2
#define DSA_DEVICE_CAPACITY     0x4
#define DSA_DEVICE_RANGE        0x8   /* dsa_check_bounds: an operand exceeds its declared bound */

/* dsa_problem.flags */
#define DSA_INDEXER_AUTO   0   /* tensor-core indexer where supported, else dp4a */
#define DSA_INDEXER_DP4A   1   /* CUDA-core dp4a dot products                     */
#define DSA_INDEXER_TC     2   /* tcgen05 tensor-core tiles (exact, fp16 operands) */
#define DSA_INDEXER_MASK   0xF
#define DSA_FLAG_NO_RELU   0x100  /* score without the per-head max(0, .)        */
#define DSA_FLAG_KV_FP8    0x200  /* latent cache stored as FP8 e4m3, one fp32
                                     scale per row ("glm53-tensorfold-spark",
                                     page 4: FP8 KV storage)                    */

/*
 * One decode-step problem.  Sizes are host values; pointers are device pointers
 * (any of them may be NULL for an entry point that does not read it).
 *
 *   R        query rows (1 per request for plain decode; several per request for
 *            chunked queries)                                 0 <= R <= 65535
 *   B        requests (packed caches)                         1 <= B <= 4096
 *   H_i,D_i  indexer heads and dim       1 <= H_i <= 128, D_i in {32,64,128,256}
 *   H_q      attention heads                                  1 <= H_q <= 128
 *   D_k,D_v  latent row width (key) and value width: D_k % 16 == 0, D_k <= 576,
 *            D_v % 32 == 0, D_v <= D_k, D_v <= 512
 *   k        top-k                                            1 <= k <= 4096
 *   L_max    >= max(row_len); the row stride of `scores`      L_max < 2^31
 *   L_total  offsets[B] (rows in k_idx and kv)                L_total < 2^31
 *   qk_abs_max  caller's bound on |q_idx| and |k_idx| (0 = 128, the int8 limit)
 *   w_abs_max   caller's bound on |w_idx| (0 = 4)
 *            The host rejects (DSA_ERR_OVERFLOW_RISK) any problem whose bound
 *            H_i * w_abs_max * D_i * qk_abs_max^2 reaches 2^31: scores are int32.
 *   softmax_scale  multiplies q . k before the softmax
 *   flags    DSA_INDEXER_* | DSA_FLAG_NO_RELU | DSA_FLAG_KV_FP8
 *   kv_scale read only with DSA_FLAG_KV_FP8 (so callers built against the
 *            shorter struct of ABI 100, which never set that flag, still work)
 *
 * FP8 cache (DSA_FLAG_KV_FP8).  Byte (j, d) of kv is an OCP FP8 E4M3 code:
 * sign, 4 exponent bits (bias 7), 3 mantissa bits; subnormals when the exponent
 * field is 0; S.1111.111 is NaN; no infinities (largest finite 448).  The row's
 * value is kv_scale[j] times the decoded code.  Attention is the same function
 * of the dequantised rows as for a bf16 cache; the codes are widened exactly
 * and the scale is applied in fp32 to the logits and the softmax weights.
 */
typedef struct dsa_problem {
  int32_t R, B, H_i, D_i, H_q, D_k, D_v, k;
  int32_t L_max;
  int32_t flags;
  int64_t L_total;
  int32_t qk_abs_max;
  int32_t w_abs_max;
  float softmax_scale;
  int32_t reserved0;
  const int8_t* q_idx;
  const int32_t* w_idx;
  const int8_t* k_idx;
  const uint16_t* q;
  const uint16_t* kv;
  const int32_t* offsets;
  const int32_t* row_offsets;
  const int32_t* row_len;
  const float* kv_scale;
} dsa_problem;

/* Library ABI version (major * 100 + minor). */
DSA_API int dsa_version(void);

/* Thread-local text of the last host-side error ("" if none). */
DSA_API const char* dsa_last_error_string(void);

/* Which indexer dsa_index_scores / dsa_decode_step will run for `p`:
 * DSA_INDEXER_DP4A or DSA_INDEXER_TC (host only; -1 if `p` is invalid). */
DSA_API int dsa_indexer_kind(const dsa_problem* p);

/* Kernels dsa_decode_step launches for problem `p`: 2 for a single query row
 * of one request with 64 attention heads and a bf16 cache (indexer, then
 * selection and attention in one kernel), else 3 (indexer, top-k, attention);
 * 0 when R = 0; -1 if `p` is invalid (host only). */
DSA_API int dsa_decode_step_kernels(const dsa_problem* p);

/* Bytes of workspace every entry point below needs for problem `p` (host only;
 * 0 if `p` is invalid -- dsa_last_error_string() says why). */
DSA_API size_t dsa_workspace_size(const dsa_problem* p);

/*
 * Step 1, the lightning indexer ("ds4 glm53-m3ultra", page 1: every cached
 * position is scored against the current query).  Writes scores[r, t] for
 * t < row_len[r]; the integer result is exact.  Reads q_idx, w_idx, k_idx,
 * offsets, row_offsets, row_len.
 */
DSA_API dsa_status dsa_index_scores(const dsa_problem* p, int32_t* scores,
                            void* ws, size_t ws_bytes, void* stream);

/*
 * Step 2, the exact ordered top-k ("ds4 glm53-m3ultra", page 1: parallel scans
 * narrow the candidates, a small surviving list is sorted, and an exact path
 * resolves ambiguous ties; same positions in the same order).  Reads
 * scores[r, 0:row_len[r]] (row stride L_max), offsets/row_offsets/row_len;
 * writes idx [R, k] (ordered by score desc, position asc; -1 past nsel[r]) and
 * nsel [R] (may be NULL).
 */
DSA_API dsa_status dsa_topk(const dsa_problem* p, const int32_t* scores, int32_t* idx,
                    int32_t* nsel, void* ws, size_t ws_bytes, void* stream);

/*
 * Step 2 without a caller workspace.  The pages have no counterpart: this is
 * an interface for callers that hold no device allocator where they call the
 * top-k (a host plugin interface that passes only input and output buffers),
 * or on a latency-critical path where a cudaMalloc, which may synchronise the
 * device, is not acceptable.
 *
 * Same inputs, outputs and results as dsa_topk.  Its scratch is a 4 MiB array
 * in the library's own device memory, fixed at load time; nothing is allocated
 * or freed.  A problem whose top-k scratch (status block, 64 B of row state,
 * the row histograms and 32 KB of survivor keys per row) exceeds 4 MiB is
 * rejected with DSA_ERR_UNSUPPORTED and a message giving both sizes; use
 * dsa_topk with a workspace then.  A row takes 40 KB to 96 KB (1 to 8
 * histogram copies, more for long rows split over many CTAs), so roughly 40
 * to 100 rows fit.
 *
 * - Every call looks the array's address up in the current device's context
 *   (cudaGetSymbolAddress, which allocates nothing), so a device reset or a
 *   new context never leaves a stale address behind.  The first call in a
 *   process may load the library's device code; make it before any stream
 *   capture begins.
 * - Every call first clears the scratch's status block, row state and
 *   histograms (cudaMemsetAsync on `stream`); the rest needs no clearing.
 * - All calls share the one array: two calls whose executions overlap (on
 *   different streams, or on different host threads without ordering) race
 *   and give wrong results.  Order them on one stream.
 * - Device status bits land in the shared array, not in a caller workspace,
 *   so dsa_read_device_status cannot report them.
 */
DSA_API dsa_status dsa_topk_static(const dsa_problem* p, const int32_t* scores, int32_t* idx,
                                   int32_t* nsel, void* stream);

/*
 * Step 3, sparse MLA attention over the selected rows only ("ds4
 * glm53-m3ultra", page 1; latent cache of "glm53-tensorfold-spark", page 4).
 * Reads q, kv (and kv_scale for an FP8 cache), offsets, row_offsets, row_len,
 * idx [R, k] and nsel [R] (NULL means min(k, row_len[r]) entries per row).
 * An index outside [0, request length) is skipped and raises
 * DSA_DEVICE_BAD_INDEX.  Writes out [R, H_q, D_v] bf16 and, if non-NULL,
 * lse [R, H_q].  A row with no selected position gets zeros (lse = -inf).
 */
DSA_API dsa_status dsa_sparse_attn(const dsa_problem* p, const int32_t* idx,
                           const int32_t* nsel, uint16_t* out, float* lse,
                           void* ws, size_t ws_bytes, void* stream);

/*
 * Steps 1-3 on one stream with no host synchronisation: the fused decode step.
 * Writes idx [R, k], nsel [R] (may be NULL) and out [R, H_q, D_v].  Scores stay
 * in the workspace.
 */
DSA_API dsa_status dsa_decode_step(const dsa_problem* p, int32_t* idx, int32_t* nsel,
                           uint16_t* out, void* ws, size_t ws_bytes, void* stream);

/*
 * Checks on the device that the operands respect the problem's declared
 * bounds: every |q_idx| and every |k_idx| of cached rows [key_row0, key_row0 +
 * key_rows) at most qk_abs_max (0 = no bound to check: int8 always fits), and
 * every |w_idx| at most w_abs_max (0 = 4).  The bounds are the caller's
 * promise (the indexer picks its exact operand format from them, and the
 * int32 overflow check relies on them); a step never re-reads the whole cache
 * to verify it, so a caller checks each key row once, when it is written to
 * the cache, and the per-step operands as it sees fit.  A violation sets
 * DSA_DEVICE_RANGE in the workspace's status word (cleared first by this
 * call); dsa_read_device_status then returns DSA_ERR_RANGE.  Reads p->R,
 * H_i, D_i, L_total, q_idx, w_idx (both may be NULL when R = 0), k_idx and the
 * bounds; ws needs 256 bytes.  One kernel, no host synchronisation.
 */
DSA_API dsa_status dsa_check_bounds(const dsa_problem* p, int64_t key_row0, int64_t key_rows, void* ws,
                                    size_t ws_bytes, void* stream);

/*
 * Synchronises `stream`, then reads the workspace's device status word into
 * *bits (DSA_DEVICE_* bits; 0 = clean).  Returns DSA_ERR_TIMEOUT,
 * DSA_ERR_DEVICE_INDEX or DSA_ERR_RANGE when the matching bit is set, else
 * DSA_OK.
 */
DSA_API dsa_status dsa_read_device_status(void* ws, void* stream, int32_t* bits);

/*
 * The same check without the bits: synchronises `stream` and returns
 * DSA_ERR_TIMEOUT, DSA_ERR_DEVICE_INDEX, DSA_ERR_RANGE or DSA_OK from the
 * workspace's device status word (a CUDA failure returns DSA_ERR_CUDA).
 */
DSA_API dsa_status dsa_get_device_status(void* ws, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* DSA_H */
