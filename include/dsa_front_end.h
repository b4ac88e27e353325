/*
 * libdsa indexer front end: the integer indexer operands of each query row,
 * projected from the row's hidden vector.
 *
 * "GLM-5.3-Flash-Alis-MLX-4bit" (page 3, the Recipe table and the note under
 * it) keeps the DSA indexer projections at 8 bits in groups of 64, packed in
 * the standard MLX affine form.  A weight matrix [O, d] is then three arrays:
 *
 *   codes   uint8 [O, d]         code 0..255 of weight (o, i); 16-byte aligned
 *   scales  bf16  [O, d / 64]    scale of group (o, i / 64); 16-byte aligned
 *   biases  bf16  [O, d / 64]    bias of group (o, i / 64); 16-byte aligned
 *
 * and weight (o, i) = scales[o, i / 64] * codes[o, i] + biases[o, i / 64].
 * (MLX packs four 8-bit codes per little-endian uint32 word: the same bytes.)
 *
 * For each query row r with hidden vector x[r] (bf16 [d]):
 *
 *   qf[h, j] = sum_i Wq[h * D_i + j, i] * x[r, i]      Wq: [H_i * D_i, d]
 *   wf[h]    = sum_i Ww[h, i] * x[r, i]                Ww: [H_i, d]
 *   sigma_h  = max_j |qf[h, j]| / q_max
 *   q_idx[r, h, j] = clamp(round(qf[h, j] / sigma_h), -q_max, q_max)
 *   u_h      = wf[h] * sigma_h,   tau = max_h |u_h| / w_max
 *   w_idx[r, h]    = clamp(round(u_h / tau), -w_max, w_max)
 *
 * round = to nearest, ties to even; codes are 0 where sigma_h or tau is 0.
 * Each head's query scale folds into its weight (sigma_h > 0 commutes with the
 * indexer's max(0, .)), so tau times the indexer's integer score approximates
 * the score of the real-valued projections.  q_max and w_max are the problem's
 * declared bounds (qk_abs_max, 0 or 128 meaning 127; w_abs_max, 0 meaning 4), so
 * the output satisfies the declarations dsa_decode_step relies on.  The pages fix
 * only the weight format; the projection of one hidden vector per row and the
 * two scales are the plainest reading that fills the indexer's integer inputs.
 *
 * Precision: the projection accumulates in fp32 (every code * x product is
 * exact; their sums are rounded), so qf and wf are within about 2^-17 of the
 * sum of |terms| of the exact values, and a code whose exact ratio lies that
 * close to a rounding midpoint may differ by one from the exact-arithmetic code.
 * The scales and the codes are then computed from those fp32 values with IEEE
 * division.  Results are deterministic (no dependence on timing).
 */
#ifndef DSA_FRONT_END_H
#define DSA_FRONT_END_H

#include "dsa.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct dsa_affine_weights {
  const uint8_t* codes;
  const uint16_t* scales;
  const uint16_t* biases;
} dsa_affine_weights;

/* Workspace bytes dsa_indexer_front_end needs for p->R rows of width d (0 and
 * the error string set when p or d is invalid). */
DSA_API size_t dsa_front_end_workspace_size(const dsa_problem* p, int32_t d);

/*
 * Reads p->R, p->H_i (1..128), p->D_i (32, 64, 128 or 256), p->qk_abs_max and
 * p->w_abs_max; d is a multiple of 512 in [512, 8192].
 *
 *   x        bf16 [R, d]             hidden vectors, 16-byte aligned
 *   wq, ww   the query projection [H_i * D_i, d] and the head-weight
 *            projection [H_i, d], as above
 *   q_idx    int8  [R, H_i, D_i]     out; 16-byte aligned
 *   w_idx    int32 [R, H_i]          out; 4-byte aligned
 *   q_scale  fp32  [R, H_i]          out, sigma; may be NULL
 *   w_scale  fp32  [R]               out, tau; may be NULL
 *   proj     fp32  [R, H_i * D_i + H_i]  out, qf then wf; may be NULL
 *   ws       at least dsa_front_end_workspace_size(p, d) bytes, 256-byte aligned
 *
 * One kernel (after a memset of the workspace's counters) on `stream`, with no
 * host synchronisation; every pointer is a device pointer owned by the caller.
 * Host validation failures return non-zero and enqueue nothing.  Its waits are
 * bounded like the step's: a wait that runs out sets DSA_DEVICE_TIMEOUT in the
 * workspace's status word (dsa_read_device_status) and the outputs are then
 * unspecified.
 */
DSA_API dsa_status dsa_indexer_front_end(const dsa_problem* p, int32_t d, const uint16_t* x,
                                         const dsa_affine_weights* wq, const dsa_affine_weights* ww,
                                         int8_t* q_idx, int32_t* w_idx, float* q_scale,
                                         float* w_scale, float* proj, void* ws, size_t ws_bytes,
                                         void* stream);

#ifdef __cplusplus
}
#endif
#endif /* DSA_FRONT_END_H */
