/*
 * libdsa test hooks: run an entry point with one of its bounded device waits
 * made to run out on purpose, so that a test can check what the library does
 * when a wait expires -- without faulting, trapping or hanging the GPU.  The
 * pages have no counterpart: these exist only to test the failure path that
 * every bounded wait in the library shares (the wait gives up after
 * `limit_ns` nanoseconds, sets DSA_DEVICE_TIMEOUT in the workspace's status
 * word, waits once more, also bounded, for any copy it still has in flight,
 * and the kernel returns; the CUDA context stays usable).
 *
 * Each hook arranges that a wait can never be satisfied while nothing is left
 * in flight: a CTA that returns without arriving at a grid barrier, or an
 * mbarrier armed for bytes whose copy is never issued.  `limit_ns` (> 0, at
 * most 10 s) replaces the normal 2 s limit of every wait in that call, so a
 * test finishes in milliseconds.  Arguments, validation and outputs are those
 * of the entry point named; after a timeout its outputs are unspecified,
 * except where stated.
 */
#ifndef DSA_TESTING_H
#define DSA_TESTING_H

#include "dsa.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * dsa_topk with CTA `skip_cta` of its cooperative grid returning before its
 * first grid barrier: the other CTAs' barrier waits run out, raise
 * DSA_DEVICE_TIMEOUT and return.  `skip_cta` must be below the grid size
 * (the device's SM count, or fewer CTAs for small problems: 0 is always
 * valid).
 */
DSA_API dsa_status dsa_test_topk_missing_arrival(const dsa_problem* p, const int32_t* scores,
                                                 int32_t* idx, int32_t* nsel, void* ws,
                                                 size_t ws_bytes, int skip_cta, int64_t limit_ns,
                                                 void* stream);

/*
 * dsa_sparse_attn with every CTA arming the barrier of its first gathered
 * tile but issuing none of the tile's row copies: each CTA's wait runs out,
 * raises DSA_DEVICE_TIMEOUT, and the rows it serves get no output -- their
 * `out` and `lse` entries are left untouched.
 */
DSA_API dsa_status dsa_test_attn_missing_gather(const dsa_problem* p, const int32_t* idx,
                                                const int32_t* nsel, uint16_t* out, float* lse,
                                                void* ws, size_t ws_bytes, int64_t limit_ns,
                                                void* stream);

/*
 * dsa_index_scores on the tensor-core indexer with the A operand in tensor
 * memory (D_i = 128, up to 128 accumulator columns per tile, L_total >= 128;
 * other shapes return DSA_ERR_UNSUPPORTED), every CTA arming the barrier of its
 * first key tile but issuing no copy for it: the converters' wait runs out,
 * the CTA's other roles stop at their next wait, and the kernel frees its
 * tensor memory and returns.
 */
DSA_API dsa_status dsa_test_indexer_missing_tile(const dsa_problem* p, int32_t* scores, void* ws,
                                                 size_t ws_bytes, int64_t limit_ns, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* DSA_TESTING_H */
