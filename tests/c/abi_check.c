/* Host-only use of libdsa from plain C99: the header compiles as C, the
 * library links, and the entry points that need no GPU behave as documented
 * (version, workspace size, host validation before any launch).  Prints one
 * line per check; exits non-zero on the first failure. */
#include <stddef.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "dsa.h"
#include "dsa_front_end.h"

#define BAD_WS ((void*)(uintptr_t)0x100010)

#define CHECK(cond, what)                                  \
  do {                                                     \
    if (!(cond)) {                                         \
      printf("FAIL %s\n", what);                           \
      return 1;                                            \
    }                                                      \
    printf("ok %s\n", what);                               \
  } while (0)

static dsa_problem mla_problem(int R, int L) {
  dsa_problem p;
  memset(&p, 0, sizeof p);
  p.R = R; p.B = 1; p.H_i = 64; p.D_i = 128; p.H_q = 64; p.D_k = 576; p.D_v = 512;
  p.k = 2048; p.L_max = L; p.L_total = L; p.softmax_scale = 1.0f / 24.0f;
  return p;
}

int main(void) {
  CHECK(dsa_version() == 101, "version 101");
  CHECK(sizeof(dsa_problem) == 136, "struct size 136");
  CHECK(offsetof(dsa_problem, L_total) == 40 && offsetof(dsa_problem, q_idx) == 64 &&
            offsetof(dsa_problem, kv_scale) == 128,
        "field offsets");

  dsa_problem p = mla_problem(1, 65536);
  const size_t ws = dsa_workspace_size(&p);
  CHECK(ws > 0 && ws % 256 == 0, "workspace size");
  dsa_problem q = mla_problem(1, 307200);
  CHECK(dsa_workspace_size(&q) > ws, "workspace grows with length");

  p.k = 0;
  CHECK(dsa_workspace_size(&p) == 0 && strstr(dsa_last_error_string(), "k=0") != NULL,
        "k = 0 rejected with a message");
  p.k = 2048;

  /* Host validation happens before any launch.  Every call below passes a
   * misaligned workspace (BAD_WS), so even a check that failed to fire would
   * be stopped by the workspace check: nothing reaches a device. */
  int32_t idx[4];
  uint16_t out[4];
  CHECK(dsa_decode_step(&p, idx, NULL, out, BAD_WS, (size_t)1 << 40, NULL) ==
            DSA_ERR_INVALID_ARG,
        "null problem pointers rejected");
  p.q_idx = (const int8_t*)(uintptr_t)0x100000;
  p.w_idx = (const int32_t*)(uintptr_t)0x100000;
  p.k_idx = (const int8_t*)(uintptr_t)0x100000;
  p.q = (const uint16_t*)(uintptr_t)0x100000;
  p.kv = (const uint16_t*)(uintptr_t)0x100000;
  p.offsets = (const int32_t*)(uintptr_t)0x100000;
  p.row_offsets = (const int32_t*)(uintptr_t)0x100000;
  p.row_len = (const int32_t*)(uintptr_t)0x100000;
  CHECK(dsa_decode_step(&p, idx, NULL, out, BAD_WS, (size_t)1 << 40, NULL) ==
            DSA_ERR_INVALID_ARG && strstr(dsa_last_error_string(), "256-byte") != NULL,
        "misaligned workspace rejected");
  p.flags = 0x400;
  CHECK(dsa_workspace_size(&p) == 0, "unknown flag rejected");
  p.flags = DSA_FLAG_KV_FP8;
  p.kv_scale = (const float*)(uintptr_t)0x100002;
  CHECK(dsa_sparse_attn(&p, idx, NULL, out, NULL, BAD_WS, (size_t)1 << 40, NULL) ==
            DSA_ERR_INVALID_ARG &&
            strstr(dsa_last_error_string(), "kv_scale") != NULL,
        "misaligned FP8 scales rejected");
  p.flags = 0;
  p.w_abs_max = 1 << 20;
  CHECK(dsa_index_scores(&p, (int32_t*)(uintptr_t)0x100000, BAD_WS, (size_t)1 << 40, NULL) ==
            DSA_ERR_OVERFLOW_RISK,
        "overflow bound rejected");
  {
    dsa_problem f = mla_problem(1, 4096);
    dsa_affine_weights w;
    w.codes = (const uint8_t*)(uintptr_t)0x100000;
    w.scales = (const uint16_t*)(uintptr_t)0x100000;
    w.biases = (const uint16_t*)(uintptr_t)0x100000;
    const size_t n = dsa_front_end_workspace_size(&f, 6144);
    CHECK(n > 0 && n % 256 == 0, "front-end workspace size");
    CHECK(dsa_indexer_front_end(&f, 6144, (const uint16_t*)(uintptr_t)0x100008, &w, &w,
                                (int8_t*)(uintptr_t)0x100000, (int32_t*)(uintptr_t)0x100000, NULL,
                                NULL, NULL, BAD_WS, n, NULL) == DSA_ERR_INVALID_ARG,
          "misaligned hidden rows rejected");
  }
  printf("all ok\n");
  return 0;
}
