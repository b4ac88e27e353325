// Sparse MLA attention over the selected latent rows: the positions are split
// over the CTAs of thread-block clusters, whose partial results are merged
// through distributed shared memory, then across clusters.
//
// For query row r and head h ("ds4 glm53-m3ultra", page 1: attention over the
// ~2048 selected positions only; latent cache of "glm53-tensorfold-spark",
// page 4: key = the whole D_k-wide latent row, value = its first D_v columns):
//   z_j = scale * q[r,h,:] . kv[idx_j, :],  o[h,:] = sum_j softmax(z)_j kv[idx_j, :D_v]
//
// attn_cluster_kernel  grid (C * Kc, head group of 16, row), cluster (C, 1, 1)
//   with C = 4 (k <= 2048) or 8, 4 warps.  With so many rows that one cluster
//   serves each (row, head group), a CTA of 16 warps serves 64 heads instead
//   (grid (C, H_q / 64, row)), so that each selected row is gathered once
//   rather than once per head group of 16.  The S = C * Kc CTAs of a (row,
//   head group) split the selected positions: CTA sp takes the tiles sp,
//   sp + S, ... of 64 positions (one tile at k = 2048).  It gathers the rows (one bulk copy per
//   whole row, as the front-axis gather of "GLM-5.3-Flash-Alis-MLX-4bit",
//   page 3), computes S = Q K^T and O += P V with bf16 mma.sync (fp32
//   accumulation) and an online softmax in fp32 (log2 domain), and leaves its
//   unnormalised O, running max m and sum l in shared memory.  After a cluster
//   barrier CTA x merges columns [x D_v / C, (x + 1) D_v / C) of the C partials
//   in CTA order.  With one cluster that is the bf16 output (round to nearest
//   even); with Kc > 1 each CTA writes its merged slice with (M, L) to the
//   workspace, and the last of the Kc CTAs of slice x to arrive (an atomic
//   counter, no waiting) merges the Kc slices in cluster order.
//
// FP8 cache (the FP8 KV storage of "glm53-tensorfold-spark", page 4): the rows
// are e4m3 codes with one fp32 scale per row.  The bulk copies land the codes in
// a staging buffer; all threads widen them to bf16 in the K buffer (exact: every
// e4m3 value is a bf16 value), after which the staging buffer takes the next
// tile's copies while this tile is computed.  The row scale s_j multiplies the
// logit (z_j = scale * s_j * q . code_j) and the softmax weight of the P V
// product (p_j s_j), both in fp32, so the result is attention over the
// dequantised rows s_j * code_j.
#include "common.cuh"
#include "ptx.cuh"

#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <math_constants.h>

namespace dsa {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
static_assert(kThreads == kAttnHeads * 8, "merge: eight lanes per head");
constexpr int kPStride = kAttnRows + 8;  // bf16 elements per P row in shared memory
constexpr int kMaxTiles = 8;             // tiles per CTA (k <= 4096 over >= 8 CTAs)
namespace cg = cooperative_groups;

struct AttnArgs {
  const uint16_t* q;
  const uint16_t* kv;      // bf16 rows, or e4m3 bytes with F8
  const float* kv_scale;   // F8: per-row scale, or null (= 1)
  const int32_t* offsets;
  const int32_t* row_offsets;
  const int32_t* row_len;
  const int32_t* idx;
  const int32_t* nsel;
  uint16_t* out;      // [R, H_q, D_v]
  float* lse;         // [R, H_q] or null
  uint32_t* status;
  float* apart;       // [R, head group, Kc, C] x (M[16], L[16], O[16][D_v / C]) when Kc > 1
  uint32_t* acnt;     // [R, head group, 16] arrivals per column slice (zeroed)
  int Kc;             // clusters per (row, head group)
  int B, H_q, D_k, D_v, k;
  int L1;             // B == 1: the request's length (L_total), known on the host
  int qs, ks;         // shared-memory row strides (elements)
  float scale_log2;
  uint64_t wait_ns;   // bound of every mbarrier wait (then DSA_DEVICE_TIMEOUT)
  int test_no_gather; // test hook: arm the first gather's barrier but issue no copy
};

__device__ int row_request(const int32_t* row_offsets, int B, int r) {
  int lo = 0, hi = B - 1;  // largest b with row_offsets[b] <= r
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (row_offsets[mid] <= r) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// NT: output n-tiles (of 8 columns) per warp; 4 warps cover 32*NT >= D_v columns.
// F8: the cache holds e4m3 codes and per-row scales.
// HG: head groups of 16 per CTA (1, or 4 for many rows: each gathered tile then
// serves 64 heads; warp w computes head group w / 4, columns (w % 4) * 8 * NT..).
template <int NT, bool F8, int HG>
__global__ void __launch_bounds__(kThreads * HG) attn_cluster_kernel(AttnArgs a) {
  constexpr int NH = kAttnHeads * HG;   // heads per CTA
  constexpr int NTH = kThreads * HG;    // threads per CTA (eight per head in the merge)
  constexpr int NW = kWarps * HG;
  static_assert(NTH == NH * 8, "merge: eight lanes per head");
  extern __shared__ __align__(16) unsigned char smem[];
  uint16_t* Qs = reinterpret_cast<uint16_t*>(smem);                          // [NH][qs]
  uint16_t* Kb = Qs + NH * a.qs;                                            // [64][ks]
  uint16_t* Ps = Kb + kAttnRows * a.ks;                                     // [HG][16][kPStride]
  float* red = reinterpret_cast<float*>(Ps + NH * kPStride);                // [2][NW][16]
  float* mls = red + 2 * NW * kAttnHeads;                                   // [NH][2]: m, l
  float* mall = mls + 2 * NH;                                               // [16][NH][2]
  float* wts = mall + 16 * NH * 2;                                          // [C][NH]
  float* invl = wts + 16 * NH;                                              // [NH]
  float* mlc = invl + NH;                                                   // [2][NH]: cluster M, L
  int* idx_s = reinterpret_cast<int*>(mlc + 2 * NH);                       // [kMaxTiles][64]
  float* sc_s = reinterpret_cast<float*>(idx_s + kMaxTiles * kAttnRows);     // F8: [kMaxTiles][64]
  uint8_t* F8s = reinterpret_cast<uint8_t*>(sc_s + kMaxTiles * kAttnRows);  // F8: [64][D_k] codes
  // [NH][D_v] partial O after the tile loop: on the K buffer (HG = 1), or on
  // the queries and the K buffer (HG = 4; 64 D_v floats <= (qs + ks) bf16 rows).
  float* Ob = reinterpret_cast<float*>(HG == 1 ? reinterpret_cast<unsigned char*>(Kb) : smem);
  __shared__ int req_s, last_s;
  __shared__ int bad_s;                        // a bounded wait of this CTA ran out
  __shared__ __align__(8) uint64_t bars[2];   // queries, K buffer

  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster.num_blocks();
  const int x = (int)cluster.block_rank();
  const int kc = (int)blockIdx.x / C;        // cluster within (row, head group)
  const int S = a.Kc * C;                    // position splits of the row
  const int sp = kc * C + x;                 // this CTA's split: tiles sp, sp + S, ...
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int hg = warp >> 2, wq = warp & 3;   // head group of the warp, its quarter
  const int g = lane >> 2, c = lane & 3;
  const int r = blockIdx.z, h0 = blockIdx.y * NH;

  const uint32_t bar_q = smem_u32(&bars[0]);
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) mbar_init(smem_u32(&bars[i]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  pdl_wait();
  pdl_trigger();
  if (tid == 0 && a.B > 1) req_s = row_request(a.row_offsets, a.B, r);
  // This CTA's selected positions (masked below once n is known).
  const int32_t* idx_row = a.idx + (int64_t)r * a.k;
  for (int i = tid; i < kMaxTiles * kAttnRows; i += NTH) {
    const int p = (sp + (i / kAttnRows) * S) * kAttnRows + (i % kAttnRows);
    idx_s[i] = p < a.k ? idx_row[p] : -1;
  }
  __syncthreads();
  // One request: offsets = {0, L_total} (documented), no lookups.
  const int b = a.B > 1 ? req_s : 0;
  const int64_t base = a.B > 1 ? a.offsets[b] : 0;
  const int L_b = a.B > 1 ? a.offsets[b + 1] - a.offsets[b] : a.L1;
  const int rl = a.row_len[r];
  const int lim = min(rl, L_b);              // valid positions of this row: [0, row_len)
  int n = a.nsel ? a.nsel[r] : min(a.k, rl);
  n = max(0, min(n, a.k));
  const int ntiles = (n + kAttnRows - 1) / kAttnRows;
  const int my_tiles = ntiles > sp ? (ntiles - sp + S - 1) / S : 0;   // <= kMaxTiles
  for (int i = tid; i < my_tiles * kAttnRows; i += NTH) {
    const int p = (sp + (i / kAttnRows) * S) * kAttnRows + (i % kAttnRows);
    int t = idx_s[i];
    if (p >= n) {
      t = -1;
    } else if (t < 0 || t >= lim) {
      raise_status(a.status, DSA_DEVICE_BAD_INDEX);
      t = -1;
    }
    idx_s[i] = t;
  }

  __syncthreads();   // idx_s final
  // Whole rows by the bulk-copy engine, issued by warp 0: queries of this head
  // group (zero rows past H_q), then per tile its 64 selected latent rows
  // (zero rows where masked).  Each buffer's barrier counts the bytes.
  const uint32_t qrowb = (uint32_t)a.D_k * 2;
  const uint32_t rowb = F8 ? (uint32_t)a.D_k : qrowb;
  if (warp == 0) {
    const int nq = min(NH, a.H_q - h0);
    if (lane == 0) mbar_expect_tx(bar_q, (uint32_t)nq * qrowb);
    __syncwarp();
    for (int hq = lane; hq < NH; hq += 32) {
      if (hq < nq)
        bulk_row(smem_u32(Qs + hq * a.qs), a.q + ((int64_t)r * a.H_q + h0 + hq) * a.D_k, qrowb, bar_q);
      else
        for (int c8 = 0; c8 < a.D_k / 8; ++c8) *reinterpret_cast<int4*>(Qs + hq * a.qs + c8 * 8) = make_int4(0, 0, 0, 0);
    }
  }
  const uint32_t kbar = smem_u32(&bars[1]);
  auto gather = [&](int i) {   // this CTA's tile i into the K (F8: staging) buffer (warp 0)
    uint16_t* Ks = Kb;
    const uint8_t* kv8 = reinterpret_cast<const uint8_t*>(a.kv);
    const int* ids = idx_s + i * kAttnRows;
    const int t0 = ids[lane], t1 = ids[lane + 32];
    const uint32_t nv = __popc(__ballot_sync(0xffffffffu, t0 >= 0)) + __popc(__ballot_sync(0xffffffffu, t1 >= 0));
    // Test hook: the barrier expects the tile's bytes but no copy is issued, so
    // the wait for it runs out (no copy is in flight when it does).
    const bool issue = !(a.test_no_gather && i == 0);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // earlier zero fills of this buffer
    if (lane == 0) mbar_expect_tx(kbar, nv * rowb);
    __syncwarp();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int j = lane + 32 * h, t = (h ? t1 : t0) >= 0 && !issue ? -2 : (h ? t1 : t0);
      if (t == -2) continue;
      if (F8) {
        if (t >= 0)
          bulk_row(smem_u32(F8s + j * a.D_k), kv8 + (base + t) * a.D_k, rowb, kbar);
        else
          for (int c16 = 0; c16 < a.D_k / 16; ++c16) *reinterpret_cast<int4*>(F8s + j * a.D_k + c16 * 16) = make_int4(0, 0, 0, 0);
      } else {
        if (t >= 0)
          bulk_row(smem_u32(Ks + j * a.ks), a.kv + (base + t) * a.D_k, rowb, kbar);
        else
          for (int c8 = 0; c8 < a.D_k / 8; ++c8) *reinterpret_cast<int4*>(Ks + j * a.ks + c8 * 8) = make_int4(0, 0, 0, 0);
      }
    }
  };
  if (warp == 0 && my_tiles > 0) gather(0);
  if (F8) {   // row scales of this CTA's positions (0 where masked), while the copies fly
    for (int i = tid; i < my_tiles * kAttnRows; i += NTH) {
      const int t = idx_s[i];
      sc_s[i] = t < 0 ? 0.f : (a.kv_scale ? __ldg(a.kv_scale + base + t) : 1.f);
    }
  }
  // A wait that runs out makes the CTA stop: it waits once more (bounded) for
  // the copies it has in flight, computes nothing further, and its cluster
  // writes no output for this (row, head group) (see the merge below).
  const bool q_ok = mbar_wait(bar_q, 0, a.status, a.wait_ns);
  int bad = __syncthreads_or(!q_ok);
  if (bad) {
    if (tid == 0) {
      mbar_wait(bar_q, 0, nullptr, a.wait_ns);
      if (my_tiles > 0) mbar_wait(kbar, 0, nullptr, a.wait_ns);
    }
    __syncthreads();
  }

  float acc[NT][4];
#pragma unroll
  for (int i = 0; i < NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  float m_run[2] = {-CUDART_INF_F, -CUDART_INF_F};
  float l_run[2] = {0.f, 0.f};

  for (int i = 0; i < my_tiles && !bad; ++i) {
    if (!F8 && warp == 0 && i > 0) gather(i);   // the previous tile's math is done (barrier below)
    const bool ok = mbar_wait(kbar, (uint32_t)i & 1u, a.status, a.wait_ns);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) mbar_wait(kbar, (uint32_t)i & 1u, nullptr, a.wait_ns);   // drain this tile's copies
      __syncthreads();
      bad = 1;
      break;
    }
    if (F8) {
      // Widen the staged codes into the K buffer (the previous tile's math is
      // done: barrier at the end of the loop), then hand the staging buffer to
      // the next tile's copies.
      const int chunks = a.D_k / 16;
      for (int e = tid; e < kAttnRows * chunks; e += NTH) {
        const int row = e / chunks, ch = e - row * chunks;
        uint4 lo, hi;
        e4m3x16_to_bf16(*reinterpret_cast<const uint4*>(F8s + row * a.D_k + ch * 16), lo, hi);
        *reinterpret_cast<uint4*>(Kb + row * a.ks + ch * 16) = lo;
        *reinterpret_cast<uint4*>(Kb + row * a.ks + ch * 16 + 8) = hi;
      }
      __syncthreads();
      if (warp == 0 && i + 1 < my_tiles) gather(i + 1);
    }
    __syncthreads();
    const uint16_t* Ks = Kb;
    const int* ids = idx_s + i * kAttnRows;
    const float* scs = sc_s + i * kAttnRows;

    // S = Q K^T for kv rows [warp*16, warp*16+16).
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
      // Two accumulator pairs (even and odd k-steps) halve the mma dependency chain.
      float s2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const int arow = (lane & 7) + ((lane >> 3) & 1) * 8, acol = (lane >> 4) * 8;
      const int brow = wq * 16 + (lane & 7) + (lane >> 4) * 8, bcol = ((lane >> 3) & 1) * 8;
      const uint32_t aaddr = smem_u32(Qs + (hg * kAttnHeads + arow) * a.qs + acol);
      const uint32_t baddr = smem_u32(Ks + brow * a.ks + bcol);
      const int nk = a.D_k / 16;
      int kk = 0;
      for (; kk + 1 < nk; kk += 2) {
        uint32_t a0, a1, a2, a3, b0, b1, b2, b3, e0, e1, e2, e3, f0, f1, f2, f3;
        ldsm_x4(aaddr + kk * 32, a0, a1, a2, a3);
        ldsm_x4(baddr + kk * 32, b0, b1, b2, b3);
        ldsm_x4(aaddr + kk * 32 + 32, e0, e1, e2, e3);
        ldsm_x4(baddr + kk * 32 + 32, f0, f1, f2, f3);
        mma16816(s[0], a0, a1, a2, a3, b0, b1);
        mma16816(s[1], a0, a1, a2, a3, b2, b3);
        mma16816(s2[0], e0, e1, e2, e3, f0, f1);
        mma16816(s2[1], e0, e1, e2, e3, f2, f3);
      }
      if (kk < nk) {
        uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
        ldsm_x4(aaddr + kk * 32, a0, a1, a2, a3);
        ldsm_x4(baddr + kk * 32, b0, b1, b2, b3);
        mma16816(s[0], a0, a1, a2, a3, b0, b1);
        mma16816(s[1], a0, a1, a2, a3, b2, b3);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        s[0][e] += s2[0][e];
        s[1][e] += s2[1][e];
      }
    }
    // Online softmax (rows g and g+8 of the head group; columns of this warp).
    float xv[2][4];
    float mx[2] = {-CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int col = wq * 16 + nt * 8 + 2 * c + (e & 1);
        const float sv = F8 ? s[nt][e] * scs[col] : s[nt][e];
        const float v = ids[col] >= 0 ? sv * a.scale_log2 : -CUDART_INF_F;
        xv[nt][e] = v;
        mx[e >> 1] = fmaxf(mx[e >> 1], v);
      }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 1));
      mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 2));
    }
    // Per-warp partial max and sum of each head, reduced over the 4 warps of
    // the head group (warps hg * 4 .. hg * 4 + 3).
    float* red_max = red;
    float* red_sum = red + NW * kAttnHeads;
    if (c == 0) {
      red_max[warp * kAttnHeads + g] = mx[0];
      red_max[warp * kAttnHeads + g + 8] = mx[1];
    }
    __syncthreads();
    float m_new[2], alpha[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float tm = -CUDART_INF_F;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) tm = fmaxf(tm, red_max[(hg * kWarps + w) * kAttnHeads + g + 8 * j]);
      m_new[j] = fmaxf(m_run[j], tm);
      alpha[j] = m_new[j] == -CUDART_INF_F ? 1.f : exp2f(m_run[j] - m_new[j]);
    }
    float ps[2] = {0.f, 0.f};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      float pv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float mm = m_new[e >> 1];
        pv[e] = (xv[nt][e] == -CUDART_INF_F) ? 0.f : exp2f(xv[nt][e] - mm);
        ps[e >> 1] += pv[e];
      }
      const int col = wq * 16 + nt * 8 + 2 * c;
      // F8: the weight of row j in O is p_j s_j (its sum l stays the plain p_j).
      const float w0 = F8 ? scs[col] : 1.f, w1 = F8 ? scs[col + 1] : 1.f;
      uint16_t* Pg = Ps + hg * kAttnHeads * kPStride;
      *reinterpret_cast<uint32_t*>(Pg + g * kPStride + col) = pack_bf16(pv[0] * w0, pv[1] * w1);
      *reinterpret_cast<uint32_t*>(Pg + (g + 8) * kPStride + col) = pack_bf16(pv[2] * w0, pv[3] * w1);
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      ps[j] += __shfl_xor_sync(0xffffffffu, ps[j], 1);
      ps[j] += __shfl_xor_sync(0xffffffffu, ps[j], 2);
    }
    if (c == 0) {
      red_sum[warp * kAttnHeads + g] = ps[0];
      red_sum[warp * kAttnHeads + g + 8] = ps[1];
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float ts = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) ts += red_sum[(hg * kWarps + w) * kAttnHeads + g + 8 * j];
      l_run[j] = l_run[j] * alpha[j] + ts;
      m_run[j] = m_new[j];
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      acc[nt][0] *= alpha[0]; acc[nt][1] *= alpha[0];
      acc[nt][2] *= alpha[1]; acc[nt][3] *= alpha[1];
    }
    // O += P V for output columns [wq*8*NT, (wq+1)*8*NT) of head group hg.
    {
      const int arow = (lane & 7) + ((lane >> 3) & 1) * 8, acol = (lane >> 4) * 8;
      const uint32_t paddr = smem_u32(Ps + (hg * kAttnHeads + arow) * kPStride + acol);
      const int vrow = (lane & 7) + ((lane >> 3) & 1) * 8, vcol = wq * 8 * NT + (lane >> 4) * 8;
      const uint32_t vaddr = smem_u32(Ks + vrow * a.ks + vcol);
#pragma unroll
      for (int kq = 0; kq < kAttnRows / 16; ++kq) {
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
    __syncthreads();  // the K buffer, Ps and red are rewritten next
  }
  __syncthreads();
  if (bad) {   // a neutral partial: nothing of this CTA enters the merge
#pragma unroll
    for (int i = 0; i < NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    m_run[0] = m_run[1] = -CUDART_INF_F;
    l_run[0] = l_run[1] = 0.f;
  }
  if (tid == 0) bad_s = bad;

  // This CTA's unnormalised partial O, m and l, for the cluster to read.
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    float* dst = Ob + (hg * kAttnHeads + g + 8 * j) * a.D_v;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int col = wq * 8 * NT + nt * 8 + 2 * c;
      if (col < a.D_v) *reinterpret_cast<float2*>(dst + col) = make_float2(acc[nt][2 * j], acc[nt][2 * j + 1]);
    }
    if (wq == 0 && c == 0) {
      mls[(hg * kAttnHeads + g + 8 * j) * 2] = m_run[j];
      mls[(hg * kAttnHeads + g + 8 * j) * 2 + 1] = l_run[j];
    }
  }
  cluster.sync();

  // Merge: weights exp2(m_c - M) per (CTA c, head), then columns of slice x.
  // Thread (head hh, CTA cc) reads that CTA's (m, l); eight lanes per head
  // reduce M and L with shuffles (C <= 8).
  int cl_bad;   // some CTA of the cluster stopped on a wait that ran out
  {
    const int hh = tid >> 3, cc = tid & 7;
    float m = -CUDART_INF_F, l = 0.f;
    int pb = 0;
    if (cc < C) {
      const float2 v = *reinterpret_cast<const float2*>(cluster.map_shared_rank(mls, cc) + hh * 2);
      m = v.x;
      l = v.y;
      pb = *cluster.map_shared_rank(&bad_s, cc);
    }
    cl_bad = __any_sync(0xffffffffu, pb);
    float M = l > 0.f ? m : -CUDART_INF_F;
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float w = l > 0.f ? exp2f(m - M) : 0.f;
    float L = w * l;
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    if (cc < C) wts[cc * NH + hh] = w;
    if (cc == 0) {
      invl[hh] = L > 0.f ? 1.f / L : 0.f;
      mlc[hh] = M;
      mlc[NH + hh] = L;
      if (a.Kc == 1 && a.lse && x == 0 && h0 + hh < a.H_q && !cl_bad)
        a.lse[(int64_t)r * a.H_q + h0 + hh] = L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -CUDART_INF_F;
    }
  }
  __syncthreads();
  const int cs = a.D_v / C;            // columns of this CTA's slice (even: D_v % 32 == 0, C <= 8)
  const int nq = NH * (cs / 4);   // column quads of this slice (cs % 4 == 0)
  const size_t pstride = 2 * NH + (size_t)NH * cs;
  const size_t slot0 = (((size_t)r * gridDim.y + blockIdx.y) * a.Kc) * C + x;   // (kc' = 0, slice x)
  float* mypart = a.Kc > 1 ? a.apart + (slot0 + (size_t)kc * C) * pstride : nullptr;
  // Two quads per thread per sweep, all 2 x C remote loads issued before the
  // (CTA-ordered) accumulation.
  for (int e0 = tid; e0 < nq; e0 += 2 * NTH) {
    float4 v[2][8];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int e = e0 + u * NTH;
      const int hh = e / (cs / 4), col = x * cs + 4 * (e % (cs / 4));
#pragma unroll
      for (int cc = 0; cc < 8; ++cc)
        if (cc < C && e < nq)
          v[u][cc] = *reinterpret_cast<const float4*>(cluster.map_shared_rank(Ob, cc) + hh * a.D_v + col);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int e = e0 + u * NTH;
      if (e >= nq) continue;
      const int hh = e / (cs / 4), col = x * cs + 4 * (e % (cs / 4));
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int cc = 0; cc < 8; ++cc)
        if (cc < C) {
          const float w = wts[cc * NH + hh];
          o.x += w * v[u][cc].x;
          o.y += w * v[u][cc].y;
          o.z += w * v[u][cc].z;
          o.w += w * v[u][cc].w;
        }
      if (a.Kc > 1) {
        *reinterpret_cast<float4*>(mypart + 2 * NH + hh * cs + (col - x * cs)) = o;
      } else if (h0 + hh < a.H_q && !cl_bad) {
        const float il = invl[hh];
        *reinterpret_cast<uint2*>(a.out + ((int64_t)r * a.H_q + h0 + hh) * a.D_v + col) =
            make_uint2(pack_bf16(o.x * il, o.y * il), pack_bf16(o.z * il, o.w * il));
      }
    }
  }
  if (a.Kc > 1 && tid < 2 * NH) mypart[tid] = mlc[tid];
  cluster.sync();   // peers may still be reading this CTA's shared memory
  if (a.Kc == 1) return;

  // Several clusters share (row, head group): the last to finish slice x merges
  // the Kc cluster partials of that slice, in cluster order.
  // Word 15 of the (row, head group)'s counters marks a cluster that stopped
  // on a wait that ran out; then no output is written for it.
  uint32_t* cnt = a.acnt + ((size_t)r * gridDim.y + blockIdx.y) * 16;
  if (tid == 0 && cl_bad) atomicOr(cnt + 15, 1u);
  __threadfence();
  __syncthreads();
  if (tid == 0) last_s = atomicAdd(cnt + x, 1u) == (uint32_t)(a.Kc - 1) && !(atomicOr(cnt + 15, 0u) & 1u);
  __syncthreads();
  if (!last_s) return;
  __threadfence();
  float* fw = mall;                    // [Kc][NH] weights of the cluster partials
  {
    const int hh = tid >> 3, q = tid & 7;   // Kc <= 8
    float m = -CUDART_INF_F, l = 0.f;
    if (q < a.Kc) {
      const float* pp = a.apart + (slot0 + (size_t)q * C) * pstride;
      m = __ldcg(pp + hh);
      l = __ldcg(pp + NH + hh);
    }
    float M = l > 0.f ? m : -CUDART_INF_F;
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float w = l > 0.f ? exp2f(m - M) : 0.f;
    float L = w * l;
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    if (q < a.Kc) fw[q * NH + hh] = w;
    if (q == 0) {
      invl[hh] = L > 0.f ? 1.f / L : 0.f;
      if (a.lse && x == 0 && h0 + hh < a.H_q)
        a.lse[(int64_t)r * a.H_q + h0 + hh] = L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -CUDART_INF_F;
    }
  }
  __syncthreads();
  for (int e = tid; e < nq; e += NTH) {
    const int hh = e / (cs / 4), cl = 4 * (e % (cs / 4));
    float4 v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (q < a.Kc)
        v[q] = __ldcg(reinterpret_cast<const float4*>(
            a.apart + (slot0 + (size_t)q * C) * pstride + 2 * NH + hh * cs + cl));
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (q < a.Kc) {
        const float w = fw[q * NH + hh];
        o.x += w * v[q].x;
        o.y += w * v[q].y;
        o.z += w * v[q].z;
        o.w += w * v[q].w;
      }
    if (h0 + hh < a.H_q) {
      const float il = invl[hh];
      *reinterpret_cast<uint2*>(a.out + ((int64_t)r * a.H_q + h0 + hh) * a.D_v + x * cs + cl) =
          make_uint2(pack_bf16(o.x * il, o.y * il), pack_bf16(o.z * il, o.w * il));
    }
  }
}

template <int NT, bool F8, int HG>
cudaError_t launch_cluster(const AttnArgs& a, dim3 grid, int C, size_t smem, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(attn_cluster_kernel<NT, F8, HG>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads * HG);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)C;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, attn_cluster_kernel<NT, F8, HG>, a);
}

// Shared memory of a CTA serving hg head groups (the kernel's layout).
size_t attn_smem(int hg, int qs, int ks, int D_k, int D_v, bool f8) {
  const size_t nh = (size_t)kAttnHeads * hg, nw = (size_t)kWarps * hg;
  const size_t qbytes = nh * qs * 2, kbytes = (size_t)kAttnRows * ks * 2;
  const size_t obytes = nh * D_v * 4;   // partial O after the tile loop, aliased (see the kernel)
  const size_t region = hg == 1 ? qbytes + (kbytes > obytes ? kbytes : obytes)
                                : (qbytes + kbytes > obytes ? qbytes + kbytes : obytes);
  size_t smem = region + nh * kPStride * 2 + 2 * nw * kAttnHeads * 4 + 2 * nh * 4 + 16 * nh * 8 +
                16 * nh * 4 + nh * 4 + 2 * nh * 4 + (size_t)kMaxTiles * kAttnRows * 4;
  if (f8) smem += (size_t)kMaxTiles * kAttnRows * 4 + (size_t)kAttnRows * D_k;   // scales, staging
  return smem;
}

}  // namespace

cudaError_t launch_attention(const dsa_problem& p, const Plan& pl, const int32_t* idx,
                             const int32_t* nsel, uint16_t* out, float* lse, char* ws,
                             cudaStream_t st, const TestHooks* hooks) {
  AttnArgs a;
  const TestHooks none;
  if (!hooks) hooks = &none;
  a.wait_ns = hooks->wait_ns;
  a.test_no_gather = hooks->attn_no_gather;
  const bool f8 = (p.flags & DSA_FLAG_KV_FP8) != 0;
  a.q = p.q; a.kv = p.kv; a.kv_scale = f8 ? p.kv_scale : nullptr;
  a.offsets = p.offsets; a.row_offsets = p.row_offsets;
  a.row_len = p.row_len; a.idx = idx; a.nsel = nsel;
  a.out = out; a.lse = lse;
  a.status = reinterpret_cast<uint32_t*>(ws + pl.off_status);
  a.apart = reinterpret_cast<float*>(ws + pl.off_apart);
  a.acnt = reinterpret_cast<uint32_t*>(ws + pl.off_acnt);
  a.B = p.B; a.H_q = p.H_q; a.D_k = p.D_k; a.D_v = p.D_v; a.k = p.k;
  a.L1 = (int)p.L_total;
  a.scale_log2 = p.softmax_scale * 1.4426950408889634f;

  int NT = 2;
  while (NT * 32 < p.D_v) NT *= 2;            // 2, 4, 8 or 16
  const int cols = NT * 32;
  a.qs = p.D_k + 8;
  a.ks = (p.D_k > cols ? p.D_k : cols) + 8;
  // Clusters of C CTAs, one 64-position tile per CTA; Kc clusters per (row,
  // head group) cover the k positions.  Clusters of 4 are placed one CTA per
  // SM (at least 116 KB of shared memory): two CTAs on an SM would share its
  // bandwidth for scattered rows (about 40 GB/s), and the gather is the
  // critical path.  Clusters of 8 so padded would not all fit in one wave.
  const int tiles = (p.k + kAttnRows - 1) / kAttnRows;
  const int C = attn_cluster_size(p.k);
  // Many rows: fewer clusters per (row, head group), each CTA looping over
  // several tiles (the workspace holds partials for this many, no more).
  const int hgroups = (p.H_q + kAttnHeads - 1) / kAttnHeads;
  const int64_t per_kc = (int64_t)p.R * hgroups * C;
  a.Kc = attn_clusters(p.R, hgroups, p.k);
  if ((tiles + C * a.Kc - 1) / (C * a.Kc) > kMaxTiles) return cudaErrorInvalidConfiguration;
  if (a.Kc > pl.attn_kc_max || a.Kc > 8) return cudaErrorInvalidConfiguration;   // the merge holds <= 8
  // So many rows that the grid of 16-head CTAs runs in many waves and one
  // cluster serves each (row, 64 heads): one CTA per (row, position split)
  // serves 4 head groups, so each selected row is gathered once instead of
  // once per head group.  bf16 cache, H_q a multiple of 64.
  const bool wide = !f8 && p.H_q % (4 * kAttnHeads) == 0 && a.Kc == 1 && per_kc > 600 &&
                    attn_clusters(p.R, p.H_q / (4 * kAttnHeads), p.k) == 1;
  if (wide) {
    const size_t smem = attn_smem(4, a.qs, a.ks, p.D_k, p.D_v, false);
    if (smem > 227u * 1024u) return cudaErrorInvalidConfiguration;
    const dim3 grid(C, p.H_q / (4 * kAttnHeads), p.R);
    switch (NT) {
      case 2: return launch_cluster<2, false, 4>(a, grid, C, smem, st);
      case 4: return launch_cluster<4, false, 4>(a, grid, C, smem, st);
      case 8: return launch_cluster<8, false, 4>(a, grid, C, smem, st);
      default: return launch_cluster<16, false, 4>(a, grid, C, smem, st);
    }
  }
  size_t smem = attn_smem(1, a.qs, a.ks, p.D_k, p.D_v, f8);
  // One CTA per SM while the grid fits in one wave.
  if (C <= 4 && per_kc * a.Kc <= 152 && smem < 116u * 1024u) smem = 116u * 1024u;
  // a.D_v / C must be even: D_v is a multiple of 32 and C <= 8.
  const dim3 grid(C * a.Kc, hgroups, p.R);
  if (f8) {
    switch (NT) {
      case 2: return launch_cluster<2, true, 1>(a, grid, C, smem, st);
      case 4: return launch_cluster<4, true, 1>(a, grid, C, smem, st);
      case 8: return launch_cluster<8, true, 1>(a, grid, C, smem, st);
      default: return launch_cluster<16, true, 1>(a, grid, C, smem, st);
    }
  }
  switch (NT) {
    case 2: return launch_cluster<2, false, 1>(a, grid, C, smem, st);
    case 4: return launch_cluster<4, false, 1>(a, grid, C, smem, st);
    case 8: return launch_cluster<8, false, 1>(a, grid, C, smem, st);
    default: return launch_cluster<16, false, 1>(a, grid, C, smem, st);
  }
}

}  // namespace dsa
