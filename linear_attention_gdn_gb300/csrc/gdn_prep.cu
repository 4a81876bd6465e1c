// gdn_prep.cu -- the UT / WY preparation of every (chunk, value head) as one
// chunk-parallel kernel: rk, rq, the chunk-local cumulative gate, KK^T / QK^T
// (tcgen05), A, T = (I + A)^-1, T' = T diag(beta gamma rk), T'' = T diag(beta),
// Aqk and the per-token scalars (gdn_ut.cuh states the algebra), written as one
// 33 KiB block per chunk and value head for the walks and the gradient kernel
// (the WY / intra / GLM-prep programs of the pages: "feat(cake_gdn_kcp) ...
// #8172" page, commit notes on those programs; "#8542" page, save-set table).
// The forward runs it before the state walk; the backward of the replay saved
// form runs it again instead of reading the blocks from the saved set.  The
// inverse's block diagonals run on the tensor cores (see prep_kernel).
#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_prof.h"
#include "gdn_ut.cuh"

namespace gdn {

constexpr int PR_THREADS = 128;
constexpr int PR_BLOCKS_PER_SM = 4;
// Shared memory (bytes, 1024-aligned tiles).  The [K; Q] tile is dead once the
// item's KK^T / QK^T MMA has completed; its space then holds, for each value
// head in turn, the FP32 A^T array, then the BF16 tiles of the inverse (D, the
// inverted diagonal blocks; L^T, then X), and finally the T', T'' and T output
// tiles.  Aqk and the scalars sit past it.
constexpr int PR_KQ = 0;                             // [K; Q] SwTile(128 x 128), 32 KB
constexpr int PR_S = 0;                              // FP32 S[64][UT_ALD]
constexpr int PR_D = 0;                              // D (inverted diagonal blocks), SwTile(64 x 64)
constexpr int PR_LX = TILE64_BYTES;                  // L^T, then X = I - N
constexpr int PR_TP = 0;                             // T', then T'' (contiguous, one bulk store)
constexpr int PR_T = 2 * TILE64_BYTES;               // T tile
constexpr int PR_AQ = 32768;                         // Aqk tile
constexpr int PR_SC = PR_AQ + TILE64_BYTES;          // scalars
constexpr int PR_SMEM = PR_SC + CB_SCAL_BYTES;
constexpr int PR_SMEM_ALLOC = PR_SMEM + 1024;
static_assert(UT_WORK_BYTES <= PR_AQ && 3 * TILE64_BYTES <= PR_AQ, "the FP32 array and the tiles lie below Aqk");
static_assert(PR_AQ % 1024 == 0 && PR_T % 1024 == 0, "swizzled tiles are 1024-aligned");
static_assert(CB_SCAL_BYTES == UT_SCAL_BYTES, "one scalar block layout");
// TMEM columns: the item's [KK^T; QK^T] (read by every value head), then the inverse's products
constexpr int PT_KK = 0, PT_INV = 64, PT_COLS = 128;

// One CTA per (chunk, q/k head): the tile load, the norms and the KK^T / QK^T
// MMA once, then the group's value heads one after another on that product
// (each head's stores drain while the next one is prepared).  Four CTAs share
// an SM, so the serial phases of one run under the others.  The UT arithmetic
// is gdn_ut.cuh's, except for the inverse's block diagonals, which run on the
// tensor cores: with D the inverted 32 x 32 diagonal blocks (FP32 forward
// substitution) and L the strictly block-lower part of A,
//   I + A = D^-1 (I + N),  N = D L,  N^2 = 0   =>   T = (I - N) D,
// two dependent M = 64 tcgen05 products (BF16 operands, FP32 accumulation).
__global__ void __launch_bounds__(PR_THREADS, PR_BLOCKS_PER_SM) prep_kernel(const __grid_constant__ PrepArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_align1024(smem_raw);
  __shared__ UtTok ut;
  __shared__ uint64_t bar, bar_kq, bar_t;
  __shared__ uint32_t tslot;
  const int c = blockIdx.x / a.H, j = blockIdx.x % a.H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (*(volatile int*)a.err) return;
  const int tok0 = a.chunk_tok0[c], L = a.chunk_len[c];

  // ---- [K; Q] tile by TMA: rows 0..63 = k tokens, 64..127 = q tokens (SwTile(128 x 128))
  if (warp == 0) tmem_alloc(&tslot, PT_COLS);
  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_init(&bar_kq, 1);
    mbar_init(&bar_t, 1);
    asm volatile("fence.mbarrier_init.release.cluster;");
    mbar_expect_tx(&bar_kq, 32768u);
    tma_load_3d(sm + PR_KQ, &a.tk, 0, j, tok0, &bar_kq);
    tma_load_3d(sm + PR_KQ + 8192, &a.tq, 0, j, tok0, &bar_kq);
    tma_load_3d(sm + PR_KQ + 16384, &a.tk, 64, j, tok0, &bar_kq);
    tma_load_3d(sm + PR_KQ + 24576, &a.tq, 64, j, tok0, &bar_kq);
  }
  // the gates of a value head (warp 3); the first head's are requested while the tile lands, each
  // later head's while the one before it is prepared
  float gb[4] = {0.f, 0.f, 0.f, 0.f};
  if (warp == 3) ut_load_gates(a.g, a.beta, a.HV, j * a.G, tok0, L, lane, gb);
  __syncthreads();
  if (!__syncthreads_and(mbar_wait(&bar_kq, 0, a.err))) {   // error path: the tile copy must land first
    if (tid == 0) mbar_drain(&bar_kq, 0);
    __syncthreads();
    if (warp == 0) tmem_dealloc(tslot, PT_COLS);
    return;
  }
  if (L < CH) {   // zero the rows past the document end (they hold the next document)
    ut_zero_tail(sm + PR_KQ, L, tid);
    __syncthreads();
  }
  ut_norm_row(sm + PR_KQ, tid, a.l2norm, ut);
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tslot;
  if (warp == 0) {
    ut_issue_kkqk(tb + PT_KK, smem_u32(sm + PR_KQ));
    mma_commit_w(&bar);
  }
  // ---- the value heads of the group, one after another, on the one KK^T / QK^T
  bool ok = true;
  uint32_t tph = 0;   // phase of bar_t (two products per value head)
  int t_pend = -1;    // error path: phase of a product whose completion was not seen (-1: none)
  float* Sm = reinterpret_cast<float*>(sm + PR_S);
  const UtInvTiles tiles{sm + PR_D, sm + PR_LX};
  const int r0 = 16 * warp + (lane >> 2), cq = 2 * (lane & 3);   // this thread's elements of T (see ut_ld_result)
  for (int hh = 0; hh < a.G; ++hh) {
    const int hv = j * a.G + hh;
    if (warp == 3) {   // ---- gates (log2 units), then the next head's loads
      const float gcur[4] = {gb[0], gb[1], gb[2], gb[3]};
      if (hh + 1 < a.G) ut_load_gates(a.g, a.beta, a.HV, hv + 1, tok0, L, lane, gb);
      ut_gates(gcur, lane, ut);
    }
    // (the first head waits for the KK^T / QK^T MMA, every later one for the previous head's copies
    // to have read the staging buffers it rewrites)
    if (hh > 0 && tid == 0) bulk_wait_read();
    ok = __syncthreads_and((hh > 0 || mbar_wait(&bar, 0, a.err)) && ok);
    tc_fence_after();
    float* sc = reinterpret_cast<float*>(sm + PR_SC);
    if (ok) {
      // ---- A^T (FP32, from the rows of KK^T), Aqk tile (rows of QK^T), scalars; the diagonal blocks
      ut_build(tb + PT_KK, warp, 0, tid, L, a.scale, ut, Sm, sm + PR_AQ, sc);
      if (tid < 64) ut_diag_blocks(Sm, tid, 1);
    }
    __syncthreads();
    if (!ok) continue;
    ok = ut_tc_inverse<PR_THREADS>(Sm, tiles, tb, PT_INV, &bar_t, tph, a.err, t_pend);
    uint32_t u[4][8];
    if (ok) {  // T', T'', T tiles (over D, X, N: the last product has read them)
      ut_ld_result<PR_THREADS>(tb, PT_INV, warp, u);
#pragma unroll
      for (int g = 0; g < 4; ++g)
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
          const int r = r0 + 8 * ((i >> 1) & 1), cc = 16 * g + 8 * (i >> 2) + cq;
          const uint32_t off = sw_off(r, cc, 64);
          const float t0 = __uint_as_float(u[g][i]), t1 = __uint_as_float(u[g][i + 1]);
          *reinterpret_cast<uint32_t*>(sm + PR_TP + off) = pack_bf16(t0 * ut.pcol[cc], t1 * ut.pcol[cc + 1]);
          *reinterpret_cast<uint32_t*>(sm + PR_TP + TILE64_BYTES + off) = pack_bf16(t0 * ut.bs[cc], t1 * ut.bs[cc + 1]);
          if (a.write_T) *reinterpret_cast<uint32_t*>(sm + PR_T + off) = pack_bf16(t0, t1);
        }
      fence_async_smem();
    }
    __syncthreads();
    if (ok && tid == 0) {   // ship the staged blocks: T' T'' (contiguous), Aqk, T, scalars
      uint8_t* cbp = a.cb + ((size_t)c * a.HV + hv) * CB_BYTES;
      bulk_store(cbp + CB_TP, sm + PR_TP, 2 * TILE64_BYTES);
      bulk_store(cbp + CB_AQK, sm + PR_AQ, TILE64_BYTES);
      if (a.write_T) bulk_store(cbp + CB_T, sm + PR_T, TILE64_BYTES);
      bulk_store(cbp + CB_SCAL, sm + PR_SC, CB_SCAL_BYTES);
      bulk_commit();
    }
  }
  if (tid == 0) bulk_wait_read();   // shared memory must outlive the copies' reads
  if (!ok && tid == 0) {   // error path (bounded waits): no MMA may outlive the CTA's TMEM
    mbar_drain(&bar, 0);
    if (t_pend >= 0) mbar_drain(&bar_t, (uint32_t)t_pend);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, PT_COLS);
}

void setup_prep_attrs() {
  cudaFuncSetAttribute(prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, PR_SMEM_ALLOC);
}
void launch_prep(const PrepArgs& a, int NC, cudaStream_t s) {
  if (NC <= 0) return;
  prof_begin(K_PREP, s);
  prep_kernel<<<NC * a.H, PR_THREADS, PR_SMEM_ALLOC, s>>>(a);
  prof_end(K_PREP, s);
}

}  // namespace gdn
