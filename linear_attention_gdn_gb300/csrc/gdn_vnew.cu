// gdn_vnew.cu -- V_new = U - W S of every (chunk, value head), recomputed from
// the saved states for the backward of the replay saved form.
//
// The replay form keeps only the state entering every chunk; the backward
// runs the UT / WY preparation again (prep_kernel: T', T'', Aqk, T and the
// scalars of every chunk) and this kernel forms, from the saved BF16 S^T,
//   W^T     = K^T T'^T,  U^T = V^T T''^T                 (tcgen05, TMEM)
//   V_new^T = U^T - S^T W^T
// exactly as the forward walk does (the same tiles, MMA shapes and BF16
// roundings, so the tiles equal the forward's bit for bit).  This is the
// pages' replay of w, u and v_new instead of saving them ("#8542" page, the
// save-set table and its full / replay forms).  There is no sequential
// dependency: one CTA per (chunk, q/k head) takes the group's value heads in
// turn on one K tile, two CTAs per SM.
#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_prof.h"

namespace gdn {

constexpr int VW_K = 0;                      // K tile, SwTile(64 x 128)
constexpr int VW_S = 16384;                  // S^T tile, SwTile(128 x 128)
constexpr int VW_V = VW_S + STATE_BYTES;     // V tile, SwTile(64 x 128)
constexpr int VW_T = VW_V + 16384;           // T' then T'' (contiguous, as in the UT block)
constexpr int VW_W = VW_T + 2 * TILE64_BYTES;   // -W^T tile, then the V_new^T staging tile, SwTile(128 x 64)
constexpr int VW_SMEM = VW_W + VN_BYTES;
constexpr int VW_SMEM_ALLOC = VW_SMEM + 1024;
static_assert(VW_S % 1024 == 0 && VW_V % 1024 == 0 && VW_T % 1024 == 0 && VW_W % 1024 == 0, "aligned tiles");
constexpr int VW_THREADS = 128;
constexpr uint32_t VW_HEAD_BYTES = STATE_BYTES + 16384 + 2 * TILE64_BYTES;   // S^T, V, T' T'' of one head
// TMEM columns: W^T, then U^T / V_new^T
constexpr int VT_W = 0, VT_U = 64;

__global__ void __launch_bounds__(VW_THREADS, 2) vnew_kernel(const __grid_constant__ VnewArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_align1024(smem_raw);
  __shared__ uint64_t bar_k, bar_ld, bar_mma;
  __shared__ uint32_t tslot;
  const int c = blockIdx.x / a.H, j = blockIdx.x % a.H;
  const int tid = threadIdx.x, warp = tid >> 5;
  if (*(volatile int*)a.err) return;
  const int tok0 = a.chunk_tok0[c], L = a.chunk_len[c];

  auto issue_head = [&](int hv) {   // S^T (saved tape), V (TMA), T' T'' (UT block) of one value head
    mbar_expect_tx(&bar_ld, VW_HEAD_BYTES);
    const size_t blk = (size_t)c * a.HV + hv;
    bulk_load(sm + VW_S, a.tape + blk * STATE_BYTES, STATE_BYTES, &bar_ld);
    tma_load_3d(sm + VW_V, &a.tv, 0, hv, tok0, &bar_ld);
    tma_load_3d(sm + VW_V + 8192, &a.tv, 64, hv, tok0, &bar_ld);
    bulk_load(sm + VW_T, a.cb + blk * CB_BYTES + CB_TP, 2 * TILE64_BYTES, &bar_ld);
  };
  if (warp == 0) tmem_alloc(&tslot, 128);
  if (tid == 0) {
    mbar_init(&bar_k, 1);
    mbar_init(&bar_ld, 1);
    mbar_init(&bar_mma, 1);
    asm volatile("fence.mbarrier_init.release.cluster;");
    mbar_expect_tx(&bar_k, 16384u);
    tma_load_3d(sm + VW_K, &a.tk, 0, j, tok0, &bar_k);
    tma_load_3d(sm + VW_K + 8192, &a.tk, 64, j, tok0, &bar_k);
  }
  // Thread 0 issues every tile request and (in warp 0) every MMA; for the error path it keeps the
  // phase of a request or a commit whose completion has not been seen yet (-1: none).
  int ld_par = -1, mma_par = -1;
  if (tid == 0 && !(a.withhold_first_load && blockIdx.x == 0)) {
    issue_head(j * a.G);
    ld_par = 0;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tslot;
  bool ok = __syncthreads_and(mbar_wait(&bar_k, 0, a.err));
  if (ok && L < CH) {   // zero the K rows past the document end (they hold the next document)
    for (int idx = tid; idx < (CH - L) * 16; idx += VW_THREADS)
      *reinterpret_cast<uint4*>(sm + VW_K + sw_chunk(L + (idx >> 4), idx & 15, 64)) = make_uint4(0u, 0u, 0u, 0u);
  }
  uint32_t mph = 0;
  const uint32_t s_k = smem_u32(sm + VW_K), s_s = smem_u32(sm + VW_S), s_v = smem_u32(sm + VW_V),
                 s_tp = smem_u32(sm + VW_T), s_tpp = smem_u32(sm + VW_T + TILE64_BYTES), s_w = smem_u32(sm + VW_W);
  for (int hh = 0; hh < a.G && ok; ++hh) {
    const int hv = j * a.G + hh;
    ok = __syncthreads_and(mbar_wait(&bar_ld, hh & 1, a.err));
    if (!ok) break;
    ld_par = -1;
    if (L < CH) {   // zero the V rows past the document end
      for (int idx = tid; idx < (CH - L) * 16; idx += VW_THREADS)
        *reinterpret_cast<uint4*>(sm + VW_V + sw_chunk(L + (idx >> 4), idx & 15, 64)) = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) {   // W^T = K^T T'^T, U^T = V^T T''^T
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_ss_w(tb + VT_W, desc_mn(s_k, 64, ks), desc_k(s_tp, 64, ks), idesc(128, 64, 1, 0), ks > 0);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_ss_w(tb + VT_U, desc_mn(s_v, 64, ks), desc_k(s_tpp, 64, ks), idesc(128, 64, 1, 0), ks > 0);
      mma_commit_w(&bar_mma);
      mma_par = (int)mph;
    }
    if (tid == 0) bulk_wait_read();   // the previous head's V_new^T store has read the staging tile
    ok = __syncthreads_and(mbar_wait(&bar_mma, mph, a.err));
    mph ^= 1;
    if (!ok) break;
    mma_par = -1;
    tc_fence_after();
    {  // -W^T -> shared (row tid = dk index), the MN-major B operand of the V_new MMA
      float w[64];
      tmem_ld32(taddr(tb, warp * 32, VT_W), w);
      tmem_ld32(taddr(tb, warp * 32, VT_W + 32), w + 32);
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {
        uint4 v;
        v.x = pack_bf16(-w[c8 * 8 + 0], -w[c8 * 8 + 1]);
        v.y = pack_bf16(-w[c8 * 8 + 2], -w[c8 * 8 + 3]);
        v.z = pack_bf16(-w[c8 * 8 + 4], -w[c8 * 8 + 5]);
        v.w = pack_bf16(-w[c8 * 8 + 6], -w[c8 * 8 + 7]);
        *reinterpret_cast<uint4*>(sm + VW_W + sw_chunk(tid, c8, 128)) = v;
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) {   // V_new^T = U^T - S^T W^T
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_ss_w(tb + VT_U, desc_k(s_s, 128, ks), desc_mn(s_w, 128, ks), idesc(128, 64, 0, 1), 1u);
      mma_commit_w(&bar_mma);
      mma_par = (int)mph;
    }
    ok = __syncthreads_and(mbar_wait(&bar_mma, mph, a.err));
    mph ^= 1;
    if (!ok) break;
    mma_par = -1;
    tc_fence_after();
    if (tid == 0 && hh + 1 < a.G) {   // S^T, V, T' T'' of this head are dead
      issue_head(hv + 1);
      ld_par = (hh + 1) & 1;
    }
    {  // V_new^T row tid -> BF16 staging tile (over -W^T, which the finished MMA no longer reads)
      float x[64];
      tmem_ld32(taddr(tb, warp * 32, VT_U), x);
      tmem_ld32(taddr(tb, warp * 32, VT_U + 32), x + 32);
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {
        uint4 v;
        v.x = pack_bf16(x[c8 * 8 + 0], x[c8 * 8 + 1]);
        v.y = pack_bf16(x[c8 * 8 + 2], x[c8 * 8 + 3]);
        v.z = pack_bf16(x[c8 * 8 + 4], x[c8 * 8 + 5]);
        v.w = pack_bf16(x[c8 * 8 + 6], x[c8 * 8 + 7]);
        *reinterpret_cast<uint4*>(sm + VW_W + sw_chunk(tid, c8, 128)) = v;
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      bulk_store(a.vn + ((size_t)c * a.HV + hv) * VN_BYTES, sm + VW_W, VN_BYTES);
      bulk_commit();
    }
  }
  if (tid == 0) bulk_wait_all();
  if (!ok && tid == 0) {   // error path (bounded waits): no copy or MMA may outlive the CTA's memory
    if (mma_par >= 0) mbar_drain(&bar_mma, (uint32_t)mma_par);
    if (ld_par >= 0) mbar_drain(&bar_ld, (uint32_t)ld_par);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, 128);
}

void setup_vnew_attrs() {
  cudaFuncSetAttribute(vnew_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, VW_SMEM_ALLOC);
}
void launch_vnew(const VnewArgs& a, int NC, cudaStream_t s) {
  if (NC <= 0) return;
  prof_begin(K_VNEW, s);
  vnew_kernel<<<NC * a.H, VW_THREADS, VW_SMEM_ALLOC, s>>>(a);
  prof_end(K_VNEW, s);
}

}  // namespace gdn
