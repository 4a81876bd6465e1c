// gdn_fwd_scan.cu -- the inter-chunk state scan with the chunk output fused.
//
// One CTA walks one chain (a document segment and one value head) chunk by
// chunk; the 128 threads own the 128 rows of S^T (row i = value column i of
// the state, kept in FP32 registers), and a BF16 copy of S^T sits in shared
// memory as a tcgen05 operand.  Per chunk, with K, Q, V the raw BF16 tiles
// (TMA, double-buffered) and T', T'', Aqk, scalars from the prep kernel:
//   W^T      = K^T T'^T                         (tcgen05, TMEM)
//   V_new^T  = V^T T''^T - S^T W^T              (= (U - W S)^T)
//   S^T     <- gamma_L S^T + (V_new^T diag(kd)) K,  kd_r = e^{G_L - G_r} rk_r
//   O^T      = diag-scaled (S^T Q^T) + V_new^T Aqk^T
// and the BF16 state entering each chunk is stored to the saved tape.  These
// are the K1 walk's state updates with the output formed from the walk's own
// tapes (the pages fuse the output into the state recurrence:
// "feat(cake_gdn_kcp) ... #8172" page, commit note on the backend's local
// programs becoming fused state recurrences).
//
// Walk modes for the intra-GPU segment split ("#8542" page: segment transfers
// M_seg and the merges that read them):
//   full (walk = 0)  every segment but a split document's first, from its true
//                    start state (after the merge); writes o, tape
//   B    (walk = 1)  segment from a zero state; writes its end state B_p^T.  The
//                    first segment of a split document starts from its true
//                    start (zero, or the document's S_in), so its B walk is its
//                    full walk: it also writes o and the tape
//   M    (walk = 2)  the segment after a split point, with U = 0 from S^T = I;
//                    its end state is M^T, the transfer of that segment
//                    (S_end = M S_start + B)
#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_prof.h"

namespace gdn {

constexpr int SC_K = 0, SC_Q = 16384, SC_V = 32768, SC_TP = 49152, SC_TPP = 57344, SC_AQK = 65536,
              SC_SCAL = 73728;
constexpr int SC_STAGE = 74752;
constexpr int SC_S = 2 * SC_STAGE;          // BF16 S^T tile, SwTile(128 x 128)
constexpr int SC_W = SC_S + STATE_BYTES;    // -W^T tile, SwTile(128 x 64)
constexpr int SC_O = SC_W + 16384;          // BF16 output staging tile [64 tok][128], SwTile(64 x 128)
constexpr int SC_SMEM = SC_O + 16384;
constexpr int SC_SMEM_ALLOC = SC_SMEM + 1024;
constexpr int SC_WORK = 256;                 // the chain and the helper warpgroup
constexpr int SC_THREADS = SC_WORK + 128;    // plus one warpgroup whose first warp issues the chain's MMAs
// registers per thread after the split (the launch gives 65536 / 384 = 168): the MMA warpgroup gives
// all but 24 back, the chain and the helper take them
constexpr int SC_REG_WORK = 240, SC_REG_MMA = 24;
static_assert(SC_WORK * SC_REG_WORK + 128 * SC_REG_MMA <= SC_THREADS * 168, "register split");

// TMEM columns: D1 (U^T, then V_new^T) and O double-buffered over consecutive chunks
constexpr int TM_D1 = 0, TM_DW = 128, TM_DS = 192, TM_O = 320, TM_AVS = 448, TM_AVN = 480;

__device__ __forceinline__ void store_state_row(uint8_t* dst, int row, const float* S) {
#pragma unroll
  for (int c8 = 0; c8 < 16; ++c8) {
    uint4 w;
    w.x = pack_bf16(S[c8 * 8 + 0], S[c8 * 8 + 1]);
    w.y = pack_bf16(S[c8 * 8 + 2], S[c8 * 8 + 3]);
    w.z = pack_bf16(S[c8 * 8 + 4], S[c8 * 8 + 5]);
    w.w = pack_bf16(S[c8 * 8 + 6], S[c8 * 8 + 7]);
    *reinterpret_cast<uint4*>(dst + sw_chunk(row, c8, 128)) = w;
  }
}

// Three warpgroups.  The chain warpgroup (warps 0-3) owns the state and runs
// the dependent chain of each chunk:
//   MMA1 (V_new^T = U^T - S^T W^T) -> V_new hop -> MMA2 (dS^T = (V_new^T
//   diag(kd)) K, and the output O^T = S^T Q'^T + V_new^T Aqk^T with
//   Q'_r = gamma_r rq_r q_r, so that o = scale O) -> S hop,
// and, while MMA1 of chunk n runs, writes the output of chunk n - 1 from its
// O buffer.  The helper warpgroup (warps 4-7) prepares chunk n + 1 while the
// chain works on chunk n (tile landing, W^T = K^T T'^T and U^T = V^T T''^T,
// the -W^T tile, Q') and streams the tiles in.  The first warp of the third
// warpgroup issues the chain's MMAs (MMA1; MMA2 then the output), so that no
// chain warp is held by the issue; the rest of that warpgroup exits.  They
// hand off through mbarriers:
//   go1       chain -> MMA warp S^T(n) is in its tile
//   go2       chain -> MMA warp the V_new^T(n) A operands are in TMEM
//   bar_wr    helper -> chain   -W^T(n), U^T(n), Q'(n) are ready
//   bar_m1    MMA1(n) done      (chain: V_new; helper: -W^T tile and D1 reuse)
//   bar_m2    MMA2(n) done      (chain: S)
//   bar_o[b]  MMA2(n) done      (chain: output(n) from O buffer b = n & 1)
//   bar_sf    chain -> helper   chunk n's stage is no longer read (V_new^T copy)
// Each completes once per use, and no waiter can fall two phases behind.
//
// KDA = true: the per-channel-decay form (one decay per key channel).  The
// stage then holds the chunk's -W^T and Kd (from kda_prep_kernel) in the K and
// Q slots, V, T'' and gamma_L; MMA1 reads -W^T from the stage (the helper only
// forms U^T), MMA2 is dS^T = V_new^T Kd, the state update scales column i of
// S^T by gamma_L[i], and the output is left to kda_out_kernel.
template <bool KDA>
__global__ void __launch_bounds__(SC_THREADS, 1) fwd_scan_kernel(const __grid_constant__ ScanArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_align1024(smem_raw);
  // go1: S^T of the chunk is in its tile (MMA1 may read it); go2: the V_new^T A operands are in TMEM
  // (MMA2 and the output MMAs may go); done: every MMA of the MMA warp has completed
  __shared__ uint64_t full_bar[2], bar_wr, bar_m1, bar_wu, bar_m2, bar_o[2], bar_sf, go1, go2, done;
  __shared__ uint32_t tslot;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int lt = tid & 127;      // row within the warpgroup = TMEM lane
  const int wq = warp & 3;       // the warp's TMEM lane quarter
  const bool chain = tid < 128;
  if (*(volatile int*)a.err) return;

  int mode, seg, hv, split = -1;
  bool write_bend = false;
  if (!a.walk) {
    mode = 0;
    seg = a.walk_seg[blockIdx.x / a.HV];
    hv = blockIdx.x % a.HV;
  } else {
    const int half = a.nsplit * a.HV;
    mode = blockIdx.x < half ? 1 : 2;
    const int bb = blockIdx.x % half;
    split = bb / a.HV;
    hv = bb % a.HV;
    // B walks run on split segment p, M walks on segment p + 1: the merges
    // use M_1 .. M_{P-1} (M_0 only ever multiplies the zero start state)
    seg = a.split_seg[split] + (mode == 2 ? 1 : 0);
    if (mode == 1 && a.seg_idx[seg] == 0) {   // a document's first segment: the full walk, plus B
      mode = 0;
      write_bend = true;
    }
  }
  const int kh = hv / a.G;
  const int c0 = a.seg_c0[seg], nch = a.seg_c1[seg] - c0;
  const bool with_o = !KDA && mode == 0 && a.o != nullptr;
  const bool with_u = mode != 2;
  const bool with_vn = mode == 0 && a.vn != nullptr;   // V_new^T tiles for the backward
  const uint32_t tx_bytes = KDA ? (with_u ? 58368u : 33792u)
                                : (mode == 0 ? (with_o ? 74752u : 50176u) : (mode == 1 ? 50176u : 25600u));
  const uint32_t cb_bytes = mode == 2 ? 8192u : (with_o ? 24576u : 16384u);
  uint8_t* s_tile = sm + SC_S;

  const int doc = a.seg_doc[seg];

  if (warp == 0) tmem_alloc(&tslot, 512);
  if (tid == 0) {
    mbar_init(&full_bar[0], 1);
    mbar_init(&full_bar[1], 1);
    mbar_init(&bar_wr, 1);
    mbar_init(&bar_m1, 1);
    mbar_init(&bar_wu, 1);
    mbar_init(&bar_m2, 1);
    mbar_init(&bar_o[0], 1);
    mbar_init(&bar_o[1], 1);
    mbar_init(&bar_sf, 1);
    mbar_init(&go1, 1);
    mbar_init(&go2, 1);
    mbar_init(&done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;");
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tslot;

  auto issue = [&](int n, int t0) {   // the tiles of chunk n (first token t0) into stage n & 1
    const int ci = c0 + n;
    uint8_t* st = sm + (n & 1) * SC_STAGE;
    uint64_t* bar = &full_bar[n & 1];
    mbar_expect_tx(bar, tx_bytes);
    if (KDA) {   // -W^T and Kd (contiguous in the block and in the stage), V, T'', gamma_L
      const uint8_t* kbp = a.cb + ((size_t)ci * a.HV + hv) * KB_BYTES;
      bulk_load(st + SC_K, kbp + KB_WT, 32768u, bar);
      if (with_u) {
        tma_load_3d(st + SC_V, &a.tv, 0, hv, t0, bar);
        tma_load_3d(st + SC_V + 8192, &a.tv, 64, hv, t0, bar);
        bulk_load(st + SC_TPP, kbp + KB_TPP, TILE64_BYTES, bar);
      }
      bulk_load(st + SC_SCAL, kbp + KB_SCAL, CB_SCAL_BYTES, bar);
      return;
    }
    const uint8_t* cbp = a.cb + ((size_t)ci * a.HV + hv) * CB_BYTES;
    tma_load_3d(st + SC_K, &a.tk, 0, kh, t0, bar);
    tma_load_3d(st + SC_K + 8192, &a.tk, 64, kh, t0, bar);
    if (with_o) {
      tma_load_3d(st + SC_Q, &a.tq, 0, kh, t0, bar);
      tma_load_3d(st + SC_Q + 8192, &a.tq, 64, kh, t0, bar);
    }
    if (with_u) {
      tma_load_3d(st + SC_V, &a.tv, 0, hv, t0, bar);
      tma_load_3d(st + SC_V + 8192, &a.tv, 64, hv, t0, bar);
    }
    bulk_load(st + SC_TP, cbp + CB_TP, cb_bytes, bar);
    bulk_load(st + SC_SCAL, cbp + CB_SCAL, CB_SCAL_BYTES, bar);
  };
  auto prefetch = [&](int n) {   // the tiles of chunk n into L2, a stage ahead of their request
    const int ci = c0 + n, t0 = a.chunk_tok0[ci];
    if (KDA) {
      const uint8_t* kbp = a.cb + ((size_t)ci * a.HV + hv) * KB_BYTES;
      bulk_prefetch(kbp + KB_WT, 32768u);
      if (with_u) {
        tma_prefetch_3d(&a.tv, 0, hv, t0);
        tma_prefetch_3d(&a.tv, 64, hv, t0);
        bulk_prefetch(kbp + KB_TPP, TILE64_BYTES);
      }
      bulk_prefetch(kbp + KB_SCAL, CB_SCAL_BYTES);
      return;
    }
    const uint8_t* cbp = a.cb + ((size_t)ci * a.HV + hv) * CB_BYTES;
    tma_prefetch_3d(&a.tk, 0, kh, t0);
    tma_prefetch_3d(&a.tk, 64, kh, t0);
    if (with_o) {
      tma_prefetch_3d(&a.tq, 0, kh, t0);
      tma_prefetch_3d(&a.tq, 64, kh, t0);
    }
    if (with_u) {
      tma_prefetch_3d(&a.tv, 0, hv, t0);
      tma_prefetch_3d(&a.tv, 64, hv, t0);
    }
    bulk_prefetch(cbp + CB_TP, cb_bytes);
    bulk_prefetch(cbp + CB_SCAL, CB_SCAL_BYTES);
  };
  if (tid == 128) {
    if (nch > 0) issue(0, a.chunk_tok0[c0]);
    if (nch > 1) issue(1, a.chunk_tok0[c0 + 1]);
    if (nch > 2) prefetch(2);
  }
  bool ok = true;
  const uint32_t sm_s = smem_u32(s_tile), sm_w = smem_u32(sm + SC_W);

  if (tid >= SC_WORK) {
    // =================== MMA warpgroup: its first warp issues MMA1, MMA2 and the output MMAs ======
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(SC_REG_MMA));
    if (warp == SC_WORK / 32) {
      bool live = true;
      for (int n = 0; n < nch && live; ++n) {
        const uint8_t* st = sm + (n & 1) * SC_STAGE;
        // MMA1: V_new^T = U^T - S^T W^T (into D1[n & 1]), once S^T, -W^T, U^T and the tiles are in
        live = mbar_wait(&go1, n & 1, a.err) && mbar_wait(&bar_wr, n & 1, a.err) &&
               mbar_wait(&full_bar[n & 1], (n >> 1) & 1, a.err);
        if (!live) break;
        tc_fence_after();
        const uint32_t d1 = tb + TM_D1 + (n & 1) * 64;
        const uint32_t b_w = KDA ? smem_u32(st + SC_K) : sm_w;   // -W^T: the stage's (KDA) or the helper's
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_ss_w(d1, desc_k(sm_s, 128, ks), desc_mn(b_w, 128, ks), idesc(128, 64, 0, 1),
                   (with_u || ks > 0) ? 1u : 0u);
        mma_commit_w(&bar_m1);
        // MMA2: dS^T = (V_new^T diag(kd)) K; then O^T = S^T Q'^T + V_new^T Aqk^T (into O[n & 1])
        if (!(live = mbar_wait(&go2, n & 1, a.err))) break;
        tc_fence_after();
        const uint32_t a_k = smem_u32(st + (KDA ? SC_Q : SC_K));   // K (scaled by kd in the A operand), or Kd
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_ts_w(tb + TM_DS, tb + TM_AVS + ks * 8, desc_mn(a_k, 64, ks), idesc(128, 128, 0, 1), ks > 0);
        mma_commit_w(&bar_m2);
        if (with_o) {   // (the O buffer n & 1 was read out by output(n - 2) in the chain's previous step)
          const uint32_t to = tb + TM_O + (n & 1) * 64;
          const uint32_t a_q = smem_u32(st + SC_Q), a_aqk = smem_u32(st + SC_AQK);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            mma_ss_w(to, desc_k(sm_s, 128, ks), desc_k(a_q, 64, ks), idesc(128, 64, 0, 0), ks > 0);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_ts_w(to, tb + TM_AVN + ks * 8, desc_k(a_aqk, 64, ks), idesc(128, 64, 0, 0), 1u);
          mma_commit_w(&bar_o[n & 1]);
        }
      }
      mma_commit_w(&done);   // arrives once every MMA this warp issued has completed
    }
    return;
  }
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(SC_REG_WORK));

  if (chain) {
    // =================== chain warpgroup ===================
    // ---- initial state (row lt of S^T): the merged start of a later segment, the document's S_in
    // for its first segment (full and B walks), else zero (the identity for M walks)
    float S[128];
    {
      const float* src = nullptr;
      int stride = 1;
      if (mode == 0 && a.seg_idx[seg] > 0) {
        src = a.s_init + ((size_t)a.seg_split[seg - 1] * a.HV + hv) * STATE_F32 + (size_t)lt * 128;
      } else if (mode != 2 && a.seg_idx[seg] == 0 && a.s_in) {   // column lt of S_in [dk][dv]
        src = a.s_in + ((size_t)doc * a.HV + hv) * STATE_F32 + lt;
        stride = 128;
      }
#pragma unroll
      for (int jj = 0; jj < 128; ++jj) S[jj] = src ? src[jj * stride] : (mode == 2 && jj == lt ? 1.f : 0.f);
      store_state_row(s_tile, lt, S);
      if (mode == 0 && a.tape) store_state_row(a.tape + ((size_t)c0 * a.HV + hv) * STATE_BYTES, lt, S);
    }
    fence_async_smem();
    named_bar(1, 128);
    if (tid == 0 && nch > 0) mbar_arrive(&go1);   // S^T of the first chunk is in its tile
    uint8_t* o_stage = sm + SC_O;
    // the output of chunk m from its O buffer (TMEM), o = scale O; thread 32 owns the staging tile's copies
    auto output = [&](int m) {
      const int L = a.chunk_len[c0 + m];
      if (tid == 32) bulk_wait_read();   // the previous output store has read the staging tile
      named_bar(1, 128);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float x[32];
        tmem_ld32(taddr(tb, wq * 32, TM_O + (m & 1) * 64 + h * 32), x);
#pragma unroll
        for (int e = 0; e < 32; ++e)
          *reinterpret_cast<__nv_bfloat16*>(o_stage + sw_off(h * 32 + e, lt, 64)) = __float2bfloat16_rn(a.scale * x[e]);
      }
      fence_async_smem();
      tc_fence_before();
      named_bar(1, 128);
      const int t0 = a.chunk_tok0[c0 + m];
      if (L < CH) {  // ragged last chunk: only its own rows (the next rows are another document's)
        for (int idx = lt; idx < L * 16; idx += 128) {
          const int r = idx >> 4, c8 = idx & 15;
          *reinterpret_cast<uint4*>(a.o + ((size_t)(t0 + r) * a.HV + hv) * D + c8 * 8) =
              *reinterpret_cast<const uint4*>(o_stage + sw_chunk(r, c8, 64));
        }
      } else if (tid == 32) {
        tma_store_3d(&a.to, o_stage, 0, hv, t0);
        tma_store_3d(&a.to, o_stage + 8192, 64, hv, t0);
        bulk_commit();
      }
    };
    for (int n = 0; n < nch && ok; ++n) {
      const uint32_t par = n & 1;
      uint8_t* st = sm + (n & 1) * SC_STAGE;
      const uint32_t a_k = smem_u32(st + SC_K), a_q = smem_u32(st + SC_Q), a_aqk = smem_u32(st + SC_AQK);
      const float* scal = reinterpret_cast<const float*>(st + SC_SCAL);
      const uint32_t d1 = tb + TM_D1 + (n & 1) * 64;
      ok = wg_sync_and(1, mbar_wait(&bar_wr, par, a.err) && mbar_wait(&full_bar[n & 1], (n >> 1) & 1, a.err));
      if (!ok) break;
      tc_fence_after();
      // (MMA1 goes out from the MMA warp)
      if (tid == 0 && n > 0) {   // chunk n - 1's V_new^T copy has been read (this chunk's tape entry may still be)
        bulk_wait_read_but1();
        mbar_arrive(&bar_sf);
      }
      if (with_o && n > 0) {   // the output of chunk n - 1, while MMA1 runs
        if (!(ok = wg_sync_and(1, mbar_wait(&bar_o[(n - 1) & 1], ((n - 1) >> 1) & 1, a.err)))) break;
        tc_fence_after();
        output(n - 1);
      }
      ok = wg_sync_and(1, mbar_wait(&bar_m1, par, a.err));
      if (!ok) break;
      tc_fence_after();
      {  // V_new^T row lt -> TMEM A operands: scaled by kd (state update), plain (output); and the BF16
         // V_new^T tile for the backward, staged in the chunk's V tile (its U^T MMA is done)
        float vn[64];
        tmem_ld32(taddr(tb, wq * 32, d1 - tb), vn);
        tmem_ld32(taddr(tb, wq * 32, d1 - tb + 32), vn + 32);
        const float* kd = scal + 64;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t ps[8], pn[8];
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const int r = q * 16 + 2 * e;
            pn[e] = pack_bf16(vn[r], vn[r + 1]);
            pn[e + 1] = pack_bf16(vn[r + 2], vn[r + 3]);
            if (KDA) {
              ps[e] = pn[e];
              ps[e + 1] = pn[e + 1];
            } else {
              const float4 k4 = *reinterpret_cast<const float4*>(kd + r);
              float t0, t1, t2, t3;
              mul2v(t0, t1, vn[r], vn[r + 1], k4.x, k4.y);
              mul2v(t2, t3, vn[r + 2], vn[r + 3], k4.z, k4.w);
              ps[e] = pack_bf16(t0, t1);
              ps[e + 1] = pack_bf16(t2, t3);
            }
          }
          tmem_st8(taddr(tb, wq * 32, TM_AVS + q * 8), ps);
          if (with_o) tmem_st8(taddr(tb, wq * 32, TM_AVN + q * 8), pn);
          if (with_vn) {
            *reinterpret_cast<uint4*>(st + SC_V + sw_chunk(lt, 2 * q, 128)) = make_uint4(pn[0], pn[1], pn[2], pn[3]);
            *reinterpret_cast<uint4*>(st + SC_V + sw_chunk(lt, 2 * q + 1, 128)) = make_uint4(pn[4], pn[5], pn[6], pn[7]);
          }
        }
        tmem_wait_st();
      }
      if (with_vn) fence_async_smem();
      tc_fence_before();
      named_bar(1, 128);
      if (tid == 0) {   // ---- MMA2 and the output MMAs go out from the MMA warp
        mbar_arrive(&go2);
        if (with_vn) {
          bulk_store(a.vn + ((size_t)(c0 + n) * a.HV + hv) * VN_BYTES, st + SC_V, VN_BYTES);
          bulk_commit();
        }
        // this chunk's tape entry has been read: the S^T tile may be rewritten
        if (with_vn) bulk_wait_read_but1();   // (the V_new^T copy just committed may still be reading)
        else bulk_wait_read();
      }
      ok = wg_sync_and(1, mbar_wait(&bar_m2, par, a.err));
      if (!ok) break;
      tc_fence_after();
      {  // S^T <- gamma_L S^T + dS^T (the S^T tile is rewritten below, after the O MMAs have read it)
        const float gL = scal[128];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          float ds[32];
          tmem_ld32(taddr(tb, wq * 32, TM_DS + h * 32), ds);
          if (KDA) {   // column i (key channel) decays by gamma_L[i]
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              const float4 gv = *reinterpret_cast<const float4*>(scal + h * 32 + e);
              fma2v(ds[e], ds[e + 1], gv.x, gv.y, S[h * 32 + e], S[h * 32 + e + 1]);
              fma2v(ds[e + 2], ds[e + 3], gv.z, gv.w, S[h * 32 + e + 2], S[h * 32 + e + 3]);
              S[h * 32 + e] = ds[e];
              S[h * 32 + e + 1] = ds[e + 1];
              S[h * 32 + e + 2] = ds[e + 2];
              S[h * 32 + e + 3] = ds[e + 3];
            }
          } else {
#pragma unroll
            for (int e = 0; e < 32; e += 2)
              fma2_to(S[h * 32 + e], S[h * 32 + e + 1], gL, S[h * 32 + e], S[h * 32 + e + 1], ds[e], ds[e + 1]);
          }
        }
        if (with_o && !mbar_wait(&bar_o[n & 1], (n >> 1) & 1, a.err)) ok = false;
        store_state_row(s_tile, lt, S);   // also the saved state entering the next chunk
      }
      fence_async_smem();
      tc_fence_before();
      ok = wg_sync_and(1, ok);
      if (!ok) break;
      if (tid == 0 && mode == 0 && a.tape && n + 1 < nch) {
        bulk_store(a.tape + ((size_t)(c0 + n + 1) * a.HV + hv) * STATE_BYTES, s_tile, STATE_BYTES);
        bulk_commit();
      }
      if (tid == 0 && n + 1 < nch) mbar_arrive(&go1);   // S^T of the next chunk is in its tile
    }
    if (ok && with_o && nch > 0) {   // the last chunk's output
      ok = wg_sync_and(1, mbar_wait(&bar_o[(nch - 1) & 1], ((nch - 1) >> 1) & 1, a.err));
      tc_fence_after();
      if (ok) output(nch - 1);
    }
    if (tid == 0 || tid == 32) bulk_wait_all();
    if (ok && (mode != 0 || write_bend)) {
      float* dst = (mode == 2 ? a.mend : a.bend) + ((size_t)split * a.HV + hv) * STATE_F32 + (size_t)lt * 128;
#pragma unroll
      for (int jj = 0; jj < 128; jj += 4)
        *reinterpret_cast<float4*>(dst + jj) = make_float4(S[jj], S[jj + 1], S[jj + 2], S[jj + 3]);
    }
    if (ok && mode == 0 && a.s_out && seg + 1 == a.seg_offsets[doc + 1]) {   // the document's S_out
      float* dst = a.s_out + ((size_t)doc * a.HV + hv) * STATE_F32 + lt;      // column lt of S [dk][dv]
#pragma unroll
      for (int jj = 0; jj < 128; ++jj) dst[jj * 128] = S[jj];
    }
  } else {
    // =================== helper warpgroup ===================
    for (int n = 0; n < nch && ok; ++n) {
      // ---- chunk n: land its tiles, W^T = K^T T'^T -> DW, U^T = V^T T''^T -> D1[n & 1], -W^T -> shared
      uint8_t* st = sm + (n & 1) * SC_STAGE;
      const int nt0 = n + 1 < nch ? a.chunk_tok0[c0 + n + 1] : 0;   // for the tile request below
      ok = wg_sync_and(2, mbar_wait(&full_bar[n & 1], (n >> 1) & 1, a.err));
      if (!ok) break;
      const int L = reinterpret_cast<const int*>(st + SC_SCAL)[129];
      if (KDA && L < CH && with_u) {   // zero the V rows past a document end (-W^T, Kd are zero there)
        for (int idx = lt; idx < (CH - L) * 16; idx += 128)
          *reinterpret_cast<uint4*>(st + SC_V + sw_chunk(L + (idx >> 4), idx & 15, 64)) = make_uint4(0u, 0u, 0u, 0u);
        fence_async_smem();
        named_bar(2, 128);
      }
      if (!KDA && L < CH) {   // zero the rows past a document end (they hold the next document)
        for (int idx = lt; idx < (CH - L) * 48; idx += 128) {
          const int t = idx / 48, rem = idx % 48, tile = rem / 16, c8 = rem % 16;
          const int off = tile == 0 ? SC_K : (tile == 1 ? SC_Q : SC_V);
          *reinterpret_cast<uint4*>(st + off + sw_chunk(L + t, c8, 64)) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_async_smem();
        named_bar(2, 128);
      }
      // MMA1(n - 1) has read the -W^T tile and the chain is done with D1[n & 1] (V_new^T of n - 2)
      if (n > 0 && !(ok = wg_sync_and(2, mbar_wait(&bar_m1, (n - 1) & 1, a.err)))) break;
      tc_fence_after();
      if (KDA) {   // U^T = V^T T''^T -> D1[n & 1] (-W^T came with the stage)
        if (with_u) {
          if (warp == 4) {
            const uint32_t a_v = smem_u32(st + SC_V), a_tpp = smem_u32(st + SC_TPP);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              mma_ss_w(tb + TM_D1 + (n & 1) * 64, desc_mn(a_v, 64, ks), desc_k(a_tpp, 64, ks),
                       idesc(128, 64, 1, 0), ks > 0);
            mma_commit_w(&bar_wu);
          }
          if (!(ok = wg_sync_and(2, mbar_wait(&bar_wu, n & 1, a.err)))) break;
          tc_fence_before();
        }
        named_bar(2, 128);
        if (tid == 128) mbar_arrive(&bar_wr);
      } else if (warp == 4) {
        const uint32_t a_k = smem_u32(st + SC_K), a_v = smem_u32(st + SC_V);
        const uint32_t a_tp = smem_u32(st + SC_TP), a_tpp = smem_u32(st + SC_TPP);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_ss_w(tb + TM_DW, desc_mn(a_k, 64, ks), desc_k(a_tp, 64, ks), idesc(128, 64, 1, 0), ks > 0);
        if (with_u) {
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_ss_w(tb + TM_D1 + (n & 1) * 64, desc_mn(a_v, 64, ks), desc_k(a_tpp, 64, ks), idesc(128, 64, 1, 0),
                     ks > 0);
        }
        mma_commit_w(&bar_wu);
      }
      if (with_o) {   // Q'_r = gamma_r rq_r q_r = (sc_r / scale) q_r in place
        const float* scal = reinterpret_cast<const float*>(st + SC_SCAL);
        const int r = lt >> 1;
        const float f = scal[r] * (1.0f / a.scale);
#pragma unroll
        for (int c8 = (lt & 1) * 8; c8 < (lt & 1) * 8 + 8; ++c8) {
          uint4* p = reinterpret_cast<uint4*>(st + SC_Q + sw_chunk(r, c8, 64));
          uint4 v = *p;
          __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 x = __bfloat1622float2(h2[e]);
            h2[e] = __floats2bfloat162_rn(x.x * f, x.y * f);
          }
          *p = v;
        }
      }
      if (!KDA) {
      if (!(ok = wg_sync_and(2, mbar_wait(&bar_wu, n & 1, a.err)))) break;
      tc_fence_after();
      {  // -W^T -> shared (row lt = dk index), the MN-major B operand of MMA1
        float w[64];
        tmem_ld32(taddr(tb, wq * 32, TM_DW), w);
        tmem_ld32(taddr(tb, wq * 32, TM_DW + 32), w + 32);
        uint8_t* wt = sm + SC_W;
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
          uint4 v;
          v.x = pack_bf16(-w[c8 * 8 + 0], -w[c8 * 8 + 1]);
          v.y = pack_bf16(-w[c8 * 8 + 2], -w[c8 * 8 + 3]);
          v.z = pack_bf16(-w[c8 * 8 + 4], -w[c8 * 8 + 5]);
          v.w = pack_bf16(-w[c8 * 8 + 6], -w[c8 * 8 + 7]);
          *reinterpret_cast<uint4*>(wt + sw_chunk(lt, c8, 128)) = v;
        }
      }
      fence_async_smem();
      tc_fence_before();
      named_bar(2, 128);
      if (tid == 128) mbar_arrive(&bar_wr);
      }
      // ---- chunk n + 1 into the stage of chunk n - 1 once the chain no longer reads it
      if (n > 0 && n + 1 < nch) {
        if (!(ok = wg_sync_and(2, mbar_wait(&bar_sf, (n - 1) & 1, a.err)))) break;
        if (tid == 128) {
          issue(n + 1, nt0);
          if (n + 2 < nch) prefetch(n + 2);
        }
      }
    }
  }
  // no MMA may outlive the TMEM allocation, and no tile copy the CTA's shared memory: on the error path
  // both are waited for whatever the error word says (bounded; a barrier phase nothing armed just
  // runs out)
  if (tid == 0 && !mbar_wait(&done, 0, a.err)) {
    mbar_drain(&done, 0);
    for (int b = 0; b < 2; ++b) {
      mbar_drain(&full_bar[b], 0);
      mbar_drain(&full_bar[b], 1);
    }
  }
  tc_fence_before();
  named_bar(3, SC_WORK);
  if (warp == 0) tmem_dealloc(tb, 512);
}

// S^T_{p+1} = S^T_p M_p^T + B_p^T, S_0 = 0, for the split segments of one
// document and value head; s_init[i] = start state of the segment after split
// i, bend[i] = B of split segment i, mend[i] = M^T of the segment after it.
__global__ void __launch_bounds__(256) merge_kernel(MergeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  float* Sp = reinterpret_cast<float*>(smem_raw);          // [128][129]
  float* Mt = Sp + 128 * 129;                              // [128][129]
  if (*(volatile int*)a.err) return;
  const int sd = blockIdx.x, hv = blockIdx.y, tid = threadIdx.x;
  const int f0 = a.sdoc_first[sd], f1 = a.sdoc_first[sd + 1];
  const size_t stride = (size_t)a.HV * STATE_F32;
  // S_1 = B_0
  for (int i = tid; i < STATE_F32; i += 256) {
    const float b = a.bend[(size_t)f0 * stride + (size_t)hv * STATE_F32 + i];
    Sp[(i >> 7) * 129 + (i & 127)] = b;
    a.s_init[(size_t)f0 * stride + (size_t)hv * STATE_F32 + i] = b;
  }
  __syncthreads();
  const int r0 = (tid >> 4) * 8, cc0 = (tid & 15) * 8;
  for (int p = f0 + 1; p < f1; ++p) {
    const float* M = a.mend + (size_t)(p - 1) * stride + (size_t)hv * STATE_F32;
    const float* B = a.bend + (size_t)p * stride + (size_t)hv * STATE_F32;
    for (int i = tid; i < STATE_F32; i += 256) Mt[(i >> 7) * 129 + (i & 127)] = M[i];
    __syncthreads();
    float acc[8][8];
#pragma unroll
    for (int x = 0; x < 8; ++x)
#pragma unroll
      for (int y = 0; y < 8; ++y) acc[x][y] = 0.f;
    for (int kk = 0; kk < 128; ++kk) {
      float sa[8], mb[8];
#pragma unroll
      for (int x = 0; x < 8; ++x) sa[x] = Sp[(r0 + x) * 129 + kk];
#pragma unroll
      for (int y = 0; y < 8; ++y) mb[y] = Mt[kk * 129 + cc0 + y];
#pragma unroll
      for (int x = 0; x < 8; ++x)
#pragma unroll
        for (int y = 0; y < 8; ++y) acc[x][y] = fmaf(sa[x], mb[y], acc[x][y]);
    }
    __syncthreads();
#pragma unroll
    for (int x = 0; x < 8; ++x)
#pragma unroll
      for (int y = 0; y < 8; ++y) {
        const int i = (r0 + x) * 128 + cc0 + y;
        const float v = acc[x][y] + B[i];
        Sp[(r0 + x) * 129 + cc0 + y] = v;
        a.s_init[(size_t)p * stride + (size_t)hv * STATE_F32 + i] = v;
      }
    __syncthreads();
  }
}

// documents without chunks: their boundary state passes through unchanged
__global__ void __launch_bounds__(256) passthrough_kernel(PassArgs a) {
  const int d = blockIdx.x;
  if (a.chunk_offsets[d + 1] != a.chunk_offsets[d]) return;
  const size_t n4 = (size_t)a.HV * STATE_F32 / 4, base = (size_t)d * a.HV * STATE_F32;
  float4* dst = reinterpret_cast<float4*>(a.dst + base);
  const float4* src = a.src ? reinterpret_cast<const float4*>(a.src + base) : nullptr;
  for (size_t i = threadIdx.x; i < n4; i += blockDim.x) dst[i] = src ? src[i] : make_float4(0.f, 0.f, 0.f, 0.f);
}
void launch_passthrough(const PassArgs& a, int N, cudaStream_t s) {
  if (N <= 0) return;
  prof_begin(K_PASS, s);
  passthrough_kernel<<<N, 256, 0, s>>>(a);
  prof_end(K_PASS, s);
}

void launch_fwd_scan(const ScanArgs& a, int nchains, cudaStream_t s) {
  if (nchains <= 0) return;
  const int id = a.walk ? K_FWD_WALK : K_FWD_SCAN;
  prof_begin(id, s);
  if (a.kda) fwd_scan_kernel<true><<<nchains, SC_THREADS, SC_SMEM_ALLOC, s>>>(a);
  else fwd_scan_kernel<false><<<nchains, SC_THREADS, SC_SMEM_ALLOC, s>>>(a);
  prof_end(id, s);
}
void launch_merge(const MergeArgs& a, int nsdoc, cudaStream_t s) {
  if (nsdoc <= 0) return;
  prof_begin(K_FWD_MERGE, s);
  merge_kernel<<<dim3(nsdoc, a.HV), 256, 2 * 128 * 129 * 4, s>>>(a);
  prof_end(K_FWD_MERGE, s);
}
void setup_fwd_scan_attrs() {
  cudaFuncSetAttribute(fwd_scan_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, SC_SMEM_ALLOC);
  cudaFuncSetAttribute(fwd_scan_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, SC_SMEM_ALLOC);
  cudaFuncSetAttribute(merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 2 * 128 * 129 * 4);
}

}  // namespace gdn
