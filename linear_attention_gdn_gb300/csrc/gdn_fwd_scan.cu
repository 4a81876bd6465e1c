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
//   full (walk = 0)  every segment, from its true start state; writes o, tape
//   B    (walk = 1)  segment from a zero state; writes its end state B_p^T
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
constexpr int SC_SIDE = SC_O + 16384;       // per-token output scales of the last two chunks (+ their L)
constexpr int SC_SMEM = SC_SIDE + 2 * 272;
constexpr int SC_SMEM_ALLOC = SC_SMEM + 1024;

// TMEM columns: D1 double-buffered (U^T, then V_new^T, of chunks n and n+1)
constexpr int TM_D1 = 0, TM_DW = 128, TM_DS = 192, TM_O1 = 320, TM_O2 = 384, TM_AVS = 448, TM_AVN = 480;

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

// The chain of one chunk is MMA1 (V_new^T = U^T - S^T W^T) -> V_new hop ->
// MMA2 (dS^T = (V_new^T diag(kd)) K, with the output products) -> S hop.
// Work that does not feed the chain runs in the shadow of its MMAs:
// W^T / U^T of chunk n+1 are issued right after MMA1(n) and their hop overlaps
// MMA2(n); the output epilogue of chunk n-1 overlaps MMA1(n).
__global__ void __launch_bounds__(128, 1) fwd_scan_kernel(const __grid_constant__ ScanArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full_bar[2], bar_m1, bar_w, bar_m2;
  __shared__ uint32_t tslot;
  const int tid = threadIdx.x, warp = tid >> 5;
  if (*(volatile int*)a.err) return;

  int mode, seg, hv, split = -1;
  if (!a.walk) {
    mode = 0;
    seg = blockIdx.x / a.HV;
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
  }
  const int kh = hv / a.G;
  const int c0 = a.seg_c0[seg], nch = a.seg_c1[seg] - c0;
  const bool with_o = mode == 0 && a.o != nullptr;
  const bool with_u = mode != 2;
  const bool with_vn = mode == 0 && a.vn != nullptr;   // V_new^T tiles for the backward
  const uint32_t tx_bytes = mode == 0 ? (with_o ? 74752u : 50176u) : (mode == 1 ? 50176u : 25600u);
  const uint32_t cb_bytes = mode == 2 ? 8192u : (with_o ? 24576u : 16384u);

  // ---- initial state (row tid of S^T)
  float S[128];
  {
    const float* src = nullptr;
    if (mode == 0 && a.seg_idx[seg] > 0)
      src = a.s_init + ((size_t)a.seg_split[seg - 1] * a.HV + hv) * STATE_F32 + (size_t)tid * 128;
#pragma unroll
    for (int jj = 0; jj < 128; ++jj) S[jj] = src ? src[jj] : (mode == 2 && jj == tid ? 1.f : 0.f);
  }
  uint8_t* s_tile = sm + SC_S;
  store_state_row(s_tile, tid, S);
  if (mode == 0 && a.tape) store_state_row(a.tape + ((size_t)c0 * a.HV + hv) * STATE_BYTES, tid, S);

  if (warp == 0) tmem_alloc(&tslot, 512);
  if (tid == 0) {
    mbar_init(&full_bar[0], 1);
    mbar_init(&full_bar[1], 1);
    mbar_init(&bar_m1, 1);
    mbar_init(&bar_w, 1);
    mbar_init(&bar_m2, 1);
    asm volatile("fence.mbarrier_init.release.cluster;");
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tslot;

  auto issue = [&](int n) {
    const int ci = c0 + n;
    uint8_t* st = sm + (n & 1) * SC_STAGE;
    uint64_t* bar = &full_bar[n & 1];
    const int t0 = a.chunk_tok0[ci];
    const uint8_t* cbp = a.cb + ((size_t)ci * a.HV + hv) * CB_BYTES;
    mbar_expect_tx(bar, tx_bytes);
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
  if (tid == 0) {
    if (nch > 0) issue(0);
    if (nch > 1) issue(1);
  }

  uint32_t ph_m1 = 0, ph_w = 0, ph_m2 = 0;
  bool ok = true;
  const uint32_t sm_s = smem_u32(s_tile), sm_w = smem_u32(sm + SC_W);
  float* side = reinterpret_cast<float*>(sm + SC_SIDE);   // [2][68]: sc[64], L

  // wait for chunk n's tiles; zero the rows past a document end (they hold the next document)
  auto land = [&](int n) -> bool {
    uint8_t* st = sm + (n & 1) * SC_STAGE;
    if (!__syncthreads_and(mbar_wait(&full_bar[n & 1], (n >> 1) & 1, a.err))) return false;
    const int L = reinterpret_cast<const int*>(st + SC_SCAL)[129];
    if (L < CH) {
      for (int idx = tid; idx < (CH - L) * 48; idx += 128) {
        const int t = idx / 48, rem = idx % 48, tile = rem / 16, c8 = rem % 16;
        const int off = tile == 0 ? SC_K : (tile == 1 ? SC_Q : SC_V);
        *reinterpret_cast<uint4*>(st + off + sw_chunk(L + t, c8, 64)) = make_uint4(0u, 0u, 0u, 0u);
      }
      fence_async_smem();
      __syncthreads();
    }
    return true;
  };
  // W^T of chunk n -> DW, U^T -> D1[n & 1]
  auto issue_wu = [&](int n) {
    uint8_t* st = sm + (n & 1) * SC_STAGE;
    const uint32_t a_k = smem_u32(st + SC_K), a_v = smem_u32(st + SC_V);
    const uint32_t a_tp = smem_u32(st + SC_TP), a_tpp = smem_u32(st + SC_TPP);
    tc_fence_after();
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      mma_ss_w(tb + TM_DW, desc_mn(a_k, 64, ks), desc_k(a_tp, 64, ks), idesc(128, 64, 1, 0), ks > 0);
    if (with_u) {
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_ss_w(tb + TM_D1 + (n & 1) * 64, desc_mn(a_v, 64, ks), desc_k(a_tpp, 64, ks), idesc(128, 64, 1, 0),
               ks > 0);
    }
    mma_commit_w(&bar_w);
  };
  // -W^T -> shared (row tid = dk index), the MN-major B operand of MMA1
  auto hop_w = [&]() {
    float w[64];
    tmem_ld32(taddr(tb, warp * 32, TM_DW), w);
    tmem_ld32(taddr(tb, warp * 32, TM_DW + 32), w + 32);
    uint8_t* wt = sm + SC_W;
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) {
      uint4 v;
      v.x = pack_bf16(-w[c8 * 8 + 0], -w[c8 * 8 + 1]);
      v.y = pack_bf16(-w[c8 * 8 + 2], -w[c8 * 8 + 3]);
      v.z = pack_bf16(-w[c8 * 8 + 4], -w[c8 * 8 + 5]);
      v.w = pack_bf16(-w[c8 * 8 + 6], -w[c8 * 8 + 7]);
      *reinterpret_cast<uint4*>(wt + sw_chunk(tid, c8, 128)) = v;
    }
    fence_async_smem();
  };
  // output of chunk n from O1, O2 (TMEM) with the saved per-token scales
  uint8_t* o_stage = sm + SC_O;
  auto output = [&](int n) {
    const float* sc = side + (n & 1) * 68;
    const int L = reinterpret_cast<const int*>(sc)[64];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float x1[32], x2[32];
      tmem_ld32(taddr(tb, warp * 32, TM_O1 + h * 32), x1);
      tmem_ld32(taddr(tb, warp * 32, TM_O2 + h * 32), x2);
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int r = h * 32 + e;
        *reinterpret_cast<__nv_bfloat16*>(o_stage + sw_off(r, tid, 64)) =
            __float2bfloat16_rn(fmaf(sc[r], x1[e], a.scale * x2[e]));
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    const int t0 = a.chunk_tok0[c0 + n];
    if (L < CH) {  // ragged last chunk: only its own rows (the next rows are another document's)
      for (int idx = tid; idx < L * 16; idx += 128) {
        const int r = idx >> 4, c8 = idx & 15;
        *reinterpret_cast<uint4*>(a.o + ((size_t)(t0 + r) * a.HV + hv) * D + c8 * 8) =
            *reinterpret_cast<const uint4*>(o_stage + sw_chunk(r, c8, 64));
      }
    } else if (tid == 0) {
      tma_store_3d(&a.to, o_stage, 0, hv, t0);
      tma_store_3d(&a.to, o_stage + 8192, 64, hv, t0);
      bulk_commit();
    }
  };

  // ---- prologue: W^T, U^T of chunk 0 and its -W^T tile
  if (nch > 0) {
    ok = land(0);
    if (ok && warp == 0) issue_wu(0);
    ok = ok && __syncthreads_and(mbar_wait(&bar_w, ph_w, a.err));
    ph_w ^= 1;
    tc_fence_after();
    if (ok) hop_w();
    tc_fence_before();
    __syncthreads();
  }
  for (int n = 0; n < nch && ok; ++n) {
    uint8_t* st = sm + (n & 1) * SC_STAGE;
    const uint32_t a_k = smem_u32(st + SC_K), a_q = smem_u32(st + SC_Q), a_aqk = smem_u32(st + SC_AQK);
    const float* scal = reinterpret_cast<const float*>(st + SC_SCAL);
    const uint32_t d1 = tb + TM_D1 + (n & 1) * 64;
    // ---- MMA1: V_new^T = U^T - S^T W^T (into D1[n & 1])
    if (warp == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_ss_w(d1, desc_k(sm_s, 128, ks), desc_mn(sm_w, 128, ks), idesc(128, 64, 0, 1),
                 (with_u || ks > 0) ? 1u : 0u);
      mma_commit_w(&bar_m1);
    }
    // ---- in its shadow: the output of chunk n - 1, then W^T / U^T of chunk n + 1
    if (with_o && n > 0) {
      tc_fence_after();
      output(n - 1);
    }
    const bool next = n + 1 < nch;
    if (next) {
      if (!(ok = land(n + 1))) break;
      if (warp == 0) issue_wu(n + 1);
    }
    ok = __syncthreads_and(mbar_wait(&bar_m1, ph_m1, a.err));
    ph_m1 ^= 1;
    if (!ok) break;
    tc_fence_after();
    {  // V_new^T row tid -> TMEM A operands: scaled by kd (state update), plain (output)
      float vn[64];
      tmem_ld32(taddr(tb, warp * 32, d1 - tb), vn);
      tmem_ld32(taddr(tb, warp * 32, d1 - tb + 32), vn + 32);
      const float* kd = scal + 64;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t ps[8], pn[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int r = q * 16 + 2 * e;
          ps[e] = pack_bf16(vn[r] * kd[r], vn[r + 1] * kd[r + 1]);
          pn[e] = pack_bf16(vn[r], vn[r + 1]);
        }
        tmem_st8(taddr(tb, warp * 32, TM_AVS + q * 8), ps);
        if (with_o) tmem_st8(taddr(tb, warp * 32, TM_AVN + q * 8), pn);
        if (with_vn) {   // staged in the -W^T tile, which MMA1 has finished reading
          uint8_t* vt = sm + SC_W;
          *reinterpret_cast<uint4*>(vt + sw_chunk(tid, 2 * q, 128)) = make_uint4(pn[0], pn[1], pn[2], pn[3]);
          *reinterpret_cast<uint4*>(vt + sw_chunk(tid, 2 * q + 1, 128)) = make_uint4(pn[4], pn[5], pn[6], pn[7]);
        }
      }
      if (with_o) {  // this chunk's output scales outlive its stage buffer
        float* sd = side + (n & 1) * 68;
        if (tid < 64) sd[tid] = scal[tid];
        if (tid == 64) reinterpret_cast<int*>(sd)[64] = reinterpret_cast<const int*>(scal)[129];
      }
      tmem_wait_st();
    }
    if (with_vn) fence_async_smem();
    tc_fence_before();
    __syncthreads();
    // ---- MMA2: dS^T = (V_new^T diag(kd)) K; O2 = V_new^T Aqk^T; O1 = S^T Q^T
    if (warp == 0) {
      if (with_vn && tid == 0) {
        bulk_store(a.vn + ((size_t)(c0 + n) * a.HV + hv) * VN_BYTES, sm + SC_W, VN_BYTES);
        bulk_commit();
      }
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_ts_w(tb + TM_DS, tb + TM_AVS + ks * 8, desc_mn(a_k, 64, ks), idesc(128, 128, 0, 1), ks > 0);
      if (with_o) {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_ts_w(tb + TM_O2, tb + TM_AVN + ks * 8, desc_k(a_aqk, 64, ks), idesc(128, 64, 0, 0), ks > 0);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_ss_w(tb + TM_O1, desc_k(sm_s, 128, ks), desc_k(a_q, 64, ks), idesc(128, 64, 0, 0), ks > 0);
      }
      mma_commit_w(&bar_m2);
      if (tid == 0) bulk_wait_read();   // earlier tape / output / V_new stores have read the tiles rewritten below
    }
    // ---- in its shadow: the -W^T tile of chunk n + 1
    if (next) {
      ok = __syncthreads_and(mbar_wait(&bar_w, ph_w, a.err));
      ph_w ^= 1;
      if (!ok) break;
      tc_fence_after();
      hop_w();
    }
    ok = __syncthreads_and(mbar_wait(&bar_m2, ph_m2, a.err));
    ph_m2 ^= 1;
    if (!ok) break;
    tc_fence_after();
    {  // S^T <- gamma_L S^T + dS^T
      const float gL = scal[128];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        float ds[32];
        tmem_ld32(taddr(tb, warp * 32, TM_DS + h * 32), ds);
#pragma unroll
        for (int e = 0; e < 32; ++e) S[h * 32 + e] = fmaf(gL, S[h * 32 + e], ds[e]);
      }
      store_state_row(s_tile, tid, S);   // also the saved state entering the next chunk
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      if (mode == 0 && a.tape && next) {
        bulk_store(a.tape + ((size_t)(c0 + n + 1) * a.HV + hv) * STATE_BYTES, s_tile, STATE_BYTES);
        bulk_commit();
      }
      if (n + 2 < nch) issue(n + 2);   // chunk n's stage is dead: its scales are in `side`
    }
  }
  if (ok && with_o && nch > 0) {
    tc_fence_after();
    output(nch - 1);
  }
  if (tid == 0) bulk_wait_read();
  if (ok && mode != 0) {
    float* dst = (mode == 1 ? a.bend : a.mend) + ((size_t)split * a.HV + hv) * STATE_F32 + (size_t)tid * 128;
#pragma unroll
    for (int jj = 0; jj < 128; jj += 4)
      *reinterpret_cast<float4*>(dst + jj) = make_float4(S[jj], S[jj + 1], S[jj + 2], S[jj + 3]);
  }
  tc_fence_before();
  __syncthreads();
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

void launch_fwd_scan(const ScanArgs& a, int nchains, cudaStream_t s) {
  if (nchains <= 0) return;
  const int id = a.walk ? K_FWD_WALK : K_FWD_SCAN;
  prof_begin(id, s);
  fwd_scan_kernel<<<nchains, 128, SC_SMEM_ALLOC, s>>>(a);
  prof_end(id, s);
}
void launch_merge(const MergeArgs& a, int nsdoc, cudaStream_t s) {
  if (nsdoc <= 0) return;
  prof_begin(K_FWD_MERGE, s);
  merge_kernel<<<dim3(nsdoc, a.HV), 256, 2 * 128 * 129 * 4, s>>>(a);
  prof_end(K_FWD_MERGE, s);
}
void setup_fwd_scan_attrs() {
  cudaFuncSetAttribute(fwd_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SC_SMEM_ALLOC);
  cudaFuncSetAttribute(merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 2 * 128 * 129 * 4);
}

}  // namespace gdn
