// gdn_kda.cu -- the per-channel-decay form (KDA) of the chunked gated delta rule:
// the same recurrence with one decay per key channel,
//   S'_t = Diag(exp(g_t)) S_{t-1},  S_t = S'_t + beta_t k^_t (v_t - S'_t^T k^_t)^T,  o_t = scale S_t^T q^_t,
// g_t in R^dk ("perf(cake_kda) ... #7097" page: the packed KDA training family beside the GDN one).
//
// Chunk form (64 tokens, entering state S; G = chunk-local cumulative log decay per channel, a
// 64 x 128 array; gamma = exp(G); every relative decay exp(G_r - G_c), c <= r, is at most 1):
//   M_rc = k^_r . (exp(G_r - G_c) k^_c),  P_rc = q^_r . (exp(G_r - G_c) k^_c)   (c <= r)
//   A = strict_tril(diag(beta) M),  T = (I + A)^-1,  T'' = T diag(beta)
//   W = T'' (gamma . K^),  U = T'' V,  V_new = U - W S
//   O = scale ((gamma . Q^) S + P V_new),  S_next = Diag(gamma_L) S + (exp(G_L - G) . K^)^T V_new
// i.e. the GDN chunk form with every decay moved inside the channel sums.
//
// Kernels here:
//   kda_prep_kernel  per (chunk, value head): G, M and P on the tensor cores, T, and the block the
//                    walks read (-W^T, Kd, T'', gamma_L, Q~, P, T, M^T)
//   kda_out_kernel   per (chunk, value head): o from the saved state and V_new^T
// The state walks are fwd_scan_kernel<true> / bwd_scan_kernel<true> (the GDN walks on this block).
//
// M and P on the tensor cores.  The relative decay does not factor into a row and a column term
// over a whole chunk without overflow, so the chunk is cut into four 16-token blocks.  For rows r of
// block a, with Gx_a the log decay entering block a (zero for a = 0),
//   exp(G_r - G_c) = exp(G_r - Gx_a) exp(Gx_a - G_c),
// the first factor at most 1 and the second at most 1 for c before block a; for c inside block a it
// is at most exp of the block's own decay range.  So, per block a (an N = 16 slice of the result),
//   M^T[:, block a] = R_a Lk[block a]^T,  P^T[:, block a] = R_a Lq[block a]^T,
//   R_a[c] = exp(Gx_a - G_c) . k^_c (c < 16 a + 16),  Lk_r = exp(G_r - Gx_a) . k^_r,  Lq likewise,
// with every factor formed from Rb_c = exp(Gx_{blk c} - G_c) . k^_c and per-channel block ratios.
// The factors stay in BF16's range while no channel decays by more than 2^-96 within one 16-token
// block; a chunk beyond that is refused with GDN_ERR_GATE_RANGE (written to the error word).
#include <algorithm>
#include <cstring>

#include "gdn.h"
#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_prof.h"
#include "gdn_ut.cuh"

namespace gdn {

// ---------------------------------------------------------------------------
// preparation
// ---------------------------------------------------------------------------
constexpr int KP_KQ = 0;        // [K; Q] SwTile(128 x 128): raw tiles, then Lk / Lq, then K~ / Q~
constexpr int KP_G = 32768;     // FP32 G [64][128]; then the two R_a tiles; then the FP32 array and the
                                // inverse's tiles; then T'' (0), T (8 KiB), -W^T (16 KiB)
constexpr int KP_B = 65536;     // Rb, then Kd; then P (0) and M^T (8 KiB)
constexpr int KP_SMEM = KP_B + 16384;
constexpr int KP_SMEM_ALLOC = KP_SMEM + 1024;
constexpr float kKdaRange = 96.f;   // log2 units: the largest decay exponent a factor may carry
// TMEM columns: [M^T | P^T] of each 16-token block (4 x 32), then the inverse's products and W^T
constexpr int KT_MP = 0, KT_INV = 128, KT_COLS = 256;
static_assert(UT_WORK_BYTES <= 32768, "the FP32 array fits in the G region");

__device__ __forceinline__ int kda_pair(int a, int b) { return a * (a - 1) / 2 + b; }   // b < a

__device__ __forceinline__ void unpack8(const uint4& w, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 x = __bfloat1622float2(h[e]);
    f[2 * e] = x.x;
    f[2 * e + 1] = x.y;
  }
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]), pack_bf16(f[6], f[7]));
}
__device__ __forceinline__ void ld8(const float* p, float (&f)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

// One CTA per (chunk, value head); two warpgroups, two CTAs per SM.
constexpr int KP_THREADS = 256;
__global__ void __launch_bounds__(KP_THREADS, 2) kda_prep_kernel(const __grid_constant__ KdaPrepArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_align1024(smem_raw);
  __shared__ __align__(16) float rk[CH], rq[CH], bs[CH];
  __shared__ __align__(16) float gx[4][D];     // log2 decay entering each 16-token block (block 0: 0)
  __shared__ __align__(16) float fab[6][D];    // exp2(gx[a] - gx[b]), b < a
  __shared__ __align__(16) float gamb[4][D];   // exp2(gx[a])
  __shared__ __align__(16) float phib[4][D];   // exp2(G_L - gx[a])
  __shared__ __align__(16) float scal[256];    // gamma_L[128]; (int) L at index 129
  __shared__ uint64_t bar_ld, bar_v[2], bar_t;
  __shared__ uint32_t tslot;
  __shared__ int unsafe;
  const int c = blockIdx.x / a.HV, hv = blockIdx.x % a.HV, j = hv / a.G;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (*(volatile int*)a.err) return;
  const int tok0 = a.chunk_tok0[c], L = a.chunk_len[c];
  uint8_t* kq = sm + KP_KQ;
  float* Gm = reinterpret_cast<float*>(sm + KP_G);
  uint8_t* rbt = sm + KP_B;
  uint8_t* kbp = a.kb + ((size_t)c * a.HV + hv) * KB_BYTES;

  if (warp == 0) tmem_alloc(&tslot, KT_COLS);
  if (tid == 0) {
    mbar_init(&bar_ld, 1);
    mbar_init(&bar_v[0], 1);
    mbar_init(&bar_v[1], 1);
    mbar_init(&bar_t, 1);
    asm volatile("fence.mbarrier_init.release.cluster;");
    unsafe = 0;
    // the K, Q tiles and the value head's 64 g rows (one TMA box; rows past L are read as zero below)
    mbar_expect_tx(&bar_ld, 32768u + 32768u);
    tma_load_3d(kq, &a.tk, 0, j, tok0, &bar_ld);
    tma_load_3d(kq + 8192, &a.tq, 0, j, tok0, &bar_ld);
    tma_load_3d(kq + 16384, &a.tk, 64, j, tok0, &bar_ld);
    tma_load_3d(kq + 24576, &a.tq, 64, j, tok0, &bar_ld);
    tma_load_3d(Gm, &a.tg, 0, hv, tok0, &bar_ld);
  }
  if (tid < CH) bs[tid] = tid < L ? a.beta[(size_t)(tok0 + tid) * a.HV + hv] : 0.f;
  __syncthreads();   // the barriers' initialisation is visible before any thread waits on them
  bool landed = __syncthreads_and(mbar_wait(&bar_ld, 0, a.err));
  if (landed && tid < 128) {  // channel tid: the cumulative decay G in log2 units (rows past L keep
                              // G_{L-1}), the block entries, the factors
    const int i = tid;
    float run = 0.f, ref = 0.f, mx = 0.f;
    for (int r = 0; r < CH; ++r) {
      if ((r & 15) == 0) {
        ref = run;
        gx[r >> 4][i] = run;
      }
      run = fmaf(r < L ? Gm[r * D + i] : 0.f, kUtLog2e, run);   // (rows past L: the next document's)
      Gm[r * D + i] = run;
      mx = fmaxf(mx, fabsf(run - ref));
    }
    const float GL = run;
    float gxv[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) gxv[b] = gx[b][i];
    float up = fmaxf(mx, GL);   // every exponent below is at most this (all <= 0 for a decay)
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      gamb[b][i] = exp2f(gxv[b]);
      phib[b][i] = exp2f(GL - gxv[b]);
      up = fmaxf(up, fmaxf(gxv[b], GL - gxv[b]));
    }
#pragma unroll
    for (int aa = 1; aa < 4; ++aa)
#pragma unroll
      for (int b = 0; b < aa; ++b) {
        fab[kda_pair(aa, b)][i] = exp2f(gxv[aa] - gxv[b]);
        up = fmaxf(up, gxv[aa] - gxv[b]);
      }
    scal[i] = exp2f(GL);
    if (!(up <= kKdaRange)) unsafe = 1;   // (also catches a NaN gate)
  }
  if (tid == 0) reinterpret_cast<int*>(scal)[129] = L;
  __syncthreads();
  const uint32_t tb = tslot;
  int vpend = 0;   // error path: versions whose completion was not seen (bit v & 1 -> bar_v, phase v >> 1)
  int t_pend = -1;
  bool ok = landed;
  if (ok && unsafe) {
    if (tid == 0) atomicCAS(a.err, 0, ST_GATE_RANGE);
    ok = false;
  }
  if (!ok) {
    if (tid == 0) mbar_drain(&bar_ld, 0);
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, KT_COLS);
    return;
  }
  if (L < CH) {
    if (tid < 128) ut_zero_tail(kq, L, tid);
    __syncthreads();
  }
  if (tid < 128) {
    const float rn = ut_row_rnorm(kq, tid, a.l2norm);
    if (tid < 64) rk[tid] = rn;
    else rq[tid - 64] = rn;
  }
  __syncthreads();
  // ---- pass 1: Lk, Lq in place; Rb (own-block reference) into its tile
#pragma unroll 2
  for (int it = 0; it < 1024 / KP_THREADS; ++it) {
    const int idx = tid + KP_THREADS * it, r = idx >> 4, c8 = idx & 15, blk = r >> 4;
    float g8[8], x8[8], kf[8], qf[8];
    ld8(Gm + r * D + 8 * c8, g8);
    ld8(&gx[blk][8 * c8], x8);
    uint4* kp = reinterpret_cast<uint4*>(kq + sw_chunk(r, c8, 128));
    uint4* qp = reinterpret_cast<uint4*>(kq + sw_chunk(64 + r, c8, 128));
    unpack8(*kp, kf);
    unpack8(*qp, qf);
    const float fk = rk[r], fq = rq[r];
    float lk[8], lq[8], rb[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float d = g8[e] - x8[e];
      const float lam = exp2f(d), ein = exp2f(-d);
      lk[e] = fk * kf[e] * lam;
      lq[e] = fq * qf[e] * lam;
      rb[e] = fk * kf[e] * ein;
    }
    *kp = pack8(lk);
    *qp = pack8(lq);
    *reinterpret_cast<uint4*>(rbt + sw_chunk(r, c8, 64)) = pack8(rb);
  }
  fence_async_smem();
  __syncthreads();
  // ---- R_a tiles (rows c < 16 a + 16: Rb scaled by exp2(gx[a] - gx[blk c]); beyond: zero) and the
  // M^T | P^T products, two buffers in the (now dead) G region
  auto build_version = [&](int v, uint8_t* dst) {
#pragma unroll 2
    for (int it = 0; it < 1024 / KP_THREADS; ++it) {
      const int idx = tid + KP_THREADS * it, r = idx >> 4, c8 = idx & 15, blk = r >> 4;
      uint4 w = make_uint4(0u, 0u, 0u, 0u);
      if (blk == v) {
        w = *reinterpret_cast<const uint4*>(rbt + sw_chunk(r, c8, 64));
      } else if (blk < v) {
        float f[8], x[8];
        unpack8(*reinterpret_cast<const uint4*>(rbt + sw_chunk(r, c8, 64)), x);
        ld8(&fab[kda_pair(v, blk)][8 * c8], f);
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] *= f[e];
        w = pack8(x);
      }
      *reinterpret_cast<uint4*>(dst + sw_chunk(r, c8, 64)) = w;
    }
  };
  auto issue_version = [&](int v, const uint8_t* vt) {   // warp 0
    const uint32_t sa = smem_u32(vt), sb = smem_u32(kq);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
      mma_ss_w(tb + KT_MP + 32 * v, desc_k(sa, 64, ks), desc_k(sb, 128, ks, 16 * v), idesc(64, 16, 0, 0), ks > 0);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
      mma_ss_w(tb + KT_MP + 32 * v + 16, desc_k(sa, 64, ks), desc_k(sb, 128, ks, 64 + 16 * v), idesc(64, 16, 0, 0),
               ks > 0);
    mma_commit_w(&bar_v[v & 1]);
  };
  auto to_mma = [&]() {
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  };
  uint8_t* vbuf0 = sm + KP_G;
  uint8_t* vbuf1 = sm + KP_G + 16384;
  build_version(0, vbuf0);
  build_version(1, vbuf1);
  to_mma();
  if (warp == 0) {
    issue_version(0, vbuf0);
    issue_version(1, vbuf1);
  }
  vpend = 3;
  ok = __syncthreads_and(mbar_wait(&bar_v[0], 0, a.err));
  if (ok) {
    vpend &= ~1;
    build_version(2, vbuf0);
    to_mma();
    if (warp == 0) issue_version(2, vbuf0);
    vpend |= 4;
    ok = __syncthreads_and(mbar_wait(&bar_v[1], 0, a.err));
  }
  if (ok) {
    vpend &= ~2;
    build_version(3, vbuf1);
    to_mma();
    if (warp == 0) issue_version(3, vbuf1);
    vpend |= 8;
    ok = __syncthreads_and(mbar_wait(&bar_v[0], 1, a.err));
  }
  if (ok) {
    vpend &= ~4;
    ok = __syncthreads_and(mbar_wait(&bar_v[1], 1, a.err));
  }
  if (ok) vpend = 0;
  tc_fence_after();
  uint32_t tph = 0;
  if (ok) {
    // ---- Kd = Rb . exp2(G_L - gx[blk]) in place; shipped now
#pragma unroll 2
    for (int it = 0; it < 1024 / KP_THREADS; ++it) {
      const int idx = tid + KP_THREADS * it, r = idx >> 4, c8 = idx & 15, blk = r >> 4;
      float f[8], x[8];
      uint4* p = reinterpret_cast<uint4*>(rbt + sw_chunk(r, c8, 64));
      unpack8(*p, x);
      ld8(&phib[blk][8 * c8], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] *= f[e];
      *p = pack8(x);
    }
    fence_async_smem();
    __syncthreads();
    if (tid == 0) {
      bulk_store(kbp + KB_KD, rbt, 16384u);
      bulk_commit();
    }
    // ---- the FP32 array: row c holds A[r][c] = beta_r M[r][c] for c < r < L (row c of M^T)
    float* Sm = reinterpret_cast<float*>(sm + KP_G);
#pragma unroll 1
    for (int blk = 2 * (warp >> 2); blk < 2 * (warp >> 2) + 2; ++blk) {   // the warpgroups split the blocks
      float mp[32];   // M^T[c][16 blk + u] at u, P^T at 16 + u (lanes 0-15 of the warp: rows 16 (warp % 4) + lane)
      tmem_ld32(taddr(tb, (warp & 3) * 32, KT_MP + 32 * blk), mp);
      if (lane < 16) {
        const int cc = 16 * (warp & 3) + lane;
#pragma unroll
        for (int u = 0; u < 16; u += 4) {
          const int r = 16 * blk + u;
          float4 v;
          v.x = (r + 0 > cc && r + 0 < L) ? bs[r + 0] * mp[u + 0] : 0.f;
          v.y = (r + 1 > cc && r + 1 < L) ? bs[r + 1] * mp[u + 1] : 0.f;
          v.z = (r + 2 > cc && r + 2 < L) ? bs[r + 2] * mp[u + 2] : 0.f;
          v.w = (r + 3 > cc && r + 3 < L) ? bs[r + 3] * mp[u + 3] : 0.f;
          *reinterpret_cast<float4*>(Sm + cc * UT_ALD + r) = v;
        }
      }
    }
    __syncthreads();
    if (tid < 64) ut_diag_blocks(Sm, tid, 1);
    __syncthreads();
    const UtInvTiles tiles{sm + KP_G, sm + KP_G + 8192};
    ok = ut_tc_inverse<KP_THREADS>(Sm, tiles, tb, KT_INV, &bar_t, tph, a.err, t_pend);
  }
  if (ok) {
    // ---- T'' and T tiles (over D and X: the last product has read them)
    {
      constexpr int NG = UtGroups<KP_THREADS>::NG;
      uint32_t u[NG][8];
      ut_ld_result<KP_THREADS>(tb, KT_INV, warp, u);
      const int r0 = 16 * (warp & 3) + (lane >> 2), cq = 2 * (lane & 3), g0 = UtGroups<KP_THREADS>::first(warp);
#pragma unroll
      for (int g = 0; g < NG; ++g)
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
          const int r = r0 + 8 * ((i >> 1) & 1), cc = 16 * (g0 + g) + 8 * (i >> 2) + cq;
          const uint32_t off = sw_off(r, cc, 64);
          const float t0 = __uint_as_float(u[g][i]), t1 = __uint_as_float(u[g][i + 1]);
          *reinterpret_cast<uint32_t*>(sm + KP_G + off) = pack_bf16(t0 * bs[cc], t1 * bs[cc + 1]);
          *reinterpret_cast<uint32_t*>(sm + KP_G + 8192 + off) = pack_bf16(t0, t1);
        }
    }
    if (tid == 0) bulk_wait_read();   // Kd has been read out of the Rb tile
    __syncthreads();
    // ---- P and M^T tiles (BF16) into the Rb tile's space, from the rows of [M^T | P^T]
#pragma unroll 1
    for (int blk = 2 * (warp >> 2); blk < 2 * (warp >> 2) + 2; ++blk) {
      float mp[32];
      tmem_ld32(taddr(tb, (warp & 3) * 32, KT_MP + 32 * blk), mp);
      if (lane < 16) {
        const int cc = 16 * (warp & 3) + lane;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float x[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int r = 16 * blk + 8 * h + e;
            x[e] = (r > cc && r < L) ? mp[8 * h + e] : 0.f;
          }
          *reinterpret_cast<uint4*>(rbt + 8192 + sw_chunk(cc, 2 * blk + h, 64)) = pack8(x);
        }
#pragma unroll
        for (int u = 0; u < 16; ++u) {   // column cc of P: P[r][cc] = P^T[cc][r] for cc <= r < L
          const int r = 16 * blk + u;
          *reinterpret_cast<__nv_bfloat16*>(rbt + sw_off(r, cc, 64)) =
              __float2bfloat16_rn((r >= cc && r < L) ? mp[16 + u] : 0.f);
        }
      }
    }
    fence_async_smem();
    __syncthreads();
    if (tid == 0) {
      bulk_store(kbp + KB_TPP, sm + KP_G, TILE64_BYTES);
      bulk_store(kbp + KB_T, sm + KP_G + 8192, TILE64_BYTES);
      bulk_store(kbp + KB_AQK, rbt, TILE64_BYTES);
      bulk_store(kbp + KB_MT, rbt + 8192, TILE64_BYTES);
      bulk_store(kbp + KB_SCAL, scal, CB_SCAL_BYTES);
      bulk_commit();
    }
    // ---- K~ = Lk . exp2(gx[blk]), Q~ likewise, in place
#pragma unroll 4
    for (int it = 0; it < 2048 / KP_THREADS; ++it) {
      const int idx = tid + KP_THREADS * it, R = idx >> 4, c8 = idx & 15, blk = (R & 63) >> 4;
      float f[8], x[8];
      uint4* p = reinterpret_cast<uint4*>(kq + sw_chunk(R, c8, 128));
      unpack8(*p, x);
      ld8(&gamb[blk][8 * c8], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] *= f[e];
      *p = pack8(x);
    }
    to_mma();
    if (warp == 0) {   // W^T = K~^T T''^T (M = 128: the key channels)
      const uint32_t sk = smem_u32(kq), st = smem_u32(sm + KP_G);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_ss_w(tb + KT_INV, desc_mn(sk, 128, ks), desc_k(st, 64, ks), idesc(128, 64, 1, 0), ks > 0);
      mma_commit_w(&bar_t);
    }
    ok = __syncthreads_and(mbar_wait(&bar_t, tph, a.err));
    if (!ok) t_pend = (int)tph;
    tph ^= 1;
    tc_fence_after();
  }
  if (ok) {
    {  // -W^T row tid % 128 (dk index) -> BF16 SwTile(128 x 64); the warpgroups split the 64 columns
      const int hw = warp >> 2;
      float w[32];
      tmem_ld32(taddr(tb, (warp & 3) * 32, KT_INV + 32 * hw), w);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = -w[8 * c + e];
        *reinterpret_cast<uint4*>(sm + KP_G + 16384 + sw_chunk(tid & 127, 4 * hw + c, 128)) = pack8(x);
      }
    }
    fence_async_smem();
    __syncthreads();
    if (tid == 0) {
      bulk_store(kbp + KB_WT, sm + KP_G + 16384, 16384u);
      bulk_store(kbp + KB_QT, kq + 8192, 8192u);              // Q~ panel 0 (rows 64-127 of the tile)
      bulk_store(kbp + KB_QT + 8192, kq + 24576, 8192u);      // Q~ panel 1
      bulk_commit();
    }
  }
  if (tid == 0) {
    bulk_wait_read();   // shared memory must outlive the copies' reads
    if (!ok) {          // error path (bounded waits): no MMA may outlive the CTA's TMEM
#pragma unroll
      for (int v = 0; v < 4; ++v)
        if (vpend & (1 << v)) mbar_drain(&bar_v[v & 1], (uint32_t)(v >> 1));
      if (t_pend >= 0) mbar_drain(&bar_t, (uint32_t)t_pend);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, KT_COLS);
}

// ---------------------------------------------------------------------------
// output: O^T = S^T Q~^T + V_new^T P^T, o = scale O
// ---------------------------------------------------------------------------
constexpr int KO_S = 0, KO_VN = 32768, KO_Q = 49152, KO_AQK = 65536, KO_O = 73728;
constexpr int KO_SMEM = KO_O + 16384;
constexpr int KO_SMEM_ALLOC = KO_SMEM + 1024;

__global__ void __launch_bounds__(128, 2) kda_out_kernel(const __grid_constant__ KdaOutArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_align1024(smem_raw);
  __shared__ uint64_t bar_ld, bar_m;
  __shared__ uint32_t tslot;
  const int c = blockIdx.x / a.HV, hv = blockIdx.x % a.HV;
  const int tid = threadIdx.x, warp = tid >> 5;
  if (*(volatile int*)a.err) return;
  const int tok0 = a.chunk_tok0[c], L = a.chunk_len[c];
  const size_t blk = (size_t)c * a.HV + hv;
  if (warp == 0) tmem_alloc(&tslot, 64);
  if (tid == 0) {
    mbar_init(&bar_ld, 1);
    mbar_init(&bar_m, 1);
    asm volatile("fence.mbarrier_init.release.cluster;");
    mbar_expect_tx(&bar_ld, (uint32_t)(STATE_BYTES + VN_BYTES + 16384 + TILE64_BYTES));
    bulk_load(sm + KO_S, a.tape + blk * STATE_BYTES, STATE_BYTES, &bar_ld);
    bulk_load(sm + KO_VN, a.vn + blk * VN_BYTES, VN_BYTES, &bar_ld);
    const uint8_t* kbp = a.kb + blk * KB_BYTES;
    bulk_load(sm + KO_Q, kbp + KB_QT, 16384u, &bar_ld);
    bulk_load(sm + KO_AQK, kbp + KB_AQK, TILE64_BYTES, &bar_ld);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tslot;
  bool ok = __syncthreads_and(mbar_wait(&bar_ld, 0, a.err));
  bool mma_out = false;
  if (ok) {
    if (warp == 0) {
      const uint32_t s_s = smem_u32(sm + KO_S), s_q = smem_u32(sm + KO_Q), s_vn = smem_u32(sm + KO_VN),
                     s_a = smem_u32(sm + KO_AQK);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_ss_w(tb, desc_k(s_s, 128, ks), desc_k(s_q, 64, ks), idesc(128, 64, 0, 0), ks > 0);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_ss_w(tb, desc_k(s_vn, 128, ks), desc_k(s_a, 64, ks), idesc(128, 64, 0, 0), 1u);
      mma_commit_w(&bar_m);
    }
    mma_out = true;
    ok = __syncthreads_and(mbar_wait(&bar_m, 0, a.err));
    if (ok) mma_out = false;
    tc_fence_after();
  }
  if (ok) {
    uint8_t* ost = sm + KO_O;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float x[32];
      tmem_ld32(taddr(tb, warp * 32, h * 32), x);
#pragma unroll
      for (int e = 0; e < 32; ++e)
        *reinterpret_cast<__nv_bfloat16*>(ost + sw_off(h * 32 + e, tid, 64)) = __float2bfloat16_rn(a.scale * x[e]);
    }
    fence_async_smem();
    __syncthreads();
    if (L < CH) {   // ragged last chunk of a document: its own rows only
      for (int idx = tid; idx < L * 16; idx += 128) {
        const int r = idx >> 4, c8 = idx & 15;
        *reinterpret_cast<uint4*>(a.o + ((size_t)(tok0 + r) * a.HV + hv) * D + c8 * 8) =
            *reinterpret_cast<const uint4*>(ost + sw_chunk(r, c8, 64));
      }
    } else if (tid == 0) {
      tma_store_3d(&a.to, ost, 0, hv, tok0);
      tma_store_3d(&a.to, ost + 8192, 64, hv, tok0);
      bulk_commit();
    }
  }
  if (tid == 0) {
    bulk_wait_all();
    if (!ok) {
      if (mma_out) mbar_drain(&bar_m, 0);
      mbar_drain(&bar_ld, 0);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, 64);
}

void setup_kda_attrs() {
  cudaFuncSetAttribute(kda_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, KP_SMEM_ALLOC);
  cudaFuncSetAttribute(kda_out_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, KO_SMEM_ALLOC);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static size_t kda_align(size_t x, size_t al) { return (x + al - 1) / al * al; }

// The KDA layouts on top of the common plan (tables and segment plan): workspace = tables, the
// per-chunk blocks (of a forward without a full saved set, and of a replay-form backward), the
// split-walk states, the forward's own tape and V_new^T when no saved set is given; then the
// backward's tapes.  Saved set = header, state tape, M_seg, V_new^T and, in the full form
// (prob->saved_form == GDN_SAVED_FULL, header form 3), the per-chunk blocks; the replay form
// (header form 2) leaves the blocks out and the backward forms them again.
gdn_status make_kda_plan(const gdn_problem* p, const int32_t* cu, Plan* P) {
  gdn_status st = make_plan(p, cu, P);
  if (st != GDN_OK) return st;
  const bool full = p->saved_form == GDN_SAVED_FULL;
  P->form = full ? 3 : 2;
  const size_t units = (size_t)P->NC * P->HV;
  const size_t st_f32 = (size_t)P->nsplit * P->HV * STATE_F32 * 4;
  size_t off = kda_align(P->o_tables[18], 1024);
  P->o_cb = off;
  off += units * KB_BYTES;
  P->o_bend = off;
  off += st_f32;
  P->o_sinit = off;
  off += st_f32;
  P->o_mend_ws = off;
  off += st_f32;
  P->o_ktape = off;
  off += units * STATE_BYTES;
  P->o_kvn = off;
  off += units * VN_BYTES;
  P->ws_fwd = off;
  off = P->o_ktape;   // the backward reuses the forward-only tape space
  P->o_dtape = off;
  off += units * STATE_BYTES;
  P->o_dvn = off;
  off += units * VN_BYTES;
  P->o_dbend = off;
  off += st_f32;
  P->o_dsinit = off;
  off += st_f32;
  P->o_vnb = 0;
  P->ws_bwd = std::max(off, P->ws_fwd);
  P->s_tape = SAVED_HEADER;
  P->s_mseg = P->s_tape + units * STATE_BYTES;
  P->s_vn = kda_align(P->s_mseg + st_f32, 1024);
  P->s_cb = full ? kda_align(P->s_vn + units * VN_BYTES, 1024) : P->s_vn;
  P->saved_bytes = full ? P->s_cb + units * KB_BYTES : P->s_vn + units * VN_BYTES;
  return GDN_OK;
}

void launch_kda_prep(const KdaPrepArgs& a, int NC, cudaStream_t s) {
  if (NC <= 0) return;
  prof_begin(K_KDA_PREP, s);
  kda_prep_kernel<<<NC * a.HV, KP_THREADS, KP_SMEM_ALLOC, s>>>(a);
  prof_end(K_KDA_PREP, s);
}

gdn_status run_kda_prep(const Plan& P, const gdn_problem* p, const void* q, const void* k, const float* g,
                        const float* beta, uint8_t* kb, uint8_t* ws, cudaStream_t s) {
  Tables t = tables_at(P, ws);
  KdaPrepArgs pa;
  memset(&pa, 0, sizeof(pa));
  if (!make_tmap(&pa.tq, q, P.T, P.H) || !make_tmap(&pa.tk, k, P.T, P.H) || !make_tmap_g(&pa.tg, g, P.T, P.HV))
    return GDN_ERR_CUDA;
  pa.g = g;
  pa.beta = beta;
  pa.chunk_tok0 = t.chunk_tok0;
  pa.chunk_len = t.chunk_len;
  pa.kb = kb;
  pa.H = P.H;
  pa.HV = P.HV;
  pa.G = P.G;
  pa.l2norm = p->l2norm ? 1 : 0;
  pa.err = reinterpret_cast<int*>(ws);
  launch_kda_prep(pa, P.NC, s);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

static gdn_status run_kda_fwd(const Plan& P, const gdn_problem* p, const void* q, const void* k, const void* v,
                              const float* g, const float* beta, const int32_t* cu_dev, void* o, void* saved,
                              uint8_t* ws, cudaStream_t s) {
  gdn_status st = run_tables(P, p, cu_dev, ws, saved, s);
  if (st != GDN_OK) return st;
  if (P.NC == 0) return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
  uint8_t* sv = static_cast<uint8_t*>(saved);
  // the per-chunk blocks: into the full-form saved set for the backward, else the workspace
  uint8_t* kb = sv && P.form == 3 ? sv + P.s_cb : ws + P.o_cb;
  st = run_kda_prep(P, p, q, k, g, beta, kb, ws, s);
  if (st != GDN_OK) return st;
  Tables t = tables_at(P, ws);
  ScanArgs sa;
  memset(&sa, 0, sizeof(sa));
  if (!make_tmap(&sa.tq, q, P.T, P.H) || !make_tmap(&sa.tk, k, P.T, P.H) || !make_tmap(&sa.tv, v, P.T, P.HV))
    return GDN_ERR_CUDA;
  sa.kda = 1;
  sa.cb = kb;
  sa.chunk_tok0 = t.chunk_tok0;
  sa.chunk_len = t.chunk_len;
  sa.seg_c0 = t.seg_c0;
  sa.seg_c1 = t.seg_c1;
  sa.seg_idx = t.seg_idx;
  sa.seg_split = t.seg_split;
  sa.split_seg = t.split_seg;
  sa.walk_seg = t.fwalk_seg;
  sa.H = P.H;
  sa.HV = P.HV;
  sa.G = P.G;
  sa.nsplit = P.nsplit;
  sa.scale = p->scale;
  sa.bend = reinterpret_cast<float*>(ws + P.o_bend);
  sa.s_init = reinterpret_cast<float*>(ws + P.o_sinit);
  sa.mend = sv ? reinterpret_cast<float*>(sv + P.s_mseg) : reinterpret_cast<float*>(ws + P.o_mend_ws);
  sa.seg_doc = t.seg_doc;
  sa.seg_offsets = t.seg_offsets;
  sa.err = reinterpret_cast<int*>(ws);
  sa.tape = sv ? sv + P.s_tape : ws + P.o_ktape;
  sa.vn = sv ? sv + P.s_vn : ws + P.o_kvn;
  sa.o = nullptr;
  if (P.nsplit > 0) {
    sa.walk = 1;
    launch_fwd_scan(sa, 2 * P.nsplit * P.HV, s);
    MergeArgs ma;
    ma.sdoc_first = t.sdoc_first;
    ma.bend = sa.bend;
    ma.mend = sa.mend;
    ma.s_init = const_cast<float*>(sa.s_init);
    ma.HV = P.HV;
    ma.err = sa.err;
    launch_merge(ma, P.nsdoc, s);
  }
  sa.walk = 0;
  launch_fwd_scan(sa, (P.NSEG - P.nsdoc) * P.HV, s);
  KdaOutArgs oa;
  memset(&oa, 0, sizeof(oa));
  if (!make_tmap(&oa.to, o, P.T, P.HV)) return GDN_ERR_CUDA;
  oa.tape = sa.tape;
  oa.vn = sa.vn;
  oa.kb = kb;
  oa.chunk_tok0 = t.chunk_tok0;
  oa.chunk_len = t.chunk_len;
  oa.o = static_cast<__nv_bfloat16*>(o);
  oa.HV = P.HV;
  oa.scale = p->scale;
  oa.err = sa.err;
  prof_begin(K_KDA_OUT, s);
  kda_out_kernel<<<P.NC * P.HV, 128, KO_SMEM_ALLOC, s>>>(oa);
  prof_end(K_KDA_OUT, s);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace gdn

using namespace gdn;

extern "C" {

gdn_status gdn_kda_saved_bytes(const gdn_problem* prob, const int32_t* cu_host, size_t* saved_bytes,
                               size_t* workspace_bytes) {
  Plan P;
  gdn_status st = make_kda_plan(prob, cu_host, &P);
  if (st != GDN_OK) return st;
  if (saved_bytes) *saved_bytes = P.saved_bytes;
  if (workspace_bytes) *workspace_bytes = P.ws_bwd;
  return GDN_OK;
}

gdn_status gdn_kda_fwd(const gdn_problem* prob, const void* q, const void* k, const void* v, const float* g,
                       const float* beta, const int32_t* cu_dev, const int32_t* cu_host, void* o, void* saved,
                       void* workspace, size_t ws_bytes, struct CUstream_st* stream) {
  Plan P;
  gdn_status st = make_kda_plan(prob, cu_host, &P);
  if (st != GDN_OK) return st;
  if (!cu_dev || !workspace || !o) return GDN_ERR_INVALID_ARG;
  if (P.T > 0 && (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(beta) ||
                  !aligned16(o)))
    return GDN_ERR_INVALID_ARG;
  if (!aligned16(workspace) || (saved && !aligned16(saved))) return GDN_ERR_INVALID_ARG;
  if (ws_bytes < P.ws_fwd) return GDN_ERR_WORKSPACE_TOO_SMALL;
  if (!device_setup()) return GDN_ERR_CUDA;
  return run_kda_fwd(P, prob, q, k, v, g, beta, cu_dev, o, saved, static_cast<uint8_t*>(workspace), stream);
}

}  // extern "C"
