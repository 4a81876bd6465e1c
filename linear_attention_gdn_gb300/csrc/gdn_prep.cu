// gdn_prep.cu -- per (chunk, value head) preparation of the chunked GDN form.
//
// For one 64-token chunk and one value head h (q/k head j = h / G):
//   rk_r, rq_r   1/sqrt(x.x + 1e-6) of k_r, q_r (or 1 with l2norm off)
//   KK^T, QK^T   one tcgen05 MMA on the stacked [K; Q] tile (M = 128)
//   G_r   = sum_{i<=r} g_i        (chunk-local cumulative gate, the pages'
//                                  "GLM prep" gate prefix rows)
//   A     = strict_tril(beta_r e^{G_r - G_j} k^_r.k^_j)        ("Akk")
//   T     = (I + A)^-1
//   Aqk   = tril(e^{G_r - G_j} q^_r.k^_j)                       ("Aqk")
//   T'    = T diag(beta gamma rk),  T'' = T diag(beta)
// so that W = T diag(beta gamma) K^ = T' K and U = T diag(beta) V = T'' V
// (the WY program's w and u; "feat(cake_gdn_kcp) ... #8172" page, commit
// notes on the intra / WY / GLM-prep programs; "#8542" page, save-set table).
//
// The inverse of the unit lower-triangular I + A is FP32 and blocked by
// 16 x 16: the four diagonal blocks by forward substitution (one lane per
// column), then the three block diagonals below them, each block from the
// finished ones (T_ij = -T_ii sum_k A_ik T_kj), on 64 lanes.
//
// Gate factors: e^{G_r - G_j} for j <= r is taken as the product
// e^{G_r - G_0} e^{G_0 - G_j} of per-token factors when the chunk's gate range
// G_0 - G_{L-1} is small enough for FP32 (below 2^100 in log2 units), and as
// one exp2f per element otherwise.
#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_prof.h"

namespace gdn {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kSafeRange = 100.f;                  // log2 units
constexpr int PR_THREADS = 128;
constexpr int PR_BLOCKS_PER_SM = 5;
constexpr int PR_ALD = 68;                           // row pitch of the FP32 A^T / T array (floats)
// Shared memory (bytes, 1024-aligned tiles).  The [K; Q] tile is dead once the
// KK^T / QK^T MMA has completed; its space then holds the FP32 array, the Aqk
// staging tile and the scalars, and finally the T' and T'' tiles (written over
// the FP32 array after every thread has read its part of T into registers).
constexpr int PR_KQ = 0;                             // [K; Q] SwTile(128 x 128), 32 KB
constexpr int PR_S = 0;                              // FP32 S[64][PR_ALD]
constexpr int PR_TP = 0;                             // T', then T'' (contiguous, one bulk store)
constexpr int PR_AQ = 17408;                         // Aqk tile
constexpr int PR_SC = PR_AQ + TILE64_BYTES;          // scalars
constexpr int PR_T = PR_SC + CB_SCAL_BYTES;          // T tile
constexpr int PR_SMEM = PR_T + TILE64_BYTES;
constexpr int PR_SMEM_ALLOC = PR_SMEM + 1024;
static_assert(64 * PR_ALD * 4 <= PR_AQ && 2 * TILE64_BYTES <= PR_AQ, "FP32 array and T', T'' fit below Aqk");
static_assert(PR_AQ % 1024 == 0 && PR_T % 1024 == 0, "swizzled tiles are 1024-aligned");
static_assert(PR_SMEM >= 32768, "the [K; Q] tile fits");

// One block diagonal d of T = (I + A)^-1 (16 x 16 blocks, 64 lanes of one value
// head): T_ij = -T_ii p with p = sum_{k=j}^{i-1} A_ik T_kj, for the 4 - d blocks
// (i, j = i - d).  S holds A[r][c] (c < r) at S[c][r] and T[r][c] (c <= r) at
// S[r][c]; the upper triangles of the diagonal blocks hold zeros (their A
// entries are dead once the diagonal blocks are inverted).  The (4 - d) * 16
// columns are spread over 64 lanes as G = 1, 2, 4 lanes per column; lane g of
// a column accumulates rows [16g/G, 16(g+1)/G) of p over the whole k range,
// the G lanes exchange their rows by shuffles, and each then forms its rows
// of T_ij.
template <int DL>
__device__ __forceinline__ void offdiag_level(float* Sm, int l) {
  constexpr int G = DL == 1 ? 1 : (DL == 2 ? 2 : 4);
  constexpr int R = 16 / G;                 // rows of p per lane
  constexpr int NCOL = (4 - DL) * 16;       // columns on this block diagonal
  const int cl = l / G, g = l % G;
  const bool act = cl < NCOL;
  const int jb = act ? cl >> 4 : 0, oi = 16 * (jb + DL), c = 16 * jb + (cl & 15);
  float p[R];
#pragma unroll
  for (int r = 0; r < R; ++r) p[r] = 0.f;
  if (act) {
#pragma unroll 4
    for (int t = 16 * jb; t < oi; ++t) {
      const float tv = Sm[t * PR_ALD + c];   // T[t][c] (zero above the diagonal of the diagonal block)
#pragma unroll
      for (int q = 0; q < R / 4; ++q) {                       // A[oi + r][t] = S[t][oi + r]
        const float4 av = *reinterpret_cast<const float4*>(Sm + t * PR_ALD + oi + g * R + 4 * q);
        fma2(p[4 * q + 0], p[4 * q + 1], av.x, av.y, tv);
        fma2(p[4 * q + 2], p[4 * q + 3], av.z, av.w, tv);
      }
    }
  }
  float pf[16];   // the whole p of this column, gathered from the G lanes
  if constexpr (G == 1) {
#pragma unroll
    for (int r = 0; r < 16; ++r) pf[r] = p[r];
  } else {
#pragma unroll
    for (int og = 0; og < G; ++og)
#pragma unroll
      for (int r = 0; r < R; ++r) pf[og * R + r] = __shfl_sync(0xffffffffu, p[r], (l & 31 & ~(G - 1)) + og);
  }
  if (act) {
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {   // T_ij[r][c] = -sum_{s <= r} T_ii[r][s] p[s]
      const int r = g * R + rr;
      float acc = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        // T_ii is zero above its diagonal: the terms s > r are skipped where r is known at compile
        // time (G = 1) and otherwise add zero
        if (G == 1 && 4 * q > rr) continue;
        const float4 tv4 = *reinterpret_cast<const float4*>(Sm + (oi + r) * PR_ALD + oi + 4 * q);
        acc = fmaf(tv4.x, pf[4 * q + 0], acc);
        if (G > 1 || 4 * q + 1 <= rr) acc = fmaf(tv4.y, pf[4 * q + 1], acc);
        if (G > 1 || 4 * q + 2 <= rr) acc = fmaf(tv4.z, pf[4 * q + 2], acc);
        if (G > 1 || 4 * q + 3 <= rr) acc = fmaf(tv4.w, pf[4 * q + 3], acc);
      }
      Sm[(oi + r) * PR_ALD + c] = -acc;
    }
  }
}

// One CTA per (chunk, q/k head): the tile load, the norms and the KK^T / QK^T
// MMA once, then the group's value heads one after another on that product
// (each head's stores drain while the next one is prepared).  Five CTAs share
// an SM, so the serial phases of one (tile load, MMA, inverse) run under the
// others.
__global__ void __launch_bounds__(PR_THREADS, PR_BLOCKS_PER_SM) prep_kernel(const __grid_constant__ PrepArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_align1024(smem_raw);
  __shared__ __align__(16) float rq[CH], rk[CH];
  __shared__ __align__(16) float Gs[CH], bs[CH], eGr[CH], eGi[CH];
  __shared__ __align__(16) float cf[CH];   // rk_j e^{G_0 - G_j}: the column factor of A and Aqk
  __shared__ __align__(16) float ca[CH];   // beta_r rk_r e^{G_r - G_0}: the row factor of A
  __shared__ __align__(16) float pcol[CH]; // beta_c e^{G_c} rk_c: the column factor of T'
  __shared__ int safe;
  __shared__ uint64_t bar, bar_kq;
  __shared__ uint32_t tslot;
  const int c = blockIdx.x / a.H, j = blockIdx.x % a.H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = tid;                   // TMEM lane = row of [KK^T; QK^T]
  if (*(volatile int*)a.err) return;
  const int tok0 = a.chunk_tok0[c], L = a.chunk_len[c];

  // ---- [K; Q] tile by TMA: rows 0..63 = k tokens, 64..127 = q tokens (SwTile(128 x 128))
  if (warp == 0) tmem_alloc(&tslot, 64);
  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_init(&bar_kq, 1);
    asm volatile("fence.mbarrier_init.release.cluster;");
    mbar_expect_tx(&bar_kq, 32768u);
    tma_load_3d(sm + PR_KQ, &a.tk, 0, j, tok0, &bar_kq);
    tma_load_3d(sm + PR_KQ + 8192, &a.tq, 0, j, tok0, &bar_kq);
    tma_load_3d(sm + PR_KQ + 16384, &a.tk, 64, j, tok0, &bar_kq);
    tma_load_3d(sm + PR_KQ + 24576, &a.tq, 64, j, tok0, &bar_kq);
  }
  // the gates of a value head (warp 3: tokens 2 lane, 2 lane + 1); the first head's are requested
  // while the tile lands, each later head's while the one before it is prepared
  float gn0 = 0.f, gn1 = 0.f, bn0 = 0.f, bn1 = 0.f;
  auto load_gates = [&](int hv_) {
    const int r0 = 2 * lane, r1 = r0 + 1;
    gn0 = gn1 = bn0 = bn1 = 0.f;
    if (r0 < L) {
      gn0 = a.g[(size_t)(tok0 + r0) * a.HV + hv_];
      bn0 = a.beta[(size_t)(tok0 + r0) * a.HV + hv_];
    }
    if (r1 < L) {
      gn1 = a.g[(size_t)(tok0 + r1) * a.HV + hv_];
      bn1 = a.beta[(size_t)(tok0 + r1) * a.HV + hv_];
    }
  };
  if (warp == 3) load_gates(j * a.G);
  __syncthreads();
  if (!__syncthreads_and(mbar_wait(&bar_kq, 0, a.err))) {
    if (warp == 0) tmem_dealloc(tslot, 64);
    return;
  }
  if (L < CH) {   // zero the rows past the document end (they hold the next document)
    for (int idx = tid; idx < (CH - L) * 32; idx += PR_THREADS) {
      const int t = idx >> 5, half = (idx >> 4) & 1, c8 = idx & 15;
      *reinterpret_cast<uint4*>(sm + PR_KQ + sw_chunk(half * 64 + L + t, c8, 128)) = make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();
  }
  {  // L2 norm of row `row` of the tile: four partial sums of 32 elements (each the sum of its even-
     // and its odd-element chain, the two run as paired FMAs), combined as (p0 + p1) + (p2 + p3)
    float pr[4];
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) {
      float se = 0.f, so = 0.f;
#pragma unroll
      for (int c8 = qq * 4; c8 < qq * 4 + 4; ++c8) {
        const uint4 val = *reinterpret_cast<const uint4*>(sm + PR_KQ + sw_chunk(row, c8, 128));
        const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&val);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(h2[e]);
          fma2v(se, so, f.x, f.y, f.x, f.y);
        }
      }
      pr[qq] = se + so;
    }
    const float ss = (pr[0] + pr[1]) + (pr[2] + pr[3]);
    const float rn = a.l2norm ? 1.0f / sqrtf(ss + 1e-6f) : 1.0f;
    if (row < 64) rk[row] = rn;
    else rq[row - 64] = rn;
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tslot;
  if (tid == 0) {
    const uint32_t sm_a = smem_u32(sm + PR_KQ);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
      mma_ss(tb, desc_k(sm_a, 128, ks), desc_k(sm_a, 128, ks), idesc(128, 64, 0, 0), ks > 0);
    mma_commit(&bar);
  }
  // ---- the value heads of the group, one after another, on the one KK^T / QK^T
  bool ok = true;
  for (int hh = 0; hh < a.G; ++hh) {
    const int hv = j * a.G + hh;
    if (warp == 3) {   // ---- gates (log2 units)
      const int r0 = 2 * lane, r1 = r0 + 1;
      const float g0 = gn0, g1 = gn1, b0 = bn0, b1 = bn1;
      if (hh + 1 < a.G) load_gates(hv + 1);
      float s = g0 + g1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += y;
      }
      const float ex = s - (g0 + g1);
      const float G0v = (ex + g0) * kLog2e, G1v = (ex + g0 + g1) * kLog2e;
      Gs[r0] = G0v;
      Gs[r1] = G1v;
      bs[r0] = b0;
      bs[r1] = b1;
      const float Gfirst = __shfl_sync(0xffffffffu, G0v, 0);
      const float Glast = __shfl_sync(0xffffffffu, G1v, 31);   // = G_{L-1} (gates past L are 0)
      eGr[r0] = exp2f(G0v - Gfirst);
      eGr[r1] = exp2f(G1v - Gfirst);
      const bool sf = (Gfirst - Glast) < kSafeRange;
      eGi[r0] = sf ? exp2f(Gfirst - G0v) : 0.f;
      eGi[r1] = sf ? exp2f(Gfirst - G1v) : 0.f;
      cf[r0] = rk[r0] * eGi[r0];
      cf[r1] = rk[r1] * eGi[r1];
      ca[r0] = b0 * rk[r0] * eGr[r0];
      ca[r1] = b1 * rk[r1] * eGr[r1];
      pcol[r0] = b0 * exp2f(G0v) * rk[r0];
      pcol[r1] = b1 * exp2f(G1v) * rk[r1];
      if (lane == 0) safe = sf;
    }
    // (the first head waits for the KK^T / QK^T MMA, every later one for the previous head's copies
    // to have read the staging buffers it rewrites)
    if (hh > 0 && tid == 0) bulk_wait_read();
    ok = __syncthreads_and((hh > 0 || mbar_wait(&bar, 0, a.err)) && ok);
    tc_fence_after();
    float* Sm = reinterpret_cast<float*>(sm + PR_S);
    if (ok) {
      // ---- A^T (FP32, from the rows of KK^T), Aqk tile (rows of QK^T), scalars
      const bool sf = safe;
#pragma unroll 1
      for (int cb0 = 0; cb0 < CH; cb0 += 32) {
        float kq[32];   // row `row` of [KK^T; QK^T], columns cb0 .. cb0 + 31
        tmem_ld32(taddr(tb, warp * 32, cb0), kq);
        if (row < 64) {
          // KK^T is symmetric, so the thread holding its row c writes row c of the transposed A:
          // S[c][r] = A[r][c] = (beta_r rk_r e^{G_r - G_0}) (rk_c e^{G_0 - G_c}) KK[c][r] for c < r < L
          const int cc = row;
          if (sf) {
            const float pc = cf[cc];
#pragma unroll
            for (int e4 = 0; e4 < 8; ++e4) {
              const int r0 = cb0 + 4 * e4;
              const float4 f = *reinterpret_cast<const float4*>(&ca[r0]);
              float4 v;
              v.x = (r0 + 0 > cc && r0 + 0 < L) ? pc * f.x * kq[4 * e4 + 0] : 0.f;
              v.y = (r0 + 1 > cc && r0 + 1 < L) ? pc * f.y * kq[4 * e4 + 1] : 0.f;
              v.z = (r0 + 2 > cc && r0 + 2 < L) ? pc * f.z * kq[4 * e4 + 2] : 0.f;
              v.w = (r0 + 3 > cc && r0 + 3 < L) ? pc * f.w * kq[4 * e4 + 3] : 0.f;
              *reinterpret_cast<float4*>(Sm + cc * PR_ALD + r0) = v;
            }
          } else {
            const float pc = rk[cc];
#pragma unroll
            for (int e4 = 0; e4 < 8; ++e4) {
              const int r0 = cb0 + 4 * e4;
              float x[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const int r = r0 + q;
                x[q] = (r > cc && r < L) ? bs[r] * rk[r] * pc * exp2f(Gs[r] - Gs[cc]) * kq[4 * e4 + q] : 0.f;
              }
              *reinterpret_cast<float4*>(Sm + cc * PR_ALD + r0) = make_float4(x[0], x[1], x[2], x[3]);
            }
          }
        } else {
          const int r = row - 64;
          const float pr = rq[r] * (sf ? eGr[r] : 1.f);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            float x[8];
            if (sf) {
              const float4 fa = *reinterpret_cast<const float4*>(&cf[cb0 + q4 * 8]);
              const float4 fb = *reinterpret_cast<const float4*>(&cf[cb0 + q4 * 8 + 4]);
              const float fv[8] = {fa.x, fa.y, fa.z, fa.w, fb.x, fb.y, fb.z, fb.w};
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const int jj = cb0 + q4 * 8 + e;
                x[e] = (jj <= r && r < L) ? pr * fv[e] * kq[q4 * 8 + e] : 0.f;
              }
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const int jj = cb0 + q4 * 8 + e;
                x[e] = (jj <= r && r < L) ? pr * rk[jj] * exp2f(Gs[r] - Gs[jj]) * kq[q4 * 8 + e] : 0.f;
              }
            }
            uint4 w;
            w.x = pack_bf16(x[0], x[1]);
            w.y = pack_bf16(x[2], x[3]);
            w.z = pack_bf16(x[4], x[5]);
            w.w = pack_bf16(x[6], x[7]);
            *reinterpret_cast<uint4*>(sm + PR_AQ + sw_chunk(r, (cb0 >> 3) + q4, 64)) = w;
          }
        }
      }
      if (row < 64) {
        const int r = row;
        float* sc = reinterpret_cast<float*>(sm + PR_SC);
        const float GL = Gs[L - 1];
        sc[r] = r < L ? a.scale * exp2f(Gs[r]) * rq[r] : 0.f;
        sc[64 + r] = r < L ? exp2f(GL - Gs[r]) * rk[r] : 0.f;
        if (r == 0) {
          sc[128] = exp2f(GL);
          reinterpret_cast<int*>(sc)[129] = L;
        }
        // ---- T = (I + A)^-1 by 16 x 16 blocks on warps 0-1 (64 lanes).  One FP32 array S[p][q]
        // (pitch PR_ALD) holds A[r][c] (c < r) at S[c][r] and T[r][c] (c <= r) at S[r][c].
        //   diagonal blocks  T_bb = (I + A_bb)^-1, forward substitution, lane = column
        //   block diagonal d T_ij = -T_ii sum_{k=j}^{i-1} A_ik T_kj (i - j = d), lane = (block, column)
        const int l = row;
        named_bar(1, 64);
        {  // diagonal blocks
          const int o = 16 * (l >> 4), cc = l & 15;
          float x[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) x[i] = (i == cc) ? 1.f : 0.f;
#pragma unroll
          for (int jq = 0; jq < 15; ++jq) {
            const float xj = x[jq];
#pragma unroll
            for (int g4 = (jq + 1) >> 2; g4 < 4; ++g4) {
              const float4 av = *reinterpret_cast<const float4*>(Sm + (o + jq) * PR_ALD + o + 4 * g4);
              // (pairs whose both rows lie below jq go as one paired FMA)
              if (4 * g4 + 0 > jq) fma2(x[4 * g4 + 0], x[4 * g4 + 1], -av.x, -av.y, xj);
              else if (4 * g4 + 1 > jq) x[4 * g4 + 1] = fmaf(-av.y, xj, x[4 * g4 + 1]);
              if (4 * g4 + 2 > jq) fma2(x[4 * g4 + 2], x[4 * g4 + 3], -av.z, -av.w, xj);
              else if (4 * g4 + 3 > jq) x[4 * g4 + 3] = fmaf(-av.w, xj, x[4 * g4 + 3]);
            }
          }
          __syncwarp();   // every lane of the block has read its A entries
#pragma unroll
          for (int i = 0; i < 16; ++i) Sm[(o + i) * PR_ALD + o + cc] = x[i];   // x[i] = 0 above the diagonal
        }
        named_bar(1, 64);
        // off-diagonal blocks, one block diagonal d at a time (then T_ij is complete for i - j = d)
        offdiag_level<1>(Sm, l);
        named_bar(1, 64);
        offdiag_level<2>(Sm, l);
        named_bar(1, 64);
        offdiag_level<3>(Sm, l);
      }
    }
    __syncthreads();   // T complete, Aqk and the scalars staged
    if (ok) {
      // ---- the T', T'', T tiles, all 128 threads: 16-byte chunks (row i, columns 8 c8 .. 8 c8 + 7);
      // first every thread reads its four chunks of T, then (after a barrier) overwrites the array
      float tv[4][8];
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        const int item = tid + PR_THREADS * it, i = item >> 3, c8 = item & 7;
        const float4 u0 = *reinterpret_cast<const float4*>(Sm + i * PR_ALD + 8 * c8);
        const float4 u1 = *reinterpret_cast<const float4*>(Sm + i * PR_ALD + 8 * c8 + 4);
        const float u[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) tv[it][e] = 8 * c8 + e <= i ? u[e] : 0.f;   // above the diagonal: A^T
      }
      __syncthreads();
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        const int item = tid + PR_THREADS * it, i = item >> 3, c8 = item & 7;
        const float4 p0 = *reinterpret_cast<const float4*>(pcol + 8 * c8);
        const float4 p1 = *reinterpret_cast<const float4*>(pcol + 8 * c8 + 4);
        const float4 q0 = *reinterpret_cast<const float4*>(bs + 8 * c8);
        const float4 q1 = *reinterpret_cast<const float4*>(bs + 8 * c8 + 4);
        const float pc[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
        const float bc[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        uint4 w1, w2, w3;
        w1.x = pack_bf16(tv[it][0] * pc[0], tv[it][1] * pc[1]);
        w1.y = pack_bf16(tv[it][2] * pc[2], tv[it][3] * pc[3]);
        w1.z = pack_bf16(tv[it][4] * pc[4], tv[it][5] * pc[5]);
        w1.w = pack_bf16(tv[it][6] * pc[6], tv[it][7] * pc[7]);
        w2.x = pack_bf16(tv[it][0] * bc[0], tv[it][1] * bc[1]);
        w2.y = pack_bf16(tv[it][2] * bc[2], tv[it][3] * bc[3]);
        w2.z = pack_bf16(tv[it][4] * bc[4], tv[it][5] * bc[5]);
        w2.w = pack_bf16(tv[it][6] * bc[6], tv[it][7] * bc[7]);
        w3.x = pack_bf16(tv[it][0], tv[it][1]);
        w3.y = pack_bf16(tv[it][2], tv[it][3]);
        w3.z = pack_bf16(tv[it][4], tv[it][5]);
        w3.w = pack_bf16(tv[it][6], tv[it][7]);
        const uint32_t off = sw_chunk(i, c8, 64);
        *reinterpret_cast<uint4*>(sm + PR_TP + off) = w1;                  // T'
        *reinterpret_cast<uint4*>(sm + PR_TP + TILE64_BYTES + off) = w2;   // T''
        if (a.write_T) *reinterpret_cast<uint4*>(sm + PR_T + off) = w3;     // T
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
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, 64);
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
