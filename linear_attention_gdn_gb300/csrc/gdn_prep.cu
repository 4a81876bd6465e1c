// gdn_prep.cu -- per (chunk, q/k head) preparation of the chunked GDN form.
//
// For one 64-token chunk and one q/k head (serving its G = HV/H value heads):
//   rk_r, rq_r   1/sqrt(x.x + 1e-6) of k_r, q_r (or 1 with l2norm off)
//   KK^T, QK^T   one tcgen05 MMA on the stacked [K; Q] tile (M = 128)
// and for every value head of the group (its gate g and beta):
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
// The inverse of the unit lower-triangular I + A is FP32 forward substitution
// in its right-looking form, one lane per column: lane c keeps column c of T
// in registers and, for j = 0..62, subtracts A[i][j] x_j from every later row
// i.  All lanes run the same unrolled instruction stream (a lane whose column
// starts after j just multiplies zeros), the A column for step j is a float4
// broadcast from shared memory, and the FMAs of one step are independent.
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
constexpr int PR_THREADS = 256;
constexpr int PR_GR = 3;                             // value heads per round (a warp pair each)
constexpr int PR_ALD = 68;                           // row pitch of the transposed A (floats)
constexpr int PR_VH = 24576;                         // per value head: A^T (17408 B), then T', T'', T tiles
constexpr int PR_AQ = PR_GR * PR_VH;                 // Aqk staging tiles, 8 KB each
constexpr int PR_SC = PR_AQ + PR_GR * TILE64_BYTES;  // scalar staging, 1 KB each
constexpr int PR_SMEM = PR_SC + PR_GR * CB_SCAL_BYTES;
constexpr int PR_SMEM_ALLOC = PR_SMEM + 1024;
static_assert(PR_VH >= 64 * PR_ALD * 4 && PR_VH >= 3 * TILE64_BYTES, "value-head region");
static_assert(PR_SMEM >= 32768, "the [K;Q] tile reuses the front of shared memory");


// One block diagonal d of T = (I + A)^-1 (16 x 16 blocks, 64 lanes of one value
// head): T_ij = -T_ii p with p = sum_{k=j}^{i-1} A_ik T_kj, for the 4 - d blocks
// (i, j = i - d).  S holds A[r][c] (c < r) at S[c][r] and T[r][c] (c <= r) at
// S[r][c].  The (4 - d) * 16 columns are spread over 64 lanes as G = 1, 2, 4
// lanes per column; lane g of a column accumulates rows [16g/G, 16(g+1)/G) of
// p over the whole k range, the G lanes exchange their rows by shuffles, and
// each then forms its rows of T_ij.
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
      const float tv = t >= c ? Sm[t * PR_ALD + c] : 0.f;   // T[t][c]
#pragma unroll
      for (int q = 0; q < R / 4; ++q) {                       // A[oi + r][t] = S[t][oi + r]
        const float4 av = *reinterpret_cast<const float4*>(Sm + t * PR_ALD + oi + g * R + 4 * q);
        p[4 * q + 0] = fmaf(av.x, tv, p[4 * q + 0]);
        p[4 * q + 1] = fmaf(av.y, tv, p[4 * q + 1]);
        p[4 * q + 2] = fmaf(av.z, tv, p[4 * q + 2]);
        p[4 * q + 3] = fmaf(av.w, tv, p[4 * q + 3]);
      }
    }
  }
  float pf[16];   // the whole p of this column, gathered from the G lanes
#pragma unroll
  for (int og = 0; og < G; ++og)
#pragma unroll
    for (int r = 0; r < R; ++r) pf[og * R + r] = __shfl_sync(0xffffffffu, p[r], (l & 31 & ~(G - 1)) + og);
  if (act) {
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {   // T_ij[r][c] = -sum_{s <= r} T_ii[r][s] p[s]
      const int r = g * R + rr;
      float acc = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 tv4 = *reinterpret_cast<const float4*>(Sm + (oi + r) * PR_ALD + oi + 4 * q);
        acc = 4 * q + 0 <= r ? fmaf(tv4.x, pf[4 * q + 0], acc) : acc;
        acc = 4 * q + 1 <= r ? fmaf(tv4.y, pf[4 * q + 1], acc) : acc;
        acc = 4 * q + 2 <= r ? fmaf(tv4.z, pf[4 * q + 2], acc) : acc;
        acc = 4 * q + 3 <= r ? fmaf(tv4.w, pf[4 * q + 3], acc) : acc;
      }
      Sm[(oi + r) * PR_ALD + c] = -acc;
    }
  }
}

__global__ void __launch_bounds__(PR_THREADS, 2) prep_kernel(const __grid_constant__ PrepArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_align1024(smem_raw);
  __shared__ float rq[CH], rk[CH];
  __shared__ float Gs[PR_GR][CH], bs[PR_GR][CH], eGr[PR_GR][CH], eGi[PR_GR][CH];
  __shared__ __align__(16) float cf[PR_GR][CH];   // rk_j e^{G_0 - G_j}: the column factor of A and Aqk
  __shared__ __align__(16) float ca[PR_GR][CH];   // beta_r rk_r e^{G_r - G_0}: the row factor of A
  __shared__ int safe[PR_GR];
  __shared__ uint64_t bar, bar_kq;
  __shared__ uint32_t tslot;
  const int c = blockIdx.x, j = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wg = tid >> 7, w4 = warp & 3;
  const int row = w4 * 32 + lane;        // TMEM lane = row of [KK^T; QK^T]
  const int cb0 = wg * 32;               // this thread's 32 columns
  if (*(volatile int*)a.err) return;
  const int tok0 = a.chunk_tok0[c], L = a.chunk_len[c];

  // ---- [K; Q] tile by TMA: rows 0..63 = k tokens, 64..127 = q tokens (SwTile(128 x 128))
  if (warp == 0) tmem_alloc(&tslot, 64);
  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_init(&bar_kq, 1);
    asm volatile("fence.mbarrier_init.release.cluster;");
    mbar_expect_tx(&bar_kq, 32768u);
    tma_load_3d(sm, &a.tk, 0, j, tok0, &bar_kq);
    tma_load_3d(sm + 8192, &a.tq, 0, j, tok0, &bar_kq);
    tma_load_3d(sm + 16384, &a.tk, 64, j, tok0, &bar_kq);
    tma_load_3d(sm + 24576, &a.tq, 64, j, tok0, &bar_kq);
  }
  // the first round's gates, requested while the tiles land
  float gq0 = 0.f, gq1 = 0.f, bq0 = 0.f, bq1 = 0.f;
  if (warp < min(PR_GR, a.G)) {
    const int hv = j * a.G + warp, r0 = 2 * lane, r1 = r0 + 1;
    if (r0 < L) {
      gq0 = a.g[(size_t)(tok0 + r0) * a.HV + hv];
      bq0 = a.beta[(size_t)(tok0 + r0) * a.HV + hv];
    }
    if (r1 < L) {
      gq1 = a.g[(size_t)(tok0 + r1) * a.HV + hv];
      bq1 = a.beta[(size_t)(tok0 + r1) * a.HV + hv];
    }
  }
  __syncthreads();
  if (!__syncthreads_and(mbar_wait(&bar_kq, 0, a.err))) {
    if (warp == 0) tmem_dealloc(tslot, 64);
    return;
  }
  if (L < CH) {   // zero the rows past the document end (they hold the next document)
    for (int idx = tid; idx < (CH - L) * 32; idx += PR_THREADS) {
      const int t = idx >> 5, half = (idx >> 4) & 1, c8 = idx & 15;
      *reinterpret_cast<uint4*>(sm + sw_chunk(half * 64 + L + t, c8, 128)) = make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();
  }
  {  // L2 norms: row tid >> 1 of the tile; four partial sums of 32 elements (two per thread),
     // combined as (p0 + p1) + (p2 + p3)
    const int rr = tid >> 1, hh = tid & 1;
    float pr[2];
#pragma unroll
    for (int qq = 0; qq < 2; ++qq) {
      float ss = 0.f;
#pragma unroll
      for (int c8 = (2 * hh + qq) * 4; c8 < (2 * hh + qq) * 4 + 4; ++c8) {
        uint4 val = *reinterpret_cast<const uint4*>(sm + sw_chunk(rr, c8, 128));
        const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&val);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float2 f = __bfloat1622float2(h2[e]);
          ss = fmaf(f.x, f.x, ss);
          ss = fmaf(f.y, f.y, ss);
        }
      }
      pr[qq] = ss;
    }
    float ss = pr[0] + pr[1];
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    const float rn = a.l2norm ? 1.0f / sqrtf(ss + 1e-6f) : 1.0f;
    if (hh == 0) {
      if (rr < 64) rk[rr] = rn;
      else rq[rr - 64] = rn;
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tslot;
  const uint32_t sm_a = smem_u32(sm);
  if (tid == 0) {
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
      mma_ss(tb, desc_k(sm_a, 128, ks), desc_k(sm_a, 128, ks), idesc(128, 64, 0, 0), ks > 0);
    mma_commit(&bar);
  }
  bool ok = __syncthreads_and(mbar_wait(&bar, 0, a.err));
  tc_fence_after();

  for (int h0 = 0; ok && h0 < a.G; h0 += PR_GR) {
    const int ng = min(PR_GR, a.G - h0);
    if (h0 > 0) {   // the previous round's output copies still read the staging buffers
      if (tid == 0) bulk_wait_read();
      __syncthreads();
    }
    // ---- gates: warp w scans value head h0 + w (log2 units)
    if (warp < ng) {
      const int hv = j * a.G + h0 + warp;
      const int r0 = 2 * lane, r1 = r0 + 1;
      float g0 = gq0, g1 = gq1, b0 = bq0, b1 = bq1;
      if (h0 > 0) {
        g0 = g1 = b0 = b1 = 0.f;
        if (r0 < L) {
          g0 = a.g[(size_t)(tok0 + r0) * a.HV + hv];
          b0 = a.beta[(size_t)(tok0 + r0) * a.HV + hv];
        }
        if (r1 < L) {
          g1 = a.g[(size_t)(tok0 + r1) * a.HV + hv];
          b1 = a.beta[(size_t)(tok0 + r1) * a.HV + hv];
        }
      }
      float s = g0 + g1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += y;
      }
      const float ex = s - (g0 + g1);
      const float G0v = (ex + g0) * kLog2e, G1v = (ex + g0 + g1) * kLog2e;
      Gs[warp][r0] = G0v;
      Gs[warp][r1] = G1v;
      bs[warp][r0] = b0;
      bs[warp][r1] = b1;
      const float Gfirst = __shfl_sync(0xffffffffu, G0v, 0);
      const float Glast = __shfl_sync(0xffffffffu, G1v, 31);   // = G_{L-1} (gates past L are 0)
      eGr[warp][r0] = exp2f(G0v - Gfirst);
      eGr[warp][r1] = exp2f(G1v - Gfirst);
      const bool sf = (Gfirst - Glast) < kSafeRange;
      eGi[warp][r0] = sf ? exp2f(Gfirst - G0v) : 0.f;
      eGi[warp][r1] = sf ? exp2f(Gfirst - G1v) : 0.f;
      cf[warp][r0] = rk[r0] * eGi[warp][r0];
      cf[warp][r1] = rk[r1] * eGi[warp][r1];
      ca[warp][r0] = b0 * rk[r0] * eGr[warp][r0];
      ca[warp][r1] = b1 * rk[r1] * eGr[warp][r1];
      if (lane == 0) safe[warp] = sf;
    }
    __syncthreads();

    // ---- A^T (FP32, rows of KK^T), Aqk tiles (rows of QK^T), scalars
    float kq[32];  // row `row` of [KK^T; QK^T], columns cb0 .. cb0 + 31 (reloaded per round)
    tmem_ld32(taddr(tb, w4 * 32, cb0), kq);
    for (int hh = 0; hh < ng; ++hh) {
      const float* Gh = Gs[hh];
      const float* bh = bs[hh];
      const bool sf = safe[hh];
      if (row < 64) {
        // KK^T is symmetric, so the thread holding its row c writes row c of the transposed A:
        // S[c][r] = A[r][c] = (beta_r rk_r e^{G_r - G_0}) (rk_c e^{G_0 - G_c}) KK[c][r] for c < r < L
        const int c = row;
        float* At = reinterpret_cast<float*>(sm + hh * PR_VH);
        if (sf) {
          const float pc = cf[hh][c];
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const int r0 = cb0 + 4 * e4;
            const float4 f = *reinterpret_cast<const float4*>(&ca[hh][r0]);
            float4 v;
            v.x = (r0 + 0 > c && r0 + 0 < L) ? pc * f.x * kq[4 * e4 + 0] : 0.f;
            v.y = (r0 + 1 > c && r0 + 1 < L) ? pc * f.y * kq[4 * e4 + 1] : 0.f;
            v.z = (r0 + 2 > c && r0 + 2 < L) ? pc * f.z * kq[4 * e4 + 2] : 0.f;
            v.w = (r0 + 3 > c && r0 + 3 < L) ? pc * f.w * kq[4 * e4 + 3] : 0.f;
            *reinterpret_cast<float4*>(At + c * PR_ALD + r0) = v;
          }
        } else {
          const float pc = rk[c];
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const int r0 = cb0 + 4 * e4;
            float x[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int r = r0 + q;
              x[q] = (r > c && r < L) ? bh[r] * rk[r] * pc * exp2f(Gh[r] - Gh[c]) * kq[4 * e4 + q] : 0.f;
            }
            *reinterpret_cast<float4*>(At + c * PR_ALD + r0) = make_float4(x[0], x[1], x[2], x[3]);
          }
        }
        const int r = row;
        if (wg == 0) {
          float* sc = reinterpret_cast<float*>(sm + PR_SC + hh * CB_SCAL_BYTES);
          const float GL = Gh[L - 1];
          sc[r] = r < L ? a.scale * exp2f(Gh[r]) * rq[r] : 0.f;
          sc[64 + r] = r < L ? exp2f(GL - Gh[r]) * rk[r] : 0.f;
          if (r == 0) {
            sc[128] = exp2f(GL);
            reinterpret_cast<int*>(sc)[129] = L;
          }
        }
      } else {
        const int r = row - 64;
        uint8_t* aq = sm + PR_AQ + hh * TILE64_BYTES;
        const float pr = rq[r] * (sf ? eGr[hh][r] : 1.f);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          float x[8];
          if (sf) {
            const float4 fa = *reinterpret_cast<const float4*>(&cf[hh][cb0 + q4 * 8]);
            const float4 fb = *reinterpret_cast<const float4*>(&cf[hh][cb0 + q4 * 8 + 4]);
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
              x[e] = (jj <= r && r < L) ? pr * rk[jj] * exp2f(Gh[r] - Gh[jj]) * kq[q4 * 8 + e] : 0.f;
            }
          }
          uint4 w;
          w.x = pack_bf16(x[0], x[1]);
          w.y = pack_bf16(x[2], x[3]);
          w.z = pack_bf16(x[4], x[5]);
          w.w = pack_bf16(x[6], x[7]);
          *reinterpret_cast<uint4*>(aq + sw_chunk(r, (cb0 >> 3) + q4, 64)) = w;
        }
      }
    }
    __syncthreads();

    // ---- T = (I + A)^-1 by 16 x 16 blocks, warp pair per value head (64 lanes).  One FP32 array
    // S[p][q] (pitch PR_ALD) holds A[r][c] (c < r) at S[c][r] and T[r][c] (c <= r) at S[r][c].
    //   diagonal blocks  T_bb = (I + A_bb)^-1, forward substitution, lane = column
    //   block diagonal d T_ij = -T_ii sum_{k=j}^{i-1} A_ik T_kj (i - j = d), lane = (block, column)
    if ((warp >> 1) < ng) {
      const int hh = warp >> 1;
      const int l = (warp & 1) * 32 + lane;
      float* Sm = reinterpret_cast<float*>(sm + hh * PR_VH);
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
            if (4 * g4 + 0 > jq) x[4 * g4 + 0] = fmaf(-av.x, xj, x[4 * g4 + 0]);
            if (4 * g4 + 1 > jq) x[4 * g4 + 1] = fmaf(-av.y, xj, x[4 * g4 + 1]);
            if (4 * g4 + 2 > jq) x[4 * g4 + 2] = fmaf(-av.z, xj, x[4 * g4 + 2]);
            if (4 * g4 + 3 > jq) x[4 * g4 + 3] = fmaf(-av.w, xj, x[4 * g4 + 3]);
          }
        }
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (i >= cc) Sm[(o + i) * PR_ALD + o + cc] = x[i];
      }
      named_bar(1 + hh, 64);
      // off-diagonal blocks, one block diagonal d at a time (then T_ij is complete for i - j = d)
      offdiag_level<1>(Sm, l);
      named_bar(1 + hh, 64);
      offdiag_level<2>(Sm, l);
      named_bar(1 + hh, 64);
      offdiag_level<3>(Sm, l);
      named_bar(1 + hh, 64);
      const int col = l;   // the tiles, lane = column
      float x[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) x[i] = i >= col ? Sm[i * PR_ALD + col] : 0.f;
      named_bar(1 + hh, 64);   // both warps of the pair are done reading A^T
      const float bc = bs[hh][col];
      const float pc = bc * exp2f(Gs[hh][col]) * rk[col];
      uint8_t* tiles = sm + hh * PR_VH;
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        const uint32_t off = sw_off(i, col, 64);
        *reinterpret_cast<__nv_bfloat16*>(tiles + off) = __float2bfloat16_rn(x[i] * pc);          // T'
        *reinterpret_cast<__nv_bfloat16*>(tiles + TILE64_BYTES + off) = __float2bfloat16_rn(x[i] * bc);  // T''
        if (a.write_T) *reinterpret_cast<__nv_bfloat16*>(tiles + 2 * TILE64_BYTES + off) = __float2bfloat16_rn(x[i]);
      }
    }
    fence_async_smem();
    __syncthreads();
    if (tid == 0) {   // ship the staged blocks: T' T'' (contiguous), Aqk, T, scalars
      for (int hh = 0; hh < ng; ++hh) {
        uint8_t* cbp = a.cb + ((size_t)c * a.HV + j * a.G + h0 + hh) * CB_BYTES;
        bulk_store(cbp + CB_TP, sm + hh * PR_VH, 2 * TILE64_BYTES);
        bulk_store(cbp + CB_AQK, sm + PR_AQ + hh * TILE64_BYTES, TILE64_BYTES);
        if (a.write_T) bulk_store(cbp + CB_T, sm + hh * PR_VH + 2 * TILE64_BYTES, TILE64_BYTES);
        bulk_store(cbp + CB_SCAL, sm + PR_SC + hh * CB_SCAL_BYTES, CB_SCAL_BYTES);
      }
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
  prep_kernel<<<dim3(NC, a.H), PR_THREADS, PR_SMEM_ALLOC, s>>>(a);
  prof_end(K_PREP, s);
}

}  // namespace gdn
