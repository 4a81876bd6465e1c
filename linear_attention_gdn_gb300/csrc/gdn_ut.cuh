// gdn_ut.cuh -- the on-chip UT / WY stage of one 64-token chunk and one value
// head, run by one 128-thread warpgroup of the preparation kernel.
//
// For the chunk's tokens r < L (q/k head j, value head h):
//   rk_r, rq_r   1/sqrt(x.x + 1e-6) of k_r, q_r (or 1 with l2norm off)
//   G_r   = sum_{i<=r} g_i        (chunk-local cumulative gate: the pages'
//                                  "GLM prep" gate prefix rows)
//   A     = strict_tril(beta_r e^{G_r - G_c} k^_r.k^_c)          ("Akk")
//   T     = (I + A)^-1
//   Aqk   = tril(e^{G_r - G_c} q^_r.k^_c)                         ("Aqk")
//   T'    = T diag(beta gamma rk),  T'' = T diag(beta)
// so that W = T diag(beta gamma) K^ = T' K and U = T diag(beta) V = T'' V are
// the WY program's w and u ("feat(cake_gdn_kcp) ... #8172" page, commit notes
// on the intra / WY / GLM-prep programs; "#8542" page, the save-set table,
// which lists gcum, Akk, Aqk, w and u among what the replay form recomputes).
// KK^T and QK^T come from one tcgen05 MMA on the stacked [K; Q] tile (M = 128)
// into 64 TMEM columns; of the unit lower-triangular inverse, the two 32 x 32
// diagonal blocks are formed here in FP32 by forward substitution (one lane
// per column), and two tensor-core products complete T (ut_tc_inverse).
//
// Gate factors: e^{G_r - G_c} for c <= r is the product e^{G_r - G_0}
// e^{G_0 - G_c} of per-token factors when the chunk's gate range G_0 - G_{L-1}
// is below 2^100 (log2 units, safe in FP32), and one exp2f per element
// otherwise.
//
// Tiles: the [K; Q] tile is a SwTile(128 x 128) with rows 0-63 the chunk's k
// tokens and rows 64-127 its q tokens (64-column panels 16 KB apart: four TMA
// boxes land it); Aqk, T', T'', T are SwTile(64 x 64) BF16.  The scalar block
// holds sc_r = scale gamma_r rq_r [64], kd_r = e^{G_L - G_r} rk_r [64],
// e^{G_L} and L (as an int), 1 KB.
#pragma once
#include <stddef.h>

#include "gdn_common.cuh"

namespace gdn {

constexpr float kUtLog2e = 1.4426950408889634f;
constexpr float kUtSafeRange = 100.f;   // log2 units
constexpr int UT_ALD = 68;              // row pitch (floats) of the FP32 A^T / T array
constexpr int UT_WORK_BYTES = 64 * UT_ALD * 4;   // 17,408: the FP32 array; T' then T'' are written over it
constexpr int UT_SCAL_BYTES = 1024;
static_assert(2 * 8192 <= UT_WORK_BYTES, "T' and T'' fit in the FP32 array's space");

// per-token factors of one chunk, shared by the warpgroup (16-byte aligned: read as float4)
struct __align__(16) UtTok {
  float rq[64], rk[64];
  float Gs[64], bs[64], eGr[64], eGi[64];
  float cf[64];     // rk_c e^{G_0 - G_c}: the column factor of A and Aqk
  float ca[64];     // beta_r rk_r e^{G_r - G_0}: the row factor of A
  float pcol[64];   // beta_c e^{G_c} rk_c: the column factor of T'
  int safe;
};
static_assert(alignof(UtTok) >= 16 && offsetof(UtTok, ca) % 16 == 0 && offsetof(UtTok, cf) % 16 == 0,
              "UtTok members are read as float4");

// Zero the rows L..63 of the [K; Q] tile (they hold the next document's tokens).
__device__ __forceinline__ void ut_zero_tail(uint8_t* kq, int L, int lt) {
  for (int idx = lt; idx < (CH - L) * 32; idx += 128) {
    const int t = idx >> 5, half = (idx >> 4) & 1, c8 = idx & 15;
    *reinterpret_cast<uint4*>(kq + sw_chunk(half * 64 + L + t, c8, 128)) = make_uint4(0u, 0u, 0u, 0u);
  }
}

// L2 norm of row lt of the [K; Q] tile: four partial sums of 32 elements (each the sum of its even-
// and its odd-element chain, the two run as paired FMAs), combined as (p0 + p1) + (p2 + p3).  The
// gradient kernel sums in the same order.
__device__ __forceinline__ float ut_row_rnorm(const uint8_t* kq, int lt, int l2norm) {
  float pr[4];
#pragma unroll
  for (int qq = 0; qq < 4; ++qq) {
    float se = 0.f, so = 0.f;
#pragma unroll
    for (int c8 = qq * 4; c8 < qq * 4 + 4; ++c8) {
      const uint4 val = *reinterpret_cast<const uint4*>(kq + sw_chunk(lt, c8, 128));
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
  return l2norm ? 1.0f / sqrtf(ss + 1e-6f) : 1.0f;
}
__device__ __forceinline__ void ut_norm_row(const uint8_t* kq, int lt, int l2norm, UtTok& u) {
  const float rn = ut_row_rnorm(kq, lt, l2norm);
  if (lt < 64) u.rk[lt] = rn;
  else u.rq[lt - 64] = rn;
}

// The gate loads of one warp (lane -> tokens 2 lane, 2 lane + 1); zero past L.
__device__ __forceinline__ void ut_load_gates(const float* g, const float* beta, int HV, int hv, int tok0, int L,
                                              int lane, float (&gb)[4]) {
  const int r0 = 2 * lane, r1 = r0 + 1;
  gb[0] = gb[1] = gb[2] = gb[3] = 0.f;
  if (r0 < L) {
    gb[0] = g[(size_t)(tok0 + r0) * HV + hv];
    gb[2] = beta[(size_t)(tok0 + r0) * HV + hv];
  }
  if (r1 < L) {
    gb[1] = g[(size_t)(tok0 + r1) * HV + hv];
    gb[3] = beta[(size_t)(tok0 + r1) * HV + hv];
  }
}

// The per-token gate factors (one warp; needs rk): cumulative gate in log2 units and the factors above.
__device__ __forceinline__ void ut_gates(const float (&gb)[4], int lane, UtTok& u) {
  const int r0 = 2 * lane, r1 = r0 + 1;
  const float g0 = gb[0], g1 = gb[1], b0 = gb[2], b1 = gb[3];
  float s = g0 + g1;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, s, o);
    if (lane >= o) s += y;
  }
  const float ex = s - (g0 + g1);
  const float G0v = (ex + g0) * kUtLog2e, G1v = (ex + g0 + g1) * kUtLog2e;
  u.Gs[r0] = G0v;
  u.Gs[r1] = G1v;
  u.bs[r0] = b0;
  u.bs[r1] = b1;
  const float Gfirst = __shfl_sync(0xffffffffu, G0v, 0);
  const float Glast = __shfl_sync(0xffffffffu, G1v, 31);   // = G_{L-1} (gates past L are 0)
  const float er0 = exp2f(G0v - Gfirst), er1 = exp2f(G1v - Gfirst);
  u.eGr[r0] = er0;
  u.eGr[r1] = er1;
  const bool sf = (Gfirst - Glast) < kUtSafeRange;
  const float ei0 = sf ? exp2f(Gfirst - G0v) : 0.f, ei1 = sf ? exp2f(Gfirst - G1v) : 0.f;
  u.eGi[r0] = ei0;
  u.eGi[r1] = ei1;
  const float k0 = u.rk[r0], k1 = u.rk[r1];
  u.cf[r0] = k0 * ei0;
  u.cf[r1] = k1 * ei1;
  u.ca[r0] = b0 * k0 * er0;
  u.ca[r1] = b1 * k1 * er1;
  u.pcol[r0] = b0 * exp2f(G0v) * k0;
  u.pcol[r1] = b1 * exp2f(G1v) * k1;
  if (lane == 0) u.safe = sf;
}

// Issue KK^T and QK^T (one M = 128, N = 64 MMA of [K; Q] against K) into 64 TMEM columns at `dst`
// (warp-uniform; one lane issues).
__device__ __forceinline__ void ut_issue_kkqk(uint32_t dst, uint32_t kq_addr) {
#pragma unroll
  for (int ks = 0; ks < 8; ++ks)
    mma_ss_w(dst, desc_k(kq_addr, 128, ks), desc_k(kq_addr, 128, ks), idesc(128, 64, 0, 0), ks > 0);
}

// From row lt of [KK^T; QK^T] in TMEM (columns `kk` .. kk + 63, lane quarter wq): threads lt < 64 write
// row lt of the transposed A into the FP32 array Sm and the chunk scalars; threads lt >= 64 write row
// lt - 64 of Aqk into `aqk` (if non-null).
__device__ __forceinline__ void ut_build(uint32_t tb, int wq, int kk, int lt, int L, float scale, const UtTok& u,
                                         float* Sm, uint8_t* aqk, float* scal) {
  const bool sf = u.safe;
  if (lt >= 64 && aqk == nullptr) return;
#pragma unroll 1
  for (int cb0 = 0; cb0 < CH; cb0 += 32) {
    float kq[32];   // row lt of [KK^T; QK^T], columns cb0 .. cb0 + 31
    tmem_ld32(taddr(tb, wq * 32, kk + cb0), kq);
    if (lt < 64) {
      // KK^T is symmetric, so the thread holding its row c writes row c of the transposed A:
      // S[c][r] = A[r][c] = (beta_r rk_r e^{G_r - G_0}) (rk_c e^{G_0 - G_c}) KK[c][r] for c < r < L
      const int cc = lt;
      if (sf) {
        const float pc = u.cf[cc];
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const int r0 = cb0 + 4 * e4;
          const float4 f = *reinterpret_cast<const float4*>(&u.ca[r0]);
          float4 v;
          v.x = (r0 + 0 > cc && r0 + 0 < L) ? pc * f.x * kq[4 * e4 + 0] : 0.f;
          v.y = (r0 + 1 > cc && r0 + 1 < L) ? pc * f.y * kq[4 * e4 + 1] : 0.f;
          v.z = (r0 + 2 > cc && r0 + 2 < L) ? pc * f.z * kq[4 * e4 + 2] : 0.f;
          v.w = (r0 + 3 > cc && r0 + 3 < L) ? pc * f.w * kq[4 * e4 + 3] : 0.f;
          *reinterpret_cast<float4*>(Sm + cc * UT_ALD + r0) = v;
        }
      } else {
        const float pc = u.rk[cc];
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const int r0 = cb0 + 4 * e4;
          float x[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int r = r0 + q;
            x[q] = (r > cc && r < L) ? u.bs[r] * u.rk[r] * pc * exp2f(u.Gs[r] - u.Gs[cc]) * kq[4 * e4 + q] : 0.f;
          }
          *reinterpret_cast<float4*>(Sm + cc * UT_ALD + r0) = make_float4(x[0], x[1], x[2], x[3]);
        }
      }
    } else {
      const int r = lt - 64;
      const float pr = u.rq[r] * (sf ? u.eGr[r] : 1.f);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        float x[8];
        if (sf) {
          const float4 fa = *reinterpret_cast<const float4*>(&u.cf[cb0 + q4 * 8]);
          const float4 fb = *reinterpret_cast<const float4*>(&u.cf[cb0 + q4 * 8 + 4]);
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
            x[e] = (jj <= r && r < L) ? pr * u.rk[jj] * exp2f(u.Gs[r] - u.Gs[jj]) * kq[q4 * 8 + e] : 0.f;
          }
        }
        uint4 w;
        w.x = pack_bf16(x[0], x[1]);
        w.y = pack_bf16(x[2], x[3]);
        w.z = pack_bf16(x[4], x[5]);
        w.w = pack_bf16(x[6], x[7]);
        *reinterpret_cast<uint4*>(aqk + sw_chunk(r, (cb0 >> 3) + q4, 64)) = w;
      }
    }
  }
  if (lt < 64) {
    const int r = lt;
    const float GL = u.Gs[L - 1];
    scal[r] = r < L ? scale * exp2f(u.Gs[r]) * u.rq[r] : 0.f;
    scal[64 + r] = r < L ? exp2f(GL - u.Gs[r]) * u.rk[r] : 0.f;
    if (r == 0) {
      scal[128] = exp2f(GL);
      reinterpret_cast<int*>(scal)[129] = L;
    }
  }
}

// The two diagonal blocks T_bb = (I + A_bb)^-1 of T (32 x 32 each), in place in Sm, on lanes l = 0..63
// (the two warps of one 64-thread group that syncs on named barrier `bar_id`; warp b takes block b):
// forward substitution in FP32, lane = column; the upper triangles of the blocks are zeroed.  Call
// after the A^T rows of ut_build are written.
__device__ __forceinline__ void ut_diag_blocks(float* Sm, int l, int bar_id) {
  named_bar(bar_id, 64);
  {
    const int o = 32 * (l >> 5), cc = l & 31;
    float x[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] = (i == cc) ? 1.f : 0.f;
#pragma unroll
    for (int jq = 0; jq < 31; ++jq) {   // x[i] -= A[i][jq] x[jq] for i > jq (row jq of the array: A[.][jq])
      const float xj = x[jq];
#pragma unroll
      for (int g4 = (jq + 1) >> 2; g4 < 8; ++g4) {
        const float4 av = *reinterpret_cast<const float4*>(Sm + (o + jq) * UT_ALD + o + 4 * g4);
        if (4 * g4 + 0 > jq) fma2(x[4 * g4 + 0], x[4 * g4 + 1], -av.x, -av.y, xj);
        else if (4 * g4 + 1 > jq) x[4 * g4 + 1] = fmaf(-av.y, xj, x[4 * g4 + 1]);
        if (4 * g4 + 2 > jq) fma2(x[4 * g4 + 2], x[4 * g4 + 3], -av.z, -av.w, xj);
        else if (4 * g4 + 3 > jq) x[4 * g4 + 3] = fmaf(-av.w, xj, x[4 * g4 + 3]);
      }
    }
    __syncwarp();   // every lane of the block has read its A entries
#pragma unroll
    for (int i = 0; i < 32; ++i) Sm[(o + i) * UT_ALD + o + cc] = x[i];   // x[i] = 0 above the diagonal
  }
}

// ---------------------------------------------------------------------------
// The rest of T = (I + A)^-1 on the tensor cores, after ut_diag_blocks.  With D the two inverted
// 32 x 32 diagonal blocks and L the strictly block-lower part of A (its lower-left 32 x 32 block),
//   I + A = D^-1 (I + N),  N = D L,  N^2 = 0   =>   T = (I - N) D,
// two dependent M = 64 tcgen05 products (BF16 operands, FP32 accumulation).  Run by all NT threads
// of the CTA; warp 0 issues.  The FP32 array Sm (row n: T_bb in n's block, A[c][n] in the later
// block's columns c) is read into registers before the tiles are written, so the tiles may lie over
// it.  T is left in TMEM columns inv .. inv + 63 (M = 64 layout; read it with ut_ld_result).  tph is
// the phase of `bar`; t_pend receives the phase of a product whose completion was not seen when a
// wait runs out (the caller drains it).
// ---------------------------------------------------------------------------
struct UtInvTiles {
  uint8_t* d;    // D, SwTile(64 x 64)
  uint8_t* lx;   // L^T, then X = I - N
};

// The 16-column groups of an M = 64, N = 64 result that warp `warp` of an NT-thread CTA reads: the
// warps of one TMEM lane quarter (warp % 4) split the four groups between them.
template <int NT>
struct UtGroups {
  static constexpr int NG = 4 * 128 / NT;   // groups per warp
  static __device__ __forceinline__ int first(int warp) { return (warp >> 2) * NG; }
};

// This thread's elements of an M = 64, N = 64 result at TMEM column `col` (the .16x256b lane map):
// u[g][i] is row 16 (warp % 4) + lane / 4 + 8 ((i >> 1) & 1), column 16 (g0 + g) + 8 (i >> 2) +
// 2 (lane % 4) + (i & 1), for the groups g0 .. g0 + NG - 1 of UtGroups<NT>.
template <int NT>
__device__ __forceinline__ void ut_ld_result(uint32_t tb, int col, int warp, uint32_t (&u)[UtGroups<NT>::NG][8]) {
  const int g0 = UtGroups<NT>::first(warp);
#pragma unroll
  for (int g = 0; g < UtGroups<NT>::NG; ++g) tmem_ld_m64_async(taddr(tb, (warp & 3) * 32, col + 16 * (g0 + g)), u[g]);
  tmem_wait_ld();
}

// NT = 128 or 256 threads (all of the CTA) take part.
template <int NT>
__device__ __forceinline__ bool ut_tc_inverse(const float* Sm, const UtInvTiles& tl, uint32_t tb, int inv,
                                              uint64_t* bar, uint32_t& tph, int* err, int& t_pend) {
  static_assert(NT == 128 || NT == 256, "one or two warpgroups");
  constexpr int NG = UtGroups<NT>::NG;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r0 = 16 * (warp & 3) + (lane >> 2), cq = 2 * (lane & 3), g0 = UtGroups<NT>::first(warp);
  {  // D and L^T as BF16 tiles from rows of the array: row n holds T_bb (columns of n's block, zero
     // above the diagonal) and, in the later block's columns c, A[c][n] = L^T[n][c]
    uint4 dch[512 / NT], lch[512 / NT];
#pragma unroll
    for (int it = 0; it < 512 / NT; ++it) {
      const int item = tid + NT * it, n = item >> 3, c8 = item & 7;
      const float4 u0 = *reinterpret_cast<const float4*>(Sm + n * UT_ALD + 8 * c8);
      const float4 u1 = *reinterpret_cast<const float4*>(Sm + n * UT_ALD + 8 * c8 + 4);
      const uint4 w = make_uint4(pack_bf16(u0.x, u0.y), pack_bf16(u0.z, u0.w), pack_bf16(u1.x, u1.y),
                                 pack_bf16(u1.z, u1.w));
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      const int bn = n >> 5, bc = c8 >> 2;
      dch[it] = bc == bn ? w : z;
      lch[it] = bc > bn ? w : z;
    }
    __syncthreads();   // the array is read: its space takes the tiles
#pragma unroll
    for (int it = 0; it < 512 / NT; ++it) {
      const int item = tid + NT * it, n = item >> 3, c8 = item & 7;
      *reinterpret_cast<uint4*>(tl.d + sw_chunk(n, c8, 64)) = dch[it];
      *reinterpret_cast<uint4*>(tl.lx + sw_chunk(n, c8, 64)) = lch[it];
    }
  }
  auto product = [&](const uint8_t* a_tile, const uint8_t* b_tile, bool b_mn) -> bool {   // TMEM = A B
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) {
      const uint32_t sa = smem_u32(a_tile), sb = smem_u32(b_tile);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_ss_w(tb + inv, desc_k(sa, 64, ks), b_mn ? desc_mn(sb, 64, ks) : desc_k(sb, 64, ks),
                 idesc(64, 64, 0, b_mn ? 1 : 0), ks > 0);
      mma_commit_w(bar);
    }
    const bool r = __syncthreads_and(mbar_wait(bar, tph, err));
    if (!r) t_pend = (int)tph;
    tph ^= 1;
    tc_fence_after();
    return r;
  };
  uint32_t u[NG][8];
  // (a K-major B tile is rows N, columns K; L^T is that form of L.  An MN-major B tile is rows K,
  // columns N: a row-major D.)
  bool ok = product(tl.d, tl.lx, false);   // N = D L
  if (ok) {  // X = I - N -> BF16 tile (over L^T, which N = D L has finished reading)
    ut_ld_result<NT>(tb, inv, warp, u);
#pragma unroll
    for (int g = 0; g < NG; ++g)
#pragma unroll
      for (int i = 0; i < 8; i += 2) {
        const int r = r0 + 8 * ((i >> 1) & 1), cc = 16 * (g0 + g) + 8 * (i >> 2) + cq;
        const float x0 = (r == cc ? 1.f : 0.f) - __uint_as_float(u[g][i]);
        const float x1 = (r == cc + 1 ? 1.f : 0.f) - __uint_as_float(u[g][i + 1]);
        *reinterpret_cast<uint32_t*>(tl.lx + sw_off(r, cc, 64)) = pack_bf16(x0, x1);
      }
  }
  ok = ok && product(tl.lx, tl.d, true);   // T = X D
  return ok;
}

}  // namespace gdn
