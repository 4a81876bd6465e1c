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
// The inverse of the unit lower-triangular I + A is taken blockwise: the two
// 32 x 32 diagonal blocks T11, T22 by FP32 forward substitution (one thread
// per column), the off-diagonal block T21 = -T22 A21 T11 by two tcgen05 MMAs
// (M = 64) on the padded 64 x 64 operands.
#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_prof.h"

namespace gdn {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int PREP_GR = 3;                            // value heads per round
constexpr int PREP_BLK = 32 * 33 + 1;                 // padded 32 x 32 FP32 block (odd stride: the
                                                      // blocks' same elements fall in different banks)
constexpr int PREP_TILES = 0;                         // Lm, Dm, Xt tiles (3 x 8 KB)
constexpr int PREP_AD = 3 * TILE64_BYTES;             // diagonal blocks of A
constexpr int PREP_TD = PREP_AD + PREP_GR * 2 * PREP_BLK * 4;   // their inverses
constexpr int PREP_A21 = PREP_TD + PREP_GR * 2 * PREP_BLK * 4;  // A21 blocks
constexpr int PREP_SMEM = PREP_A21 + PREP_GR * PREP_BLK * 4;
constexpr int PREP_SMEM_ALLOC = PREP_SMEM + 1024;
static_assert(PREP_SMEM >= 32768, "the [K;Q] tile reuses the front of shared memory");

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return (uint8_t*)(((uintptr_t)p + 1023) & ~(uintptr_t)1023);
}

__global__ void __launch_bounds__(128, 2) prep_kernel(PrepArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  __shared__ float rq[CH], rk[CH];
  __shared__ float Gs[PREP_GR][CH], bs[PREP_GR][CH];
  __shared__ uint64_t bar;
  __shared__ uint32_t tslot;
  const int c = blockIdx.x, j = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (*(volatile int*)a.err) return;
  const int tok0 = a.chunk_tok0[c], L = a.chunk_len[c];

  // ---- [K; Q] tile: rows 0..63 = k tokens, 64..127 = q tokens (zero past L)
  for (int idx = tid; idx < 128 * 16; idx += 128) {
    const int row = idx >> 4, c8 = idx & 15, r = row & 63;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (r < L) {
      const __nv_bfloat16* src = (row < 64 ? a.k : a.q) + ((size_t)(tok0 + r) * a.H + j) * D + c8 * 8;
      val = __ldg(reinterpret_cast<const uint4*>(src));
    }
    *reinterpret_cast<uint4*>(sm + sw_chunk(row, c8, 128)) = val;
  }
  if (warp == 0) tmem_alloc(&tslot, 128);
  if (tid == 0) {
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;");
  }
  __syncthreads();
  {  // L2 norms (row tid of the tile)
    float ss = 0.f;
#pragma unroll
    for (int c8 = 0; c8 < 16; ++c8) {
      uint4 val = *reinterpret_cast<const uint4*>(sm + sw_chunk(tid, c8, 128));
      const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&val);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float2 f = __bfloat1622float2(h2[e]);
        ss = fmaf(f.x, f.x, ss);
        ss = fmaf(f.y, f.y, ss);
      }
    }
    const float rn = a.l2norm ? 1.0f / sqrtf(ss + 1e-6f) : 1.0f;
    if (tid < 64) rk[tid] = rn;
    else rq[tid - 64] = rn;
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tslot;
  const uint32_t sm_a = smem_u32(sm);
  uint32_t ph = 0;
  if (tid == 0) {
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
      mma_ss(tb, desc_k(sm_a, 128, ks), desc_k(sm_a, 128, ks), idesc(128, 64, 0, 0), ks > 0);
    mma_commit(&bar);
  }
  bool ok = __syncthreads_and(mbar_wait(&bar, ph, a.err));
  ph ^= 1;
  tc_fence_after();
  float kq[64];  // row tid of [KK^T; QK^T]
  if (ok) {
    tmem_ld32(taddr(tb, warp * 32, 0), kq);
    tmem_ld32(taddr(tb, warp * 32, 32), kq + 32);
  }
  tc_fence_before();
  __syncthreads();  // the [K;Q] tile is dead from here on

  float* Ad = reinterpret_cast<float*>(sm + PREP_AD);
  float* Td = reinterpret_cast<float*>(sm + PREP_TD);
  float* A21s = reinterpret_cast<float*>(sm + PREP_A21);
  uint8_t* Lm = sm + PREP_TILES;
  uint8_t* Dm = Lm + TILE64_BYTES;
  uint8_t* Xt = Dm + TILE64_BYTES;

  for (int h0 = 0; ok && h0 < a.G; h0 += PREP_GR) {
    const int ng = min(PREP_GR, a.G - h0);
    // ---- gates: warp w scans value head h0 + w
    if (warp < ng) {
      const int hv = j * a.G + h0 + warp;
      const int r0 = 2 * lane, r1 = r0 + 1;
      float g0 = 0.f, g1 = 0.f, b0 = 0.f, b1 = 0.f;
      if (r0 < L) {
        g0 = a.g[(size_t)(tok0 + r0) * a.HV + hv];
        b0 = a.beta[(size_t)(tok0 + r0) * a.HV + hv];
      }
      if (r1 < L) {
        g1 = a.g[(size_t)(tok0 + r1) * a.HV + hv];
        b1 = a.beta[(size_t)(tok0 + r1) * a.HV + hv];
      }
      float s = g0 + g1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += y;
      }
      const float ex = s - (g0 + g1);
      // cumulative gate in log2 units: every exponential below is exp2f of a difference
      Gs[warp][r0] = (ex + g0) * kLog2e;
      Gs[warp][r1] = (ex + g0 + g1) * kLog2e;
      bs[warp][r0] = b0;
      bs[warp][r1] = b1;
    }
    __syncthreads();

    // ---- A blocks (threads 0..63, row r of KK^T); Aqk and scalars (64..127)
    for (int hh = 0; hh < ng; ++hh) {
      const int hv = j * a.G + h0 + hh;
      uint8_t* cbp = a.cb + ((size_t)c * a.HV + hv) * CB_BYTES;
      const float* Gh = Gs[hh];
      const float* bh = bs[hh];
      if (tid < 64) {
        const int r = tid;
        const float Gr = Gh[r], br = bh[r] * rk[r];
        float* A0 = Ad + (hh * 2 + 0) * PREP_BLK;
        float* A1 = Ad + (hh * 2 + 1) * PREP_BLK;
        float* A2 = A21s + hh * PREP_BLK;
#pragma unroll
        for (int jj = 0; jj < 64; ++jj) {
          const float val = (jj < r && r < L) ? br * rk[jj] * exp2f(Gr - Gh[jj]) * kq[jj] : 0.f;
          if (r < 32) {
            if (jj < 32) A0[r * 33 + jj] = val;
          } else if (jj >= 32) {
            A1[(r - 32) * 33 + (jj - 32)] = val;
          } else {
            A2[(r - 32) * 33 + jj] = val;
          }
        }
        float* sc = reinterpret_cast<float*>(cbp + CB_SCAL);
        const float GL = Gh[L - 1];
        sc[r] = r < L ? a.scale * exp2f(Gr) * rq[r] : 0.f;
        sc[64 + r] = r < L ? exp2f(GL - Gr) * rk[r] : 0.f;
        if (r == 0) {
          sc[128] = exp2f(GL);
          reinterpret_cast<int*>(sc)[129] = L;
        }
      } else {
        const int r = tid - 64;
        const float Gr = Gh[r], qr = rq[r];
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j0 = c8 * 8 + 2 * e, j1 = j0 + 1;
            const float v0 = (j0 <= r && r < L) ? qr * rk[j0] * exp2f(Gr - Gh[j0]) * kq[j0] : 0.f;
            const float v1 = (j1 <= r && r < L) ? qr * rk[j1] * exp2f(Gr - Gh[j1]) * kq[j1] : 0.f;
            w[e] = pack_bf16(v0, v1);
          }
          *reinterpret_cast<uint4*>(cbp + CB_AQK + sw_chunk(r, c8, 64)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    }
    __syncthreads();

    // ---- diagonal 32x32 inverses by forward substitution, jobs (head, block, column)
    {
      const int njobs = ng * 64;
      for (int rnd = 0; rnd * 128 < njobs; ++rnd) {
        const int jidx = rnd * 128 + ((rnd & 1) ? 127 - tid : tid);
        if (jidx >= njobs) continue;
        const int col = jidx / (2 * ng), rest = jidx % (2 * ng);
        const float* A = Ad + rest * PREP_BLK;   // rest = hh * 2 + blk
        float* X = Td + rest * PREP_BLK;
        for (int i = 0; i < col; ++i) X[i * 33 + col] = 0.f;
        X[col * 33 + col] = 1.f;
        for (int i = col + 1; i < 32; ++i) {
          float s = 0.f;
          for (int jj = col; jj < i; ++jj) s = fmaf(A[i * 33 + jj], X[jj * 33 + col], s);
          X[i * 33 + col] = -s;
        }
      }
    }
    __syncthreads();

    // ---- T21 = -T22 A21 T11 on the tensor cores, then T', T'' (and T)
    for (int hh = 0; ok && hh < ng; ++hh) {
      const int hv = j * a.G + h0 + hh;
      uint8_t* cbp = a.cb + ((size_t)c * a.HV + hv) * CB_BYTES;
      const float* T0 = Td + (hh * 2 + 0) * PREP_BLK;
      const float* T1 = Td + (hh * 2 + 1) * PREP_BLK;
      const float* A2 = A21s + hh * PREP_BLK;
      auto dval = [&](int r, int cc) -> float {
        if (r < 32) return cc < 32 ? T0[r * 33 + cc] : 0.f;
        return cc >= 32 ? T1[(r - 32) * 33 + (cc - 32)] : 0.f;
      };
      {  // Lm = [[0,0],[A21,0]], Dm = blockdiag(T11, T22), BF16
        const int r = tid >> 1, half = tid & 1;
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8) {
          const int c8 = half * 4 + q8;
          uint32_t wl[4], wd[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int cc = c8 * 8 + 2 * e;
            const float l0 = (r >= 32 && cc < 32) ? A2[(r - 32) * 33 + cc] : 0.f;
            const float l1 = (r >= 32 && cc + 1 < 32) ? A2[(r - 32) * 33 + cc + 1] : 0.f;
            wl[e] = pack_bf16(l0, l1);
            wd[e] = pack_bf16(dval(r, cc), dval(r, cc + 1));
          }
          *reinterpret_cast<uint4*>(Lm + sw_chunk(r, c8, 64)) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
          *reinterpret_cast<uint4*>(Dm + sw_chunk(r, c8, 64)) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
        }
      }
      fence_async_smem();
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
      if (tid == 0) {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_ss(tb + 64, desc_k(smem_u32(Lm), 64, ks), desc_mn(smem_u32(Dm), 64, ks), idesc(64, 64, 0, 1),
                 ks > 0);
        mma_commit(&bar);
      }
      ok = __syncthreads_and(mbar_wait(&bar, ph, a.err));
      ph ^= 1;
      tc_fence_after();
      if (!ok) break;
      {  // X = Lm Dm (M = 64 layout: warp w, lanes 0..15 hold rows 16w + lane)
        float x[64];
        tmem_ld32(taddr(tb, warp * 32, 64), x);
        tmem_ld32(taddr(tb, warp * 32, 96), x + 32);
        if (lane < 16) {
          const int r = warp * 16 + lane;
#pragma unroll
          for (int c8 = 0; c8 < 8; ++c8) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) w[e] = pack_bf16(x[c8 * 8 + 2 * e], x[c8 * 8 + 2 * e + 1]);
            *reinterpret_cast<uint4*>(Xt + sw_chunk(r, c8, 64)) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      fence_async_smem();
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
      if (tid == 0) {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_ss(tb + 64, desc_k(smem_u32(Dm), 64, ks), desc_mn(smem_u32(Xt), 64, ks), idesc(64, 64, 0, 1),
                 ks > 0);
        mma_commit(&bar);
      }
      ok = __syncthreads_and(mbar_wait(&bar, ph, a.err));
      ph ^= 1;
      tc_fence_after();
      if (!ok) break;
      {  // T = Dm - [[0,0],[Y21,0]] with Y = Dm X; write T'', T' (and T)
        float y[64];
        tmem_ld32(taddr(tb, warp * 32, 64), y);
        tmem_ld32(taddr(tb, warp * 32, 96), y + 32);
        if (lane < 16) {
          const int r = warp * 16 + lane;
          const float* Gh = Gs[hh];
          const float* bh = bs[hh];
#pragma unroll
          for (int c8 = 0; c8 < 8; ++c8) {
            uint32_t wp[4], wpp[4], wt[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float tv[2], tpp[2], tp[2];
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                const int cc = c8 * 8 + 2 * e + u;
                tv[u] = dval(r, cc) - ((r >= 32 && cc < 32) ? y[cc] : 0.f);
                tpp[u] = tv[u] * bh[cc];
                tp[u] = tpp[u] * exp2f(Gh[cc]) * rk[cc];
              }
              wt[e] = pack_bf16(tv[0], tv[1]);
              wpp[e] = pack_bf16(tpp[0], tpp[1]);
              wp[e] = pack_bf16(tp[0], tp[1]);
            }
            const uint32_t off = sw_chunk(r, c8, 64);
            *reinterpret_cast<uint4*>(cbp + CB_TP + off) = make_uint4(wp[0], wp[1], wp[2], wp[3]);
            *reinterpret_cast<uint4*>(cbp + CB_TPP + off) = make_uint4(wpp[0], wpp[1], wpp[2], wpp[3]);
            if (a.write_T) *reinterpret_cast<uint4*>(cbp + CB_T + off) = make_uint4(wt[0], wt[1], wt[2], wt[3]);
          }
        }
      }
      tc_fence_before();
      __syncthreads();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, 128);
}

void setup_prep_attrs() {
  cudaFuncSetAttribute(prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, PREP_SMEM_ALLOC);
}
void launch_prep(const PrepArgs& a, int NC, cudaStream_t s) {
  if (NC <= 0) return;
  prof_begin(K_PREP, s);
  prep_kernel<<<dim3(NC, a.H), 128, PREP_SMEM_ALLOC, s>>>(a);
  prof_end(K_PREP, s);
}

}  // namespace gdn
