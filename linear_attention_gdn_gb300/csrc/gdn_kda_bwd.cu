// gdn_kda_bwd.cu -- backward of the per-channel-decay (KDA) chunk form.
//
// Per chunk and value head (notation of gdn_kda.cu; dS = gradient of the state leaving the chunk,
// dX = dV_new from the adjoint walk, S and X = V_new from the saved set), reversing
//   O = scale (Q~ S + P X),  S_next = Diag(gamma_L) S + Kd^T X,  X = T'' V - T'' K~ S:
//   dQg = scale dO S^T        -> dq^ += gamma . dQg,       dG += Q~ . dQg
//   dKd = X dS^T              -> dk^ += E . dKd,           dG -= Kd . dKd,  dG_L += sum_r Kd . dKd
//   dG_L += gamma_L . rowsum(dS . S)
//   dW = -dX S^T,  dT = (dX V^T + dW K~^T) diag(beta)
//   dv = beta . (T^T dX),  dY = T^T dW -> dk^ += beta gamma . dY,  dG += beta K~ . dY
//   dA = -T^T dT T^T (strictly lower),  dM = diag(beta) dA,  dP = scale dO X^T (c <= r)
//   dbeta_r = V_r . (T^T dX)_r + K~_r . dY_r + sum_c dA_rc M_rc
//   rowM_r = sum_c dM_rc exp(G_r - G_c) . k^_c,  rowP_r likewise with dP (c < r),
//   col_c = sum_r (dM_rc k^_r + dP_rc q^_r) . exp(G_r - G_c) (r > c):
//     dk^ += rowM + col + dP_rr q^,  dq^ += rowP + dP_rr k^,  dG += k^ . rowM + q^ . rowP - k^ . col
//   (the diagonal of dP has no dG term: q^_r . dP_rr k^_r enters once with each sign)
//   dg = reverse cumulative sum of dG within the chunk (dG_L added at the last token)
// then the L2-norm backward of the q/k group sums (the reverse of the KDA oracle's per-token lines,
// "perf(cake_kda) ... #7097" page for the family; the chunk algebra is the GDN one of the
// "feat(cake_gdn_kcp) ... #8172" page with every decay inside the channel sums).
//
// The decay-weighted products rowM, rowP, col run on the tensor cores per pair of 16-token blocks
// (a, b), with Gx_a the log decay entering block a and every token carrying its own block's factor:
// Lk_r = k^_r exp(G_r - Gx_{blk r}), Lq_r likewise, Rb_c = k^_c exp(Gx_{blk c} - G_c), so that
// exp(G_r - G_c) k^_c = exp(G_r - Gx_a) F(a, b) Rb_c with F(a, b) = exp(Gx_a - Gx_b) per channel.
// The block products (one K = 16 MMA step each) are summed with F in FP32 afterwards.
//
// kda_grad_kernel: one CTA of 512 threads per (chunk, q/k head); the group's value heads one after
// another, each a fixed sequence of MMA groups and CUDA-core passes (no overlap between heads); dq^
// and dk^ accumulate over the heads in TMEM.
#include <cstring>

#include "gdn.h"
#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_prof.h"
#include "gdn_ut.cuh"

namespace gdn {

struct KdaGradArgs {
  CUtensorMap tq, tk, tv, tdo, tg, tdg;
  const float* g;
  const float* beta;
  const uint8_t* kb;      // [NC][HV][KB_BYTES] (T, M^T)
  const uint8_t* tape;    // saved S^T per chunk
  const uint8_t* dtape;   // dS'^T per chunk
  const uint8_t* vn;      // saved V_new^T per chunk
  const uint8_t* dvn;     // dV_new^T per chunk
  const int* chunk_tok0;
  const int* chunk_len;
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  float* dg;
  float* dbeta;
  int NC, H, HV, G, l2norm;
  float scale;
  int* err;
};

// shared memory (bytes, 1024-aligned regions)
constexpr int KG_KQ = 0;          // [K; Q] raw tile of the item, SwTile(128 x 128)
constexpr int KG_G = 32768;       // FP32 G [64][128] (log2 units) of the value head
constexpr int KG_T = 65536;       // T
constexpr int KG_MT = 73728;      // M^T
constexpr int KG_X = 81920;       // 128 KiB reused by the phases of a value head:
constexpr int KX_S = 0, KX_DS = 32768, KX_VN = 65536, KX_DV = 81920, KX_DO = 98304, KX_V = 114688;   // MA
constexpr int KX_WD = 0, KX_KT = 16384;                                      // dW^T, K~ (MB)
constexpr int KX_DT = 32768, KX_R1 = 40960, KX_DM = 49152, KX_DMT = 57344, KX_DP = 65536, KX_DPT = 73728;
constexpr int KX_LK = 81920, KX_LQ = 98304, KX_RB = 114688;                   // after MA
constexpr int KG_SMEM = KG_X + 131072;
constexpr int KG_SMEM_ALLOC = KG_SMEM + 1024;
// TMEM columns
constexpr int KGT_DQ = 0, KGT_DK = 64, KGT_A0 = 128, KGT_A1 = 192, KGT_A2 = 256, KGT_A3 = 320, KGT_A4 = 384,
              KGT_A5 = 448;
// the decay-weighted products (every other result is dead by then): Z_b (64 - 16 b columns each, from
// column 16 b of the result), Zp_b, then Y_a (16 a + 16 columns each) over the Z columns
// dG^T of the value head takes over A1 once A1 is read; the decay-weighted products then use the other
// result columns: Z_b (64 - 16 b columns each, from column 16 b of the result) from column 256, Zp_b
// at kZPCol[b], and Y_a (16 a + 16 columns each) over the Z columns
constexpr int KGT_DG = KGT_A1, KGT_Z = 256;
__constant__ int kZOff[4] = {0, 64, 112, 144};
__constant__ int kZPCol[4] = {128, 416, 464, 496};
__constant__ int kYOff[4] = {0, 16, 48, 96};

__device__ __forceinline__ int kg_pair(int a, int b) { return a * (a - 1) / 2 + b; }   // b < a

// four warpgroups; thread t owns row t % 128 (TMEM lane) and KG_CW of the 64 token columns of a result
constexpr int KG_WG = 4;
constexpr int KG_THREADS = 128 * KG_WG;
constexpr int KG_CW = 64 / KG_WG;
constexpr int KG_NH = KG_CW / 16;   // 16-column groups per thread
static_assert(KG_CW % 16 == 0, "whole 16-column groups per thread");

// sum over the 32 lanes of a warp of column `lane & 15` of v[16] (fixed order)
__device__ __forceinline__ float kg_colsum16(float (&v)[16], int lane) {
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int kq = 0; kq < o; ++kq) {
      const float mine = up ? v[kq + o] : v[kq];
      const float other = up ? v[kq] : v[kq + o];
      v[kq] = mine + __shfl_xor_sync(0xffffffffu, other, o);
    }
  }
  return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 16);
}

// sum over the 32 lanes of a warp of column `lane` of v[32] (fixed order)
__device__ __forceinline__ float colsum32(float (&v)[32], int lane) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int kq = 0; kq < o; ++kq) {
      const float mine = up ? v[kq + o] : v[kq];
      const float other = up ? v[kq] : v[kq + o];
      v[kq] = mine + __shfl_xor_sync(0xffffffffu, other, o);
    }
  }
  return v[0];
}

__device__ __forceinline__ void kg_unpack8(const uint4& w, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 x = __bfloat1622float2(h[e]);
    f[2 * e] = x.x;
    f[2 * e + 1] = x.y;
  }
}
__device__ __forceinline__ uint4 kg_pack8(const float* f) {
  return make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]), pack_bf16(f[6], f[7]));
}
__device__ __forceinline__ float bf16_at(const uint8_t* tile, int r, int c, int R) {
  return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(tile + sw_off(r, c, R)));
}

__global__ void __launch_bounds__(KG_THREADS, 1) kda_grad_kernel(const __grid_constant__ KdaGradArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_align1024(smem_raw);
  __shared__ __align__(16) float rk[CH], rq[CH], bs[CH];
  __shared__ __align__(16) float gx[4][D];     // log2 decay entering each 16-token block
  __shared__ __align__(16) float fab[6][D];    // exp2(gx[a] - gx[b]), b < a
  __shared__ __align__(16) float glL[D];       // log2 G_L per channel
  __shared__ __align__(16) float dgl[KG_WG][D];   // partial dG_L per key channel (per warpgroup)
  __shared__ __align__(16) float red[8][CH];   // per-warp partial column sums
  __shared__ __align__(16) float rowdb[KG_WG][CH];   // partial row sums (per warpgroup's columns)
  __shared__ __align__(16) float cum[KG_WG][D];      // per-warpgroup totals of the reverse cumulative sum
  __shared__ __align__(16) float pdiag[CH];    // dP_rr (kept out of the decay-weighted products)
  __shared__ uint64_t bar_qk, bar_ld, bar_g, bar_m;
  __shared__ uint32_t tslot;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, wg = tid >> 7, lt = tid & 127, wq = warp & 3;
  const int c0 = KG_CW * wg;   // this thread's columns (tokens) of a 64-column result
  const int c = blockIdx.x / a.H, j = blockIdx.x % a.H;
  if (*(volatile int*)a.err) return;
  const int tok0 = a.chunk_tok0[c], L = a.chunk_len[c];
  uint8_t* kq = sm + KG_KQ;
  float* Gm = reinterpret_cast<float*>(sm + KG_G);
  uint8_t* X = sm + KG_X;
  if (warp == 0) tmem_alloc(&tslot, 512);
  if (tid == 0) {
    mbar_init(&bar_qk, 1);
    mbar_init(&bar_ld, 1);
    mbar_init(&bar_g, 1);
    mbar_init(&bar_m, 1);
    asm volatile("fence.mbarrier_init.release.cluster;");
    mbar_expect_tx(&bar_qk, 32768u);
    tma_load_3d(kq, &a.tk, 0, j, tok0, &bar_qk);
    tma_load_3d(kq + 8192, &a.tq, 0, j, tok0, &bar_qk);
    tma_load_3d(kq + 16384, &a.tk, 64, j, tok0, &bar_qk);
    tma_load_3d(kq + 24576, &a.tq, 64, j, tok0, &bar_qk);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tslot;
  uint32_t mph = 0, ldph = 0;
  bool mma_pend = false, ld_pend = false, qk_pend = true;
  bool ok = __syncthreads_and(mbar_wait(&bar_qk, 0, a.err));
  if (ok) {
    qk_pend = false;
    if (L < CH && tid < 128) ut_zero_tail(kq, L, tid);
    __syncthreads();
    if (tid < 128) {
      const float rn = ut_row_rnorm(kq, tid, a.l2norm);
      if (tid < 64) rk[tid] = rn;
      else rq[tid - 64] = rn;
    }
    __syncthreads();
  }
  auto kraw = [&](int r, int i) { return bf16_at(kq, r, i, 128); };
  auto qraw = [&](int r, int i) { return bf16_at(kq, 64 + r, i, 128); };
  auto tldc = [&](int col, float* o) {   // this thread's KG_CW columns of a result
    if constexpr (KG_CW == 32) tmem_ld32(taddr(tb, wq * 32, col + c0), o);
    else tmem_ld16(taddr(tb, wq * 32, col + c0), o);
  };
  auto tld16c = [&](int col, float* o) { tmem_ld16(taddr(tb, wq * 32, col), o); };   // absolute column
  auto tst16c = [&](int col, const float* v) { tmem_st16(taddr(tb, wq * 32, col), v); };
  constexpr int kZPColH[4] = {128, 416, 464, 496};   // (kZPCol, as compile-time values for the MMA issue)

  auto to_tc = [&]() {   // generic smem / TMEM writes -> visible to the next MMAs
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  };
  auto commit = [&]() {
    mma_commit(&bar_m);
    mma_pend = true;
  };
  auto mma_wait = [&]() -> bool {   // the last commit (only one is ever outstanding)
    const bool r = __syncthreads_and(mbar_wait(&bar_m, mph, a.err));
    if (r) {
      mph ^= 1;
      mma_pend = false;
    }
    tc_fence_after();
    return r;
  };
  // M = 64 results: this thread's rows ra, ra + 8 and, per load g, columns c0 + 16 g + 8 (i >> 2) +
  // 2 (lane & 3) + (i & 1) for value i
  const int ra = 16 * wq + (lane >> 2);
  auto ld_m64 = [&](int col, uint32_t (&u)[KG_NH][8]) {
#pragma unroll
    for (int g = 0; g < KG_NH; ++g) tmem_ld_m64_async(taddr(tb, wq * 32, col + c0 + 16 * g), u[g]);
    tmem_wait_ld();
  };
  const uint32_t s_s = smem_u32(X + KX_S), s_ds = smem_u32(X + KX_DS), s_vn = smem_u32(X + KX_VN),
                 s_dv = smem_u32(X + KX_DV), s_do = smem_u32(X + KX_DO), s_v = smem_u32(X + KX_V),
                 s_t = smem_u32(sm + KG_T), s_wd = smem_u32(X + KX_WD), s_kt = smem_u32(X + KX_KT),
                 s_dt = smem_u32(X + KX_DT), s_r1 = smem_u32(X + KX_R1), s_dm = smem_u32(X + KX_DM),
                 s_dmt = smem_u32(X + KX_DMT), s_dp = smem_u32(X + KX_DP), s_dpt = smem_u32(X + KX_DPT),
                 s_lk = smem_u32(X + KX_LK), s_lq = smem_u32(X + KX_LQ), s_rb = smem_u32(X + KX_RB);

  for (int hh = 0; hh < a.G && ok; ++hh) {
    const int hv = j * a.G + hh;
    const size_t blk = (size_t)c * a.HV + hv;
    if (tid == 0) {   // this value head's tiles
      bulk_wait_read();   // the last value head's dg copy has read its staging tile
      const uint8_t* kbp = a.kb + blk * KB_BYTES;
      // the 64 g rows first, on their own barrier (rows past L are read as zero below): the decay
      // cumsum runs while the rest lands
      mbar_expect_tx(&bar_g, 32768u);
      tma_load_3d(Gm, &a.tg, 0, hv, tok0, &bar_g);
      mbar_expect_tx(&bar_ld, (uint32_t)(2 * STATE_BYTES + 2 * VN_BYTES + 2 * 16384 + 2 * TILE64_BYTES));
      bulk_load(X + KX_S, a.tape + blk * STATE_BYTES, STATE_BYTES, &bar_ld);
      bulk_load(X + KX_DS, a.dtape + blk * STATE_BYTES, STATE_BYTES, &bar_ld);
      bulk_load(X + KX_VN, a.vn + blk * VN_BYTES, VN_BYTES, &bar_ld);
      bulk_load(X + KX_DV, a.dvn + blk * VN_BYTES, VN_BYTES, &bar_ld);
      tma_load_3d(X + KX_DO, &a.tdo, 0, hv, tok0, &bar_ld);
      tma_load_3d(X + KX_DO + 8192, &a.tdo, 64, hv, tok0, &bar_ld);
      tma_load_3d(X + KX_V, &a.tv, 0, hv, tok0, &bar_ld);
      tma_load_3d(X + KX_V + 8192, &a.tv, 64, hv, tok0, &bar_ld);
      bulk_load(sm + KG_T, kbp + KB_T, TILE64_BYTES, &bar_ld);
      bulk_load(sm + KG_MT, kbp + KB_MT, TILE64_BYTES, &bar_ld);
      if (hh + 1 < a.G) {   // the next value head's tiles into L2 while this one is worked on (a hint)
        const size_t nb = blk + 1;
        bulk_prefetch(a.tape + nb * STATE_BYTES, STATE_BYTES);
        bulk_prefetch(a.dtape + nb * STATE_BYTES, STATE_BYTES);
        bulk_prefetch(a.vn + nb * VN_BYTES, VN_BYTES);
        bulk_prefetch(a.dvn + nb * VN_BYTES, VN_BYTES);
        tma_prefetch_3d(&a.tdo, 0, hv + 1, tok0);
        tma_prefetch_3d(&a.tdo, 64, hv + 1, tok0);
        tma_prefetch_3d(&a.tv, 0, hv + 1, tok0);
        tma_prefetch_3d(&a.tv, 64, hv + 1, tok0);
        bulk_prefetch(a.kb + nb * KB_BYTES + KB_T, TILE64_BYTES);
        bulk_prefetch(a.kb + nb * KB_BYTES + KB_MT, TILE64_BYTES);
        tma_prefetch_3d(&a.tg, 0, hv + 1, tok0);
      }
    }
    ld_pend = true;
    if (tid < CH) bs[tid] = tid < L ? a.beta[(size_t)(tok0 + tid) * a.HV + hv] : 0.f;
    ok = __syncthreads_and(mbar_wait(&bar_g, ldph, a.err));
    if (!ok) break;
    if (tid < 128) {   // channel tid: cumulative decay (log2 units), block entries, block ratios
      const int i = tid;
      float run = 0.f;
      for (int r = 0; r < CH; ++r) {
        if ((r & 15) == 0) gx[r >> 4][i] = run;
        run = fmaf(r < L ? Gm[r * D + i] : 0.f, kUtLog2e, run);   // (rows past L: the next document's)
        Gm[r * D + i] = run;
      }
      glL[i] = run;
#pragma unroll
      for (int aa = 1; aa < 4; ++aa)
#pragma unroll
        for (int b = 0; b < aa; ++b) fab[kg_pair(aa, b)][i] = exp2f(gx[aa][i] - gx[b][i]);
    }
    ok = __syncthreads_and(mbar_wait(&bar_ld, ldph, a.err));   // the other tiles
    if (!ok) break;
    ldph ^= 1;
    ld_pend = false;
    if (L < CH) {   // zero the dO, V rows past the document end
      for (int idx = tid; idx < (CH - L) * 32; idx += KG_THREADS) {
        const int t = idx >> 5, tile = (idx >> 4) & 1, c8 = idx & 15;
        *reinterpret_cast<uint4*>(X + (tile ? KX_V : KX_DO) + sw_chunk(L + t, c8, 64)) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    to_tc();
    // ---- MA: S dO^T (A1), dS X^T (A3), dO X^T (A4), S dX^T (A0), dX V^T (A5), dX^T T (A2)
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        mma_ss(tb + KGT_A4, desc_k(s_do, 64, ks), desc_mn(s_vn, 128, ks), idesc(64, 64, 0, 1), ks > 0);
        mma_ss(tb + KGT_A1, desc_mn(s_s, 128, ks), desc_k(s_do, 64, ks), idesc(128, 64, 1, 0), ks > 0);
        mma_ss(tb + KGT_A3, desc_mn(s_ds, 128, ks), desc_mn(s_vn, 128, ks), idesc(128, 64, 1, 1), ks > 0);
        mma_ss(tb + KGT_A0, desc_mn(s_s, 128, ks), desc_mn(s_dv, 128, ks), idesc(128, 64, 1, 1), ks > 0);
        mma_ss(tb + KGT_A5, desc_mn(s_dv, 128, ks), desc_k(s_v, 64, ks), idesc(64, 64, 1, 0), ks > 0);
      }
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_ss(tb + KGT_A2, desc_k(s_dv, 128, ks), desc_mn(s_t, 64, ks), idesc(128, 64, 0, 1), ks > 0);
      commit();
    }
    {  // while MA runs: gamma_L . <S, dS'> per key channel over this thread's 64 value rows
      const int i = lt;
      float acc0 = 0.f, acc1 = 0.f;
      for (int jj = (128 / KG_WG) * wg; jj < (128 / KG_WG) * (wg + 1); jj += 2) {
        acc0 = fmaf(bf16_at(X + KX_S, jj, i, 128), bf16_at(X + KX_DS, jj, i, 128), acc0);
        acc1 = fmaf(bf16_at(X + KX_S, jj + 1, i, 128), bf16_at(X + KX_DS, jj + 1, i, 128), acc1);
      }
      dgl[wg][i] = exp2f(glL[i]) * (acc0 + acc1);
    }
    if (!(ok = mma_wait())) break;
    // ---- HA: dW^T (= -A0) and K~ tiles for MB; dv from A2
    {
      const int i = lt;
      float w[KG_CW], x[KG_CW];
      tldc(KGT_A0, w);
      tldc(KGT_A2, x);
#pragma unroll
      for (int q4 = 0; q4 < KG_CW / 8; ++q4) {
        float t8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) t8[e] = -w[q4 * 8 + e];
        *reinterpret_cast<uint4*>(X + KX_WD + sw_chunk(i, (c0 >> 3) + q4, 128)) = kg_pack8(t8);
      }
#pragma unroll
      for (int e = 0; e < KG_CW; ++e) {   // dv[r][j] = beta_r (T^T dX)[r][j], row lt = j
        const int r = c0 + e;
        if (r < L) a.dv[((size_t)(tok0 + r) * a.HV + hv) * D + i] = __float2bfloat16_rn(bs[r] * x[e]);
      }
    }
#pragma unroll
    for (int it = 0; it < 1024 / KG_THREADS; ++it) {   // K~[r] = rk_r k_r . exp2(G_r)
      const int idx = tid + KG_THREADS * it, r = idx >> 4, c8 = idx & 15;
      float kf[8], y[8];
      kg_unpack8(*reinterpret_cast<const uint4*>(kq + sw_chunk(r, c8, 128)), kf);
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = rk[r] * kf[e] * exp2f(Gm[r * D + 8 * c8 + e]);
      *reinterpret_cast<uint4*>(X + KX_KT + sw_chunk(r, c8, 64)) = kg_pack8(y);
    }
    to_tc();
    // ---- MB: dW K~^T (A0, M = 64), dY^T = dW^T T (A2)
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_ss(tb + KGT_A0, desc_mn(s_wd, 128, ks), desc_k(s_kt, 64, ks), idesc(64, 64, 1, 0), ks > 0);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_ss(tb + KGT_A2, desc_k(s_wd, 128, ks), desc_mn(s_t, 64, ks), idesc(128, 64, 0, 1), ks > 0);
      commit();
    }
    {  // side work: the A1 (dO S^T)^T and A3 (dKd^T) terms into dq^T, dk^T, dG_L and dG^T, which takes
       // over A1's columns for the rest of the value head
      const int i = lt;
      const float GLi = glL[i];
      float kdsum = 0.f;
#pragma unroll 1
      for (int h = 0; h < KG_NH; ++h) {
        const int cb = c0 + 16 * h;
        float p1[16], p3[16], aq[16], ak[16], dg[16];
        tld16c(KGT_A1 + cb, p1);
        tld16c(KGT_A3 + cb, p3);
        if (hh > 0) {
          tld16c(KGT_DQ + cb, aq);
          tld16c(KGT_DK + cb, ak);
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) aq[e] = ak[e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int r = cb + e;
          const float Gri = Gm[r * D + i];
          const float gm = exp2f(Gri), Ee = exp2f(GLi - Gri);
          const float qh = rq[r] * qraw(r, i), kh = rk[r] * kraw(r, i);
          aq[e] = fmaf(a.scale * gm, p1[e], aq[e]);
          ak[e] = fmaf(Ee, p3[e], ak[e]);
          const float kdp = kh * Ee * p3[e];
          dg[e] = a.scale * qh * gm * p1[e] - kdp;
          kdsum += kdp;
        }
        tst16c(KGT_DQ + cb, aq);
        tst16c(KGT_DK + cb, ak);
        tst16c(KGT_DG + cb, dg);
      }
      tmem_wait_st();
      dgl[wg][i] += kdsum;
    }
    if (!(ok = mma_wait())) break;
    // ---- HB: dT = (dX V^T + dW K~^T) diag(beta), dbeta column sums of T . (those), dP tiles; dY terms
    {
      uint32_t u6a[KG_NH][8], u6b[KG_NH][8], u2[KG_NH][8];
      ld_m64(KGT_A5, u6a);
      ld_m64(KGT_A0, u6b);
      ld_m64(KGT_A4, u2);
      float tbs[KG_NH][4];
#pragma unroll
      for (int g = 0; g < KG_NH; ++g)
#pragma unroll
        for (int q = 0; q < 4; ++q) tbs[g][q] = 0.f;
#pragma unroll
      for (int g = 0; g < KG_NH; ++g)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int r = ra + 8 * hr;
#pragma unroll
          for (int hb = 0; hb < 2; ++hb) {
            const int i0 = hb * 4 + hr * 2;   // values i0, i0 + 1: columns cc, cc + 1
            const int cc = c0 + 16 * g + 8 * hb + 2 * (lane & 3);
            float dt[2], dp[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float s6 = __uint_as_float(u6a[g][i0 + e]) + __uint_as_float(u6b[g][i0 + e]);
              dt[e] = bs[cc + e] * s6;
              tbs[g][hb * 2 + e] = fmaf(bf16_at(sm + KG_T, r, cc + e, 64), s6, tbs[g][hb * 2 + e]);
              // the diagonal dP_rr k^_r (into dq^_r) and dP_rr q^_r (into dk^_r) are added exactly in the
              // final pass: their dG terms cancel (q^_r . rowP_r against k^_r . col_r), which the two
              // differently rounded block products would not do
              const bool live = cc + e < r && r < L;
              dp[e] = live ? a.scale * __uint_as_float(u2[g][i0 + e]) : 0.f;
              if (cc + e == r) pdiag[r] = r < L ? a.scale * __uint_as_float(u2[g][i0 + e]) : 0.f;
            }
            const uint32_t off = sw_off(r, cc, 64);
            *reinterpret_cast<uint32_t*>(X + KX_DT + off) = pack_bf16(dt[0], dt[1]);
            *reinterpret_cast<uint32_t*>(X + KX_DP + off) = pack_bf16(dp[0], dp[1]);
            *reinterpret_cast<__nv_bfloat16*>(X + KX_DPT + sw_off(cc, r, 64)) = __float2bfloat16_rn(dp[0]);
            *reinterpret_cast<__nv_bfloat16*>(X + KX_DPT + sw_off(cc + 1, r, 64)) = __float2bfloat16_rn(dp[1]);
          }
        }
      // column sums over the warp's 16 rows: lanes with equal lane & 3 hold the same columns
#pragma unroll
      for (int g = 0; g < KG_NH; ++g)
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int o = 4; o <= 16; o <<= 1) tbs[g][q] += __shfl_xor_sync(0xffffffffu, tbs[g][q], o);
      if (lane < 4) {
#pragma unroll
        for (int g = 0; g < KG_NH; ++g)
#pragma unroll
          for (int q = 0; q < 4; ++q) red[wq][c0 + 16 * g + 8 * (q >> 1) + 2 * lane + (q & 1)] = tbs[g][q];
      }
    }
    {  // dY^T (A2): dk^T += beta gamma . dY, dG^T += beta K~ . dY
      const int i = lt;
#pragma unroll 1
      for (int h = 0; h < KG_NH; ++h) {
        const int cb = c0 + 16 * h;
        float y[16], ak[16], dg[16];
        tld16c(KGT_A2 + cb, y);
        tld16c(KGT_DK + cb, ak);
        tld16c(KGT_DG + cb, dg);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int r = cb + e;
          const float bg = bs[r] * exp2f(Gm[r * D + i]);
          ak[e] = fmaf(bg, y[e], ak[e]);
          dg[e] = fmaf(bg * rk[r] * kraw(r, i), y[e], dg[e]);
        }
        tst16c(KGT_DK + cb, ak);
        tst16c(KGT_DG + cb, dg);
      }
      tmem_wait_st();
    }
    to_tc();
    // ---- M4: R1 = dT T^T (A5)
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_ss(tb + KGT_A5, desc_k(s_dt, 64, ks), desc_k(s_t, 64, ks), idesc(64, 64, 0, 0), ks > 0);
      commit();
    }
    // while M4 runs: the block-relative tiles Lk, Lq (exp2(G_r - gx[blk]) . k^, q^) and Rb (exp2(gx[blk] - G_c) . k^)
#pragma unroll 2
    for (int it = 0; it < 1024 / KG_THREADS; ++it) {
      const int idx = tid + KG_THREADS * it, r = idx >> 4, c8 = idx & 15, bk = r >> 4;
      float kf[8], qf[8], lk[8], lq[8], rb[8];
      kg_unpack8(*reinterpret_cast<const uint4*>(kq + sw_chunk(r, c8, 128)), kf);
      kg_unpack8(*reinterpret_cast<const uint4*>(kq + sw_chunk(64 + r, c8, 128)), qf);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float d = Gm[r * D + 8 * c8 + e] - gx[bk][8 * c8 + e];
        const float lam = exp2f(d), ein = exp2f(-d);
        lk[e] = rk[r] * kf[e] * lam;
        lq[e] = rq[r] * qf[e] * lam;
        rb[e] = rk[r] * kf[e] * ein;
      }
      *reinterpret_cast<uint4*>(X + KX_LK + sw_chunk(r, c8, 64)) = kg_pack8(lk);
      *reinterpret_cast<uint4*>(X + KX_LQ + sw_chunk(r, c8, 64)) = kg_pack8(lq);
      *reinterpret_cast<uint4*>(X + KX_RB + sw_chunk(r, c8, 64)) = kg_pack8(rb);
    }
    if (!(ok = mma_wait())) break;
    {  // R1 -> BF16 tile for M5
      uint32_t u[KG_NH][8];
      ld_m64(KGT_A5, u);
#pragma unroll
      for (int g = 0; g < KG_NH; ++g)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr)
#pragma unroll
          for (int hb = 0; hb < 2; ++hb) {
            const int i0 = hb * 4 + hr * 2, cc = c0 + 16 * g + 8 * hb + 2 * (lane & 3);
            *reinterpret_cast<uint32_t*>(X + KX_R1 + sw_off(ra + 8 * hr, cc, 64)) =
                pack_bf16(__uint_as_float(u[g][i0]), __uint_as_float(u[g][i0 + 1]));
          }
    }
    to_tc();
    // ---- M5: T^T R1 = -dA (A0)
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_ss(tb + KGT_A0, desc_mn(s_t, 64, ks), desc_mn(s_r1, 64, ks), idesc(64, 64, 1, 1), ks > 0);
      commit();
    }
    if (!(ok = mma_wait())) break;
    {  // dA (strictly lower, rows < L): dM = diag(beta) dA tiles; dbeta row sums of dA . M
      uint32_t u[KG_NH][8];
      ld_m64(KGT_A0, u);
      float rsum[2] = {0.f, 0.f};
#pragma unroll
      for (int g = 0; g < KG_NH; ++g)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int r = ra + 8 * hr;
#pragma unroll
          for (int hb = 0; hb < 2; ++hb) {
            const int i0 = hb * 4 + hr * 2, cc = c0 + 16 * g + 8 * hb + 2 * (lane & 3);
            float dm[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const bool live = cc + e < r && r < L;
              const float dA = live ? -__uint_as_float(u[g][i0 + e]) : 0.f;
              rsum[hr] = fmaf(dA, bf16_at(sm + KG_MT, cc + e, r, 64), rsum[hr]);
              dm[e] = bs[r] * dA;
            }
            *reinterpret_cast<uint32_t*>(X + KX_DM + sw_off(r, cc, 64)) = pack_bf16(dm[0], dm[1]);
            *reinterpret_cast<__nv_bfloat16*>(X + KX_DMT + sw_off(cc, r, 64)) = __float2bfloat16_rn(dm[0]);
            *reinterpret_cast<__nv_bfloat16*>(X + KX_DMT + sw_off(cc + 1, r, 64)) = __float2bfloat16_rn(dm[1]);
          }
        }
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        rsum[hr] += __shfl_xor_sync(0xffffffffu, rsum[hr], 1);
        rsum[hr] += __shfl_xor_sync(0xffffffffu, rsum[hr], 2);
      }
      if ((lane & 3) == 0) {
        rowdb[wg][ra] = rsum[0];
        rowdb[wg][ra + 8] = rsum[1];
      }
    }
    // ---- the decay-weighted products, one 16-token block pair per MMA step (K = 16):
    //   Z_b[i][r]  = sum_{c in b} Rb[c][i] dM[r][c]   (r >= 16 b)   rowM_r = Lk-side factor . sum_b F(a, b) Z_b
    //   Zp_b       likewise with dP                                  rowP_r
    //   Y_a[i][c]  = sum_{r in a} Lk[r][i] dM[r][c] + Lq[r][i] dP[r][c]   (c < 16 a + 16)
    //                                                                col_c = sum_{a >= b} F(a, b) Y_a
    // with F(a, b) = exp2(gx[a] - gx[b]) per channel applied in FP32 afterwards, so both sides of every
    // pair (r, c) carry the same BF16 roundings (Lk_r, Rb_c, dM_rc) and cancel in the cumulative sum.
    if (tid == 0) {
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int n = 64 - 16 * b;
        mma_ss(tb + KGT_Z + kZOff[b], desc_mn(s_rb, 64, b), desc_k(s_dm, 64, b, 16 * b), idesc(128, n, 1, 0), 0u);
        mma_ss(tb + kZPColH[b], desc_mn(s_rb, 64, b), desc_k(s_dp, 64, b, 16 * b), idesc(128, n, 1, 0), 0u);
      }
      commit();
    }
    if (!(ok = mma_wait())) break;
    {  // rows: rowM = sum_b F(a, b) Z_b, rowP likewise (block a of the row); then dq^T += lam rowP + dP_rr k^,
       // dk^T += lam rowM + dP_rr q^, dG^T += Lk rowM + Lq rowP
      const int i = lt;
#pragma unroll 1
      for (int h = 0; h < KG_NH; ++h) {
        const int aa = (c0 >> 4) + h, cb = c0 + 16 * h;
        float rm[16], rp[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) rm[e] = rp[e] = 0.f;
        for (int b = 0; b <= aa; ++b) {   // Z_b and Zp_b of the block pair: two loads, one wait
          const float f = b == aa ? 1.f : fab[kg_pair(aa, b)][i];
          uint32_t zm[16], zp[16];
          tmem_ld16_async(taddr(tb, wq * 32, KGT_Z + kZOff[b] + 16 * (aa - b)), zm);
          tmem_ld16_async(taddr(tb, wq * 32, kZPCol[b] + 16 * (aa - b)), zp);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            rm[e] = fmaf(f, __uint_as_float(zm[e]), rm[e]);
            rp[e] = fmaf(f, __uint_as_float(zp[e]), rp[e]);
          }
        }
        float aq[16], ak[16], dg[16];
        {
          uint32_t uq[16], uk[16];
          tmem_ld16_async(taddr(tb, wq * 32, KGT_DQ + cb), uq);
          tmem_ld16_async(taddr(tb, wq * 32, KGT_DK + cb), uk);
          tmem_wait_ld();
          as_float16(uq, aq);
          as_float16(uk, ak);
        }
        tld16c(KGT_DG + cb, dg);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int r = cb + e;
          const float lam = exp2f(Gm[r * D + i] - gx[aa][i]);
          const float kh = rk[r] * kraw(r, i), qh = rq[r] * qraw(r, i);
          aq[e] += lam * rp[e] + pdiag[r] * kh;
          ak[e] += lam * rm[e] + pdiag[r] * qh;
          // (k^ lam and q^ lam as the BF16 Lk, Lq that the column products read: see below)
          dg[e] += bf16_at(X + KX_LK, r, i, 64) * rm[e] + bf16_at(X + KX_LQ, r, i, 64) * rp[e];
        }
        tst16c(KGT_DQ + cb, aq);
        tst16c(KGT_DK + cb, ak);
        tst16c(KGT_DG + cb, dg);
      }
      tmem_wait_st();
    }
    to_tc();   // (the Z columns are read before the Y products overwrite them)
    if (tid == 0) {
#pragma unroll
      for (int aa = 0; aa < 4; ++aa) {
        const int n = 16 * (aa + 1);
        mma_ss(tb + KGT_Z + kYOff[aa], desc_mn(s_lk, 64, aa), desc_k(s_dmt, 64, aa), idesc(128, n, 1, 0), 0u);
        mma_ss(tb + KGT_Z + kYOff[aa], desc_mn(s_lq, 64, aa), desc_k(s_dpt, 64, aa), idesc(128, n, 1, 0), 1u);
      }
      commit();
    }
    if (!(ok = mma_wait())) break;
    {  // columns: col = sum_{a >= b} F(a, b) Y_a (block b of the column); dk^T += ein col, dG^T -= Rb col
       // (Rb = k^ ein in BF16, as the row products read it, so that each pair (r, c) cancels in the
       // cumulative sum to FP32 accuracy)
      const int i = lt;
#pragma unroll 1
      for (int h = 0; h < KG_NH; ++h) {
        const int b = (c0 >> 4) + h, cb = c0 + 16 * h;
        float cl[16], y[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) cl[e] = 0.f;
        int aa = b;
        for (; aa + 1 < 4; aa += 2) {   // two Y blocks per wait
          const float f0 = aa == b ? 1.f : fab[kg_pair(aa, b)][i], f1 = fab[kg_pair(aa + 1, b)][i];
          uint32_t y0[16], y1[16];
          tmem_ld16_async(taddr(tb, wq * 32, KGT_Z + kYOff[aa] + cb), y0);
          tmem_ld16_async(taddr(tb, wq * 32, KGT_Z + kYOff[aa + 1] + cb), y1);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) cl[e] = fmaf(f1, __uint_as_float(y1[e]), fmaf(f0, __uint_as_float(y0[e]), cl[e]));
        }
        if (aa < 4) {
          const float f = aa == b ? 1.f : fab[kg_pair(aa, b)][i];
          tld16c(KGT_Z + kYOff[aa] + cb, y);
#pragma unroll
          for (int e = 0; e < 16; ++e) cl[e] = fmaf(f, y[e], cl[e]);
        }
        float ak[16], dg[16];
        {
          uint32_t uk[16], ug[16];
          tmem_ld16_async(taddr(tb, wq * 32, KGT_DK + cb), uk);
          tmem_ld16_async(taddr(tb, wq * 32, KGT_DG + cb), ug);
          tmem_wait_ld();
          as_float16(uk, ak);
          as_float16(ug, dg);
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int r = cb + e;
          const float ein = exp2f(gx[b][i] - Gm[r * D + i]);
          ak[e] += ein * cl[e];
          dg[e] -= bf16_at(X + KX_RB, r, i, 64) * cl[e];
        }
        tst16c(KGT_DK + cb, ak);
        tst16c(KGT_DG + cb, dg);
      }
      tmem_wait_st();
    }
    {  // dG_L at the last token, then dg = reverse cumulative sum of dG over the chunk's tokens
      const int i = lt;
      float gl = 0.f;
#pragma unroll
      for (int w = 0; w < KG_WG; ++w) gl += dgl[w][i];
      float acc = 0.f;
#pragma unroll 1
      for (int h = KG_NH - 1; h >= 0; --h) {   // this thread's columns, high to low
        const int cb = c0 + 16 * h;
        float dg[16];
        tld16c(KGT_DG + cb, dg);
#pragma unroll
        for (int e = 15; e >= 0; --e) {
          const int r = cb + e;
          float x = r < L ? dg[e] : 0.f;
          if (r == L - 1) x += gl;
          acc += x;
          dg[e] = acc;
        }
        tst16c(KGT_DG + cb, dg);
      }
      cum[wg][i] = acc;
      tmem_wait_st();
    }
    __syncthreads();
    {
      const int i = lt;
      float add = 0.f;   // the later columns' totals
      for (int w = wg + 1; w < KG_WG; ++w) add += cum[w][i];
#pragma unroll 1
      for (int h = 0; h < KG_NH; ++h) {
        const int cb = c0 + 16 * h;
        float dg[16];
        tld16c(KGT_DG + cb, dg);
        if (L == CH) {   // staged as FP32 [64 tokens][128] over the dead tiles, then one TMA store
          float* dgs = reinterpret_cast<float*>(X);
#pragma unroll
          for (int e = 0; e < 16; ++e) dgs[(cb + e) * D + i] = dg[e] + add;
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int r = cb + e;
            if (r < L) a.dg[((size_t)(tok0 + r) * a.HV + hv) * D + i] = dg[e] + add;
          }
        }
      }
      if (tid < L) {
        float db = 0.f;
#pragma unroll
        for (int w = 0; w < KG_WG; ++w) db += rowdb[w][tid];
#pragma unroll
        for (int w = 0; w < 4; ++w) db += red[w][tid];
        a.dbeta[(size_t)(tok0 + tid) * a.HV + hv] = db;
      }
    }
    if (L == CH) fence_async_smem();   // the staged dg, for the copy below
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (L == CH && tid == 0) {   // (the next value head's loads wait for it to have read its tile)
      tma_store_3d(&a.tdg, X, 0, hv, tok0);
      bulk_commit();
    }
  }
  if (ok) {  // ---- item end: the L2-norm backward of the group sums dq^, dk^; dq, dk
    const int i = lt;
    float aq[KG_CW], ak[KG_CW], pq[KG_CW], pk[KG_CW];
    tldc(KGT_DQ, aq);
    tldc(KGT_DK, ak);
#pragma unroll
    for (int e = 0; e < KG_CW; ++e) {
      pq[e] = qraw(c0 + e, i) * aq[e];
      pk[e] = kraw(c0 + e, i) * ak[e];
    }
    if constexpr (KG_CW == 32) {
      const float sq = colsum32(*reinterpret_cast<float(*)[32]>(pq), lane);
      const float sk = colsum32(*reinterpret_cast<float(*)[32]>(pk), lane);
      red[wq][c0 + lane] = sq;
      red[4 + wq][c0 + lane] = sk;
    } else {
      const float sq = kg_colsum16(*reinterpret_cast<float(*)[16]>(pq), lane);
      const float sk = kg_colsum16(*reinterpret_cast<float(*)[16]>(pk), lane);
      if (lane < 16) {
        red[wq][c0 + lane] = sq;
        red[4 + wq][c0 + lane] = sk;
      }
    }
    __syncthreads();
    if (tid < CH) {
      float xq = 0.f, xk = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        xq += red[w][tid];
        xk += red[4 + w][tid];
      }
      const float nq = rq[tid], nk = rk[tid];
      rowdb[0][tid] = xq * nq * nq * nq;
      rowdb[1][tid] = xk * nk * nk * nk;
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < KG_CW; ++e) {
      const int r = c0 + e;
      if (r >= L) continue;
      float oq = aq[e], ok2 = ak[e];
      if (a.l2norm) {
        oq = rq[r] * aq[e] - qraw(r, i) * rowdb[0][r];
        ok2 = rk[r] * ak[e] - kraw(r, i) * rowdb[1][r];
      }
      a.dq[((size_t)(tok0 + r) * a.H + j) * D + i] = __float2bfloat16_rn(oq);
      a.dk[((size_t)(tok0 + r) * a.H + j) * D + i] = __float2bfloat16_rn(ok2);
    }
  }
  if (tid == 0) bulk_wait_all();   // the last dg copy out of shared memory
  if (tid == 0 && !ok) {   // error path (bounded waits): nothing may land in or read this CTA's memory
    if (mma_pend) mbar_drain(&bar_m, mph);
    if (ld_pend) {
      mbar_drain(&bar_g, ldph);
      mbar_drain(&bar_ld, ldph);
    }
    if (qk_pend) mbar_drain(&bar_qk, 0);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, 512);
}

void setup_kda_bwd_attrs() {
  cudaFuncSetAttribute(kda_grad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, KG_SMEM_ALLOC);
}

gdn_status run_kda_prep(const Plan& P, const gdn_problem* p, const void* q, const void* k, const float* g,
                        const float* beta, uint8_t* kb, uint8_t* ws, cudaStream_t s);

static gdn_status run_kda_bwd(const Plan& P, const gdn_problem& pr, const void* q, const void* k, const void* v,
                              const float* g, const float* beta, const int32_t* cu_dev, const void* dO,
                              const void* saved, void* dq, void* dk, void* dv, float* dg, float* dbeta,
                              uint8_t* ws, cudaStream_t s) {
  gdn_status st = run_tables(P, &pr, cu_dev, ws, nullptr, s);
  if (st != GDN_OK) return st;
  launch_check_saved(P, pr, saved, ws, s);
  if (P.NC == 0) return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
  // the per-chunk blocks: the forward's, from a full-form saved set, else formed again (the replay of
  // the decay products and UT blocks); then the adjoint walks
  const uint8_t* sv = static_cast<const uint8_t*>(saved);
  uint8_t* kb = P.form == 3 ? const_cast<uint8_t*>(sv) + P.s_cb : ws + P.o_cb;
  if (P.form != 3) {
    st = run_kda_prep(P, &pr, q, k, g, beta, kb, ws, s);
    if (st != GDN_OK) return st;
  }
  st = run_bwd_walks(P, pr, q, k, dO, kb, 1, saved, nullptr, nullptr, ws, s);
  if (st != GDN_OK) return st;
  Tables t = tables_at(P, ws);
  KdaGradArgs ga;
  memset(&ga, 0, sizeof(ga));
  if (!make_tmap(&ga.tq, q, P.T, P.H) || !make_tmap(&ga.tk, k, P.T, P.H) || !make_tmap(&ga.tv, v, P.T, P.HV) ||
      !make_tmap(&ga.tdo, dO, P.T, P.HV) || !make_tmap_g(&ga.tg, g, P.T, P.HV) ||
      !make_tmap_g(&ga.tdg, dg, P.T, P.HV))
    return GDN_ERR_CUDA;
  ga.g = g;
  ga.beta = beta;
  ga.kb = kb;
  ga.tape = sv + P.s_tape;
  ga.dtape = ws + P.o_dtape;
  ga.vn = sv + P.s_vn;
  ga.dvn = ws + P.o_dvn;
  ga.chunk_tok0 = t.chunk_tok0;
  ga.chunk_len = t.chunk_len;
  ga.dq = static_cast<__nv_bfloat16*>(dq);
  ga.dk = static_cast<__nv_bfloat16*>(dk);
  ga.dv = static_cast<__nv_bfloat16*>(dv);
  ga.dg = dg;
  ga.dbeta = dbeta;
  ga.NC = P.NC;
  ga.H = P.H;
  ga.HV = P.HV;
  ga.G = P.G;
  ga.l2norm = pr.l2norm ? 1 : 0;
  ga.scale = pr.scale;
  ga.err = reinterpret_cast<int*>(ws);
  prof_begin(K_KDA_GRAD, s);
  kda_grad_kernel<<<P.NC * P.H, KG_THREADS, KG_SMEM_ALLOC, s>>>(ga);
  prof_end(K_KDA_GRAD, s);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace gdn

using namespace gdn;

extern "C" gdn_status gdn_kda_bwd(const gdn_problem* prob, const void* q, const void* k, const void* v,
                                  const float* g, const float* beta, const int32_t* cu_dev, const int32_t* cu_host,
                                  const void* dO, const void* saved, void* dq, void* dk, void* dv, float* dg,
                                  float* dbeta, void* workspace, size_t ws_bytes, struct CUstream_st* stream) {
  Plan P;
  gdn_status st = make_kda_plan(prob, cu_host, &P);
  if (st != GDN_OK) return st;
  if (!cu_dev || !workspace || !saved) return GDN_ERR_INVALID_ARG;
  if (P.T > 0 && (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(beta) ||
                  !aligned16(dO) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(dg) ||
                  !aligned16(dbeta)))
    return GDN_ERR_INVALID_ARG;
  if (!aligned16(workspace) || !aligned16(saved)) return GDN_ERR_INVALID_ARG;
  if (ws_bytes < P.ws_bwd) return GDN_ERR_WORKSPACE_TOO_SMALL;
  if (!device_setup()) return GDN_ERR_CUDA;
  return run_kda_bwd(P, *prob, q, k, v, g, beta, cu_dev, dO, saved, dq, dk, dv, dg, dbeta,
                     static_cast<uint8_t*>(workspace), stream);
}
