// gdn_bwd.cu -- backward of the chunked GDN form.
//
// Per chunk (local positions r, S = state entering, dS' = gradient of the
// state leaving the chunk, P = scale), reversing the forward equations
//   V_new = U - W S,  O = P (diag(gamma) Q^ S + Aqk V_new),
//   S' = gamma_L S + Kd^T V_new:
//   dV_new = P Aqk^T dO + Kd dS'
//   dS     = gamma_L dS' + P (diag(gamma) Q^)^T dO - W^T dV_new      (reverse scan)
// and the chunk-local gradients (dq^, dk^, dv, dbeta, dG -> dg) from the
// UT / WY relations W = T diag(beta gamma) K^, U = T diag(beta) V,
// T = (I + A)^-1 (dA = -T^T dT T^T on the strict lower triangle).  These are
// the adjoint walk and the dA / dv and fused-gradient programs of the
// flashinfer Cake GDN pages ("feat(cake_gdn_kcp) ... #8172" page, commit
// notes on the K2 walk, kcp_dav and the fused-gradient program; "#8542" page:
// the backward's merges read the M_seg plane of the forward).
//
// Kernels:
//   bwd_scan_kernel   reverse dS walk per (segment, value head); writes the
//                     BF16 dS' tape (gradient leaving each chunk), or, in the
//                     split's zero-start mode, the adjoint at a segment start
//   merge_bwd_kernel  dS_end(p) = dS_end(p+1) M_{p+1} + B'_{p+1} over segments
//   grad_kernel       per (chunk, q/k head): everything chunk-local, summing
//                     dq^, dk^ over the group's value heads, then the L2-norm
//                     backward
#include "gdn.h"
#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_prof.h"

namespace gdn {

constexpr float kLog2e = 1.4426950408889634f;

bool make_tmap(CUtensorMap* m, const void* base, int64_t T, int heads);
gdn_status run_tables(const Plan& P, const gdn_problem* p, const int32_t* cu_dev, uint8_t* ws, void* saved,
                      cudaStream_t s);
gdn_status run_prep(const Plan& P, const gdn_problem* p, const void* q, const void* k, const float* g,
                    const float* beta, uint8_t* ws, uint8_t* cb, int write_T, cudaStream_t s);

struct BScanArgs {
  CUtensorMap tq, tk, tdo;
  const uint8_t* cb;
  const int* chunk_tok0;
  const int* seg_c0;
  const int* seg_c1;
  const int* seg_split;
  const int* split_seg;
  int HV, G, nsplit, walk;
  float scale;
  uint8_t* dtape;        // [NC][HV][STATE_BYTES]
  uint8_t* dvn;          // [NC][HV][VN_BYTES] dV_new^T tiles (full walks)
  const float* ds_init;  // [nsplit][HV][STATE_F32]: adjoint at the end of split segment i
  float* dbend;          // [nsplit][HV][STATE_F32]
  int* err;
};

struct GradArgs {
  CUtensorMap tq, tk, tv, tdo;
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const float* g;
  const float* beta;
  const uint8_t* cb;
  const uint8_t* tape;    // saved S^T per chunk
  const uint8_t* dtape;   // dS'^T per chunk
  const uint8_t* vn;      // V_new^T per chunk (saved by the forward)
  const uint8_t* dvn;     // dV_new^T per chunk (written by the adjoint walk)
  const int* chunk_tok0;
  const int* chunk_len;
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  float* dg;
  float* dbeta;
  int H, HV, G, l2norm;
  float scale;
  int* err;
};

struct MergeBwdArgs {
  const int* sdoc_first;
  const float* dbend;
  const float* mend;
  float* ds_init;
  int HV;
  int* err;
};

struct CheckArgs {
  const uint8_t* saved;
  SavedHeader expect;
  int* err;
};

// ===========================================================================
// reverse dS scan
// ===========================================================================
constexpr int BS_K = 0, BS_Q = 16384, BS_DO = 32768, BS_TP = 49152, BS_AQK = 57344, BS_SCAL = 65536;
constexpr int BS_STAGE = 66560;
constexpr int BS_DS = 2 * BS_STAGE;           // BF16 dS'^T tile
constexpr int BS_W = BS_DS + STATE_BYTES;     // -W^T tile, SwTile(128 x 64)
constexpr int BS_DV = BS_W + 16384;           // dV_new^T staging, SwTile(128 x 64)
constexpr int BS_SMEM = BS_DV + VN_BYTES;
constexpr int BS_SMEM_ALLOC = BS_SMEM + 1024;
constexpr int BT_DW = 0, BT_DX = 64, BT_DY = 128, BT_DS = 192, BT_ADV = 320, BT_ADO = 352;

__device__ __forceinline__ void store_row128(uint8_t* dst, int row, const float* S) {
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

__device__ __forceinline__ float ld_bf16(const uint8_t* tile, int r, int c, int R) {
  return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(tile + sw_off(r, c, R)));
}

__global__ void __launch_bounds__(128, 1) bwd_scan_kernel(const __grid_constant__ BScanArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full_bar[2], mma_bar;
  __shared__ uint32_t tslot;
  const int tid = threadIdx.x, warp = tid >> 5;
  if (*(volatile int*)a.err) return;

  int seg, hv, split = -1;
  if (!a.walk) {
    seg = blockIdx.x / a.HV;
    hv = blockIdx.x % a.HV;
  } else {  // zero-start reverse walk of the segment after split point `split`
    split = blockIdx.x / a.HV;
    hv = blockIdx.x % a.HV;
    seg = a.split_seg[split] + 1;
  }
  const int kh = hv / a.G;
  const int c0 = a.seg_c0[seg], nch = a.seg_c1[seg] - c0;

  float dS[128];
  {
    const float* src = nullptr;
    if (!a.walk && a.seg_split[seg] >= 0)
      src = a.ds_init + ((size_t)a.seg_split[seg] * a.HV + hv) * STATE_F32 + (size_t)tid * 128;
#pragma unroll
    for (int jj = 0; jj < 128; ++jj) dS[jj] = src ? src[jj] : 0.f;
  }
  uint8_t* ds_tile = sm + BS_DS;
  store_row128(ds_tile, tid, dS);

  if (warp == 0) tmem_alloc(&tslot, 512);
  if (tid == 0) {
    mbar_init(&full_bar[0], 1);
    mbar_init(&full_bar[1], 1);
    mbar_init(&mma_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;");
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tslot;

  // iteration `it` processes chunk c0 + nch - 1 - it
  auto issue = [&](int it) {
    const int ci = c0 + nch - 1 - it;
    uint8_t* st = sm + (it & 1) * BS_STAGE;
    uint64_t* bar = &full_bar[it & 1];
    const int t0 = a.chunk_tok0[ci];
    const uint8_t* cbp = a.cb + ((size_t)ci * a.HV + hv) * CB_BYTES;
    mbar_expect_tx(bar, (uint32_t)BS_STAGE);
    tma_load_3d(st + BS_K, &a.tk, 0, kh, t0, bar);
    tma_load_3d(st + BS_K + 8192, &a.tk, 64, kh, t0, bar);
    tma_load_3d(st + BS_Q, &a.tq, 0, kh, t0, bar);
    tma_load_3d(st + BS_Q + 8192, &a.tq, 64, kh, t0, bar);
    tma_load_3d(st + BS_DO, &a.tdo, 0, hv, t0, bar);
    tma_load_3d(st + BS_DO + 8192, &a.tdo, 64, hv, t0, bar);
    bulk_load(st + BS_TP, cbp + CB_TP, TILE64_BYTES, bar);
    bulk_load(st + BS_AQK, cbp + CB_AQK, TILE64_BYTES, bar);
    bulk_load(st + BS_SCAL, cbp + CB_SCAL, CB_SCAL_BYTES, bar);
  };
  if (tid == 0) {
    if (nch > 0) issue(0);
    if (nch > 1) issue(1);
  }
  uint32_t mph = 0;
  bool ok = true;
  const uint32_t sm_ds = smem_u32(ds_tile), sm_w = smem_u32(sm + BS_W);
  for (int it = 0; it < nch && ok; ++it) {
    const int ci = c0 + nch - 1 - it;
    uint8_t* st = sm + (it & 1) * BS_STAGE;
    const uint32_t a_k = smem_u32(st + BS_K), a_q = smem_u32(st + BS_Q), a_do = smem_u32(st + BS_DO);
    const uint32_t a_tp = smem_u32(st + BS_TP), a_aqk = smem_u32(st + BS_AQK);
    const float* scal = reinterpret_cast<const float*>(st + BS_SCAL);
    ok = __syncthreads_and(mbar_wait(&full_bar[it & 1], (it >> 1) & 1, a.err));
    if (!ok) break;
    const int L = reinterpret_cast<const int*>(scal)[129];
    if (L < CH) {
      for (int idx = tid; idx < (CH - L) * 48; idx += 128) {
        const int t = idx / 48, rem = idx % 48, tile = rem / 16, c8 = rem % 16;
        const int off = tile == 0 ? BS_K : (tile == 1 ? BS_Q : BS_DO);
        *reinterpret_cast<uint4*>(st + off + sw_chunk(L + t, c8, 64)) = make_uint4(0u, 0u, 0u, 0u);
      }
      fence_async_smem();
      __syncthreads();
    }
    tc_fence_after();
    if (tid == 0) {
      // the dS'^T tile (written and fenced last iteration) is this chunk's tape entry
      if (!a.walk) {
        bulk_store(a.dtape + ((size_t)ci * a.HV + hv) * STATE_BYTES, ds_tile, STATE_BYTES);
        bulk_commit();
      }
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_ss(tb + BT_DW, desc_mn(a_k, 64, ks), desc_k(a_tp, 64, ks), idesc(128, 64, 1, 0), ks > 0);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_ss(tb + BT_DX, desc_mn(a_do, 64, ks), desc_mn(a_aqk, 64, ks), idesc(128, 64, 1, 1), ks > 0);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_ss(tb + BT_DY, desc_k(sm_ds, 128, ks), desc_k(a_k, 64, ks), idesc(128, 64, 0, 0), ks > 0);
      mma_commit(&mma_bar);
    }
    {  // (P gamma_r rq_r dO[r][tid]) -> TMEM A operand, while the MMAs run
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t p8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int r = q * 16 + 2 * e;
          p8[e] = pack_bf16(scal[r] * ld_bf16(st + BS_DO, r, tid, 64), scal[r + 1] * ld_bf16(st + BS_DO, r + 1, tid, 64));
        }
        tmem_st8(taddr(tb, warp * 32, BT_ADO + q * 8), p8);
      }
    }
    ok = __syncthreads_and(mbar_wait(&mma_bar, mph, a.err));
    mph ^= 1;
    if (!ok) break;
    tc_fence_after();
    {
      float w[64];
      tmem_ld32(taddr(tb, warp * 32, BT_DW), w);
      tmem_ld32(taddr(tb, warp * 32, BT_DW + 32), w + 32);
      uint8_t* wt = sm + BS_W;
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {
        uint4 v;
        v.x = pack_bf16(-w[c8 * 8 + 0], -w[c8 * 8 + 1]);
        v.y = pack_bf16(-w[c8 * 8 + 2], -w[c8 * 8 + 3]);
        v.z = pack_bf16(-w[c8 * 8 + 4], -w[c8 * 8 + 5]);
        v.w = pack_bf16(-w[c8 * 8 + 6], -w[c8 * 8 + 7]);
        *reinterpret_cast<uint4*>(wt + sw_chunk(tid, c8, 128)) = v;
      }
      const float* kd = scal + 64;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float x[32], y[32];
        tmem_ld32(taddr(tb, warp * 32, BT_DX + h * 32), x);
        tmem_ld32(taddr(tb, warp * 32, BT_DY + h * 32), y);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t p8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int j = q * 16 + 2 * e, r = h * 32 + j;
            p8[e] = pack_bf16(fmaf(a.scale, x[j], kd[r] * y[j]), fmaf(a.scale, x[j + 1], kd[r + 1] * y[j + 1]));
          }
          tmem_st8(taddr(tb, warp * 32, BT_ADV + h * 16 + q * 8), p8);
          if (!a.walk) {
            uint8_t* dvt = sm + BS_DV;
            const int c8 = h * 4 + q * 2;
            *reinterpret_cast<uint4*>(dvt + sw_chunk(tid, c8, 128)) = make_uint4(p8[0], p8[1], p8[2], p8[3]);
            *reinterpret_cast<uint4*>(dvt + sw_chunk(tid, c8 + 1, 128)) = make_uint4(p8[4], p8[5], p8[6], p8[7]);
          }
        }
      }
      tmem_wait_st();
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
      if (!a.walk) {   // this chunk's dV_new^T for the gradient kernel
        bulk_store(a.dvn + ((size_t)ci * a.HV + hv) * VN_BYTES, sm + BS_DV, VN_BYTES);
        bulk_commit();
      }
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_ts(tb + BT_DS, tb + BT_ADV + ks * 8, desc_k(sm_w, 128, ks), idesc(128, 128, 0, 0), ks > 0);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_ts(tb + BT_DS, tb + BT_ADO + ks * 8, desc_mn(a_q, 64, ks), idesc(128, 128, 0, 1), 1u);
      mma_commit(&mma_bar);
      bulk_wait_read();   // the tape copies have read the dS'^T and dV_new^T tiles rewritten next
    }
    ok = __syncthreads_and(mbar_wait(&mma_bar, mph, a.err));
    mph ^= 1;
    if (!ok) break;
    tc_fence_after();
    {
      const float gL = scal[128];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        float x[32];
        tmem_ld32(taddr(tb, warp * 32, BT_DS + h * 32), x);
#pragma unroll
        for (int e = 0; e < 32; ++e) dS[h * 32 + e] = fmaf(gL, dS[h * 32 + e], x[e]);
      }
      store_row128(ds_tile, tid, dS);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && it + 2 < nch) issue(it + 2);
  }
  if (tid == 0) bulk_wait_all();
  if (ok && a.walk) {
    float* dst = a.dbend + ((size_t)split * a.HV + hv) * STATE_F32 + (size_t)tid * 128;
#pragma unroll
    for (int jj = 0; jj < 128; jj += 4)
      *reinterpret_cast<float4*>(dst + jj) = make_float4(dS[jj], dS[jj + 1], dS[jj + 2], dS[jj + 3]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, 512);
}

// dS^T_end(i) = dS^T_end(i+1) M + B'^T(i), walking the split segments of one
// document backwards; M = M_{p+1}, stored transposed (mend[i] = M_{p+1}^T).
__global__ void __launch_bounds__(256) merge_bwd_kernel(MergeBwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  float* Sp = reinterpret_cast<float*>(smem_raw);   // [128][129]
  float* Mt = Sp + 128 * 129;                       // Mt[kk][c] = M[kk][c] = mend[c][kk]
  if (*(volatile int*)a.err) return;
  const int sd = blockIdx.x, hv = blockIdx.y, tid = threadIdx.x;
  const int f0 = a.sdoc_first[sd], f1 = a.sdoc_first[sd + 1];
  const size_t stride = (size_t)a.HV * STATE_F32;
  for (int i = tid; i < STATE_F32; i += 256) {
    const float b = a.dbend[(size_t)(f1 - 1) * stride + (size_t)hv * STATE_F32 + i];
    Sp[(i >> 7) * 129 + (i & 127)] = b;
    a.ds_init[(size_t)(f1 - 1) * stride + (size_t)hv * STATE_F32 + i] = b;
  }
  __syncthreads();
  const int r0 = (tid >> 4) * 8, cc0 = (tid & 15) * 8;
  for (int p = f1 - 2; p >= f0; --p) {
    const float* M = a.mend + (size_t)p * stride + (size_t)hv * STATE_F32;
    const float* B = a.dbend + (size_t)p * stride + (size_t)hv * STATE_F32;
    for (int i = tid; i < STATE_F32; i += 256) Mt[(i & 127) * 129 + (i >> 7)] = M[i];
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
        a.ds_init[(size_t)p * stride + (size_t)hv * STATE_F32 + i] = v;
      }
    __syncthreads();
  }
}

__global__ void check_saved_kernel(CheckArgs a) {
  const SavedHeader* h = reinterpret_cast<const SavedHeader*>(a.saved);
  const SavedHeader& e = a.expect;
  if (h->magic != e.magic || h->version != e.version || h->T != e.T || h->N != e.N || h->H != e.H ||
      h->HV != e.HV || h->dk != e.dk || h->dv != e.dv || h->l2norm != e.l2norm || h->NC != e.NC ||
      h->NSEG != e.NSEG || h->nsplit != e.nsplit || h->seg_len != e.seg_len || h->scale_bits != e.scale_bits ||
      h->cu_hash != e.cu_hash)
    atomicCAS(a.err, 0, ST_SAVED_MISMATCH);
}

// ===========================================================================
// chunk gradients
// ===========================================================================
// Shared memory of the chunk-gradient kernel (bytes; tiles 1024-aligned).
constexpr int GK_Q = 0, GK_K = 16384, GK_KQ = 32768, GK_V = 50176, GK_DO = 66560, GK_DV = 82944,
              GK_VN = 99328, GK_S = 115712, GK_DS = 148480, GK_T = 181248, GK_SCAL = 189440, GK_WD = 190464;
constexpr int GK_SMEM = 206848;
constexpr int GK_SMEM_ALLOC = GK_SMEM + 1024;
constexpr int GK_KQLD = 68;   // row pitch (floats) of the FP32 [QK^T lower | KK^T upper] table
static_assert(GK_KQ + 64 * GK_KQLD * 4 <= GK_V, "KQ table");
// regions reused once their first contents are dead
constexpr int GK_H1 = GK_DO, GK_H2 = GK_DO + 8192;   // after MA (dO dead)
constexpr int GK_DT = GK_DV, GK_R1 = GK_DV + 8192;   // after MA (dV_new dead)
constexpr int GK_F1 = GK_WD, GK_F2 = GK_WD + 8192;   // after MB (dW dead)
// TMEM columns: dq^T, dk^T accumulators of the group, then six 64-column results
constexpr int GT_DQ = 0, GT_DK = 64, GT_A0 = 128, GT_A1 = 192, GT_A2 = 256, GT_A3 = 320, GT_A4 = 384, GT_A5 = 448;

constexpr int GK_NWG = 4;                    // warpgroups; each takes GK_CW of the 64 token columns
constexpr int GK_CW = 64 / GK_NWG;
constexpr int GK_THREADS = 128 * GK_NWG;

// sum over the 32 lanes of a warp of column `lane & 15` of v[16] (fixed order)
__device__ __forceinline__ float colsum16(float (&v)[16], int lane) {
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

__device__ __forceinline__ void store_chunk8(uint8_t* tile, int r, int c8, int R, const float* x) {
  uint4 w;
  w.x = pack_bf16(x[0], x[1]);
  w.y = pack_bf16(x[2], x[3]);
  w.z = pack_bf16(x[4], x[5]);
  w.w = pack_bf16(x[6], x[7]);
  *reinterpret_cast<uint4*>(tile + sw_chunk(r, c8, R)) = w;
}

// One CTA per (chunk, q/k head); its value heads one after another.  Every
// operand of the first MMA group of a value head comes from memory: S and
// dS' from the two tapes, V_new^T from the forward, dV_new^T from the
// adjoint walk, V, dO, and T from the saved UT block.  Per value head:
//   MA  S dV_new^T (= -dW^T), S dO^T, X^T = dV_new^T T, dKd^T = dS' V_new^T,
//       dO V_new^T (-> dAqk), dV_new V^T                       (44 MMAs)
//   MB  dW K^T, Y^T = dW^T T
//   M4  R1 = dT T^T, K^T H1 (+= dq^T), Q^T H2 (+= dk^T)
//   M5  T^T R1 (= -dA)
//   M6  K^T F1 + K^T F2 (+= dk^T)
// Each CUDA-core pass first writes what the next group reads, hands off, and
// does its side work (dv, column-scaled dq / dk terms, per-token partial
// sums) while that group runs.  The next value head's loads are requested as
// soon as the buffers they land in are dead.
__global__ void __launch_bounds__(GK_THREADS, 1) grad_kernel(const __grid_constant__ GradArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t bar_qk, bar_vn, bar_sv, bar_do, bar_dt, mma_bar;
  __shared__ float gall[8][CH], ball[8][CH];   // the group's gates, prefetched (first 8 value heads)
  __shared__ uint32_t tslot;
  __shared__ float rq[CH], rk[CH], Gs[CH], bs[CH], gs[CH], decs[CH], eGr[CH], eGi[CH];
  __shared__ int gsafe;
  __shared__ float part[6][4][CH];             // per-token partial sums, one row per 32-lane quarter
  __shared__ float colC[2][4][CH];             // column sums of C (dAqk . Aqk, dA . A) per quarter
  __shared__ float rowC[GK_NWG][CH], rowB[GK_NWG][CH], sdot[GK_THREADS / 32];
  const int c = blockIdx.x, j = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wg = tid >> 7, w4 = warp & 3;
  const int row = w4 * 32 + lane;          // TMEM lane / M = 128 row of this thread
  const int cb0 = wg * GK_CW;              // first of this thread's GK_CW columns
  const int r64 = w4 * 16 + lane;          // M = 64 row (valid for lane < 16)
  if (*(volatile int*)a.err) return;
  const int tok0 = a.chunk_tok0[c], L = a.chunk_len[c];

  if (warp == 0) tmem_alloc(&tslot, 512);
  if (tid == 0) {
    mbar_init(&bar_qk, 1);
    mbar_init(&bar_vn, 1);
    mbar_init(&bar_sv, 1);
    mbar_init(&bar_do, 1);
    mbar_init(&bar_dt, 1);
    mbar_init(&mma_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;");
  }
  __syncthreads();
  const uint32_t tb = tslot;
  const size_t tile_idx0 = (size_t)c * a.HV;
  auto issue_vn = [&](int hv) {   // V_new^T
    mbar_expect_tx(&bar_vn, (uint32_t)VN_BYTES);
    bulk_load(sm + GK_VN, a.vn + (tile_idx0 + hv) * VN_BYTES, VN_BYTES, &bar_vn);
  };
  auto issue_sv = [&](int hv) {   // S, dS', V and the chunk scalars
    mbar_expect_tx(&bar_sv, (uint32_t)(2 * STATE_BYTES + 16384 + CB_SCAL_BYTES));
    bulk_load(sm + GK_S, a.tape + (tile_idx0 + hv) * STATE_BYTES, STATE_BYTES, &bar_sv);
    bulk_load(sm + GK_DS, a.dtape + (tile_idx0 + hv) * STATE_BYTES, STATE_BYTES, &bar_sv);
    tma_load_3d(sm + GK_V, &a.tv, 0, hv, tok0, &bar_sv);
    tma_load_3d(sm + GK_V + 8192, &a.tv, 64, hv, tok0, &bar_sv);
    bulk_load(sm + GK_SCAL, a.cb + (tile_idx0 + hv) * CB_BYTES + CB_SCAL, CB_SCAL_BYTES, &bar_sv);
  };
  auto issue_do = [&](int hv) {
    mbar_expect_tx(&bar_do, 16384u);
    tma_load_3d(sm + GK_DO, &a.tdo, 0, hv, tok0, &bar_do);
    tma_load_3d(sm + GK_DO + 8192, &a.tdo, 64, hv, tok0, &bar_do);
  };
  auto issue_dt = [&](int hv) {   // dV_new^T and T
    mbar_expect_tx(&bar_dt, (uint32_t)(VN_BYTES + TILE64_BYTES));
    bulk_load(sm + GK_DV, a.dvn + (tile_idx0 + hv) * VN_BYTES, VN_BYTES, &bar_dt);
    bulk_load(sm + GK_T, a.cb + (tile_idx0 + hv) * CB_BYTES + CB_T, TILE64_BYTES, &bar_dt);
  };
  if (tid == 0) {
    mbar_expect_tx(&bar_qk, 32768u);
    tma_load_3d(sm + GK_Q, &a.tq, 0, j, tok0, &bar_qk);
    tma_load_3d(sm + GK_Q + 8192, &a.tq, 64, j, tok0, &bar_qk);
    tma_load_3d(sm + GK_K, &a.tk, 0, j, tok0, &bar_qk);
    tma_load_3d(sm + GK_K + 8192, &a.tk, 64, j, tok0, &bar_qk);
    issue_vn(j * a.G);
    issue_sv(j * a.G);
    issue_do(j * a.G);
    issue_dt(j * a.G);
  }
  for (int i = tid; i < min(a.G, 8) * CH; i += GK_THREADS) {   // gates of the group
    const int hh = i / CH, r = i % CH;
    const size_t gi = (size_t)(tok0 + r) * a.HV + j * a.G + hh;
    gall[hh][r] = r < L ? a.g[gi] : 0.f;
    ball[hh][r] = r < L ? a.beta[gi] : 0.f;
  }
  __syncthreads();

  uint32_t mph = 0;
  bool ok = true;
  auto mma_sync_wait = [&]() -> bool {
    bool r = __syncthreads_and(mbar_wait(&mma_bar, mph, a.err));
    mph ^= 1;
    tc_fence_after();
    return r;
  };
  auto handoff = [&]() {   // generic smem/TMEM writes -> visible to the next MMAs
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  };
  const uint32_t s_q = smem_u32(sm + GK_Q), s_k = smem_u32(sm + GK_K), s_v = smem_u32(sm + GK_V),
                 s_do = smem_u32(sm + GK_DO), s_s = smem_u32(sm + GK_S), s_ds = smem_u32(sm + GK_DS),
                 s_t = smem_u32(sm + GK_T), s_wd = smem_u32(sm + GK_WD), s_dv = smem_u32(sm + GK_DV),
                 s_vn = smem_u32(sm + GK_VN), s_dt = smem_u32(sm + GK_DT), s_r1 = smem_u32(sm + GK_R1),
                 s_h1 = smem_u32(sm + GK_H1), s_h2 = smem_u32(sm + GK_H2), s_f1 = smem_u32(sm + GK_F1),
                 s_f2 = smem_u32(sm + GK_F2);
  const float* scal = reinterpret_cast<const float*>(sm + GK_SCAL);
  float* KQ = reinterpret_cast<float*>(sm + GK_KQ);
  auto tld = [&](int col, float* out) { tmem_ld16(taddr(tb, w4 * 32, col + cb0), out); };
  // issue several TMEM loads, then wait once
  auto tld2 = [&](int c0_, float* o0, int c1_, float* o1) {
    uint32_t r0[16], r1[16];
    tmem_ld16_async(taddr(tb, w4 * 32, c0_ + cb0), r0);
    tmem_ld16_async(taddr(tb, w4 * 32, c1_ + cb0), r1);
    tmem_wait_ld();
    as_float16(r0, o0);
    as_float16(r1, o1);
  };

  float dq_acc[GK_CW], dk_acc[GK_CW];   // the column-scaled dq^T, dk^T terms [row][cb0 + e]
#pragma unroll
  for (int e = 0; e < GK_CW; ++e) dq_acc[e] = dk_acc[e] = 0.f;

  for (int h = 0; h < a.G && ok; ++h) {
    const int hv = j * a.G + h;
    const uint32_t vph = h & 1;   // phase of the per-value-head barriers
    if (h == 0) {
      ok = __syncthreads_and(mbar_wait(&bar_qk, 0, a.err));
      if (!ok) break;
      if (L < CH) {   // zero the Q, K rows past the document end (they hold the next document)
        for (int idx = tid; idx < (CH - L) * 32; idx += GK_THREADS) {
          const int t = idx >> 5, tile = (idx >> 4) & 1, c8 = idx & 15;
          *reinterpret_cast<uint4*>(sm + (tile ? GK_K : GK_Q) + sw_chunk(L + t, c8, 64)) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      if (tid < 128) {   // L2 norms of the q/k rows
        const uint8_t* tile = sm + (tid < 64 ? GK_K : GK_Q);
        const int r = tid & 63;
        float ss = 0.f;
        if (r < L) {   // same summation order as the prep kernel's norms
#pragma unroll
          for (int c8 = 0; c8 < 16; ++c8) {
            const uint4 val = *reinterpret_cast<const uint4*>(tile + sw_chunk(r, c8, 64));
            const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&val);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = __bfloat1622float2(h2[e]);
              ss = fmaf(f.x, f.x, ss);
              ss = fmaf(f.y, f.y, ss);
            }
          }
        }
        const float rn = a.l2norm ? 1.0f / sqrtf(ss + 1e-6f) : 1.0f;
        if (tid < 64) rk[r] = rn;
        else rq[r] = rn;
      }
      // KK^T and QK^T (M = 64) -> the FP32 table: QK^T on and below the diagonal, KK^T above
      handoff();
      if (tid == 0) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          mma_ss(tb + GT_A0, desc_k(s_k, 64, ks), desc_k(s_k, 64, ks), idesc(64, 64, 0, 0), ks > 0);
          mma_ss(tb + GT_A1, desc_k(s_q, 64, ks), desc_k(s_k, 64, ks), idesc(64, 64, 0, 0), ks > 0);
        }
        mma_commit(&mma_bar);
      }
      if (!(ok = mma_sync_wait())) break;
      float kk[GK_CW], qk[GK_CW];
      tld2(GT_A0, kk, GT_A1, qk);
      if (lane < 16) {
#pragma unroll
        for (int e = 0; e < GK_CW; e += 4) {
          const int cc = cb0 + e;
          float4 v;
          v.x = cc + 0 <= r64 ? qk[e + 0] : kk[e + 0];
          v.y = cc + 1 <= r64 ? qk[e + 1] : kk[e + 1];
          v.z = cc + 2 <= r64 ? qk[e + 2] : kk[e + 2];
          v.w = cc + 3 <= r64 ? qk[e + 3] : kk[e + 3];
          *reinterpret_cast<float4*>(KQ + r64 * GK_KQLD + cc) = v;
        }
      }
      tc_fence_before();   // the TMEM reads above precede the first MA
    }
    if (warp == 0) {  // gates of this value head
      const int r0 = 2 * lane, r1 = r0 + 1;
      float g0 = 0.f, g1 = 0.f, b0 = 0.f, b1 = 0.f;
      if (h < 8) {
        g0 = gall[h][r0];
        g1 = gall[h][r1];
        b0 = ball[h][r0];
        b1 = ball[h][r1];
      } else {
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
      // cumulative gate in log2 units (the prep kernel's convention)
      const float G0v = (ex + g0) * kLog2e, G1v = (ex + g0 + g1) * kLog2e;
      Gs[r0] = G0v;
      Gs[r1] = G1v;
      bs[r0] = b0;
      bs[r1] = b1;
      gs[r0] = r0 < L ? exp2f(G0v) : 0.f;
      gs[r1] = r1 < L ? exp2f(G1v) : 0.f;
      // per-token gate factors: e^{G_r - G_j} = eGr[r] eGi[j] when the chunk's range is FP32-safe
      const float Gfirst = __shfl_sync(0xffffffffu, G0v, 0);
      const float Glast = __shfl_sync(0xffffffffu, G1v, 31);
      const bool sf = (Gfirst - Glast) < 100.f;
      eGr[r0] = exp2f(G0v - Gfirst);
      eGr[r1] = exp2f(G1v - Gfirst);
      eGi[r0] = sf ? exp2f(Gfirst - G0v) : 0.f;
      eGi[r1] = sf ? exp2f(Gfirst - G1v) : 0.f;
      decs[r0] = r0 < L ? exp2f(Glast - G0v) : 0.f;
      decs[r1] = r1 < L ? exp2f(Glast - G1v) : 0.f;
      if (lane == 0) gsafe = sf;
    }
    // this value head's tiles
    ok = __syncthreads_and(mbar_wait(&bar_vn, vph, a.err) & mbar_wait(&bar_sv, vph, a.err) &
                           mbar_wait(&bar_do, vph, a.err) & mbar_wait(&bar_dt, vph, a.err));
    if (!ok) break;
    const bool sfac = gsafe;
    auto gamma_rc = [&](int r, int cc) -> float {   // e^{G_r - G_c}, c <= r
      return sfac ? eGr[r] * eGi[cc] : exp2f(Gs[r] - Gs[cc]);
    };
    const float gL = scal[128];
    if (L < CH) {  // zero rows past the document end in the V, dO tiles
      for (int idx = tid; idx < (CH - L) * 32; idx += GK_THREADS) {
        const int t = idx >> 5, tile = (idx >> 4) & 1, c8 = idx & 15;
        *reinterpret_cast<uint4*>(sm + (tile ? GK_DO : GK_V) + sw_chunk(L + t, c8, 64)) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    handoff();
    // ---- MA
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        mma_ss(tb + GT_A4, desc_k(s_do, 64, ks), desc_mn(s_vn, 128, ks), idesc(64, 64, 0, 1), ks > 0);
        mma_ss(tb + GT_A0, desc_mn(s_s, 128, ks), desc_mn(s_dv, 128, ks), idesc(128, 64, 1, 1), ks > 0);
        mma_ss(tb + GT_A1, desc_mn(s_s, 128, ks), desc_k(s_do, 64, ks), idesc(128, 64, 1, 0), ks > 0);
        mma_ss(tb + GT_A3, desc_mn(s_ds, 128, ks), desc_mn(s_vn, 128, ks), idesc(128, 64, 1, 1), ks > 0);
        mma_ss(tb + GT_A5, desc_mn(s_dv, 128, ks), desc_k(s_v, 64, ks), idesc(64, 64, 1, 0), ks > 0);
      }
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_ss(tb + GT_A2, desc_k(s_dv, 128, ks), desc_mn(s_t, 64, ks), idesc(128, 64, 0, 1), ks > 0);
      mma_commit(&mma_bar);
    }
    if (!(ok = mma_sync_wait())) break;
    if (tid == 0 && h + 1 < a.G) issue_vn(hv + 1);   // V_new^T is dead from here on
    // HA: dW^T = -(S dV_new^T) -> shared for MB; X^T kept for the side work
    float x[GK_CW];
    {
      float w[GK_CW];
      tld2(GT_A0, w, GT_A2, x);
#pragma unroll
      for (int q4 = 0; q4 < GK_CW / 8; ++q4) {
        float t8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) t8[e] = -w[q4 * 8 + e];
        store_chunk8(sm + GK_WD, row, (cb0 >> 3) + q4, 128, t8);
      }
    }
    handoff();
    // ---- MB: dW K^T (M = 64), Y^T = dW^T T
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_ss(tb + GT_A0, desc_mn(s_wd, 128, ks), desc_k(s_k, 64, ks), idesc(64, 64, 1, 0), ks > 0);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_ss(tb + GT_A2, desc_k(s_wd, 128, ks), desc_mn(s_t, 64, ks), idesc(128, 64, 0, 1), ks > 0);
      mma_commit(&mma_bar);
    }
    {  // HA side work: dv, the column-scaled dq / dk terms, partial sums for dbeta / dg
      float cb[GK_CW];
      __nv_bfloat16* dvp = a.dv + ((size_t)tok0 * a.HV + hv) * D + row;
#pragma unroll
      for (int e = 0; e < GK_CW; ++e) {
        const int cc = cb0 + e;
        if (cc < L) dvp[(size_t)cc * a.HV * D] = __float2bfloat16_rn(bs[cc] * x[e]);
        cb[e] = ld_bf16(sm + GK_V, cc, row, 64) * x[e];
      }
      const float sb = colsum16(cb, lane);
      float y[GK_CW], z[GK_CW];
      tld2(GT_A1, y, GT_A3, z);   // S dO^T (row = dk index), dKd^T (row = dk index)
#pragma unroll
      for (int e = 0; e < GK_CW; ++e) {
        const int cc = cb0 + e;
        const float pg = a.scale * gs[cc];
        dq_acc[e] = fmaf(pg, y[e], dq_acc[e]);
        dk_acc[e] = fmaf(decs[cc], z[e], dk_acc[e]);
        y[e] = pg * rq[cc] * ld_bf16(sm + GK_Q, cc, row, 64) * y[e];
        z[e] = rk[cc] * ld_bf16(sm + GK_K, cc, row, 64) * z[e];
      }
      const float sg = colsum16(y, lane);
      const float sz = colsum16(z, lane);
      // <S, dS'> over this thread's quarter of the row
      float sd = 0.f;
#pragma unroll
      for (int c8 = wg * (16 / GK_NWG); c8 < (wg + 1) * (16 / GK_NWG); ++c8) {   // 16-byte chunks in swizzle order
        const uint4 sa = *reinterpret_cast<const uint4*>(sm + GK_S + sw_chunk(row, c8, 128));
        const uint4 sb4 = *reinterpret_cast<const uint4*>(sm + GK_DS + sw_chunk(row, c8, 128));
        const __nv_bfloat162* ha = reinterpret_cast<const __nv_bfloat162*>(&sa);
        const __nv_bfloat162* hb = reinterpret_cast<const __nv_bfloat162*>(&sb4);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 fa = __bfloat1622float2(ha[e]), fb = __bfloat1622float2(hb[e]);
          sd = fmaf(fa.x, fb.x, sd);
          sd = fmaf(fa.y, fb.y, sd);
        }
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) sd += __shfl_xor_sync(0xffffffffu, sd, o);
      if (lane == 0) sdot[warp] = sd;
      if (lane < GK_CW) {
        part[0][w4][cb0 + lane] = sb;
        part[1][w4][cb0 + lane] = sg;
        part[2][w4][cb0 + lane] = sz;
      }
    }
    if (!(ok = mma_sync_wait())) break;
    if (tid == 0 && h + 1 < a.G) issue_sv(hv + 1);   // S, dS', V, scalars are dead from here on
    {  // HB: the token-pair terms -> H1, H2, dT for M4; dAqk . Aqk -> row / column sums of C
      float daq[GK_CW], t1[GK_CW], t2[GK_CW];
      tld(GT_A4, daq);
      tld2(GT_A5, t1, GT_A0, t2);
      float cm[GK_CW], rc = 0.f;
      const int r = r64;
      const bool rv = lane < 16;
#pragma unroll
      for (int q4 = 0; q4 < GK_CW / 8; ++q4) {
        float h1[8], h2[8], dt[8];
        const float4 qa = *reinterpret_cast<const float4*>(KQ + (rv ? r : 0) * GK_KQLD + cb0 + q4 * 8);
        const float4 qb = *reinterpret_cast<const float4*>(KQ + (rv ? r : 0) * GK_KQLD + cb0 + q4 * 8 + 4);
        const float qk[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int jj = q4 * 8 + e, cc = cb0 + jj;
          const bool live = rv && cc <= r && r < L;
          const float gam = live ? gamma_rc(r, cc) : 0.f;
          const float dA = live ? a.scale * daq[jj] : 0.f;
          cm[jj] = dA * gam * rq[r & 63] * rk[cc] * qk[e];
          rc += cm[jj];
          h1[e] = rk[cc] * gam * dA;
          h2[e] = rq[r & 63] * gam * dA;
          dt[e] = bs[cc] * fmaf(gs[cc] * rk[cc], t2[jj], t1[jj]);
        }
        if (rv) {
          store_chunk8(sm + GK_H1, r, (cb0 >> 3) + q4, 64, h1);
          store_chunk8(sm + GK_H2, r, (cb0 >> 3) + q4, 64, h2);
          store_chunk8(sm + GK_DT, r, (cb0 >> 3) + q4, 64, dt);
        }
      }
      if (rv) rowC[wg][r] = rc;
      const float cs = colsum16(cm, lane);
      if (lane < GK_CW) colC[0][w4][cb0 + lane] = cs;
    }
    handoff();
    // ---- M4: R1 = dT T^T (M = 64), K^T H1 (+= dq^T), Q^T H2 (+= dk^T)
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        mma_ss(tb + GT_A5, desc_k(s_dt, 64, ks), desc_k(s_t, 64, ks), idesc(64, 64, 0, 0), ks > 0);
        mma_ss(tb + GT_DQ, desc_mn(s_k, 64, ks), desc_k(s_h1, 64, ks), idesc(128, 64, 1, 0), (h > 0 || ks > 0));
        mma_ss(tb + GT_DK, desc_mn(s_q, 64, ks), desc_mn(s_h2, 64, ks), idesc(128, 64, 1, 1), (h > 0 || ks > 0));
      }
      mma_commit(&mma_bar);
    }
    {  // HB side work: Y^T = dW^T T (rows = dk index) -> dk, partial sums
      float yv[GK_CW];
      tld(GT_A2, yv);
#pragma unroll
      for (int e = 0; e < GK_CW; ++e) {
        const int cc = cb0 + e;
        dk_acc[e] = fmaf(bs[cc] * gs[cc], yv[e], dk_acc[e]);
        yv[e] *= rk[cc] * ld_bf16(sm + GK_K, cc, row, 64);
      }
      const float sy = colsum16(yv, lane);
      if (lane < GK_CW) part[3][w4][cb0 + lane] = sy;
    }
    if (!(ok = mma_sync_wait())) break;
    if (tid == 0 && h + 1 < a.G) issue_do(hv + 1);   // the dO region (H1, H2) is dead
    {  // H4: R1 -> shared for M5
      float r1v[GK_CW];
      tld(GT_A5, r1v);
      if (lane < 16) {
#pragma unroll
        for (int q4 = 0; q4 < GK_CW / 8; ++q4) store_chunk8(sm + GK_R1, r64, (cb0 >> 3) + q4, 64, r1v + q4 * 8);
      }
    }
    handoff();
    // ---- M5: T^T R1 (= -dA, M = 64)
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_ss(tb + GT_A0, desc_mn(s_t, 64, ks), desc_mn(s_r1, 64, ks), idesc(64, 64, 1, 1), ks > 0);
      mma_commit(&mma_bar);
    }
    if (!(ok = mma_sync_wait())) break;
    if (tid == 0 && h + 1 < a.G) issue_dt(hv + 1);   // dV_new^T (dT, R1) and T are dead
    {  // H5: dA rows -> F1, F2 for M6; dbeta row terms; dA . A -> column sums of C
      float xa[GK_CW];
      tld(GT_A0, xa);
      const int r = r64;
      const bool rv = lane < 16;
      const float br = bs[r & 63];
      float rb = 0.f, cm[GK_CW];
#pragma unroll
      for (int q4 = 0; q4 < GK_CW / 8; ++q4) {
        float f1[8], f2[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int jj = q4 * 8 + e, cc = cb0 + jj;
          const bool live = rv && cc < r && r < L;
          const float gam = live ? gamma_rc(r, cc) : 0.f;
          const float dA = live ? -xa[jj] : 0.f;
          const float kk = live ? KQ[cc * GK_KQLD + r] : 0.f;   // KK^T[r][cc], kept above the diagonal
          const float base = dA * gam * rk[r & 63] * rk[cc] * kk;   // dA . (A / beta_r)
          rb += base;
          cm[jj] = br * base;
          const float E = dA * br * gam;
          f1[e] = rk[cc] * E;
          f2[e] = rk[r & 63] * E;
        }
        if (rv) {
          store_chunk8(sm + GK_F1, r, (cb0 >> 3) + q4, 64, f1);
          store_chunk8(sm + GK_F2, r, (cb0 >> 3) + q4, 64, f2);
        }
      }
      if (rv) rowB[wg][r] = rb;
      const float cs = colsum16(cm, lane);
      if (lane < GK_CW) colC[1][w4][cb0 + lane] = cs;
    }
    handoff();
    // ---- M6: K^T F1 + K^T F2 (+= dk^T).  Not waited for here: the next
    // group's commit (or the final one) covers it.
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_ss(tb + GT_DK, desc_mn(s_k, 64, ks), desc_k(s_f1, 64, ks), idesc(128, 64, 1, 0), 1u);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_ss(tb + GT_DK, desc_mn(s_k, 64, ks), desc_mn(s_f2, 64, ks), idesc(128, 64, 1, 1), 1u);
    }
    // ---- per-token totals: dbeta, dG -> dg
    if (tid < CH) {
      const int r = tid;
      float sb = 0.f, sg = 0.f, sz = 0.f, sy = 0.f, cr = 0.f, rbs = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        sb += part[0][w][r];
        sg += part[1][w][r];
        sz += part[2][w][r];
        sy += part[3][w][r];
        cr -= colC[0][w][r] + colC[1][w][r];
      }
#pragma unroll
      for (int w = 0; w < GK_NWG; ++w) {
        cr += rowC[w][r];
        rbs += rowB[w][r];
      }
      const float z = decs[r] * sz;
      // row sums - column sums of C = dAqk . Aqk + dA . A (the second row sum is beta_r times rowB)
      float dG = sg - z + bs[r] * gs[r] * sy + cr + bs[r] * rbs;
      const float db = sb + gs[r] * sy + rbs;
      // chunk-end terms: gamma_L <S, dS'> and sum_c z_c
      float zs = z;
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) zs += __shfl_xor_sync(0xffffffffu, zs, o);
      __shared__ float zpart[2], wtot[2];
      if (lane == 0) zpart[warp] = zs;
      named_bar(1, 64);
      if (r == L - 1) {
        float sd = 0.f;
#pragma unroll
        for (int w = 0; w < GK_THREADS / 32; ++w) sd += sdot[w];
        dG += gL * sd + zpart[0] + zpart[1];
      }
      if (r >= L) dG = 0.f;
      // dg_r = sum_{i >= r} dG_i: reverse scan within each warp, then add the later warp's total
      float acc = dG;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float yy = __shfl_down_sync(0xffffffffu, acc, o);
        if (lane + o < 32) acc += yy;
      }
      if (lane == 0) wtot[warp] = acc;
      named_bar(1, 64);
      if (warp == 0) acc += wtot[1];
      if (r < L) {
        a.dg[(size_t)(tok0 + r) * a.HV + hv] = acc;
        a.dbeta[(size_t)(tok0 + r) * a.HV + hv] = db;
      }
    }
    __syncthreads();
  }

  // ---- the MMA-accumulated dq^T, dk^T; L2-norm backward of the group sums; dq, dk
  if (ok) {
    if (tid == 0) mma_commit(&mma_bar);
    ok = mma_sync_wait();
  }
  if (ok) {
    {
      float xq[GK_CW], xk[GK_CW];
      tld2(GT_DQ, xq, GT_DK, xk);
#pragma unroll
      for (int e = 0; e < GK_CW; ++e) {
        dq_acc[e] += xq[e];
        dk_acc[e] += xk[e];
      }
    }
    float pq[GK_CW], pk[GK_CW];
#pragma unroll
    for (int e = 0; e < GK_CW; ++e) {
      const int cc = cb0 + e;
      pq[e] = ld_bf16(sm + GK_Q, cc, row, 64) * dq_acc[e];
      pk[e] = ld_bf16(sm + GK_K, cc, row, 64) * dk_acc[e];
    }
    const float sq = colsum16(pq, lane), sk = colsum16(pk, lane);
    if (lane < GK_CW) {
      part[4][w4][cb0 + lane] = sq;
      part[5][w4][cb0 + lane] = sk;
    }
    __syncthreads();
    __nv_bfloat16* dqp = a.dq + ((size_t)tok0 * a.H + j) * D + row;
    __nv_bfloat16* dkp = a.dk + ((size_t)tok0 * a.H + j) * D + row;
#pragma unroll
    for (int e = 0; e < GK_CW; ++e) {
      const int cc = cb0 + e;
      if (cc >= L) continue;
      float outq = dq_acc[e], outk = dk_acc[e];
      if (a.l2norm) {
        float xq = 0.f, xk = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          xq += part[4][w][cc];
          xk += part[5][w][cc];
        }
        const float nq = rq[cc], nk = rk[cc];
        outq = nq * dq_acc[e] - ld_bf16(sm + GK_Q, cc, row, 64) * xq * nq * nq * nq;
        outk = nk * dk_acc[e] - ld_bf16(sm + GK_K, cc, row, 64) * xk * nk * nk * nk;
      }
      dqp[(size_t)cc * a.H * D] = __float2bfloat16_rn(outq);
      dkp[(size_t)cc * a.H * D] = __float2bfloat16_rn(outk);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, 512);
}

// ===========================================================================
// host side
// ===========================================================================
void setup_bwd_attrs() {
  cudaFuncSetAttribute(bwd_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, BS_SMEM_ALLOC);
  cudaFuncSetAttribute(grad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, GK_SMEM_ALLOC);
  cudaFuncSetAttribute(merge_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 2 * 128 * 129 * 4);
}

gdn_status run_bwd(const Plan& P, const gdn_problem& pr, const void* q, const void* k, const void* v,
                   const float* g, const float* beta, const int32_t* cu_dev, const void* dO, const void* saved,
                   void* dq, void* dk, void* dv, float* dg, float* dbeta, uint8_t* ws, cudaStream_t s) {
  gdn_status st = run_tables(P, &pr, cu_dev, ws, nullptr, s);
  if (st != GDN_OK) return st;
  {
    CheckArgs ca;
    ca.saved = static_cast<const uint8_t*>(saved);
    SavedHeader h;
    memset(&h, 0, sizeof(h));
    h.magic = SAVED_MAGIC;
    h.version = SAVED_VERSION;
    h.T = P.T;
    h.N = P.N;
    h.H = P.H;
    h.HV = P.HV;
    h.dk = pr.dk;
    h.dv = pr.dv;
    h.l2norm = pr.l2norm ? 1 : 0;
    h.NC = P.NC;
    h.NSEG = P.NSEG;
    h.nsplit = P.nsplit;
    h.seg_len = P.seg_len;
    memcpy(&h.scale_bits, &pr.scale, 4);
    h.cu_hash = P.cu_hash;
    ca.expect = h;
    ca.err = reinterpret_cast<int*>(ws);
    prof_begin(K_CHECK_SAVED, s);
    check_saved_kernel<<<1, 1, 0, s>>>(ca);
    prof_end(K_CHECK_SAVED, s);
  }
  if (P.NC == 0) return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
  // the per-chunk UT blocks come from the saved set (written by the forward)
  Tables t = tables_at(P, ws);
  const uint8_t* sv = static_cast<const uint8_t*>(saved);
  BScanArgs ba;
  memset(&ba, 0, sizeof(ba));
  if (!make_tmap(&ba.tq, q, P.T, P.H) || !make_tmap(&ba.tk, k, P.T, P.H) || !make_tmap(&ba.tdo, dO, P.T, P.HV))
    return GDN_ERR_CUDA;
  ba.cb = sv + P.s_cb;
  ba.chunk_tok0 = t.chunk_tok0;
  ba.seg_c0 = t.seg_c0;
  ba.seg_c1 = t.seg_c1;
  ba.seg_split = t.seg_split;
  ba.split_seg = t.split_seg;
  ba.HV = P.HV;
  ba.G = P.G;
  ba.nsplit = P.nsplit;
  ba.scale = pr.scale;
  ba.dtape = ws + P.o_dtape;
  ba.dvn = ws + P.o_dvn;
  ba.ds_init = reinterpret_cast<const float*>(ws + P.o_dsinit);
  ba.dbend = reinterpret_cast<float*>(ws + P.o_dbend);
  ba.err = reinterpret_cast<int*>(ws);
  if (P.nsplit > 0) {
    ba.walk = 1;
    prof_begin(K_BWD_WALK, s);
    bwd_scan_kernel<<<P.nsplit * P.HV, 128, BS_SMEM_ALLOC, s>>>(ba);
    prof_end(K_BWD_WALK, s);
    MergeBwdArgs ma;
    ma.sdoc_first = t.sdoc_first;
    ma.dbend = ba.dbend;
    ma.mend = reinterpret_cast<const float*>(sv + P.s_mseg);
    ma.ds_init = reinterpret_cast<float*>(ws + P.o_dsinit);
    ma.HV = P.HV;
    ma.err = ba.err;
    prof_begin(K_BWD_MERGE, s);
    merge_bwd_kernel<<<dim3(P.nsdoc, P.HV), 256, 2 * 128 * 129 * 4, s>>>(ma);
    prof_end(K_BWD_MERGE, s);
  }
  ba.walk = 0;
  prof_begin(K_BWD_SCAN, s);
  bwd_scan_kernel<<<P.NSEG * P.HV, 128, BS_SMEM_ALLOC, s>>>(ba);
  prof_end(K_BWD_SCAN, s);

  GradArgs ga;
  memset(&ga, 0, sizeof(ga));
  ga.tq = ba.tq;
  ga.tk = ba.tk;
  ga.tdo = ba.tdo;
  if (!make_tmap(&ga.tv, v, P.T, P.HV)) return GDN_ERR_CUDA;
  ga.q = static_cast<const __nv_bfloat16*>(q);
  ga.k = static_cast<const __nv_bfloat16*>(k);
  ga.g = g;
  ga.beta = beta;
  ga.cb = sv + P.s_cb;
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
  ga.H = P.H;
  ga.HV = P.HV;
  ga.G = P.G;
  ga.l2norm = pr.l2norm ? 1 : 0;
  ga.scale = pr.scale;
  ga.err = reinterpret_cast<int*>(ws);
  prof_begin(K_GRAD, s);
  grad_kernel<<<dim3(P.NC, P.H), GK_THREADS, GK_SMEM_ALLOC, s>>>(ga);
  prof_end(K_GRAD, s);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace gdn
