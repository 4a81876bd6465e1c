// gdn_conv1d.cu -- the short causal convolution + SiLU front of the GDN layer.
//
// Over packed documents (restart at every cu_seqlens boundary), per channel c
// of the C packed q/k/v channels, with a depthwise kernel of W <= 4 taps:
//   z[t, c] = b[c] + sum_i w[c, i] x[t - (W-1) + i, c]   (zero before the document start)
//   y[t, c] = z sigma(z)
// and the backward, dz = dy sigma(z) (1 + z (1 - sigma(z))):
//   dx[s, c] = sum_i w[c, i] dz[s + (W-1) - i, c]  (inside s's document)
//   dw[c, i] = sum_t dz[t, c] x[t - (W-1) + i, c],  db[c] = sum_t dz[t, c]
// The pages time their GDN layer with this convolution over the 10,240 packed
// q/k/v channels in front ("#8542" page: the B23 shape description and the
// family's conv1d + SiLU training backend; its save-set table keeps at most
// three history rows, a four-tap kernel).
//
// Both directions are bandwidth-bound: a CTA of 128 threads owns 512
// channels (four BF16 channels, one 8-byte vector, per thread) and a
// contiguous token range, which it walks in order with the last W - 1 input
// rows (and, backward, the last W values of dz) in registers, so every
// element is read from HBM once plus a halo of W - 1 rows per range.  The
// forward requests rows in batches of 16, one batch ahead of their use, over
// ranges of 256 tokens.  The backward (ranges of 1,024 tokens) has its x and dy
// rows brought into a ring of three shared-memory stages of 8 rows by bulk
// copies; it writes per-range partial sums of dw and db, and a second kernel
// adds them in range order, so the result does not depend on scheduling.  Its
// workspace opens with a 16-byte status word (gdn_device_status reads it).
#include <algorithm>
#include <cstring>
#include <mutex>

#include "gdn.h"
#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_prof.h"

namespace gdn {

constexpr int CV_THREADS = 128;
constexpr int CV_VEC = 4;                         // channels per thread
constexpr int CV_CH = CV_THREADS * CV_VEC;        // channels per CTA
constexpr int CV_MAXW = 4;
constexpr int CV_UF = 16;                         // rows requested together (forward)
constexpr int CV_RF = 256;                        // tokens per range (forward)
constexpr int CV_RB = 1024;                       // tokens per range (backward: one dw / db partial each)
// backward: the x and dy rows land in a ring of shared-memory stages by bulk copies, so the bytes
// in flight do not cost registers
constexpr int CV_NS = 3;                          // stages in the ring
constexpr int CV_RSB = 8;                         // rows per stage (x and dy)
constexpr int CV_ROWB = CV_CH * 2;                // bytes of one CTA row of one tensor
constexpr int CV_SMEM_B = CV_NS * 2 * CV_RSB * CV_ROWB;   // 48 KB
constexpr int CV_WS_HEAD = 16;                    // the backward workspace opens with the status word

struct ConvArgs {
  CUtensorMap tx, tdy;   // the backward's row boxes of x and dy (when tma is set)
  const __nv_bfloat16* x;
  const float* w;        // [C][W]
  const float* b;        // [C] or null
  const int* cu;         // [N+1]
  const __nv_bfloat16* dy;
  __nv_bfloat16* y;      // forward output
  __nv_bfloat16* dx;     // backward output
  float* part;           // [S][W+1][C] partial dw (rows 0..W-1) and db (row W) per token range
  int* err;              // device status word (backward)
  float* dw;             // [C][W]
  float* db;             // [C]
  int64_t T;
  int N, C, W, R;        // R: tokens per range (grid.y ranges)
  int tma;               // backward: stages land as two TMA boxes (C a multiple of 256), else row copies
};

__device__ __forceinline__ uint2 ld_raw(const __nv_bfloat16* p) {
  return __ldg(reinterpret_cast<const uint2*>(p));
}
__device__ __forceinline__ void unpack_row(const uint2 u, float (&v)[CV_VEC]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int e = 0; e < CV_VEC / 2; ++e) {
    const float2 f = __bfloat1622float2(h[e]);
    v[2 * e] = f.x;
    v[2 * e + 1] = f.y;
  }
}
__device__ __forceinline__ void ld_row(const __nv_bfloat16* p, float (&v)[CV_VEC]) { unpack_row(ld_raw(p), v); }
__device__ __forceinline__ void st_row(__nv_bfloat16* p, const float (&v)[CV_VEC]) {
  uint2 u;
  u.x = pack_bf16(v[0], v[1]);
  u.y = pack_bf16(v[2], v[3]);
  *reinterpret_cast<uint2*>(p) = u;
}
// 1 / (1 + e^{-z}) with the fast exponential and division (a few ulp; the result is rounded to
// BF16 or feeds an FP32 gradient)
__device__ __forceinline__ float sigmoidf(float z) { return __fdividef(1.0f, 1.0f + __expf(-z)); }

// the document containing token t: the largest d with cu[d] <= t (skipping empty documents)
__device__ __forceinline__ int doc_of(const int* cu, int N, int64_t t) {
  int lo = 0, hi = N;   // cu[lo] <= t < cu[hi] (t < T = cu[N])
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cu[mid] <= t) lo = mid;
    else hi = mid;
  }
  return lo;
}

// One thread's state for W taps: the taps and bias of its channels, the last W - 1 input rows
// (hist[W-2] the newest; zero before the document start), and the document bookkeeping.
template <int W>
struct ConvThread {
  static constexpr int H = W > 1 ? W - 1 : 1;
  float w[W][CV_VEC], b[CV_VEC];
  float hist[H][CV_VEC];
  int start, next, d;

  __device__ __forceinline__ void setup(const ConvArgs& a, int c0, int64_t lo) {
#pragma unroll
    for (int e = 0; e < CV_VEC; ++e) {
#pragma unroll
      for (int i = 0; i < W; ++i) w[i][e] = a.w[(size_t)(c0 + e) * W + i];
      b[e] = a.b ? a.b[c0 + e] : 0.f;
    }
    d = doc_of(a.cu, a.N, lo);
    start = a.cu[d];
    next = a.cu[d + 1];
#pragma unroll
    for (int j = 0; j < H; ++j) {   // hist[j] = x[lo - (W-1) + j]
      const int64_t s = lo - (W - 1) + j;
      if (W > 1 && s >= start) ld_row(a.x + s * a.C + c0, hist[j]);
      else
#pragma unroll
        for (int e = 0; e < CV_VEC; ++e) hist[j][e] = 0.f;
    }
  }
  // advance the document bookkeeping to token t; a new document clears the history
  __device__ __forceinline__ void enter(const ConvArgs& a, int64_t t) {
    if (t < next) return;
    while (d + 1 < a.N && a.cu[d + 1] <= t) ++d;
    start = a.cu[d];
    next = a.cu[d + 1];
#pragma unroll
    for (int j = 0; j < H; ++j)
#pragma unroll
      for (int e = 0; e < CV_VEC; ++e) hist[j][e] = 0.f;
  }
  // z of the row xt; xs[i] = the input tap i multiplies; then xt joins the history
  // (channels in pairs: one paired FMA per tap and pair, each half rounding as fmaf)
  __device__ __forceinline__ void step(const float (&xt)[CV_VEC], float (&z)[CV_VEC], float (&xs)[W][CV_VEC]) {
#pragma unroll
    for (int e = 0; e < CV_VEC; ++e) {
#pragma unroll
      for (int i = 0; i < W - 1; ++i) xs[i][e] = hist[i][e];
      xs[W - 1][e] = xt[e];
    }
#pragma unroll
    for (int e = 0; e < CV_VEC; e += 2) {
      float a0 = b[e], a1 = b[e + 1];
#pragma unroll
      for (int i = 0; i < W; ++i) fma2v(a0, a1, w[i][e], w[i][e + 1], xs[i][e], xs[i][e + 1]);
      z[e] = a0;
      z[e + 1] = a1;
    }
#pragma unroll
    for (int e = 0; e < CV_VEC; ++e) {
#pragma unroll
      for (int j = 0; j + 1 < W - 1; ++j) hist[j][e] = hist[j + 1][e];
      if (W > 1) hist[H - 1][e] = xt[e];
    }
  }
};

// one forward row: y[t] from x[t] and the history
template <int W>
__device__ __forceinline__ void fwd_row(const ConvArgs& a, ConvThread<W>& th, int64_t t, uint2 xraw, int c0) {
  th.enter(a, t);
  float xt[CV_VEC], z[CV_VEC], xs[W][CV_VEC], y[CV_VEC];
  unpack_row(xraw, xt);
  th.step(xt, z, xs);
#pragma unroll
  for (int e = 0; e < CV_VEC; e += 2) mul2v(y[e], y[e + 1], z[e], z[e + 1], sigmoidf(z[e]), sigmoidf(z[e + 1]));
  st_row(a.y + t * a.C + c0, y);
}

template <int W>
__global__ void __launch_bounds__(CV_THREADS) conv_fwd_kernel(const ConvArgs a) {
  const int c0 = (blockIdx.x * CV_THREADS + threadIdx.x) * CV_VEC;
  const int64_t lo = (int64_t)blockIdx.y * a.R, hi = min(a.T, lo + a.R);
  if (c0 >= a.C || lo >= hi) return;
  ConvThread<W> th;
  th.setup(a, c0, lo);
  // rows are requested one batch ahead of their use
  uint2 nx[CV_UF];
#pragma unroll
  for (int u = 0; u < CV_UF; ++u)
    if (lo + u < hi) nx[u] = ld_raw(a.x + (lo + u) * a.C + c0);
  for (int64_t t0 = lo; t0 < hi; t0 += CV_UF) {
    uint2 xr[CV_UF];
#pragma unroll
    for (int u = 0; u < CV_UF; ++u) {
      xr[u] = nx[u];
      if (t0 + CV_UF + u < hi) nx[u] = ld_raw(a.x + (t0 + CV_UF + u) * a.C + c0);
    }
#pragma unroll
    for (int u = 0; u < CV_UF; ++u) {
      const int64_t t = t0 + u;
      if (t >= hi) break;
      fwd_row<W>(a, th, t, xr[u], c0);
    }
  }
}

// Backward over the range [lo, hi): dz for rows [lo, hi + W - 1) (the last W - 1 only feed dx of
// rows below hi), dx for rows [lo, hi), partial dw / db over rows [lo, hi).  BwdState holds a
// thread's window of dz and its partial sums; row() takes one row t.
template <int W>
struct BwdState {
  float dzw[W][CV_VEC];   // dz of rows t - (W-1) .. t (dzw[W-1] the newest)
  int dsw[W];             // the document start of each of those rows (-1: past the end)
  float pw[W][CV_VEC], pb[CV_VEC];

  __device__ __forceinline__ void init() {
#pragma unroll
    for (int j = 0; j < W; ++j) {
      dsw[j] = -1;
#pragma unroll
      for (int e = 0; e < CV_VEC; ++e) dzw[j][e] = 0.f;
    }
#pragma unroll
    for (int e = 0; e < CV_VEC; ++e) {
      pb[e] = 0.f;
#pragma unroll
      for (int i = 0; i < W; ++i) pw[i][e] = 0.f;
    }
  }
  __device__ __forceinline__ void row(const ConvArgs& a, ConvThread<W>& th, int64_t t, int64_t lo, int64_t hi,
                                      uint2 xraw, uint2 graw, int c0) {
    float dz[CV_VEC];
    int ds = -1;
    if (t < a.T) {
      th.enter(a, t);
      ds = th.start;
      float xt[CV_VEC], gt[CV_VEC], z[CV_VEC], xs[W][CV_VEC];
      unpack_row(xraw, xt);
      unpack_row(graw, gt);
      th.step(xt, z, xs);
#pragma unroll
      for (int e = 0; e < CV_VEC; e += 2) {   // dz = (dy sg) (1 + z (1 - sg)), channels in pairs
        const float s0 = sigmoidf(z[e]), s1 = sigmoidf(z[e + 1]);
        float u0, u1, v0 = 1.f, v1 = 1.f, p0, p1;
        fma2_to(u0, u1, -1.f, s0, s1, 1.f, 1.f);   // 1 - sg
        fma2v(v0, v1, z[e], z[e + 1], u0, u1);      // 1 + z (1 - sg)
        mul2v(p0, p1, gt[e], gt[e + 1], s0, s1);
        mul2v(dz[e], dz[e + 1], p0, p1, v0, v1);
      }
      if (t < hi) {
#pragma unroll
        for (int e = 0; e < CV_VEC; e += 2) {
          fma2v(pb[e], pb[e + 1], dz[e], dz[e + 1], 1.f, 1.f);   // (dz times 1, plus pb: exactly pb + dz)
#pragma unroll
          for (int i = 0; i < W; ++i) fma2v(pw[i][e], pw[i][e + 1], dz[e], dz[e + 1], xs[i][e], xs[i][e + 1]);
        }
      }
    } else {
#pragma unroll
      for (int e = 0; e < CV_VEC; ++e) dz[e] = 0.f;
    }
#pragma unroll
    for (int j = 0; j + 1 < W; ++j) {
      dsw[j] = dsw[j + 1];
#pragma unroll
      for (int e = 0; e < CV_VEC; ++e) dzw[j][e] = dzw[j + 1][e];
    }
    dsw[W - 1] = ds;
#pragma unroll
    for (int e = 0; e < CV_VEC; ++e) dzw[W - 1][e] = dz[e];
    // dx of row s = t - (W-1), the oldest slot: tap i sees dz of row s + (W-1) - i, slot W-1-i,
    // when that row is in s's document
    const int64_t s = t - (W - 1);
    if (s >= lo && s < hi) {
      float dx[CV_VEC];
#pragma unroll
      for (int e = 0; e < CV_VEC; e += 2) {
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int i = W - 1; i >= 0; --i)
          if (dsw[W - 1 - i] == dsw[0])
            fma2v(a0, a1, th.w[i][e], th.w[i][e + 1], dzw[W - 1 - i][e], dzw[W - 1 - i][e + 1]);
        dx[e] = a0;
        dx[e + 1] = a1;
      }
      st_row(a.dx + s * a.C + c0, dx);
    }
  }
  __device__ __forceinline__ void finish(const ConvArgs& a, int c0) {
    float* pp = a.part + (size_t)blockIdx.y * (W + 1) * a.C + c0;
#pragma unroll
    for (int i = 0; i < W; ++i)
      *reinterpret_cast<float4*>(pp + (size_t)i * a.C) = make_float4(pw[i][0], pw[i][1], pw[i][2], pw[i][3]);
    *reinterpret_cast<float4*>(pp + (size_t)W * a.C) = make_float4(pb[0], pb[1], pb[2], pb[3]);
  }
};

// The backward: thread 0 keeps CV_NS - 1 stages of rows in flight (one bulk copy of the
// CTA's channels per row and tensor, the x rows of a stage then its dy rows); every thread reads
// its 8 bytes of each row from shared memory.
template <int W>
__global__ void __launch_bounds__(CV_THREADS) conv_bwd_kernel(const __grid_constant__ ConvArgs a) {
  extern __shared__ __align__(128) uint8_t cv_sm[];
  __shared__ uint64_t full[CV_NS];
  const int cb = blockIdx.x * CV_CH, nchan = min(CV_CH, a.C - cb);
  const int c0 = cb + threadIdx.x * CV_VEC;
  const bool on = c0 < a.C;
  const int64_t lo = (int64_t)blockIdx.y * a.R, hi = min(a.T, lo + a.R);
  if (lo >= hi || *(volatile int*)a.err) return;
  const int64_t end = hi + W - 1, lim = min(end, a.T);
  const int nst = (int)((end - lo + CV_RSB - 1) / CV_RSB);
  constexpr int STAGE = 2 * CV_RSB * CV_ROWB;   // x rows, then dy rows
  if (threadIdx.x == 0) {
#pragma unroll
    for (int i = 0; i < CV_NS; ++i) mbar_init(&full[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;");
  }
  __syncthreads();
  auto issue = [&](int st) {   // thread 0: the rows of stage st below lim into slot st % CV_NS
    const int64_t r0 = lo + (int64_t)st * CV_RSB;
    const int64_t left = lim - r0;
    const int nr = left <= 0 ? 0 : (left < CV_RSB ? (int)left : CV_RSB);
    uint8_t* base = cv_sm + (st % CV_NS) * STAGE;
    uint64_t* bar = &full[st % CV_NS];
    if (a.tma) {   // one box per tensor: CV_RSB rows of this CTA's 512 channels (past T or C: zero)
      mbar_expect_tx(bar, (uint32_t)(2 * CV_RSB * CV_ROWB));
      tma_load_3d(base, &a.tx, 0, 2 * (int)blockIdx.x, (int)r0, bar);
      tma_load_3d(base + CV_RSB * CV_ROWB, &a.tdy, 0, 2 * (int)blockIdx.x, (int)r0, bar);
      return;
    }
    mbar_expect_tx(bar, (uint32_t)(2 * nr * nchan * 2));
    for (int r = 0; r < nr; ++r) {
      bulk_load(base + r * CV_ROWB, a.x + (r0 + r) * a.C + cb, nchan * 2, bar);
      bulk_load(base + (CV_RSB + r) * CV_ROWB, a.dy + (r0 + r) * a.C + cb, nchan * 2, bar);
    }
  };
  if (threadIdx.x == 0)
    for (int st = 0; st < min(CV_NS - 1, nst); ++st) issue(st);
  ConvThread<W> th;
  if (on) th.setup(a, c0, lo);
  BwdState<W> bs;
  bs.init();
  for (int st = 0; st < nst; ++st) {
    if (threadIdx.x == 0 && st + CV_NS - 1 < nst) issue(st + CV_NS - 1);   // into the slot freed last
    if (!__syncthreads_and(mbar_wait(&full[st % CV_NS], (st / CV_NS) & 1, a.err))) {
      // error path (bounded): the copies still landing in the other slots land before the CTA's memory
      // goes (of a slot's two phase parities one completed last; the other completes when its copy
      // lands, else its wait runs out)
      if (threadIdx.x == 0)
        for (int i = 0; i < CV_NS; ++i) {
          mbar_drain(&full[i], 0);
          mbar_drain(&full[i], 1);
        }
      return;
    }
    const uint8_t* base = cv_sm + (st % CV_NS) * STAGE + threadIdx.x * 8;
    if (on) {
#pragma unroll
      for (int u = 0; u < CV_RSB; ++u) {
        const int64_t t = lo + (int64_t)st * CV_RSB + u;
        if (t >= end) break;
        uint2 xr = make_uint2(0u, 0u), gr = make_uint2(0u, 0u);
        if (t < lim) {
          xr = *reinterpret_cast<const uint2*>(base + u * CV_ROWB);
          gr = *reinterpret_cast<const uint2*>(base + (CV_RSB + u) * CV_ROWB);
        }
        bs.row(a, th, t, lo, hi, xr, gr, c0);
      }
    }
    __syncthreads();   // every thread is done with the slot
  }
  if (on) bs.finish(a, c0);
}

// dw, db: the ranges' partial sums added in range order
__global__ void __launch_bounds__(256) conv_reduce_kernel(const ConvArgs a, int S) {
  const int c = blockIdx.x * 256 + threadIdx.x;
  if (c >= a.C) return;
  for (int i = 0; i <= a.W; ++i) {
    float acc = 0.f;
    for (int s = 0; s < S; ++s) acc += a.part[((size_t)s * (a.W + 1) + i) * a.C + c];
    if (i < a.W) a.dw[(size_t)c * a.W + i] = acc;
    else if (a.db) a.db[c] = acc;
  }
}

// token ranges of R tokens (the last one shorter): S of them
static int conv_ranges(int64_t T, int R) { return (int)((T + R - 1) / R); }

// the backward kernel's shared memory (48 KB dynamic plus its barriers) needs the opt-in, once per
// device
static bool conv_setup() {
  static std::mutex mu;
  static bool done[128] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return false;
  std::lock_guard<std::mutex> lk(mu);
  if (!done[dev]) {
    bool ok = cudaFuncSetAttribute(conv_bwd_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   CV_SMEM_B) == cudaSuccess;
    ok = ok && cudaFuncSetAttribute(conv_bwd_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    CV_SMEM_B) == cudaSuccess;
    ok = ok && cudaFuncSetAttribute(conv_bwd_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    CV_SMEM_B) == cudaSuccess;
    ok = ok && cudaFuncSetAttribute(conv_bwd_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    CV_SMEM_B) == cudaSuccess;
    if (!ok) return false;
    done[dev] = true;
  }
  return true;
}

}  // namespace gdn

using namespace gdn;

extern "C" {

static gdn_status conv_check(const gdn_conv_problem* p, const int32_t* cu) {
  if (!p || !cu) return GDN_ERR_INVALID_ARG;
  // C a multiple of 8: a row of a CTA's channels is a whole number of 16-byte units (bulk copies)
  if (p->N < 1 || p->C <= 0 || p->C % 8 != 0 || p->W < 1 || p->W > CV_MAXW || p->T < 0)
    return p->W > CV_MAXW ? GDN_ERR_UNSUPPORTED : GDN_ERR_INVALID_ARG;
  if (cu[0] != 0 || (int64_t)cu[p->N] != p->T) return GDN_ERR_INVALID_ARG;
  for (int i = 0; i < p->N; ++i)
    if (cu[i + 1] < cu[i]) return GDN_ERR_INVALID_ARG;
  return GDN_OK;
}

static bool al16(const void* q) { return q && ((uintptr_t)q & 15) == 0; }

gdn_status gdn_conv1d_workspace_bytes(const gdn_conv_problem* p, const int32_t* cu_host, size_t* ws_bytes) {
  gdn_status st = conv_check(p, cu_host);
  if (st != GDN_OK) return st;
  if (!ws_bytes) return GDN_ERR_INVALID_ARG;
  *ws_bytes = CV_WS_HEAD + (p->T > 0 ? (size_t)conv_ranges(p->T, CV_RB) * (p->W + 1) * p->C * sizeof(float) : 0);
  return GDN_OK;
}

gdn_status gdn_conv1d_fwd(const gdn_conv_problem* p, const void* x, const float* w, const float* b,
                          const int32_t* cu_dev, const int32_t* cu_host, void* y, struct CUstream_st* stream) {
  gdn_status st = conv_check(p, cu_host);
  if (st != GDN_OK) return st;
  if (!cu_dev || !al16(w) || (b && !al16(b))) return GDN_ERR_INVALID_ARG;
  if (p->T == 0) return GDN_OK;
  if (!al16(x) || !al16(y)) return GDN_ERR_INVALID_ARG;
  ConvArgs a;
  memset(&a, 0, sizeof(a));
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.w = w;
  a.b = b;
  a.cu = cu_dev;
  a.y = static_cast<__nv_bfloat16*>(y);
  a.T = p->T;
  a.N = p->N;
  a.C = p->C;
  a.W = p->W;
  a.R = CV_RF;
  const int S = conv_ranges(p->T, CV_RF);
  if (S > 65535) return GDN_ERR_UNSUPPORTED;   // grid.y: more than 16.7 M tokens
  const dim3 grid((p->C + CV_CH - 1) / CV_CH, S);
  prof_begin(K_CONV_FWD, stream);
  switch (p->W) {
    case 1: conv_fwd_kernel<1><<<grid, CV_THREADS, 0, stream>>>(a); break;
    case 2: conv_fwd_kernel<2><<<grid, CV_THREADS, 0, stream>>>(a); break;
    case 3: conv_fwd_kernel<3><<<grid, CV_THREADS, 0, stream>>>(a); break;
    default: conv_fwd_kernel<4><<<grid, CV_THREADS, 0, stream>>>(a); break;
  }
  prof_end(K_CONV_FWD, stream);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status gdn_conv1d_bwd(const gdn_conv_problem* p, const void* x, const float* w, const float* b,
                          const int32_t* cu_dev, const int32_t* cu_host, const void* dy, void* dx, float* dw,
                          float* db, void* workspace, size_t ws_bytes, struct CUstream_st* stream) {
  gdn_status st = conv_check(p, cu_host);
  if (st != GDN_OK) return st;
  if (!cu_dev || !al16(w) || (b && !al16(b)) || !al16(dw) || (db && !al16(db))) return GDN_ERR_INVALID_ARG;
  size_t need = 0;
  gdn_conv1d_workspace_bytes(p, cu_host, &need);
  if (ws_bytes < need) return GDN_ERR_WORKSPACE_TOO_SMALL;
  if (!al16(workspace)) return GDN_ERR_INVALID_ARG;
  if (p->T > 0 && (!al16(x) || !al16(dy) || !al16(dx))) return GDN_ERR_INVALID_ARG;
  if (cudaMemsetAsync(workspace, 0, CV_WS_HEAD, stream) != cudaSuccess) return GDN_ERR_CUDA;   // status OK
  if (p->T == 0) {   // no tokens: zero gradients of the taps and the bias
    if (cudaMemsetAsync(dw, 0, sizeof(float) * (size_t)p->C * p->W, stream) != cudaSuccess) return GDN_ERR_CUDA;
    if (db && cudaMemsetAsync(db, 0, sizeof(float) * (size_t)p->C, stream) != cudaSuccess) return GDN_ERR_CUDA;
    return GDN_OK;
  }
  ConvArgs a;
  memset(&a, 0, sizeof(a));
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.w = w;
  a.b = b;
  a.cu = cu_dev;
  a.dy = static_cast<const __nv_bfloat16*>(dy);
  a.dx = static_cast<__nv_bfloat16*>(dx);
  a.err = static_cast<int*>(workspace);
  a.part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + CV_WS_HEAD);
  a.dw = dw;
  a.db = db;
  a.T = p->T;
  a.N = p->N;
  a.C = p->C;
  a.W = p->W;
  a.R = CV_RB;
  a.tma = p->C % 256 == 0 && make_tmap_rows(&a.tx, x, p->T, p->C, CV_RSB) &&
          make_tmap_rows(&a.tdy, dy, p->T, p->C, CV_RSB);
  const int S = conv_ranges(p->T, CV_RB);
  const dim3 grid((p->C + CV_CH - 1) / CV_CH, S);
  if (!conv_setup()) return GDN_ERR_CUDA;
  prof_begin(K_CONV_BWD, stream);
  switch (p->W) {
    case 1: conv_bwd_kernel<1><<<grid, CV_THREADS, CV_SMEM_B, stream>>>(a); break;
    case 2: conv_bwd_kernel<2><<<grid, CV_THREADS, CV_SMEM_B, stream>>>(a); break;
    case 3: conv_bwd_kernel<3><<<grid, CV_THREADS, CV_SMEM_B, stream>>>(a); break;
    default: conv_bwd_kernel<4><<<grid, CV_THREADS, CV_SMEM_B, stream>>>(a); break;
  }
  conv_reduce_kernel<<<(p->C + 255) / 256, 256, 0, stream>>>(a, S);
  prof_end(K_CONV_BWD, stream);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // extern "C"
