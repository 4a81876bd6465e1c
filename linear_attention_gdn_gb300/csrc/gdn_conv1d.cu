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
// element is read from HBM once plus a halo of W - 1 rows per range.  Rows are
// requested four at a time before any is used.  The backward writes per-range
// partial sums of dw and db; a second kernel adds them in range order, so the
// result does not depend on scheduling.
#include <algorithm>
#include <cstring>

#include "gdn.h"
#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_prof.h"

namespace gdn {

int sm_count();

constexpr int CV_THREADS = 128;
constexpr int CV_VEC = 4;                         // channels per thread
constexpr int CV_CH = CV_THREADS * CV_VEC;        // channels per CTA
constexpr int CV_MAXW = 4;
constexpr int CV_U = 4;                           // rows requested together

struct ConvArgs {
  const __nv_bfloat16* x;
  const float* w;        // [C][W]
  const float* b;        // [C] or null
  const int* cu;         // [N+1]
  const __nv_bfloat16* dy;
  __nv_bfloat16* y;      // forward output
  __nv_bfloat16* dx;     // backward output
  float* part;           // [S][W+1][C] partial dw (rows 0..W-1) and db (row W) per token range
  float* dw;             // [C][W]
  float* db;             // [C]
  int64_t T;
  int N, C, W, R;        // R: tokens per range (grid.y ranges)
};

__device__ __forceinline__ void ld_row(const __nv_bfloat16* p, float (&v)[CV_VEC]) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int e = 0; e < CV_VEC / 2; ++e) {
    const float2 f = __bfloat1622float2(h[e]);
    v[2 * e] = f.x;
    v[2 * e + 1] = f.y;
  }
}
__device__ __forceinline__ void st_row(__nv_bfloat16* p, const float (&v)[CV_VEC]) {
  uint2 u;
  u.x = pack_bf16(v[0], v[1]);
  u.y = pack_bf16(v[2], v[3]);
  *reinterpret_cast<uint2*>(p) = u;
}
__device__ __forceinline__ float sigmoidf(float z) { return 1.0f / (1.0f + expf(-z)); }

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

// per-thread setup shared by both directions: taps, bias, the document of the first row, and the
// last W - 1 input rows before it (zero where they precede the document start)
struct ConvThread {
  float w[CV_MAXW][CV_VEC], b[CV_VEC];
  float xw[CV_MAXW - 1][CV_VEC];   // xw[W-2] is the row just before the current one
  int start, next;                 // current document's first token, the next document's
  int d;
};

__device__ __forceinline__ void conv_setup(const ConvArgs& a, int c0, int64_t lo, ConvThread& th) {
#pragma unroll
  for (int i = 0; i < CV_MAXW; ++i)
#pragma unroll
    for (int e = 0; e < CV_VEC; ++e) th.w[i][e] = i < a.W ? a.w[(size_t)(c0 + e) * a.W + i] : 0.f;
#pragma unroll
  for (int e = 0; e < CV_VEC; ++e) th.b[e] = a.b ? a.b[c0 + e] : 0.f;
  th.d = doc_of(a.cu, a.N, lo);
  th.start = a.cu[th.d];
  th.next = a.cu[th.d + 1];
#pragma unroll
  for (int j = 0; j < CV_MAXW - 1; ++j) {   // xw[j] = x[lo - (W-1) + j]
    const int64_t s = lo - (a.W - 1) + j;
    if (j < a.W - 1 && s >= th.start) ld_row(a.x + s * a.C + c0, th.xw[j]);
    else
#pragma unroll
      for (int e = 0; e < CV_VEC; ++e) th.xw[j][e] = 0.f;
  }
}

// advance the document bookkeeping to token t; true when t starts a document (history reset)
__device__ __forceinline__ bool conv_enter(const ConvArgs& a, int64_t t, ConvThread& th) {
  if (t < th.next) return false;
  while (th.d + 1 < a.N && a.cu[th.d + 1] <= t) ++th.d;
  th.start = a.cu[th.d];
  th.next = a.cu[th.d + 1];
  return true;
}

// z for the current row xt, the history in th.xw; then shift xt into the history
__device__ __forceinline__ void conv_z(const ConvArgs& a, const float (&xt)[CV_VEC], ConvThread& th,
                                       float (&z)[CV_VEC], float (&xs)[CV_MAXW][CV_VEC]) {
  // xs[i] = x[t - (W-1) + i]: the input that tap i multiplies
#pragma unroll
  for (int i = 0; i < CV_MAXW; ++i)
#pragma unroll
    for (int e = 0; e < CV_VEC; ++e)
      xs[i][e] = i < a.W - 1 ? th.xw[i][e] : (i == a.W - 1 ? xt[e] : 0.f);
#pragma unroll
  for (int e = 0; e < CV_VEC; ++e) {
    float acc = th.b[e];
#pragma unroll
    for (int i = 0; i < CV_MAXW; ++i) acc = fmaf(th.w[i][e], xs[i][e], acc);
    z[e] = acc;
  }
  // the history moves down one row: xw[j] <- xw[j + 1] for j < W - 2, xw[W - 2] <- xt
#pragma unroll
  for (int j = 0; j < CV_MAXW - 1; ++j) {
    constexpr int LAST = CV_MAXW - 2;
    const int up = j < LAST ? j + 1 : LAST;   // (a compile-time index)
#pragma unroll
    for (int e = 0; e < CV_VEC; ++e) {
      const float nx = j < a.W - 2 ? th.xw[up][e] : xt[e];
      if (j <= a.W - 2) th.xw[j][e] = nx;
    }
  }
}

__device__ __forceinline__ void conv_reset(ConvThread& th) {
#pragma unroll
  for (int j = 0; j < CV_MAXW - 1; ++j)
#pragma unroll
    for (int e = 0; e < CV_VEC; ++e) th.xw[j][e] = 0.f;
}

__global__ void __launch_bounds__(CV_THREADS) conv_fwd_kernel(const ConvArgs a) {
  const int c0 = (blockIdx.x * CV_THREADS + threadIdx.x) * CV_VEC;
  const int64_t lo = (int64_t)blockIdx.y * a.R, hi = min(a.T, lo + a.R);
  if (c0 >= a.C || lo >= hi) return;
  ConvThread th;
  conv_setup(a, c0, lo, th);
  for (int64_t t0 = lo; t0 < hi; t0 += CV_U) {
    float xr[CV_U][CV_VEC];
#pragma unroll
    for (int u = 0; u < CV_U; ++u)
      if (t0 + u < hi) ld_row(a.x + (t0 + u) * a.C + c0, xr[u]);
#pragma unroll
    for (int u = 0; u < CV_U; ++u) {
      const int64_t t = t0 + u;
      if (t >= hi) break;
      if (conv_enter(a, t, th)) conv_reset(th);
      float z[CV_VEC], xs[CV_MAXW][CV_VEC], y[CV_VEC];
      conv_z(a, xr[u], th, z, xs);
#pragma unroll
      for (int e = 0; e < CV_VEC; ++e) y[e] = z[e] * sigmoidf(z[e]);
      st_row(a.y + t * a.C + c0, y);
    }
  }
}

// Backward over the range [lo, hi): dz for rows [lo, hi + W - 1) (the last W - 1 only feed dx of
// rows below hi), dx for rows [lo, hi), partial dw / db over rows [lo, hi).
__global__ void __launch_bounds__(CV_THREADS) conv_bwd_kernel(const ConvArgs a) {
  const int c0 = (blockIdx.x * CV_THREADS + threadIdx.x) * CV_VEC;
  const int64_t lo = (int64_t)blockIdx.y * a.R, hi = min(a.T, lo + a.R);
  if (c0 >= a.C || lo >= hi) return;
  ConvThread th;
  conv_setup(a, c0, lo, th);
  float dzw[CV_MAXW][CV_VEC];   // dz of rows t' - (W-1) .. t' (dzw[W-1] newest)
  int dsw[CV_MAXW];             // the document start of each of those rows (-1: none)
#pragma unroll
  for (int j = 0; j < CV_MAXW; ++j) {
    dsw[j] = -1;
#pragma unroll
    for (int e = 0; e < CV_VEC; ++e) dzw[j][e] = 0.f;
  }
  float pw[CV_MAXW][CV_VEC], pb[CV_VEC];
#pragma unroll
  for (int e = 0; e < CV_VEC; ++e) {
    pb[e] = 0.f;
#pragma unroll
    for (int i = 0; i < CV_MAXW; ++i) pw[i][e] = 0.f;
  }
  const int64_t end = hi + a.W - 1;
  for (int64_t t0 = lo; t0 < end; t0 += CV_U) {
    float xr[CV_U][CV_VEC], gr[CV_U][CV_VEC];
#pragma unroll
    for (int u = 0; u < CV_U; ++u)
      if (t0 + u < end && t0 + u < a.T) {
        ld_row(a.x + (t0 + u) * a.C + c0, xr[u]);
        ld_row(a.dy + (t0 + u) * a.C + c0, gr[u]);
      }
#pragma unroll
    for (int u = 0; u < CV_U; ++u) {
      const int64_t t = t0 + u;
      if (t >= end) break;
      float dz[CV_VEC];
      int ds = -1;
      if (t < a.T) {
        if (conv_enter(a, t, th)) conv_reset(th);
        ds = th.start;
        float z[CV_VEC], xs[CV_MAXW][CV_VEC];
        conv_z(a, xr[u], th, z, xs);
#pragma unroll
        for (int e = 0; e < CV_VEC; ++e) {
          const float sg = sigmoidf(z[e]);
          dz[e] = gr[u][e] * sg * (1.0f + z[e] * (1.0f - sg));
        }
        if (t < hi) {
#pragma unroll
          for (int e = 0; e < CV_VEC; ++e) {
            pb[e] += dz[e];
#pragma unroll
            for (int i = 0; i < CV_MAXW; ++i) pw[i][e] = fmaf(dz[e], xs[i][e], pw[i][e]);
          }
        }
      } else {
#pragma unroll
        for (int e = 0; e < CV_VEC; ++e) dz[e] = 0.f;
      }
      // window of the last W rows' dz
#pragma unroll
      for (int j = 0; j < CV_MAXW - 1; ++j) {
        dsw[j] = dsw[j + 1];
#pragma unroll
        for (int e = 0; e < CV_VEC; ++e) dzw[j][e] = dzw[j + 1][e];
      }
      dsw[CV_MAXW - 1] = ds;
#pragma unroll
      for (int e = 0; e < CV_VEC; ++e) dzw[CV_MAXW - 1][e] = dz[e];
      // dx of row s = t - (W-1): taps i see dz of row s + (W-1) - i = window slot CV_MAXW - 1 - i
      const int64_t s = t - (a.W - 1);
      if (s >= lo && s < hi) {
        int sds = -2;   // the document start of row s, which sits in slot CV_MAXW - W
#pragma unroll
        for (int slot = 0; slot < CV_MAXW; ++slot)
          if (slot == CV_MAXW - a.W) sds = dsw[slot];
        float dx[CV_VEC];
#pragma unroll
        for (int e = 0; e < CV_VEC; ++e) {
          float acc = 0.f;
#pragma unroll
          for (int i = CV_MAXW - 1; i >= 0; --i) {
            const int slot = CV_MAXW - 1 - i;
            if (i < a.W && dsw[slot] == sds) acc = fmaf(th.w[i][e], dzw[slot][e], acc);
          }
          dx[e] = acc;
        }
        st_row(a.dx + s * a.C + c0, dx);
      }
    }
  }
  float* pp = a.part + (size_t)blockIdx.y * (a.W + 1) * a.C + c0;
#pragma unroll
  for (int i = 0; i < CV_MAXW; ++i)
    if (i < a.W) *reinterpret_cast<float4*>(pp + (size_t)i * a.C) = make_float4(pw[i][0], pw[i][1], pw[i][2], pw[i][3]);
  *reinterpret_cast<float4*>(pp + (size_t)a.W * a.C) = make_float4(pb[0], pb[1], pb[2], pb[3]);
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

// token ranges: enough CTAs to fill the GPU four times over, at least 64 tokens each
static void conv_ranges(int64_t T, int C, int sms, int* S, int* R) {
  const int nblk = (C + CV_CH - 1) / CV_CH;
  int64_t s = std::max<int64_t>(1, (4 * (int64_t)sms + nblk - 1) / nblk);
  s = std::min<int64_t>(s, std::max<int64_t>(1, (T + 63) / 64));
  const int64_t r = std::max<int64_t>(1, (T + s - 1) / s);
  *R = (int)std::min<int64_t>(r, INT32_MAX);
  *S = (int)((T + r - 1) / r);
}

}  // namespace gdn

using namespace gdn;

extern "C" {

static gdn_status conv_check(const gdn_conv_problem* p, const int32_t* cu) {
  if (!p || !cu) return GDN_ERR_INVALID_ARG;
  if (p->N < 1 || p->C <= 0 || p->C % CV_VEC != 0 || p->W < 1 || p->W > CV_MAXW || p->T < 0)
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
  int S = 0, R = 0;
  conv_ranges(p->T, p->C, sm_count(), &S, &R);
  *ws_bytes = p->T > 0 ? (size_t)S * (p->W + 1) * p->C * sizeof(float) : 0;
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
  int S = 0;
  conv_ranges(p->T, p->C, sm_count(), &S, &a.R);
  prof_begin(K_CONV_FWD, stream);
  conv_fwd_kernel<<<dim3((p->C + CV_CH - 1) / CV_CH, S), CV_THREADS, 0, stream>>>(a);
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
  if (p->T > 0 && (!al16(x) || !al16(dy) || !al16(dx) || !al16(workspace))) return GDN_ERR_INVALID_ARG;
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
  a.part = static_cast<float*>(workspace);
  a.dw = dw;
  a.db = db;
  a.T = p->T;
  a.N = p->N;
  a.C = p->C;
  a.W = p->W;
  int S = 0;
  conv_ranges(p->T, p->C, sm_count(), &S, &a.R);
  prof_begin(K_CONV_BWD, stream);
  conv_bwd_kernel<<<dim3((p->C + CV_CH - 1) / CV_CH, S), CV_THREADS, 0, stream>>>(a);
  conv_reduce_kernel<<<(p->C + 255) / 256, 256, 0, stream>>>(a, S);
  prof_end(K_CONV_BWD, stream);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // extern "C"
