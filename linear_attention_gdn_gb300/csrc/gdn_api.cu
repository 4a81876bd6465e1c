// gdn_api.cu -- host layer of the C ABI declared in include/gdn.h:
// argument validation, the segment planner, workspace / saved-set layouts,
// TMA tensor maps and the launch sequence of each entry point.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include "gdn.h"
#include "gdn_internal.h"
#include "gdn_prof.h"

namespace gdn {
void launch_tables(const TableArgs& a, cudaStream_t s);
void launch_prep(const PrepArgs& a, int NC, cudaStream_t s);
void launch_fwd_scan(const ScanArgs& a, int nchains, cudaStream_t s);
void launch_passthrough(const PassArgs& a, int N, cudaStream_t s);
void launch_merge(const MergeArgs& a, int nsdoc, cudaStream_t s);
void setup_fwd_scan_attrs();
void setup_bwd_attrs();
void setup_prep_attrs();
void setup_vnew_attrs();
void setup_kda_attrs();
void setup_kda_bwd_attrs();
gdn_status run_bwd(const Plan& P, const gdn_problem& pr, const void* q, const void* k, const void* v,
                   const float* g, const float* beta, const int32_t* cu_dev, const void* dO, const void* saved,
                   void* dq, void* dk, void* dv, float* dg, float* dbeta, const float* ds_out, float* ds_in,
                   uint8_t* ws, cudaStream_t s);
}  // namespace gdn

using namespace gdn;

namespace gdn {

// ---------------------------------------------------------------------------
// plan and layouts
// ---------------------------------------------------------------------------


static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int sm_count() {
  int dev = 0, n = 152;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) n = 152;
  }
  return n > 0 ? n : 152;
}

static gdn_status validate_problem(const gdn_problem* p, const int32_t* cu) {
  if (!p || !cu) return GDN_ERR_INVALID_ARG;
  if (p->N < 1 || p->T < 0 || p->H < 1 || p->HV < 1) return GDN_ERR_INVALID_ARG;
  if (p->dk != 128 || p->dv != 128) return GDN_ERR_UNSUPPORTED;
  if (p->HV % p->H != 0) return GDN_ERR_UNSUPPORTED;
  if (p->T > (int64_t)INT32_MAX / 2) return GDN_ERR_UNSUPPORTED;
  if (p->segments < 0) return GDN_ERR_INVALID_ARG;
  if (p->saved_form != GDN_SAVED_FULL && p->saved_form != GDN_SAVED_REPLAY) return GDN_ERR_INVALID_ARG;
  if (cu[0] != 0) return GDN_ERR_INVALID_ARG;
  for (int i = 0; i < p->N; ++i)
    if (cu[i + 1] < cu[i]) return GDN_ERR_INVALID_ARG;
  if ((int64_t)cu[p->N] != p->T) return GDN_ERR_INVALID_ARG;
  return GDN_OK;
}

// The segment planner.  A scan chain is one (segment, value head); chains of
// one document share nothing, so a long document is cut into segments whose
// transfer operators are composed by the merge kernel.  Splitting costs two
// extra walks per split segment (B and M), so it pays only when the longest
// chains would otherwise leave most SMs idle: the planner splits a document
// of n chunks when n exceeds both 512 and three times the balanced per-SM
// share of all chain steps, into P = ceil(n / share) segments of equal length
// (the walks of one launch run in waves of one CTA per SM, so a short last
// segment would leave its wave idle).
static void plan_segments(const gdn_problem* p, const int32_t* cu, int* seg_len, int* split_min,
                          int* max_doc) {
  int64_t total = 0;
  int mx = 0;
  for (int i = 0; i < p->N; ++i) {
    const int n = (cu[i + 1] - cu[i] + CHUNK - 1) / CHUNK;
    total += n;
    mx = std::max(mx, n);
  }
  *max_doc = mx;
  if (p->segments > 0) {
    const int s = std::max(1, (mx + p->segments - 1) / p->segments);
    *seg_len = s;
    *split_min = s;
    return;
  }
  const int64_t share = (total * p->HV + sm_count() - 1) / sm_count();
  if (mx > 512 && mx > 3 * share) {
    const int64_t parts = (mx + share - 1) / share;
    *seg_len = (int)std::max<int64_t>(256, (mx + parts - 1) / parts);
    *split_min = *seg_len;
  } else {
    *seg_len = std::max(mx, 1);
    *split_min = INT32_MAX;
  }
}

gdn_status make_plan(const gdn_problem* p, const int32_t* cu, Plan* P) {
  gdn_status st = validate_problem(p, cu);
  if (st != GDN_OK) return st;
  P->T = p->T;
  P->N = p->N;
  P->H = p->H;
  P->HV = p->HV;
  P->G = p->HV / p->H;
  P->form = p->saved_form;
  P->sms = sm_count();
  plan_segments(p, cu, &P->seg_len, &P->split_min, &P->max_doc_chunks);
  int NC = 0, NSEG = 0, nsplit = 0, nsdoc = 0, n_empty = 0;
  uint32_t h = 0u;
  for (int i = 0; i < p->N; ++i) {
    const int n = (cu[i + 1] - cu[i] + CHUNK - 1) / CHUNK;
    const int Pd = n > P->split_min ? (n + P->seg_len - 1) / P->seg_len : (n > 0 ? 1 : 0);
    NC += n;
    NSEG += Pd;
    n_empty += n == 0 ? 1 : 0;
    if (Pd > 1) {
      nsplit += Pd - 1;
      nsdoc += 1;
    }
    h += cu_entry_hash(i, cu[i + 1]);
  }
  P->NC = NC;
  P->NSEG = NSEG;
  P->nsplit = nsplit;
  P->nsdoc = nsdoc;
  P->n_empty = n_empty;
  P->cu_hash = h;
  // workspace
  size_t off = 256;   // control block (error word)
  const int counts[19] = {P->N + 1, P->N + 1, P->N + 1, NC, NC, NC, NSEG, NSEG, NSEG, NSEG, NSEG, nsplit,
                          nsdoc + 1, P->N + 1, NSEG - nsdoc, NSEG - nsdoc, NSEG - nsdoc, NSEG - nsdoc, 0};
  for (int i = 0; i < 19; ++i) {
    P->o_tables[i] = off;
    off = align_up(off + (size_t)counts[i] * 4, 256);
  }
  off = align_up(off, 1024);
  // the UT blocks of a forward without a full saved set, and of a replay-form backward
  P->o_cb = off;
  off += (size_t)NC * P->HV * CB_BYTES;
  const size_t st_f32 = (size_t)nsplit * P->HV * STATE_F32 * 4;
  P->o_bend = off;
  off += st_f32;
  P->o_sinit = off;
  off += st_f32;
  P->o_mend_ws = off;
  off += st_f32;
  P->ws_fwd = off;
  P->o_dtape = off;
  off += (size_t)NC * P->HV * STATE_BYTES;
  P->o_dvn = off;
  off += (size_t)NC * P->HV * VN_BYTES;
  P->o_dbend = off;
  off += st_f32;
  P->o_dsinit = off;
  off += st_f32;
  P->o_vnb = 0;
  if (P->form == GDN_SAVED_REPLAY) {
    P->o_vnb = off;
    off += (size_t)NC * P->HV * VN_BYTES;
  }
  P->ws_bwd = off;
  // saved set: header, state tape, M_seg; the full form adds the UT blocks and V_new^T
  P->s_tape = SAVED_HEADER;
  P->s_mseg = P->s_tape + (size_t)NC * P->HV * STATE_BYTES;
  P->s_cb = align_up(P->s_mseg + st_f32, 1024);
  if (P->form == GDN_SAVED_FULL) {
    P->s_vn = P->s_cb + (size_t)NC * P->HV * CB_BYTES;
    P->saved_bytes = P->s_vn + (size_t)NC * P->HV * VN_BYTES;
  } else {
    P->s_vn = P->s_cb;
    P->saved_bytes = P->s_cb;
  }
  return GDN_OK;
}


static SavedHeader header_of(const Plan& P, const gdn_problem* p) {
  SavedHeader h;
  memset(&h, 0, sizeof(h));
  h.magic = SAVED_MAGIC;
  h.version = SAVED_VERSION;
  h.T = P.T;
  h.N = P.N;
  h.H = P.H;
  h.HV = P.HV;
  h.dk = p->dk;
  h.dv = p->dv;
  h.l2norm = p->l2norm ? 1 : 0;
  h.NC = P.NC;
  h.NSEG = P.NSEG;
  h.nsplit = P.nsplit;
  h.seg_len = P.seg_len;
  memcpy(&h.scale_bits, &p->scale, 4);
  h.cu_hash = P.cu_hash;
  h.form = P.form;
  return h;
}

// ---------------------------------------------------------------------------
// TMA tensor maps and one-time per-device setup
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// token-major BF16 tensor [T][heads][128]; box = 64 features x 1 head x 64 tokens
bool make_tmap(CUtensorMap* m, const void* base, int64_t T, int heads) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {128, (cuuint64_t)heads, (cuuint64_t)std::max<int64_t>(T, 1)};
  cuuint64_t strides[2] = {128 * 2, (cuuint64_t)heads * 128 * 2};
  cuuint32_t box[3] = {64, 1, 64};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_g(CUtensorMap* m, const float* base, int64_t T, int heads) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {128, (cuuint64_t)heads, (cuuint64_t)std::max<int64_t>(T, 1)};
  cuuint64_t strides[2] = {128 * 4, (cuuint64_t)heads * 128 * 4};
  cuuint32_t box[3] = {128, 1, 64};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_rows(CUtensorMap* m, const void* base, int64_t T, int C, int rows) {
  auto fn = encode_fn();
  if (!fn || C % 256 != 0) return false;
  cuuint64_t dims[3] = {256, (cuuint64_t)(C / 256), (cuuint64_t)std::max<int64_t>(T, 1)};
  cuuint64_t strides[2] = {256 * 2, (cuuint64_t)C * 2};
  cuuint32_t box[3] = {256, 2, (cuuint32_t)rows};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool device_setup() {
  static std::mutex mu;
  static bool done[128] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return false;
  std::lock_guard<std::mutex> lk(mu);
  if (!done[dev]) {
    setup_fwd_scan_attrs();
    setup_bwd_attrs();
    setup_prep_attrs();
    setup_vnew_attrs();
    setup_kda_attrs();
    setup_kda_bwd_attrs();
    done[dev] = true;
  }
  return true;
}


// ---------------------------------------------------------------------------
// launch counters and optional per-kernel event timing
// ---------------------------------------------------------------------------
static const char* const kKernelNames[K_NUM] = {
    "tables_scan_kernel", "tables_fill_kernel", "prep_kernel",    "fwd_scan_kernel(walk)",
    "merge_kernel",       "fwd_scan_kernel",    "check_saved_kernel", "bwd_scan_kernel(walk)",
    "merge_bwd_kernel",   "bwd_scan_kernel",    "grad_kernel",        "passthrough_kernel",
    "conv_fwd_kernel",    "conv_bwd_kernel(+reduce)", "vnew_kernel",      "kda_prep_kernel",
    "kda_out_kernel",     "kda_grad_kernel",    "walk_order_kernel"};
struct ProfRec {
  int id;
  cudaEvent_t e0, e1;
};
static std::mutex g_prof_mu;
static bool g_prof_on = false;
static long long g_launches[K_NUM] = {};
static std::vector<ProfRec> g_recs;
static std::vector<cudaEvent_t> g_pool;
static cudaEvent_t g_open[K_NUM] = {};

static cudaEvent_t pool_get() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

void prof_begin(int id, cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_launches[id] += 1;
  if (!g_prof_on) return;
  cudaEvent_t e = pool_get();
  cudaEventRecord(e, s);
  g_open[id] = e;
}
void prof_end(int id, cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_prof_on || !g_open[id]) return;
  cudaEvent_t e = pool_get();
  cudaEventRecord(e, s);
  g_recs.push_back({id, g_open[id], e});
  g_open[id] = nullptr;
}

bool aligned16(const void* p) { return p && ((uintptr_t)p & 15) == 0; }

// ---------------------------------------------------------------------------
// forward
// ---------------------------------------------------------------------------
gdn_status run_tables(const Plan& P, const gdn_problem* p, const int32_t* cu_dev, uint8_t* ws, void* saved,
                      cudaStream_t s) {
  if (cudaMemsetAsync(ws, 0, 256, s) != cudaSuccess) return GDN_ERR_CUDA;
  TableArgs ta;
  ta.cu = cu_dev;
  ta.T = P.T;
  ta.cu_hash = P.cu_hash;
  ta.N = P.N;
  ta.NC = P.NC;
  ta.NSEG = P.NSEG;
  ta.nsplit = P.nsplit;
  ta.nsdoc = P.nsdoc;
  ta.seg_len = P.seg_len;
  ta.split_min = P.split_min;
  ta.t = tables_at(P, ws);
  ta.err = reinterpret_cast<int*>(ws);
  ta.hdr = header_of(P, p);
  ta.saved = static_cast<uint8_t*>(saved);
  launch_tables(ta, s);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status run_prep(const Plan& P, const gdn_problem* p, const void* q, const void* k, const float* g,
                    const float* beta, uint8_t* ws, uint8_t* cb, int write_T, cudaStream_t s) {
  Tables t = tables_at(P, ws);
  PrepArgs pa;
  if (!make_tmap(&pa.tq, q, P.T, P.H) || !make_tmap(&pa.tk, k, P.T, P.H)) return GDN_ERR_CUDA;
  pa.q = static_cast<const __nv_bfloat16*>(q);
  pa.k = static_cast<const __nv_bfloat16*>(k);
  pa.g = g;
  pa.beta = beta;
  pa.chunk_tok0 = t.chunk_tok0;
  pa.chunk_len = t.chunk_len;
  pa.cb = cb;
  pa.H = P.H;
  pa.HV = P.HV;
  pa.G = P.G;
  pa.l2norm = p->l2norm ? 1 : 0;
  pa.write_T = write_T;
  pa.scale = p->scale;
  pa.err = reinterpret_cast<int*>(ws);
  launch_prep(pa, P.NC, s);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

static gdn_status run_fwd(const Plan& P, const gdn_problem* p, const void* q, const void* k, const void* v,
                          const float* g, const float* beta, const int32_t* cu_dev, const float* s_in, void* o,
                          float* s_out, void* saved, uint8_t* ws, cudaStream_t s) {
  gdn_status st = run_tables(P, p, cu_dev, ws, saved, s);
  if (st != GDN_OK) return st;
  if (s_out && P.n_empty > 0) {   // documents without chunks pass S_in straight through
    PassArgs pa;
    pa.chunk_offsets = tables_at(P, ws).chunk_offsets;
    pa.src = s_in;
    pa.dst = s_out;
    pa.HV = P.HV;
    launch_passthrough(pa, P.N, s);
  }
  if (P.NC == 0) return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
  // with a full-form saved set, the per-chunk UT blocks (with T) go into it for the backward; else
  // they are the walk's scratch in the workspace
  const bool full = saved && P.form == GDN_SAVED_FULL;
  uint8_t* cb = full ? static_cast<uint8_t*>(saved) + P.s_cb : ws + P.o_cb;
  st = run_prep(P, p, q, k, g, beta, ws, cb, full ? 1 : 0, s);
  if (st != GDN_OK) return st;
  Tables t = tables_at(P, ws);
  ScanArgs sa;
  memset(&sa, 0, sizeof(sa));
  if (!make_tmap(&sa.tq, q, P.T, P.H) || !make_tmap(&sa.tk, k, P.T, P.H) || !make_tmap(&sa.tv, v, P.T, P.HV))
    return GDN_ERR_CUDA;
  sa.cb = cb;
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
  sa.mend = saved ? reinterpret_cast<float*>(static_cast<uint8_t*>(saved) + P.s_mseg)
                  : reinterpret_cast<float*>(ws + P.o_mend_ws);
  sa.seg_doc = t.seg_doc;
  sa.seg_offsets = t.seg_offsets;
  sa.s_in = s_in;
  sa.s_out = s_out;
  sa.err = reinterpret_cast<int*>(ws);
  // (the first segment of a split document walks in full in the split launch: it writes o and the tape)
  sa.tape = saved ? static_cast<uint8_t*>(saved) + P.s_tape : nullptr;
  sa.vn = full ? static_cast<uint8_t*>(saved) + P.s_vn : nullptr;
  sa.o = static_cast<__nv_bfloat16*>(o);
  if (o && !make_tmap(&sa.to, o, P.T, P.HV)) return GDN_ERR_CUDA;
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
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace gdn

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------
extern "C" {

const char* gdn_status_string(gdn_status s) {
  switch (s) {
    case GDN_OK: return "ok";
    case GDN_ERR_INVALID_ARG: return "invalid argument";
    case GDN_ERR_UNSUPPORTED: return "unsupported problem (dk, dv must be 128 and HV a multiple of H)";
    case GDN_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case GDN_ERR_SAVED_MISMATCH: return "saved set does not match this problem";
    case GDN_ERR_CUDA: return "CUDA error";
    case GDN_ERR_TIMEOUT: return "a bounded device wait ran out";
    case GDN_ERR_DEVICE: return "device-side error";
    case GDN_ERR_GATE_RANGE: return "a per-channel decay too steep within 16 tokens (KDA)";
  }
  return "unknown status";
}

gdn_status gdn_saved_bytes(const gdn_problem* prob, const int32_t* cu_host, size_t* saved_bytes,
                           size_t* workspace_bytes) {
  Plan P;
  gdn_status st = make_plan(prob, cu_host, &P);
  if (st != GDN_OK) return st;
  if (saved_bytes) *saved_bytes = P.saved_bytes;
  if (workspace_bytes) *workspace_bytes = P.ws_bwd;
  return GDN_OK;
}

int32_t gdn_plan_segment_chunks(const gdn_problem* prob, const int32_t* cu_host) {
  Plan P;
  if (make_plan(prob, cu_host, &P) != GDN_OK) return 0;
  return P.split_min == INT32_MAX ? P.max_doc_chunks : P.seg_len;
}

gdn_status gdn_fwd_states(const gdn_problem* prob, const void* q, const void* k, const void* v, const float* g,
                          const float* beta, const int32_t* cu_dev, const int32_t* cu_host, const float* s_in,
                          void* o, float* s_out, void* saved, void* workspace, size_t ws_bytes,
                          struct CUstream_st* stream) {
  Plan P;
  gdn_status st = make_plan(prob, cu_host, &P);
  if (st != GDN_OK) return st;
  if (!cu_dev || !workspace || (!o && !saved && !s_out)) return GDN_ERR_INVALID_ARG;
  if (P.T > 0 && (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(beta) ||
                  (o && !aligned16(o))))
    return GDN_ERR_INVALID_ARG;
  if ((s_in && !aligned16(s_in)) || (s_out && !aligned16(s_out))) return GDN_ERR_INVALID_ARG;
  if (!aligned16(workspace) || (saved && !aligned16(saved))) return GDN_ERR_INVALID_ARG;
  if (ws_bytes < P.ws_fwd) return GDN_ERR_WORKSPACE_TOO_SMALL;
  if (!device_setup()) return GDN_ERR_CUDA;
  return run_fwd(P, prob, q, k, v, g, beta, cu_dev, s_in, o, s_out, saved, static_cast<uint8_t*>(workspace),
                 stream);
}

gdn_status gdn_fwd(const gdn_problem* prob, const void* q, const void* k, const void* v, const float* g,
                   const float* beta, const int32_t* cu_dev, const int32_t* cu_host, void* o, void* saved,
                   void* workspace, size_t ws_bytes, struct CUstream_st* stream) {
  if (!o && !saved) return GDN_ERR_INVALID_ARG;
  return gdn_fwd_states(prob, q, k, v, g, beta, cu_dev, cu_host, nullptr, o, nullptr, saved, workspace, ws_bytes,
                        stream);
}

gdn_status gdn_bwd_states(const gdn_problem* prob, const void* q, const void* k, const void* v, const float* g,
                          const float* beta, const int32_t* cu_dev, const int32_t* cu_host, const void* dO,
                          const float* ds_out, const void* saved, void* dq, void* dk, void* dv, float* dg,
                          float* dbeta, float* ds_in, void* workspace, size_t ws_bytes,
                          struct CUstream_st* stream) {
  Plan P;
  gdn_status st = make_plan(prob, cu_host, &P);
  if (st != GDN_OK) return st;
  if (!cu_dev || !workspace || !saved) return GDN_ERR_INVALID_ARG;
  if (P.T > 0 && (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(beta) ||
                  !aligned16(dO) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(dg) ||
                  !aligned16(dbeta)))
    return GDN_ERR_INVALID_ARG;
  if ((ds_out && !aligned16(ds_out)) || (ds_in && !aligned16(ds_in))) return GDN_ERR_INVALID_ARG;
  if (!aligned16(workspace) || !aligned16(saved)) return GDN_ERR_INVALID_ARG;
  if (ws_bytes < P.ws_bwd) return GDN_ERR_WORKSPACE_TOO_SMALL;
  if (!device_setup()) return GDN_ERR_CUDA;
  return run_bwd(P, *prob, q, k, v, g, beta, cu_dev, dO, saved, dq, dk, dv, dg, dbeta, ds_out, ds_in,
                 static_cast<uint8_t*>(workspace), stream);
}

gdn_status gdn_bwd(const gdn_problem* prob, const void* q, const void* k, const void* v, const float* g,
                   const float* beta, const int32_t* cu_dev, const int32_t* cu_host, const void* dO,
                   const void* saved, void* dq, void* dk, void* dv, float* dg, float* dbeta, void* workspace,
                   size_t ws_bytes, struct CUstream_st* stream) {
  return gdn_bwd_states(prob, q, k, v, g, beta, cu_dev, cu_host, dO, nullptr, saved, dq, dk, dv, dg, dbeta,
                        nullptr, workspace, ws_bytes, stream);
}

gdn_status gdn_ckpt_fwd_bwd(const gdn_problem* prob, const void* q, const void* k, const void* v,
                            const float* g, const float* beta, const int32_t* cu_dev, const int32_t* cu_host,
                            const void* dO, void* o, void* dq, void* dk, void* dv, float* dg, float* dbeta,
                            void* saved_scratch, void* workspace, size_t ws_bytes, struct CUstream_st* stream) {
  Plan P;
  gdn_status st = make_plan(prob, cu_host, &P);
  if (st != GDN_OK) return st;
  if (!saved_scratch) return GDN_ERR_INVALID_ARG;
  // the checkpointed forward (no states kept), then the recompute forward
  // that writes the saved set, then the backward; with o == NULL the first
  // forward would produce nothing and is skipped
  if (o) {
    st = gdn_fwd(prob, q, k, v, g, beta, cu_dev, cu_host, o, nullptr, workspace, ws_bytes, stream);
    if (st != GDN_OK) return st;
  }
  st = gdn_fwd(prob, q, k, v, g, beta, cu_dev, cu_host, nullptr, saved_scratch, workspace, ws_bytes, stream);
  if (st != GDN_OK) return st;
  return gdn_bwd(prob, q, k, v, g, beta, cu_dev, cu_host, dO, saved_scratch, dq, dk, dv, dg, dbeta, workspace,
                 ws_bytes, stream);
}

gdn_status gdn_chunk_table_offsets(const gdn_problem* prob, const int32_t* cu_host, size_t offsets[4],
                                   int32_t* num_chunks) {
  Plan P;
  gdn_status st = make_plan(prob, cu_host, &P);
  if (st != GDN_OK) return st;
  if (!offsets || !num_chunks) return GDN_ERR_INVALID_ARG;
  offsets[0] = P.o_tables[0];   // chunk_offsets
  offsets[1] = P.o_tables[3];   // chunk_doc
  offsets[2] = P.o_tables[4];   // chunk_tok0
  offsets[3] = P.o_tables[5];   // chunk_len
  *num_chunks = P.NC;
  return GDN_OK;
}


gdn_status gdn_backward_tape_offsets(const gdn_problem* prob, const int32_t* cu_host, size_t offsets[4]) {
  Plan P;
  gdn_status st = make_plan(prob, cu_host, &P);
  if (st != GDN_OK) return st;
  if (!offsets) return GDN_ERR_INVALID_ARG;
  const bool replay = P.form == GDN_SAVED_REPLAY;
  offsets[0] = replay ? P.o_cb : 0;
  offsets[1] = replay ? P.o_vnb : 0;
  offsets[2] = P.o_dtape;
  offsets[3] = P.o_dvn;
  return GDN_OK;
}

void gdn_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_on = on != 0;
}

int gdn_profile_read(gdn_kernel_stat* out, int max_entries) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  double ms[K_NUM] = {};
  long long timed[K_NUM] = {};
  for (const ProfRec& r : g_recs) {
    float t = 0.f;
    if (cudaEventSynchronize(r.e1) == cudaSuccess && cudaEventElapsedTime(&t, r.e0, r.e1) == cudaSuccess) {
      ms[r.id] += t;
      timed[r.id] += 1;
    }
    g_pool.push_back(r.e0);
    g_pool.push_back(r.e1);
  }
  g_recs.clear();
  int n = 0;
  for (int i = 0; i < K_NUM; ++i) {
    if (g_launches[i] == 0) continue;
    if (out && n < max_entries) {
      out[n].name = kKernelNames[i];
      out[n].launches = g_launches[i];
      out[n].timed_launches = timed[i];
      out[n].total_ms = ms[i];
    }
    ++n;
    g_launches[i] = 0;
  }
  return n;
}

gdn_status gdn_device_status(void* workspace, struct CUstream_st* stream) {
  if (!workspace) return GDN_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return GDN_ERR_CUDA;
  int e = 0;
  if (cudaMemcpy(&e, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return GDN_ERR_CUDA;
  if (e < 0 || e > 8) return GDN_ERR_DEVICE;
  return (gdn_status)e;
}

}  // extern "C"
