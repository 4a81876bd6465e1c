// gdn_internal.h -- layouts and kernel argument blocks shared by the host
// layer (gdn_api.cu) and the kernels.  Not part of the public ABI.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

constexpr int CHUNK = 64;   // tokens per chunk

// ---- per (chunk, value head) block written by the prep kernel ----
// T' = T diag(beta gamma rk), T'' = T diag(beta), Aqk = tril(Q^ K^T . Gamma),
// T = (I + A)^-1 (backward only), all BF16 SwTile(64 x 64); then scalars.
constexpr int CB_TP = 0;
constexpr int CB_TPP = 8192;
constexpr int CB_AQK = 16384;
constexpr int CB_T = 24576;
constexpr int CB_SCAL = 32768;   // float sc[64], kd[64], gL, (int) L
constexpr int CB_SCAL_BYTES = 1024;
constexpr int CB_BYTES = 33792;
constexpr int TILE64_BYTES = 8192;

// ---- per (chunk, value head) block of the per-channel-decay (KDA) form, written by kda_prep_kernel ----
// With G the chunk-local cumulative log decay per key channel (a 64 x 128 array), gamma = exp(G):
constexpr int KB_WT = 0;         // -W^T = -(T'' (gamma . K^))^T, BF16 SwTile(128 x 64) (rows: dk index)
constexpr int KB_KD = 16384;     // Kd = exp(G_L - G) . K^, BF16 SwTile(64 x 128)
constexpr int KB_TPP = 32768;    // T'' = T diag(beta), SwTile(64 x 64)
constexpr int KB_SCAL = 40960;   // float gamma_L[128] (per key channel); (int) L at float index 129
constexpr int KB_QT = 41984;     // Q~ = gamma . Q^, SwTile(64 x 128)
constexpr int KB_AQK = 58368;    // P = tril_incl(Q^_r . (exp(G_r - G_c) . K^_c)), SwTile(64 x 64)
constexpr int KB_T = 66560;      // T = (I + A)^-1, SwTile(64 x 64)
constexpr int KB_MT = 74752;     // M^T, M = strict_tril(K^_r . (exp(G_r - G_c) . K^_c)), SwTile(64 x 64)
constexpr int KB_BYTES = 82944;

// one saved state: BF16 S^T (dv rows x dk cols) as SwTile(128 x 128)
constexpr int STATE_BYTES = 32768;
constexpr int STATE_F32 = 128 * 128;   // an FP32 S^T, row-major [dv][dk]
constexpr int SAVED_HEADER = 4096;
// one chunk's V_new^T (forward) or dV_new^T (adjoint walk): BF16 SwTile(128 x 64)
constexpr int VN_BYTES = 16384;

// saved-set header (first bytes of `saved`)
struct SavedHeader {
  uint32_t magic, version;
  int64_t T;
  int32_t N, H, HV, dk, dv, l2norm;
  int32_t NC, NSEG, nsplit, seg_len;
  uint32_t scale_bits, cu_hash;
  int32_t form, pad;   // saved form (0 full, 1 replay)
};
constexpr uint32_t SAVED_MAGIC = 0x4744'4e31u;   // "GDN1"
constexpr uint32_t SAVED_VERSION = 4;

// ---- device tables built by the table kernel ----
struct Tables {
  int* chunk_offsets;  // [N+1]
  int* chunk_doc;      // [NC]
  int* chunk_tok0;     // [NC]
  int* chunk_len;      // [NC]
  int* seg_offsets;    // [N+1]  segments per document, prefix sum
  int* split_offsets;  // [N+1]  split segments (transfer walks) per document, prefix sum
  int* seg_doc;        // [NSEG]
  int* seg_c0;         // [NSEG] first chunk (global index)
  int* seg_c1;         // [NSEG] one past the last chunk
  int* seg_idx;        // [NSEG] index of the segment within its document
  int* seg_split;      // [NSEG] index in the split list, or -1
  int* split_seg;      // [nsplit] segments that get transfer walks (p < P-1 of split docs)
  int* sdoc_first;     // [nsdoc+1] first split index of each split document
  int* sdoc_offsets;   // [N+1]  split documents before each document, prefix sum
  int* fwalk_seg;      // [NSEG - nsdoc] segments whose full forward walk runs after the merge: all
                       //        but the first segment of each split document (that one runs with
                       //        the transfer walks, from its true start)
  int* bwalk_seg;      // [NSEG - nsdoc] segments whose full reverse walk runs after the backward
                       //        merge: all but the last segment of each split document
                       // (both in longest-first order: the walks' CTAs take them in list order)
  int* fwalk_doc;      // [NSEG - nsdoc] the same two lists in segment order, from which the ordered
  int* bwalk_doc;      //        ones are made
};

// Hash of one cu_seqlens entry (document d ends at token `end`): murmur3's
// 32-bit finaliser of the entry mixed with its index.  The hash of a whole
// cu_seqlens is the sum of its entries' hashes mod 2^32, which the host and
// the table kernel both compute (the kernel in parallel, in any order).
__host__ __device__ inline uint32_t fmix32(uint32_t h) {
  h ^= h >> 16;
  h *= 0x85ebca6bu;
  h ^= h >> 13;
  h *= 0xc2b2ae35u;
  h ^= h >> 16;
  return h;
}
__host__ __device__ inline uint32_t cu_entry_hash(int d, int end) {
  return fmix32((uint32_t)end ^ fmix32((uint32_t)d + 0x9e3779b9u));
}

struct TableArgs {
  const int* cu;
  int64_t T;
  uint32_t cu_hash;         // sum over d of cu_entry_hash(d, cu[d + 1]) of the host copy
  int N, NC, NSEG, nsplit, nsdoc;
  int seg_len, split_min;   // a document of n chunks is split iff n > split_min
  Tables t;
  int* err;
  SavedHeader hdr;          // written into `saved` when it is non-null
  uint8_t* saved;
};

struct PrepArgs {
  CUtensorMap tq, tk;
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const float* g;
  const float* beta;
  const int* chunk_tok0;
  const int* chunk_len;
  uint8_t* cb;        // [NC][HV][CB_BYTES]
  int H, HV, G, l2norm, write_T;
  float scale;
  int* err;
};

struct ScanArgs {
  CUtensorMap tq, tk, tv, to;
  const uint8_t* cb;
  const int* chunk_tok0;
  const int* chunk_len;
  const int* seg_c0;
  const int* seg_c1;
  const int* seg_idx;
  const int* seg_split;
  const int* split_seg;
  const int* walk_seg;        // walk = 0: the segments to walk (one per CTA group of HV)
  int H, HV, G, nsplit, walk;   // walk = 0: full walks after the merge; 1: B and M walks (the first
                                // segment of a split document walks in full here, writing its B)
  float scale;
  uint8_t* tape;              // [NC][HV][STATE_BYTES] or null
  uint8_t* vn;                // [NC][HV][VN_BYTES] V_new^T tiles, or null
  __nv_bfloat16* o;           // [T][HV][128] or null
  const float* s_init;        // [nsplit][HV][STATE_F32]: start of the segment after split segment i
  float* bend;                // [nsplit][HV][STATE_F32]
  float* mend;                // [nsplit][HV][STATE_F32]
  const int* seg_doc;         // [NSEG]
  const int* seg_offsets;     // [N+1]
  const float* s_in;          // [N][HV][128][128] FP32 S entering each document, or null (zero)
  float* s_out;               // [N][HV][128][128] FP32 S leaving each document, or null
  int kda;                    // 1: per-channel decay; cb holds KB_BYTES blocks (-W^T, Kd, T'', gamma_L)
  int* err;
};

// the per-channel-decay preparation of every (chunk, value head)
struct KdaPrepArgs {
  CUtensorMap tq, tk, tg;
  const float* g;             // [T][HV][128] log decay per key channel
  const float* beta;          // [T][HV]
  const int* chunk_tok0;
  const int* chunk_len;
  uint8_t* kb;                // [NC][HV][KB_BYTES] out
  int H, HV, G, l2norm;
  int* err;
};

// o = scale (Q~ S + P V_new) of every (chunk, value head), from the states and V_new^T
struct KdaOutArgs {
  CUtensorMap to;
  const uint8_t* tape;        // [NC][HV][STATE_BYTES] S^T entering each chunk
  const uint8_t* vn;          // [NC][HV][VN_BYTES] V_new^T
  const uint8_t* kb;          // [NC][HV][KB_BYTES]
  const int* chunk_tok0;
  const int* chunk_len;
  __nv_bfloat16* o;
  int HV;
  float scale;
  int* err;
};

// V_new^T of every (chunk, value head) from the saved states (replay form)
struct VnewArgs {
  CUtensorMap tk, tv;
  const uint8_t* tape;        // [NC][HV][STATE_BYTES] saved S^T
  const uint8_t* cb;          // [NC][HV][CB_BYTES] UT blocks of this call
  const int* chunk_tok0;
  const int* chunk_len;
  uint8_t* vn;                // [NC][HV][VN_BYTES] out
  int H, HV, G;
  int withhold_first_load;    // test hook: CTA 0 never requests its first tiles, so its bounded wait
                              // runs out and the call reports GDN_ERR_TIMEOUT (nothing is left in flight)
  int* err;
};

// boundary states of documents without chunks: dst[d] = src[d] (zero if src is null)
struct PassArgs {
  const int* chunk_offsets;   // [N+1]
  const float* src;           // [N][HV][STATE_F32] or null
  float* dst;                 // [N][HV][STATE_F32]
  int HV;
};

struct MergeArgs {
  const int* sdoc_first;
  const float* bend;
  const float* mend;
  float* s_init;
  int HV;
  int* err;
};

// host-side plan of one call (sizes, segment plan, buffer offsets)
struct Plan {
  int64_t T;
  int N, H, HV, G;
  int NC, NSEG, nsplit, nsdoc, seg_len, split_min, max_doc_chunks;
  int n_empty;   // documents without tokens
  int form;      // saved form: 0 full (UT blocks and V_new^T saved), 1 replay (the backward recomputes them)
  int sms;   // SMs of the current device (persistent grids)
  uint32_t cu_hash;
  // workspace offsets (bytes)
  size_t o_tables[19];
  size_t o_cb, o_bend, o_sinit, o_mend_ws;
  size_t o_dtape, o_dvn, o_dbend, o_dsinit;   // backward
  size_t o_vnb;                               // backward, replay form: recomputed V_new^T tiles
  size_t o_ktape, o_kvn;                      // KDA forward without a saved set: its tape and V_new^T
  size_t ws_fwd, ws_bwd;
  // saved offsets
  size_t s_tape, s_mseg, s_cb, s_vn, saved_bytes;
};

inline Tables tables_at(const Plan& P, uint8_t* ws) {
  Tables t;
  int** f[18] = {&t.chunk_offsets, &t.seg_offsets, &t.split_offsets, &t.chunk_doc,    &t.chunk_tok0, &t.chunk_len,
                 &t.seg_doc,       &t.seg_c0,      &t.seg_c1,        &t.seg_idx,      &t.seg_split,  &t.split_seg,
                 &t.sdoc_first,    &t.sdoc_offsets, &t.fwalk_seg,    &t.bwalk_seg,    &t.fwalk_doc,  &t.bwalk_doc};
  for (int i = 0; i < 18; ++i) *f[i] = reinterpret_cast<int*>(ws + P.o_tables[i]);
  return t;
}

// ---- host layer (gdn_api.cu) pieces that the KDA entry points (gdn_kda.cu) share ----
gdn_status make_plan(const gdn_problem* p, const int32_t* cu, Plan* P);
gdn_status make_kda_plan(const gdn_problem* p, const int32_t* cu, Plan* P);
bool device_setup();
bool aligned16(const void* p);
bool make_tmap(CUtensorMap* m, const void* base, int64_t T, int heads);
// FP32 [T][heads][128] (the per-channel log decay g): boxes of 64 tokens x 128 channels of one head,
// no swizzle, rows past T read as zero
bool make_tmap_g(CUtensorMap* m, const float* base, int64_t T, int heads);
// BF16 [T][C] with C a multiple of 256, seen as [T][C / 256][256]: boxes of `rows` tokens x 512 channels
// (two 256-channel halves, so a box lands as `rows` rows of 1 KB), no swizzle, rows past T read as zero
bool make_tmap_rows(CUtensorMap* m, const void* base, int64_t T, int C, int rows);
gdn_status run_tables(const Plan& P, const gdn_problem* p, const int32_t* cu_dev, uint8_t* ws, void* saved,
                      cudaStream_t s);
void launch_fwd_scan(const ScanArgs& a, int nchains, cudaStream_t s);
void launch_merge(const MergeArgs& a, int nsdoc, cudaStream_t s);
void launch_check_saved(const Plan& P, const gdn_problem& pr, const void* saved, uint8_t* ws, cudaStream_t s);
gdn_status run_bwd_walks(const Plan& P, const gdn_problem& pr, const void* q, const void* k, const void* dO,
                         const uint8_t* cb, int kda, const void* saved, const float* ds_out, float* ds_in,
                         uint8_t* ws, cudaStream_t s);

}  // namespace gdn
