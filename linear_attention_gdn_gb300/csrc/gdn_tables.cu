// gdn_tables.cu -- the varlen chunk-index builder.
//
// From cu_seqlens it builds, bit-exactly, the chunk tables every other kernel
// indexes (chunks of 64 tokens restart at each document start; the last chunk
// of a document holds len mod 64 tokens or a full chunk) and the segment plan
// of the intra-GPU split: a document of n > split_min chunks is cut into
// ceil(n / seg_len) segments of seg_len chunks (the last one shorter).  The
// flashinfer Cake GDN pages keep four chunk tables plus a segment table built
// from cu_seqlens ("feat(cake_gdn_kcp) ... #8172" page, commit note on the
// backend's fifth table); their contents are not printed, so these tables are
// this library's own definition.
#include <algorithm>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_prof.h"

namespace gdn {

// Block-wide exclusive scan of 4 counters (1024 threads).
__device__ __forceinline__ void block_scan4(int v[4], int excl[4], int total[4]) {
  __shared__ int warp_sums[32][4];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    int x = v[m];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    incl[m] = x;
    if (lane == 31) warp_sums[warp][m] = x;
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      int x = warp_sums[lane][m];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      warp_sums[lane][m] = x;   // inclusive over warps
    }
  }
  __syncthreads();
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    int before = warp ? warp_sums[warp - 1][m] : 0;
    excl[m] = before + incl[m] - v[m];
    total[m] = warp_sums[31][m];
  }
  __syncthreads();
}

__global__ void __launch_bounds__(1024) tables_scan_kernel(TableArgs a) {
  __shared__ uint32_t s_hash;
  __shared__ int s_bad;
  if (threadIdx.x == 0) {
    s_hash = 0u;
    s_bad = 0;
  }
  __syncthreads();
  int carry[4] = {0, 0, 0, 0};   // chunks, segments, split segments, split documents
  uint32_t hsum = 0u;            // this thread's share of the cu_seqlens hash
  int bad = 0;
  for (int base = 0; base < a.N; base += 1024) {
    const int d = base + (int)threadIdx.x;
    int v[4] = {0, 0, 0, 0};
    if (d < a.N) {
      const int lo = a.cu[d], hi = a.cu[d + 1];
      hsum += cu_entry_hash(d, hi);
      bad |= hi < lo;
      const int len = hi < lo ? 0 : hi - lo;
      const int n = (len + CH - 1) / CH;
      const int P = n > a.split_min ? (n + a.seg_len - 1) / a.seg_len : (n > 0 ? 1 : 0);
      v[0] = n;
      v[1] = P;
      v[2] = P > 1 ? P - 1 : 0;
      v[3] = P > 1 ? 1 : 0;
    }
    int excl[4], total[4];
    block_scan4(v, excl, total);
    if (d < a.N) {
      a.t.chunk_offsets[d] = carry[0] + excl[0];
      a.t.seg_offsets[d] = carry[1] + excl[1];
      a.t.split_offsets[d] = carry[2] + excl[2];
      a.t.sdoc_offsets[d] = carry[3] + excl[3];
      if (v[3] && carry[3] + excl[3] <= a.nsdoc) a.t.sdoc_first[carry[3] + excl[3]] = carry[2] + excl[2];
    }
#pragma unroll
    for (int m = 0; m < 4; ++m) carry[m] += total[m];
  }
  atomicAdd(&s_hash, hsum);   // a sum mod 2^32: the order of the additions does not matter
  if (bad) atomicOr(&s_bad, 1);
  __syncthreads();
  if (threadIdx.x == 0) {
    a.t.chunk_offsets[a.N] = carry[0];
    a.t.seg_offsets[a.N] = carry[1];
    a.t.split_offsets[a.N] = carry[2];
    a.t.sdoc_offsets[a.N] = carry[3];
    if (carry[3] <= a.nsdoc) a.t.sdoc_first[carry[3]] = carry[2];
    // The host planned from its copy of cu_seqlens.  The device copy must hold
    // the same values: cu[0] = 0, non-decreasing, cu[N] = T, and the same hash
    // of every entry (which catches, say, two documents with swapped lengths,
    // where every count above still agrees).  On any mismatch the error word
    // is set here, before the fill kernel and every later kernel of the call,
    // which all skip their work once it is set.
    if (a.cu[0] != 0 || (int64_t)a.cu[a.N] != a.T || s_bad || s_hash != a.cu_hash || carry[0] != a.NC ||
        carry[1] != a.NSEG || carry[2] != a.nsplit || carry[3] != a.nsdoc)
      atomicCAS(a.err, 0, 1 /* GDN_ERR_INVALID_ARG */);
    else if (a.saved)
      *reinterpret_cast<SavedHeader*>(a.saved) = a.hdr;
  }
}

// largest d in [0, n) with off[d] <= x  (off non-decreasing, off[0] <= x)
__device__ __forceinline__ int find_owner(const int* off, int n, int x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (off[mid] <= x) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(256) tables_fill_kernel(TableArgs a) {
  if (*(volatile int*)a.err) return;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < a.NC) {
    const int d = find_owner(a.t.chunk_offsets, a.N, i);
    const int t0 = a.cu[d] + (i - a.t.chunk_offsets[d]) * CH;
    a.t.chunk_doc[i] = d;
    a.t.chunk_tok0[i] = t0;
    a.t.chunk_len[i] = min(CH, a.cu[d + 1] - t0);
  }
  if (i < a.NSEG) {
    const int d = find_owner(a.t.seg_offsets, a.N, i);
    const int p = i - a.t.seg_offsets[d];
    const int P = a.t.seg_offsets[d + 1] - a.t.seg_offsets[d];
    const int cd0 = a.t.chunk_offsets[d], cd1 = a.t.chunk_offsets[d + 1];
    int c0 = cd0, c1 = cd1;
    if (P > 1) {
      c0 = cd0 + p * a.seg_len;
      c1 = min(c0 + a.seg_len, cd1);
    }
    a.t.seg_doc[i] = d;
    a.t.seg_c0[i] = c0;
    a.t.seg_c1[i] = c1;
    a.t.seg_idx[i] = p;
    int sp = -1;
    if (P > 1 && p < P - 1) {
      sp = a.t.split_offsets[d] + p;
      a.t.split_seg[sp] = i;
    }
    a.t.seg_split[i] = sp;
    // the segments walked in full after the merges: in the forward all but a split document's first
    // segment, in the backward all but its last (those walk from their true start / end with the
    // transfer walks); both lists in segment order here, longest first after walk_order_kernel
    const int sd = a.t.sdoc_offsets[d];
    if (!(P > 1 && p == 0)) a.t.fwalk_doc[i - sd - (P > 1 ? 1 : 0)] = i;
    if (!(P > 1 && p == P - 1)) a.t.bwalk_doc[i - sd] = i;
  }
}

// The full walks' segment lists in longest-first order, stable among equal lengths (a walk's length is
// its chunk count).  With more chains than SMs, the walks' CTAs start in list order: longest first
// leaves the short chains for the last wave, where segment order can leave a long document's chains
// to start after the others and end late (the classic longest-processing-time-first rule).
// blockIdx.y selects the list (0 forward, 1 backward); each thread ranks one entry by counting the
// entries ahead of it; lists longer than WO_MAX keep segment order.
constexpr int WO_MAX = 8192;
__global__ void __launch_bounds__(256) walk_order_kernel(Tables t, int n, const int* err) {
  __shared__ int len_s[WO_MAX];
  if (*(volatile const int*)err) return;
  const int* src = blockIdx.y == 0 ? t.fwalk_doc : t.bwalk_doc;
  int* dst = blockIdx.y == 0 ? t.fwalk_seg : t.bwalk_seg;
  if (n > WO_MAX) {
    for (int k = blockIdx.x * blockDim.x + threadIdx.x; k < n; k += gridDim.x * blockDim.x) dst[k] = src[k];
    return;
  }
  for (int k = threadIdx.x; k < n; k += blockDim.x) len_s[k] = t.seg_c1[src[k]] - t.seg_c0[src[k]];
  __syncthreads();
  for (int k = blockIdx.x * blockDim.x + threadIdx.x; k < n; k += gridDim.x * blockDim.x) {
    const int lk = len_s[k];
    int rank = 0;
    for (int j = 0; j < n; ++j) {
      const int lj = len_s[j];
      rank += (lj > lk || (lj == lk && j < k)) ? 1 : 0;
    }
    dst[rank] = src[k];
  }
}

void launch_tables(const TableArgs& a, cudaStream_t s) {
  prof_begin(K_TABLES_SCAN, s);
  tables_scan_kernel<<<1, 1024, 0, s>>>(a);
  prof_end(K_TABLES_SCAN, s);
  const int n = a.NC > a.NSEG ? a.NC : a.NSEG;
  if (n > 0) {
    prof_begin(K_TABLES_FILL, s);
    tables_fill_kernel<<<(n + 255) / 256, 256, 0, s>>>(a);
    prof_end(K_TABLES_FILL, s);
  }
  const int nw = a.NSEG - a.nsdoc;
  if (nw > 0) {
    prof_begin(K_WALK_ORDER, s);
    walk_order_kernel<<<dim3((unsigned)std::min((nw + 255) / 256, 64), 2), 256, 0, s>>>(a.t, nw, a.err);
    prof_end(K_WALK_ORDER, s);
  }
}

}  // namespace gdn
