// gdn_common.cuh -- sm_103a building blocks shared by the GDN kernels:
// swizzled shared-memory tiles, tcgen05 descriptors / MMA / TMEM access,
// mbarriers with bounded waits, TMA and bulk copies.
//
// Tile convention ("SwTile"): a row-major tile of R rows whose rows are 128
// bytes of BF16 split into 64-column panels; panel p holds columns
// [64p, 64p + 64) of every row, rows at a 128-byte pitch, and the 16-byte
// chunk j of row r sits at chunk position j ^ (r % 8) (the 128-byte swizzle
// TMA's SWIZZLE_128B mode writes).  Panels start on 1024-byte boundaries.
// Such a tile is at the same time
//   - a K-major tcgen05 operand whose M/N extent is the rows and K the columns
//   - an MN-major operand whose K extent is the rows and M/N the columns.
// A TMA box of [64 rows][64 BF16] with SWIZZLE_128B lands as one panel.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace gdn {

constexpr int CH = 64;   // chunk length
constexpr int D = 128;   // head dim (dk = dv)

// error codes mirrored from gdn.h
constexpr int ST_TIMEOUT = 6;
constexpr int ST_DEVICE = 7;
constexpr int ST_SAVED_MISMATCH = 4;
constexpr int ST_GATE_RANGE = 8;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// The first 1024-byte boundary in a dynamic shared-memory array.  The offset is
// added to the array itself (not to an integer copy of its address), so that
// the compiler keeps the result in the shared address space and every access
// through it stays a shared-memory access.
__device__ __forceinline__ uint8_t* smem_align1024(uint8_t* raw) {
  return raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
}

// ----------------------------------------------------------------------------
// SwTile addressing
// ----------------------------------------------------------------------------
__host__ __device__ __forceinline__ uint32_t sw_off(int r, int c, int R) {
  return (uint32_t)((c >> 6) * (R * 128) + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) + (c & 7) * 2);
}
// byte offset of the 16-byte chunk holding columns [8*c8, 8*c8 + 8) of row r
__host__ __device__ __forceinline__ uint32_t sw_chunk(int r, int c8, int R) {
  return (uint32_t)((c8 >> 3) * (R * 128) + r * 128 + (((c8 & 7) ^ (r & 7)) << 4));
}

// ----------------------------------------------------------------------------
// tcgen05 descriptors
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;           // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;           // 128-byte swizzle
  return d;
}
// K-major operand: tile rows = M (or N), columns = K; k-step ks = columns [16ks, 16ks+16).
// `R` is the tile's row count (it sets the panel pitch); row0 (multiple of 8)
// selects a row sub-range.
__device__ __forceinline__ uint64_t desc_k(uint32_t tile, int R, int ks, int row0 = 0) {
  return sdesc(tile + (uint32_t)((ks >> 2) * (R * 128) + row0 * 128 + (ks & 3) * 32), 0, 1024);
}
// MN-major operand: tile rows = K, columns = M (or N); k-step ks = rows [16ks, 16ks+16).
// panel0 selects the first 64-column panel used.
__device__ __forceinline__ uint64_t desc_mn(uint32_t tile, int R, int ks, int panel0 = 0) {
  return sdesc(tile + (uint32_t)(panel0 * (R * 128) + ks * 2048), (uint32_t)(R * 128), 1024);
}
// instruction descriptor: BF16 x BF16 -> FP32, dense
__host__ __device__ constexpr uint32_t idesc(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(id), "r"(acc));
}
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(id), "r"(acc));
}
// Warp-uniform issue: the whole warp executes these (descriptors stay in
// uniform registers) and one lane chosen by elect.sync issues the instruction.
__device__ __forceinline__ void mma_ss_w(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n.reg .pred p, e;\nsetp.ne.b32 p, %4, 0;\nelect.sync _|e, 0xffffffff;\n"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(id), "r"(acc));
}
__device__ __forceinline__ void mma_ts_w(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n.reg .pred p, e;\nsetp.ne.b32 p, %4, 0;\nelect.sync _|e, 0xffffffff;\n"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(id), "r"(acc));
}
__device__ __forceinline__ void mma_commit_w(uint64_t* bar) {
  asm volatile(
      "{\n.reg .pred e;\nelect.sync _|e, 0xffffffff;\n"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(smem_u32(bar)));
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
      smem_u32(bar)));
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;"); }

// TMEM allocation (one full warp executes these)
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
               "r"(ncols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t base, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(ncols));
}
// TMEM address of (lane, column); warp w may touch lanes [32*(w%4), 32*(w%4)+32)
__device__ __forceinline__ uint32_t taddr(uint32_t base, int lane, int col) {
  return base + ((uint32_t)lane << 16) + (uint32_t)col;
}

#define GDN_TMEM_LD16(addr, r)                                                                      \
  asm volatile(                                                                                     \
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14," \
      "%15}, [%16];"                                                                                \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),       \
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),    \
        "=r"(r[14]), "=r"(r[15])                                                                    \
      : "r"(addr))

// start loading 16 consecutive FP32 columns of this thread's lane (complete with tmem_wait_ld)
__device__ __forceinline__ void tmem_ld16_async(uint32_t addr, uint32_t (&r)[16]) { GDN_TMEM_LD16(addr, r); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void as_float16(const uint32_t (&r)[16], float* out) {
#pragma unroll
  for (int j = 0; j < 16; ++j) out[j] = __uint_as_float(r[j]);
}
// load 16 consecutive FP32 columns of this thread's lane
__device__ __forceinline__ void tmem_ld16(uint32_t addr, float* out) {
  uint32_t r[16];
  GDN_TMEM_LD16(addr, r);
  asm volatile("tcgen05.wait::ld.sync.aligned;");
#pragma unroll
  for (int j = 0; j < 16; ++j) out[j] = __uint_as_float(r[j]);
}
// load 32 consecutive columns (two x16 loads, one wait)
__device__ __forceinline__ void tmem_ld32(uint32_t addr, float* out) {
  uint32_t r[16], s[16];
  GDN_TMEM_LD16(addr, r);
  GDN_TMEM_LD16(addr + 16, s);
  asm volatile("tcgen05.wait::ld.sync.aligned;");
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    out[j] = __uint_as_float(r[j]);
    out[16 + j] = __uint_as_float(s[j]);
  }
}
// store 8 consecutive 32-bit columns of this thread's lane
__device__ __forceinline__ void tmem_st8(uint32_t addr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(addr), "r"(v[0]),
      "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]));
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;"); }
// store 16 consecutive FP32 columns of this thread's lane
__device__ __forceinline__ void tmem_st16(uint32_t addr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          addr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
      "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
      "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])));
}
// 16 rows x 16 columns of an M = 64 result (the rows sit in lanes [0, 16) of the
// warp's 32-lane quarter), spread over the whole warp (.16x256b.x2): value i of
// thread t is row t / 4 + 8 ((i >> 1) & 1), column 8 (i >> 2) + 2 (t % 4) + (i & 1)
// relative to the address.  Completes with tmem_wait_ld().
__device__ __forceinline__ void tmem_ld_m64_async(uint32_t addr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x2.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(addr));
}

// d0 = a0 b + d0, d1 = a1 b + d1 as one paired FP32 FMA (each component rounds as fmaf)
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b) {
  const float2 r = __ffma2_rn(make_float2(a0, a1), make_float2(b, b), make_float2(d0, d1));
  d0 = r.x;
  d1 = r.y;
}

// (d0, d1) = (b a0 + c0, b a1 + c1) as one paired FP32 FMA
__device__ __forceinline__ void fma2_to(float& d0, float& d1, float b, float a0, float a1, float c0, float c1) {
  const float2 r = __ffma2_rn(make_float2(a0, a1), make_float2(b, b), make_float2(c0, c1));
  d0 = r.x;
  d1 = r.y;
}

// (d0, d1) += (a0 b0, a1 b1) and (d0, d1) = (a0 b0, a1 b1) as paired FP32 instructions
__device__ __forceinline__ void fma2v(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  const float2 r = __ffma2_rn(make_float2(a0, a1), make_float2(b0, b1), make_float2(d0, d1));
  d0 = r.x;
  d1 = r.y;
}
__device__ __forceinline__ void mul2v(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  const float2 r = __fmul2_rn(make_float2(a0, a1), make_float2(b0, b1));
  d0 = r.x;
  d1 = r.y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ----------------------------------------------------------------------------
// mbarriers (bounded waits)
// ----------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes));
}
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
// Wait for phase `parity` of `bar` to complete.  Gives up after ~1 s (or at
// once if the call's error word is already set), records GDN_ERR_TIMEOUT and
// returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* err) {
  uint32_t done = 0;
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity));
    if (done) return true;
    if ((it & 1023) == 0) {
      uint64_t now = globaltimer();
      if (it == 0) t0 = now;
      else if (now - t0 > 1000000000ull || *(volatile int*)err != 0) {
        atomicCAS(err, 0, ST_TIMEOUT);
        return false;
      }
    }
  }
}

// Wait up to ~1 s for phase `parity` of `bar`, whatever the error word says: on an
// error path, lets copies this CTA already has in flight land before it exits.
// Returns whether the phase completed.
__device__ __forceinline__ bool mbar_drain(uint64_t* bar, uint32_t parity) {
  uint32_t done = 0;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 0;; ++it) {
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity));
    if (done) return true;
    if ((it & 1023) == 1023 && globaltimer() - t0 > 1000000000ull) return false;
  }
}

// ----------------------------------------------------------------------------
// TMA and bulk copies (completion counted on an mbarrier)
// ----------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
      "%4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}
// L2 prefetch of one box of a 3-D tensor map (a hint: nothing waits for it)
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(map), "r"(x), "r"(y),
               "r"(z)
               : "memory");
}
// L2 prefetch of a contiguous range; bytes multiple of 16, 16-byte aligned (a hint)
__device__ __forceinline__ void bulk_prefetch(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
// plain bulk copy global -> shared; bytes multiple of 16, both 16-byte aligned
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// bulk copy shared -> global (bulk-group completion); both 16-byte aligned
__device__ __forceinline__ void bulk_store(void* gdst, const void* ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(smem_u32(ssrc)),
               "r"(bytes)
               : "memory");
}
// TMA tile store shared -> global of one box of a 3-D tensor map
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* ssrc, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(map),
               "r"(x), "r"(y), "r"(z), "r"(smem_u32(ssrc))
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// wait until the source reads of every committed bulk group are done (its shared memory may be rewritten)
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// the same, except that the most recently committed group may still be reading
__device__ __forceinline__ void bulk_wait_read_but1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// wait until every committed bulk group has completed
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// barrier over one 128-thread warpgroup (named barrier `id`) that also ANDs `v` across it
__device__ __forceinline__ bool wg_sync_and(int id, bool v) {
  uint32_t r;
  asm volatile(
      "{\n.reg .pred p, q;\nsetp.ne.u32 q, %1, 0;\nbar.red.and.pred p, %2, 128, q;\nselp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id));
  return r != 0;
}
// barrier `id` over `n` threads that also ANDs `v` across them
__device__ __forceinline__ bool bar_and(int id, int n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n.reg .pred p, q;\nsetp.ne.u32 q, %1, 0;\nbar.red.and.pred p, %2, %3, q;\nselp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(n));
  return r != 0;
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads));
}

}  // namespace gdn
