// gdn_probe.cu -- the tensor-pipe probe behind the roofline's own BF16 peak:
// one CTA per SM issues back-to-back BF16 tcgen05 products (M = 128, N = 256,
// K = 16, the largest single-CTA shape) on operand tiles resident in shared
// memory, accumulating into one TMEM tile.  No operand moves during the loop,
// so the rate is what the tensor cores alone sustain at the running clock: the
// ceiling a kernel of this library could reach with perfect operand delivery.
#include <cuda_runtime.h>

#include "gdn.h"
#include "gdn_common.cuh"

namespace gdn {

constexpr int PB_THREADS = 128;
constexpr int PB_A = 0;                    // A: 128 rows x 64 K columns, one 128-byte swizzled panel (16 KB)
constexpr int PB_B = 16384;                // B: 256 rows x 64 K columns (32 KB)
constexpr int PB_SMEM = PB_B + 32768;
constexpr int PB_SMEM_ALLOC = PB_SMEM + 1024;
constexpr int PB_M = 128, PB_N = 256, PB_K = 16, PB_KSTEPS = 4;   // four K = 16 steps per panel

__global__ void __launch_bounds__(PB_THREADS, 1) tensor_probe_kernel(int iters, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_align1024(smem_raw);
  __shared__ uint64_t bar;
  __shared__ uint32_t tslot;
  const int tid = threadIdx.x, warp = tid >> 5;
  // zero operands: the values do not matter to the rate, and zeros keep the sums finite
  for (int i = tid; i < PB_SMEM / 16; i += PB_THREADS) reinterpret_cast<uint4*>(sm)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_async_smem();
  if (warp == 0) tmem_alloc(&tslot, PB_N);
  if (tid == 0) {
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tslot, sa = smem_u32(sm + PB_A), sb = smem_u32(sm + PB_B);
  if (warp == 0) {
    for (int it = 0; it < iters; ++it)
#pragma unroll
      for (int ks = 0; ks < PB_KSTEPS; ++ks)
        mma_ss_w(tb, desc_k(sa, PB_M, ks), desc_k(sb, PB_N, ks), idesc(PB_M, PB_N, 0, 0), (it | ks) != 0);
    mma_commit_w(&bar);   // arrives once every product above has completed
  }
  if (!__syncthreads_and(mbar_wait(&bar, 0, err)) && tid == 0) mbar_drain(&bar, 0);
  tc_fence_after();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, PB_N);
}

}  // namespace gdn

extern "C" gdn_status gdn_tensor_probe(int32_t iters, int32_t* dev_err, double* flops, cudaStream_t stream) {
  using namespace gdn;
  if (iters <= 0 || iters > (1 << 20) || !dev_err || !flops) return GDN_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return GDN_ERR_CUDA;
  if (cudaFuncSetAttribute(tensor_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, PB_SMEM_ALLOC) !=
      cudaSuccess)
    return GDN_ERR_CUDA;
  tensor_probe_kernel<<<sms, PB_THREADS, PB_SMEM_ALLOC, stream>>>(iters, dev_err);
  if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
  *flops = 2.0 * PB_M * PB_N * PB_K * PB_KSTEPS * (double)iters * (double)sms;
  return GDN_OK;
}
