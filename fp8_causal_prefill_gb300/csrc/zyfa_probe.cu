// Tensor-core rate probe: the dense FP8 (kind::f8f6f4) and BF16 (kind::f16) MMA throughput of this GPU,
// measured with the same instruction forms, operand layouts and issue pattern as the attention kernel.
//
// The attention kernel's headline figure is a fraction of the FP8 tensor peak (captivela ZYFA article,
// "Angka Nyata": FP8 prefill throughput quoted as a share of the FP8 peak).  The probe gives that peak
// as a measurement: one persistent CTA per SM; one elected lane of warp 0 issues back-to-back
// M=128, N=256 MMAs (four 32-byte K steps of a 128-byte swizzled row each) into one TMEM accumulator,
// with both operands resident in shared memory; the clock64 span of each CTA is written out, so the
// host gets both the wall-clock rate (CUDA events) and the per-SM FLOP per cycle.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/zyfa.h"
#include "ptx.cuh"

namespace {

using namespace zyfa::ptx;

constexpr int kProbeThreads = 128;
constexpr int kProbeM = 128, kProbeN = 256;
constexpr int kABytes = kProbeM * 128, kBBytes = kProbeN * 128;
// shared memory above 114 KiB keeps it to one CTA per SM
constexpr int kProbeSmem = 1024 + 128 * 1024;
constexpr long long kProbeWaitLimit = 1ll << 33;  // a few seconds of SM clocks

__global__ void __launch_bounds__(kProbeThreads, 1)
    zyfa_mma_rate_kernel(int fp8, int iters, long long* cycles, int* timed_out) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t done;
  __shared__ uint32_t tmem_base;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* p = smem_raw + (base - raw);
  // operands: finite e4m3 / bf16 bit patterns of small magnitude (the clock under load depends on the
  // operand values, so they are not all zero)
  for (int i = threadIdx.x; i < (kABytes + kBBytes) / 4; i += kProbeThreads) {
    const uint32_t h = (static_cast<uint32_t>(i) * 2654435761u) ^ 0x5bd1e995u;
    reinterpret_cast<uint32_t*>(p)[i] = fp8 ? (h & 0xA7A7A7A7u) : (h & 0xBC7FBC7Fu);
  }
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&done), 1);
    fence_mbar_init();
  }
  const int warp = threadIdx.x >> 5;
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_base), kProbeN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  if (warp == 0) {
    const uint64_t ad = smem_desc(base, 16, 1024, kSwizzle128B);
    const uint64_t bd = smem_desc(base + kABytes, 16, 1024, kSwizzle128B);
    const uint32_t idesc = fp8 ? idesc_dense(kFmtE4M3, kFmtE4M3, false, false, kProbeM, kProbeN)
                               : idesc_dense(kFmtBF16, kFmtBF16, false, false, kProbeM, kProbeN);
    const long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const uint32_t acc = (it | ks) != 0 ? 1u : 0u;
        if (fp8) mma_f8_ss(tmem, ad + ks * 2, bd + ks * 2, idesc, acc);
        else mma_f16_ss(tmem, ad + ks * 2, bd + ks * 2, idesc, acc);
      }
    }
    tc_commit(smem_u32(&done));
    const int never = 0;
    const bool ok = mbar_wait_warp(smem_u32(&done), 0, &never, kProbeWaitLimit);
    const long long t1 = clock64();
    if ((threadIdx.x & 31) == 0) {
      cycles[blockIdx.x] = t1 - t0;
      if (!ok) atomicOr(timed_out, 1);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kProbeN);
}

}  // namespace

extern "C" {

long long zyfa_probe_mma_flops_per_iter(int fp8) {
  // four K steps of 32 bytes: 4 x 32 e4m3 or 4 x 16 bf16 products per output, 2 FLOP each
  return 2ll * kProbeM * kProbeN * (fp8 ? 128 : 64);
}

zyfa_status_t zyfa_probe_mma_rate(int fp8, int iters, int grid, long long* cycles, int* timed_out,
                                  cudaStream_t stream) {
  if ((fp8 != 0 && fp8 != 1) || iters < 1 || grid < 1 || !cycles || !timed_out) return ZYFA_ERR_INVALID_ARG;
  if (cudaFuncSetAttribute(zyfa_mma_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kProbeSmem) !=
      cudaSuccess)
    return ZYFA_ERR_CUDA;
  zyfa_mma_rate_kernel<<<grid, kProbeThreads, kProbeSmem, stream>>>(fp8, iters, cycles, timed_out);
  return cudaGetLastError() == cudaSuccess ? ZYFA_OK : ZYFA_ERR_CUDA;
}

}  // extern "C"
