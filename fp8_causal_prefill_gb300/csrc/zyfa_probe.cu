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

// ---- The attention kernel's own MMA forms, one at a time (same instruction kinds, shapes, operand
// sources and shared-memory layouts as its score and PV MMAs), each iteration issued back to back by
// one elected lane with no other work in the loop.  Forms:
//   0  FP8 score tile: S = Q K^T, M=128, N=128, D=128 (four 32-byte K steps), both operands in shared memory
//   1  FP8 PV: O += P [V | 1], block-scaled (e8m0 factors in TMEM), M=128, N=144, 128 keys, P in TMEM
//   2  form 0 then form 1 (one query tile's work per K/V tile)
//   3  the FP8 score tile as two N=64 halves (Q read twice from shared memory)
//   4  BF16 score tile: M=128, N=128, D=128 (eight K steps over two 128-byte chunks)
//   5  BF16 score tile of the MLA shape: M=128, N=64, D=192 (twelve K steps over three chunks)
// Shared memory (1024-byte aligned): Q 48 KB | K 48 KB | V 16 KB | ones 16 KB.  TMEM: S at column 0,
// O at 256, P at 416, scale factors at 480 (P) and 496 (V).
constexpr int kFormSmem = 1024 + 128 * 1024;
constexpr int kNumForms = 6;

__host__ __device__ constexpr long long form_flops(int form) {
  return form == 0 || form == 3 ? 2ll * 128 * 128 * 128
         : form == 1            ? 2ll * 128 * 144 * 128
         : form == 2            ? 2ll * 128 * 128 * 128 + 2ll * 128 * 144 * 128
         : form == 4            ? 2ll * 128 * 128 * 128
         : form == 5            ? 2ll * 128 * 64 * 192
                                : -1;
}

template <int FORM>
__global__ void __launch_bounds__(kProbeThreads, 1) zyfa_mma_form_kernel(int iters, long long* cycles, int* timed_out) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t done;
  __shared__ uint32_t tmem_base;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* p = smem_raw + (base - raw);
  constexpr uint32_t kQ = 0, kK = 48 * 1024, kV = 96 * 1024, kOnes = 112 * 1024, kEnd = 128 * 1024;
  constexpr bool kBf16 = FORM >= 4;
  // finite operands of small magnitude (e4m3 or bf16 bit patterns); e4m3 1.0 in the ones atom
  for (uint32_t i = threadIdx.x; i < kEnd / 4; i += kProbeThreads) {
    const uint32_t h = (i * 2654435761u) ^ 0x5bd1e995u;
    reinterpret_cast<uint32_t*>(p)[i] = i >= kOnes / 4 ? 0x38383838u : (kBf16 ? (h & 0xBC7FBC7Fu) : (h & 0xA7A7A7A7u));
  }
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&done), 1);
    fence_mbar_init();
  }
  const int warp = threadIdx.x >> 5;
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  // P codes and the scale factors (2^0) of P and V, each warp its lane quarter
  {
    const uint32_t lanes = static_cast<uint32_t>(warp * 32) << 16;
    uint32_t r[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) r[i] = 0x30303030u + static_cast<uint32_t>(i);
    tmem_st16(tmem + lanes + 416, r);
    tmem_st16(tmem + lanes + 432, r);
    tmem_st4(tmem + lanes + 480, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
    tmem_st4(tmem + lanes + 496, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
    tmem_st4(tmem + lanes + 500, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) {
    // K-major Q and K: 128-byte swizzled chunks of R rows, R * 128 bytes apart; a 32-byte K step moves
    // the start address by 2 (16-byte units), a chunk by R * 8
    const uint64_t qd = smem_desc(base + kQ, 16, 1024, kSwizzle128B);
    const uint64_t kd = smem_desc(base + kK, 16, 1024, kSwizzle128B);
    const uint64_t vd = smem_desc(base + kV, kOnes - kV, 1024, kSwizzle128B);  // MN-major V, ones atom by LBO
    constexpr uint32_t kN = FORM == 3 || FORM == 5 ? 64 : 128;
    constexpr int kChunks = FORM == 5 ? 3 : (FORM == 4 ? 2 : 1);
    const uint32_t idesc_s = kBf16 ? idesc_dense(kFmtBF16, kFmtBF16, false, false, 128, kN)
                                   : idesc_dense(kFmtE4M3, kFmtE4M3, false, false, 128, kN);
    auto score = [&](int it, uint32_t d, uint64_t bd) {
#pragma unroll
      for (int c = 0; c < kChunks; ++c)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t a = qd + c * (128 * 8) + ks * 2, b = bd + c * (kN * 8) + ks * 2;
          const uint32_t acc = (it | c | ks) != 0 ? 1u : 0u;
          if constexpr (kBf16) mma_f16_ss(d, a, b, idesc_s, acc);
          else mma_f8_ss(d, a, b, idesc_s, acc);
        }
    };
    auto pv = [&](int it) {
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_mxf8_ts(tmem + 256, tmem + 416 + ks * 8, vd + (ks * 32 * 128) / 16,
                    idesc_block_scaled(kFmtE4M3, kFmtE4M3, true, 128, 144, ks, 0), tmem + 480, tmem + 496,
                    (it | ks) != 0 ? 1u : 0u);
    };
    const long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
      if constexpr (FORM == 0 || FORM == 2 || FORM == 4 || FORM == 5) score(it, tmem, kd);
      if constexpr (FORM == 3) {
        score(it, tmem, kd);
        score(it, tmem + 64, kd + 64 * 8);  // keys 64..127: rows 64.. of the K tile
      }
      if constexpr (FORM == 1 || FORM == 2) pv(it);
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
  if (warp == 0) tmem_dealloc(tmem, 512);
}

template <int FORM>
zyfa_status_t launch_form(int iters, int grid, long long* cycles, int* timed_out, cudaStream_t stream) {
  if (cudaFuncSetAttribute(zyfa_mma_form_kernel<FORM>, cudaFuncAttributeMaxDynamicSharedMemorySize, kFormSmem) !=
      cudaSuccess)
    return ZYFA_ERR_CUDA;
  zyfa_mma_form_kernel<FORM><<<grid, kProbeThreads, kFormSmem, stream>>>(iters, cycles, timed_out);
  return cudaGetLastError() == cudaSuccess ? ZYFA_OK : ZYFA_ERR_CUDA;
}

}  // namespace

extern "C" {

long long zyfa_probe_mma_form_flops_per_iter(int form) { return form_flops(form); }

zyfa_status_t zyfa_probe_mma_form_rate(int form, int iters, int grid, long long* cycles, int* timed_out,
                                       cudaStream_t stream) {
  if (form < 0 || form >= kNumForms || iters < 1 || grid < 1 || !cycles || !timed_out) return ZYFA_ERR_INVALID_ARG;
  switch (form) {
    case 0: return launch_form<0>(iters, grid, cycles, timed_out, stream);
    case 1: return launch_form<1>(iters, grid, cycles, timed_out, stream);
    case 2: return launch_form<2>(iters, grid, cycles, timed_out, stream);
    case 3: return launch_form<3>(iters, grid, cycles, timed_out, stream);
    case 4: return launch_form<4>(iters, grid, cycles, timed_out, stream);
    default: return launch_form<5>(iters, grid, cycles, timed_out, stream);
  }
}

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
