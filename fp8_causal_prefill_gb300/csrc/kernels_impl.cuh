// Launch wrapper shared by the FP8 and BF16 kernel translation units.
#pragma once
#include <atomic>
#include <cstdint>

#include "launch.h"
#include "zyfa_fwd.cuh"

namespace zyfa {

template <bool FP8, int DQK, int DV>
int smem_bytes() {
  return Cfg<FP8, DQK, DV, tile_keys<FP8, DQK, DV>()>::kSmemBytes;
}

template <bool FP8, int DQK, int DV>
int epi_cols() {
  return Cfg<FP8, DQK, DV, tile_keys<FP8, DQK, DV>()>::kEpiCols;
}

template <bool FP8, int DQK, int DV, bool EXACT>
cudaError_t launch_fwd(const LaunchArgs& a) {
  constexpr int BN = tile_keys<FP8, DQK, DV>();
  using C = Cfg<FP8, DQK, DV, BN>;
  auto kernel = zyfa_fwd_kernel<FP8, DQK, DV, BN, EXACT>;
  // the shared-memory opt-in is an attribute of the function on the current device: set it once per
  // device (a host-side cost of several microseconds that short launches would otherwise pay)
  static std::atomic<uint64_t> attr_set{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0;
  if (!bit || !(attr_set.load(std::memory_order_acquire) & bit)) {
    const cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (err != cudaSuccess) return err;
    attr_set.fetch_or(bit, std::memory_order_acq_rel);
  }
  Params p;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.q_descale = a.q_descale;
  p.k_descale = a.k_descale;
  p.v_descale = a.v_descale;
  p.B = a.B;
  p.S = a.S;
  p.H = a.H;
  p.H_kv = a.H_kv;
  p.softmax_scale = a.softmax_scale;
  p.num_units = a.num_units;
  p.qb_end = a.qb_end;
  p.status = a.status;
  p.stall_loads = a.stall_loads;
  p.lse = a.lse;
  p.desc_per_head = a.desc_per_head;
  p.no_block_scale = a.no_block_scale;
  p.rescale_binades = a.rescale_binades;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = a.stream;
  return cudaLaunchKernelEx(&cfg, kernel, p, a.maps);
}

}  // namespace zyfa
