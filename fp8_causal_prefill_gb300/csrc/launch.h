// Host-side launch interface between the C ABI (zyfa_api.cu) and the kernel translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

namespace zyfa {

struct LaunchArgs {
  const void* q;
  void* out;
  const float* q_descale;
  const float* k_descale;
  const float* v_descale;
  int B, S, H, H_kv;
  float softmax_scale;
  int num_units;
  int* status;
  int grid;
  CUtensorMap tm_q, tm_k0, tm_k1, tm_v;
  cudaStream_t stream;
};

// Defined for <true,64,64>, <true,128,128>, <true,192,128> in zyfa_kernels_fp8.cu and for the same
// head shapes with FP8 = false in zyfa_kernels_bf16.cu.
template <bool FP8, int DQK, int DV>
cudaError_t launch_fwd(const LaunchArgs& a);

// Dynamic shared memory the kernel instantiation needs (bytes).
template <bool FP8, int DQK, int DV>
int smem_bytes();

}  // namespace zyfa
