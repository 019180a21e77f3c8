// Host-side launch interface between the C ABI (zyfa_api.cu) and the kernel translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

namespace zyfa {

// 4-D tensor maps over [B][S][heads][D]; *0 move 128-byte chunks of a row, *1 its 64-byte tail chunk.
struct Maps {
  CUtensorMap q0, q1, k0, k1, v;
  CUtensorMap o;  // bf16 output, stored by TMA from a per-warp staging tile
};

struct LaunchArgs {
  void* out;
  const float* q_descale;
  const float* k_descale;
  const float* v_descale;
  int B, S, H, H_kv;
  float softmax_scale;
  int num_units;
  int qb_end;  // last query block (exclusive) of the processed range
  int* status;
  int stall_loads;    // nonzero only for the stalled-pipeline self-test
  float* lse;         // optional log-sum-exp output [B,H,S]
  int desc_per_head;  // descales indexed by (batch, KV head)
  int no_block_scale; // exact P only: round against the row reference, no per-block scaling
  int rescale_binades;  // block-scaled FP8: largest lag of the row reference before a rescale
  int grid;
  Maps maps;
  cudaStream_t stream;
};

// Keys per K/V tile of an instantiation (the TMA box height of the K and V maps).
template <bool FP8, int DQK, int DV>
constexpr int tile_keys() {
  return (!FP8 && DQK == 192) ? 64 : 128;
}

// Defined for the head shapes (64,64), (128,128), (192,128): FP8 with Lean P in zyfa_kernels_fp8.cu,
// FP8 with exact P (EXACT = true) in zyfa_kernels_fp8_exact.cu, BF16 in zyfa_kernels_bf16.cu.
template <bool FP8, int DQK, int DV, bool EXACT>
cudaError_t launch_fwd(const LaunchArgs& a);

// Dynamic shared memory the kernel instantiation needs (bytes).
template <bool FP8, int DQK, int DV>
int smem_bytes();

// Output columns per TMA store box of the instantiation's epilogue (32, or 16 where shared memory
// is short); the output map's box is 32 rows x this many columns.
template <bool FP8, int DQK, int DV>
int epi_cols();

}  // namespace zyfa
