// FP8 e4m3 instantiations of the causal prefill kernel (Lean P).
#include "kernels_impl.cuh"

namespace zyfa {
template cudaError_t launch_fwd<true, 64, 64, false>(const LaunchArgs&);
template cudaError_t launch_fwd<true, 128, 128, false>(const LaunchArgs&);
template cudaError_t launch_fwd<true, 192, 128, false>(const LaunchArgs&);
template int smem_bytes<true, 64, 64>();
template int epi_cols<true, 64, 64>();
template int smem_bytes<true, 128, 128>();
template int epi_cols<true, 128, 128>();
template int smem_bytes<true, 192, 128>();
template int epi_cols<true, 192, 128>();
}  // namespace zyfa
