// BF16 instantiations of the causal prefill kernel (same schedule as FP8).
#include "kernels_impl.cuh"

namespace zyfa {
template cudaError_t launch_fwd<false, 64, 64, false>(const LaunchArgs&);
template cudaError_t launch_fwd<false, 128, 128, false>(const LaunchArgs&);
template cudaError_t launch_fwd<false, 192, 128, false>(const LaunchArgs&);
template int smem_bytes<false, 64, 64>();
template int epi_cols<false, 64, 64>();
template int smem_bytes<false, 128, 128>();
template int epi_cols<false, 128, 128>();
template int smem_bytes<false, 192, 128>();
template int epi_cols<false, 192, 128>();
}  // namespace zyfa
