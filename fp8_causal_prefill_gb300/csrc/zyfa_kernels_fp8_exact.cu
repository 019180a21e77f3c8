// FP8 e4m3 instantiations of the causal prefill kernel with exact P (hardware exponential and e4m3
// rounding per probability in place of Lean P), the comparison point for the Lean-P ablation.
#include "kernels_impl.cuh"

namespace zyfa {
template cudaError_t launch_fwd<true, 64, 64, true>(const LaunchArgs&);
template cudaError_t launch_fwd<true, 128, 128, true>(const LaunchArgs&);
template cudaError_t launch_fwd<true, 192, 128, true>(const LaunchArgs&);
}  // namespace zyfa
