// Kernel instance: head dim 64, bf16 inputs/outputs.
#include "fa_fwd_kernel.cuh"

namespace fa {
int launch_d64_bf16(const LaunchArgs& a, cudaStream_t s) { return launch_instance<64, true>(a, s); }
}  // namespace fa
