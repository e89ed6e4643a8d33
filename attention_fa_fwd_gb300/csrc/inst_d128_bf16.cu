// Kernel instance: head dim 128, bf16 inputs/outputs.
#include "fa_fwd_kernel.cuh"

namespace fa {
int launch_d128_bf16(const LaunchArgs& a, cudaStream_t s) { return launch_instance<128, true>(a, s); }
}  // namespace fa
