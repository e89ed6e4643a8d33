// Kernel instance: head dim 64, f16 inputs/outputs.
#include "fa_fwd_kernel.cuh"

namespace fa {
int launch_d64_f16(const LaunchArgs& a, cudaStream_t s) { return launch_instance<64, false>(a, s); }
}  // namespace fa
