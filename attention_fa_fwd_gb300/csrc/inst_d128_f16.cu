// Kernel instance: head dim 128, f16 inputs/outputs.
#include "fa_fwd_kernel.cuh"

namespace fa {
int launch_d128_f16(const LaunchArgs& a, cudaStream_t s) { return launch_instance<128, false>(a, s); }
}  // namespace fa
