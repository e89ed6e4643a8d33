// Kernel instance: one-tile layout, head dim 64, bf16 inputs/outputs.
#include "fa_fwd_wide.cuh"

namespace fa {
int launch_wide_d64_bf16(const LaunchArgs& a, cudaStream_t s) { return launch_wide_instance<64, true>(a, s); }
}  // namespace fa
