// Kernel instance: one-tile layout, head dim 128, f16 inputs/outputs.
#include "fa_fwd_wide.cuh"

namespace fa {
int launch_wide_d128_f16(const LaunchArgs& a, cudaStream_t s) { return launch_wide_instance<128, false>(a, s); }
}  // namespace fa
