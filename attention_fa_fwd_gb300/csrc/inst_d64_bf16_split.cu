// Kernel instance: head dim 64, bf16 inputs/outputs, split over key chunks.
#include "fa_fwd_kernel.cuh"

namespace fa {
int launch_d64_bf16_split(const LaunchArgs& a, cudaStream_t s)
{
    if (a.p.tpu == 1) return launch_d64_bf16_split_kp(a, s);
    return launch_instance<64, true, true>(a, s);
}
}  // namespace fa
