// Kernel instance: head dim 64, bf16 inputs/outputs, one pass (no split of the key range).
#include "fa_fwd_kernel.cuh"

namespace fa {
int launch_d64_bf16(const LaunchArgs& a, cudaStream_t s)
{
    if (a.p.split_chunk > 0) return launch_d64_bf16_split(a, s);
    if (a.p.tpu == 1) return launch_d64_bf16_kp(a, s);
    return launch_instance<64, true, false>(a, s);
}
}  // namespace fa
