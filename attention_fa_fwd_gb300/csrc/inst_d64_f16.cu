// Kernel instance: head dim 64, f16 inputs/outputs, one pass (no split of the key range).
#include "fa_fwd_kernel.cuh"

namespace fa {
int launch_d64_f16(const LaunchArgs& a, cudaStream_t s)
{
    if (a.p.split_chunk > 0) return launch_d64_f16_split(a, s);
    if (a.p.tpu == 1) return launch_d64_f16_kp(a, s);
    return launch_instance<64, false, false>(a, s);
}
}  // namespace fa
