// Kernel instance: head dim 128, f16 inputs/outputs, one pass (no split of the key range).
#include "fa_fwd_kernel.cuh"

namespace fa {
int launch_d128_f16(const LaunchArgs& a, cudaStream_t s)
{
    if (a.p.split_chunk > 0) return launch_d128_f16_split(a, s);
    return launch_instance<128, false, false>(a, s);
}
}  // namespace fa
