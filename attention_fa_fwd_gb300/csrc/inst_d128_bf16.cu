// Kernel instance: head dim 128, bf16 inputs/outputs, one pass (no split of the key range).
#include "fa_fwd_kernel.cuh"

namespace fa {
int launch_d128_bf16(const LaunchArgs& a, cudaStream_t s)
{
    if (a.p.split_chunk > 0) return launch_d128_bf16_split(a, s);
    return launch_instance<128, true, false>(a, s);
}
}  // namespace fa
