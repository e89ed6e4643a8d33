// Kernel instance: head dim 64, bf16 inputs/outputs, key range split into
// chunks, one query tile per unit, in the decoupled order (P_t in its own TMEM
// columns, so the next QK_t is issued before PV_t).
#include "fa_fwd_kernel.cuh"

namespace fa {
int launch_d64_bf16_split_dec(const LaunchArgs& a, cudaStream_t s)
{
    return launch_instance<64, true, true, true>(a, s);
}
}  // namespace fa
