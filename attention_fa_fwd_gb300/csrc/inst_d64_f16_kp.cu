// Kernel instance: head dim 64, fp16 inputs/outputs, one pass, one query tile
// per unit as a key-parity unit (the two tile slots take the query tile's
// even and odd key tiles; the epilogue merges them).
#include "fa_fwd_kernel.cuh"

namespace fa {
int launch_d64_f16_kp(const LaunchArgs& a, cudaStream_t s)
{
    return launch_instance<64, false, false, true>(a, s);
}
}  // namespace fa
