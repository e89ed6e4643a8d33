// Kernel instance: head dim 64, fp16 inputs/outputs, key range split into
// chunks, one query tile per unit as a key-parity unit (the two tile slots
// take the chunk's even and odd key tiles; the epilogue merges them).
#include "fa_fwd_kernel.cuh"

namespace fa {
int launch_d64_f16_split_kp(const LaunchArgs& a, cudaStream_t s)
{
    return launch_instance<64, false, true, true>(a, s);
}
}  // namespace fa
