// Kernel instance: head dim 64, bf16 inputs/outputs, key range split into
// chunks, one query tile per unit as a key-parity unit (the two tile slots
// take the chunk's even and odd key tiles; the epilogue merges them).
#include "fa_fwd_kernel.cuh"

namespace fa {
int launch_d64_bf16_split_kp(const LaunchArgs& a, cudaStream_t s)
{
    return launch_instance<64, true, true, true>(a, s);
}
}  // namespace fa
