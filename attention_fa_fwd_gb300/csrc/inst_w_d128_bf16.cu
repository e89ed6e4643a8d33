// Kernel instance: one-tile layout, head dim 128, bf16 inputs/outputs.
#include "fa_fwd_wide.cuh"

namespace fa {
int launch_wide_d128_bf16(const LaunchArgs& a, cudaStream_t s) { return launch_wide_instance<128, true>(a, s); }
int wide_smem_bytes_for(int D) { return D == 64 ? WideCfg<64>::kSmemBytes : WideCfg<128>::kSmemBytes; }
}  // namespace fa
