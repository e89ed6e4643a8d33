// Launch parameters shared by the host launcher and the kernel instances.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fa {

constexpr int kBM = 128;       // query rows per tile (one TMEM lane per row)
constexpr int kBN = 128;       // keys per K/V tile
constexpr int kThreads = 512;  // 4 warpgroups: softmax x2, correction/epilogue, load+MMA

// Work-unit schedule and problem constants, identical for every CTA.
struct Params {
    float* lse;                 // [B*H, S] fp32 output
    unsigned int* status;       // device status word (bounded-wait give-ups)
    unsigned long long timeout_ns;
    int BH;                     // B * H
    int S;                      // sequence length
    int n_qtiles;               // ceil(S / 128)
    int n_kv;                   // ceil(S / 128)
    int tpu;                    // query tiles per work unit: 1 or 2
    int n_qgroups;              // ceil(n_qtiles / tpu)
    int n_units;                // BH * n_qgroups
    int head_group;             // heads whose units are interleaved, longest first
    int causal;                 // 1: key j allowed for query i iff j <= i
    int mask_last;              // the last K/V tile of a query tile needs masking
    float scale_log2;           // scale * log2(e)
};

struct LaunchArgs {
    CUtensorMap tm_q, tm_k, tm_v, tm_o;
    Params p;
    int grid;
};

// One launcher per (head dim, dtype) instance; each lives in its own
// translation unit.  Returns a cudaError_t.
int launch_d64_f16(const LaunchArgs& a, cudaStream_t s);
int launch_d64_bf16(const LaunchArgs& a, cudaStream_t s);
int launch_d128_f16(const LaunchArgs& a, cudaStream_t s);
int launch_d128_bf16(const LaunchArgs& a, cudaStream_t s);

// Dynamic shared memory of the instance for head dim D.
int smem_bytes_for(int D);

// Kernel that waits on a barrier nobody arrives on (bounded-wait self-test).
int launch_wait_selftest(unsigned int* status, unsigned long long timeout_ns, cudaStream_t s);

}  // namespace fa
