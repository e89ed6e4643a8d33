// Split-KV merge: every output row has one partial (O_c normalised by its own
// row sum, fp32, and LSE_c) per key chunk.  The row's result is the softmax
// over all its keys, i.e. the chunks weighted by exp(LSE_c - LSE):
//   LSE = m + ln sum_c exp(LSE_c - m),  m = max_c LSE_c
//   O   = sum_c exp(LSE_c - LSE) O_c
// One thread per (row, 4 consecutive columns); HBM-bound and tiny next to the
// attention kernel.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_fwd_common.h"

namespace fa {

namespace {

template <bool kBF16>
__global__ void merge_kernel(MergeArgs a)
{
    const int per_row = a.D / 4;
    const long long total = (long long)a.BH * a.S * per_row;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int d4 = (int)(i % per_row);
        const long long rs = i / per_row;
        const int s = (int)(rs % a.S);
        const int bh = (int)(rs / a.S);
        const int qt = s / 128, row = s % 128;
        const int qg = qt / a.tpu, t = qt % a.tpu;
        int base = bh * a.units_per_head;
        for (int g = 0; g < qg; ++g) base += split_chunks(g, a.tpu, a.n_qtiles, a.n_kv, a.causal, a.chunk);
        const int n = (kv_tiles_of(qt, a.n_kv, a.causal) + a.chunk - 1) / a.chunk;
        float m = -INFINITY;
        for (int c = 0; c < n; ++c) m = fmaxf(m, a.ws_lse[((size_t)(base + c) * a.tpu + t) * 128 + row]);
        float sum = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c = 0; c < n; ++c) {
            const size_t slot = ((size_t)(base + c) * a.tpu + t) * 128 + row;
            const float w = expf(a.ws_lse[slot] - m);
            const float4 v = *reinterpret_cast<const float4*>(a.ws_o + slot * a.D + 4 * d4);
            sum += w;
            acc.x += w * v.x;
            acc.y += w * v.y;
            acc.z += w * v.z;
            acc.w += w * v.w;
        }
        const float inv = 1.f / sum;
        const size_t out = ((size_t)bh * a.S + s) * a.D + 4 * d4;
        if constexpr (kBF16) {
            __nv_bfloat162* o = reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(a.o) + out);
            o[0] = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
            o[1] = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
        } else {
            __half2* o = reinterpret_cast<__half2*>(static_cast<__half*>(a.o) + out);
            o[0] = __floats2half2_rn(acc.x * inv, acc.y * inv);
            o[1] = __floats2half2_rn(acc.z * inv, acc.w * inv);
        }
        if (d4 == 0) a.lse[(size_t)bh * a.S + s] = m + logf(sum);
    }
}

}  // namespace

int launch_merge(const MergeArgs& a, cudaStream_t s)
{
    const long long total = (long long)a.BH * a.S * (a.D / 4);
    long long blocks = (total + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    if (a.bf16)
        merge_kernel<true><<<(unsigned)blocks, 256, 0, s>>>(a);
    else
        merge_kernel<false><<<(unsigned)blocks, 256, 0, s>>>(a);
    return (int)cudaGetLastError();
}

}  // namespace fa
