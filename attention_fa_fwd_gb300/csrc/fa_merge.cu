// Split-KV merge: every output row has one partial per key chunk (O_c, already
// normalised by the chunk's own row sum, fp32, and LSE_c).  The row's result is
// the softmax over all its keys, i.e. the chunks weighted by their share of the
// softmax mass ("FlashAttention的Triton性能考古学", 核心算法回顾, applied to
// whole chunks):
//   LSE = m + ln sum_c exp(LSE_c - m),  m = max_c LSE_c
//   O   = sum_c exp(LSE_c - LSE) O_c
//
// One block per (batch*head, query tile, 32 rows).  The partials come from L2
// and each dependent load costs a full round trip, so the block first turns
// each row's LSE_c into weights in shared memory (one thread per row), then
// every thread takes (row, 8 columns) slices and issues the loads of eight
// chunks before it does any arithmetic; neighbouring threads read and write
// neighbouring columns of a row.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_fwd_common.h"

namespace fa {

namespace {

constexpr int kMergeThreads = 256;
constexpr int kRows = 32;          // rows of a query tile per block
constexpr int kMaxChunks = 64;     // weights kept in shared memory per row
constexpr int kBatch = 8;          // chunks whose loads are in flight together

template <bool kBF16>
__device__ __forceinline__ uint32_t pack16(float lo, float hi)
{
    if constexpr (kBF16) {
        const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&v);
    } else {
        const __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&v);
    }
}

__device__ __forceinline__ void fma8(float (&acc)[8], float w, const float4& v0, const float4& v1)
{
    acc[0] = fmaf(w, v0.x, acc[0]);
    acc[1] = fmaf(w, v0.y, acc[1]);
    acc[2] = fmaf(w, v0.z, acc[2]);
    acc[3] = fmaf(w, v0.w, acc[3]);
    acc[4] = fmaf(w, v1.x, acc[4]);
    acc[5] = fmaf(w, v1.y, acc[5]);
    acc[6] = fmaf(w, v1.z, acc[6]);
    acc[7] = fmaf(w, v1.w, acc[7]);
}

template <bool kBF16>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(MergeArgs a)
{
    __shared__ float w[kMaxChunks][kRows];
    __shared__ float mi[2][kRows];     // per row: max LSE_c and 1 / sum (chunks beyond kMaxChunks)
    __shared__ int first_s;
    // launched as a programmatic dependent of the attention kernel: wait until
    // that grid has completed and its partials are visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int blocks_per_tile = 128 / kRows;
    const int tile = blockIdx.x / blocks_per_tile, r0 = (blockIdx.x % blocks_per_tile) * kRows;
    const int bh = tile / a.n_qtiles, qt = tile % a.n_qtiles;
    const int qg = qt / a.tpu, t = qt % a.tpu;
    const int n = (kv_tiles_of(qt, a.n_qtiles, a.causal) + a.chunk - 1) / a.chunk;
    if (threadIdx.x == 0) {
        int first = bh * a.units_per_head;
        for (int g = 0; g < qg; ++g) first += split_chunks(g, a.tpu, a.n_qtiles, a.n_qtiles, a.causal, a.chunk);
        first_s = first;
    }
    __syncthreads();
    const size_t step = (size_t)a.tpu * 128;            // slots between consecutive chunks of a row
    const size_t slot0 = ((size_t)first_s * a.tpu + t) * 128 + r0;
    // weights: thread r < kRows owns row r0 + r; the LSE_c are loaded kBatch at
    // a time (independent loads, one round trip per batch), with a running
    // maximum and a sum rescaled as the maximum moves
    if (threadIdx.x < kRows) {
        const int r = threadIdx.x;
        const float* lse_c = a.ws_lse + slot0 + r;
        float m = -INFINITY, sum = 0.f;
        for (int c0 = 0; c0 < n; c0 += kBatch) {
            float x[kBatch];
#pragma unroll
            for (int i = 0; i < kBatch; ++i) x[i] = c0 + i < n ? lse_c[(c0 + i) * step] : -INFINITY;
            float mb = x[0];
#pragma unroll
            for (int i = 1; i < kBatch; ++i) mb = fmaxf(mb, x[i]);
            const float mn = fmaxf(m, mb);
            float sb = 0.f;
#pragma unroll
            for (int i = 0; i < kBatch; ++i) sb += __expf(x[i] - mn);
            sum = sum * __expf(m - mn) + sb;   // m = -inf only before the first batch, where sum = 0
            m = mn;
#pragma unroll
            for (int i = 0; i < kBatch; ++i)
                if (c0 + i < n && c0 + i < kMaxChunks) w[c0 + i][r] = x[i];
        }
        const float inv = 1.f / sum;
        for (int c = 0; c < n && c < kMaxChunks; ++c) w[c][r] = __expf(w[c][r] - m) * inv;
        mi[0][r] = m;
        mi[1][r] = inv;
        const int qrow = qt * 128 + r0 + r;
        if (qrow < a.S) a.lse[(size_t)bh * a.S + qrow] = m + logf(sum);
    }
    __syncthreads();
    // one (row, 8 columns) slice per thread and pass; neighbouring threads take
    // neighbouring columns of a row, so reads and writes are coalesced
    const int per_row = a.D / 8;
    for (int idx = threadIdx.x; idx < kRows * per_row; idx += kMergeThreads) {
        const int r = idx / per_row, c8 = idx % per_row;
        const int qrow = qt * 128 + r0 + r;
        if (qrow >= a.S) continue;
        const float* src = a.ws_o + (slot0 + r) * a.D + c8 * 8;
        const size_t cstep = step * a.D;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int c0 = 0; c0 < n; c0 += kBatch) {
            float4 v[kBatch][2];
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                if (c0 + i < n) {
                    const float4* p = reinterpret_cast<const float4*>(src + (size_t)(c0 + i) * cstep);
                    v[i][0] = p[0];
                    v[i][1] = p[1];
                } else {
                    v[i][0] = v[i][1] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                const int c = c0 + i;
                float wc = 0.f;
                if (c < n) wc = c < kMaxChunks ? w[c][r] : __expf(a.ws_lse[slot0 + r + c * step] - mi[0][r]) * mi[1][r];
                fma8(acc, wc, v[i][0], v[i][1]);
            }
        }
        uint16_t* dst = static_cast<uint16_t*>(a.o) + ((size_t)bh * a.S + qrow) * a.D + c8 * 8;
        *reinterpret_cast<uint4*>(dst) = make_uint4(pack16<kBF16>(acc[0], acc[1]), pack16<kBF16>(acc[2], acc[3]),
                                                    pack16<kBF16>(acc[4], acc[5]), pack16<kBF16>(acc[6], acc[7]));
    }
}

}  // namespace

// Launched with programmatic stream serialisation: the attention kernel lets
// its dependents launch from its start, so this grid is scheduled while the
// attention grid still runs and its blocks take SMs as they free up;
// griddepcontrol.wait above still orders every read after the partials.
int launch_merge(const MergeArgs& a, bool bf16, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.BH * (unsigned)a.n_qtiles * (128 / kRows), 1, 1);
    cfg.blockDim = dim3(kMergeThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = bf16 ? cudaLaunchKernelEx(&cfg, merge_kernel<true>, a) : cudaLaunchKernelEx(&cfg, merge_kernel<false>, a);
    return (int)e;
}

}  // namespace fa
