// Self-tests of two device building blocks:
// - the bounded mbarrier wait: one CTA waits on a barrier that no thread ever
//   arrives on; the wait gives up after the time limit, records its site in
//   the status word and the kernel returns normally;
// - the FMA-pipe exponential ptx::f2_exp2_poly, evaluated element-wise so a
//   test can hold it to its error bound.
#include "fa_fwd_common.h"
#include "ptx.cuh"

namespace fa {

constexpr uint32_t kSiteSelftest = 0x700;

__global__ void wait_selftest_kernel(unsigned int* status, unsigned long long timeout_ns)
{
    __shared__ __align__(8) unsigned long long bar;
    __shared__ uint32_t abort_word;
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_u32(&bar), 1);
        abort_word = 0u;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    const ptx::WaitCtx wc{ptx::smem_u32(&abort_word), timeout_ns, status};
    ptx::mbar_wait(wc, ptx::smem_u32(&bar), 0u, kSiteSelftest);
    __syncthreads();
}

int launch_wait_selftest(unsigned int* status, unsigned long long timeout_ns, cudaStream_t s)
{
    wait_selftest_kernel<<<1, 32, 0, s>>>(status, timeout_ns);
    return (int)cudaGetLastError();
}

// y[i] = 2^x[i] by ptx::f2_exp2_poly; elements go through it in pairs (the
// second of an odd tail pairs with itself).
__global__ void exp2_poly_selftest_kernel(const float* __restrict__ x, float* __restrict__ y, int n)
{
    const int pairs = (n + 1) / 2;
    for (int k = blockIdx.x * blockDim.x + threadIdx.x; k < pairs; k += gridDim.x * blockDim.x) {
        const int i0 = 2 * k, i1 = (2 * k + 1 < n) ? 2 * k + 1 : 2 * k;
        float y0, y1;
        ptx::f2_unpack(ptx::f2_exp2_poly(x[i0], x[i1]), y0, y1);
        y[i0] = y0;
        if (i1 != i0) y[i1] = y1;
    }
}

int launch_exp2_poly_selftest(const float* x, float* y, int n, cudaStream_t s)
{
    const int pairs = (n + 1) / 2;
    const int blocks = (pairs + 255) / 256 < 1024 ? (pairs + 255) / 256 : 1024;
    exp2_poly_selftest_kernel<<<blocks, 256, 0, s>>>(x, y, n);
    return (int)cudaGetLastError();
}

}  // namespace fa
