// Self-test of the bounded mbarrier wait: one CTA waits on a barrier that no
// thread ever arrives on.  The wait gives up after the time limit, records its
// site in the status word and the kernel returns normally.
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

}  // namespace fa
