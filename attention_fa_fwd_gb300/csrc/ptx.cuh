// Inline-PTX building blocks for sm_103a: mbarriers with bounded waits, TMA
// tensor copies, tcgen05 (tensor memory allocation, MMA, commit, TMEM loads and
// stores) and the shared-memory / instruction descriptors tcgen05.mma reads.
//
// The mbarrier wait is written out by hand ("G6: Cluster 与 2CTA 探索", V40:
// a library wait whose retry path the compiler outlined spilled the barrier
// address onto the critical path).  Unlike the page's loop it is bounded: after
// a time limit it records where it gave up and returns false, and every caller
// unwinds, so a lost arrival can never hang the GPU.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace fa {
namespace ptx {

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// The warp's index in the block, broadcast from lane 0 so the compiler can
// prove it warp-uniform: code under branches on it then stays on the uniform
// datapath (tcgen05 takes its descriptors and tensor-memory addresses from
// uniform registers).  Measured 4-9% over threadIdx.x / 32 at the kernel's
// role dispatch (inside the roles the warp's quarter stays threadIdx.x-based:
// broadcasting it too measured 1-2% slower on the large workloads).
__device__ __forceinline__ int warp_id_uniform()
{
    return __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t ld_shared_volatile(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void st_shared_volatile(uint32_t addr, uint32_t v)
{
    asm volatile("st.volatile.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void ld_shared_v4(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// ---- mbarrier ---------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// The issuing instructions below take a predicate `on`: a role that runs on a
// whole warp (so the warp never diverges) issues them from one lane without a
// branch around them.
__device__ __forceinline__ void mbar_arrive(uint32_t bar, uint32_t on = 1u)
{
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %1, 0;\n\t"
        "@q mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];\n\t}" ::"r"(bar), "r"(on)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes, uint32_t on = 1u)
{
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t"
        "@q mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(bar), "r"(bytes),
        "r"(on)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t"
        ".reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t"
        "}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Where a CTA gives up: the abort word in shared memory (other roles poll it and
// unwind), the time limit, and the device status word the host reads.
struct WaitCtx {
    uint32_t abort_addr;
    unsigned long long timeout_ns;
    unsigned int* status;
};

// Wait for the phase of `bar` with parity `parity`.  Returns false when the CTA
// aborts: this wait ran past the limit (it records `site`, non-zero) or another
// role of the CTA already gave up.
__device__ __forceinline__ bool mbar_wait(const WaitCtx& w, uint32_t bar, uint32_t parity, uint32_t site)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 15u) == 0u) {
            if (ld_shared_volatile(w.abort_addr) != 0u) return false;
            if (globaltimer_ns() - t0 > w.timeout_ns) {
                st_shared_volatile(w.abort_addr, 1u);
                atomicCAS(w.status, 0u, site);
                return false;
            }
        }
    }
}

// Warp-wide wait: every lane polls the barrier, so the warp stays converged
// while it waits (a lane-0 poll with the other lanes parked in __syncwarp kept
// the warp diverged for the whole wait and cost 7-13% of throughput), and one
// vote gives all lanes the same outcome, so they never disagree about an abort.
__device__ __forceinline__ bool mbar_wait_warp(const WaitCtx& w, uint32_t bar, uint32_t parity, uint32_t site)
{
    const bool ok = mbar_wait(w, bar, parity, site);
    return __all_sync(0xffffffffu, ok);
}

// Teardown wait: ignores the abort word (it is used after an abort, to let the
// CTA's own copies and MMAs finish before shared and tensor memory go away).
__device__ __forceinline__ bool mbar_wait_drain(const WaitCtx& w, uint32_t bar, uint32_t parity, uint32_t site)
{
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 15u) == 15u && globaltimer_ns() - t0 > w.timeout_ns) {
            atomicCAS(w.status, 0u, site);
            return false;
        }
    }
}

// Shared-memory word with release / acquire semantics at CTA scope: a step
// counter one warp publishes after its data, another polls before reading it.
__device__ __forceinline__ void st_release_shared(uint32_t addr, uint32_t v, uint32_t on = 1u)
{
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t"
        "@q st.release.cta.shared::cta.u32 [%0], %1;\n\t}" ::"r"(addr), "r"(v), "r"(on)
        : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_shared(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// Warp-wide bounded wait until the counter at `addr` reaches `target`
// (counters only grow): every lane polls with acquire semantics (the warp
// stays converged), and one vote gives all lanes the same outcome.  Same
// give-up rules as mbar_wait.
__device__ __forceinline__ bool flag_wait_warp(const WaitCtx& w, uint32_t addr, uint32_t target, uint32_t site)
{
    bool ok = true;
    if (ld_acquire_shared(addr) < target) {
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t it = 1;; ++it) {
            if (ld_acquire_shared(addr) >= target) break;
            if ((it & 15u) == 0u) {
                if (ld_shared_volatile(w.abort_addr) != 0u) {
                    ok = false;
                    break;
                }
                if (globaltimer_ns() - t0 > w.timeout_ns) {
                    st_shared_volatile(w.abort_addr, 1u);
                    atomicCAS(w.status, 0u, site);
                    ok = false;
                    break;
                }
            }
        }
    }
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---- TMA ----------------------------------------------------------------------

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 3-D tiled load into shared memory; completes `bytes` on `bar`.
__device__ __forceinline__ void tma_load_3d(const CUtensorMap* m, uint32_t dst, uint32_t bar, int x, int y, int z,
                                            uint32_t on = 1u)
{
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %6, 0;\n\t"
        "@q cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
        "\n\t}" ::"r"(dst), "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(bar), "r"(on)
        : "memory");
}

// 3-D tiled store from shared memory (bulk-group completion).  Out-of-range rows
// of the box are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* m, uint32_t src, int x, int y, int z)
{
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];"
                 ::"l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(src)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Generic-proxy shared-memory writes -> visible to the async proxy (TMA store).
__device__ __forceinline__ void fence_proxy_async_shared()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- registers per warpgroup ------------------------------------------------------

template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc()
{
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec()
{
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ---- tcgen05: tensor memory -------------------------------------------------------

// Whole warp: allocate `ncols` TMEM columns, address written to shared `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// ---- tcgen05: MMA -------------------------------------------------------------------

// D[tmem] (+)= A[smem] * B[smem]
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate, uint32_t on = 1u)
{
    asm volatile(
        "{\n\t"
        ".reg .pred p, q;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.ne.b32 q, %5, 0;\n\t"
        "@q tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
        "}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(on)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate, uint32_t on = 1u)
{
    asm volatile(
        "{\n\t"
        ".reg .pred p, q;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.ne.b32 q, %5, 0;\n\t"
        "@q tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
        "}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(on)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar, uint32_t on = 1u)
{
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %1, 0;\n\t"
        "@q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar), "r"(on)
        : "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (tiles 1024-byte aligned).
//   bits  0-13 start address >> 4      bits 16-29 leading byte offset >> 4
//   bits 32-45 stride byte offset >> 4 bits 46-47 descriptor version (1)
//   bits 61-63 layout: 2 = 128-byte swizzle
// The low word (start address, leading byte offset) is what changes from one
// operand to the next; the high word is fixed by the layout.  Issuers that
// step through a tile keep only the low word and add start-address steps to
// it (a shared address below 256 KB never carries out of its 14 bits).
__device__ __forceinline__ uint32_t sdesc_lo(uint32_t saddr, uint32_t lbo)
{
    return ((saddr >> 4) & 0x3FFFu) | (((lbo >> 4) & 0x3FFFu) << 16);
}
__host__ __device__ constexpr uint32_t sdesc_hi_sw128(uint32_t sbo)
{
    return ((sbo >> 4) & 0x3FFFu) | (1u << (46 - 32)) | (2u << (61 - 32));
}
__device__ __forceinline__ uint64_t sdesc_join(uint32_t lo, uint32_t hi)
{
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(hi));
    return d;
}
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    return sdesc_join(sdesc_lo(saddr, lbo), sdesc_hi_sw128(sbo));
}

// Instruction descriptor of kind::f16 with fp32 accumulation.
//   bits 4-5 D format (1 = f32)   bits 7-9 / 10-12 A / B format (0 = f16, 1 = bf16)
//   bit 15 / 16 A / B major (0 = K-major, 1 = MN-major)
//   bits 17-22 N >> 3             bits 24-28 M >> 4
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool bf16, bool b_mn_major)
{
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// ---- tcgen05: TMEM <-> registers (32 data-path lanes x 32-bit) ---------------------
// A warp reaches TMEM lanes 32*(warp % 4) .. +31; lane L of the warp gets lane
// base+L, consecutive columns in consecutive registers.

#define FA_R8(i) "=r"(r[i + 0]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                 "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define FA_W8(i) "r"(r[i + 0]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), \
                 "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])

// Load 32 columns and wait for them (the wait sits in the same asm statement so
// no use of r[] can be scheduled before it).
__device__ __forceinline__ void tmem_ld32_wait(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : FA_R8(0), FA_R8(8), FA_R8(16), FA_R8(24)
        : "r"(taddr)
        : "memory");
}

// Load 32 columns without waiting (several loads may be in flight; follow
// with tmem_wait_ld and reg_fence before using the registers).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r)
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : FA_R8(0), FA_R8(8), FA_R8(16), FA_R8(24)
        : "r"(taddr)
        : "memory");
}

// Load 32 columns without waiting and, in the same instruction, reduce them to
// their maximum (per thread = per TMEM lane): the row maximum of a 32-column
// slice comes with the load.
__device__ __forceinline__ void tmem_ld32_max(uint32_t taddr, uint32_t* r, float& mx)
{
    asm volatile(
        "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, %32, [%33];"
        : FA_R8(0), FA_R8(8), FA_R8(16), FA_R8(24), "=f"(mx)
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Compiler-level fence: every use of r[] depends on a (volatile, hence ordered)
// statement placed after the wait, so no use can be hoisted above it.
template <int N>
__device__ __forceinline__ void reg_fence(uint32_t (&r)[N])
{
#pragma unroll
    for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}

template <int N>
__device__ __forceinline__ void reg_fence(float (&r)[N])
{
#pragma unroll
    for (int i = 0; i < N; ++i) asm volatile("" : "+f"(r[i]));
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
        ::"r"(taddr), FA_W8(0), FA_W8(8)
        : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
        ::"r"(taddr), FA_W8(0), FA_W8(8), FA_W8(16), FA_W8(24)
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

#undef FA_R8
#undef FA_W8

// ---- arithmetic -------------------------------------------------------------------

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float lg2(float x)
{
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---- packed fp32 pairs (one instruction, two lanes of work) -------------------

__device__ __forceinline__ uint64_t f2_pack(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t r;
    asm("fma.rn.ftz.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("add.rn.ftz.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("mul.rn.ftz.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// 2^x for a pair of floats on the FMA pipe instead of the XU (MUFU).
//   x = n + f, n = rint(x): adding M = 1.5 * 2^23 + 127 rounds x to an integer
//   and leaves n + 127 in the low bits of the sum t; t - M = n exactly; f in
//   [-1/2, 1/2].  2^f: degree-3 polynomial minimising the relative error on
//   [-1/2, 1/2] (Remez exchange; attention_fa_fwd_gb300/exp2_poly_fit.py
//   prints these coefficients; max relative error 7.5e-5).  2^n: the low nine
//   bits of t shifted to the exponent field, which is exactly 2^n for n in
//   [-127, 128] (n = -127 gives +0).  x is clamped at -127 first, so -inf and
//   very negative arguments give 0, as ex2.approx.ftz does.  Results below
//   2^-126 flush to zero (the final multiply is .ftz).
__device__ __forceinline__ uint64_t f2_exp2_poly(float x0, float x1)
{
    constexpr float kM = 12583039.0f;   // 1.5 * 2^23 + 127
    constexpr float kC0 = 0.9999280572f, kC1 = 0.6932609677f, kC2 = 0.2426111251f, kC3 = 0.05517166853f;
    const uint64_t x = f2_pack(fmaxf(x0, -127.f), fmaxf(x1, -127.f));
    const uint64_t t = f2_add(x, f2_pack(kM, kM));
    const uint64_t n = f2_add(t, f2_pack(-kM, -kM));
    const uint64_t f = f2_fma(n, f2_pack(-1.f, -1.f), x);
    uint64_t p = f2_fma(f, f2_pack(kC3, kC3), f2_pack(kC2, kC2));
    p = f2_fma(p, f, f2_pack(kC1, kC1));
    p = f2_fma(p, f, f2_pack(kC0, kC0));
    float t0, t1;
    f2_unpack(t, t0, t1);
    return f2_mul(p, f2_pack(__uint_as_float(__float_as_uint(t0) << 23), __uint_as_float(__float_as_uint(t1) << 23)));
}

// max of three fp32 values in one instruction
__device__ __forceinline__ float max3(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Two fp32 values -> one 32-bit word of two 16-bit values, round to nearest
// even; `lo` lands in the low half (the lower column / element index).
template <bool kBF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    uint32_t d;
    if constexpr (kBF16)
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// Two fp32 values -> two fp16 in one word, nearest even, saturating at +-65504
// (finite inputs never become infinite); `lo` in the low half.
__device__ __forceinline__ uint32_t pack2_f16_satfinite(float lo, float hi)
{
    uint32_t d;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// x rounded to the 16-bit type (nearest even), returned as fp32: the value an
// element packed by pack2 carries into the MMA.
template <bool kBF16>
__device__ __forceinline__ float round16(float x)
{
    const uint32_t d = pack2<kBF16>(x, x);
    if constexpr (kBF16) {
        return __uint_as_float(d << 16);   // a bf16 is the upper half of the fp32 with its value
    } else {
        float r;
        asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.f32.f16 %0, lo;\n\t}" : "=f"(r) : "r"(d));
        return r;
    }
}

}  // namespace ptx
}  // namespace fa
