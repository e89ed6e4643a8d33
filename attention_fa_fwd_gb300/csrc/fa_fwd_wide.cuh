// Fused attention forward for sm_103a, one-tile layout: a persistent,
// warp-specialised kernel whose work unit is one 128-row query tile, walked
// over the keys in wide steps of 192 keys.
//
// It computes what the two-tile kernel of fa_fwd_kernel.cuh computes - per
// (batch*head, query row i): O_i = sum_j softmax(s_i)_j v_j and
// LSE_i = ln sum_j exp(s_ij) with s_ij = scale * q_i . k_j over the allowed
// keys ("CUDA手写masked multi-head attention", section 3.1), tile by tile with
// the running statistics of online softmax and one division at the end
// ("FlashAttention的Triton性能考古学", 核心算法回顾 and 关键优化：反转循环顺序) -
// with a different schedule of the tensor core:
//
// * Scores S (fp32, one TMEM column per key) and P (16-bit, two keys per
//   column, two buffers) live in separate TMEM regions.  The next step's QK^T
//   is issued as soon as both softmax warpgroups have read S into registers
//   ("S free"), so the tensor core computes S(j+1) while the softmax turns
//   S(j) into P(j); P(j) goes to the buffer P*V(j-1) is not reading, so the
//   softmax of step j+1 can start the moment it has published P(j).
// * Both softmax warpgroups work on the same 128 rows, each on one half of a
//   step's keys (TMEM lane quadrants tie a warp to 32 rows).  They trade their
//   half-row maxima through shared memory once per step (a step counter with
//   release/acquire semantics per warp, polled by the partner warp: an
//   mbarrier round trip measured 560 cycles per step here), so both take the
//   same re-base decisions and P is relative to one base per row.
// * One MMA instruction carries more work (N = 192 keys for QK^T), so
//   the single issuing thread's waits and commits cost less per FLOP, and the
//   MMAs queued behind it cover more tensor time.
// * The steps of consecutive units form one stream: the next unit's first
//   QK^T is issued while the current unit's last P is being computed, and its
//   Q tile is loaded ahead (two Q buffers), so unit boundaries leave no gap.
//
// Rescale: the conditional re-base of "G6: Cluster 与 2CTA 探索", V41 (base b
// moves only when the row maximum passes b + T; T = 15 for fp16, 30 for bf16,
// as in the two-tile kernel), warp-wide as there; the softmax warps rescale O
// in TMEM themselves ("G6", V44), each warpgroup its half of O's columns,
// after the previous P*V has completed; the first P*V half of the step writes
// every column of O, so it waits for warpgroup 1 too (see kBarPA).  bf16 rows
// normalise O by l + dl, dl adding per step the rounding of each half's
// largest p to bf16 (as the two-tile kernel does).  This layout keeps P in
// bf16 for bf16 inputs (no conversion of V).
//
// CTA layout (512 threads, one CTA per SM):
//   warps 0-3   softmax, keys [0, BN/2) of each step
//   warps 4-7   softmax, keys [BN/2, BN) of each step
//   warps 8-11  epilogue: O / l, LSE, 16-bit O stored from registers
//   warp 12     TMA producer: Q tiles (two buffers), ring of K/V slots
//   warp 13     tcgen05 MMA issuer (one thread) and TMEM owner
//   warps 14-15 idle (they complete the fourth warpgroup for setmaxnreg)
//
// Tensor memory (512 columns): S [0, 192), P [192, 288) and [288, 384) for
// even and odd steps, O from 384 (one buffer of D columns at head dim 128;
// two of 64 at head dim 64, so an epilogue never holds up the next unit's
// first P*V).  The commit that announces S(j) also covers P*V(j-2), so P's
// buffer for step j is free whenever S(j) is.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "fa_fwd_common.h"
#include "fa_fwd_kernel.cuh"
#include "ptx.cuh"

namespace fa {

template <int D>
struct WideCfg {
    static_assert(D == 64 || D == 128, "head dim");
    static constexpr int kBN = kWideBN;                  // keys per step
    static constexpr int kNC = kBN / 2;                  // key columns per softmax warpgroup
    static constexpr int kQBytes = kBM * D * 2;          // one Q tile (16-bit)
    static constexpr int kQBoxBytes = kBM * 128;         // 128 rows x 64 columns
    static constexpr int kKVBoxBytes = kBN * 128;        // kBN rows x 64 columns
    static constexpr int kKVBytes = kBN * D * 2;         // one K or V tile of a step
    static constexpr int kBoxes = D / 64;
    static constexpr int kQBufs = 2;
    static constexpr int kOBufs = (D == 64) ? 2 : 1;
    // K/V ring: K of step s+1 and V of step s alternate through it.  Three
    // slots (D=128) give every copy the time of two MMA groups between the
    // release of the entry it overwrites and its first use; at D=64 the
    // groups are shorter and the tiles smaller, so the ring is deeper.
    static constexpr int kSlots = (D == 128) ? 3 : 6;
    static constexpr int kOffQ = 0;
    static constexpr int kOffKV = kOffQ + kQBufs * kQBytes;
    static constexpr int kOffX = kOffKV + kSlots * kKVBytes;        // [2 parity][2 half][128] half-row maxima
    static constexpr int kOffXFlag = kOffX + 2 * 2 * kBM * 4;       // [8] per softmax warp: steps published
    static constexpr int kOffSt = kOffXFlag + 8 * 4;                // [kOBufs][2 half][128] float4 row statistics
    static constexpr int kOffBars = kOffSt + kOBufs * 2 * kBM * 16;
    enum : int {
        kBarQFull = 0,      // [2] Q tile landed (TMA tx)
        kBarQEmpty = 2,     // [2] last QK of the Q tile finished (commit)
        kBarSFull = 4,      // scores of the step in TMEM (commit)
        kBarSFree = 5,      // both softmax warpgroups read S (8 warps)
        // [2] per P buffer: P of keys [0, BN/2) (PA) or [BN/2, BN) (PB) in
        // TMEM, O rescaled.  PB: warpgroup 1's 4 warps.  PA: warpgroup 0's 4
        // warps and warpgroup 1's 4: the first P*V half writes every column
        // of O, so it must also wait until warpgroup 1 has left O alone (its
        // half of O's columns rescaled, when the step rescales).  One barrier
        // per buffer, not one per role: the softmax may publish the next
        // step's P before the issuer has waited on this step's, and a single
        // barrier would then complete two phases and read as incomplete.
        kBarPA = 6,
        kBarPB = 8,
        kBarPVDone = 10,    // the step's P*V finished: O may be rescaled (commit)
        kBarOFull = 11,     // [2] the unit's last P*V finished (commit)
        kBarOEmpty = 13,    // [2] epilogue read O (4 warps)
        kBarStFull = 15,    // [2] row statistics of the unit in shared memory (8 warps)
        kBarStEmpty = 17,   // [2] epilogue took them (4 warps)
        kBarDrain = 19,     // MMA drain at exit (commit)
        kBarKVFull = 20,    // [kSlots] K or V tile landed (TMA tx)
    };
    static constexpr int kBarKVEmpty = kBarKVFull + kSlots;   // [kSlots] its last MMA finished (commit)
    static constexpr int kNumBars = kBarKVEmpty + kSlots;
    static constexpr int kOffCtl = kOffBars + kNumBars * 8;   // [0] TMEM base, [1] abort
    static constexpr int kSmemBytes = kOffCtl + 16 + 1024;    // + slack to align the base to 1 KB
    static constexpr uint32_t kColS = 0;
    static constexpr uint32_t kColP = kBN;       // two buffers of kBN / 2 columns
    static constexpr uint32_t kColO = 384;
    static_assert(kColP + kBN <= kColO && kColO + kOBufs * D <= 512, "TMEM budget");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// Register budget per warpgroup after setmaxnreg: softmax x2, epilogue, control.
// 2 * 184 + 64 + 80 = 512 = 65536 registers / 128 threads.
struct WideRegs {   // the spill-free split ptxas -v reports for all four instances
    static constexpr uint32_t kSoftmax = 184, kEpilogue = 64, kControl = 80;
};
static_assert(2 * WideRegs::kSoftmax + WideRegs::kEpilogue + WideRegs::kControl == 512, "register split");

__device__ __forceinline__ uint32_t smem_u32_of(const void* p) { return ptx::smem_u32(p); }

// Phase timing of the FA_TRACE build: a role's first thread sums the SM clock
// between consecutive marks into eight 32-bit registers and writes them (and
// the number of steps) to the trace buffer once, at the end, so no store
// lands in the middle of the timed work.  The production build has none of it.
#ifdef FA_TRACE
struct PhaseClock {
    uint32_t acc[8];
    uint32_t n;
    uint32_t t;
    __device__ __forceinline__ void start()
    {
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0u;
        n = 0u;
        t = (uint32_t)clock64();
    }
    __device__ __forceinline__ void mark(int k)
    {
        const uint32_t now = (uint32_t)clock64();
        acc[k] += now - t;
        t = now;
    }
    __device__ __forceinline__ void flush(const Params& p, int role) const
    {
        if ((int)blockIdx.x >= p.trace_ctas || p.trace_cap < 9) return;
        unsigned long long* dst = p.trace + ((size_t)blockIdx.x * kTraceRoles + role) * (size_t)p.trace_cap;
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[i] = acc[i];
        dst[8] = n;
    }
};
#define WT_DECL(cond) PhaseClock wt; const bool wt_on = (cond); if (wt_on) wt.start()
#define WT_MARK(k) do { if (wt_on) wt.mark(k); } while (0)
#define WT_STEP() do { if (wt_on) ++wt.n; } while (0)
#define WT_FLUSH(role) do { if (wt_on) wt.flush(p, role); } while (0)
#else
#define WT_DECL(cond) (void)0
#define WT_MARK(k) (void)0
#define WT_STEP() (void)0
#define WT_FLUSH(role) (void)0
#endif

// One work unit of the one-tile layout: a query tile and its number of steps.
struct WideUnit {
    int status;   // kUnitDone, kUnitOk or kUnitSkip
    int bh;
    int q_tile;
    int n;        // key steps of kBN keys: up to the diagonal (causal) or S
};

// The r-th unit of this CTA (the schedules of unit_at, one query tile per unit).
template <int BN>
__device__ __forceinline__ WideUnit wide_unit_at(int r, const Params& p)
{
    const Unit u = unit_at<false>(r, p);
    WideUnit w;
    w.status = u.status;
    w.bh = u.bh;
    w.q_tile = u.q_tile[0];
    const int kv_end = p.causal ? min(p.S, (w.q_tile + 1) * kBM) : p.S;
    w.n = (kv_end + BN - 1) / BN;
    return w;
}

// The first unit after r that is not skipped (or the end): every role walks
// the same list, the loader and the issuer look one unit ahead.
template <int BN>
__device__ __forceinline__ WideUnit wide_next_unit(int& r, const Params& p)
{
    WideUnit u;
    do {
        ++r;
        u = wide_unit_at<BN>(r, p);
    } while (u.status == kUnitSkip);
    return u;
}

// ---------------------------------------------------------------------------------
// Softmax warpgroup w (0: first half of a step's keys, 1: second half); one
// thread per query row.
template <int D, bool kBF16>
__device__ __forceinline__ void wide_softmax_role(const Params& p, const ptx::WaitCtx& wc, int w, uint32_t tmem,
                                                  uint32_t bars, float* xchg, float4* stats)
{
    using C = WideCfg<D>;
    constexpr int NC = C::kNC;
    const int lane = threadIdx.x & 31;
    const int wq = (threadIdx.x >> 5) & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_base + C::kColS + (uint32_t)(w * NC);
    const uint32_t tP = tmem + lane_base + C::kColP + (uint32_t)(w * (NC / 2));   // + (step & 1) * BN/2
    const float sl2 = p.scale_log2;
    const uint32_t bar_p = bars + 8 * (w ? C::kBarPB : C::kBarPA);   // + (step & 1)
    const uint32_t flag_own = smem_u32_of(xchg) + (uint32_t)(C::kOffXFlag - C::kOffX) + 4u * (uint32_t)(w * 4 + wq);
    const uint32_t flag_partner = smem_u32_of(xchg) + (uint32_t)(C::kOffXFlag - C::kOffX) + 4u * (uint32_t)((1 - w) * 4 + wq);
    uint32_t st = 0;    // steps of this CTA so far (one S, one P, one P*V each)
    uint32_t cnt = 0;   // units of this CTA so far
    WT_DECL((threadIdx.x & 127) == 0);

    for (int r = 0;; ++r) {
        const WideUnit un = wide_unit_at<C::kBN>(r, p);
        if (un.status == kUnitDone) break;
        if (un.status == kUnitSkip) continue;
        const int ob = C::kOBufs == 2 ? (int)(cnt & 1u) : 0;
        const uint32_t tO = tmem + lane_base + C::kColO + (uint32_t)(ob * D + w * (D / 2));
        const int qrow = un.q_tile * kBM + row;
        const int klim = p.causal ? min(qrow, p.S - 1) : p.S - 1;   // last key this row may see
        const int kmin = p.causal ? min(un.q_tile * kBM, p.S - 1) : p.S - 1;   // the same for the tile's first row
        float b = -INFINITY;   // base of the row, base-2 scaled units
        float l = 0.f;         // sum of 2^(x - b) over this half's keys: gives the LSE
        float dl = 0.f;        // bf16: rounding of each step's largest p of this half (see the two-tile kernel)
        for (int j = 0; j < un.n; ++j, ++st) {
            if (!ptx::mbar_wait_warp(wc, bars + 8 * C::kBarSFull, st & 1u, kSiteSoftmax | C::kBarSFull)) return;
            WT_MARK(4);
            ptx::tc_fence_after();
            uint32_t sr[NC];
            float pm[NC / 32];
#pragma unroll
            for (int c = 0; c < NC / 32; ++c) ptx::tmem_ld32_max(tS + 32 * c, sr + 32 * c, pm[c]);
            ptx::tmem_wait_ld();
            ptx::reg_fence(sr);
            ptx::reg_fence(pm);
            // S is in registers: the issuer may compute the next step's scores
            ptx::tc_fence_before();
            __syncwarp();
            ptx::mbar_arrive(bars + 8 * C::kBarSFree, lane == 0);
            WT_MARK(0);
            float* s = reinterpret_cast<float*>(sr);
            const int k0 = j * C::kBN + w * NC;   // first key of this half
            float mraw;
            if (k0 + NC - 1 > kmin) {
                // keys beyond the sequence and (causal) keys after the row
                const int lim = klim - k0;
#pragma unroll
                for (int c = 0; c < NC; ++c) s[c] = (c <= lim) ? s[c] : -INFINITY;
                // maximum over what is left: four chains of three-input max
                float m[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int c = 0; c < NC; c += 8) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) m[k] = ptx::max3(m[k], s[c + 2 * k], s[c + 2 * k + 1]);
                }
                mraw = fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
            } else {
                mraw = pm[0];
#pragma unroll
                for (int c = 1; c < NC / 32; ++c) mraw = fmaxf(mraw, pm[c]);
            }
            // trade half-row maxima with the partner warp (same rows, other half)
            float* xs = xchg + (st & 1u) * (2 * kBM);
            xs[w * kBM + row] = mraw;
            __syncwarp();
            ptx::st_release_shared(flag_own, st + 1u, lane == 0);
            WT_MARK(5);
            if (!ptx::flag_wait_warp(wc, flag_partner, st + 1u, kSiteSoftmax | 0xF0u)) return;
            WT_MARK(6);
            const float mx = fmaxf(mraw, xs[(1 - w) * kBM + row]) * sl2;
            WT_MARK(1);
            // conditional re-base (see the two-tile kernel): both warps of the
            // pair see the same maxima and bases, so they decide alike
            const float cand = fmaxf(b, mx);
            const bool rebase = cand > b + rebase_threshold<kBF16>();
            const bool rescale = j > 0 && __any_sync(0xffffffffu, rebase);
            float h = 1.f;
            if (rebase || rescale) {
                h = ptx::ex2(b - cand);   // 0 on the first step (b = -inf); 1 if cand == b
                b = cand;
            }
            // warpgroup 1 without a rescale this step leaves O alone: the first
            // P*V half (warpgroup 0's keys, every column of O) need not wait for it
            if (w == 1 && !rescale) ptx::mbar_arrive(bars + 8 * (C::kBarPA + (st & 1u)), lane == 0);
            // p = 2^(s * scale*log2e - b), packed to 16 bits two keys a word and
            // stored 32 keys at a time into this step's P buffer
            const float nb = (b == -INFINITY) ? 0.f : -b;
            const uint64_t c2 = ptx::f2_pack(sl2, sl2), nb2 = ptx::f2_pack(nb, nb);
            uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
            if constexpr (kBF16) {
                // this half's largest p, by the same FMA and ex2 the loop below uses
                const float pmx = ptx::ex2(fmaf(mraw, sl2, nb));
                dl = fmaf(dl, h, ptx::round16<kBF16>(pmx) - pmx);
            }
            const uint32_t tPb = tP + (st & 1u) * (uint32_t)(C::kBN / 2);
#pragma unroll
            for (int c = 0; c < NC / 32; ++c) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float x0, x1;
                    ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(s[32 * c + 2 * i], s[32 * c + 2 * i + 1]), c2, nb2), x0, x1);
                    const float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1);
                    acc[i & 3] = ptx::f2_add(acc[i & 3], ptx::f2_pack(p0, p1));
                    pk[i] = ptx::pack2<kBF16>(p0, p1);
                }
                ptx::tmem_st16(tPb + 16 * c, pk);
            }
            WT_MARK(2);
            if (rescale) {
                // O is stable once the previous step's P*V has completed; this
                // warp's 32 rows of this half of O scaled by 2^(b_old - b_new)
                if (!ptx::mbar_wait_warp(wc, bars + 8 * C::kBarPVDone, (st - 1) & 1u, kSiteSoftmax | C::kBarPVDone))
                    return;
                ptx::tc_fence_after();
#pragma unroll
                for (int c0 = 0; c0 < D / 2; c0 += 32) {
                    uint32_t o[32];
                    ptx::tmem_ld32_wait(tO + c0, o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * h);
                    ptx::tmem_st32(tO + c0, o);
                }
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            __syncwarp();
            ptx::mbar_arrive(bar_p + 8 * (st & 1u), lane == 0);
            // warpgroup 1's rescaled half of O, for the first P*V half
            if (w == 1 && rescale) ptx::mbar_arrive(bars + 8 * (C::kBarPA + (st & 1u)), lane == 0);
            WT_MARK(3);
            WT_STEP();
            float sa, sb;
            ptx::f2_unpack(ptx::f2_add(ptx::f2_add(acc[0], acc[1]), ptx::f2_add(acc[2], acc[3])), sa, sb);
            l = fmaf(l, h, sa + sb);
        }
        // hand this half's (l, l + dl) and the base to the epilogue
        const uint32_t ph_st = ((cnt / C::kOBufs) & 1u) ^ 1u;
        if (!ptx::mbar_wait_warp(wc, bars + 8 * (C::kBarStEmpty + ob), ph_st, kSiteSoftmax | (C::kBarStEmpty + ob)))
            return;
        stats[(ob * 2 + w) * kBM + row] = make_float4(l, l + dl, b, 0.f);
        __syncwarp();
        ptx::mbar_arrive(bars + 8 * (C::kBarStFull + ob), lane == 0);
        ++cnt;
    }
    WT_FLUSH(w);
}

// ---------------------------------------------------------------------------------
// Epilogue warpgroup: per unit, O / l, LSE, 16-bit O stored from registers
// (each thread writes its row: whole 32-byte sectors).
template <int D, bool kBF16>
__device__ __forceinline__ void wide_epilogue_role(const Params& p, const ptx::WaitCtx& wc, uint32_t tmem,
                                                   uint32_t bars, const float4* stats)
{
    using C = WideCfg<D>;
    const int lane = threadIdx.x & 31;
    const int wq = (threadIdx.x >> 5) & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    uint32_t cnt = 0;
    for (int r = 0;; ++r) {
        const WideUnit un = wide_unit_at<C::kBN>(r, p);
        if (un.status == kUnitDone) break;
        if (un.status == kUnitSkip) continue;
        const int ob = C::kOBufs == 2 ? (int)(cnt & 1u) : 0;
        const uint32_t par = (cnt / C::kOBufs) & 1u;
        if (!ptx::mbar_wait_warp(wc, bars + 8 * (C::kBarOFull + ob), par, kSiteEpilogue | (C::kBarOFull + ob)) ||
            !ptx::mbar_wait_warp(wc, bars + 8 * (C::kBarStFull + ob), par, kSiteEpilogue | (C::kBarStFull + ob)))
            return;
        ptx::tc_fence_after();
        const float4 s0 = stats[(ob * 2 + 0) * kBM + row];
        const float4 s1 = stats[(ob * 2 + 1) * kBM + row];
        __syncwarp();
        ptx::mbar_arrive(bars + 8 * (C::kBarStEmpty + ob), lane == 0);
        const float inv = 1.0f / (s0.y + s1.y);
        const int qrow = un.q_tile * kBM + row;
        const bool in = qrow < p.S;
        if (in) p.lse[(size_t)un.bh * (size_t)p.S + (size_t)qrow] = (s0.z + ptx::lg2(s0.x + s1.x)) * kLn2;
        const uint64_t il2 = ptx::f2_pack(inv, inv);
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + ((size_t)un.bh * p.S + qrow) * D);
        const uint32_t tO = tmem + lane_base + C::kColO + (uint32_t)(ob * D);
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[32];
            ptx::tmem_ld32_wait(tO + c0, o);
            if (c0 + 32 == D) {
                // every column read: the issuer may start the next unit's P*V here
                ptx::tc_fence_before();
                __syncwarp();
                ptx::mbar_arrive(bars + 8 * (C::kBarOEmpty + ob), lane == 0);
            }
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float x0, x1;
                ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])), il2),
                               x0, x1);
                pk[i] = ptx::pack2<kBF16>(x0, x1);
            }
            if (in) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    dst[c0 / 8 + i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
            }
        }
        ++cnt;
    }
}

// ---------------------------------------------------------------------------------
// TMA producer (one thread).  Ring entries in the order the issuer uses them:
// K of the CTA's first step, then per step s the K of step s+1 (if any, the
// next unit's first step included) and the V of step s.
template <int D>
__device__ __forceinline__ void wide_load_role(const Params& p, const ptx::WaitCtx& wc, const CUtensorMap* tm_q,
                                               const CUtensorMap* tm_k, const CUtensorMap* tm_v, uint32_t smem_base,
                                               uint32_t bars)
{
    const uint32_t ex = (threadIdx.x & 31) == 0 ? 1u : 0u;   // the lane that issues (the whole warp runs the role)
    using C = WideCfg<D>;
    uint32_t e = 0;        // ring entries issued
    uint32_t nq = 0;       // Q tiles issued
    bool ok = true;
    auto load_q = [&](const WideUnit& u) {
        const uint32_t qb = nq & 1u;
        if (!ptx::mbar_wait(wc, bars + 8 * (C::kBarQEmpty + qb), ((nq >> 1) & 1u) ^ 1u, kSiteLoad | (C::kBarQEmpty + qb))) {
            ok = false;
            return;
        }
        const uint32_t fb = bars + 8 * (C::kBarQFull + qb);
        ptx::mbar_arrive_expect_tx(fb, C::kQBytes, ex);
        const uint32_t dst = smem_base + C::kOffQ + qb * C::kQBytes;
#pragma unroll
        for (int bx = 0; bx < C::kBoxes; ++bx)
            ptx::tma_load_3d(tm_q, dst + bx * C::kQBoxBytes, fb, bx * 64, u.q_tile * kBM, u.bh, ex);
        ++nq;
    };
    auto load_kv = [&](const CUtensorMap* m, const WideUnit& u, int j) {
        const uint32_t slot = e % C::kSlots;
        if (!ptx::mbar_wait(wc, bars + 8 * (C::kBarKVEmpty + slot), ((e / C::kSlots) & 1u) ^ 1u,
                            kSiteLoad | (C::kBarKVEmpty + slot))) {
            ok = false;
            return;
        }
        const uint32_t fb = bars + 8 * (C::kBarKVFull + slot);
        ptx::mbar_arrive_expect_tx(fb, C::kKVBytes, ex);
        const uint32_t dst = smem_base + C::kOffKV + slot * C::kKVBytes;
#pragma unroll
        for (int bx = 0; bx < C::kBoxes; ++bx)
            ptx::tma_load_3d(m, dst + bx * C::kKVBoxBytes, fb, bx * 64, j * C::kBN, u.bh, ex);
        ++e;
    };

    int r = -1;
    WideUnit un = wide_next_unit<C::kBN>(r, p);
    if (un.status == kUnitOk) {
        load_q(un);
        if (ok) load_kv(tm_k, un, 0);
    }
    while (ok && un.status == kUnitOk) {
        int rn = r;
        WideUnit nx = un;
        for (int j = 0; j < un.n && ok; ++j) {
            if (j + 1 < un.n) {
                load_kv(tm_k, un, j + 1);
            } else {
                nx = wide_next_unit<C::kBN>(rn, p);
                if (nx.status == kUnitOk) {
                    load_q(nx);
                    if (ok) load_kv(tm_k, nx, 0);
                }
            }
            if (ok) load_kv(tm_v, un, j);
        }
        if (!ok) break;
        r = rn;
        un = nx;
    }
    // Every issued copy must land before the CTA exits (after an abort, too).
    for (uint32_t b = 0; b < 2u && b < nq; ++b) {
        const uint32_t last = nq - 1 - ((nq - 1 - b) % 2u);   // last Q tile issued into buffer b
        ptx::mbar_wait_drain(wc, bars + 8 * (C::kBarQFull + b), (last >> 1) & 1u, kSiteDrain | (C::kBarQFull + b));
    }
    for (uint32_t s = 0; s < (uint32_t)C::kSlots && s < e; ++s) {
        const uint32_t last = e - 1 - ((e - 1 - s) % C::kSlots);   // last entry in slot s
        ptx::mbar_wait_drain(wc, bars + 8 * (C::kBarKVFull + s), (last / C::kSlots) & 1u,
                             kSiteDrain | (C::kBarKVFull + s));
    }
}

// ---------------------------------------------------------------------------------
// tcgen05 MMA issuer (one thread).  Per step s: QK^T of step s+1 once the
// softmax has read S(s), then P*V of step s in two halves as each softmax
// warpgroup publishes its half of P.
template <int D, bool kBF16>
__device__ __forceinline__ void wide_mma_role(const Params& p, const ptx::WaitCtx& wc, uint32_t tmem,
                                              uint32_t smem_base, uint32_t bars)
{
    const uint32_t ex = (threadIdx.x & 31) == 0 ? 1u : 0u;   // the lane that issues (the whole warp runs the role)
    using C = WideCfg<D>;
    constexpr uint32_t kIdescQK = ptx::idesc_f16(kBM, C::kBN, kBF16, false);   // Q, K both K-major
    constexpr uint32_t kIdescPV = ptx::idesc_f16(kBM, D, kBF16, true);         // V is MN-major (D contiguous)
    constexpr uint32_t kDescHi = ptx::sdesc_hi_sw128(1024);
    constexpr int kHalfK = C::kBN / 32;   // K=16 MMAs per half of P

    // S = Q K^T: M = 128 rows, N = kBN keys, K = D in steps of 16
    auto issue_qk = [&](uint32_t qb, uint32_t slot) {
        const uint32_t qa = ptx::sdesc_lo(smem_base + C::kOffQ + qb * C::kQBytes, 16);
        const uint32_t kb = ptx::sdesc_lo(smem_base + C::kOffKV + slot * C::kKVBytes, 16);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t oa = ((kk >> 2) * C::kQBoxBytes + (kk & 3) * 32) >> 4;
            const uint32_t ob = ((kk >> 2) * C::kKVBoxBytes + (kk & 3) * 32) >> 4;
            ptx::mma_ss(tmem + C::kColS, ptx::sdesc_join(qa + oa, kDescHi), ptx::sdesc_join(kb + ob, kDescHi),
                        kIdescQK, kk > 0 ? 1u : 0u, ex);
        }
    };
    // O += P V for one half of the keys: A = P from TMEM (16 keys = 8 columns
    // per MMA), B = V [kBN keys x D], 64-column boxes kKVBoxBytes apart.
    auto issue_pv = [&](uint32_t slot, uint32_t ob, uint32_t pb, int half, bool acc) {
        const uint32_t vl = ptx::sdesc_lo(smem_base + C::kOffKV + slot * C::kKVBytes, C::kKVBoxBytes);
#pragma unroll
        for (int k4 = 0; k4 < kHalfK; ++k4) {
            const int kk = half * kHalfK + k4;
            ptx::mma_ts(tmem + C::kColO + ob * D, tmem + C::kColP + pb * (C::kBN / 2) + kk * 8,
                        ptx::sdesc_join(vl + ((kk * 16 * 128) >> 4), kDescHi), kIdescPV, (acc || kk > 0) ? 1u : 0u, ex);
        }
    };
    auto kv_wait = [&](uint32_t e) {
        const uint32_t slot = e % C::kSlots;
        return ptx::mbar_wait(wc, bars + 8 * (C::kBarKVFull + slot), (e / C::kSlots) & 1u,
                              kSiteMma | (C::kBarKVFull + slot));
    };

    uint32_t e = 0;     // ring entries consumed (same order as the loader's)
    uint32_t st = 0;    // steps
    uint32_t cnt = 0;   // units
    WT_DECL(ex != 0u);
    int r = -1;
    WideUnit un = wide_next_unit<C::kBN>(r, p);
    if (un.status == kUnitOk) {
        // the CTA's first QK
        if (!ptx::mbar_wait(wc, bars + 8 * C::kBarQFull, 0u, kSiteMma | C::kBarQFull) || !kv_wait(0)) goto done;
        ptx::tc_fence_after();
        issue_qk(0, 0);
        ptx::mma_commit(bars + 8 * C::kBarSFull, ex);
        ptx::mma_commit(bars + 8 * C::kBarKVEmpty, ex);
        if (un.n == 1) ptx::mma_commit(bars + 8 * C::kBarQEmpty, ex);
        e = 1;
    }
    while (un.status == kUnitOk) {
        int rn = r;
        WideUnit nx = un;
        const uint32_t ob = C::kOBufs == 2 ? (cnt & 1u) : 0u;
        for (int j = 0; j < un.n; ++j, ++st) {
            // QK^T of the next step (this unit's, or the next unit's first)
            bool have_next = j + 1 < un.n;
            uint32_t nqb = cnt & 1u;
            int nj = j + 1, nn = un.n;
            if (!have_next) {
                nx = wide_next_unit<C::kBN>(rn, p);
                have_next = nx.status == kUnitOk;
                nqb = (cnt + 1) & 1u;
                nj = 0;
                nn = nx.n;
            }
            WT_MARK(0);
            if (have_next) {
                if (!ptx::mbar_wait(wc, bars + 8 * C::kBarSFree, st & 1u, kSiteMma | C::kBarSFree)) goto done;
                WT_MARK(1);
                if (nj == 0 && !ptx::mbar_wait(wc, bars + 8 * (C::kBarQFull + nqb), ((cnt + 1) >> 1) & 1u,
                                               kSiteMma | (C::kBarQFull + nqb)))
                    goto done;
                const uint32_t ek = e++;
                if (!kv_wait(ek)) goto done;
                WT_MARK(2);
                ptx::tc_fence_after();
                issue_qk(nqb, ek % C::kSlots);
                ptx::mma_commit(bars + 8 * C::kBarSFull, ex);
                ptx::mma_commit(bars + 8 * (C::kBarKVEmpty + ek % C::kSlots), ex);
                if (nj == nn - 1) ptx::mma_commit(bars + 8 * (C::kBarQEmpty + nqb), ex);
                WT_MARK(3);
            }
            // P*V of this step
            const uint32_t ev = e++;
            if (j == 0 && !ptx::mbar_wait(wc, bars + 8 * (C::kBarOEmpty + ob), ((cnt / C::kOBufs) & 1u) ^ 1u,
                                          kSiteMma | (C::kBarOEmpty + ob)))
                goto done;
            if (!kv_wait(ev)) goto done;
            WT_MARK(4);
            const uint32_t pb = st & 1u, ph_p = (st >> 1) & 1u;   // P buffer and its phase
            if (!ptx::mbar_wait(wc, bars + 8 * (C::kBarPA + pb), ph_p, kSiteMma | (C::kBarPA + pb))) goto done;
            WT_MARK(5);
            ptx::tc_fence_after();
            issue_pv(ev % C::kSlots, ob, pb, 0, j > 0);
            if (!ptx::mbar_wait(wc, bars + 8 * (C::kBarPB + pb), ph_p, kSiteMma | (C::kBarPB + pb))) goto done;
            WT_MARK(6);
            ptx::tc_fence_after();
            issue_pv(ev % C::kSlots, ob, pb, 1, true);
            ptx::mma_commit(bars + 8 * C::kBarPVDone, ex);
            ptx::mma_commit(bars + 8 * (C::kBarKVEmpty + ev % C::kSlots), ex);
            if (j == un.n - 1) ptx::mma_commit(bars + 8 * (C::kBarOFull + ob), ex);
            WT_MARK(7);
            WT_STEP();
        }
        ++cnt;
        r = rn;
        un = nx;
    }
done:
    // every MMA must be complete before tensor memory is released
    ptx::mma_commit(bars + 8 * C::kBarDrain, ex);
    ptx::mbar_wait_drain(wc, bars + 8 * C::kBarDrain, 0u, kSiteDrain | C::kBarDrain);
    WT_FLUSH(kTrMma);
}

// ---------------------------------------------------------------------------------
template <int D, bool kBF16>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_wide_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ Params p)
{
    using C = WideCfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw);
    const uint32_t bars = base + C::kOffBars;
    float* xchg = reinterpret_cast<float*>(smem + C::kOffX);
    float4* stats = reinterpret_cast<float4*>(smem + C::kOffSt);
    volatile uint32_t* ctl = reinterpret_cast<volatile uint32_t*>(smem + C::kOffCtl);
    const int warp = ptx::warp_id_uniform();
    const int lane = threadIdx.x & 31;
    // the next kernel in the stream may be scheduled now (see the two-tile kernel)
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            ptx::mbar_init(bars + 8 * (C::kBarQFull + t), 1);
            ptx::mbar_init(bars + 8 * (C::kBarQEmpty + t), 1);
            ptx::mbar_init(bars + 8 * (C::kBarOFull + t), 1);
            ptx::mbar_init(bars + 8 * (C::kBarOEmpty + t), 4);
            ptx::mbar_init(bars + 8 * (C::kBarStFull + t), 8);
            ptx::mbar_init(bars + 8 * (C::kBarStEmpty + t), 4);
        }
        ptx::mbar_init(bars + 8 * C::kBarSFull, 1);
        ptx::mbar_init(bars + 8 * C::kBarSFree, 8);
        for (int t = 0; t < 2; ++t) {
            ptx::mbar_init(bars + 8 * (C::kBarPA + t), 8);
            ptx::mbar_init(bars + 8 * (C::kBarPB + t), 4);
        }
        ptx::mbar_init(bars + 8 * C::kBarPVDone, 1);
        for (int q = 0; q < 8; ++q) ptx::st_shared_volatile(base + C::kOffXFlag + 4 * q, 0u);
        ptx::mbar_init(bars + 8 * C::kBarDrain, 1);
        for (int s = 0; s < C::kSlots; ++s) {
            ptx::mbar_init(bars + 8 * (C::kBarKVFull + s), 1);
            ptx::mbar_init(bars + 8 * (C::kBarKVEmpty + s), 1);
        }
        ctl[1] = 0u;
        ptx::fence_mbar_init();
    }
    if (warp == 12 && lane == 0) {
        ptx::prefetch_tmap(&tm_q);
        ptx::prefetch_tmap(&tm_k);
        ptx::prefetch_tmap(&tm_v);
    }
    if (warp == 13) {
        ptx::tmem_alloc(base + C::kOffCtl, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = ctl[0];
    const ptx::WaitCtx wc{base + C::kOffCtl + 4, p.timeout_ns, p.status};
    // global memory only after the previous grid in the stream has completed
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp < 8) {
        ptx::setmaxnreg_inc<WideRegs::kSoftmax>();
        wide_softmax_role<D, kBF16>(p, wc, warp >> 2, tmem, bars, xchg, stats);
    } else if (warp < 12) {
        ptx::setmaxnreg_dec<WideRegs::kEpilogue>();
        wide_epilogue_role<D, kBF16>(p, wc, tmem, bars, stats);
    } else {
        ptx::setmaxnreg_dec<WideRegs::kControl>();
        // the loader and the MMA issuer run on all 32 lanes of their warp (one
        // lane issues), so neither warp diverges while it waits
        if (warp == 12) {
            wide_load_role<D>(p, wc, &tm_q, &tm_k, &tm_v, base, bars);
        } else if (warp == 13) {
            wide_mma_role<D, kBF16>(p, wc, tmem, base, bars);
        }
        __syncwarp();
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 13) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

template <int D, bool kBF16>
int launch_wide_instance(const LaunchArgs& a, cudaStream_t stream)
{
    auto kern = fa_fwd_wide_kernel<D, kBF16>;
    cudaError_t e = cudaSuccess;
    if (!smem_opt_in_done(reinterpret_cast<const void*>(kern), a.device)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, WideCfg<D>::kSmemBytes);
        if (e != cudaSuccess) return (int)e;
        smem_opt_in_mark(reinterpret_cast<const void*>(kern), a.device);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = WideCfg<D>::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, a.tm_q, a.tm_k, a.tm_v, a.p);
    return (int)e;
}

}  // namespace fa
