// Fused attention forward for sm_103a: a persistent, warp-specialised kernel
// built on TMA, mbarriers and tcgen05 (tensor memory + single-thread MMA).
//
// What is computed, per (batch*head, query row i):
//   s_ij = scale * q_i . k_j for allowed keys j (all j; or j <= i when causal)
//   O_i  = sum_j softmax(s_i)_j v_j,   LSE_i = ln sum_j exp(s_ij)
// ("CUDA手写masked multi-head attention", section 3.1), tile by tile with the
// running statistics of online softmax and one division at the end
// ("FlashAttention的Triton性能考古学", 核心算法回顾 and 关键优化：反转循环顺序:
// the query tile is loaded once and the key loop is inner).
//
// CTA layout (512 threads, one CTA per SM, persistent over work units):
//   warps 0-3   softmax warpgroup of query tile 0 (one thread per row)
//   warps 4-7   softmax warpgroup of query tile 1
//   warps 8-11  correction/epilogue warpgroup: the final correction O / l,
//               LSE, bf16/fp16 convert, shared-memory staging and TMA store;
//               for one-pass bf16 launches the softmax warpgroups run the
//               epilogue (epi_in_softmax) and these warps convert V tiles
//   warp 12     TMA producer: Q tiles, then a ring of K/V slots
//   warp 13     tcgen05 MMA issuer (one thread) and TMEM owner
//   warps 14-15 bf16 inputs: convert V tiles to fp16 in shared memory (P is
//               fp16, see p_is_bf16); fp16 inputs: idle (they complete the
//               fourth warpgroup for setmaxnreg)
//
// A work unit is one (batch*head, group of 1 or 2 query tiles of 128 rows).  TMEM
// (512 columns x 128 lanes, fp32) holds S0 | S1 | O0 | O1: the scores of each
// query tile, and its output accumulator.  P (16-bit) overwrites the first half
// of its S region and feeds the P*V MMA straight from TMEM ("G6", V37: P stays
// in TMEM, the "ts" form of tcgen05.mma).
//
// MMA issue order per key tile j ("G6", V39, interleave):
//   PV0(j), QK0(j+1), PV1(j), QK1(j+1)
// so the tensor core computes one tile's scores while the other tile's softmax
// runs (the FA_SCORE_ROTATION build option issues QK(j+1) earlier still at
// D=64, into a third score buffer; see Cfg::kRot).  The softmax publishes P
// once it is complete and the issuer sends the tile's P*V after that one wait
// (the FA_PV_SPLIT build option publishes it in two halves instead, "G6",
// V43).
//
// Softmax uses the conditional rescale of "G6", V41, in the base-2 domain: the
// row base b only moves when the tile maximum exceeds b + T, so p = 2^(x - b)
// lies in (0, 2^T].  The page uses T = 8 with fp16 P summed in half2; here P is
// summed in fp32, so T is set by P's type alone: 15 for fp16 (2^15 < 65504)
// and 30 for bf16 (fp32's exponent range), which makes rescales much rarer on
// inputs whose row maxima keep rising.  The row maximum of an unmasked tile comes with the TMEM
// load (tcgen05.ld.red .max; "G6", V41: "4 ld.red").  When a row's base moves,
// the softmax warp owning it rescales its 32 rows of O in TMEM before it
// publishes P ("G6", V44: the rescale moved into the softmax warpgroups; here
// too a separate correction handshake measured ~16% slower).  Because
// tcgen05.commit covers every earlier MMA of the issuing thread, the commit
// that announces S_t(j) also guarantees PV_t(j-1) has finished, so O_t is
// stable when the softmax rescales it.
//
// Causal masking: with 128 x 128 tiles a query tile's diagonal is exactly its
// last key tile; later key tiles are skipped, only the diagonal tile (and a
// ragged last key tile) pays for the mask.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "fa_fwd_common.h"
#include "ptx.cuh"

namespace fa {

// Re-base threshold T in log2 units ("G6", V41 uses base + 8): p <= 2^T must be
// finite in P's 16-bit type; the row sums and O accumulate in fp32.
template <bool kBF16>
__host__ __device__ constexpr float rebase_threshold() { return kBF16 ? 30.0f : 15.0f; }

// Where a re-base puts the base: the tile maximum plus this much (log2 units).
// Any base gives the same result in real arithmetic; above the maximum, p
// starts at 2^-overshoot <= 1 and the next re-base waits until the row maximum
// rises by T + overshoot instead of T, which matters for fp16 P (T = 15) on
// inputs whose maxima keep rising; p of 2^-20 of the row's largest stays
// inside fp16's range (its subnormals reach 2^-24).
template <bool kBF16>
__host__ __device__ constexpr float rebase_overshoot() { return kBF16 ? 0.0f : 8.0f; }

// P's 16-bit type.  P*V takes P and V of one type (tcgen05.mma kind::f16), and
// bf16's 8-bit significand rounds P to 2^-9: on inputs whose rows are nearly
// one-hot over large values of V that moves some elements of O past the
// rounding midpoint of the bf16 output.  So for bf16 inputs two otherwise idle
// warps convert each V tile to fp16 in shared memory once it lands
// (vconvert_role), and P is fp16 for both input types; Q K^T stays bf16.
// FA_BF16_P=1 builds keep bf16 P and V (the build option exists to measure
// the conversion's cost).
#ifndef FA_BF16_P
#define FA_BF16_P 0
#endif
template <bool kBF16>
__host__ __device__ constexpr bool p_is_bf16() { return kBF16 && FA_BF16_P != 0; }
template <bool kBF16>
__host__ __device__ constexpr bool converts_v() { return kBF16 && FA_BF16_P == 0; }

// Pairs out of every 16 whose exponentials use ptx::f2_exp2_poly (the FMA
// pipe) instead of ex2.approx (the XU): the split of the exponential work the
// "Triton" page's MIO-bottleneck section motivates.  Off by default: on GB300
// the XU retires ex2 fast enough that the extra FMA-pipe instructions cost
// more than they save (the build option exists to measure that).
#ifndef FA_EXP2_POLY_PAIRS
#define FA_EXP2_POLY_PAIRS 0
#endif
constexpr int kExp2PolyPairs = FA_EXP2_POLY_PAIRS;

// "G6", V44 layout: each softmax warpgroup also runs the epilogue of its own
// query tile (wait for the last PV, O / l, LSE, 16-bit O stored from
// registers), and the correction/epilogue warpgroup idles.  Off by default:
// the separate epilogue is off the critical path here (the MMA issuer waits
// on it at unit starts only), while in the softmax warpgroups it delays the
// tile's next unit (the build option exists to measure that).  Split-KV
// instances keep the separate epilogue.
#ifndef FA_EPILOGUE_IN_SOFTMAX
#define FA_EPILOGUE_IN_SOFTMAX 0
#endif
constexpr bool kEpilogueInSoftmax = FA_EPILOGUE_IN_SOFTMAX != 0;

// Where the epilogue runs: in the softmax warpgroups with the V44 build option
// (split-KV instances keep the separate epilogue: it writes the fp32
// partials).  The conversion of V tiles (bf16 inputs) takes warps 14-15; the
// epilogue warpgroup in the softmax warpgroups and all six warps converting
// measured slower (train 1105 vs 1125, stress 1140 vs 1235 TFLOPS): the
// conversion's cost is issue slots, not latency.
template <bool kBF16, bool kSplit, bool kKP>
__host__ __device__ constexpr bool epi_in_softmax() { return kEpilogueInSoftmax && !kSplit && !kKP; }
template <bool kBF16, bool kSplit, bool kKP>
__host__ __device__ constexpr int conv_warps() { return converts_v<kBF16>() ? (epi_in_softmax<kBF16, kSplit, kKP>() ? 6 : 2) : 0; }
// P published in two halves (keys 0-63, then 64-127), the first P*V half
// issued after the first ("G6", V43's PV split, so that half of P*V overlaps
// the second half of the exponentials).  Off by default: the MMA issuer's
// extra wait and fence per slot and step cost more than the overlap gains
// (train 1328-1337 against 1373-1376 TFLOPS, wide 853 against 873-875,
// 1x1x16384x64 401 against 415; the build option exists to measure that).
#ifndef FA_PV_SPLIT
#define FA_PV_SPLIT 0
#endif
constexpr bool kPVSplit = FA_PV_SPLIT != 0;

// Three rotating score buffers at D=64 (Cfg::kRot): each slot's next scores
// are computed while its softmax still works on the current ones.  Off by
// default: the hand-off chain they remove is not what bounds the D=64
// launches (measured slower, the build option exists to measure that).
#ifndef FA_SCORE_ROTATION
#define FA_SCORE_ROTATION 0
#endif
constexpr bool kScoreRotation = FA_SCORE_ROTATION != 0;
static_assert(kExp2PolyPairs >= 0 && kExp2PolyPairs <= 16, "FA_EXP2_POLY_PAIRS must be in [0, 16]");
constexpr float kLn2 = 0.693147180559945309f;

// Register budget per warpgroup after setmaxnreg: softmax x2, epilogue, control
// (load + MMA).  The four add up to 512 = 65536 registers / 128 threads; the
// splits are the spill-free ones ptxas -v reports for each head dim and type
//
template <int D, bool kBF16, bool kSplit, bool kKP> struct RegSplit {   // D=128 one pass, D=64 split-KV
    static constexpr uint32_t kSoftmax = 184, kEpilogue = 56, kControl = 88;
};
template <bool kBF16, bool kKP> struct RegSplit<64, kBF16, false, kKP> {
    static constexpr uint32_t kSoftmax = 184, kEpilogue = 72, kControl = 72;
};
// key-parity units (kKP): the epilogue merges two accumulators
template <bool kBF16> struct RegSplit<64, kBF16, false, true> {
    static constexpr uint32_t kSoftmax = 176, kEpilogue = 88, kControl = 72;
};
template <bool kBF16> struct RegSplit<64, kBF16, true, true> {
    static constexpr uint32_t kSoftmax = 176, kEpilogue = 88, kControl = 72;
};
template <int D, bool kBF16, bool kSplit, bool kKP>
constexpr bool reg_split_fits()
{
    using R = RegSplit<D, kBF16, kSplit, kKP>;
    return 2 * R::kSoftmax + R::kEpilogue + R::kControl == 512;
}
static_assert(reg_split_fits<128, false, false, false>() && reg_split_fits<128, false, true, false>() &&
                  reg_split_fits<64, false, false, false>() && reg_split_fits<64, false, false, true>() &&
                  reg_split_fits<64, false, true, false>() && reg_split_fits<64, false, true, true>(),
              "register split must add up to 512");

// Barrier indices inside the barrier array.  The score and P barriers come in
// kStepBars per tile slot, taken in turn by the slot's key steps with
// FA_SCORE_ROTATION (Cfg::kRot), else only the slot's first one.  The spacing
// matters without the rotation too: with the two slots' score, P-half and
// P-full barriers adjacent (one 16-byte chunk per pair) the D=128 launches ran
// 1.5% (4x32x4096) and 3% (1x32x16384) slower than with these 24-byte gaps;
// wider gaps (16, 32 or 128 bytes per barrier) measured no better.
constexpr int kStepBars = 3;
// Bytes from one barrier to the next in shared memory.
constexpr uint32_t kBarStride = 8;
enum : int {
    kBarQFull = 0,      // [2] Q tile t landed (TMA tx)
    kBarQEmpty = 2,     // [2] last QK of tile t finished (commit)
    kBarSFull = 4,      // [2][kStepBars] scores of slot t's step ready (commit)
    kBarPHalf = 10,     // [2][kStepBars] P keys 0-63 in TMEM, O_t rescaled (4 softmax warps; FA_PV_SPLIT)
    kBarPFull = 16,     // [2][kStepBars] P in TMEM, O_t rescaled (4 softmax warps)
    kBarOFull = 22,     // [2] last PV of tile t finished (commit)
    kBarOEmpty = 24,    // [2] epilogue done reading O_t (4 epilogue warps)
    kBarStFull = 26,    // [2] row statistics of tile t in shared memory (4 softmax warps)
    kBarStEmpty = 28,   // [2] epilogue took the statistics (4 epilogue warps)
    kBarPVDone = 30,    // [2][2] a P*V of slot t that is not the unit's last finished (commit)
    kBarDrain = 34,     // MMA drain at exit (commit)
    kBarKVFull = 35,    // [slots] K or V tile landed (TMA tx)
};

template <int D, bool kKP = false>
struct Cfg {
    static_assert(D == 64 || D == 128, "head dim");
    static_assert(!kKP || D == 64, "key-parity units: head dim 64");
    static constexpr int kTileBytes = kBM * D * 2;          // one Q, K or V tile (16-bit)
    static constexpr int kBoxBytes = kBM * 64 * 2;          // one 128-row x 64-column swizzle box
    static constexpr int kBoxes = D / 64;
    // Key-parity units (kKP, one query tile per unit at D=64): a ring entry
    // holds two key tiles, 2j and 2j+1 of step j (the even one for tile slot 0,
    // the odd one for slot 1), so the ring keeps its 128 KB in 4 double slots.
    static constexpr int kSlotBytes = kKP ? 2 * kTileBytes : kTileBytes;
    static constexpr int kSlots = kKP ? 4 : ((D == 128) ? 4 : 8);   // K/V ring (K and V share it)
    static constexpr int kOffQ = 0;
    static constexpr int kOffKV = kOffQ + 2 * kTileBytes;
    static constexpr int kOffStage = kOffKV + kSlots * kSlotBytes;   // one O box for the TMA store
    static constexpr int kOffStats = kOffStage + kBoxBytes;          // float4 (l, b, l_norm, 0) [2][128]
    // Ring entries free in pairs: V_j with the next K_{j+1} (they free
    // together), a unit's last V with the next unit's first K, entry 0 alone;
    // pair p = (2p - 1, 2p) has empty barrier p % kPairs, one commit each.
    // At D=64 they also land in pairs (kFullPairs): a step's K_j and V_j,
    // entries (2q, 2q+1), share full barrier q % kPairs (one arrival and one
    // tile of bytes from each copy), so the wait for K_j before QK(j) also
    // covers V_j for PV(j).  That makes QK(j+1) wait for V_{j+1} too: with the
    // 8-slot ring there is slack for it, with D=128's 4 slots there is not
    // (measured 5-9% slower there, 2-3% faster at D=64).  kSlots barriers are
    // reserved per side.
    static constexpr bool kFullPairs = (D == 64) && !(kKP && kScoreRotation);
    // Two-tile units: the softmax warp that sees a key step's last scores
    // frees the pair (V_{j-1}, K_j) (that step's last QK comes after the
    // previous step's every P*V), not a commit from the MMA issuer.
    static constexpr bool kSoftmaxRelease = (D == 64) && !kKP && !kScoreRotation;
    // Two-tile units at D=128: no release at all.  The loader waits, before
    // reusing the pair (V_{j-1}, K_j)'s slots, on the score barrier of step
    // j's last QK itself (that commit completes when the same MMAs do).  Each
    // slot's score barriers then alternate between two: the loader runs at
    // most one step behind them, so a parity wait never aliases (the 8-entry
    // ring at D=64 would let it run three behind).
    static constexpr bool kLoaderOnScores = (D == 128) && !kKP && !kScoreRotation;
    static constexpr int kPairs = kSlots / 2;
    static constexpr int kBarKVEmpty = kBarKVFull + kSlots;
    __device__ static constexpr uint32_t pair_of(uint32_t entry) { return (entry + 1u) / 2u; }
    // [slots] a V tile converted to fp16 in place (bf16 inputs; 2 warps).  K
    // and V alternate through an even number of slots, so V tiles always use
    // the odd slots and each of these barriers completes once per V tile there.
    static constexpr int kBarVConv = kBarKVEmpty + kSlots;
    static constexpr int kNumBars = kBarVConv + kSlots;
    static constexpr int kOffBars = kOffStats + 2 * kBM * 16;
    static constexpr int kOffCtl = kOffBars + kNumBars * (int)kBarStride;          // [0] TMEM base, [1] abort, [2] epilogue go
    static constexpr int kSmemBytes = kOffCtl + 16 + 1024;            // + slack to align the base to 1 KB
    // TMEM columns.  D=128: S0 | S1 | O0 | O1; P_t overwrites the first half of
    // S_t, so the next QK_t must wait for PV_t (the issuer orders them).
    // D=64 (kRot): three score buffers SB0 | SB1 | SB2 and O0 | O1 fill the 512
    // columns.  A unit's key steps, slot by slot in issue order, are its ops
    // 0, 1, 2, ...; op m's scores (and then its P) live in buffer m % 3, and
    // the QK of op m + 3 is issued right after the PV of op m, so each slot's
    // next scores are computed while its softmax still works on the current
    // ones (with two buffers they could only follow the PV).  In key-parity
    // units the two slots hold one query tile's even and odd key tiles: O0
    // and O1 are two partial accumulators the epilogue merges.
    static constexpr bool kRot = (D == 64) && kScoreRotation;
    static constexpr int kSBufs = kRot ? 3 : 2;
    static_assert(kSBufs <= kStepBars, "one step barrier per score buffer");
    __device__ static constexpr uint32_t col_s(int t) { return t ? 128u : 0u; }
    __device__ static constexpr uint32_t col_sb(uint32_t b) { return 128u * b; }
    __device__ static constexpr uint32_t col_o(int t) { return (kRot ? 384u : 256u) + (t ? (uint32_t)D : 0u); }
    __device__ static constexpr uint32_t col_p(int t) { return col_s(t); }
};


static_assert(Cfg<64, true>::kSmemBytes <= Cfg<64>::kSmemBytes, "key-parity instances fit the D=64 launch geometry");

// bf16 inputs with K and V on separate full barriers (D=128): the V
// converters announce V_j only once K_{j+1} has landed too, so the MMA
// issuer's one wait per key step for the converted V_j also covers the next
// QKs' K (its own wait for K_{j+1} and the fence after it go: one wait and one
// fence fewer per step on the issuing thread).  K_{j+1} lands right after V_j.
template <int D, bool kBF16, bool kKP>
__host__ __device__ constexpr bool conv_covers_k() { return converts_v<kBF16>() && !Cfg<D, kKP>::kFullPairs && !Cfg<D, kKP>::kRot; }

struct Unit {
    int status;      // kUnitDone, kUnitOk or kUnitSkip
    int id;          // position of the unit in the schedule (split: its workspace slot)
    int bh;
    int j0;          // first key step of the unit (0 unless split)
    int kt0;         // key-parity units: first key tile (step j of slot t is key tile kt0 + 2j + t)
    int q_tile[2];   // query tile index of each tile of the unit
    int nkv[2];      // end (exclusive) of the key tiles tile t visits; 0 = tile absent
    int last[2];     // the tile's last key tile overall: the one the mask applies to
    int nmax;        // max of nkv
};

enum : int { kUnitDone = 0, kUnitOk = 1, kUnitSkip = 2 };

// A unit's ops (kRot): the key steps of its two slots in issue order.  While
// both slots have steps left, op 2i is slot 0's step j0 + i and op 2i + 1 slot
// 1's; after that the slot with more steps runs alone.
struct OpMap {
    int j0, cm, tl, n;   // first step, steps both slots run, the longer slot, op count
    __device__ __forceinline__ OpMap(const Unit& un) {
        const int c0 = un.nkv[0] > un.j0 ? un.nkv[0] - un.j0 : 0;
        const int c1 = un.nkv[1] > un.j0 ? un.nkv[1] - un.j0 : 0;
        j0 = un.j0;
        cm = min(c0, c1);
        tl = c0 > c1 ? 0 : 1;
        n = c0 + c1;
    }
    __device__ __forceinline__ int slot(int m) const { return m < 2 * cm ? (m & 1) : tl; }
    __device__ __forceinline__ int step(int m) const { return m < 2 * cm ? j0 + (m >> 1) : j0 + m - cm; }
    // op of slot t's step j
    __device__ __forceinline__ int op(int t, int j) const { return j - j0 < cm ? 2 * (j - j0) + t : j - j0 + cm; }
    __device__ __forceinline__ bool first_of_step(int m) const { return m >= 2 * cm || !(m & 1); }
    __device__ __forceinline__ bool last_of_step(int m) const { return m >= 2 * cm || (m & 1); }
};

// The r-th work unit of this CTA; every role of the CTA walks the same list.
//
// kSchedSnake: units ordered group of `head_group` heads by group, longest
// first inside a group (causal: the last query tiles); CTA c takes, in round r,
// entry r*G + c (r even) or r*G + G-1-c (r odd), a snake over a list of falling
// cost.  Without the mask (all units cost the same) the group is one head and
// consecutive CTAs share a head's K/V.
//
// kSchedPairs (causal): query group g of a head is paired with group
// n_qgroups-1-g, so every pair costs the same; CTA c takes pair (r/2)*G + c, its
// long unit on even r and its short unit on odd r.  Pairs are ordered head by
// head, so the CTAs of a round share few heads and the short unit re-reads K/V
// the long one just brought into L2.  With an odd group count the middle group
// pairs with itself and its second slot is skipped.
//
// kSchedTable (causal launches of several rounds, up to kSchedTableMaxUnits
// units): the host's list schedule, carried in Params (per-CTA offsets and unit
// indices bh * n_qgroups + qg); CTA c runs its list in order.  The host builds
// it longest first inside groups of heads, each unit to the least loaded CTA.
//
// Split-KV launches take (head, query group, key chunk) units in dense order.
// Returned by value: a unit the caller keeps by reference becomes
// address-taken and its fields are reloaded from local memory in the MMA
// issuer's inner loop (measured: 8% slower).
template <bool kSplit, bool kKP = false>
__device__ __forceinline__ Unit unit_at(int r, const Params& p)
{
    const long long G = gridDim.x, c = blockIdx.x;
    Unit un;
    un.status = kUnitOk;
    un.j0 = 0;
    int bh, qg;
    if constexpr (kSplit) {
        // (head, query group, key chunk), dense and in that order
        const long long u = (long long)r * G + c;
        un.status = u >= p.n_units ? kUnitDone : kUnitOk;
        const int ui = (int)u;
        bh = ui / p.units_per_head;
        int rem = ui - bh * p.units_per_head;
        qg = 0;
        for (int n = split_chunks(0, p.tpu, p.n_qtiles, p.n_kv, p.causal, p.split_chunk);
             rem >= n && qg + 1 < p.n_qgroups;
             n = split_chunks(qg, p.tpu, p.n_qtiles, p.n_kv, p.causal, p.split_chunk)) {
            rem -= n;
            ++qg;
        }
        un.j0 = rem * p.split_chunk;
        un.id = ui;
    } else if (p.sched == kSchedTable) {
        // the host's list schedule: this CTA's units, in order
        const int at = (int)p.tab_off[c] + r;
        un.status = at >= (int)p.tab_off[c + 1] ? kUnitDone : kUnitOk;
        const int u = un.status == kUnitOk ? (int)p.tab_unit[at] : 0;
        bh = u / p.n_qgroups;
        qg = u - bh * p.n_qgroups;
        un.id = u;
    } else if (p.sched == kSchedPairs) {
        // 32-bit arithmetic: pair indices stay below 2^31 (a 64-bit division
        // would bring in a called subroutine and slowed the whole kernel)
        const long long pl = (long long)(r >> 1) * G + c;
        un.status = pl >= p.n_pairs ? kUnitDone : kUnitOk;
        const int pi = (int)pl;
        const int h = pi / p.pairs_per_head;
        const int k = pi - h * p.pairs_per_head;
        const int longer = p.n_qgroups - 1 - k;
        if (un.status == kUnitOk && (r & 1) && k == longer) un.status = kUnitSkip;
        bh = h;
        qg = (r & 1) ? k : longer;
        un.id = 2 * pi + (r & 1);
    } else {
        const long long u = (long long)r * G + ((r & 1) ? (G - 1 - c) : c);
        un.status = u >= p.n_units ? kUnitDone : kUnitOk;
        const int per_group = p.head_group * p.n_qgroups;
        const int g = (int)u / per_group;
        const int w = (int)u - g * per_group;
        const int h0 = g * p.head_group;
        const int hg = min(p.head_group, p.BH - h0);
        const int rank = w / hg;
        bh = h0 + (w - rank * hg);
        qg = p.causal ? (p.n_qgroups - 1 - rank) : rank;
        un.id = (int)u;
    }
    un.bh = bh;
    un.nmax = 0;
    un.kt0 = 0;
    if constexpr (kKP) {
        // key-parity unit: one query tile (p.tpu == 1); its key tiles
        // [kt0, end) alternate between slot 0 (even steps of the unit's own
        // count) and slot 1, step j holding tiles kt0 + 2j and kt0 + 2j + 1
        const int qt = qg;
        const int total = kv_tiles_of(qt, p.n_kv, p.causal);
        const int kt0 = un.j0;
        const int end = kSplit ? min(kt0 + p.split_chunk, total) : total;
        const int count = end > kt0 ? end - kt0 : 0;
        un.kt0 = kt0;
        un.j0 = 0;
        un.q_tile[0] = un.q_tile[1] = qt;
        un.last[0] = un.last[1] = total - 1;
        un.nkv[0] = (count + 1) / 2;
        un.nkv[1] = count / 2;
        un.nmax = un.nkv[0];
    } else {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int qt = qg * p.tpu + t;
            const bool active = (t < p.tpu) && (qt < p.n_qtiles);
            const int total = kv_tiles_of(qt, p.n_kv, p.causal);
            un.q_tile[t] = qt;
            un.last[t] = total - 1;
            if constexpr (kSplit) {
                const int end = min(un.j0 + p.split_chunk, total);
                un.nkv[t] = (active && end > un.j0) ? end : 0;
            } else {
                un.nkv[t] = active ? total : 0;
            }
            un.nmax = max(un.nmax, un.nkv[t]);
        }
    }
    return un;
}

// Event trace: compiled in only with -DFA_TRACE (a separate library); the
// production kernel contains none of it.
#ifdef FA_TRACE
__device__ __forceinline__ void trace_event(const Params& p, int role, uint32_t& n, uint32_t ev, uint32_t arg)
{
    if ((int)blockIdx.x < p.trace_ctas && (int)n < p.trace_cap) {
        const unsigned long long t = clock64();
        p.trace[((size_t)blockIdx.x * kTraceRoles + role) * (size_t)p.trace_cap + n] =
            ((unsigned long long)ev << 56) | ((unsigned long long)(arg & 0xFFFFu) << 40) | (t & 0xFFFFFFFFFFull);
        ++n;
    }
}
#define FA_TRACE_DECL uint32_t tr_n = 0
#define FA_TRACE_EV(cond, role, ev, arg) \
    do {                                 \
        if (cond) trace_event(p, role, tr_n, ev, arg); \
    } while (0)
#else
#define FA_TRACE_DECL (void)0
#define FA_TRACE_EV(cond, role, ev, arg) (void)0
#endif

// Wait-site codes recorded in the status word: role << 8 | barrier index.
// Status word of a CTA that found O not finite with bf16 inputs: V held a value
// beyond fp16's range (its P*V runs in fp16), or an input was not finite.
constexpr uint32_t kSiteRangeV = 0x800;
enum : uint32_t { kSiteSoftmax = 0x100, kSiteEpilogue = 0x300, kSiteLoad = 0x400, kSiteMma = 0x500,
                  kSiteDrain = 0x600 };

// ---------------------------------------------------------------------------------
// Softmax warpgroup t: one thread per query row of tile t.
template <int D, bool kBF16, bool kSplit, bool kKP>
__device__ __forceinline__ void softmax_role(const Params& p, const ptx::WaitCtx& wc, int t, uint32_t tmem,
                                             uint32_t bars, float4* stats)
{
    // kKP: key-parity units (one query tile; slot t takes its key tiles
    // kt0 + 2j + t, with its own base, sum and accumulator O_t, merged by the
    // epilogue).  Otherwise slot t is query tile t of the unit.
    using C = Cfg<D, kKP>;
    const int lane = threadIdx.x & 31;
    const int wq = (threadIdx.x >> 5) & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tO = tmem + lane_base + C::col_o(t);
    const float sl2 = p.scale_log2;
    // ph_s: phase bit of step barrier i at bit i; sb: the step barrier this
    // slot takes next (kRot: in turn over kSBufs, else always 0); pvd: kRot's
    // P*V-done waits so far (two barriers in turn)
    uint32_t ph_s = 0, ph_te = 0, ph_o = 0, sb = 0, pvd = 0;
    FA_TRACE_DECL;
    [[maybe_unused]] const bool tr = (threadIdx.x & 127) == 0;   // the warpgroup's trace events (FA_TRACE builds)

    uint32_t kv_next = 0;   // kSoftmaxRelease: the ring entry of the next unit's first K
    for (int r = 0;; ++r) {
        const Unit un = unit_at<kSplit, kKP>(r, p);
        if (un.status == kUnitDone) break;
        if (un.status == kUnitSkip) continue;
        const uint32_t kvb = kv_next;   // K_j is ring entry kvb + 2(j - j0)
        kv_next += 2u * (uint32_t)max(0, un.nmax - un.j0);
        // t is a runtime value: select instead of indexing, so the unit stays in registers
        const int nkv = t ? un.nkv[1] : un.nkv[0];
        const int q_tile = t ? un.q_tile[1] : un.q_tile[0];
        // the masked tile: the row's last key tile (always nkv - 1 without a split)
        const int last = (kSplit || kKP) ? (t ? un.last[1] : un.last[0]) : nkv - 1;
        if (nkv == 0) continue;
        float b = -INFINITY;   // base of the row, base-2 scaled units
        float l = 0.f;         // running sum of 2^(x - b): gives the LSE
        // bf16 inputs: O is normalised by l + dl, where dl sums, per key tile,
        // the rounding of the tile's largest p to P's 16-bit type.  The MMAs
        // weight V with the rounded P; when one key dominates a row, its
        // rounding (2^-12 relative for fp16 P, 2^-9 for bf16 P) would otherwise
        // scale that row of O, and a bf16 O in [4, 8) is already rounded to
        // within 2^-6 (without dl the stress workload's worst row measured
        // 1.1e-3 off).  fp16 inputs round O to 2^-11 relative: dl stays 0.
        float dl = 0.f;
        const OpMap om(un);
        for (int j = un.j0; j < nkv; ++j) {
            const int kt = kKP ? un.kt0 + 2 * j + t : j;   // the key tile in S_t
            // this step's scores (then its P): slot t's own columns, or (kRot)
            // the buffer of the step's op
            const uint32_t tS = tmem + lane_base +
                                (C::kRot ? C::col_sb((uint32_t)om.op(t, j) % (uint32_t)C::kSBufs) : C::col_s(t));
            const uint32_t tP = tS;
            const uint32_t bstep = (uint32_t)(kStepBars * t) + sb;
            // the step's P barrier: in turn with the scores' under kRot, else the slot's first
            const uint32_t bpub = C::kRot ? bstep : (uint32_t)(kStepBars * t);
            if (!ptx::mbar_wait_warp(wc, bars + kBarStride * (kBarSFull + bstep), (ph_s >> sb) & 1u, kSiteSoftmax | (kBarSFull + bstep)))
                return;
            ph_s ^= 1u << sb;
            if constexpr (C::kRot)
                sb = sb + 1u == (uint32_t)C::kSBufs ? 0u : sb + 1u;
            else if constexpr (C::kLoaderOnScores)
                sb ^= 1u;
            if constexpr (C::kSoftmaxRelease) {
                // this step's last QK (slot 1's, or slot 0's when slot 1 is
                // done or absent) has finished, and with it every P*V of the
                // step before: V_{j-1} and K_j are free
                if ((t == 1 || j >= un.nkv[1]) && wq == 0)
                    ptx::mbar_arrive(bars + kBarStride * (C::kBarKVEmpty + C::pair_of(kvb + 2u * (uint32_t)(j - un.j0)) % C::kPairs),
                                     lane == 0);
            }
            // kRot: the slot's previous P*V may still run; it must finish
            // before O is rescaled, and its barrier is consumed once per step
            auto pv_done_wait = [&]() -> bool {
                const uint32_t b = kBarPVDone + 2 * t + (pvd & 1u);
                const bool ok = ptx::mbar_wait_warp(wc, bars + kBarStride * b, (pvd >> 1) & 1u, kSiteSoftmax | b);
                ++pvd;
                return ok;
            };
            FA_TRACE_EV(tr, t, kEvSReady, j);
            ptx::tc_fence_after();
            // scores of the row; each 32-column load also returns its maximum
            uint32_t sr[128];
            float pm[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) ptx::tmem_ld32_max(tS + 32 * c, sr + 32 * c, pm[c]);
            ptx::tmem_wait_ld();
            ptx::reg_fence(sr);
            ptx::reg_fence(pm);
            FA_TRACE_EV(tr, t, kEvSLoaded, j);
            float* s = reinterpret_cast<float*>(sr);
            float mraw;
            if (p.mask_last && kt == last) {
                // keys beyond the sequence, and (causal) keys after this row
                const int qrow = q_tile * kBM + row;
                int lim = p.S - 1 - kt * kBN;
                if (p.causal) lim = min(lim, qrow - kt * kBN);
#pragma unroll
                for (int c = 0; c < 128; ++c) s[c] = (c <= lim) ? s[c] : -INFINITY;
                // maximum over what is left: four chains of three-input max
                float m[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) m[k] = ptx::max3(s[32 * k], s[32 * k + 1], s[32 * k + 2]);
#pragma unroll
                for (int i = 3; i < 31; i += 2) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) m[k] = ptx::max3(m[k], s[32 * k + i], s[32 * k + i + 1]);
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) m[k] = fmaxf(m[k], s[32 * k + 31]);
                mraw = fmaxf(ptx::max3(m[0], m[1], m[2]), m[3]);
            } else {
                mraw = fmaxf(ptx::max3(pm[0], pm[1], pm[2]), pm[3]);
            }
            const float mx = mraw * sl2;
            // conditional re-base: keep b unless the maximum passed b + T.  The O
            // rescale below is warp-wide (collective TMEM accesses), so when one
            // row of the warp re-bases, every row of the warp re-bases to its
            // own candidate at no extra cost: all 32 restart with the full
            // margin, and the next warp rescale waits for a row to climb T more.
            const float cand = fmaxf(b, mx);
            const bool rebase = cand > b + rebase_threshold<p_is_bf16<kBF16>()>();
            const bool rescale = j > un.j0 && __any_sync(0xffffffffu, rebase);
#ifdef FA_DEBUG_STATS
            if (p.dbg_count != nullptr && j > un.j0) {
                // the debug build counts the kernel's own re-bases
                const unsigned rows = __popc(__ballot_sync(0xffffffffu, rebase));
                if (lane == 0 && rows > 0u) {
                    atomicAdd(p.dbg_count + 0, 1ull);
                    atomicAdd(p.dbg_count + 1, (unsigned long long)rows);
                }
            }
#endif
            float h = 1.f;
            if (rebase || rescale) {
                // a row that re-bases moves to its maximum plus the overshoot; a
                // row the warp carries along only moves if that lies above its
                // base (never by the overshoot again: repeated, that would push
                // its p towards fp16's underflow)
                const float nb_new = fmaxf(b, mx + rebase_overshoot<p_is_bf16<kBF16>()>());
                h = ptx::ex2(b - nb_new);   // 0 on the first tile (b = -inf)
                b = nb_new;
            }
            FA_TRACE_EV(tr, t, kEvMaxDone, j);
            if (rescale) {
                if constexpr (C::kRot) {
                    if (!pv_done_wait()) return;
                }
                // this warp's 32 rows of O_t are scaled by 2^(b_old - b_new)
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t o[32];
                    ptx::tmem_ld32_wait(tO + c0, o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * h);
                    ptx::tmem_st32(tO + c0, o);
                }
                FA_TRACE_EV(tr, t, kEvRescale, j);
            }
            // p = 2^(s * scale*log2e - b): one packed FMA per pair, two ex2,
            // packed row sums in four independent accumulators; P is published
            // once complete (with FA_PV_SPLIT also after its first 64 keys)
            const float nb = (b == -INFINITY) ? 0.f : -b;
            const uint64_t c2 = ptx::f2_pack(sl2, sl2), nb2 = ptx::f2_pack(nb, nb);
            uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
            if constexpr (kBF16) {
                // the tile maximum's p, by the same FMA and ex2 the loop below uses
                const float pm = ptx::ex2(fmaf(mraw, sl2, nb));
                dl = fmaf(dl, h, ptx::round16<p_is_bf16<kBF16>()>(pm) - pm);
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float x0, x1;
                    ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(s[c * 32 + 2 * i], s[c * 32 + 2 * i + 1]), c2, nb2), x0, x1);
                    float p0, p1;
                    if (kExp2PolyPairs > 0 && ((i + 1) * kExp2PolyPairs / 16) != (i * kExp2PolyPairs / 16)) {
                        ptx::f2_unpack(ptx::f2_exp2_poly(x0, x1), p0, p1);   // spread evenly over the 16 pairs
                    } else {
                        p0 = ptx::ex2(x0);
                        p1 = ptx::ex2(x1);
                    }
                    acc[i & 3] = ptx::f2_add(acc[i & 3], ptx::f2_pack(p0, p1));
                    pk[i] = ptx::pack2<p_is_bf16<kBF16>()>(p0, p1);
                }
                ptx::tmem_st16(tP + c * 16, pk);
                if ((kPVSplit && c == 1) || c == 3) {
                    // publish P (and the rescaled O) for the MMA issuer: whole,
                    // or with FA_PV_SPLIT keys 0-63 at c == 1
                    ptx::tmem_wait_st();
                    ptx::tc_fence_before();
                    __syncwarp();
                    ptx::mbar_arrive(bars + kBarStride * ((c == 1 ? kBarPHalf : kBarPFull) + bpub), lane == 0);
                    if (c == 1) FA_TRACE_EV(tr, t, kEvExpDone, j);
                }
            }
            FA_TRACE_EV(tr, t, kEvPDone, j);
            if constexpr (C::kRot) {
                if (j > un.j0 && !rescale && !pv_done_wait()) return;
            }
            float sa, sb;
            ptx::f2_unpack(ptx::f2_add(ptx::f2_add(acc[0], acc[1]), ptx::f2_add(acc[2], acc[3])), sa, sb);
            l = fmaf(l, h, sa + sb);
        }
#ifdef FA_DEBUG_STATS
        if (!kSplit && !kKP && p.dbg_rows != nullptr) {
            // the debug build writes each row's final base and row sum
            const int qrow = q_tile * kBM + row;
            if (qrow < p.S) {
                float* d = p.dbg_rows + 2 * ((size_t)un.bh * p.S + qrow);
                d[0] = b;
                d[1] = l;
            }
        }
#endif
        if constexpr (epi_in_softmax<kBF16, kSplit, kKP>()) {
            // this tile's epilogue, here: O_t is final once its last PV completed
            if (!ptx::mbar_wait_warp(wc, bars + kBarStride * (kBarOFull + t), ph_o, kSiteSoftmax | (kBarOFull + t))) return;
            ph_o ^= 1u;
            ptx::tc_fence_after();
            const int qrow = q_tile * kBM + row;
            const bool in = qrow < p.S;
            if (in) p.lse[(size_t)un.bh * (size_t)p.S + (size_t)qrow] = (b + ptx::lg2(l)) * kLn2;
            const float inv_l = 1.0f / (l + dl);
            const uint64_t il2 = ptx::f2_pack(inv_l, inv_l);
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + ((size_t)un.bh * p.S + qrow) * D);
            float osum = 0.f;   // converted V: a value beyond fp16's range makes O (and this sum) not finite
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t o[32];
                ptx::tmem_ld32_wait(tO + c0, o);
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float x0, x1;
                    ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])), il2),
                                   x0, x1);
                    if constexpr (converts_v<kBF16>()) osum += fabsf(x0) + fabsf(x1);
                    pk[i] = ptx::pack2<kBF16>(x0, x1);
                }
                if (in) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[c0 / 8 + i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                }
            }
            if (converts_v<kBF16>() && in && !(osum <= 3.0e38f)) atomicCAS(p.status, 0u, kSiteRangeV);
            ptx::tc_fence_before();
            __syncwarp();
            ptx::mbar_arrive(bars + kBarStride * (kBarOEmpty + t), lane == 0);
        } else {
            // hand (l, b) of every row to the epilogue
            if (!ptx::mbar_wait_warp(wc, bars + kBarStride * (kBarStEmpty + t), ph_te ^ 1u, kSiteSoftmax | (kBarStEmpty + t)))
                return;
            ph_te ^= 1u;
            stats[t * kBM + row] = make_float4(l, b, l + dl, 0.f);
            __syncwarp();
            ptx::mbar_arrive(bars + kBarStride * (kBarStFull + t), lane == 0);
        }
    }
}

// ---------------------------------------------------------------------------------
// Correction/epilogue warpgroup: per unit and query tile, the final correction
// O_t / l, the LSE, conversion to 16 bits, shared-memory staging, TMA store.
template <int D, bool kBF16, bool kSplit, bool kKP>
__device__ __forceinline__ void correction_epilogue_role(const Params& p, const ptx::WaitCtx& wc,
                                                         const CUtensorMap* tm_o, uint32_t tmem, uint32_t smem_base,
                                                         uint32_t bars, const float4* stats, volatile uint32_t* ctl_go)
{
    using C = Cfg<D, kKP>;
    const int lane = threadIdx.x & 31;
    const int wq = (threadIdx.x >> 5) & 3;
    const int row = wq * 32 + lane;
    const bool leader = (threadIdx.x == 8 * 32);
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t stage = smem_base + C::kOffStage;
    volatile uint32_t* go = ctl_go;   // leader's wait outcome, read by all 128 threads
    uint32_t ph_o = 0u, ph_t = 0u;   // phase bit of tile t at bit t
    FA_TRACE_DECL;
    if constexpr (epi_in_softmax<kBF16, kSplit, kKP>()) return;   // the softmax warpgroups run the epilogue

    for (int r = 0;; ++r) {
        const Unit un = unit_at<kSplit, kKP>(r, p);
        if (un.status == kUnitDone) break;
        if (un.status == kUnitSkip) continue;
        if constexpr (kKP) {
            // key-parity unit: the unit's one query tile has two partial
            // results, slot 0 (its even key tiles: O_0, base b0, sum l0) and
            // slot 1 (odd: O_1, b1, l1; absent when the unit has one key tile);
            // with m = max(b0, b1) and w_h = 2^(b_h - m) the row's sum is
            // w0 l0 + w1 l1 and its O is (w0 O_0 + w1 O_1) / (w0 l0' + w1 l1')
            // (l' the normaliser, l + dl)
            if (un.nkv[0] == 0) continue;
            const bool has1 = un.nkv[1] > 0;
            if (wq == 0) {   // the leader's warp waits, all lanes together
                bool ok = ptx::mbar_wait(wc, bars + kBarStride * kBarOFull, ph_o & 1u, kSiteEpilogue | kBarOFull) &&
                          ptx::mbar_wait(wc, bars + kBarStride * kBarStFull, ph_t & 1u, kSiteEpilogue | kBarStFull);
                if (has1)
                    ok = ok &&
                         ptx::mbar_wait(wc, bars + kBarStride * (kBarOFull + 1), (ph_o >> 1) & 1u, kSiteEpilogue | (kBarOFull + 1)) &&
                         ptx::mbar_wait(wc, bars + kBarStride * (kBarStFull + 1), (ph_t >> 1) & 1u, kSiteEpilogue | (kBarStFull + 1));
                ok = __all_sync(0xffffffffu, ok);
                if (leader) go[0] = ok ? 1u : 0u;
            }
            ptx::named_bar_sync(1, 128);
            if (go[0] == 0u) goto done;
            const uint32_t flip = has1 ? 3u : 1u;
            ph_o ^= flip;
            ph_t ^= flip;
            ptx::tc_fence_after();
            const float4 s0 = stats[row];
            const float4 s1 = has1 ? stats[kBM + row] : make_float4(0.f, -INFINITY, 0.f, 0.f);
            __syncwarp();
            ptx::mbar_arrive(bars + kBarStride * kBarStEmpty, lane == 0);
            ptx::mbar_arrive(bars + kBarStride * (kBarStEmpty + 1), has1 && lane == 0);
            const float m = fmaxf(s0.y, s1.y);   // b0 is finite: the unit's first key tile is unmasked for every row
            const float w0 = ptx::ex2(s0.y - m), w1 = has1 ? ptx::ex2(s1.y - m) : 0.f;
            const float lsum = w0 * s0.x + w1 * s1.x;
            const float inv_l = 1.0f / (w0 * s0.z + w1 * s1.z);
            const float c0 = w0 * inv_l, c1 = w1 * inv_l;
            const float row_lse = (m + ptx::lg2(lsum)) * kLn2;
            const uint32_t tO0 = tmem + lane_base + C::col_o(0), tO1 = tmem + lane_base + C::col_o(1);
            static_assert(D == 64, "key-parity units: D=64");
            float osum = 0.f;   // converted V: a value beyond fp16's range makes O (and this sum) not finite
            // O_0 and O_1, 32 columns at a time (O_1 only when slot 1 ran)
            auto merged = [&](int c0c, uint32_t (&oa)[32], uint32_t (&ob)[32]) {
                ptx::tmem_ld32(tO0 + c0c, oa);
                if (has1) ptx::tmem_ld32(tO1 + c0c, ob);
                ptx::tmem_wait_ld();
                ptx::reg_fence(oa);
                ptx::reg_fence(ob);
            };
            if constexpr (kSplit) {
                const size_t slot = (size_t)un.id * kBM + row;   // one tile per unit
                float* dst = p.ws_o + slot * D;
#pragma unroll 1
                for (int c0c = 0; c0c < D; c0c += 32) {
                    uint32_t oa[32], ob[32];
                    merged(c0c, oa, ob);
#pragma unroll
                    for (int i = 0; i < 32; i += 4) {
                        float x[4];
#pragma unroll
                        for (int e2 = 0; e2 < 4; ++e2)
                            x[e2] = has1 ? fmaf(__uint_as_float(oa[i + e2]), c0, __uint_as_float(ob[i + e2]) * c1)
                                         : __uint_as_float(oa[i + e2]) * c0;
                        if constexpr (converts_v<kBF16>()) osum += (fabsf(x[0]) + fabsf(x[1])) + (fabsf(x[2]) + fabsf(x[3]));
                        *reinterpret_cast<float4*>(dst + c0c + i) = make_float4(x[0], x[1], x[2], x[3]);
                    }
                }
                if (converts_v<kBF16>() && !(osum <= 3.0e38f)) atomicCAS(p.status, 0u, kSiteRangeV);
                p.ws_lse[slot] = row_lse;
                ptx::tc_fence_before();
                __syncwarp();
                ptx::mbar_arrive(bars + kBarStride * kBarOEmpty, lane == 0);
                ptx::mbar_arrive(bars + kBarStride * (kBarOEmpty + 1), has1 && lane == 0);
                continue;
            }
            const int qrow = un.q_tile[0] * kBM + row;
            if (qrow < p.S) p.lse[(size_t)un.bh * (size_t)p.S + (size_t)qrow] = row_lse;
#ifdef FA_DEBUG_STATS
            if (p.dbg_rows != nullptr && qrow < p.S) {
                // the debug build's per-row base and sum: the merged ones
                float* d = p.dbg_rows + 2 * ((size_t)un.bh * p.S + qrow);
                d[0] = m;
                d[1] = lsum;
            }
#endif
            // the staging box is free once the previous TMA store has read it
            if (leader) ptx::bulk_wait_read0();
            ptx::named_bar_sync(1, 128);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t oa[32], ob[32];
                merged(half * 32, oa, ob);
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float a = has1 ? fmaf(__uint_as_float(oa[2 * i]), c0, __uint_as_float(ob[2 * i]) * c1)
                                         : __uint_as_float(oa[2 * i]) * c0;
                    const float b2 = has1 ? fmaf(__uint_as_float(oa[2 * i + 1]), c0, __uint_as_float(ob[2 * i + 1]) * c1)
                                          : __uint_as_float(oa[2 * i + 1]) * c0;
                    if constexpr (converts_v<kBF16>()) osum += fabsf(a) + fabsf(b2);
                    pk[i] = ptx::pack2<kBF16>(a, b2);
                }
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int chunk = half * 4 + cc;   // 16-byte chunk of the 128-byte row
                    const uint32_t addr = stage + row * 128 + ((chunk ^ (row & 7)) << 4);
                    ptx::st_shared_v4(addr, pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            ptx::mbar_arrive(bars + kBarStride * kBarOEmpty, lane == 0);
            ptx::mbar_arrive(bars + kBarStride * (kBarOEmpty + 1), has1 && lane == 0);
            ptx::fence_proxy_async_shared();
            ptx::named_bar_sync(1, 128);
            if (leader) {
                ptx::tma_store_3d(tm_o, stage, 0, un.q_tile[0] * kBM, un.bh);
                ptx::bulk_commit();
            }
            if (converts_v<kBF16>() && qrow < p.S && !(osum <= 3.0e38f)) atomicCAS(p.status, 0u, kSiteRangeV);
            continue;
        } else {
            // one named barrier carries the leader's wait outcome to all 128
            // threads, so the warpgroup never splits over an abort
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                if (un.nkv[t] == 0) continue;
                if (wq == 0) {   // the leader's warp waits, all lanes together
                    const bool ok = __all_sync(0xffffffffu,
                                               ptx::mbar_wait(wc, bars + kBarStride * (kBarOFull + t), (ph_o >> t) & 1u,
                                                              kSiteEpilogue | (kBarOFull + t)) &&
                                                   ptx::mbar_wait(wc, bars + kBarStride * (kBarStFull + t), (ph_t >> t) & 1u,
                                                                  kSiteEpilogue | (kBarStFull + t)));
                    if (leader) go[0] = ok ? 1u : 0u;
                }
                ptx::named_bar_sync(1, 128);
                if (go[0] == 0u) goto done;
                ph_o ^= 1u << t;
                ph_t ^= 1u << t;
                FA_TRACE_EV(leader, kTrEpilogue, kEvOFull, t);
                ptx::tc_fence_after();
                const float4 st = stats[t * kBM + row];
                __syncwarp();
                ptx::mbar_arrive(bars + kBarStride * (kBarStEmpty + t), lane == 0);
                const float inv_l = 1.0f / st.z;   // the sum of the P values the MMAs used
                const float row_lse = (st.y + ptx::lg2(st.x)) * kLn2;
                if constexpr (kSplit) {
                    // split-KV partial: this chunk's O (normalised by its own row
                    // sum) and LSE, fp32, into the workspace slot of the unit
                    const size_t slot = ((size_t)un.id * p.tpu + t) * kBM + row;
                    float* dst = p.ws_o + slot * D;
                    const uint32_t tO = tmem + lane_base + C::col_o(t);
                    float osum = 0.f;   // converted V: a value beyond fp16's range makes O (and this sum) not finite
#pragma unroll 1
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t o[32];
                        ptx::tmem_ld32_wait(tO + c0, o);
#pragma unroll
                        for (int i = 0; i < 32; i += 4) {
                            const float4 x = make_float4(__uint_as_float(o[i]) * inv_l, __uint_as_float(o[i + 1]) * inv_l,
                                                         __uint_as_float(o[i + 2]) * inv_l, __uint_as_float(o[i + 3]) * inv_l);
                            if constexpr (converts_v<kBF16>()) osum += (fabsf(x.x) + fabsf(x.y)) + (fabsf(x.z) + fabsf(x.w));
                            *reinterpret_cast<float4*>(dst + c0 + i) = x;
                        }
                    }
                    if (converts_v<kBF16>() && !(osum <= 3.0e38f)) atomicCAS(p.status, 0u, kSiteRangeV);
                    p.ws_lse[slot] = row_lse;
                    ptx::tc_fence_before();
                    __syncwarp();
                    ptx::mbar_arrive(bars + kBarStride * (kBarOEmpty + t), lane == 0);
                    FA_TRACE_EV(leader, kTrEpilogue, kEvEpiDone, t);
                    continue;
                }
                const int qrow = un.q_tile[t] * kBM + row;
                if (qrow < p.S) p.lse[(size_t)un.bh * (size_t)p.S + (size_t)qrow] = row_lse;
                const uint32_t tO = tmem + lane_base + C::col_o(t);
                float osum = 0.f;   // converted V: a value beyond fp16's range makes O (and this sum) not finite
#pragma unroll 1
                for (int box = 0; box < C::kBoxes; ++box) {
                    // the staging box is free once the previous TMA store has read it
                    if (leader) ptx::bulk_wait_read0();
                    ptx::named_bar_sync(1, 128);
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        uint32_t o[32];
                        ptx::tmem_ld32_wait(tO + box * 64 + half * 32, o);
                        uint32_t pk[16];
                        const uint64_t il2 = ptx::f2_pack(inv_l, inv_l);
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            float a, b2;
                            ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])), il2),
                                           a, b2);
                            if constexpr (converts_v<kBF16>()) osum += fabsf(a) + fabsf(b2);
                            pk[i] = ptx::pack2<kBF16>(a, b2);
                        }
#pragma unroll
                        for (int cc = 0; cc < 4; ++cc) {
                            const int chunk = half * 4 + cc;   // 16-byte chunk of the 128-byte row
                            const uint32_t addr = stage + row * 128 + ((chunk ^ (row & 7)) << 4);
                            ptx::st_shared_v4(addr, pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
                        }
                    }
                    if (box == C::kBoxes - 1) {
                        ptx::tc_fence_before();
                        __syncwarp();
                        ptx::mbar_arrive(bars + kBarStride * (kBarOEmpty + t), lane == 0);
                    }
                    ptx::fence_proxy_async_shared();
                    ptx::named_bar_sync(1, 128);
                    if (leader) {
                        ptx::tma_store_3d(tm_o, stage, box * 64, un.q_tile[t] * kBM, un.bh);
                        ptx::bulk_commit();
                    }
                }
                if (converts_v<kBF16>() && qrow < p.S && !(osum <= 3.0e38f)) atomicCAS(p.status, 0u, kSiteRangeV);
                FA_TRACE_EV(leader, kTrEpilogue, kEvEpiDone, t);
            }
        }
    }
done:
    if (leader) ptx::bulk_wait0();
}

// ---------------------------------------------------------------------------------
// TMA producer (one thread).
template <int D, bool kSplit, bool kKP>
__device__ __forceinline__ void load_role(const Params& p, const ptx::WaitCtx& wc, const CUtensorMap* tm_q,
                                          const CUtensorMap* tm_k, const CUtensorMap* tm_v, uint32_t smem_base,
                                          uint32_t bars)
{
    const uint32_t ex = (threadIdx.x & 31) == 0 ? 1u : 0u;   // the lane that issues (the whole warp runs the role)
    using C = Cfg<D, kKP>;
    uint32_t ph_qe = 0u;       // phase bit of Q buffer t at bit t
    uint32_t q_issued = 0u;    // bit t: a Q load into buffer t was issued
    uint32_t kv_count = 0;
    bool ok = true;
    FA_TRACE_DECL;
    // kLoaderOnScores: the release of key step g (counted over the CTA's
    // units) is the score barrier of its last QK: slot s's n-th step, kept as
    // s << 31 | n for the last two steps (h[g & 1]); cnt0 / cnt1 count each
    // slot's steps so far, g the steps
    uint32_t g = 0, cnt0 = 0, cnt1 = 0, h0 = 0, h1 = 0;
    for (int r = 0; ok; ++r) {
        const Unit un = unit_at<kSplit, kKP>(r, p);
        if (un.status == kUnitDone) break;
        if (un.status == kUnitSkip) continue;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            if (!ok || un.nkv[t] == 0 || (kKP && t == 1)) continue;   // key-parity units: one Q tile
            if (!ptx::mbar_wait(wc, bars + kBarStride * (kBarQEmpty + t), ((ph_qe >> t) & 1u) ^ 1u, kSiteLoad | (kBarQEmpty + t))) {
                ok = false;
                continue;
            }
            ph_qe ^= 1u << t;
            const uint32_t fb = bars + kBarStride * (kBarQFull + t);
            ptx::mbar_arrive_expect_tx(fb, C::kTileBytes, ex);
            const uint32_t dst = smem_base + C::kOffQ + t * C::kTileBytes;
#pragma unroll
            for (int bx = 0; bx < C::kBoxes; ++bx)
                ptx::tma_load_3d(tm_q, dst + bx * C::kBoxBytes, fb, bx * 64, un.q_tile[t] * kBM, un.bh, ex);
            q_issued |= 1u << t;
            FA_TRACE_EV(ex != 0u, kTrLoad, kEvQLoad, t);
        }
        for (int j = un.j0; j < un.nmax && ok; ++j) {
            // two-tile units: slot 1, when present, has every step of the unit
            const uint32_t last = j < un.nkv[1] ? 1u : 0u;
            const uint32_t info = (last << 31) | (last ? cnt1 : cnt0);
#pragma unroll 1
            for (int kind = 0; kind < 2; ++kind) {
                const uint32_t idx = kv_count;
                const uint32_t slot = idx % C::kSlots;
                if (C::kLoaderOnScores && idx >= (uint32_t)C::kSlots) {
                    // K_j reuses the slots freed by step g - 2, V_j by step g - 1
                    const uint32_t hs = ((g + (uint32_t)kind) & 1u) ? h1 : h0;
                    const uint32_t sl = hs >> 31, n = hs & 0x7FFFFFFFu;
                    const uint32_t b = kBarSFull + kStepBars * sl + (n & 1u);
                    if (!ptx::mbar_wait(wc, bars + kBarStride * b, (n >> 1) & 1u, kSiteLoad | b)) {
                        ok = false;
                        break;
                    }
                } else if (idx >= (uint32_t)C::kSlots) {
                    // the entry this copy overwrites must be freed: its pair's release
                    const uint32_t pr = C::pair_of(idx - C::kSlots);
                    const uint32_t b = C::kBarKVEmpty + pr % C::kPairs;
                    if (!ptx::mbar_wait(wc, bars + kBarStride * b, (pr / C::kPairs) & 1u, kSiteLoad | b)) {
                        ok = false;
                        break;
                    }
                }
                if (kind == 0) {   // step g - 2's entry is used: step g's takes its place
                    if (g & 1u) h1 = info; else h0 = info;
                }
                ++kv_count;
                const uint32_t fb = bars + kBarStride * (kBarKVFull + (C::kFullPairs ? (idx / 2u) % C::kPairs : slot));
                ptx::mbar_arrive_expect_tx(fb, C::kSlotBytes, ex);
                const uint32_t dst = smem_base + C::kOffKV + slot * C::kSlotBytes;
                const CUtensorMap* m = kind ? tm_v : tm_k;
                // key-parity units: the step's two key tiles kt0 + 2j (slot 0)
                // and kt0 + 2j + 1 (slot 1; past the sequence it is zero-filled)
                // in one 256-row copy (their tensor maps have 256-row boxes)
                const int row0 = (kKP ? un.kt0 + 2 * j : j) * kBN;
#pragma unroll
                for (int bx = 0; bx < C::kBoxes; ++bx)
                    ptx::tma_load_3d(m, dst + bx * C::kBoxBytes, fb, bx * 64, row0, un.bh, ex);
                FA_TRACE_EV(ex != 0u, kTrLoad, kEvKVLoad, idx);
            }
            if (j < un.nkv[0]) ++cnt0;
            if (j < un.nkv[1]) ++cnt1;
            ++g;
        }
    }
    // Every issued copy must land before the CTA exits (after an abort, too).
#pragma unroll
    for (int t = 0; t < 2; ++t)
        if ((q_issued >> t) & 1u)
            ptx::mbar_wait_drain(wc, bars + kBarStride * (kBarQFull + t), ((ph_qe >> t) & 1u) ^ 1u, kSiteDrain | (kBarQFull + t));
    if (!C::kFullPairs) {
        for (uint32_t s = 0; s < (uint32_t)C::kSlots && s < kv_count; ++s) {
            const uint32_t last = kv_count - 1 - ((kv_count - 1 - s) % C::kSlots);   // last use of slot s
            ptx::mbar_wait_drain(wc, bars + kBarStride * (kBarKVFull + s), (last / C::kSlots) & 1u,
                                 kSiteDrain | (kBarKVFull + s));
        }
    } else if (kv_count > 0) {
        const uint32_t qmax = (kv_count - 1) / 2;   // the last pair with a copy issued
        // a pair left with only its K copy (an abort in between) gets its
        // second arrival here, so its phase completes once that copy lands
        if (kv_count & 1u) ptx::mbar_arrive(bars + kBarStride * (kBarKVFull + qmax % C::kPairs), ex);
        for (uint32_t b = 0; b < (uint32_t)C::kPairs && b <= qmax; ++b) {
            const uint32_t q = qmax - ((qmax - b) % C::kPairs);   // last pair on barrier b
            ptx::mbar_wait_drain(wc, bars + kBarStride * (kBarKVFull + b), (q / C::kPairs) & 1u, kSiteDrain | (kBarKVFull + b));
        }
    }
}

// ---------------------------------------------------------------------------------
// V converter (bf16 inputs; warps 14-15, and the epilogue warpgroup's warps 8-11
// when the epilogue runs in the softmax warpgroups): each V tile, once it has
// landed, is rewritten in place from bf16 to fp16 (element by element, so the
// swizzled layout stays valid), made visible to the tensor core's reads
// (fence.proxy.async) and announced on its slot's conversion barrier.  The walk
// over units and key tiles is the loader's: K_j, then V_j, for every key tile
// of every unit.  A value beyond fp16's range becomes infinite, so O does too;
// the epilogues check O and record kSiteRangeV (no per-element check here).
template <int D, bool kSplit, bool kKP, int kWarps>
__device__ __forceinline__ void vconvert_role(const Params& p, const ptx::WaitCtx& wc, uint32_t smem_base,
                                              uint32_t bars, int conv_tid)
{
    using C = Cfg<D, kKP>;
    const int lane = threadIdx.x & 31;
    uint32_t kv_count = 0;
    for (int r = 0;; ++r) {
        const Unit un = unit_at<kSplit, kKP>(r, p);
        if (un.status == kUnitDone) break;
        if (un.status == kUnitSkip) continue;
        for (int j = un.j0; j < un.nmax; ++j) {
            const uint32_t iv = kv_count + 1;   // K_j's entry, then V_j's
            kv_count += 2;
            bool ok;
            if constexpr (C::kFullPairs) {
                const uint32_t q = iv / 2u, b = kBarKVFull + q % C::kPairs;
                ok = ptx::mbar_wait_warp(wc, bars + kBarStride * b, (q / C::kPairs) & 1u, kSiteLoad | 0x80u | b);
            } else {
                const uint32_t slot = iv % C::kSlots;
                ok = ptx::mbar_wait_warp(wc, bars + kBarStride * (kBarKVFull + slot), (iv / C::kSlots) & 1u,
                                         kSiteLoad | 0x80u | (kBarKVFull + slot));
            }
            if (!ok) return;
            const uint32_t tile = smem_base + C::kOffKV + (iv % C::kSlots) * C::kSlotBytes;
            // eight 16-byte chunks in flight per thread: the conversion's latency
            // sits in front of the tile's first P*V (unrolled 2: train 1088,
            // 8: 1152, 16: 1106 TFLOPS)
#pragma unroll 8
            for (uint32_t off = (uint32_t)conv_tid * 16u; off < (uint32_t)C::kSlotBytes; off += 32u * kWarps * 16u) {
                uint32_t w[4];
                ptx::ld_shared_v4(tile + off, w);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    w[k] = ptx::pack2<false>(__uint_as_float(w[k] << 16), __uint_as_float(w[k] & 0xFFFF0000u));
                ptx::st_shared_v4(tile + off, w[0], w[1], w[2], w[3]);
            }
            ptx::fence_proxy_async_shared();
            __syncwarp();
            if constexpr (conv_covers_k<D, true, kKP>()) {
                // K_{j+1} (a unit's first K the issuer waits for itself)
                if (j + 1 < un.nmax) {
                    const uint32_t ik = iv + 1u, slot = ik % C::kSlots;
                    if (!ptx::mbar_wait_warp(wc, bars + kBarStride * (kBarKVFull + slot), (ik / C::kSlots) & 1u,
                                             kSiteLoad | 0x80u | (kBarKVFull + slot)))
                        return;
                }
            }
            ptx::mbar_arrive(bars + kBarStride * (C::kBarVConv + iv % C::kSlots), lane == 0);
        }
    }
}

// ---------------------------------------------------------------------------------
// tcgen05 MMA issuer (one thread).
template <int D, bool kBF16, bool kSplit, bool kKP>
__device__ __forceinline__ void mma_role(const Params& p, const ptx::WaitCtx& wc, uint32_t tmem, uint32_t smem_base,
                                         uint32_t bars)
{
    const uint32_t ex = (threadIdx.x & 31) == 0 ? 1u : 0u;   // the lane that issues (the whole warp runs the role)
    using C = Cfg<D, kKP>;
    constexpr uint32_t kIdescQK = ptx::idesc_f16(kBM, kBN, kBF16, false);   // Q, K both K-major
    constexpr uint32_t kIdescPV = ptx::idesc_f16(kBM, D, p_is_bf16<kBF16>(), true);   // V MN-major (D contiguous)
    uint32_t ph_q = 0u, ph_ph = 0u, ph_p = 0u, ph_oe = 0u;   // phase bit of tile t at bit t
    uint32_t sq = 0u;   // kLoaderOnScores: bit t, which of slot t's two score barriers the next QK commits to
    uint32_t kv_count = 0;
    FA_TRACE_DECL;

    // at D=64 K_j and V_j land on one barrier (see Cfg): waiting for K_j (the
    // unit's first QK, or QK(j) in the step before) also covers V_j for PV(j)
    auto kv_wait = [&](uint32_t idx) -> bool {
        if constexpr (C::kFullPairs) {
            const uint32_t q = idx / 2u, b = kBarKVFull + q % C::kPairs;
            return ptx::mbar_wait(wc, bars + kBarStride * b, (q / C::kPairs) & 1u, kSiteMma | b);
        } else {
            const uint32_t slot = idx % C::kSlots;
            return ptx::mbar_wait(wc, bars + kBarStride * (kBarKVFull + slot), (idx / C::kSlots) & 1u,
                                  kSiteMma | (kBarKVFull + slot));
        }
    };
    // V_j converted to fp16 (bf16 inputs): the tile the P*V MMAs read
    auto v_wait = [&](uint32_t idx) -> bool {
        if constexpr (converts_v<kBF16>()) {
            const uint32_t slot = idx % C::kSlots;
            return ptx::mbar_wait(wc, bars + kBarStride * (C::kBarVConv + slot), (idx / C::kSlots) & 1u,
                                  kSiteMma | (C::kBarVConv + slot));
        } else {
            return kv_wait(idx);
        }
    };
    // frees the pair of ring entries ending at `idx` (see Cfg): one commit
    auto kv_release = [&](uint32_t idx) { ptx::mma_commit(bars + kBarStride * (C::kBarKVEmpty + C::pair_of(idx) % C::kPairs), ex); };
    // S_t = Q_t K^T: M = 128 rows, N = 128 keys, K = D in steps of 16 (32 bytes
    // inside a 128-byte swizzled row; the next 64 columns sit in the next box).
    // Descriptors are built once per tile and stepped by adding the offset to
    // the start-address field of their low word: the issuing thread's
    // instructions per MMA are part of what keeps the tensor pipe fed
    // (measured: +4.5% against rebuilding each descriptor).
    constexpr uint32_t kDescHi = ptx::sdesc_hi_sw128(1024);
    auto issue_qk = [&](int t, uint32_t idx, uint32_t scol) {
        // key-parity units: one Q tile; slot t's key tile is the entry's t-th half
        const uint32_t qa = ptx::sdesc_lo(smem_base + C::kOffQ + (kKP ? 0 : t) * C::kTileBytes, 16);
        const uint32_t kb = ptx::sdesc_lo(
            smem_base + C::kOffKV + (idx % C::kSlots) * C::kSlotBytes + (kKP ? t * C::kTileBytes : 0), 16);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4;
            ptx::mma_ss(tmem + scol, ptx::sdesc_join(qa + off, kDescHi), ptx::sdesc_join(kb + off, kDescHi),
                        kIdescQK, kk > 0 ? 1u : 0u, ex);
        }
    };
    // O_t += P_t V: A = P from TMEM (16 keys = 8 columns per step), B = V tile
    // [128 keys x D], D contiguous: 8-key groups 1024 bytes apart, 64-column
    // boxes kBoxBytes apart.
    // One half: keys 64*half .. 64*half+63 (four K=16 steps).
    auto issue_pv = [&](int t, uint32_t idx, int half, bool acc, uint32_t pcol) {
        const uint32_t vb = smem_base + C::kOffKV + (idx % C::kSlots) * C::kSlotBytes + (kKP ? t * C::kTileBytes : 0);
        const uint32_t vl = ptx::sdesc_lo(vb, C::kBoxBytes);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
            const int kk = half * 4 + k4;
            ptx::mma_ts(tmem + C::col_o(t), tmem + pcol + kk * 8,
                        ptx::sdesc_join(vl + ((kk * 16 * 128) >> 4), kDescHi), kIdescPV, (acc || kk > 0) ? 1u : 0u, ex);
        }
    };

    if constexpr (C::kRot) {
        // Three score buffers: op m's QK writes buffer m % 3 and the QK of op
        // m + 3 follows the PV of op m (Cfg::kRot).  Per-slot state in bit
        // fields, since the slot of an op is a run-time value: qb / pb, 2 bits
        // per slot, the step barrier its next QK commits to / its next P wait
        // reads; pph, the phase bit of P barrier 3t + i at that bit; pvn, bit
        // t, which of slot t's two P*V-done barriers comes next.
        uint32_t qb = 0u, pb = 0u, pph = 0u, pvn = 0u;
        auto next3 = [](uint32_t f, int t) {
            const uint32_t i = (f >> (2 * t)) & 3u;
            return (f & ~(3u << (2 * t))) | ((i == 2u ? 0u : i + 1u) << (2 * t));
        };
        for (int r = 0;; ++r) {
            const Unit un = unit_at<kSplit, kKP>(r, p);
            if (un.status == kUnitDone) break;
            if (un.status == kUnitSkip) continue;
            const OpMap om(un);
            if (om.n == 0) continue;
            // K_j is entry kvb + 2(j - j0) of the ring, V_j the entry after it
            const uint32_t kvb = kv_count;
            FA_TRACE_EV(ex != 0u, kTrMma, kEvUnit, un.id);
            int k_in = un.j0 - 1;   // the last step whose K has been waited for
            // the QK of op m: slot t's step j into buffer m % 3
            auto qk_op = [&](int m) -> bool {
                const int t = om.slot(m), j = om.step(m);
                if (j == un.j0 && (!kKP || t == 0)) {
                    // key-parity units: both slots read slot 0's Q buffer
                    if (!ptx::mbar_wait(wc, bars + kBarStride * (kBarQFull + t), (ph_q >> t) & 1u, kSiteMma | (kBarQFull + t)))
                        return false;
                    ph_q ^= 1u << t;
                }
                const uint32_t ik = kvb + 2u * (uint32_t)(j - un.j0);
                if (j > k_in) {
                    if (!kv_wait(ik)) return false;
                    k_in = j;
                }
                ptx::tc_fence_after();
                FA_TRACE_EV(ex != 0u, kTrMma, kEvQKGo, ((uint32_t)t << 12) | j);
                issue_qk(t, ik, C::col_sb((uint32_t)m % 3u));
                const uint32_t b = kBarSFull + kStepBars * t + ((qb >> (2 * t)) & 3u);
                ptx::mma_commit(bars + kBarStride * b, ex);
                qb = next3(qb, t);
                FA_TRACE_EV(ex != 0u, kTrMma, kEvQK, ((uint32_t)t << 12) | j);
                // Q is free after its last QK: the unit's last op (key-parity
                // units), else slot t's last step
                if (kKP ? m == om.n - 1 : j == (t ? un.nkv[1] : un.nkv[0]) - 1)
                    ptx::mma_commit(bars + kBarStride * (kBarQEmpty + (kKP ? 0 : t)), ex);
                return true;
            };
            for (int m = 0; m < om.n && m < 3; ++m)
                if (!qk_op(m)) goto done;
            kv_release(kvb);
            for (int m = 0; m < om.n; ++m) {
                const int t = om.slot(m), j = om.step(m);
                const uint32_t bi = (uint32_t)(kStepBars * t) + ((pb >> (2 * t)) & 3u);
                const uint32_t pcol = C::col_sb((uint32_t)m % 3u);
                const uint32_t iv = kvb + 2u * (uint32_t)(j - un.j0) + 1u;
                FA_TRACE_EV(ex != 0u, kTrMma, kEvPWait, ((uint32_t)t << 12) | j);
                const uint32_t bp = kPVSplit ? kBarPHalf + bi : kBarPFull + bi;   // the first P wait
                if (!ptx::mbar_wait(wc, bars + kBarStride * bp, (pph >> bi) & 1u, kSiteMma | bp)) goto done;
                if (j == un.j0) {
                    // O_t is overwritten: the previous unit's epilogue must have read it
                    if (!ptx::mbar_wait(wc, bars + kBarStride * (kBarOEmpty + t), ((ph_oe >> t) & 1u) ^ 1u,
                                        kSiteMma | (kBarOEmpty + t)))
                        goto done;
                    ph_oe ^= 1u << t;
                }
                // V_j, before the step's first P*V (at D=64 with fp16 inputs
                // the wait for K_j covered it)
                if (!(C::kFullPairs && !converts_v<kBF16>()) && om.first_of_step(m) && !v_wait(iv)) goto done;
                ptx::tc_fence_after();
                FA_TRACE_EV(ex != 0u, kTrMma, kEvPVGo, ((uint32_t)t << 12) | j);
                issue_pv(t, iv, 0, j > un.j0, pcol);
                FA_TRACE_EV(ex != 0u, kTrMma, kEvPVMid, ((uint32_t)t << 12) | j);
                if constexpr (kPVSplit) {
                    if (!ptx::mbar_wait(wc, bars + kBarStride * (kBarPFull + bi), (pph >> bi) & 1u, kSiteMma | (kBarPFull + bi)))
                        goto done;
                    ptx::tc_fence_after();
                }
                pph ^= 1u << bi;
                pb = next3(pb, t);
                issue_pv(t, iv, 1, true, pcol);
                FA_TRACE_EV(ex != 0u, kTrMma, kEvPV, ((uint32_t)t << 12) | j);
                if (j == (t ? un.nkv[1] : un.nkv[0]) - 1) {
                    ptx::mma_commit(bars + kBarStride * (kBarOFull + t), ex);
                } else {
                    ptx::mma_commit(bars + kBarStride * (kBarPVDone + 2 * t + ((pvn >> t) & 1u)), ex);
                    pvn ^= 1u << t;
                }
                // V_j with K_{j+1}: every QK on K_{j+1} (ops up to m + 2) is issued
                if (om.last_of_step(m) && j + 1 < un.nmax) kv_release(iv + 1u);
                if (m + 3 < om.n && !qk_op(m + 3)) goto done;
            }
            kv_count = kvb + 2 * (un.nmax - un.j0);
        }
    } else for (int r = 0;; ++r) {
        const Unit un = unit_at<kSplit, kKP>(r, p);
        if (un.status == kUnitDone) break;
        if (un.status == kUnitSkip) continue;
        // K_j is entry kvb + 2(j - j0) of the ring, V_j the entry after it
        const uint32_t kvb = kv_count;
        FA_TRACE_EV(ex != 0u, kTrMma, kEvUnit, un.id);
        // the unit's first QKs, tile by tile: Q_1 frees only with the previous
        // unit's very last QK and lands last, so QK_0 (and tile 0's softmax)
        // need not wait for it
        bool k_in = false;
        // key-parity units read one Q buffer from both slots: it is released
        // by the slot whose QK on it comes last in issue order
        const int qe_slot = kKP ? (un.nkv[0] > un.nkv[1] ? 0 : 1) : 0;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            if (un.nkv[t] == 0) continue;
            if (!kKP || t == 0) {
                if (!ptx::mbar_wait(wc, bars + kBarStride * (kBarQFull + t), (ph_q >> t) & 1u, kSiteMma | (kBarQFull + t)))
                    goto done;
                ph_q ^= 1u << t;
            }
            if (!k_in) {
                if (!kv_wait(kvb)) goto done;
                k_in = true;
            }
            ptx::tc_fence_after();
            issue_qk(t, kvb, C::col_s(t));
            ptx::mma_commit(bars + kBarStride * (kBarSFull + kStepBars * t + ((sq >> t) & 1u)), ex);
            if constexpr (C::kLoaderOnScores) sq ^= 1u << t;
            FA_TRACE_EV(ex != 0u, kTrMma, kEvQK, (uint32_t)t << 12);
            if (un.nkv[t] == un.j0 + 1 && (!kKP || t == qe_slot))
                ptx::mma_commit(bars + kBarStride * (kBarQEmpty + (kKP ? 0 : t)), ex);
        }
        if constexpr (!C::kSoftmaxRelease && !C::kLoaderOnScores) kv_release(kvb);
        for (int j = un.j0; j < un.nmax; ++j) {
            const uint32_t iv = kvb + 2 * (j - un.j0) + 1, ik = iv + 1;
            bool v_ready = C::kFullPairs && !converts_v<kBF16>(), k_ready = false;
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                if (j < un.nkv[t]) {
                    FA_TRACE_EV(ex != 0u, kTrMma, kEvPWait, ((uint32_t)t << 12) | j);
                    // P_t (with FA_PV_SPLIT: its first half)
                    const uint32_t bp = (kPVSplit ? kBarPHalf : kBarPFull) + kStepBars * t;
                    if (!ptx::mbar_wait(wc, bars + kBarStride * bp, (ph_ph >> t) & 1u, kSiteMma | bp)) goto done;
                    ph_ph ^= 1u << t;
                    if (j == un.j0) {
                        // O_t is overwritten: the previous unit's epilogue must have read it
                        if (!ptx::mbar_wait(wc, bars + kBarStride * (kBarOEmpty + t), ((ph_oe >> t) & 1u) ^ 1u,
                                            kSiteMma | (kBarOEmpty + t)))
                            goto done;
                        ph_oe ^= 1u << t;
                    }
                    if (!v_ready) {
                        if (!v_wait(iv)) goto done;
                        v_ready = true;
                    }
                    ptx::tc_fence_after();
                    FA_TRACE_EV(ex != 0u, kTrMma, kEvPVGo, ((uint32_t)t << 12) | j);
                    issue_pv(t, iv, 0, j > un.j0, C::col_p(t));
                    FA_TRACE_EV(ex != 0u, kTrMma, kEvPVMid, ((uint32_t)t << 12) | j);
                    if constexpr (kPVSplit) {
                        if (!ptx::mbar_wait(wc, bars + kBarStride * (kBarPFull + kStepBars * t), (ph_p >> t) & 1u,
                                            kSiteMma | (kBarPFull + kStepBars * t)))
                            goto done;
                        ph_p ^= 1u << t;
                        ptx::tc_fence_after();
                    }
                    issue_pv(t, iv, 1, true, C::col_p(t));
                    FA_TRACE_EV(ex != 0u, kTrMma, kEvPV, ((uint32_t)t << 12) | j);
                    if (j == un.nkv[t] - 1) ptx::mma_commit(bars + kBarStride * (kBarOFull + t), ex);
                }
                if (j + 1 < un.nkv[t]) {
                    if (!k_ready) {
                        // (bf16 at D=128: covered by this step's wait for the converted V_j)
                        if constexpr (!conv_covers_k<D, kBF16, kKP>()) {
                            if (!kv_wait(ik)) goto done;
                            ptx::tc_fence_after();
                        }
                        k_ready = true;
                    }
                    FA_TRACE_EV(ex != 0u, kTrMma, kEvQKGo, ((uint32_t)t << 12) | (j + 1));
                    issue_qk(t, ik, C::col_s(t));
                    ptx::mma_commit(bars + kBarStride * (kBarSFull + kStepBars * t + ((sq >> t) & 1u)), ex);
                    if constexpr (C::kLoaderOnScores) sq ^= 1u << t;
                    FA_TRACE_EV(ex != 0u, kTrMma, kEvQK, ((uint32_t)t << 12) | (j + 1));
                    if (j + 1 == un.nkv[t] - 1 && (!kKP || t == qe_slot))
                        ptx::mma_commit(bars + kBarStride * (kBarQEmpty + (kKP ? 0 : t)), ex);
                }
            }
            // V_j and K_{j+1} together; a unit's last V goes with the next
            // unit's first K (released after that unit's first QKs)
            if (!C::kSoftmaxRelease && !C::kLoaderOnScores && j + 1 < un.nmax) kv_release(ik);
        }
        kv_count = kvb + 2 * (un.nmax - un.j0);
    }
done:
    // every MMA must be complete before tensor memory is released
    ptx::mma_commit(bars + kBarStride * kBarDrain, ex);
    ptx::mbar_wait_drain(wc, bars + kBarStride * kBarDrain, 0u, kSiteDrain | kBarDrain);
}

// ---------------------------------------------------------------------------------
template <int D, bool kBF16, bool kSplit, bool kKP>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  const __grid_constant__ Params p)
{
    using C = Cfg<D, kKP>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw);
    const uint32_t bars = base + C::kOffBars;
    float4* stats = reinterpret_cast<float4*>(smem + C::kOffStats);
    volatile uint32_t* ctl = reinterpret_cast<volatile uint32_t*>(smem + C::kOffCtl);
    const int warp = ptx::warp_id_uniform();
    const int lane = threadIdx.x & 31;
    FA_TRACE_DECL;
    FA_TRACE_EV(threadIdx.x == 0, kTrKernel, kEvEntry, 0);
    // The next kernel in the stream (the split-KV merge, or the next pass) may
    // be scheduled now: it waits for this grid to complete before it touches
    // global memory, and meanwhile sets itself up on SMs this grid leaves.
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            ptx::mbar_init(bars + kBarStride * (kBarQFull + t), 1);
            ptx::mbar_init(bars + kBarStride * (kBarQEmpty + t), 1);
            for (int i = 0; i < kStepBars; ++i) {
                ptx::mbar_init(bars + kBarStride * (kBarSFull + kStepBars * t + i), 1);
                ptx::mbar_init(bars + kBarStride * (kBarPHalf + kStepBars * t + i), 4);
                ptx::mbar_init(bars + kBarStride * (kBarPFull + kStepBars * t + i), 4);
            }
            ptx::mbar_init(bars + kBarStride * (kBarPVDone + 2 * t), 1);
            ptx::mbar_init(bars + kBarStride * (kBarPVDone + 2 * t + 1), 1);
            ptx::mbar_init(bars + kBarStride * (kBarOFull + t), 1);
            ptx::mbar_init(bars + kBarStride * (kBarOEmpty + t), 4);
            ptx::mbar_init(bars + kBarStride * (kBarStFull + t), 4);
            ptx::mbar_init(bars + kBarStride * (kBarStEmpty + t), 4);
        }
        ptx::mbar_init(bars + kBarStride * kBarDrain, 1);
        for (int s = 0; s < C::kSlots; ++s) {
            ptx::mbar_init(bars + kBarStride * (kBarKVFull + s), C::kFullPairs ? 2 : 1);   // (K_j's and V_j's copies)
            ptx::mbar_init(bars + kBarStride * (C::kBarKVEmpty + s), 1);
            ptx::mbar_init(bars + kBarStride * (C::kBarVConv + s), conv_warps<kBF16, kSplit, kKP>() > 0 ? conv_warps<kBF16, kSplit, kKP>() : 1);
        }
        ctl[1] = 0u;
        ptx::fence_mbar_init();
    }
    if (warp == 12 && lane == 0) {
        ptx::prefetch_tmap(&tm_q);
        ptx::prefetch_tmap(&tm_k);
        ptx::prefetch_tmap(&tm_v);
        ptx::prefetch_tmap(&tm_o);
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
    // Launched as a programmatic dependent: the setup above (shared and tensor
    // memory only) overlapped the previous grid's tail; every global access
    // (inputs it may have written, outputs and workspace it may still read)
    // comes after that grid has completed and its writes are visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    FA_TRACE_EV(threadIdx.x == 0, kTrKernel, kEvSetup, 0);

    if (warp < 8) {
        ptx::setmaxnreg_inc<RegSplit<D, kBF16, kSplit, kKP>::kSoftmax>();
        softmax_role<D, kBF16, kSplit, kKP>(p, wc, warp >> 2, tmem, bars, stats);
    } else if (warp < 12) {
        ptx::setmaxnreg_dec<RegSplit<D, kBF16, kSplit, kKP>::kEpilogue>();
        if constexpr (conv_warps<kBF16, kSplit, kKP>() == 6)
            vconvert_role<D, kSplit, kKP, 6>(p, wc, base, bars, threadIdx.x - 8 * 32);
        else
            correction_epilogue_role<D, kBF16, kSplit, kKP>(p, wc, &tm_o, tmem, base, bars, stats, ctl + 2);
    } else {
        ptx::setmaxnreg_dec<RegSplit<D, kBF16, kSplit, kKP>::kControl>();
        // the loader and the MMA issuer run on all 32 lanes of their warp (one
        // lane issues), so neither warp diverges while it waits
        if (warp == 12) {
            load_role<D, kSplit, kKP>(p, wc, &tm_q, &tm_k, &tm_v, base, bars);
        } else if (warp == 13) {
            mma_role<D, kBF16, kSplit, kKP>(p, wc, tmem, base, bars);
        } else if constexpr (conv_warps<kBF16, kSplit, kKP>() == 6) {
            vconvert_role<D, kSplit, kKP, 6>(p, wc, base, bars, 128 + threadIdx.x - 14 * 32);
        } else if constexpr (conv_warps<kBF16, kSplit, kKP>() == 2) {
            vconvert_role<D, kSplit, kKP, 2>(p, wc, base, bars, threadIdx.x - 14 * 32);
        }
        __syncwarp();
    }

    ptx::tc_fence_before();
    __syncthreads();
    FA_TRACE_EV(threadIdx.x == 0, kTrKernel, kEvExit, 0);
    if (warp == 13) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

template <int D, bool kBF16, bool kSplit, bool kKP = false>
int launch_instance(const LaunchArgs& a, cudaStream_t stream)
{
    auto kern = fa_fwd_kernel<D, kBF16, kSplit, kKP>;
    // the shared-memory opt-in is a per-device property of the kernel: set it
    // on the first launch on each device only (it costs a driver call)
    cudaError_t e = cudaSuccess;
    if (!smem_opt_in_done(reinterpret_cast<const void*>(kern), a.device)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D, kKP>::kSmemBytes);
        if (e != cudaSuccess) return (int)e;
        smem_opt_in_mark(reinterpret_cast<const void*>(kern), a.device);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg<D, kKP>::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, a.tm_q, a.tm_k, a.tm_v, a.tm_o, a.p);
    return (int)e;
}

}  // namespace fa
