// Host side of the C ABI declared in include/fa_fwd.h: argument checks, TMA
// tensor maps, launch geometry and the work-unit schedule, dispatch to the
// kernel instances.  Nothing here allocates device memory.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <mutex>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "fa_fwd.h"
#include "fa_fwd_common.h"
#include "fa_fwd_kernel.cuh"

namespace {

using fa::kBM;

// Device status word: a bounded wait that gives up stores its site here.
__device__ unsigned int g_fa_status = 0u;

#ifdef FA_TRACE
// Trace buffer of the FA_TRACE build, set with fa_trace_set.
unsigned long long* g_trace = nullptr;
int g_trace_ctas = 0, g_trace_cap = 0;
#endif
#ifdef FA_DEBUG_STATS
// Side buffers of the FA_DEBUG_STATS build, set with fa_debug_stats_set.
float* g_dbg_rows = nullptr;
unsigned long long* g_dbg_count = nullptr;
#endif

constexpr int kMaxDevices = 64;

// Kernel layout of one-pass launches (fa_fwd_set_layout): 0 = automatic.
std::atomic<int> g_layout{0};
constexpr int kLayoutAuto = 0, kLayoutTwoTile = 1, kLayoutOneTile = 2;

// The layout a one-pass launch of head dim D uses.
int resolve_layout(int /*D*/)
{
    const int l = g_layout.load(std::memory_order_relaxed);
    return l == kLayoutAuto ? kLayoutTwoTile : l;
}
std::atomic<int> g_num_sms[kMaxDevices];     // 0 = not queried yet
std::atomic<int> g_cc[kMaxDevices];          // major*10 + minor, 0 = not queried yet
std::atomic<void*> g_status_addr[kMaxDevices];   // device address of g_fa_status, nullptr = not looked up

unsigned long long timeout_ns()
{
    static const unsigned long long ns = [] {
        const char* e = std::getenv("FA_WAIT_TIMEOUT_MS");
        long long ms = e ? std::atoll(e) : 0;
        if (ms <= 0) ms = 4000;
        return (unsigned long long)ms * 1000000ull;
    }();
    return ns;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// SM count and compute capability of the current device (cached per device).
int device_props(int* num_sms, int* cc)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
    int n = g_num_sms[dev].load(std::memory_order_relaxed);
    int c = g_cc[dev].load(std::memory_order_relaxed);
    if (n == 0 || c == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return FA_ERR_CUDA;
        c = major * 10 + minor;
        g_num_sms[dev].store(n, std::memory_order_relaxed);
        g_cc[dev].store(c, std::memory_order_relaxed);
    }
    *num_sms = n;
    *cc = c;
    return FA_OK;
}

int check_args(int B, int H, int S, int D, int causal, int dtype)
{
    if (B < 1 || H < 1 || S < 1) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    // every tensor stays below 2^31 elements (the header's size limit)
    const long long rows = (long long)B * H * S;
    if (rows * (long long)(D > 0 ? D : 1) >= (1ll << 31)) return FA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
    if (dtype != FA_DTYPE_F16 && dtype != FA_DTYPE_BF16) return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---- causal schedule planner ------------------------------------------------
// The kernel walks a list of work units ordered group by group (`head_group`
// heads per group), longest first inside a group, CTA c taking entries in snake
// order (see unit_at / decode_unit in fa_fwd_kernel.cuh).  Larger groups balance
// the causal triangle better; smaller groups keep the K/V of the heads in flight
// within L2.  The planner replays the assignment for the group sizes whose K/V
// fits the budget (group_candidates) and keeps the best-balanced one (the
// smallest such group within 0.5% of the best).  Results are cached per shape.

constexpr long long kGroupKVBudget = 160ll << 20;   // bytes of K/V per group of heads

// Load of the most loaded CTA over the mean, with the cost of a unit taken as
// its key tiles plus a fixed per-unit overhead of two tiles.
double snake_imbalance(int BH, int n_qtiles, int tpu, int n_qgroups, long long units, int grid, int hg,
                       std::vector<double>& load)
{
    load.assign((size_t)grid, 0.0);
    const long long per_group = (long long)hg * n_qgroups;
    double total = 0.0;
    for (long long u = 0; u < units; ++u) {
        const long long r = u / grid, pos = u % grid;
        const long long c = (r & 1) ? (grid - 1 - pos) : pos;
        const long long g = u / per_group, w = u - g * per_group;
        const long long h0 = g * hg;
        const long long hgg = hg < BH - h0 ? hg : BH - h0;
        const long long rank = w / hgg;
        const long long qg = n_qgroups - 1 - rank;
        double cost = 2.0;
        for (int t = 0; t < tpu; ++t) {
            const long long qt = qg * tpu + t;
            if (qt < n_qtiles) cost += (double)(qt + 1);
        }
        load[(size_t)c] += cost;
        total += cost;
    }
    double mx = 0.0;
    for (double x : load) mx = x > mx ? x : mx;
    return mx / (total / grid);
}

// Head-group sizes the planners replay: every size up to 32 (where the
// balance moves most from one size to the next; the sizes picked for the
// measured shapes are 4 to 26), then sizes about 12% apart up to `cap`.
// Replaying every size up to the budget took seconds for launches of many
// short heads (65536 heads of 128 keys: 5120 sizes x 65536 units).
std::vector<int> group_candidates(long long cap)
{
    std::vector<int> c;
    for (long long hg = 1; hg <= cap && hg <= 32; ++hg) c.push_back((int)hg);
    for (long long hg = 36; hg < cap; hg = hg + hg / 8) c.push_back((int)hg);
    if (cap > 32) c.push_back((int)cap);
    return c;
}

int plan_head_group(int BH, int S, int D, int n_qtiles, int tpu, int n_qgroups, long long units, int grid)
{
    struct Entry { int BH, S, D, grid, hg; };
    static std::mutex mu;
    static std::vector<Entry> cache;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (const Entry& e : cache)
            if (e.BH == BH && e.S == S && e.D == D && e.grid == grid) return e.hg;
    }
    const long long kv_head_bytes = 2ll * S * D * 2;
    long long cap = kGroupKVBudget / kv_head_bytes;
    if (cap < 1) cap = 1;
    if (cap > BH) cap = BH;
    int pick = 1;   // one query group per head: every unit costs the same
    if (n_qgroups > 1) {
        const std::vector<int> cand = group_candidates(cap);
        std::vector<double> load, score(cand.size());
        double best = 1e30;
        for (size_t i = 0; i < cand.size(); ++i) {
            score[i] = snake_imbalance(BH, n_qtiles, tpu, n_qgroups, units, grid, cand[i], load);
            best = std::min(best, score[i]);
        }
        for (size_t i = 0; i < cand.size(); ++i)
            if (score[i] <= best + 0.005) {
                pick = cand[i];
                break;
            }
    }
    std::lock_guard<std::mutex> lock(mu);
    if (cache.size() >= 256) cache.erase(cache.begin());
    cache.push_back({BH, S, D, grid, pick});
    return pick;
}

// ---- table schedule ----------------------------------------------------------
// For causal launches of several rounds that fit the table, the host computes a
// list schedule instead of a closed form: the units, ordered group by group
// (head_group heads at a time, so the heads in flight share L2) and longest
// first inside a group, go one at a time to the CTA with the least modelled work
// so far (a unit costs its key tiles plus two for its fixed part).  That is
// longest-processing-time list scheduling per group.  Its balance moves with the
// group size, so the planner replays it for the group sizes whose K/V fits
// kTableKVBudget (group_candidates) and keeps the smallest within 0.5% of the
// best.  It
// balances the causal triangle where mirror pairs leave rounds half-empty and a
// snake needs all heads in one group (modelled, most loaded CTA over the mean:
// 4x32x4096 1.04 pairs, 1.008 here with 8-head groups; 8x16x2048 1.19 pairs,
// 1.026 here).  Tables are cached per shape; each launch carries its copy in the
// kernel parameters.
constexpr long long kTableKVBudget = 64ll << 20;   // bytes of K/V per group of heads

struct SchedTable {
    int BH, S, D, tpu, causal, grid, hg;
    std::vector<unsigned short> off, unit;
};

// Assigns the units (heads in groups of hg) to `grid` CTAs; returns the most
// loaded CTA's modelled work over the mean, and the per-CTA lists if `per`.
double list_schedule(int BH, int n_qtiles, int tpu, int causal, int grid, int hg,
                     std::vector<std::vector<unsigned short>>* per)
{
    const int n_qgroups = (n_qtiles + tpu - 1) / tpu;
    auto cost = [&](int qg) {
        int last = qg * tpu + tpu - 1;
        if (last > n_qtiles - 1) last = n_qtiles - 1;
        return (double)fa::kv_tiles_of(last, n_qtiles, causal) + 2.0;
    };
    if (per) per->assign((size_t)grid, {});
    // min-heap of (load, cta), ties to the lower CTA
    std::vector<std::pair<double, int>> heap;
    heap.reserve((size_t)grid);
    for (int c = 0; c < grid; ++c) heap.push_back({0.0, c});
    auto later = [](const std::pair<double, int>& a, const std::pair<double, int>& b) {
        return a.first > b.first || (a.first == b.first && a.second > b.second);
    };
    std::make_heap(heap.begin(), heap.end(), later);
    double total = 0.0;
    for (int h0 = 0; h0 < BH; h0 += hg) {
        const int h1 = std::min(BH, h0 + hg);
        for (int rank = 0; rank < n_qgroups; ++rank) {
            const int qg = causal ? n_qgroups - 1 - rank : rank;
            const double w = cost(qg);
            for (int h = h0; h < h1; ++h) {
                std::pop_heap(heap.begin(), heap.end(), later);
                if (per) (*per)[(size_t)heap.back().second].push_back((unsigned short)(h * n_qgroups + qg));
                heap.back().first += w;
                total += w;
                std::push_heap(heap.begin(), heap.end(), later);
            }
        }
    }
    double mx = 0.0;
    for (const auto& e : heap) mx = std::max(mx, e.first);
    return mx / (total / grid);
}

bool table_applies(int causal, long long units, int grid)
{
    return causal && units > grid && units <= fa::kSchedTableMaxUnits && grid <= fa::kSchedTableMaxCtas;
}

// The table for this shape (built and cached on first use); copies it into *p
// when p is not null and returns its head group.
int table_plan(int BH, int S, int D, int n_qtiles, int tpu, int causal, int grid, fa::Params* p)
{
    static std::mutex mu;
    static std::vector<SchedTable> cache;   // recent shapes
    std::lock_guard<std::mutex> lock(mu);
    const SchedTable* t = nullptr;
    for (const SchedTable& e : cache)
        if (e.BH == BH && e.S == S && e.D == D && e.tpu == tpu && e.causal == causal && e.grid == grid) {
            t = &e;
            break;
        }
    if (!t) {
        const long long kv_head_bytes = 2ll * S * D * 2;
        long long cap = kTableKVBudget / kv_head_bytes;
        cap = std::max(1ll, std::min(cap, (long long)BH));
        const int n_qgroups = (n_qtiles + tpu - 1) / tpu;
        int pick = 1;   // one query group per head: every unit costs the same
        if (n_qgroups > 1) {
            const std::vector<int> cand = group_candidates(cap);
            std::vector<double> score(cand.size());
            double best = 1e30;
            for (size_t i = 0; i < cand.size(); ++i) {
                score[i] = list_schedule(BH, n_qtiles, tpu, causal, grid, cand[i], nullptr);
                best = std::min(best, score[i]);
            }
            for (size_t i = 0; i < cand.size(); ++i)
                if (score[i] <= best + 0.005) {
                    pick = cand[i];
                    break;
                }
        }
        SchedTable n{BH, S, D, tpu, causal, grid, pick, {}, {}};
        std::vector<std::vector<unsigned short>> per;
        list_schedule(BH, n_qtiles, tpu, causal, grid, pick, &per);
        n.off.assign((size_t)grid + 1, 0);
        for (int c = 0; c < grid; ++c) {
            n.off[(size_t)c] = (unsigned short)n.unit.size();
            n.unit.insert(n.unit.end(), per[(size_t)c].begin(), per[(size_t)c].end());
        }
        n.off[(size_t)grid] = (unsigned short)n.unit.size();
        if (cache.size() >= 16) cache.erase(cache.begin());
        cache.push_back(std::move(n));
        t = &cache.back();
    }
    if (p) {
        std::copy(t->off.begin(), t->off.end(), p->tab_off);
        std::copy(t->unit.begin(), t->unit.end(), p->tab_unit);
    }
    return t->hg;
}

// Work-unit geometry (see the schedule comment in fa_fwd_kernel.cuh).  The
// one-tile layout (fa_fwd_wide.cuh) always takes one query tile per unit.
void plan(int B, int H, int S, int D, int causal, int num_sms, fa_launch_info_t* info, fa::Params* p,
          int layout)
{
    const int BH = B * H;
    const int n_qtiles = (S + kBM - 1) / kBM;
    const bool one_tile = layout == kLayoutOneTile;
    // two query tiles per unit (ping-pong softmax) once there is enough work for
    // two units per SM; otherwise one, so small problems still fill the GPU
    const int tpu = (!one_tile && (long long)BH * n_qtiles >= 2ll * num_sms) ? 2 : 1;
    const int n_qgroups = (n_qtiles + tpu - 1) / tpu;
    const long long units = (long long)BH * n_qgroups;
    const int grid = (int)(units < num_sms ? units : num_sms);
    // Causal units differ in cost.  The snake over head groups balances best
    // (the planner replays it), but each of its rounds holds about
    // grid / head_group units of a head; with fewer than four, CTAs rarely share
    // a head's K/V in L2 and the re-reads go to DRAM (4x32x4096x128 bf16: 1.1 GB
    // per launch against 0.4 GB, and under a one-second loop the GPU hits its
    // power cap).  Then the mirror-pair schedule is used instead: slightly worse
    // balance, but a CTA's two units share one head and a round covers few heads.
    // With a single round every CTA takes one unit.  Without the mask every unit
    // costs the same and heads simply go in order.  Causal launches of several
    // rounds that fit the parameter table take the host's list schedule instead
    // (see table_plan), which gets both balance and locality.
    int head_group = 1;
    bool pairs = false;
    const bool table = table_applies(causal, units, grid);
    if (table) {
        head_group = table_plan(BH, S, D, n_qtiles, tpu, causal, grid, p);
    } else if (causal && units > grid) {
        head_group = plan_head_group(BH, S, D, n_qtiles, tpu, n_qgroups, units, grid);
        pairs = grid < 4 * head_group;
    } else if (causal) {
        head_group = plan_head_group(BH, S, D, n_qtiles, tpu, n_qgroups, units, grid);
    }
    const int pairs_per_head = (n_qgroups + 1) / 2;
    if (info) {
        info->grid = grid;
        info->block = fa::kThreads;
        info->smem_bytes = one_tile ? fa::wide_smem_bytes_for(D) : fa::smem_bytes_for(D);
        info->tiles_per_unit = tpu;
        info->units = (int)units;
        info->head_group = head_group;
        info->num_sms = num_sms;
        info->schedule = table ? 2 : (pairs ? 1 : 0);
        info->layout = one_tile ? kLayoutOneTile : kLayoutTwoTile;
        info->key_step = one_tile ? fa::kWideBN : fa::kBN;
    }
    if (p) {
        p->BH = BH;
        p->S = S;
        p->n_qtiles = n_qtiles;
        p->n_kv = n_qtiles;
        p->tpu = tpu;
        p->n_qgroups = n_qgroups;
        p->n_units = (int)units;
        p->sched = table ? fa::kSchedTable : (pairs ? fa::kSchedPairs : fa::kSchedSnake);
        p->head_group = head_group;
        p->pairs_per_head = pairs_per_head;
        p->n_pairs = (long long)BH * pairs_per_head;
        p->causal = causal;
        p->mask_last = (causal || (S % fa::kBN) != 0) ? 1 : 0;
        p->split_chunk = 0;
        p->units_per_head = 0;
        p->ws_o = nullptr;
        p->ws_lse = nullptr;
    }
}

// ---- split-KV planner ---------------------------------------------------------
// When one pass has fewer work units than SMs (few heads, short rows), the key
// range of every query group is cut into chunks of `chunk` key tiles, each a
// unit of its own; the largest chunk that still gives every SM a unit is used.
// Returns false when one pass already fills the GPU or no split would help.
struct SplitPlan {
    int chunk, tpu, n_qtiles, n_qgroups, units_per_head;
    long long units;
};

// Cost model of the split planner, in SM cycles measured on GB300 for this
// kernel: one key step of a one-tile unit (softmax, PV and QK strictly in
// series), one key step of a two-tile unit (the tiles interleave), the fixed
// part of a unit (Q and first K/V loads, epilogue with the partial's write),
// and the merge: a fixed part (the second launch, its wait for the attention
// grid, three dependent L2 round trips; fitted to measured split times) plus
// its partial bytes read.  Small problems whose one pass is short (the
// batch-1, 16-head, 1024-token case: 17 us) stay one pass.
constexpr double kStep1 = 3450.0, kStep2 = 3900.0, kUnitFixed = 5800.0;
constexpr double kMergeFixed = 20000.0, kMergeBytesPerCycle = 1500.0;

// Split only problems that leave SMs idle, and only when the estimated
// makespan of the best (tiles per unit, chunk) beats one pass by 10%.
bool plan_split_search(int BH, int S, int causal, int num_sms, SplitPlan* sp)
{
    const int n_qtiles = (S + kBM - 1) / kBM;
    const int tpu1 = ((long long)BH * n_qtiles >= 2ll * num_sms) ? 2 : 1;
    const int ng1 = (n_qtiles + tpu1 - 1) / tpu1;
    const long long units1 = (long long)BH * ng1;
    if (units1 >= num_sms) return false;
    // one pass: one unit per CTA; the longest unit sets the time
    const double step1 = tpu1 == 2 ? kStep2 : kStep1;
    const double one_pass = fa::kv_tiles_of(n_qtiles - 1, n_qtiles, causal) * step1 + kUnitFixed;
    double best = one_pass;
    bool found = false;
    for (int tpu = 1; tpu <= (n_qtiles >= 2 ? 2 : 1); ++tpu) {
        const int n_qgroups = (n_qtiles + tpu - 1) / tpu;
        for (int c = 1; c < n_qtiles; ++c) {
            int uph = 0;
            for (int g = 0; g < n_qgroups; ++g) uph += fa::split_chunks(g, tpu, n_qtiles, n_qtiles, causal, c);
            const long long units = (long long)BH * uph;
            const long long rounds = (units + num_sms - 1) / num_sms;
            const double merge_bytes = (double)units * tpu * kBM * 64 * sizeof(float);   // per 64 columns of D
            const double cost = rounds * (c * (tpu == 2 ? kStep2 : kStep1) + kUnitFixed) + kMergeFixed +
                                merge_bytes / kMergeBytesPerCycle;
            if (cost < best && units < (1ll << 30)) {
                best = cost;
                found = true;
                sp->chunk = c;
                sp->tpu = tpu;
                sp->n_qtiles = n_qtiles;
                sp->n_qgroups = n_qgroups;
                sp->units_per_head = uph;
                sp->units = units;
            }
        }
    }
    return found && best < 0.9 * one_pass;
}

// The search walks every (tiles per unit, chunk) over every query group, which
// is O(n_qtiles^2): tens of microseconds of host time for long rows, more than
// the kernels of a small problem take.  Callers repeat shapes (the workspace
// query, then the call; every step of a loop), so recent answers are kept.
struct SplitMemo {
    int BH, S, causal, num_sms;
    bool found;
    SplitPlan sp;
};
constexpr int kSplitMemo = 16;
std::mutex g_split_mu;
SplitMemo g_split_memo[kSplitMemo];
int g_split_n = 0, g_split_next = 0;

bool plan_split(int BH, int S, int causal, int num_sms, SplitPlan* sp)
{
    {
        std::lock_guard<std::mutex> lk(g_split_mu);
        for (int i = 0; i < g_split_n; ++i) {
            const SplitMemo& m = g_split_memo[i];
            if (m.BH == BH && m.S == S && m.causal == causal && m.num_sms == num_sms) {
                if (m.found) *sp = m.sp;
                return m.found;
            }
        }
    }
    SplitMemo m{BH, S, causal, num_sms, false, SplitPlan{}};
    m.found = plan_split_search(BH, S, causal, num_sms, &m.sp);
    {
        std::lock_guard<std::mutex> lk(g_split_mu);
        g_split_memo[g_split_next] = m;
        g_split_next = (g_split_next + 1) % kSplitMemo;
        if (g_split_n < kSplitMemo) ++g_split_n;
    }
    if (m.found) *sp = m.sp;
    return m.found;
}

// partial O then partial LSE of every (unit, tile, row)
size_t split_workspace_bytes(const SplitPlan& sp, int D)
{
    return (size_t)sp.units * sp.tpu * kBM * (size_t)(D + 1) * sizeof(float);
}

// [B*H, S, D] 16-bit tensor, `rows`-row x 64-column boxes, 128-byte swizzle.
int make_tmap(CUtensorMap* m, const void* ptr, int BH, int S, int D, int dtype, int rows = kBM)
{
    auto fn = encode_fn();
    if (!fn) return FA_ERR_CUDA;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)BH};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)S * D * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(m, dtype == FA_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                          3, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

namespace fa {
int smem_bytes_for(int D) { return D == 64 ? Cfg<64>::kSmemBytes : Cfg<128>::kSmemBytes; }

namespace {
// (kernel, devices with the opt-in set) for the few kernel instances there are
constexpr int kOptInSlots = 32;
std::mutex g_opt_in_mu;
const void* g_opt_in_kern[kOptInSlots];
unsigned long long g_opt_in_devs[kOptInSlots];
int g_opt_in_n = 0;
}  // namespace

bool smem_opt_in_done(const void* kern, int device)
{
    std::lock_guard<std::mutex> lk(g_opt_in_mu);
    for (int i = 0; i < g_opt_in_n; ++i)
        if (g_opt_in_kern[i] == kern) return (g_opt_in_devs[i] >> (device & 63)) & 1ull;
    return false;
}

void smem_opt_in_mark(const void* kern, int device)
{
    std::lock_guard<std::mutex> lk(g_opt_in_mu);
    for (int i = 0; i < g_opt_in_n; ++i)
        if (g_opt_in_kern[i] == kern) {
            g_opt_in_devs[i] |= 1ull << (device & 63);
            return;
        }
    if (g_opt_in_n < kOptInSlots) {   // a full table only means the opt-in is set again on every launch
        g_opt_in_kern[g_opt_in_n] = kern;
        g_opt_in_devs[g_opt_in_n] = 1ull << (device & 63);
        ++g_opt_in_n;
    }
}
}  // namespace fa

extern "C" {

const char* fa_strerror(int status)
{
    switch (status) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported head dim, dtype or device (needs D in {64,128}, fp16/bf16, sm_103)";
    case FA_ERR_MISALIGNED: return "tensor pointer not 16-byte aligned";
    case FA_ERR_CUDA: return "CUDA runtime/driver error";
    case FA_ERR_TIMEOUT: return "a bounded in-kernel wait timed out";
    case FA_ERR_SCRATCH: return "problem needs more split-KV scratch than the library's static array holds";
    case FA_ERR_RANGE: return "bf16 input V holds a value beyond fp16's range (+-65504): results invalid";
    default: return "unknown status";
    }
}

int fa_fwd_launch_info(int B, int H, int S, int D, int causal, int dtype, fa_launch_info_t* info)
{
    if (!info) return FA_ERR_INVALID_ARG;
    int rc = check_args(B, H, S, D, causal, dtype);
    if (rc != FA_OK) return rc;
    int num_sms = 0, cc = 0;
    rc = device_props(&num_sms, &cc);
    if (rc != FA_OK) return rc;
    plan(B, H, S, D, causal, num_sms, info, nullptr, resolve_layout(D));
    return FA_OK;
}

int fa_fwd_plan(int B, int H, int S, int D, int causal, int dtype, int num_sms, fa_launch_info_t* info)
{
    if (!info || num_sms < 1) return FA_ERR_INVALID_ARG;
    const int rc = check_args(B, H, S, D, causal, dtype);
    if (rc != FA_OK) return rc;
    plan(B, H, S, D, causal, num_sms, info, nullptr, resolve_layout(D));
    return FA_OK;
}

int fa_fwd_set_layout(int layout)
{
    if (layout < kLayoutAuto || layout > kLayoutOneTile) return -1;
    return g_layout.exchange(layout);
}

int fa_fwd_schedule_table(int B, int H, int S, int D, int causal, int dtype, int num_sms, unsigned short* offsets,
                          int offsets_cap, unsigned short* units, int units_cap, int* n_ctas, int* n_units)
{
    if (!offsets || !units || !n_ctas || !n_units || num_sms < 1 || offsets_cap < 0 || units_cap < 0)
        return FA_ERR_INVALID_ARG;
    const int rc = check_args(B, H, S, D, causal, dtype);
    if (rc != FA_OK) return rc;
    std::vector<fa::Params> hold(1);   // the table makes Params large: keep it off the stack
    fa::Params* p = hold.data();
    fa_launch_info_t info;
    plan(B, H, S, D, causal, num_sms, &info, p, resolve_layout(D));
    if (p->sched != fa::kSchedTable) return FA_ERR_UNSUPPORTED;
    const int nu = (int)p->tab_off[info.grid];
    if (offsets_cap < info.grid + 1 || units_cap < nu) return FA_ERR_INVALID_ARG;
    std::copy(p->tab_off, p->tab_off + info.grid + 1, offsets);
    std::copy(p->tab_unit, p->tab_unit + nu, units);
    *n_ctas = info.grid;
    *n_units = nu;
    return FA_OK;
}

}  // extern "C"

namespace {

// Common checks of the forward entry points; fills the SM count.
int check_call(const void* q, const void* k, const void* v, const void* o, const float* lse, int B, int H, int S,
               int D, int causal, float scale, int dtype, int* num_sms)
{
    if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
    if (!(scale > 0.0f) || !std::isfinite(scale)) return FA_ERR_INVALID_ARG;
    int rc = check_args(B, H, S, D, causal, dtype);
    if (rc != FA_OK) return rc;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return FA_ERR_MISALIGNED;
    int cc = 0;
    rc = device_props(num_sms, &cc);
    if (rc != FA_OK) return rc;
    if (cc != 103) return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

// One attention launch (and, with a split plan, the merge launch after it).
int run_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int S, int D, int causal,
            float scale, int dtype, int num_sms, const SplitPlan* sp, float* ws, cudaStream_t s)
{
    fa::LaunchArgs a;
    fa_launch_info_t info;
    const int layout = sp ? kLayoutTwoTile : resolve_layout(D);
    plan(B, H, S, D, causal, num_sms, &info, &a.p, layout);
    a.grid = info.grid;
    if (cudaGetDevice(&a.device) != cudaSuccess || a.device < 0 || a.device >= kMaxDevices) return FA_ERR_CUDA;
    const int BH = B * H;
    if (sp) {
        a.p.tpu = sp->tpu;
        a.p.n_qgroups = sp->n_qgroups;
        a.p.n_units = (int)sp->units;
        a.p.split_chunk = sp->chunk;
        a.p.units_per_head = sp->units_per_head;
        a.p.sched = fa::kSchedSnake;
        a.p.ws_o = ws;
        a.p.ws_lse = ws + (size_t)sp->units * sp->tpu * kBM * D;
        a.grid = (int)(sp->units < num_sms ? sp->units : num_sms);
    }
    a.p.lse = lse;
    a.p.o = o;
    a.p.scale_log2 = (float)((double)scale * 1.4426950408889634);
    a.p.timeout_ns = timeout_ns();
    a.p.trace = nullptr;
    a.p.trace_ctas = 0;
    a.p.trace_cap = 0;
    a.p.dbg_rows = nullptr;
    a.p.dbg_count = nullptr;
#ifdef FA_DEBUG_STATS
    a.p.dbg_rows = g_dbg_rows;
    a.p.dbg_count = g_dbg_count;
#endif
#ifdef FA_TRACE
    a.p.trace = g_trace;
    a.p.trace_ctas = g_trace_ctas;
    a.p.trace_cap = g_trace_cap;
#endif
    void* status = g_status_addr[a.device].load(std::memory_order_acquire);
    if (!status) {
        if (cudaGetSymbolAddress(&status, g_fa_status) != cudaSuccess) return FA_ERR_CUDA;
        g_status_addr[a.device].store(status, std::memory_order_release);
    }
    a.p.status = static_cast<unsigned int*>(status);
    int e;
    if (layout == kLayoutOneTile) {
        const int kv_rows = fa::kWideBN;
        if (make_tmap(&a.tm_q, q, BH, S, D, dtype) != FA_OK ||
            make_tmap(&a.tm_k, k, BH, S, D, dtype, kv_rows) != FA_OK ||
            make_tmap(&a.tm_v, v, BH, S, D, dtype, kv_rows) != FA_OK)
            return FA_ERR_CUDA;
        if (D == 64)
            e = dtype == FA_DTYPE_BF16 ? fa::launch_wide_d64_bf16(a, s) : fa::launch_wide_d64_f16(a, s);
        else
            e = dtype == FA_DTYPE_BF16 ? fa::launch_wide_d128_bf16(a, s) : fa::launch_wide_d128_f16(a, s);
        return e == (int)cudaSuccess ? FA_OK : FA_ERR_CUDA;
    }
    // key-parity units (D=64, one query tile per unit) load a step's two key
    // tiles with one 256-row copy
    const int kv_rows = (D == 64 && a.p.tpu == 1) ? 2 * kBM : kBM;
    if (make_tmap(&a.tm_q, q, BH, S, D, dtype) != FA_OK || make_tmap(&a.tm_k, k, BH, S, D, dtype, kv_rows) != FA_OK ||
        make_tmap(&a.tm_v, v, BH, S, D, dtype, kv_rows) != FA_OK || make_tmap(&a.tm_o, o, BH, S, D, dtype) != FA_OK)
        return FA_ERR_CUDA;

    if (D == 64)
        e = dtype == FA_DTYPE_BF16 ? fa::launch_d64_bf16(a, s) : fa::launch_d64_f16(a, s);
    else
        e = dtype == FA_DTYPE_BF16 ? fa::launch_d128_bf16(a, s) : fa::launch_d128_f16(a, s);
    if (e != (int)cudaSuccess) return FA_ERR_CUDA;
    if (sp) {
        fa::MergeArgs m;
        m.ws_o = a.p.ws_o;
        m.ws_lse = a.p.ws_lse;
        m.o = o;
        m.lse = lse;
        m.BH = BH;
        m.S = S;
        m.D = D;
        m.n_qtiles = sp->n_qtiles;
        m.n_qgroups = sp->n_qgroups;
        m.tpu = sp->tpu;
        m.causal = causal;
        m.chunk = sp->chunk;
        m.units_per_head = sp->units_per_head;
        if (fa::launch_merge(m, dtype == FA_DTYPE_BF16, s) != (int)cudaSuccess) return FA_ERR_CUDA;
    }
    return FA_OK;
}

}  // namespace

extern "C" {

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int S, int D, int causal,
           float scale, int dtype, cudaStream_t stream)
{
    int num_sms = 0;
    const int rc = check_call(q, k, v, o, lse, B, H, S, D, causal, scale, dtype, &num_sms);
    if (rc != FA_OK) return rc;
    return run_fwd(q, k, v, o, lse, B, H, S, D, causal, scale, dtype, num_sms, nullptr, nullptr, stream);
}

int fa_fwd_splitkv_workspace(int B, int H, int S, int D, int causal, int dtype, size_t* bytes)
{
    if (!bytes) return FA_ERR_INVALID_ARG;
    int rc = check_args(B, H, S, D, causal, dtype);
    if (rc != FA_OK) return rc;
    int num_sms = 0, cc = 0;
    rc = device_props(&num_sms, &cc);
    if (rc != FA_OK) return rc;
    SplitPlan sp;
    *bytes = plan_split(B * H, S, causal, num_sms, &sp) ? split_workspace_bytes(sp, D) : 0;
    return FA_OK;
}

int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int S, int D,
                   int causal, float scale, int dtype, void* workspace, size_t workspace_bytes, cudaStream_t stream)
{
    int num_sms = 0;
    const int rc = check_call(q, k, v, o, lse, B, H, S, D, causal, scale, dtype, &num_sms);
    if (rc != FA_OK) return rc;
    SplitPlan sp;
    if (!plan_split(B * H, S, causal, num_sms, &sp))
        return run_fwd(q, k, v, o, lse, B, H, S, D, causal, scale, dtype, num_sms, nullptr, nullptr, stream);
    if (!workspace || workspace_bytes < split_workspace_bytes(sp, D)) return FA_ERR_INVALID_ARG;
    if (!aligned16(workspace)) return FA_ERR_MISALIGNED;
    return run_fwd(q, k, v, o, lse, B, H, S, D, causal, scale, dtype, num_sms, &sp, static_cast<float*>(workspace),
                   stream);
}

namespace {

// The pipelined host-buffer path: the B*H heads are cut into chunks of whole
// heads (a multiple of 4, so every chunk's LSE slice stays 16-byte aligned)
// and the chunks go round-robin over a few library-owned streams, so chunk
// c+1 uploads while chunk c computes and chunk c-1 downloads.  Streams and
// events are host objects created once per device; nothing is allocated on
// the device.  The enqueue is serialised per device, so the shared events
// are recorded and waited on in matching pairs.
constexpr int kIoStreams = 3;
constexpr int kIoMaxChunks = 8;
constexpr size_t kIoMinBytes = size_t(32) << 20;     // below this one pass is enqueued as is
constexpr size_t kIoChunkBytes = size_t(48) << 20;   // input bytes per chunk, about

struct IoPipe {
    std::mutex mu;
    bool ready = false;
    cudaStream_t st[kIoStreams];
    cudaEvent_t start, done[kIoStreams];
};
IoPipe g_io[kMaxDevices];

int io_pipe_init(IoPipe& io)
{
    if (io.ready) return FA_OK;
    for (int i = 0; i < kIoStreams; ++i)
        if (cudaStreamCreateWithFlags(&io.st[i], cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&io.done[i], cudaEventDisableTiming) != cudaSuccess)
            return FA_ERR_CUDA;
    if (cudaEventCreateWithFlags(&io.start, cudaEventDisableTiming) != cudaSuccess) return FA_ERR_CUDA;
    io.ready = true;
    return FA_OK;
}

// Heads per chunk for a pass of BH heads; 0 means "do not chunk".
int io_heads_per_chunk(int BH, size_t head_bytes)
{
    const size_t in_bytes = 3 * (size_t)BH * head_bytes;
    if (BH < 8 || in_bytes < kIoMinBytes) return 0;
    int chunks = (int)std::min<size_t>(kIoMaxChunks, std::max<size_t>(2, in_bytes / kIoChunkBytes));
    chunks = std::min(chunks, BH / 4);
    if (chunks < 2) return 0;
    const int hc = ((BH + chunks - 1) / chunks + 3) / 4 * 4;
    return hc < BH ? hc : 0;
}

}  // namespace

int fa_fwd_hostio(const void* q_h, const void* k_h, const void* v_h, void* o_h, float* lse_h, void* q_d, void* k_d,
                  void* v_d, void* o_d, float* lse_d, int B, int H, int S, int D, int causal, float scale, int dtype,
                  cudaStream_t stream)
{
    if (!q_h || !k_h || !v_h || !o_h || !lse_h || !q_d || !k_d || !v_d || !o_d || !lse_d)
        return FA_ERR_INVALID_ARG;
    if (!(scale > 0.0f) || !std::isfinite(scale)) return FA_ERR_INVALID_ARG;
    int rc = check_args(B, H, S, D, causal, dtype);
    if (rc != FA_OK) return rc;
    const void* ptrs[10] = {q_h, k_h, v_h, o_h, lse_h, q_d, k_d, v_d, o_d, lse_d};
    for (const void* p : ptrs)
        if (!aligned16(p)) return FA_ERR_MISALIGNED;
    const size_t n = (size_t)B * H * S * D * 2, nl = (size_t)B * H * S * sizeof(float);
    cudaStream_t s = stream;
    const int BH = B * H;
    const size_t head_bytes = (size_t)S * D * 2, head_lse = (size_t)S * sizeof(float);
    const int hc = io_heads_per_chunk(BH, head_bytes);
    if (hc > 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
        IoPipe& io = g_io[dev];
        std::lock_guard<std::mutex> lock(io.mu);
        if ((rc = io_pipe_init(io)) != FA_OK) return rc;
        // the chunks start after the caller's earlier work on `stream` ...
        if (cudaEventRecord(io.start, s) != cudaSuccess) return FA_ERR_CUDA;
        for (int i = 0; i < kIoStreams; ++i)
            if (cudaStreamWaitEvent(io.st[i], io.start, 0) != cudaSuccess) return FA_ERR_CUDA;
        auto at = [](const void* base, size_t off) {
            return static_cast<char*>(const_cast<void*>(base)) + off;
        };
        int used = 0;
        for (int h0 = 0, c = 0; h0 < BH; h0 += hc, ++c) {
            const int nh = std::min(hc, BH - h0);
            cudaStream_t cs = io.st[c % kIoStreams];
            used = std::max(used, c % kIoStreams + 1);
            const size_t off = (size_t)h0 * head_bytes, bytes = (size_t)nh * head_bytes;
            const size_t loff = (size_t)h0 * head_lse, lbytes = (size_t)nh * head_lse;
            if (cudaMemcpyAsync(at(q_d, off), at(q_h, off), bytes, cudaMemcpyHostToDevice, cs) != cudaSuccess ||
                cudaMemcpyAsync(at(k_d, off), at(k_h, off), bytes, cudaMemcpyHostToDevice, cs) != cudaSuccess ||
                cudaMemcpyAsync(at(v_d, off), at(v_h, off), bytes, cudaMemcpyHostToDevice, cs) != cudaSuccess)
                return FA_ERR_CUDA;
            // heads are independent: a chunk is the pass of B = 1, H = nh on its slices
            rc = fa_fwd(at(q_d, off), at(k_d, off), at(v_d, off), at(o_d, off),
                        reinterpret_cast<float*>(at(lse_d, loff)), 1, nh, S, D, causal, scale, dtype, cs);
            if (rc != FA_OK) return rc;
            if (cudaMemcpyAsync(at(o_h, off), at(o_d, off), bytes, cudaMemcpyDeviceToHost, cs) != cudaSuccess ||
                cudaMemcpyAsync(at(lse_h, loff), at(lse_d, loff), lbytes, cudaMemcpyDeviceToHost, cs) != cudaSuccess)
                return FA_ERR_CUDA;
        }
        // ... and the caller's later work on `stream` waits for all of them
        for (int i = 0; i < used; ++i)
            if (cudaEventRecord(io.done[i], io.st[i]) != cudaSuccess ||
                cudaStreamWaitEvent(s, io.done[i], 0) != cudaSuccess)
                return FA_ERR_CUDA;
        return FA_OK;
    }
    if (cudaMemcpyAsync(q_d, q_h, n, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(k_d, k_h, n, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(v_d, v_h, n, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return FA_ERR_CUDA;
    rc = fa_fwd(q_d, k_d, v_d, o_d, lse_d, B, H, S, D, causal, scale, dtype, stream);
    if (rc != FA_OK) return rc;
    if (cudaMemcpyAsync(o_h, o_d, n, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyAsync(lse_h, lse_d, nl, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return FA_ERR_CUDA;
    return FA_OK;
}

int fa_device_status(cudaStream_t stream, int clear, unsigned int* site)
{
    if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
    unsigned int v = 0u;
    if (cudaMemcpyFromSymbol(&v, g_fa_status, sizeof(v)) != cudaSuccess) return FA_ERR_CUDA;
    if (clear && v != 0u) {
        const unsigned int zero = 0u;
        if (cudaMemcpyToSymbol(g_fa_status, &zero, sizeof(zero)) != cudaSuccess) return FA_ERR_CUDA;
    }
    if (site) *site = v;
    if (v == 0u) return FA_OK;
    return (v & 0xF00u) == fa::kSiteRangeV ? FA_ERR_RANGE : FA_ERR_TIMEOUT;
}

int fa_selftest_wait_timeout(unsigned int timeout_us, cudaStream_t stream)
{
    if (timeout_us < 1u || timeout_us > 10000000u) return FA_ERR_INVALID_ARG;
    void* status = nullptr;
    if (cudaGetSymbolAddress(&status, g_fa_status) != cudaSuccess) return FA_ERR_CUDA;
    const int e = fa::launch_wait_selftest(static_cast<unsigned int*>(status), (unsigned long long)timeout_us * 1000ull, stream);
    return e == (int)cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_selftest_exp2_poly(const float* x, float* y, int n, cudaStream_t stream)
{
    if (n < 0 || (n > 0 && (x == nullptr || y == nullptr))) return FA_ERR_INVALID_ARG;
    if (n == 0) return FA_OK;
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) % alignof(float) != 0) return FA_ERR_MISALIGNED;
    const int e = fa::launch_exp2_poly_selftest(x, y, n, stream);
    return e == (int)cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

#ifdef FA_DEBUG_STATS
// Debug-statistics build only ("CUDA手写masked multi-head attention", 6.3: a
// debug mode that hands each row's running maximum and sum to the host).  Every
// later one-pass fa_fwd writes, per row (b*H + h, i), its final base b and row
// sum l = sum over the row's keys of 2^(x - b), x the scaled score in base 2,
// into rows ([B*H, S, 2] fp32, device, caller-owned), and adds to counters[0]
// the warp rescales of O and to counters[1] the row re-bases after a row's
// first key tile (device, 2 x u64, caller-owned, zeroed by the caller).  Both
// null: off.  ln2 * (b + log2 l) is the row's LSE.
int fa_debug_stats_set(float* rows, unsigned long long* counters)
{
    if ((rows == nullptr) != (counters == nullptr)) return FA_ERR_INVALID_ARG;
    g_dbg_rows = rows;
    g_dbg_count = counters;
    return FA_OK;
}

// The re-base rule of P's type for `dtype` inputs: threshold T and overshoot,
// both in base-2 units (a re-base happens when the tile maximum passes b + T
// and moves b to the maximum plus the overshoot).
int fa_debug_rebase_rule(int dtype, float* threshold, float* overshoot)
{
    if (!threshold || !overshoot || (dtype != FA_DTYPE_F16 && dtype != FA_DTYPE_BF16)) return FA_ERR_INVALID_ARG;
    const bool p_bf16 = dtype == FA_DTYPE_BF16 ? fa::p_is_bf16<true>() : fa::p_is_bf16<false>();
    *threshold = p_bf16 ? fa::rebase_threshold<true>() : fa::rebase_threshold<false>();
    *overshoot = p_bf16 ? fa::rebase_overshoot<true>() : fa::rebase_overshoot<false>();
    return FA_OK;
}
#endif

#ifdef FA_TRACE
// Trace build only: every later fa_fwd records events of CTAs [0, ctas) into
// `buf` (device, ctas * 6 * cap 64-bit words, caller-owned, zeroed by the caller).
int fa_trace_set(unsigned long long* buf, int ctas, int cap)
{
    if ((buf == nullptr) != (ctas == 0) || ctas < 0 || cap < 0) return FA_ERR_INVALID_ARG;
    g_trace = buf;
    g_trace_ctas = ctas;
    g_trace_cap = cap;
    return FA_OK;
}
#endif

}  // extern "C"

// ---- split-KV without allocation -------------------------------------------------
// Scratch for fa_fwd_splitkv_static: a file-scope device array, so a caller
// that cannot allocate device memory still gets the split path.  Each device
// that loads the library holds these bytes until the process exits.

namespace {

constexpr size_t kStaticScratchBytes = 32ull << 20;   // 32 MiB

static __device__ __align__(256) unsigned char g_fa_static_scratch[kStaticScratchBytes];

// Device address of the array, looked up once per device (with that device
// current) and cached; in host code the symbol itself is not a device address.
std::atomic<void*> g_static_scratch_ptr[kMaxDevices];

int static_scratch(void** ptr)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
    void* p = g_static_scratch_ptr[dev].load(std::memory_order_acquire);
    if (!p) {
        if (cudaGetSymbolAddress(&p, g_fa_static_scratch) != cudaSuccess || !p) return FA_ERR_CUDA;
        g_static_scratch_ptr[dev].store(p, std::memory_order_release);
    }
    *ptr = p;
    return FA_OK;
}

}  // namespace

extern "C" int fa_fwd_splitkv_static(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                                     int S, int D, int causal, float scale, int dtype, cudaStream_t stream)
{
    int num_sms = 0;
    int rc = check_call(q, k, v, o, lse, B, H, S, D, causal, scale, dtype, &num_sms);
    if (rc != FA_OK) return rc;
    SplitPlan sp;
    if (!plan_split(B * H, S, causal, num_sms, &sp))
        return run_fwd(q, k, v, o, lse, B, H, S, D, causal, scale, dtype, num_sms, nullptr, nullptr, stream);
    if (split_workspace_bytes(sp, D) > kStaticScratchBytes) return FA_ERR_SCRATCH;
    void* ws = nullptr;
    rc = static_scratch(&ws);
    if (rc != FA_OK) return rc;
    return run_fwd(q, k, v, o, lse, B, H, S, D, causal, scale, dtype, num_sms, &sp, static_cast<float*>(ws), stream);
}
