// Launch parameters shared by the host launcher and the kernel instances.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fa {

constexpr int kBM = 128;       // query rows per tile (one TMEM lane per row)
constexpr int kBN = 128;       // keys per K/V tile
constexpr int kThreads = 512;  // 4 warpgroups: softmax x2, correction/epilogue, load+MMA
// Table schedule capacity: the table travels in the kernel parameters (16-bit
// unit indices and offsets), so it serves launches of up to this many units on
// up to this many CTAs; larger launches use the closed-form schedules.
constexpr int kSchedTableMaxUnits = 6144;
constexpr int kSchedTableMaxCtas = 160;

// Work-unit schedule and problem constants, identical for every CTA.
struct Params {
    float* lse;                 // [B*H, S] fp32 output
    void* o;                    // [B*H, S, D] 16-bit output (stores outside the TMA path)
    unsigned int* status;       // device status word (bounded-wait give-ups)
    unsigned long long timeout_ns;
    int BH;                     // B * H
    int S;                      // sequence length
    int n_qtiles;               // ceil(S / 128)
    int n_kv;                   // ceil(S / 128)
    int tpu;                    // query tiles per work unit: 1 or 2
    int n_qgroups;              // ceil(n_qtiles / tpu)
    int n_units;                // BH * n_qgroups
    int sched;                  // kSchedSnake, kSchedPairs or kSchedTable
    int head_group;             // snake: heads whose units are interleaved, longest first
    int pairs_per_head;         // pairs: ceil(n_qgroups / 2)
    long long n_pairs;          // pairs: BH * pairs_per_head
    int causal;                 // 1: key j allowed for query i iff j <= i
    int mask_last;              // the last K/V tile of a query tile needs masking
    float scale_log2;           // scale * log2(e)
    // Split-KV mode (split_chunk > 0): a unit covers key tiles
    // [chunk * split_chunk, (chunk + 1) * split_chunk) of one query group and
    // writes its O (normalised by its own row sums, fp32) and LSE to the
    // workspace; the merge kernel combines the chunks of each row.
    int split_chunk;            // key tiles per chunk, 0 = no split
    int units_per_head;         // split: sum over query groups of their chunk counts
    float* ws_o;                // split: [n_units][tpu][128][D] fp32
    float* ws_lse;              // split: [n_units][tpu][128] fp32
    // Event trace (used only by the FA_TRACE build): per traced CTA and role,
    // `trace_cap` 64-bit records of event, argument and SM clock.
    unsigned long long* trace;
    int trace_ctas;
    int trace_cap;
    // Debug statistics (used only by the FA_DEBUG_STATS build; null otherwise):
    // per row (b*H + h, i) its final base b and row sum l = sum 2^(x - b)
    // ([B*H, S, 2] fp32), and two counters: warp rescales of O, row re-bases
    // after a row's first key tile.
    float* dbg_rows;
    unsigned long long* dbg_count;
    // Table schedule (kSchedTable): CTA c runs units tab_unit[tab_off[c]] ..
    // tab_unit[tab_off[c + 1] - 1] in that order; a unit is bh * n_qgroups + qg.
    // Kept last: the kernel takes Params as a __grid_constant__ parameter and
    // reads the table from parameter space.
    unsigned short tab_off[kSchedTableMaxCtas + 1];
    unsigned short tab_unit[kSchedTableMaxUnits];
};

// Split-KV merge: one block per (batch*head, query tile) combines the tile's
// chunk partials into O (16-bit) and LSE.
struct MergeArgs {
    const float* ws_o;
    const float* ws_lse;
    void* o;
    float* lse;
    int BH, S, D, n_qtiles, n_qgroups, tpu, causal, chunk, units_per_head;
};
int launch_merge(const MergeArgs& a, bool bf16, cudaStream_t s);

// Trace roles and events (FA_TRACE build).  A record is
// event << 56 | (arg & 0xFFFF) << 40 | (clock64 & (2^40 - 1)).
enum TraceRole : int { kTrSoftmax0 = 0, kTrSoftmax1 = 1, kTrEpilogue = 2, kTrLoad = 3, kTrMma = 4, kTrKernel = 5,
                       kTraceRoles = 6 };
enum TraceEvent : unsigned {
    kEvSReady = 1,      // softmax: scores of key tile j visible (arg j)
    kEvPDone = 2,       // softmax: P of key tile j published (arg j)
    kEvRescale = 3,     // softmax: O rescaled in TMEM (arg j)
    kEvSLoaded = 4,     // softmax: scores in registers (arg j)
    kEvMaxDone = 5,     // softmax: row maximum and re-base decision done (arg j)
    kEvExpDone = 6,     // softmax: first half of P published (arg j)
    kEvUnit = 10,       // MMA: unit starts (arg unit index)
    kEvQK = 11,         // MMA: QK issued (arg t << 12 | j)
    kEvPV = 12,         // MMA: PV issued (arg t << 12 | j)
    kEvPWait = 13,      // MMA: starts waiting for P (arg t << 12 | j)
    kEvPVGo = 14,       // MMA: first half of P ready, first PV half about to issue (arg t << 12 | j)
    kEvPVMid = 15,      // MMA: first PV half issued (arg t << 12 | j)
    kEvQKGo = 16,       // MMA: about to issue QK (arg t << 12 | j)
    kEvQLoad = 20,      // load: Q tile issued (arg t)
    kEvKVLoad = 21,     // load: K or V tile issued (arg ring index)
    kEvOFull = 30,      // epilogue: O of tile t complete (arg t)
    kEvEpiDone = 31,    // epilogue: tile t stored (arg t)
    kEvEntry = 40,      // kernel: thread 0 entered
    kEvSetup = 41,      // kernel: barriers initialised, TMEM allocated
    kEvExit = 42,       // kernel: all roles done, before TMEM is freed
};

enum : int { kSchedSnake = 0, kSchedPairs = 1, kSchedTable = 2 };

// Key tiles a query tile visits: all of them, or up to its diagonal when causal.
__host__ __device__ inline int kv_tiles_of(int q_tile, int n_kv, int causal)
{
    return causal ? (q_tile + 1 < n_kv ? q_tile + 1 : n_kv) : n_kv;
}

// Split-KV: number of key chunks of query group qg (its last tile sets the range).
__host__ __device__ inline int split_chunks(int qg, int tpu, int n_qtiles, int n_kv, int causal, int chunk)
{
    int last_tile = qg * tpu + tpu - 1;
    if (last_tile > n_qtiles - 1) last_tile = n_qtiles - 1;
    return (kv_tiles_of(last_tile, n_kv, causal) + chunk - 1) / chunk;
}


struct LaunchArgs {
    CUtensorMap tm_q, tm_k, tm_v, tm_o;
    Params p;
    int grid;
    int device;   // current CUDA device (0..63): the launcher sets per-device kernel attributes once
};

// One launcher per (head dim, dtype) instance; each lives in its own
// translation unit.  Returns a cudaError_t.
int launch_d64_f16(const LaunchArgs& a, cudaStream_t s);
int launch_d64_bf16(const LaunchArgs& a, cudaStream_t s);
int launch_d128_f16(const LaunchArgs& a, cudaStream_t s);
int launch_d128_bf16(const LaunchArgs& a, cudaStream_t s);
int launch_d64_f16_split(const LaunchArgs& a, cudaStream_t s);
int launch_d64_bf16_split(const LaunchArgs& a, cudaStream_t s);
int launch_d128_f16_split(const LaunchArgs& a, cudaStream_t s);
int launch_d128_bf16_split(const LaunchArgs& a, cudaStream_t s);
int launch_d64_f16_kp(const LaunchArgs& a, cudaStream_t s);
int launch_d64_bf16_kp(const LaunchArgs& a, cudaStream_t s);
int launch_d64_f16_split_kp(const LaunchArgs& a, cudaStream_t s);
int launch_d64_bf16_split_kp(const LaunchArgs& a, cudaStream_t s);

// One-tile layout (fa_fwd_wide.cuh): one 128-row query tile per unit, steps of
// kWideBN keys.  LaunchArgs::tm_o is not used; its K and V maps have boxes of
// kWideBN rows (the kernel's expected bytes per copy assume exactly that).
constexpr int kWideBN = 192;
int launch_wide_d64_f16(const LaunchArgs& a, cudaStream_t s);
int launch_wide_d64_bf16(const LaunchArgs& a, cudaStream_t s);
int launch_wide_d128_f16(const LaunchArgs& a, cudaStream_t s);
int launch_wide_d128_bf16(const LaunchArgs& a, cudaStream_t s);
int wide_smem_bytes_for(int D);

// Dynamic shared memory of the instance for head dim D.
int smem_bytes_for(int D);

// Whether the large shared-memory opt-in of kernel `kern` is already set on
// `device`, and recording that it is.  Keyed by the kernel's own address, so
// several builds of this library loaded into one process never share an entry.
bool smem_opt_in_done(const void* kern, int device);
void smem_opt_in_mark(const void* kern, int device);

// Kernel that waits on a barrier nobody arrives on (bounded-wait self-test).
int launch_wait_selftest(unsigned int* status, unsigned long long timeout_ns, cudaStream_t s);
int launch_exp2_poly_selftest(const float* x, float* y, int n, cudaStream_t s);

}  // namespace fa
