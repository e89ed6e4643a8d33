/*
 * fa_fwd.h - C ABI of the GB300 (sm_103a) fused attention forward pass.
 *
 * The operation (one call = the whole hot path):
 *
 *   O    = softmax(Q K^T * scale + mask) V
 *   LSE_i = ln sum_j exp(scale * q_i . k_j)      over the keys j row i may see
 *
 * for every (batch b, head h) independently.  The formula is the one of
 * "CUDA手写masked multi-head attention", section 3.1 (Attention公式的CUDA语义
 * 重写); the causal mask keeps the lower triangle (key j <= query i), as the
 * same section's mask code and comment state, and masked scores count as -inf.
 * The computation is tiled with online softmax ("FlashAttention的Triton性能考古学",
 * sections 核心算法回顾 and 关键优化：反转循环顺序: running max and sum per row,
 * one normalisation at the end), so the S x S score matrix never reaches device
 * memory, and uses the conditional rescale of "G6: Cluster 与 2CTA 探索", V41:
 * a row keeps its base until its maximum rises by more than 2^15 (fp16) or 2^30
 * (bf16) in scaled base-2 units (the page's 2^8, widened to what P's type holds),
 * and O is rescaled only then, 32 rows at a time.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Layout     q, k, v, o: contiguous [B, H, S, D] tensors of `dtype` (row-major,
 *            D fastest).  lse: contiguous [B, H, S] float32.  Q, K and V share
 *            S (self-attention, square mask).
 * Pointers   "device" pointers must be addressable by the current CUDA device
 *            (cudaMalloc / torch CUDA tensors); "host" pointers are ordinary or
 *            pinned host memory.  All tensor pointers must be 16-byte aligned.
 * Ownership  The caller allocates and frees every buffer; no call allocates
 *            device memory.  Loading the library reserves, on every device
 *            that runs any of its entry points, one static 32 MiB device
 *            array: the scratch of fa_fwd_splitkv_static, which keeps the
 *            partial results of the last split call made through that entry
 *            point (see it for the sharing and race rules).  Beyond that the
 *            library keeps no per-call state; it caches per device the SM
 *            count, the status word's address and each kernel's shared-memory
 *            opt-in, and per shape the launch schedule and the split-KV plan
 *            (host memory, guarded for concurrent use).
 * Streams    `stream` is a cudaStream_t (NULL = legacy default stream).  Work
 *            is enqueued on it and the call returns without synchronising;
 *            calls on different streams may run concurrently.  Each pass is
 *            launched as a programmatic dependent of the work before it on
 *            the stream: its blocks may be scheduled while that work
 *            finishes, but touch no global memory until it has completed, so
 *            ordering on the stream is that of any kernel.  fa_fwd,
 *            fa_fwd_splitkv and fa_fwd_splitkv_static can be captured into
 *            CUDA graphs (the kernels' parameters carry everything a launch
 *            needs); fa_fwd_splitkv_static only after one uncaptured call on
 *            the device, which looks up the address of its scratch array.
 * Errors     Every entry point returns an fa_status_t and never aborts, throws
 *            or prints.  Invalid arguments are rejected before anything is
 *            enqueued.
 * Sizes      B, H, S >= 1 with B*H*S*D < 2^31 elements per tensor; D in {64,
 *            128}; dtype fp16 or bf16; any S (tails are masked in the kernel).
 */
#ifndef FA_FWD_H
#define FA_FWD_H

#include <stddef.h>

/* The CUDA runtime's stream handle, declared here so that this header needs no
 * CUDA include; identical to the runtime's own typedef. */
#ifndef __CUDA_RUNTIME_API_H__
typedef struct CUstream_st* cudaStream_t;
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_DTYPE_F16 = 0,   /* IEEE binary16 inputs and output, fp32 accumulation */
    FA_DTYPE_BF16 = 1   /* bfloat16 inputs and output, fp32 accumulation */
} fa_dtype_t;

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,  /* null pointer, B/H/S < 1, causal not 0/1, scale not finite or <= 0,
                                sizes overflowing 2^31 elements */
    FA_ERR_UNSUPPORTED = 2,  /* D not in {64, 128}, unknown dtype, current device not compute capability 10.3 */
    FA_ERR_MISALIGNED = 3,   /* a tensor pointer not 16-byte aligned */
    FA_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed (launch, copy, tensor map) */
    FA_ERR_TIMEOUT = 5,      /* a bounded in-kernel wait gave up (reported by fa_device_status) */
    FA_ERR_SCRATCH = 6,      /* fa_fwd_splitkv_static: the problem needs more than its static scratch */
    FA_ERR_RANGE = 7         /* bf16 inputs: O came out not finite - V held an element beyond +-65504 (fp16's
                                range) or an input was not finite (reported by fa_device_status) */
} fa_status_t;

/*
 * fa_fwd - the fused attention forward pass on device buffers.
 *
 *   q, k, v  device, read-only, [B, H, S, D] of dtype
 *   o        device, written, [B, H, S, D] of dtype; O rounded to nearest-even
 *   lse      device, written, [B, H, S] float32, natural log of the row sums of
 *            exp(scaled scores) over the allowed keys
 *   causal   0 = no mask, 1 = key j allowed for query i iff j <= i
 *   scale    multiplier of Q K^T, finite and > 0 (usually 1/sqrt(D))
 *   dtype    an fa_dtype_t
 *   stream   the CUDA stream the work is enqueued on
 *
 * One kernel launch per call.  o and lse must not overlap q, k or v.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int B, int H, int S, int D, int causal, float scale, int dtype, cudaStream_t stream);

/*
 * fa_fwd_splitkv - fa_fwd for problems too small to fill the GPU in one pass.
 *
 * When one pass would give fewer work units than the device has SMs (few
 * heads and short sequences) and a cost model of the kernel predicts a
 * shorter run, the key range of every query tile group is cut into chunks of
 * key tiles processed as separate units: each writes the softmax-normalised
 * partial O of its keys (fp32) and their LSE into `workspace`, and a second
 * kernel combines the chunks of every row, O = sum_c exp(LSE_c - LSE) O_c
 * with LSE = ln sum_c exp(LSE_c) - the online softmax merge of
 * "FlashAttention的Triton性能考古学" (核心算法回顾) applied to whole chunks.
 * Otherwise the call is exactly fa_fwd and ignores `workspace`.
 *
 *   workspace        device, caller-owned scratch of at least the size that
 *                    fa_fwd_splitkv_workspace reports, 16-byte aligned; its
 *                    contents need no initialisation and are overwritten
 *   workspace_bytes  its size
 *
 * Two launches (attention, merge) on `stream`; calls that share a workspace
 * must not overlap.
 * FA_ERR_INVALID_ARG if the workspace is missing or too small while a split
 * is needed; otherwise errors as fa_fwd.
 */
int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                   int B, int H, int S, int D, int causal, float scale, int dtype,
                   void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * fa_fwd_splitkv_workspace - bytes of workspace fa_fwd_splitkv needs for this
 * problem on the current device (0: no split, the call runs one pass).
 * Host only; errors as fa_fwd's argument checks.
 */
int fa_fwd_splitkv_workspace(int B, int H, int S, int D, int causal, int dtype, size_t* bytes);

/*
 * fa_fwd_splitkv_static - fa_fwd_splitkv for callers that cannot allocate.
 *
 * No counterpart on the source pages: this entry point exists for callers that
 * must not or cannot call cudaMalloc - runtimes that forbid allocation after
 * start-up (fixed memory budgets, real-time serving loops), or code that runs
 * under another framework's allocator and holds no handle to it - but still
 * want the split path for small problems.  It allocates nothing: its split
 * scratch is a static device array of 32 MiB (2^25 bytes) inside the library,
 * which every GPU that loads the library holds until the process exits.
 *
 * Same arguments, layouts and results as fa_fwd_splitkv, without the
 * workspace.  The first call on a device looks up that device's address of the
 * array (cudaGetSymbolAddress, with the device current) and caches it; make
 * that first call before any stream capture.  All calls on a device share the
 * one array: calls whose work overlaps on the GPU (different streams, or
 * threads) race on it and must be serialised by the caller.  The array keeps
 * the last call's partial results; nothing in it needs clearing, since a call
 * writes every partial it reads.  Returns FA_ERR_SCRATCH, launching nothing,
 * when the split plan needs more than 32 MiB (fa_fwd_splitkv_workspace reports
 * the need); otherwise errors as fa_fwd_splitkv.  Problems that one pass
 * already fits run as fa_fwd and use no scratch.
 */
int fa_fwd_splitkv_static(const void* q, const void* k, const void* v, void* o, float* lse,
                          int B, int H, int S, int D, int causal, float scale, int dtype, cudaStream_t stream);

/*
 * fa_fwd_hostio - the same pass with host-side inputs and outputs.
 *
 * Host->device copies of q_h, k_h, v_h into the caller's device buffers q_d,
 * k_d, v_d; fa_fwd on them into o_d, lse_d; device->host copies of o_d, lse_d
 * into o_h, lse_h.  Returns once everything is enqueued; the caller
 * synchronises `stream` before reading o_h / lse_h.  Host buffers should be
 * pinned for the copies to be asynchronous.  Same layouts, sizes and errors as
 * fa_fwd; all ten pointers must be non-null and 16-byte aligned.
 *
 * Passes that move 32 MiB or more of input over at least 8 heads are cut into
 * up to 8 chunks of whole heads (multiples of 4), enqueued round-robin on
 * three streams the library creates once per device, so the copies of one
 * chunk overlap the compute of another (the attention of a head does not
 * depend on the other heads; results are identical to one pass).  That work
 * is ordered after what the caller enqueued on `stream` before the call, and
 * `stream` waits for all of it, so work enqueued on `stream` after the call
 * sees the results.  Enqueueing is serialised per device across threads.
 */
int fa_fwd_hostio(const void* q_h, const void* k_h, const void* v_h, void* o_h, float* lse_h,
                  void* q_d, void* k_d, void* v_d, void* o_d, float* lse_d,
                  int B, int H, int S, int D, int causal, float scale, int dtype, cudaStream_t stream);

/* Launch geometry fa_fwd would use for a problem on the current device. */
typedef struct {
    int grid;            /* CTAs launched (persistent: <= SM count) */
    int block;           /* threads per CTA */
    int smem_bytes;      /* dynamic shared memory per CTA */
    int tiles_per_unit;  /* 128-row query tiles per work unit (1 or 2) */
    int units;           /* work units = B*H * ceil(query tiles / tiles_per_unit) */
    int head_group;      /* snake schedule: heads scheduled together (longest units first) */
    int num_sms;         /* SM count of the current device */
    int schedule;        /* 0 = snake over units, 1 = causal mirror pairs, 2 = host list schedule
                            (fa_fwd_schedule_table); see the kernel source */
    int layout;          /* 1 = two query tiles per unit, 2 = one query tile per unit (fa_fwd_set_layout) */
    int key_step;        /* keys per step of a unit's key loop: 128 (layout 1) or 192 (layout 2) */
} fa_launch_info_t;

/*
 * fa_fwd_launch_info - fills *info for fa_fwd(B, H, S, D, causal, dtype).
 * Host only: queries the current device's SM count, launches nothing.
 * Errors as fa_fwd's argument checks (pointers are not examined).
 */
int fa_fwd_launch_info(int B, int H, int S, int D, int causal, int dtype, fa_launch_info_t* info);

/*
 * fa_fwd_plan - the same geometry for a device with `num_sms` SMs (>= 1).
 * Pure host computation: touches no device, so it works without a GPU.
 */
int fa_fwd_plan(int B, int H, int S, int D, int causal, int dtype, int num_sms, fa_launch_info_t* info);

/*
 * fa_fwd_set_layout - the kernel layout of one-pass launches, process-wide.
 *
 * Not on the pages: two layouts of the same computation, kept side by side so
 * they can be measured against each other.
 *   0  automatic (the default): the library picks per launch
 *   1  two 128-row query tiles per work unit, 128-key steps, the two softmax
 *      warpgroups alternating between the tiles (the ping-pong of "G6: Cluster
 *      与 2CTA 探索", V37-V39, on one CTA)
 *   2  one query tile per work unit, 192-key steps, both softmax warpgroups on
 *      the tile (each on half of a step's keys), scores and probabilities in
 *      separate tensor-memory regions so the next step's Q K^T overlaps the
 *      softmax
 * Split-KV launches (fa_fwd_splitkv) always use layout 1.  Results agree to
 * within rounding, not bit for bit, across layouts; each layout is
 * deterministic.  Returns the previous setting, or -1 (nothing changed) for
 * a value outside 0..2.  Calls already enqueued are not affected.
 */
int fa_fwd_set_layout(int layout);

/*
 * fa_fwd_schedule_table - the table schedule fa_fwd uses for a causal launch
 * of several rounds (schedule == 2 in fa_fwd_plan) on a device with `num_sms`
 * SMs.  Not on the pages: causal units differ in length ("CUDA手写masked
 * multi-head attention", section 2.1: the upper triangle does no work), and the
 * host balances them by longest-first list scheduling inside groups of heads
 * whose K/V fit in L2 together; the table travels in the kernel parameters.
 *
 * Pure host computation (no device).  On success writes n_ctas + 1 offsets to
 * offsets[] (capacity offsets_cap) and n_units unit indices to units[]
 * (capacity units_cap): CTA c runs units[offsets[c]] .. units[offsets[c+1]-1]
 * in that order, a unit index being bh * ceil(query tiles / tiles_per_unit) +
 * query group.  Returns FA_OK; FA_ERR_UNSUPPORTED when the launch uses a
 * closed-form schedule instead; FA_ERR_INVALID_ARG for a null pointer,
 * num_sms < 1 or a buffer that is too small; otherwise as fa_fwd's checks.
 */
int fa_fwd_schedule_table(int B, int H, int S, int D, int causal, int dtype, int num_sms,
                          unsigned short* offsets, int offsets_cap, unsigned short* units, int units_cap,
                          int* n_ctas, int* n_units);

/*
 * fa_device_status - the device status word of the kernels.
 *
 * Every wait inside the kernels gives up after a time limit (default 4 s,
 * FA_WAIT_TIMEOUT_MS overrides it when the library is loaded), records the
 * wait site in a device status word and makes its CTA exit cleanly.  With
 * bf16 inputs the two-tile layout computes P*V in fp16 (P and V of one type;
 * bf16's 8-bit significand on P measurably moves O past the output's rounding
 * midpoints on near one-hot rows), converting V to fp16 in shared memory: an
 * element of V beyond +-65504 becomes infinite, and a CTA whose O comes out
 * not finite records site 0x800.  This
 * call synchronises `stream`, reads the word, clears it if `clear` is non-zero
 * and returns FA_OK, FA_ERR_RANGE (site 0x800) or FA_ERR_TIMEOUT (any other
 * site); *site (if non-null) receives the recorded site code (0 = none).
 * FA_ERR_CUDA if the synchronisation fails.
 */
int fa_device_status(cudaStream_t stream, int clear, unsigned int* site);

/*
 * fa_selftest_wait_timeout - exercises the bounded wait used by the kernels.
 *
 * Launches one CTA that waits on a shared-memory barrier nothing ever arrives
 * on, with a limit of `timeout_us` microseconds (1..10^7).  The wait gives up,
 * records its site in the status word and the kernel returns.  Returns FA_OK
 * once enqueued; read the outcome with fa_device_status.  Faults and hangs
 * nothing: the context stays usable.
 */
int fa_selftest_wait_timeout(unsigned int timeout_us, cudaStream_t stream);

/*
 * fa_selftest_exp2_poly - evaluates the FMA-pipe exponential the softmax can
 * use for part of its exponentials (build option FA_EXP2_POLY_PAIRS; off in
 * the default build): y[i] = 2^x[i] for i < n.
 *
 * The method is the range reduction 2^x = 2^n * 2^f (n = rint(x),
 * f in [-1/2, 1/2]) with a degree-3 minimax polynomial for 2^f; the split of
 * the exponential work between units follows the MIO-bottleneck section of
 * "FlashAttention的Triton性能考古学".  Relative error <= 7.5e-5 for results
 * >= 2^-126 (x >= -125.9); arguments <= -127 (and -inf) give +0.
 *
 * x, y: device pointers to n floats (4-byte aligned), caller-owned; n >= 0
 * (n = 0 launches nothing).  Enqueued on `stream`, returns at once.
 * FA_ERR_INVALID_ARG for n < 0 or a null pointer with n > 0,
 * FA_ERR_MISALIGNED for a pointer not 4-byte aligned, FA_ERR_CUDA if the
 * launch fails.
 */
int fa_selftest_exp2_poly(const float* x, float* y, int n, cudaStream_t stream);

/* Human-readable text for an fa_status_t; never NULL. */
const char* fa_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* FA_FWD_H */
