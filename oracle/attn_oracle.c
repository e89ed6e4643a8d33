/*
 * fp64 CPU oracle for the fused attention forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * bench's CPU-baseline leg may build, load or call this file.  It shares no
 * code, header, table or helper with the CUDA path, and the CUDA path never
 * calls it.
 *
 * Every array is contiguous.  q, k, v and o are [BH][S][D] float64 (BH = B*H),
 * lse is [BH][S] float64.  The 16-bit inputs are widened exactly by the caller.
 * Arithmetic is IEEE double; the file must be compiled without -ffast-math.
 *
 * What each function follows:
 *
 *  fa_oracle_attention      The definition O = softmax(Q K^T * scale + mask) V
 *                           of "CUDA手写masked multi-head attention", section 3.1
 *                           (the "+" before the mask was lost in the page text),
 *                           with the causal mask of the same section: only the
 *                           lower triangle (key j <= query i) is kept and masked
 *                           scores become -inf.  The full S x S score matrix of
 *                           each head is materialised.  LSE_i = ln sum_j
 *                           exp(s_ij) over the allowed j, in natural log.
 *  fa_oracle_attention_rows The same definition for a list of (head, row)
 *                           pairs: one score row at a time, for sequences whose
 *                           S x S matrix does not fit in host memory.
 *  fa_oracle_online         The tiled online softmax of "FlashAttention的Triton
 *                           性能考古学", sections 核心算法回顾 and 关键优化：反转
 *                           循环顺序: running max m and running sum l per row,
 *                           one key block at a time, the accumulator rescaled by
 *                           exp(m_old - m_new), and one division at the end.
 *  fa_oracle_lazy           The conditional rescale of "G6: Cluster 与 2CTA 探索",
 *                           V41 (Conditional Scale): base-2 domain, a row base b
 *                           that only moves when the tile maximum exceeds b by
 *                           more than a threshold (8 on the page), so p lies in
 *                           (0, 2^threshold].  The probabilities fed to P*V may be
 *                           rounded to fp16 or bf16 as the GPU does; the row sum
 *                           uses the unrounded values.  This is an algorithm
 *                           model, used to pin the recurrence and to predict the
 *                           GPU's error budget and rescale counts.
 *
 * A row with no allowed key (impossible for a square causal mask, defined for
 * completeness) gets O = 0 and LSE = -inf.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static int allowed(int causal, int64_t i, int64_t j) { return !causal || j <= i; }

static double dot(const double* a, const double* b, int64_t D)
{
    double acc = 0.0;
    for (int64_t d = 0; d < D; ++d) acc += a[d] * b[d];
    return acc;
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int fa_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- the definition, full score matrix per head ------------------------- */
int fa_oracle_attention(const double* q, const double* k, const double* v,
                        int64_t BH, int64_t S, int64_t D, int causal, double scale,
                        double* o, double* lse, int nthreads)
{
    if (BH < 0 || S < 0 || D < 1) return 1;
    set_threads(nthreads);
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t h = 0; h < BH; ++h) {
        const double* qh = q + h * S * D;
        const double* kh = k + h * S * D;
        const double* vh = v + h * S * D;
        double* oh = o + h * S * D;
        double* lh = lse + h * S;
        double* s = (double*)malloc((size_t)(S > 0 ? S : 1) * (size_t)(S > 0 ? S : 1) * sizeof(double));
        if (!s) {
#pragma omp atomic write
            failed = 1;
            continue;
        }
        /* scores s_ij = scale * q_i . k_j, masked entries -inf */
        for (int64_t i = 0; i < S; ++i)
            for (int64_t j = 0; j < S; ++j)
                s[i * S + j] = allowed(causal, i, j) ? scale * dot(qh + i * D, kh + j * D, D)
                                                     : -INFINITY;
        for (int64_t i = 0; i < S; ++i) {
            double* row = s + i * S;
            double m = -INFINITY;
            for (int64_t j = 0; j < S; ++j) if (row[j] > m) m = row[j];
            double* oi = oh + i * D;
            for (int64_t d = 0; d < D; ++d) oi[d] = 0.0;
            if (m == -INFINITY) { lh[i] = -INFINITY; continue; }
            double sum = 0.0;
            for (int64_t j = 0; j < S; ++j) sum += exp(row[j] - m);
            double L = m + log(sum);
            lh[i] = L;
            /* P_ij = exp(s_ij - LSE_i); O_i = sum_j P_ij v_j */
            for (int64_t j = 0; j < S; ++j) {
                double p = exp(row[j] - L);
                if (p == 0.0) continue;
                const double* vj = vh + j * D;
                for (int64_t d = 0; d < D; ++d) oi[d] += p * vj[d];
            }
        }
        free(s);
    }
    return failed ? 2 : 0;
}

/* ---- the definition, one score row at a time, for sampled rows ---------- */
int fa_oracle_attention_rows(const double* q, const double* k, const double* v,
                             int64_t BH, int64_t S, int64_t D, int causal, double scale,
                             int64_t nrows, const int64_t* heads, const int64_t* rows,
                             double* o_rows, double* lse_rows, int nthreads)
{
    if (BH < 0 || S < 0 || D < 1 || nrows < 0) return 1;
    for (int64_t r = 0; r < nrows; ++r)
        if (heads[r] < 0 || heads[r] >= BH || rows[r] < 0 || rows[r] >= S) return 1;
    set_threads(nthreads);
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t h = heads[r], i = rows[r];
        const double* qi = q + (h * S + i) * D;
        const double* kh = k + h * S * D;
        const double* vh = v + h * S * D;
        double* oi = o_rows + r * D;
        double* s = (double*)malloc((size_t)(S > 0 ? S : 1) * sizeof(double));
        if (!s) {
#pragma omp atomic write
            failed = 1;
            continue;
        }
        double m = -INFINITY;
        for (int64_t j = 0; j < S; ++j) {
            s[j] = allowed(causal, i, j) ? scale * dot(qi, kh + j * D, D) : -INFINITY;
            if (s[j] > m) m = s[j];
        }
        for (int64_t d = 0; d < D; ++d) oi[d] = 0.0;
        if (m == -INFINITY) { lse_rows[r] = -INFINITY; free(s); continue; }
        double sum = 0.0;
        for (int64_t j = 0; j < S; ++j) sum += exp(s[j] - m);
        double L = m + log(sum);
        lse_rows[r] = L;
        for (int64_t j = 0; j < S; ++j) {
            double p = exp(s[j] - L);
            if (p == 0.0) continue;
            const double* vj = vh + j * D;
            for (int64_t d = 0; d < D; ++d) oi[d] += p * vj[d];
        }
        free(s);
    }
    return failed ? 2 : 0;
}

/* ---- textbook online softmax over key blocks of `tile` keys -------------- */
int fa_oracle_online(const double* q, const double* k, const double* v,
                     int64_t BH, int64_t S, int64_t D, int causal, double scale,
                     int64_t tile, double* o, double* lse, int nthreads)
{
    if (BH < 0 || S < 0 || D < 1 || tile < 1) return 1;
    set_threads(nthreads);
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t h = 0; h < BH; ++h) {
        const double* kh = k + h * S * D;
        const double* vh = v + h * S * D;
        double* acc = (double*)malloc((size_t)D * sizeof(double));
        double* sblk = (double*)malloc((size_t)tile * sizeof(double));
        if (!acc || !sblk) {
            free(acc); free(sblk);
#pragma omp atomic write
            failed = 1;
            continue;
        }
        /* Q block outer (one row at a time here), key blocks inner */
        for (int64_t i = 0; i < S; ++i) {
            const double* qi = q + (h * S + i) * D;
            double m = -INFINITY, l = 0.0;
            for (int64_t d = 0; d < D; ++d) acc[d] = 0.0;
            for (int64_t j0 = 0; j0 < S; j0 += tile) {
                int64_t n = (S - j0 < tile) ? S - j0 : tile;
                double mb = -INFINITY;
                for (int64_t t = 0; t < n; ++t) {
                    int64_t j = j0 + t;
                    sblk[t] = allowed(causal, i, j) ? scale * dot(qi, kh + j * D, D) : -INFINITY;
                    if (sblk[t] > mb) mb = sblk[t];
                }
                double m_new = (mb > m) ? mb : m;
                if (m_new == -INFINITY) continue;          /* nothing allowed yet */
                double corr = exp(m - m_new);              /* 0 when m was -inf */
                l *= corr;
                for (int64_t d = 0; d < D; ++d) acc[d] *= corr;
                for (int64_t t = 0; t < n; ++t) {
                    double p = exp(sblk[t] - m_new);
                    if (p == 0.0) continue;
                    l += p;
                    const double* vj = vh + (j0 + t) * D;
                    for (int64_t d = 0; d < D; ++d) acc[d] += p * vj[d];
                }
                m = m_new;
            }
            double* oi = o + (h * S + i) * D;
            if (m == -INFINITY) {
                for (int64_t d = 0; d < D; ++d) oi[d] = 0.0;
                lse[h * S + i] = -INFINITY;
                continue;
            }
            for (int64_t d = 0; d < D; ++d) oi[d] = acc[d] / l;   /* deferred normalisation */
            lse[h * S + i] = m + log(l);
        }
        free(acc);
        free(sblk);
    }
    return failed ? 2 : 0;
}

/* ---- rounding of a probability to a 16-bit format, round-to-nearest-even -- */
/* mant_bits counts the implicit bit (11 for fp16, 8 for bf16); emin is the
 * exponent of the smallest normal (-14 for fp16, -126 for bf16).  Values are
 * non-negative and far below either format's overflow threshold here. */
static double round_to_format(double x, int mant_bits, int emin)
{
    if (x == 0.0 || !isfinite(x)) return x;
    int e;
    frexp(x, &e);                   /* x = f * 2^e, f in [0.5, 1) -> unit exponent e-1 */
    int ue = e - 1;
    if (ue < emin) ue = emin;       /* subnormal range keeps the smallest spacing */
    double ulp = ldexp(1.0, ue - (mant_bits - 1));
    return rint(x / ulp) * ulp;     /* rint: ties to even under the default mode */
}

/* p_round: 0 = none, 1 = fp16, 2 = bf16.
 * stats (may be NULL), 3 doubles: number of re-bases after a row's first
 * non-empty tile, largest p seen, number of (row, tile) steps. */
int fa_oracle_lazy(const double* q, const double* k, const double* v,
                   int64_t BH, int64_t S, int64_t D, int causal, double scale,
                   int64_t tile, double threshold, int p_round,
                   double* o, double* lse, double* stats, int nthreads)
{
    if (BH < 0 || S < 0 || D < 1 || tile < 1 || !(threshold >= 0.0) || p_round < 0 || p_round > 2)
        return 1;
    set_threads(nthreads);
    const double c = scale * M_LOG2E;      /* scores move to the base-2 domain */
    double rebases = 0.0, pmax = 0.0, steps = 0.0;
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+:rebases, steps) reduction(max:pmax)
    for (int64_t h = 0; h < BH; ++h) {
        const double* kh = k + h * S * D;
        const double* vh = v + h * S * D;
        double* acc = (double*)malloc((size_t)D * sizeof(double));
        double* sblk = (double*)malloc((size_t)tile * sizeof(double));
        if (!acc || !sblk) {
            free(acc); free(sblk);
#pragma omp atomic write
            failed = 1;
            continue;
        }
        for (int64_t i = 0; i < S; ++i) {
            const double* qi = q + (h * S + i) * D;
            double b = -INFINITY, l = 0.0;
            int started = 0;
            for (int64_t d = 0; d < D; ++d) acc[d] = 0.0;
            for (int64_t j0 = 0; j0 < S; j0 += tile) {
                int64_t n = (S - j0 < tile) ? S - j0 : tile;
                double tmax = -INFINITY;                 /* max of the raw dot products */
                for (int64_t t = 0; t < n; ++t) {
                    int64_t j = j0 + t;
                    sblk[t] = allowed(causal, i, j) ? dot(qi, kh + j * D, D) : -INFINITY;
                    if (sblk[t] > tmax) tmax = sblk[t];
                }
                if (tmax == -INFINITY) continue;         /* tile fully masked for this row */
                steps += 1.0;
                double cand = (tmax * c > b) ? tmax * c : b;
                double history = 1.0;
                if (cand > b + threshold) {              /* re-base only past the threshold */
                    history = exp2(b - cand);            /* 0 when b was -inf */
                    if (started) rebases += 1.0;
                    b = cand;
                }
                started = 1;
                l *= history;
                for (int64_t d = 0; d < D; ++d) acc[d] *= history;
                for (int64_t t = 0; t < n; ++t) {
                    if (sblk[t] == -INFINITY) continue;
                    double p = exp2(sblk[t] * c - b);    /* in (0, 2^threshold] */
                    if (p > pmax) pmax = p;
                    l += p;
                    double pu = p_round == 1 ? round_to_format(p, 11, -14)
                              : p_round == 2 ? round_to_format(p, 8, -126) : p;
                    const double* vj = vh + (j0 + t) * D;
                    for (int64_t d = 0; d < D; ++d) acc[d] += pu * vj[d];
                }
            }
            double* oi = o + (h * S + i) * D;
            if (!started) {
                for (int64_t d = 0; d < D; ++d) oi[d] = 0.0;
                lse[h * S + i] = -INFINITY;
                continue;
            }
            for (int64_t d = 0; d < D; ++d) oi[d] = acc[d] / l;
            lse[h * S + i] = M_LN2 * (b + log2(l));      /* back to natural log */
        }
        free(acc);
        free(sblk);
    }
    if (stats) { stats[0] = rebases; stats[1] = pmax; stats[2] = steps; }
    return failed ? 2 : 0;
}

/* Exposed for the pins: the 16-bit rounding used by the model above. */
double fa_oracle_round_f16(double x) { return round_to_format(x, 11, -14); }
double fa_oracle_round_bf16(double x) { return round_to_format(x, 8, -126); }
