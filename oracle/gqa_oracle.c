/*
 * gqa_oracle.c -- CPU oracle for fused grouped-query flash-attention prefill.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain definition that the
 * CUDA path is checked against.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load it.  It shares no code, header, table
 * or helper with the CUDA library, and the CUDA library never calls it.
 *
 * Sources (web pages this follows):
 *   [HIPEP]  ROCm/hip-ep PR #622, "perf(gqa): support sliding windows in the
 *            fused flash prefill kernel" (includes the attention-sinks commits).
 *   [SGL]    sgl-project/sglang PR #34468, "gfx950 SWA prefix trim".
 *
 * What is computed (the plain definition; the fused kernel reaches the same
 * result by skipping provably empty tiles and by an online softmax, see
 * [SGL] commit 1 "bit-identical" and the "Numerics" section):
 *
 *   For sequence b with P = prefix_lens[b] cached keys and E = cu[b+1]-cu[b]
 *   new queries, its keys/values live at rows kv_indptr[b] .. +P+E-1 of k/v,
 *   ordered [prefix | extend].  Query row i (0 <= i < E) sits at position
 *   pos = P + i.  Query head h reads KV head h / (Hq/Hkv).
 *
 *   1. score s_j = scale * <q[row,h,:], k[base+j,g,:]> for EVERY key j in
 *      [0, P+E)  (the full row is materialised, masked keys included);
 *   2. explicit mask: key j is kept iff j <= pos (causal) and, when a window
 *      w > 0 is given, j >= pos - w + 1 ([HIPEP] window commit: the per-row
 *      lower bound is the one the decomposed causal mask kernel uses, so a
 *      row sees exactly w keys including itself; window = 1 means "itself
 *      only", [HIPEP] window-harness commit);
 *   3. sink-augmented softmax: an extra logit x joins the denominator only
 *      ([HIPEP] sink-fold commit): x = sinks[h] (natural-log logit, NOT
 *      multiplied by scale) in per-head mode, x = 0 in smooth_softmax mode
 *      (the "+1" of the third sink mode, [HIPEP] sink-harness commit), and no
 *      extra term otherwise;
 *         m   = max(max_{kept} s_j, x)     (x included only for stability)
 *         z   = sum_{kept} exp(s_j - m) + [x present] exp(x - m)
 *         out = sum_{kept} exp(s_j - m) * v[base+j,g,:] / z
 *         lse = m + log(z)
 *   4. a row with no kept key gets out = 0 and lse = -inf ([HIPEP] sink-fold
 *      commit: such a row is skipped and keeps a clamped denominator).
 *
 *   Optional custom mask (gqa_oracle_prefill_masked): one more condition on
 *   a key, ANDed with the causal and window conditions of step 2 ([SGL]
 *   PR body: custom-mask and causal conjuncts can only empty a tile
 *   further; the custom mask combined with a sliding window is the EAGLE
 *   target-verify route of [SGL] commit 1).  The mask is a bitmap over each
 *   sequence's extend keys: extend key P + j' is kept for extend row i only
 *   if bit j' of row i is set; the prefix keys are not covered by it.
 *   Layout: 32-bit words, row i of sequence b at words
 *   mask_indptr[b] + i*W .. + W - 1 with W = ceil(E / 32), bit j' % 32 of
 *   word j' / 32.
 *
 * Precision: every input is the exact value of the caller's 16-bit number,
 * widened to double; all arithmetic is double (the pages' own references
 * accumulate in fp32; double is at least as exact).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Mask predicate of step 2 (causal + optional window). */
static int oracle_keep(long pos, long j, int window)
{
    if (j > pos) return 0;                       /* causal */
    if (window > 0 && j < pos - window + 1) return 0; /* window lower bound */
    return 1;
}

/* Custom-mask condition (see above): 1 for a prefix key or without a mask,
 * else bit (j - P) of row i of sequence b's bitmap. */
static int oracle_custom_keep(const uint32_t* mask, const int32_t* mask_indptr, int b,
                              long E, long P, long i, long j)
{
    if (mask == NULL || j < P) return 1;
    const long jp = j - P;
    const long W = (E + 31) / 32;
    const uint32_t word = mask[(long)mask_indptr[b] + i * W + jp / 32];
    return (int)((word >> (jp % 32)) & 1u);
}

/* Reports how many threads the oracle will use (for the CPU-baseline line). */
int gqa_oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Checks the ragged-batch metadata: cu[0] = 0, non-decreasing, each
 * sequence's KV span equals prefix + extend and stays inside total_kv. */
static int oracle_check_meta(const int32_t* cu, const int32_t* prefix,
                             const int32_t* kv_indptr, int num_seqs,
                             long total_q, long total_kv)
{
    if (num_seqs < 0) return -1;
    if (num_seqs == 0) return 0;
    if (cu[0] != 0) return -1;
    for (int b = 0; b < num_seqs; ++b) {
        long E = (long)cu[b + 1] - cu[b];
        if (E < 0 || prefix[b] < 0) return -1;
        if ((long)kv_indptr[b + 1] - kv_indptr[b] != (long)prefix[b] + E) return -1;
        if (kv_indptr[b] < 0 || kv_indptr[b + 1] > total_kv) return -1;
    }
    if (cu[num_seqs] > total_q) return -1;
    return 0;
}

/*
 * gqa_oracle_prefill -- steps 1-4 above for every (sequence, query head,
 * query row), or only for the token rows whose row_select entry is nonzero
 * (row_select may be NULL = all rows).  Unselected rows of out/lse are left
 * untouched.
 *
 *   q   [total_q,  Hq,  d]  double
 *   k,v [total_kv, Hkv, d]  double
 *   out [total_q,  Hq,  d]  double      lse [total_q, Hq] double (may be NULL)
 *   sinks [Hq] double or NULL; smooth nonzero selects the "+1" mode.
 * Returns 0, or -1 on inconsistent arguments.
 */
int gqa_oracle_prefill_masked(const double* q, const double* k, const double* v,
                              const int32_t* cu_seqlens_q, const int32_t* prefix_lens,
                              const int32_t* kv_indptr, int num_seqs, long total_q,
                              long total_kv, int Hq, int Hkv, int d, double scale,
                              int window, const double* sinks, int smooth,
                              const uint8_t* row_select, double* out, double* lse,
                              const uint32_t* custom_mask, const int32_t* mask_indptr);

int gqa_oracle_prefill(const double* q, const double* k, const double* v,
                       const int32_t* cu_seqlens_q, const int32_t* prefix_lens,
                       const int32_t* kv_indptr, int num_seqs, long total_q,
                       long total_kv, int Hq, int Hkv, int d, double scale,
                       int window, const double* sinks, int smooth,
                       const uint8_t* row_select, double* out, double* lse)
{
    return gqa_oracle_prefill_masked(q, k, v, cu_seqlens_q, prefix_lens, kv_indptr, num_seqs,
                                     total_q, total_kv, Hq, Hkv, d, scale, window, sinks,
                                     smooth, row_select, out, lse, NULL, NULL);
}

/*
 * gqa_oracle_prefill_masked -- gqa_oracle_prefill with the optional custom
 * mask (custom_mask and mask_indptr both NULL: no mask).  mask_indptr
 * [num_seqs+1] must step by E_b * ceil(E_b / 32) words per sequence.
 */
int gqa_oracle_prefill_masked(const double* q, const double* k, const double* v,
                              const int32_t* cu_seqlens_q, const int32_t* prefix_lens,
                              const int32_t* kv_indptr, int num_seqs, long total_q,
                              long total_kv, int Hq, int Hkv, int d, double scale,
                              int window, const double* sinks, int smooth,
                              const uint8_t* row_select, double* out, double* lse,
                              const uint32_t* custom_mask, const int32_t* mask_indptr)
{
    if (Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv != 0) return -1;
    if (sinks != NULL && smooth) return -1;
    if (oracle_check_meta(cu_seqlens_q, prefix_lens, kv_indptr, num_seqs,
                          total_q, total_kv) != 0)
        return -1;
    if ((custom_mask == NULL) != (mask_indptr == NULL)) return -1;
    if (mask_indptr != NULL) {
        if (num_seqs > 0 && mask_indptr[0] < 0) return -1;
        for (int b = 0; b < num_seqs; ++b) {
            const long E = (long)cu_seqlens_q[b + 1] - cu_seqlens_q[b];
            if ((long)mask_indptr[b + 1] - mask_indptr[b] != E * ((E + 31) / 32)) return -1;
        }
    }
    const int G = Hq / Hkv;
    const long n_pairs = (long)num_seqs * Hq;

#pragma omp parallel
    {
        double* s = NULL;
        long s_cap = 0;
        double* acc = (double*)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 1)
        for (long bh = 0; bh < n_pairs; ++bh) {
            const int b = (int)(bh / Hq);
            const int h = (int)(bh % Hq);
            const int g = h / G;
            const long P = prefix_lens[b];
            const long E = (long)cu_seqlens_q[b + 1] - cu_seqlens_q[b];
            const long L = P + E;
            const long base = kv_indptr[b];
            if (L > s_cap) {
                free(s);
                s = (double*)malloc(sizeof(double) * (size_t)L);
                s_cap = L;
            }
            const int has_x = (sinks != NULL) || smooth;
            const double x = (sinks != NULL) ? sinks[h] : 0.0;
            for (long i = 0; i < E; ++i) {
                const long row = cu_seqlens_q[b] + i;
                if (row_select != NULL && !row_select[row]) continue;
                const long pos = P + i;
                const double* qr = q + ((size_t)row * Hq + h) * d;
                /* step 1: the full score row */
                for (long j = 0; j < L; ++j) {
                    const double* kr = k + ((size_t)(base + j) * Hkv + g) * d;
                    double dot = 0.0;
                    for (int t = 0; t < d; ++t) dot += qr[t] * kr[t];
                    s[j] = scale * dot;
                }
                /* step 2 + 3: masked, sink-augmented softmax */
                int any = 0;
                double m = -INFINITY;
                for (long j = 0; j < L; ++j) {
                    if (!oracle_keep(pos, j, window)) continue;
                    if (!oracle_custom_keep(custom_mask, mask_indptr, b, E, P, i, j)) continue;
                    if (!any || s[j] > m) m = s[j];
                    any = 1;
                }
                double* o = out + ((size_t)row * Hq + h) * d;
                if (!any) { /* step 4 */
                    for (int t = 0; t < d; ++t) o[t] = 0.0;
                    if (lse) lse[(size_t)row * Hq + h] = -INFINITY;
                    continue;
                }
                if (has_x && x > m) m = x;
                double z = 0.0;
                for (int t = 0; t < d; ++t) acc[t] = 0.0;
                for (long j = 0; j < L; ++j) {
                    if (!oracle_keep(pos, j, window)) continue;
                    if (!oracle_custom_keep(custom_mask, mask_indptr, b, E, P, i, j)) continue;
                    const double p = exp(s[j] - m);
                    z += p;
                    const double* vr = v + ((size_t)(base + j) * Hkv + g) * d;
                    for (int t = 0; t < d; ++t) acc[t] += p * vr[t];
                }
                if (has_x) z += exp(x - m);
                for (int t = 0; t < d; ++t) o[t] = acc[t] / z;
                if (lse) lse[(size_t)row * Hq + h] = m + log(z);
            }
        }
        free(s);
        free(acc);
    }
    return 0;
}

/*
 * gqa_oracle_tile_census -- the tile bookkeeping a tiled kernel must reach,
 * derived from the mask predicate itself and not from any floor formula.
 *
 * A work unit is (sequence b, KV head g, query tile t) covering the query
 * positions q0 = t*rows .. min(q0+rows, E)-1 of sequence b (all G query heads
 * of the group share these positions, so the mask does not depend on the
 * head).  Keys are cut into tiles [n0, n0+block_n) with n0 a multiple of
 * block_n counted from the start of the sequence's KV ([SGL] commit 2: one
 * loop over prefix and extend together).
 *
 * For each unit, with a tile "live" when some (real row, key) pair in it is
 * kept, and "masked" when some (real row, key) pair in it is not kept:
 *   kv_lo    = block_n * (index of the first live tile)
 *   n_tiles  = last live tile - first live tile + 1
 *   n_masked = number of masked tiles among those n_tiles
 * A kernel that walks exactly [kv_lo, kv_lo + n_tiles*block_n) never visits a
 * tile holding no kept element below the window ([SGL] commit 1: the loop
 * floor; [HIPEP] window commit: start at the first tile any row can reach)
 * and needs the per-element mask only on the n_masked tiles.
 *
 * Key intervals are used instead of a per-key loop: for real row pos the kept
 * keys are exactly [lo(pos), pos] with lo = max(0, pos-w+1) (or 0 without a
 * window), so a tile holds a kept key of that row iff it intersects that
 * interval, and a non-kept key iff it is not contained in it.
 *
 * Records are written in (b, g, t) order, 6 int32 each:
 *   b, g, q0, kv_lo, n_tiles, n_masked.
 * Returns the number of units, or -1 if max_units is too small / bad args.
 */
long gqa_oracle_tile_census(const int32_t* cu_seqlens_q, const int32_t* prefix_lens,
                            int num_seqs, int Hkv, int rows, int block_n,
                            int window, int32_t* records, long max_units)
{
    if (rows <= 0 || block_n <= 0 || Hkv <= 0 || num_seqs < 0) return -1;
    long n = 0;
    for (int b = 0; b < num_seqs; ++b) {
        const long P = prefix_lens[b];
        const long E = (long)cu_seqlens_q[b + 1] - cu_seqlens_q[b];
        const long L = P + E;
        const long n_key_tiles = (L + block_n - 1) / block_n;
        for (int g = 0; g < Hkv; ++g) {
            for (long q0 = 0; q0 < E; q0 += rows) {
                const long q_end = (q0 + rows < E) ? q0 + rows : E;
                long first = -1, last = -1;
                for (long tile = 0; tile < n_key_tiles; ++tile) {
                    const long n0 = tile * block_n, n1 = n0 + block_n - 1;
                    for (long i = q0; i < q_end; ++i) {
                        const long pos = P + i;
                        long lo = (window > 0) ? pos - window + 1 : 0;
                        if (lo < 0) lo = 0;
                        if (n0 <= pos && n1 >= lo) {
                            if (first < 0) first = tile;
                            last = tile;
                            break;
                        }
                    }
                }
                long masked = 0;
                for (long tile = first; tile >= 0 && tile <= last; ++tile) {
                    const long n0 = tile * block_n, n1 = n0 + block_n - 1;
                    for (long i = q0; i < q_end; ++i) {
                        const long pos = P + i;
                        long lo = (window > 0) ? pos - window + 1 : 0;
                        if (lo < 0) lo = 0;
                        if (n0 < lo || n1 > pos) { ++masked; break; }
                    }
                }
                if (n >= max_units) return -1;
                int32_t* r = records + 6 * n;
                r[0] = b;
                r[1] = g;
                r[2] = (int32_t)q0;
                r[3] = (first < 0) ? 0 : (int32_t)(first * block_n);
                r[4] = (first < 0) ? 0 : (int32_t)(last - first + 1);
                r[5] = (int32_t)masked;
                ++n;
            }
        }
    }
    return n;
}
