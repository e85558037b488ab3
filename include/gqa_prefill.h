/*
 * gqa_prefill.h -- C ABI of libgqa_prefill.so: fused grouped-query
 * flash-attention prefill for gpt-oss-style layers on sm_103a.
 *
 * The operation (what one call computes) follows two pages:
 *   ROCm/hip-ep PR #622, "perf(gqa): support sliding windows in the fused
 *   flash prefill kernel": the sink folded into the softmax denominator
 *   (sink-fold commit), the smooth_softmax "+1" mode (sink-gate and
 *   sink-harness commits), the per-row window bound and the KV-loop start
 *   tile (window-in-v5 commit and the PR body "Why" / "A NaN the window
 *   introduces"), and the decline-instead-of-miscompute rule (sink-fold
 *   commit);
 *   sgl-project/sglang PR #34468, "gfx950 SWA prefix trim": one KV loop over
 *   [cached prefix | extend] with a BLOCK_N-aligned floor (commit 2), and the
 *   window-bounded prefix layout (commit 1).
 *
 * Definition.  Sequence b has P_b = prefix_lens[b] cached keys followed by
 * E_b = cu_seqlens_q[b+1] - cu_seqlens_q[b] new tokens.  Query row i of the
 * sequence sits at position P_b + i and, for query head h, attends to key j
 * of KV head h / (Hq/Hkv) iff j <= P_b + i and (window <= 0 or
 * j >= P_b + i - window + 1): window counts the keys a row sees, itself
 * included, so window = 1 is "itself only".  With s_j = scale * <q, k_j>
 * over the kept keys and x the sink logit (sinks[h] in per-head mode, 0 in
 * smooth_softmax mode, absent otherwise):
 *     out = sum_j e^{s_j} v_j / (sum_j e^{s_j} + e^{x})
 *     lse = log(sum_j e^{s_j} + e^{x})        (natural log)
 * The sink is a natural-log logit and is NOT multiplied by scale.  A row
 * with no kept key (impossible for real rows with consistent metadata)
 * gets out = 0 and lse = -inf.
 *
 * Layouts (all row-major, dense, caller-owned device memory):
 *   q, out  [total_q,  Hq,  d]   16-bit (dtype), 16-byte aligned base
 *   k, v    [total_kv, Hkv, d]   same dtype; sequence b's keys are rows
 *           kv_indptr[b] .. kv_indptr[b+1]-1, ordered [prefix | extend], so
 *           kv_indptr[b+1] - kv_indptr[b] == P_b + E_b.  For a windowed
 *           layer the caller may hand only the last min(prefix, window)
 *           prefix rows (window-bounded layout): positions are relative to
 *           the first supplied key, and the result is the same.
 *   cu_seqlens_q  int32 [num_seqs+1], cu[0] = 0, non-decreasing, cu[B] <= total_q
 *   prefix_lens   int32 [num_seqs]
 *   kv_indptr     int32 [num_seqs+1], kv_indptr[B] <= total_kv
 *   sinks         fp32 [Hq] or NULL
 *   lse           fp32 [total_q, Hq] or NULL
 * Every row of k and v in [0, total_kv) must hold finite values: the kernel
 * reads whole key tiles and relies on masked probabilities being exact zeros.
 *
 * Ownership and asynchrony: the library allocates nothing per call and keeps
 * only a process-wide launch-configuration cache.  A call validates its host
 * arguments, enqueues one kernel on `stream` (a cudaStream_t; NULL = legacy
 * default stream) and returns without synchronising; it never copies device
 * data to the host.  Rows of out/lse that belong to no sequence are not
 * written.
 *
 * Errors: invalid host arguments return GQA_ERR_INVALID before any launch;
 * shapes the kernels do not implement return GQA_ERR_UNSUPPORTED (the call
 * declines rather than computing something else); a failed launch returns
 * GQA_ERR_CUDA.  Device metadata is checked by the kernel itself: if
 * cu_seqlens_q / prefix_lens / kv_indptr are inconsistent the kernel writes
 * nothing and raises GQA_DEV_BAD_METADATA in the device status word, read
 * with gqa_prefill_get_device_status().  Every wait inside the kernel is
 * bounded; a wait that runs out raises GQA_DEV_TIMEOUT instead of hanging.
 */
#ifndef GQA_PREFILL_H
#define GQA_PREFILL_H

#include <stddef.h>
#include <stdint.h>

/* Symbols of the C ABI; the library is built with hidden visibility otherwise. */
#if defined(__GNUC__)
#define GQA_API __attribute__((visibility("default")))
#else
#define GQA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of q, k, v and out. */
enum { GQA_F16 = 0, GQA_BF16 = 1 };

/* Host-side return codes. */
enum {
    GQA_OK = 0,
    GQA_ERR_INVALID = -1,
    GQA_ERR_UNSUPPORTED = -2,
    GQA_ERR_CUDA = -3
};

/* Device status word bits (gqa_prefill_get_device_status). */
enum {
    GQA_DEV_TIMEOUT = 1,       /* a bounded wait inside a kernel ran out */
    GQA_DEV_BAD_METADATA = 2   /* cu_seqlens_q / prefix_lens / kv_indptr inconsistent */
};

/*
 * gqa_flash_prefill -- the fused prefill (see the definition above).
 *   num_seqs     B >= 0.  The kernel keeps each launch's sequence metadata in
 *                shared memory, 512 sequences at most: a call with more runs
 *                as ceil(B / 512) launches, in stream order, over consecutive
 *                groups of 512 sequences.
 *   total_q      rows of q/out (>= cu_seqlens_q[B]); 0 means no work
 *   total_kv     rows of k/v (>= kv_indptr[B])
 *   max_seqlen_q optional host hint, max_b E_b (0 = unknown); only used to
 *                pick a launch configuration, never to bound work
 *   Hq, Hkv      query / KV heads, Hq % Hkv == 0; G = Hq/Hkv must divide 128
 *   d            head dim: 64, 128 or 256
 *   dtype        GQA_F16 or GQA_BF16
 *   scale        multiplier of q.k (> 0, finite), usually 1/sqrt(d)
 *   window       <= 0: causal only; else keys (pos - window, pos]
 *   sinks        per-head logits or NULL; smooth_softmax must then be 0
 *   smooth_softmax nonzero: +1 in the denominator (sinks must be NULL)
 * Returns GQA_OK or a negative GQA_ERR_* code.
 */
GQA_API int gqa_flash_prefill(const void* q, const void* k, const void* v,
                      const int32_t* cu_seqlens_q, const int32_t* prefix_lens,
                      const int32_t* kv_indptr, int num_seqs, int total_q,
                      int total_kv, int max_seqlen_q, int Hq, int Hkv, int d,
                      int dtype, float scale, int window, const float* sinks,
                      int smooth_softmax, void* out, float* lse, void* stream);

/*
 * gqa_flash_prefill_masked -- gqa_flash_prefill with a custom mask ANDed
 * into the causal and window conditions: one more condition on a key, which
 * can only remove keys (sgl-project/sglang PR #34468, "gfx950 SWA prefix
 * trim": the custom mask combined with a sliding window, the EAGLE
 * target-verify route of commit 1, and the PR body's note that custom-mask
 * and causal conjuncts can only empty a tile further, so the loop floor is
 * unchanged).
 *
 *   custom_mask       device uint32 words, 4-byte aligned: per sequence a
 *                     bitmap over its extend keys.  Row i (0 <= i < E_b) of
 *                     sequence b occupies words mask_indptr[b] + i * W_b ..
 *                     + W_b - 1, W_b = ceil(E_b / 32); extend key j' (key
 *                     P_b + j' of the sequence) is kept for row i only if bit
 *                     j' % 32 of word j' / 32 is set.  Prefix keys are not
 *                     covered by the bitmap (only the causal and window
 *                     conditions apply to them); bits above the row's own
 *                     position are ignored (causality removes those keys).
 *   mask_indptr       device int32 [num_seqs + 1]: mask_indptr[b + 1] -
 *                     mask_indptr[b] == E_b * W_b, mask_indptr[0] >= 0.
 *   total_mask_words  words in custom_mask (>= mask_indptr[num_seqs]).
 *
 * A row left with no key gets out = 0 and lse = -inf, as in
 * gqa_flash_prefill.  Inconsistent mask metadata raises
 * GQA_DEV_BAD_METADATA like the other metadata.  Head dims, dtypes, sink
 * modes, windows and KV layouts as gqa_flash_prefill (the contiguous KV
 * layout only); the key tile is 128 (d = 64, full attention) or 64.
 * Returns as gqa_flash_prefill; GQA_ERR_INVALID also for a NULL or
 * misaligned mask.
 */
GQA_API int gqa_flash_prefill_masked(const void* q, const void* k, const void* v,
                                     const int32_t* cu_seqlens_q, const int32_t* prefix_lens,
                                     const int32_t* kv_indptr, int num_seqs, int total_q,
                                     int total_kv, int max_seqlen_q, int Hq, int Hkv, int d,
                                     int dtype, float scale, int window, const float* sinks,
                                     int smooth_softmax, const uint32_t* custom_mask,
                                     const int32_t* mask_indptr, long long total_mask_words,
                                     void* out, float* lse, void* stream);

/*
 * gqa_flash_prefill_paged -- the same operation as gqa_flash_prefill with K
 * and V held in a page pool, the way serving stacks hand over a cached prefix
 * (the kv_indices / window_kv_indices page tables of SGLang PR #34468).
 *
 *   k_pages, v_pages   device [num_pages, page_size, Hkv, d], q's dtype,
 *                      16-byte aligned.
 *   kv_page_indptr     device int32 [num_seqs + 1]: the pages of sequence b
 *                      are kv_page_indices[kv_page_indptr[b] ..
 *                      kv_page_indptr[b+1]), in key order; there must be
 *                      exactly ceil((prefix_lens[b] + E_b) / page_size).
 *   kv_page_indices    device int32 [num_page_entries], page numbers in
 *                      [0, num_pages).
 *   page_size          tokens per page: a multiple of 8 that divides, or is
 *                      divided by, the kernel's key tile of 64 or 128 (every
 *                      power of two from 8 qualifies); else GQA_ERR_UNSUPPORTED.
 *
 * Key j of sequence b is slot j % page_size of page
 * kv_page_indices[kv_page_indptr[b] + j / page_size]; prefix_lens[b] counts
 * the prefix keys the pages hold (the whole prefix, or its last
 * min(prefix, window) keys for a window-bounded table), exactly as the
 * contiguous layout.  Other arguments, layouts and return codes as
 * gqa_flash_prefill.  A page count that disagrees with the lengths is
 * reported through GQA_DEV_BAD_METADATA with nothing written; a page number
 * outside the pool raises GQA_DEV_BAD_METADATA as well, and the rows of that
 * call are then unspecified.
 */
GQA_API int gqa_flash_prefill_paged(const void* q, const void* k_pages,
                                    const void* v_pages, const int32_t* cu_seqlens_q,
                                    const int32_t* prefix_lens,
                                    const int32_t* kv_page_indptr,
                                    const int32_t* kv_page_indices,
                                    int num_page_entries, int page_size,
                                    int num_pages, int num_seqs, int total_q,
                                    int max_seqlen_q, int Hq, int Hkv, int d,
                                    int dtype, float scale, int window,
                                    const float* sinks, int smooth_softmax,
                                    void* out, float* lse, void* stream);

/* num_splits value selecting the balanced split (see below). */
#define GQA_SPLITS_BALANCED (-1)

/*
 * gqa_flash_prefill_splitkv -- the same operation as gqa_flash_prefill, with
 * each work unit's key tiles divided into num_splits contiguous ranges
 * processed by separate CTAs, for calls whose units would not fill the GPU
 * (short query chunks over long cached prefixes).  Each range produces an
 * fp32 partial (O relative to its own running maximum, the maximum, the
 * denominator); a second kernel combines the partials of a unit with the
 * log-sum-exp merge and folds the sink in once, the partial-result combine
 * that SGLang PR #34468 ("gfx950 SWA prefix trim") uses for its
 * context-parallel path.  The result equals the unsplit call up to rounding.
 *
 * With num_splits = GQA_SPLITS_BALANCED the call is one kernel whose
 * resident CTAs take equal shares of all the call's key tiles (the units
 * laid end to end in the order they are dealt), so that no CTA idles while
 * others finish a last wave: for calls whose units do not divide evenly over
 * the CTAs (a 512-token chunk's 256 units on 304 resident CTAs).  A unit that
 * share boundaries cut runs as pieces on consecutive CTAs; each piece writes
 * an fp32 partial and counts itself with an atomic, and the piece that
 * completes the count merges the unit's partials (the same log-sum-exp merge,
 * in a fixed order, so the result is the same run to run) and writes the
 * rows.  No CTA waits on another.  Declined (GQA_ERR_UNSUPPORTED) when one
 * launch has more query tiles than the kernel's shared-memory scratch holds
 * (about 16,000 at d = 64) or more than 2^31 key tiles in all.
 *
 *   num_splits       0: the library's choice (splits only when the units fill
 *                    less than half the resident CTAs), else 1..16; 1 is the
 *                    unsplit kernel and needs no workspace;
 *                    GQA_SPLITS_BALANCED: the balanced split.
 *   workspace        device memory owned by the caller, 256-byte aligned, at
 *                    least the size gqa_prefill_splitkv_workspace() reports
 *                    for the same shapes and num_splits; only scratch (its
 *                    contents before and after the call are meaningless: the
 *                    balanced split's count words carry a per-launch tag, and
 *                    words with another tag count as zero), and must not be
 *                    shared by calls that may run concurrently.
 *   workspace_bytes  its size.
 *
 * Other arguments, layouts and return codes as gqa_flash_prefill; a missing
 * or too small workspace returns GQA_ERR_INVALID before any launch.  Two
 * kernels are enqueued on `stream` (one for the balanced split).
 */
GQA_API int gqa_flash_prefill_splitkv(const void* q, const void* k, const void* v,
                              const int32_t* cu_seqlens_q,
                              const int32_t* prefix_lens, const int32_t* kv_indptr,
                              int num_seqs, int total_q, int total_kv,
                              int max_seqlen_q, int Hq, int Hkv, int d, int dtype,
                              float scale, int window, const float* sinks,
                              int smooth_softmax, void* out, float* lse,
                              int num_splits, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * gqa_flash_prefill_splitkv_noalloc -- gqa_flash_prefill_splitkv without a
 * caller workspace: the partials live in a 32 MiB (33,554,432-byte) array of
 * device memory defined at file scope in the library, so the call allocates
 * nothing.  The paper has no counterpart; the entry point exists for callers
 * that may not allocate device memory.
 *
 *   num_splits  as gqa_flash_prefill_splitkv (0 = the library's choice).
 *
 * Arguments are validated exactly as gqa_flash_prefill_splitkv does, and with
 * the same return codes (empty work is GQA_OK only after that validation).
 * The plan that launches is the plan whose workspace layout is checked:
 * shapes needing more than the array (gqa_prefill_splitkv_workspace for the
 * same arguments) return GQA_ERR_UNSUPPORTED before any launch.  Nothing in
 * the array has to start at zero: every value the merge reads is written
 * earlier in the same call.  The array is one per device and process: calls
 * that overlap in time on a device (other streams, other host threads) race
 * on it, so the caller must order them.  The first splitting call on a
 * device looks up the array's device address (again after a device reset
 * creates a new context); make that first call before any stream capture.
 * GQA_ERR_CUDA if the address cannot be obtained.
 */
GQA_API int gqa_flash_prefill_splitkv_noalloc(const void* q, const void* k, const void* v,
                                              const int32_t* cu_seqlens_q,
                                              const int32_t* prefix_lens,
                                              const int32_t* kv_indptr, int num_seqs,
                                              int total_q, int total_kv, int max_seqlen_q,
                                              int Hq, int Hkv, int d, int dtype, float scale,
                                              int window, const float* sinks,
                                              int smooth_softmax, void* out, float* lse,
                                              int num_splits, void* stream);

/*
 * Host only: the split count gqa_flash_prefill_splitkv will use for these
 * shapes and num_splits (0 = the library's choice) in *splits_used, and the
 * workspace it needs in *bytes (0 when the call does not split).  For
 * GQA_SPLITS_BALANCED, *splits_used is GQA_SPLITS_BALANCED and *bytes covers
 * two partial tiles per resident CTA plus 32 bytes per work unit.  Returns
 * GQA_OK, GQA_ERR_INVALID or GQA_ERR_UNSUPPORTED as gqa_prefill_plan.
 */
GQA_API int gqa_prefill_splitkv_workspace(int num_seqs, int total_q, int max_seqlen_q,
                                  int Hq, int Hkv, int d, int dtype, int window,
                                  int num_splits, int* splits_used,
                                  size_t* bytes);

/*
 * Launch plan of a call with these shapes (host only, no device access).
 * A work unit is (sequence, KV head, query positions): the kernel's 128-row
 * MMA tile packs the G query heads of one KV head over 128 / G query
 * positions, a unit holds q_tiles such tiles (rows_per_unit = q_tiles * 128
 * / G positions) that walk the same keys in tiles of block_n, so every K/V
 * tile brought on chip serves q_tiles * 128 rows.
 */
typedef struct {
    int rows_per_unit;  /* query positions per unit (128 / G) */
    int block_n;        /* keys per KV tile */
    int kv_stages;      /* K/V shared-memory ring depth */
    int ctas_per_sm;    /* resident CTAs per SM the launch assumes */
    int grid;           /* CTAs launched (persistent) */
    int max_units;      /* upper bound on unit records: Hkv * (ceil(total_q/rows) + B'),
                           B' = min(B, 512), times the launches ceil(B / 512) */
    int q_tiles;        /* 128-row query tiles per unit: 1, or 2 (one CTA per SM) */
} gqa_prefill_plan_t;

GQA_API int gqa_prefill_plan(int num_seqs, int total_q, int max_seqlen_q, int Hq,
                     int Hkv, int d, int dtype, int window,
                     gqa_prefill_plan_t* plan);

/*
 * gqa_flash_prefill_debug -- same computation as gqa_flash_prefill, and each
 * work unit also writes one record of 8 int32 into unit_log (device memory,
 * capacity max_units records from gqa_prefill_plan; caller pre-fills it,
 * e.g. with -1) at the unit's index:
 *   b, g, q0, kv_lo, n_tiles, n_masked, cta, order
 * kv_lo / n_tiles are the key tiles the unit walked (kv_lo relative to the
 * sequence's first key), n_masked how many of them needed the per-element
 * mask, cta the CTA that ran it and order its position in that CTA's list.
 * With more than 512 sequences, launch i (sequences from 512 i on) writes its
 * records from record i * (max_units / launches) on, and its b counts from
 * that launch's first sequence.
 */
GQA_API int gqa_flash_prefill_debug(const void* q, const void* k, const void* v,
                            const int32_t* cu_seqlens_q,
                            const int32_t* prefix_lens, const int32_t* kv_indptr,
                            int num_seqs, int total_q, int total_kv,
                            int max_seqlen_q, int Hq, int Hkv, int d, int dtype,
                            float scale, int window, const float* sinks,
                            int smooth_softmax, void* out, float* lse,
                            void* stream, int32_t* unit_log);

/*
 * Force the KV tile size for later calls in this process (0 restores the
 * configuration cache's choice).  Valid values: 64, 96 or 128; 96 exists for
 * d = 64 only and d = 256 allows 64 only (a call whose d has no kernel for
 * the forced size returns GQA_ERR_UNSUPPORTED).  Returns GQA_OK or
 * GQA_ERR_INVALID.  Meant for tests and tuning.
 */
GQA_API int gqa_prefill_force_block_n(int block_n);

/*
 * Force the number of 128-row query tiles per work unit for later calls in
 * this process (0 restores the configuration cache's choice): 1, or 2 (two
 * query tiles walk the same key tiles, so each K/V tile loaded serves 256
 * rows; one CTA per SM with a deeper K/V ring).  2 exists for block_n 64 and
 * 128 at d = 64 and block_n 64 at d = 128; a call whose shape has no such
 * kernel returns GQA_ERR_UNSUPPORTED.  Returns GQA_OK or GQA_ERR_INVALID.
 * Meant for tests and tuning.
 */
GQA_API int gqa_prefill_force_q_tiles(int q_tiles);

/*
 * Launch-configuration tuning.  The configuration cache is keyed on (d, a
 * power-of-two bucket of max_seqlen_q, Hq, G, windowed, dtype), never on the
 * KV length.  With tuning on (this call, or GQA_PREFILL_TUNE=1 in the
 * environment before the first call), the first call for an untuned key times
 * every candidate tile size on the caller's stream (without the sink) and
 * keeps the fastest (candidates: block_n 64, 96, 128 with one query tile per
 * unit and 64, 128 with two, where the head dim has the kernel); that call
 * synchronises its stream, and tuning is skipped
 * while the stream is being captured.  GQA_PREFILL_TUNE_DEBUG=1 prints the
 * timings.  enable: 0 or 1.  Returns GQA_OK or GQA_ERR_INVALID.
 */
GQA_API int gqa_prefill_set_tuning(int enable);

/* Forget every cached configuration (tuned or default).  Returns GQA_OK. */
GQA_API int gqa_prefill_clear_config_cache(void);

/*
 * The cached configuration for a call with these shapes: *block_n = 0 (and
 * *q_tiles = 0) if the key has no entry yet; *tuned = 1 if the entry came
 * from a timed sweep.  q_tiles may be NULL.
 */
GQA_API int gqa_prefill_config_block_n(int total_q, int max_seqlen_q, int Hq, int Hkv,
                               int d, int dtype, int window, int* block_n,
                               int* q_tiles, int* tuned);

/*
 * Failure-detection self-test: launches one thread that waits, through the
 * same bounded wait the prefill kernel uses, on a barrier nothing completes.
 * The wait gives up after timeout_ms (1..10000), records GQA_DEV_TIMEOUT in
 * the device status word and returns; the call synchronises `stream`, then
 * reads and clears the status word into *status (expected GQA_DEV_TIMEOUT).
 * The CUDA context stays usable afterwards.
 */
GQA_API int gqa_prefill_selftest_timeout(int timeout_ms, void* stream, int* status);

/*
 * Read and clear the device status word of the current device (bits
 * GQA_DEV_*).  Synchronises the device first.  Returns GQA_OK or
 * GQA_ERR_CUDA; *status receives the bits.
 */
GQA_API int gqa_prefill_get_device_status(int* status);



/*
 * gqa_prefill_get_stream_status -- the same status word, read without a
 * device-wide synchronisation: a one-thread kernel enqueued on `stream`
 * takes the word and clears it in one atomic exchange, and the call waits
 * for `stream` only.  *status then holds every bit raised by kernels that
 * completed before that point of `stream` (in particular all earlier calls
 * on `stream`), and possibly bits from kernels still running on other
 * streams; no bit is lost between the read and the clear.  Up to 64 host
 * threads may read concurrently.  Returns GQA_OK, GQA_ERR_INVALID for a NULL
 * status, or GQA_ERR_CUDA.
 */
GQA_API int gqa_prefill_get_stream_status(void* stream, int* status);

/* Call flag: the metadata arrays are ready (see gqa_prefill_set_call_flags). */
#define GQA_FLAG_METADATA_READY 1u

/*
 * Flags for the prefill calls made later by the calling host thread (until
 * changed; 0 at thread start).  Not an operation of the pages: a launch
 * detail of this library.
 *
 * GQA_FLAG_METADATA_READY: the caller guarantees that the metadata arrays a
 * call reads (cu_seqlens_q, prefix_lens, kv_indptr or kv_page_indptr,
 * mask_indptr) are not written by any kernel that may still be running when
 * the call's kernel starts, for example because they were uploaded once per
 * batch, before the layers' kernels.  The kernels are launched with
 * programmatic dependent launch and may start while the previous kernel in
 * the stream finishes: with this flag, a kernel reads and checks the
 * metadata and plans its work before it waits for that kernel, instead of
 * after (measured on the 16k prefill step: 2.4% faster).  Everything else
 * (q, k, v, page tables, masks, sinks) is still read after the wait, and
 * nothing is written before it.  Breaking the guarantee can give wrong
 * results without any error.
 *
 * Returns GQA_OK, or GQA_ERR_INVALID for unknown flag bits (flags unchanged).
 */
GQA_API int gqa_prefill_set_call_flags(unsigned int flags);

/* The calling host thread's call flags. */
GQA_API unsigned int gqa_prefill_get_call_flags(void);

/* Static text for a GQA_* return code. */
GQA_API const char* gqa_prefill_status_string(int code);

/* Library version, e.g. "0.1.0". */
GQA_API const char* gqa_prefill_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GQA_PREFILL_H */
