/*
 * locks.h -- C ABI of the LOCKS sparse long-context decode library (GB300, sm_103a).
 *
 * Method: "LOCKS: Page-Local Compact Key Summaries for Efficient Long-Context
 * Decoding" (J. Hwang, arXiv 2607.24555).  Section references below are to
 * that paper's technical summary:
 *   §2 "Method: LOCKS" -- page-local spectral decomposition, quantisation,
 *      reconstruction and selection (the equation for s_j(q)), group-shared
 *      selection (GQA), implementation notes (full CUDA graph, summaries built
 *      off the decode critical path when a page is finalised);
 *   abstract -- the summary alone gives each page an estimate of its
 *      attention mass (a log-sum-exp); only the highest-ranked pages are
 *      attended, and ranking them touches no cached key or value.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor arguments are DEVICE pointers owned by the caller.  The library
 *    never allocates, frees or synchronises inside the decode entry points, so
 *    a sequence of calls can be captured into a CUDA graph.  Every call is
 *    asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream).
 *    One exception: `out` (the attention result) may also be page-locked host
 *    memory that the device addresses with the same pointer (cudaHostAlloc'd
 *    memory under unified addressing; locks_device_accessible() says whether
 *    a pointer qualifies).  The kernels then store the result straight into
 *    host memory (on a Grace system, over NVLink-C2C), and the caller reads
 *    it once `stream` has completed: no separate device-to-host copy.
 *  - All device pointers must be 16-byte aligned.
 *  - Host-side validation runs before any launch; on failure nothing is
 *    launched and an error code is returned.  A failed launch returns
 *    LOCKS_ERR_CUDA.
 *  - Data-dependent problems found on the device (a block id outside
 *    [0, num_blocks), a sequence longer than its block-table row, a wait that
 *    ran out) never fault: the kernel skips the offending access and ORs a
 *    LOCKS_FLAG_* bit into the status word at the start of `workspace`;
 *    locks_read_status() returns it (that call synchronises `stream`).
 *    Every wait on an mbarrier is bounded (about one second of %globaltimer);
 *    when one runs out the kernel flags LOCKS_FLAG_TIMEOUT and returns.
 *  - Fixed shape: head_dim d = 128, page_size B = 16, group_size G = 4, and
 *    either quantised summaries at rank r = 8 (quant = 1, the method's
 *    records) or unquantised fp32 summaries of rank 1 <= r <= 16 (quant = 0,
 *    a debug and reference configuration: at r = 16 a record reproduces its
 *    page's keys exactly, so s_j is the exact page log-sum-exp).  Other
 *    values return LOCKS_ERR_UNSUPPORTED.
 *
 * Tensor layouts
 * --------------
 *  q            bf16 [batch][H_kv*G][128]; query head h*G+g belongs to KV head h.
 *  k_cache,
 *  v_cache      bf16 [num_blocks][H_kv][16][128]; one physical block holds one
 *               16-token page for every KV head; a page-head is 4096 contiguous
 *               bytes.
 *  block_table  int32 [batch][max_pages]; logical page j of request b lives in
 *               physical block block_table[b][j].
 *  seq_lens     int32 [batch]; L_b = tokens cached for request b INCLUDING the
 *               token being decoded (its K/V already written).  Full pages:
 *               n_b = L_b / 16; the tail page n_b holds t_b = L_b % 16 tokens
 *               (none when t_b = 0) and has no summary yet.
 *  summaries    uint8 [num_blocks][H_kv][784]; record of page-head (blk, h) at
 *               byte (blk*H_kv + h)*784.  Only blocks passed to
 *               locks_build_summaries hold valid records.
 *  scores       fp32 [batch][H_kv][max_pages][G]; s_j for full pages j < n_b.
 *  selected     int32 [batch][H_kv][budget_pages]; logical page indices, sorted
 *               ascending; only the first n_selected[b][h] entries are valid.
 *  n_selected   int32 [batch][H_kv] = min(budget_pages, n_b).
 *  out          fp32 [batch][H_kv*G][128].
 *
 * Summary record (784 bytes per page-head; ~9.6 % of the page-head's 8192 KV
 * bytes, §2 "about 10 % at B = 16, r = 8")
 * ---------------------------------------------------------------------------
 *  The page's 16 keys k_i are centred on mu = mean_i k_i; X = K - mu.  The
 *  top-8 eigenpairs (lambda_k, w_k) of the 16x16 Gram matrix X X^T give the
 *  orthonormal key-space basis V[:,k] = X^T w_k / sqrt(lambda_k) and the token
 *  coefficients c[i,k] = w_k[i] sqrt(lambda_k); directions with
 *  lambda_k <= 1e-6 lambda_1 are zero.  Sign: for each k the coefficient of
 *  largest magnitude over the 16 tokens is positive.  Quantisation is
 *  symmetric with one fp32 scale per tensor: s = max|x| / qmax, code =
 *  round-half-even(x / s) (s = 0 gives codes 0); V: int4 in [-7, 7]
 *  (two's-complement nibbles), mu and c: int8 in [-127, 127].
 *  Byte map (d = 0..127, k = 0..7, i = 0..15):
 *   [0,512)   V code (dim, k): s = dim/16, w = dim%16, hh = w/8, t = (w%8)/2,
 *             e = w%2, p = s/2, sp = s%2, m = 2*sp + hh + 4*e;
 *             byte 64*k + 16*t + 4*p + m/2, high nibble iff m is odd.
 *   [512,640) mu code (dim): byte 512 + 32*t + 4*s + 2*hh + e.
 *   [640,768) c code (i, k): nt = i/8, gid = i%8, tk = k/2, ek = k%2;
 *             byte 640 + 4*(4*gid + tk) + 2*nt + ek.
 *   [768,784) fp32 little-endian: s_V, s_mu, s_c, tail energy
 *             sum_{k>8} lambda_k (diagnostic of §3 Thm. 1; not used by scoring).
 *  The byte map puts each lane's share of a tensor-core fragment in one
 *  contiguous 16/32/4-byte run, so the scorer loads it with single vector loads.
 *
 * Unquantised record (quant = 0, rank r): 528 + 576 r bytes per page-head,
 * fp32 little-endian: [mu: 128][V: 128 x r, V[dim][k] at dim * r + k]
 * [C: 16 x r, c[i][k] at i * r + k][tail energy sum_{k>r} lambda_k, 0, 0, 0];
 * the same centroid, eigenpairs, ranking, sign and zero-floor rules.
 */
#ifndef LOCKS_H
#define LOCKS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t (struct CUstream_st *). */
typedef struct CUstream_st *locks_stream_t;

typedef enum {
  LOCKS_OK = 0,
  LOCKS_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, negative size, ... */
  LOCKS_ERR_UNSUPPORTED = 2,  /* a shape this build does not implement */
  LOCKS_ERR_WORKSPACE = 3,    /* workspace smaller than locks_workspace_bytes */
  LOCKS_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
  LOCKS_ERR_TIMEOUT = 5       /* locks_read_status / locks_noalloc_read_status: the flags
                                 read include LOCKS_FLAG_TIMEOUT (they are still returned) */
} locks_status;

typedef struct {
  int32_t head_dim;      /* d: 128 */
  int32_t page_size;     /* B: 16 */
  int32_t rank;          /* r: 8 (quant = 1) or 1..16 (quant = 0) */
  int32_t num_kv_heads;  /* H_kv >= 1 */
  int32_t group_size;    /* G: 4 query heads per KV head */
  int32_t quant;         /* 1: int4 basis, int8 centroid/coefficients; 0: fp32 */
} locks_cfg;

/* Status-word bits written by the kernels (see locks_read_status). */
#define LOCKS_FLAG_BAD_BLOCK   1u  /* a block id outside [0, num_blocks) was skipped */
#define LOCKS_FLAG_BAD_SEQLEN  2u  /* L_b < 0 or ceil(L_b/16) > max_pages; request skipped */
#define LOCKS_FLAG_TIMEOUT     4u  /* a bounded wait on an mbarrier ran out */
#define LOCKS_FLAG_BAD_SELECT  8u  /* a selected index outside [0, n_b) was skipped */

/* Bytes of one page-head summary record (784 for quant = 1, 528 + 576 r for
 * quant = 0), 0 for an unsupported cfg. */
size_t locks_summary_bytes(const locks_cfg *cfg);

/* Workspace bytes needed by score/select and sparse/dense decode for this
 * batch shape (one workspace may be shared by all calls of a step, used in
 * stream order).  Host only, no CUDA call. */
locks_status locks_workspace_bytes(const locks_cfg *cfg, int32_t batch, int32_t max_pages,
                                   int32_t budget_pages, size_t *bytes);

/* Zero a workspace before its first use (the status word and the merge
 * tickets must start at zero; the kernels keep the tickets at zero after
 * every call).  Enqueues one memset on `stream`. */
locks_status locks_workspace_init(void *workspace, size_t workspace_bytes, locks_stream_t stream);

/* 1 when the current device's kernels can dereference p: device or managed
 * memory, or page-locked host memory whose device pointer equals p (the
 * form `out` may take); 0 otherwise, including NULL and pointers the CUDA
 * runtime does not know (pageable host memory).  Host-side query, no launch
 * and no synchronisation.  The paper has no counterpart: it is a check for
 * callers that hand `out` in host memory. */
int32_t locks_device_accessible(const void *p);

/* Synchronise `stream`, copy the status word to *flags and clear it.
 * Returns LOCKS_ERR_TIMEOUT (with *flags written) when a bounded wait ran
 * out since the last read, LOCKS_OK otherwise. */
locks_status locks_read_status(void *workspace, uint32_t *flags, locks_stream_t stream);

/* Diagnostic of the bounded waits (the paper has no counterpart): one CTA
 * runs the library's bounded mbarrier wait on a barrier that never completes
 * (it waits for two arrivals and gets one), with a limit of limit_us
 * microseconds (1 .. 100000), after issuing one 256-byte bulk copy from `src`
 * (device, 16-byte aligned) into shared memory on a second barrier.  The wait
 * gives up after the limit and ORs LOCKS_FLAG_TIMEOUT into the status word at
 * the start of `workspace`; the kernel then waits for its copy and returns, so
 * the context stays usable.  result (device uint32[4], 16-byte aligned):
 * [0] = 1 if the wait ran out, [1] = 1 if the copy landed, [2] = the sum of
 * the 64 copied 32-bit words, [3] = low bits of the %globaltimer when the wait
 * gave up. */
locks_status locks_check_bounded_wait(const void *src, uint32_t *result, uint32_t limit_us, void *workspace,
                                      size_t workspace_bytes, locks_stream_t stream);

/* Page summary builder, §2 "page-local spectral decomposition" and
 * "quantisation": for each of the n_build physical blocks in block_ids
 * (device int32) and each KV head, read the 16 keys of k_cache and write the
 * 784-byte record described above into `summaries`.  Meant to run when pages
 * are finalised (prefill, or a page crossing), off the decode critical path.
 * Block ids outside [0, num_blocks) are skipped and flagged.  Uses only the
 * status word of `workspace` (workspace may be NULL: no flag is reported). */
locks_status locks_build_summaries(const locks_cfg *cfg, const void *k_cache, int64_t num_blocks,
                                   const int32_t *block_ids, int32_t n_build, void *summaries,
                                   void *workspace, size_t workspace_bytes, locks_stream_t stream);

/* Page-crossing build, §2 "page-local spectral decomposition" ("when a page
 * is finalised") and "implementation" (full CUDA graph): the records of
 * block_ids[0, min(*n_pending, max_pending)), in the same format and to the
 * same accuracy as locks_build_summaries (codes within one of the exact
 * decomposition's; built for latency with a tridiagonal eigensolver, so not
 * bit for bit the bulk builder's), where n_pending points to a device int32
 * that the kernel reads.  One captured
 * graph thus serves every decode step, whatever number of requests crossed a
 * page boundary at that step (at most max_pending, e.g. one per request).
 * Entries at or past *n_pending are not read.  Launch it before
 * locks_decode_step on the same stream so the newly full pages are scored.
 * n_pending must be 4-byte aligned. */
locks_status locks_build_pending(const locks_cfg *cfg, const void *k_cache, int64_t num_blocks,
                                 const int32_t *block_ids, const int32_t *n_pending, int32_t max_pending,
                                 void *summaries, void *workspace, size_t workspace_bytes,
                                 locks_stream_t stream);

/* Scoring pass, §2 "reconstruction and selection" (the s_j(q) equation):
 * for every request b, KV head h and full page j < n_b, read the page's
 * record (and nothing else of the cache) and write, for each query head g of
 * the group, s_j = log sum_i exp((q.mu_j + (V_j^T q).c_i) / sqrt(d)) into
 * `scores` (or into the workspace when scores is NULL). */
locks_status locks_score(const locks_cfg *cfg, const void *q, const void *summaries,
                         int64_t num_blocks, const int32_t *block_table, const int32_t *seq_lens,
                         int32_t batch, int32_t max_pages, float *scores,
                         void *workspace, size_t workspace_bytes, locks_stream_t stream);

/* Selection pass, §2 "reconstruction and selection" and "group-shared
 * selection (GQA)": Z_{b,h,g} = logsumexp over full pages of s_j; share =
 * exp(s_j - Z); the group's table is the mean share over its G query heads;
 * the min(budget_pages, n_b) largest entries (lower page index on ties) are
 * written to selected[b][h][...] in ascending page order and their count to
 * n_selected[b][h].  `scores` must be what locks_score was given.  One
 * thread-block cluster per (b, h) -- 8 CTAs when all of them fit on the GPU
 * at once, else 2 (or 4 or 8 when a CTA's slice of max_pages would exceed
 * 16,384 pages) -- computes Z from the scores and selects by an exact
 * cluster-wide radix select.  Needs max_pages <= 131072,
 * else LOCKS_ERR_UNSUPPORTED. */
locks_status locks_select(const locks_cfg *cfg, const int32_t *seq_lens, int32_t batch,
                          int32_t max_pages, int32_t budget_pages, const float *scores,
                          int32_t *selected, int32_t *n_selected,
                          void *workspace, size_t workspace_bytes, locks_stream_t stream);

/* locks_score followed by locks_select on the same stream. */
locks_status locks_score_select(const locks_cfg *cfg, const void *q, const void *summaries,
                                int64_t num_blocks, const int32_t *block_table,
                                const int32_t *seq_lens, int32_t batch, int32_t max_pages,
                                int32_t budget_pages, float *scores, int32_t *selected,
                                int32_t *n_selected, void *workspace, size_t workspace_bytes,
                                locks_stream_t stream);

/* Sparse paged decode attention, §2 / abstract (only the selected pages are read):
 * for each (b, h) and each of the G query heads of the group,
 * out = softmax(sm_scale * q K^T) V over the tokens of the selected full
 * pages plus the t_b tokens of the open tail page (always attended).  All G
 * heads share each K/V page read.  Split-K over pages with an online-softmax
 * merge.  sm_scale is normally 1/sqrt(128). */
locks_status locks_sparse_decode(const locks_cfg *cfg, const void *q, const void *k_cache,
                                 const void *v_cache, int64_t num_blocks,
                                 const int32_t *block_table, const int32_t *seq_lens,
                                 const int32_t *selected, const int32_t *n_selected,
                                 int32_t batch, int32_t max_pages, int32_t budget_pages,
                                 float sm_scale, float *out, void *workspace,
                                 size_t workspace_bytes, locks_stream_t stream);

/* Selection and sparse attention fused, §2 "Reconstruction and selection",
 * "Group-shared selection (GQA)" and the implementation note that scoring,
 * selection and sparse attention run back to back with no host round trip:
 * the same results as locks_select followed by locks_sparse_decode (it writes
 * `selected`, `n_selected` and `out`), computed by one thread-block cluster of
 * 8 CTAs per (request, KV head) that keeps the selection on chip and merges
 * the split attention through distributed shared memory.  It is launched as a
 * programmatic dependent of the preceding kernel on `stream` (normally
 * locks_score), so its set-up overlaps that kernel's tail.  Needs
 * budget_pages <= 2047 and max_pages <= 131072, else LOCKS_ERR_UNSUPPORTED. */
locks_status locks_select_sparse_decode(const locks_cfg *cfg, const void *q, const void *k_cache,
                                        const void *v_cache, int64_t num_blocks,
                                        const int32_t *block_table, const int32_t *seq_lens,
                                        int32_t batch, int32_t max_pages, int32_t budget_pages,
                                        const float *scores, int32_t *selected, int32_t *n_selected,
                                        float sm_scale, float *out, void *workspace,
                                        size_t workspace_bytes, locks_stream_t stream);

/* One whole LOCKS decode step for a batch: locks_score, then either
 * locks_select_sparse_decode (when batch * num_kv_heads clusters of 8 CTAs
 * fit on the GPU at once and max_pages <= 32768) or locks_select followed by
 * locks_sparse_decode (larger batches, where the cluster kernel would run in
 * many waves, and longer contexts, where its long per-CTA slices cost more).
 * Each kernel after the first is a programmatic dependent of the one before
 * it.  Same results either way; same limits as the fused call. */
locks_status locks_decode_step(const locks_cfg *cfg, const void *q, const void *summaries,
                               const void *k_cache, const void *v_cache, int64_t num_blocks,
                               const int32_t *block_table, const int32_t *seq_lens, int32_t batch,
                               int32_t max_pages, int32_t budget_pages, float sm_scale, float *scores,
                               int32_t *selected, int32_t *n_selected, float *out, void *workspace,
                               size_t workspace_bytes, locks_stream_t stream);

/* The decode step at a page crossing, §2 "page-local spectral decomposition"
 * (a page is summarised when it is finalised) and "implementation" (full CUDA
 * graph): the same results as building, for every request whose current
 * token completed a page (L_b % 16 == 0, page L_b / 16 - 1), that page's
 * record for every KV head into `summaries`, then locks_decode_step.  The
 * build is launched first and the scorer as its programmatic dependent: the
 * scorer streams every other page's record while the build runs and copies
 * the new pages' records only after it has ended.  Requests whose length is
 * not a multiple of 16 build nothing; the pages are derived from seq_lens and
 * the block table on the device, so one captured graph serves any batch.
 * Same arguments, layouts and limits as locks_decode_step (summaries is
 * written). */
locks_status locks_decode_step_crossing(const locks_cfg *cfg, const void *q, void *summaries,
                                        const void *k_cache, const void *v_cache, int64_t num_blocks,
                                        const int32_t *block_table, const int32_t *seq_lens, int32_t batch,
                                        int32_t max_pages, int32_t budget_pages, float sm_scale, float *scores,
                                        int32_t *selected, int32_t *n_selected, float *out, void *workspace,
                                        size_t workspace_bytes, locks_stream_t stream);

/* Dense comparator (the full-cache attention LOCKS is measured against):
 * the same computation over every cached token of each request. */
locks_status locks_dense_decode(const locks_cfg *cfg, const void *q, const void *k_cache,
                                const void *v_cache, int64_t num_blocks,
                                const int32_t *block_table, const int32_t *seq_lens,
                                int32_t batch, int32_t max_pages, float sm_scale, float *out,
                                void *workspace, size_t workspace_bytes, locks_stream_t stream);

/* ---------------------------------------------------------------------------
 * Shared-basis ablation, §3 "impossibility of shared projections": the
 * comparison selector the method is measured against, which scores every page
 * of a KV head through ONE rank-rho basis U (fp32 [H_kv][128][rho], the
 * caller's, e.g. the top principal directions of the head's centred keys;
 * 1 <= rho <= 64) instead of each page's own.  Record per page-head, fp32,
 * 512 + 64 rho bytes: [mu: 128][c: 16 x rho, c[i][k] = U[:,k].(k_i - mu)].
 * Score: s_j = log sum_i exp((q.mu + (U^T q).c_i) / sqrt(d)), written to the
 * same table as locks_score's, so locks_select and locks_sparse_decode run on
 * it unchanged.  Block ids outside the cache are flagged and skipped.
 * ------------------------------------------------------------------------ */
locks_status locks_shared_basis_build(const locks_cfg *cfg, const void *k_cache, int64_t num_blocks,
                                      const int32_t *block_ids, int32_t n_build, const float *basis, int32_t rho,
                                      void *records, void *workspace, size_t workspace_bytes,
                                      locks_stream_t stream);

locks_status locks_shared_basis_score(const locks_cfg *cfg, const void *q, const float *basis, int32_t rho,
                                      const void *records, int64_t num_blocks, const int32_t *block_table,
                                      const int32_t *seq_lens, int32_t batch, int32_t max_pages, float *scores,
                                      void *workspace, size_t workspace_bytes, locks_stream_t stream);

/* ---------------------------------------------------------------------------
 * Context-parallel shards: one request's full pages split over several GPUs.
 *
 * §2 "Reconstruction and selection" / "Group-shared selection (GQA)" normalise
 * each query head's page scores over all of a request's pages, and §4 places
 * the method at 1M+ token contexts.  When a request's pages are split over
 * n_shards GPUs (shard r holds the contiguous logical pages starting at
 * page_offset[b]; only the last shard may hold the open tail page), each shard
 * runs the calls below on its own cache and block table, with shard_lens[b]
 * its own token count in place of seq_lens.  Between them the caller gathers
 * three small results from every shard (an all-gather over any transport:
 * the kernels never wait on another GPU):
 *   1. locks_score (unchanged), then locks_cp_score_pairs -> pairs
 *      float [batch][H_kv][G][2];  gather -> pairs_all [n_shards][...];
 *   2. locks_cp_select_local -> this shard's top-min(budget, n) pages as
 *      candidates: cand_pages int32 [batch][H_kv][budget] (global page
 *      indices, ascending), cand_keys uint32 (same shape; the selection key,
 *      fp32 bits of the page's group-mean share), cand_counts int32
 *      [batch][H_kv];  gather all three over shards;
 *   3. locks_cp_merge_select -> the global top-k restricted to this shard
 *      (local page indices, ascending) in selected / n_selected; then
 *      locks_cp_sparse_decode_partial -> states float [batch][H_kv*G][130]
 *      (per query head: m in log2 units, l, unnormalised o[128]);
 *      gather -> states_all [n_shards][...];  locks_cp_merge_attention -> out.
 * The selection equals the one-GPU selection up to the rounding of Z_g (keys
 * are computed by the same code on every shard; ties go to the lower global
 * page index); the output is attention over the union of the shards'
 * selected pages plus the tail.  n_shards * budget_pages <= 16384.
 * ------------------------------------------------------------------------ */

/* Per (request, KV head, query head): max over the shard's full pages of
 * s_j*log2(e) and the sum of 2^(s_j*log2(e) - max) -> pairs (16-byte aligned).
 * `scores` as given to locks_score (NULL: the workspace's). */
locks_status locks_cp_score_pairs(const locks_cfg *cfg, const int32_t *shard_lens, int32_t batch,
                                  int32_t max_pages, const float *scores, float *pairs, void *workspace,
                                  size_t workspace_bytes, locks_stream_t stream);

/* The shard's local selection with Z_g from every shard's pairs, written as
 * candidates (see above).  page_offset: device int32 [batch]. */
locks_status locks_cp_select_local(const locks_cfg *cfg, const int32_t *shard_lens, const int32_t *page_offset,
                                   int32_t batch, int32_t max_pages, int32_t budget_pages, const float *scores,
                                   const float *pairs_all, int32_t n_shards, int32_t *cand_pages,
                                   uint32_t *cand_keys, int32_t *cand_counts, void *workspace,
                                   size_t workspace_bytes, locks_stream_t stream);

/* The k = min(budget, total candidates) largest candidates of all shards
 * (key descending, lower global page first); this shard's share of them as
 * local page indices, ascending. */
locks_status locks_cp_merge_select(const locks_cfg *cfg, const int32_t *page_offset, int32_t batch,
                                   int32_t budget_pages, int32_t n_shards, int32_t shard,
                                   const int32_t *cand_pages_all, const uint32_t *cand_keys_all,
                                   const int32_t *cand_counts_all, int32_t *selected, int32_t *n_selected,
                                   locks_stream_t stream);

/* locks_sparse_decode over the shard's selected pages (and its tail page, if
 * it holds one), writing the unnormalised state instead of `out`. */
locks_status locks_cp_sparse_decode_partial(const locks_cfg *cfg, const void *q, const void *k_cache,
                                            const void *v_cache, int64_t num_blocks, const int32_t *block_table,
                                            const int32_t *shard_lens, const int32_t *selected,
                                            const int32_t *n_selected, int32_t batch, int32_t max_pages,
                                            int32_t budget_pages, float sm_scale, float *states, void *workspace,
                                            size_t workspace_bytes, locks_stream_t stream);

/* out[b][hq][:] = sum_r 2^(m_r - M) o_r / sum_r 2^(m_r - M) l_r over the
 * shards' states (zero when every shard's l is zero). */
locks_status locks_cp_merge_attention(const locks_cfg *cfg, int32_t batch, int32_t n_shards,
                                      const float *states_all, float *out, locks_stream_t stream);

/* Sparse decode attention without a caller-provided workspace.  The paper
 * has no counterpart: this exists for callers that cannot allocate device
 * memory (an engine that gave all of HBM to its KV-cache pool, a
 * latency-critical path where cudaMalloc would synchronise the device, a host
 * integration with no allocator).  Same computation, arguments, layouts,
 * validation and split-K plan as locks_sparse_decode; the scratch (split
 * partials, merge tickets, status word) is one fixed 8 MiB device array
 * inside the library, resident on every GPU that loads it until exit.
 * Allocates nothing.  The first call in a CUDA context looks up that array's
 * address there (make it before any stream capture); each call clears the
 * merge tickets with one cudaMemsetAsync on `stream`.  Device-side flags
 * (LOCKS_FLAG_*) accumulate in the array's status word until
 * locks_noalloc_read_status reads and clears them.  Calls share the array:
 * calls that overlap on the GPU race.  Returns LOCKS_ERR_WORKSPACE, before
 * any CUDA call, when batch * num_kv_heads exceeds 4025 (request, KV head)
 * units, the most whose partial states fit in 8 MiB. */
locks_status locks_sparse_decode_noalloc(const locks_cfg *cfg, const void *q, const void *k_cache,
                                         const void *v_cache, int64_t num_blocks,
                                         const int32_t *block_table, const int32_t *seq_lens,
                                         const int32_t *selected, const int32_t *n_selected,
                                         int32_t batch, int32_t max_pages, int32_t budget_pages,
                                         float sm_scale, float *out, locks_stream_t stream);

/* Status word of locks_sparse_decode_noalloc, without a workspace: synchronise
 * `stream`, copy the flags accumulated by the calls since the last read to
 * *flags and clear them; LOCKS_ERR_TIMEOUT as for locks_read_status.  The
 * paper has no counterpart (see above). */
locks_status locks_noalloc_read_status(uint32_t *flags, locks_stream_t stream);

/* Static description of a status code. */
const char *locks_status_str(locks_status status);

#ifdef __cplusplus
}
#endif

#endif /* LOCKS_H */
