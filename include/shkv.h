/*
 * shkv.h -- C ABI of libshkv: shared-KV multi-decoder paged decode attention
 * for NVIDIA GB300 (sm_103a).
 *
 * The problem, as the pages state it:
 *   - PrefillShare (Sec. 3.3, Sec. 7; Eqs. 8-9): one frozen base prefill
 *     module writes a single KV cache C_base, held in vLLM PagedAttention
 *     blocks (pages); N task-specific decode modules all consume that one
 *     cache; a returning session runs a partial prefill on its new tokens
 *     only and hands the extended cache on.
 *   - ICaRus (key designs 2 and 3): all decoders share one frozen logical
 *     encoder, so their KV caches are bitwise identical and stored once; the
 *     decoders' queries are concatenated along the head axis and attend the
 *     same KV together, so each KV byte is read once per step instead of once
 *     per model.
 *
 * Conventions for every call:
 *   - All device buffers are caller-owned (the library allocates no device
 *     memory).  Pointers are device pointers unless a parameter says "host".
 *     Device pointers must be 16-byte aligned.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued asynchronously on it; argument errors are
 *     returned synchronously before anything is enqueued.
 *   - bf16 means IEEE bfloat16 bit patterns (uint16_t storage).
 *   - Calls on one pool are not thread-safe; use one host thread per pool.
 *   - Device-side faults never trap: a bad page index, an inconsistent
 *     sequence length or a pipeline wait that runs over its time limit sets a
 *     bit in the pool's error word, the affected data is skipped (zero
 *     contribution), and shkv_check_errors() reports it.
 */
#ifndef SHKV_H
#define SHKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SHKV_OK = 0,
    SHKV_ERR_INVALID_ARG = 1,   /* null / misaligned pointer, bad size, shape mismatch */
    SHKV_ERR_CAPACITY = 2,      /* a sequence would exceed max_pages_per_seq * page_size */
    SHKV_ERR_UNSUPPORTED = 3,   /* outside the supported set (see shkv_decode_attention) */
    SHKV_ERR_CUDA = 4,          /* a CUDA runtime call failed */
    SHKV_ERR_DEVICE = 5         /* shkv_check_errors found device error bits */
} shkv_status;

/* Bits of the device error word. */
#define SHKV_ERRF_PAGE_OOB 0x1u   /* block-table entry outside [0, num_pages) */
#define SHKV_ERRF_SEQ_LEN 0x2u    /* device seq_lens disagrees with the pool's host copy */
#define SHKV_ERRF_TIMEOUT 0x4u    /* a pipeline wait exceeded its time limit */
#define SHKV_ERRF_PIPELINE 0x8u   /* a pipeline slot held a stage other than the one expected */

/* Largest batch a single decode / append call accepts. */
#define SHKV_MAX_BATCH 1024

typedef struct shkv_pool shkv_pool; /* opaque host handle, owns no device memory */

/*
 * Pool description.  The pool is the paged KV cache of PrefillShare Sec. 3.3
 * (vLLM blocks), shared by every decoder (ICaRus key design 2).
 *   k_pages, v_pages  device bf16 [num_pages, num_kv_heads, page_size, head_dim]
 *   block_table       device int32 [max_batch, max_pages_per_seq]; entry
 *                     (b, i) is the physical page of request b's logical page
 *                     i.  The caller fills it; one table serves all decoders.
 *   seq_lens          device int32 [max_batch]; cached tokens per request.
 *                     After creation the pool owns its contents: change it
 *                     only through shkv_append_kv / shkv_pool_set_seq_lens.
 *   error_word        device uint32 (one word), zeroed by shkv_pool_create.
 *   initial_seq_lens  host int32 [max_batch] or NULL (all zero); copied to
 *                     seq_lens and to the pool's host copy at creation.
 */
typedef struct {
    int32_t num_pages;
    int32_t page_size;        /* 16 or 32 tokens */
    int32_t num_kv_heads;
    int32_t head_dim;         /* 64 or 128 */
    int32_t max_batch;
    int32_t max_pages_per_seq;
    void *k_pages;
    void *v_pages;
    int32_t *block_table;
    int32_t *seq_lens;
    uint32_t *error_word;
    const int32_t *initial_seq_lens; /* host, nullable */
} shkv_pool_config;

/*
 * Create a pool handle over caller-owned memory.  Validates the description,
 * builds the TMA descriptors of the K and V pools, writes the initial
 * sequence lengths and zeroes the error word (synchronously, on the current
 * device).  Errors: SHKV_ERR_INVALID_ARG, SHKV_ERR_UNSUPPORTED (page size or
 * head dim), SHKV_ERR_CUDA.  On success *out receives the handle.
 */
shkv_status shkv_pool_create(const shkv_pool_config *cfg, shkv_pool **out);

/* Release the host handle.  Device memory stays with the caller. */
shkv_status shkv_pool_destroy(shkv_pool *pool);

/*
 * Set the cached length of requests [0, batch) from host array `lens`
 * (each in [0, max_pages_per_seq * page_size]).  Updates the pool's host copy
 * and copies to seq_lens on `stream`, then synchronizes `stream`.
 * Errors: SHKV_ERR_INVALID_ARG, SHKV_ERR_CAPACITY, SHKV_ERR_CUDA.
 */
shkv_status shkv_pool_set_seq_lens(shkv_pool *pool, int32_t batch, const int32_t *lens,
                                   void *stream);

/* Copy the pool's host copy of the lengths of requests [0, batch) to host
 * array `lens`.  No device work. */
shkv_status shkv_pool_get_seq_lens(const shkv_pool *pool, int32_t batch, int32_t *lens);

/*
 * Partial-prefill append (PrefillShare Sec. 3.3 / Sec. 7: a cache hit runs
 * prefill on the new tokens only and hands the extended cache on).  For every
 * request b < batch and new token t < n_new_tokens:
 *   pool[block_table[b][(L_b+t)/P], g, (L_b+t)%P, :] = new[b, t, g, :]
 * for K and V and every KV head g, then L_b += n_new_tokens.  A bit-exact
 * copy.  The block table must already map the pages the new tokens land in.
 *   k_new, v_new  device bf16 [batch, n_new_tokens, num_kv_heads, head_dim]
 * Errors: SHKV_ERR_INVALID_ARG; SHKV_ERR_CAPACITY if L_b + n_new_tokens
 * exceeds max_pages_per_seq * page_size; SHKV_ERR_CUDA.  A block-table entry
 * outside the pool sets SHKV_ERRF_PAGE_OOB and that token is not written.
 */
shkv_status shkv_append_kv(shkv_pool *pool, int32_t batch, int32_t n_new_tokens,
                           const void *k_new, const void *v_new, void *stream);

/*
 * Bytes of device workspace shkv_decode_attention needs for this shape: a
 * region of SHKV_COUNT_REGION_BYTES at the front holding the per-(request,
 * KV head) arrival counters of every call, then the split-KV partials.
 */
#define SHKV_COUNT_REGION_BYTES (1u << 20)
shkv_status shkv_decode_workspace_size(const shkv_pool *pool, int32_t batch, int32_t n_models,
                                       int32_t hq_per_model, size_t *bytes);

/*
 * Shared-KV decode attention (ICaRus key design 3 over the PrefillShare
 * paged cache).  The n_models decoders' queries are stacked model-major
 * along the head axis, row r = m * hq_per_model + h; query head h of every
 * decoder uses KV head g = h / (hq_per_model / num_kv_heads).  For each
 * request b < batch and row r:
 *   s_t = scale * <q[b, r, :], K_b[t, g, :]>   for t < L_b (no causal mask)
 *   out[b, r, :] = sum_t softmax(s)_t V_b[t, g, :]
 *   lse_out[b, r] = ln sum_t exp(s_t)
 * where K_b / V_b are read through the shared block table.  Each KV page of
 * each head is read from HBM once for all n_models * group stacked rows.
 * Long contexts are split across SMs (flash-decoding) and the splits merged
 * by log-sum-exp inside the same launch.
 *   q        device bf16 [batch, n_models * hq_per_model, head_dim]
 *   out      device bf16, same shape (round to nearest even from fp32)
 *   lse_out  device fp32 [batch, n_models * hq_per_model], or NULL
 *   workspace, workspace_bytes
 *            device scratch of at least shkv_decode_workspace_size() bytes.
 *            Its counter region (the first SHKV_COUNT_REGION_BYTES) must be
 *            zero before its first use; every call that completes without
 *            device error bits leaves it zero again and writes nothing else
 *            there, so one workspace serves calls of any shape in turn.
 *            Calls sharing one workspace must not overlap on the GPU.
 * Two interchangeable consumers implement the same result: warp-level
 * mma.sync tiles and, for head_dim 128, tcgen05 tiles with the accumulators
 * in tensor memory (tokens along the MMA's M dimension, 128-token stages).
 * shkv_decode_consumer() reports which one a call runs;
 * shkv_pool_set_decode_consumer() names one for a pool where the shape
 * allows it (no call reads the process environment).
 * Supported: batch in [1, SHKV_MAX_BATCH], every L_b >= 1,
 * hq_per_model % num_kv_heads == 0, rows per KV head
 * n_models * hq_per_model / num_kv_heads <= 64,
 * batch * num_kv_heads <= SHKV_COUNT_REGION_BYTES / 4.
 * Errors: SHKV_ERR_INVALID_ARG (null pointers, L_b == 0, shapes),
 * SHKV_ERR_UNSUPPORTED (outside the set above), SHKV_ERR_CUDA.
 */
shkv_status shkv_decode_attention(shkv_pool *pool, int32_t batch, int32_t n_models,
                                  int32_t hq_per_model, const void *q, float scale, void *out,
                                  float *lse_out, void *workspace, size_t workspace_bytes,
                                  void *stream);

/*
 * Causal partial-prefill attention (PrefillShare Sec. 3.3: on a prefix-cache
 * hit the shared prefill module runs only on the new tokens, extending the
 * cached prefix).  Call after shkv_append_kv has put the n_new tokens' K/V
 * into the pool: request b then holds L_b tokens, the last n_new of them new,
 * and new token i (position L_b - n_new + i) attends every key at a position
 * <= its own -- the whole cached prefix and the new tokens causally.
 *   q        device bf16 [batch, n_new, hq_per_model, head_dim] (the prefill
 *            module's query heads; head h uses KV head h / (Hq / Hkv))
 *   out      device bf16, same shape;  lse_out device fp32 [batch, n_new,
 *            hq_per_model] (natural log) or NULL
 * Tensor-core kernel (tcgen05): a tile is floor(128 / G) new tokens x the G
 * query heads of one KV head, stacked on the MMA M dimension; one CTA takes
 * two consecutive tiles of a (request, KV head) and streams its pages once
 * for both, the CTAs ordered longest first.
 * Supported: head_dim 128, page size 16 or 32, G <= 128, batch <=
 * SHKV_MAX_BATCH.  Errors: SHKV_ERR_INVALID_ARG (null / misaligned pointers,
 * a request shorter than n_new), SHKV_ERR_UNSUPPORTED, SHKV_ERR_CUDA; page
 * and length disagreements set the error word as in decode.
 */
shkv_status shkv_prefill_attention(shkv_pool *pool, int32_t batch, int32_t n_new, int32_t hq_per_model,
                                   const void *q, float scale, void *out, float *lse_out, void *stream);

/*
 * Per-decoder unique tails (PrefillShare Sec. 3.3-4 and Eqs. 8-9: decode
 * starts from the shared base cache and each decoder extends it with its own
 * generated-token cache Delta C_t; the shared prefix is stored once, each
 * decoder's tail N times in total).  Decoder m of request b attends the
 * concatenation of the shared prefix (the pool's block table, L_b tokens)
 * and its own tail (the tail table, T_{b,m} tokens, 0 allowed).  Tail pages
 * live in the same page pool.
 */
typedef struct shkv_tails shkv_tails;

typedef struct {
    int32_t max_batch;                 /* requests */
    int32_t n_models;                  /* decoders per request (N) */
    int32_t max_tail_pages;            /* block-table width of one tail */
    int32_t *block_table;              /* device int32 [max_batch, n_models, max_tail_pages], caller-owned */
    int32_t *tail_lens;                /* device int32 [max_batch, n_models], caller-owned */
    const int32_t *initial_tail_lens;  /* host int32 [max_batch * n_models] or NULL (all zero) */
} shkv_tails_config;

/*
 * Tails over `pool`'s pages.  Writes the initial lengths to tail_lens and
 * shares (and clears) the pool's error word.  The pool must outlive the
 * tails.  Errors: SHKV_ERR_INVALID_ARG, SHKV_ERR_CAPACITY (an initial length
 * above max_tail_pages * page_size), SHKV_ERR_CUDA.
 */
shkv_status shkv_tails_create(shkv_pool *pool, const shkv_tails_config *cfg, shkv_tails **out);
shkv_status shkv_tails_destroy(shkv_tails *tails);

/* Host-side lengths of the first `batch` requests' tails, [batch * n_models]
 * (set: also copied to the device on `stream`, which is synchronised). */
shkv_status shkv_tails_set_lens(shkv_tails *tails, int32_t batch, const int32_t *tail_lens, void *stream);
shkv_status shkv_tails_get_lens(const shkv_tails *tails, int32_t batch, int32_t *tail_lens);

/*
 * Append n_new_tokens to every decoder's tail (its generated tokens' K/V):
 * k_new / v_new device bf16 [batch, n_models, T, Hkv, d]; same rules and
 * errors as shkv_append_kv, per (request, decoder).
 */
shkv_status shkv_tails_append(shkv_tails *tails, int32_t batch, int32_t n_new_tokens, const void *k_new,
                              const void *v_new, void *stream);

/* Workspace bytes for shkv_decode_attention_tails (its counter region zero
 * before the first use, as for shkv_decode_attention; kept between calls). */
shkv_status shkv_decode_tails_workspace_size(const shkv_pool *pool, const shkv_tails *tails, int32_t batch,
                                             int32_t hq_per_model, size_t *bytes);

/*
 * shkv_decode_attention where every decoder also attends its own tail:
 * out[b, m*Hq + h] = softmax attention over [shared prefix ++ tail(b, m)].
 * q / out / lse_out as in shkv_decode_attention with n_models = the tails'
 * n_models.  One pass over the pages: a small kernel lays out each request's
 * unit (its shared pages, then each decoder's tail pages, read from the
 * device block and tail tables with the host copies of the lengths), then
 * the decode kernel streams every unit once for all N*G stacked rows, a tail
 * page being attended by its own decoder's G rows only.  The layout kernel
 * runs while the previous kernel of `stream` is still running (one warp per
 * request, beside that kernel's CTAs).  It writes its tables at an offset of
 * `workspace` whose bytes miss every buffer that this library's previous
 * call on `stream` reads or writes (that call's workspace bytes, queries,
 * outputs, tables, appended K/V, merge inputs), under whatever pointers; when
 * no offset does, or the library has no record of a call on `stream`, it
 * first waits for the previous kernel.  It reads the block and tail tables
 * without waiting for that kernel.  So a kernel enqueued on `stream` right
 * before this call that lets programmatic dependents start
 * (griddepcontrol.launch_dependents / cudaTriggerProgrammaticLaunchCompletion)
 * must by then be done writing those tables and done with any bytes of
 * `workspace`; copies, kernels launched without programmatic stream
 * serialization and this library's own kernels are fine.  Supported:
 * batch * n_models <= SHKV_MAX_BATCH, n_models <= 254, rest as
 * shkv_decode_attention.  Errors as shkv_decode_attention (the device copies
 * of the lengths are not compared: SHKV_ERRF_SEQ_LEN is not raised here).
 */
shkv_status shkv_decode_attention_tails(shkv_pool *pool, shkv_tails *tails, int32_t batch, int32_t hq_per_model,
                                        const void *q, float scale, void *out, float *lse_out, void *workspace,
                                        size_t workspace_bytes, void *stream);

/*
 * Page bookkeeping for the shared pool (host only, no CUDA): refcounted
 * prefix-cache pages and transfer pages.
 *
 * PrFaaS (hybrid prefix cache pool): prefix-cache blocks are reused within
 * the cluster and must be block-aligned and completely filled; transfer-cache
 * blocks serve one cross-cluster transfer and are dropped when it is done.
 * ICaRus key design 2: all task models share the frozen base encoder, so a
 * prefix cached while serving one agent is a hit for every later agent.
 *
 * A full block (page_size tokens) is keyed by a hash chain over token ids
 * with the parent block's hash, and matched only if the parent and the token
 * ids are equal.  Pages whose reference count drops to zero stay indexed
 * (idle, least recently used first) until a new allocation needs a page.
 * The caller fills the pages it is handed (prefill / handoff /
 * shkv_append_kv) and writes them into block tables; several requests may
 * reference one page.
 */
typedef struct shkv_pages shkv_pages;

typedef struct {
    int32_t num_pages;
    int32_t free_pages;          /* never used, or released private/transfer pages */
    int32_t cached_idle_pages;   /* indexed prefix pages no request references */
    int32_t referenced_pages;    /* pages with a reference count > 0 */
    int32_t indexed_blocks;      /* full blocks in the prefix index */
    int32_t transfer_pages;      /* transfer pages currently allocated */
    int64_t block_lookups;       /* full blocks looked up by acquire */
    int64_t block_hits;          /* of which were cached */
} shkv_pages_info;

/* A manager for pages 0 .. num_pages-1 of page_size tokens. */
shkv_status shkv_pages_create(int32_t num_pages, int32_t page_size, shkv_pages **out);
shkv_status shkv_pages_destroy(shkv_pages *pages);

/*
 * Pages for a request whose prompt is tokens[0 .. n_tokens): the longest
 * prefix of full blocks found in the index is reused (reference +1 each),
 * the remaining ceil(n_tokens / page_size) - hits pages are new private
 * pages (reference 1) taken from the free pages, else from the idle cached
 * pages in LRU order (dropped from the index).
 *   pages            host int32 [max_pages]: receives the request's pages
 *   n_cached_tokens  receives hits * page_size (tokens already in the pool)
 * Errors: SHKV_ERR_INVALID_ARG; SHKV_ERR_CAPACITY (more than max_pages
 * blocks, or not enough pages: nothing is kept).
 */
shkv_status shkv_pages_acquire(shkv_pages *pages, const int32_t *tokens, int32_t n_tokens, int32_t *out_pages,
                               int32_t max_pages, int32_t *n_cached_tokens);

/*
 * After the request's pages hold its K/V: enter its full blocks (not a
 * partial last block) into the prefix index.  Blocks already indexed (this
 * request's hits, or the same content published by another request) are
 * left as they are.  Errors: SHKV_ERR_INVALID_ARG (a page not referenced,
 * or a transfer page).
 */
shkv_status shkv_pages_publish(shkv_pages *pages, const int32_t *tokens, int32_t n_tokens, const int32_t *req_pages);

/* Drop one reference from each page (a finished request or transfer). */
shkv_status shkv_pages_release(shkv_pages *pages, const int32_t *req_pages, int32_t n_pages);

/* n pages for one transfer (reference 1, never indexed). */
shkv_status shkv_pages_alloc_transfer(shkv_pages *pages, int32_t n_pages, int32_t *out_pages);

shkv_status shkv_pages_stats(const shkv_pages *pages, shkv_pages_info *info);
shkv_status shkv_pages_refcount(const shkv_pages *pages, int32_t page, int32_t *count);

/* Consumer kernels of shkv_decode_attention. */
#define SHKV_CONSUMER_AUTO (-1)
#define SHKV_CONSUMER_MMA_SYNC 0
#define SHKV_CONSUMER_TCGEN05 1

/*
 * Name the consumer kernel that shkv_decode_attention and
 * shkv_decode_attention_tails run on this pool: SHKV_CONSUMER_AUTO (the
 * default set at creation: tcgen05 for head_dim 128 and 16 to 64 rows per KV
 * head, mma.sync otherwise), SHKV_CONSUMER_MMA_SYNC or SHKV_CONSUMER_TCGEN05.
 * Both compute the same result; naming one serves tests and measurements.
 * tcgen05 is taken only where the shape allows it (head_dim 128, at most 64
 * rows per KV head); elsewhere mma.sync runs.  Host-only, no device work.
 * Errors: SHKV_ERR_INVALID_ARG (null pool, unknown value).
 */
shkv_status shkv_pool_set_decode_consumer(shkv_pool *pool, int32_t consumer);

/*
 * Which consumer shkv_decode_attention would run on this pool for n_models
 * decoders of hq_per_model query heads, given the pool's consumer setting:
 * *consumer = SHKV_CONSUMER_MMA_SYNC or SHKV_CONSUMER_TCGEN05.  Host-only; no
 * device work.  Errors: SHKV_ERR_INVALID_ARG (null pointers, counts < 1),
 * SHKV_ERR_UNSUPPORTED (hq_per_model % num_kv_heads != 0 or more than 64
 * rows per KV head).
 */
shkv_status shkv_decode_consumer(const shkv_pool *pool, int32_t n_models, int32_t hq_per_model,
                                 int32_t *consumer);

/*
 * Log-sum-exp merge of split-KV partials (the flash-decoding reduction for
 * long contexts).  For every (b, row):
 *   M = max_s lse_part[s, b, row];  w_s = exp(lse_part[s, b, row] - M)
 *   out[b, row, :] = sum_s w_s o_part[s, b, row, :] / sum_s w_s
 *   lse_out[b, row] = M + ln sum_s w_s
 * Partials with lse = -inf carry no weight; a row whose partials are all
 * -inf gets out = 0 and lse = -inf.
 *   o_part   device fp32 [n_splits, batch, rows, head_dim] (each partial
 *            already normalised by its own softmax sum)
 *   lse_part device fp32 [n_splits, batch, rows] (natural log)
 *   out      device bf16 [batch, rows, head_dim]
 *   lse_out  device fp32 [batch, rows], or NULL
 * head_dim must be a multiple of 4.  Errors: SHKV_ERR_INVALID_ARG, SHKV_ERR_CUDA.
 */
shkv_status shkv_splitkv_merge(int32_t n_splits, int32_t batch, int32_t rows, int32_t head_dim,
                               const float *o_part, const float *lse_part, void *out,
                               float *lse_out, void *stream);

/*
 * Synchronize `stream`, then read and clear the pool's device error word.
 * *flags receives the SHKV_ERRF_* bits.  Returns SHKV_ERR_DEVICE if any bit
 * was set, SHKV_OK otherwise (SHKV_ERR_CUDA if the stream reported an error).
 */
shkv_status shkv_check_errors(shkv_pool *pool, void *stream, uint32_t *flags);

/*
 * Self-test of the bounded waits (no counterpart on the pages): enqueues on
 * `stream` one small kernel whose only waiting thread waits, with the wait
 * every kernel of this library uses, for a barrier that nothing completes.
 * After the wait's limit (2 s of device time) it gives up, sets
 * SHKV_ERRF_TIMEOUT in the pool's error word and the kernel exits; it reads
 * and writes nothing else.  shkv_check_errors then reports the bit.  For
 * checking on the device at hand that a stalled pipeline ends with an error
 * status instead of a hang, and that the context stays usable after it.
 * Errors: SHKV_ERR_INVALID_ARG for a null pool, SHKV_ERR_CUDA if the launch
 * fails.
 */
shkv_status shkv_selftest_bounded_wait(shkv_pool *pool, void *stream);

/*
 * Host-only view of how shkv_decode_attention divides work (no device
 * needed).  The (request, KV head, page) chunks, ordered request-major, are
 * cut into `num_ctas` contiguous, non-empty ranges, one per persistent CTA,
 * of equal estimated cost for the consumer that runs them; a (request, head)
 * whose pages straddle a cut is split and merged by log-sum-exp.  Cost, in
 * tokens of one KV head streamed: each (request, head) pays its ring stages
 * whole (128 tokens on tcgen05, min(page_size, 32) on mma.sync) plus a fixed
 * amount; on tcgen05 a cut inside a (request, head) adds the second piece's
 * segment work and both pieces' partials and merge, and the fixed amounts
 * grow with the stacked rows n_models * hq_per_model / num_kv_heads.
 *   seq_lens      host int32 [batch] (each >= 1)
 *   n_models, hq_per_model   as in shkv_decode_attention
 *   consumer      SHKV_CONSUMER_MMA_SYNC or SHKV_CONSUMER_TCGEN05: the kernel
 *                 the plan is for (shkv_decode_consumer names the one a pool
 *                 would run)
 *   max_ctas      upper bound on CTAs (normally the SM count)
 *   cta_begin     host int64 [max_ctas + 1] or NULL; receives the first
 *                 chunk of every CTA and, at [num_ctas], the total chunk count
 *   num_ctas      receives the CTA count used
 *   num_splits    receives the number of (request, head) units that are split
 * Errors: SHKV_ERR_INVALID_ARG (null num_ctas, unknown consumer, counts < 1,
 * batch above SHKV_MAX_BATCH, a length < 1, page_size above 255),
 * SHKV_ERR_UNSUPPORTED (hq_per_model % num_kv_heads != 0, more than 64 rows
 * per KV head, more than INT32_MAX chunks).
 */
shkv_status shkv_plan_decode(int32_t batch, const int32_t *seq_lens, int32_t page_size,
                             int32_t num_kv_heads, int32_t n_models, int32_t hq_per_model,
                             int32_t consumer, int32_t max_ctas, int64_t *cta_begin,
                             int32_t *num_ctas, int32_t *num_splits);

/*
 * Bytes of the library's static device scratch used by
 * shkv_decode_attention_noalloc.
 */
#define SHKV_NOALLOC_SCRATCH_BYTES (8u << 20)

/*
 * shkv_decode_attention without a caller-provided workspace.  The pages have
 * no counterpart to this call: it exists for callers that cannot call
 * cudaMalloc -- code hosted inside a framework that owns all device memory
 * through its own allocator or a fixed memory budget and offers no
 * allocation hook, or code on a latency-critical path where cudaMalloc's
 * implicit device synchronisation is not acceptable.
 *
 * Same arguments, layouts, results and errors as shkv_decode_attention, minus
 * the workspace.  The split-KV scratch is a file-scope static device array of
 * SHKV_NOALLOC_SCRATCH_BYTES (8 MiB) that every GPU which loads the library
 * holds until the process exits.
 *   - The call allocates nothing: no cudaMalloc / cudaFree / allocating
 *     library routine.  Once every argument check has passed, it clears the
 *     scratch's arrival counters with cudaMemsetAsync on `stream`, then
 *     launches; a rejected call enqueues nothing.
 *   - Set-up: the first call in a CUDA context (the current device, which
 *     must be the pool's device) looks up the scratch's device address with
 *     cudaGetSymbolAddress and caches it under the context's unique ID, so a
 *     new context (after cudaDeviceReset, or one the caller creates) gets
 *     its own lookup and never a stale address.  Make the first call in a
 *     context before any stream capture in it.
 *   - All calls on a device share the one array, which keeps the last call's
 *     contents; calls whose executions overlap on the GPU (different streams
 *     without ordering) race on it and give wrong results.
 * Errors: those of shkv_decode_attention; SHKV_ERR_UNSUPPORTED if the scratch
 * this shape needs exceeds SHKV_NOALLOC_SCRATCH_BYTES (that is
 * shkv_decode_workspace_size less its counter region, plus this call's
 * batch * num_kv_heads counters rounded up to 256 bytes: the scratch's
 * counters are cleared by every call); SHKV_ERR_INVALID_ARG if the current
 * device is not the pool's.
 */
shkv_status shkv_decode_attention_noalloc(shkv_pool *pool, int32_t batch, int32_t n_models,
                                          int32_t hq_per_model, const void *q, float scale,
                                          void *out, float *lse_out, void *stream);

/*
 * Divide a decode batch among world_size replicas (host only, no CUDA).
 * PrefillShare's framework scope runs decode in a data-parallel pool of
 * GPUs; the decode step shards by request with no exchange step, so each
 * replica holds and streams only the pages of the requests it owns.
 * Requests are taken longest first (by pages, ceil(seq_lens[b] / page_size),
 * ties by index) and each goes to the replica with the fewest pages so far
 * (ties to the lower rank): every replica computes the same assignment from
 * the same lengths.  The heaviest replica holds at most the mean plus the
 * largest single request.
 *   seq_lens    host int32 [batch], each >= 0
 *   owner       host int32 [batch]: receives the replica of each request
 *   rank_pages  host int64 [world_size] or NULL: receives each replica's
 *               pages (unique KV bytes = pages * page_size * num_kv_heads *
 *               head_dim * 4)
 * Errors: SHKV_ERR_INVALID_ARG (null pointers, negative length,
 * page_size < 1, world_size < 1).
 */
shkv_status shkv_partition_requests(int32_t batch, const int32_t *seq_lens, int32_t page_size,
                                    int32_t world_size, int32_t *owner, int64_t *rank_pages);

/* Static description of a status code. */
const char *shkv_status_string(shkv_status status);

#ifdef __cplusplus
}
#endif

#endif /* SHKV_H */
