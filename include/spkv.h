/*
 * spkv.h -- C ABI of the GB300 (sm_103a) block-sparse paged-KV decode library.
 *
 * One decode step over a paged, head-major KV cache runs as
 *
 *   paged_kv_append      write the new token's K/V rows, refresh the pooled-key summaries
 *   score_blocks         block scores from the pooled keys (two-stage pooling)
 *   decode_append_score  a decode step's paged_kv_append + score_blocks in one launch
 *   select_topk          per-KV-head top-k pages: eviction-head budget k_e + query budget k_q
 *   resident_setdiff     selected pages that are not resident (swap-in list)
 *   lru_bucket_update    64-bucket LRU recency update and victim choice
 *   select_resident_update  select_topk + resident_setdiff + lru_bucket_update in one call
 *   retrieve_pages       swap-in of the missing pages from a host pool into resident slots
 *   sparse_decode_attn_slots  attention reading the selected pages from their resident slots
 *   sparse_decode_attn   split-K flash decoding over the selected pages
 *   lazy_rope_decode_attn  the same with deferred RoPE (query rotated once per document)
 *   lazy_rope_decode_attn_docs  the same over shared cached documents, scheduled by document
 *   lazy_rope_prefill_attn a tile of new query rows over cached documents (tcgen05)
 *   lazy_rope_prefill_step   the same plus the new rows' causal attention among themselves
 *   lazy_alibi_prefill_attn  the prefill step for models with ALiBi position biases
 *   attn_column_scores   PyramidKV-style key scores of a prompt's last rows (tcgen05)
 *   attn_column_scores_lse  the same from row log-sum-exps the attention already produced
 *   score_blocks_dir, sparse_decode_attn_dir, retrieve_pages_dir  the same calls through a
 *                        two-level page directory (spkv_pagemap_* manages one)
 *
 * Sources (web pages, cited by title and section):
 *   [NOSA] "NOSA: Native and Offloadable Sparse Attention", sections "Method 1: the NOSA
 *          algorithm" and "Method 2: the NOSI system".
 *   [Spin] "Unifying Sparse Attention with Hierarchical Memory for Scalable Long-Context LLM
 *          Serving", section 2A "Unified partition abstraction" and 2B "Dynamic,
 *          locality-aware KV management".
 *   [Lazy] "LazyAttention", sections "Core idea: deferred positional encoding",
 *          "Technical implementation 2. Decoding" and "Mathematical equivalence".
 *   [FA]   "How KV sparsity achieves 1.5x acceleration for vLLM" (Novita AI), section
 *          "2. Attention modification".
 *
 * Conventions for every entry point
 *   - Pointers named "device" are CUDA device memory owned by the caller (for example
 *     allocated by PyTorch); the library never frees them.  Host pointers are marked "host".
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream) and
 *     never synchronise, except spkv_get_device_error.
 *   - Argument errors are detected on the host before any launch and return SPKV_EINVAL.
 *     A failed launch returns SPKV_ECUDA.  No C++ exception crosses this boundary.
 *   - Malformed *device* data (a page id, physical page or slot out of range) never faults:
 *     the kernel skips the entry and sets a bit in the handle's device error word, which
 *     spkv_get_device_error reports (bits SPKV_DEVERR_*).
 *   - Fixed shapes: head_dim 128, page 64 tokens, pooling sub-block 16 tokens, group size
 *     G = Hq / Hk with 1 <= G <= 16.  Other values return SPKV_EUNSUPPORTED.
 *   - bf16 is IEEE bfloat16; accumulation is fp32.
 *   - A handle serves one stream at a time; calls on one handle must not overlap on the GPU.
 *   - "unit" = one (request b, kv head h) pair, u = b * Hk + h.
 */
#ifndef SPKV_H_
#define SPKV_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum spkv_status {
  SPKV_OK = 0,
  SPKV_EINVAL = -1,        /* bad argument, detected on the host, nothing launched */
  SPKV_ENOMEM = -2,        /* device or host allocation failed (create only) */
  SPKV_ECUDA = -3,         /* a CUDA call or kernel launch failed */
  SPKV_EDEVICE = -4,       /* the device error word was non-zero (spkv_get_device_error) */
  SPKV_ETIMEOUT = -5,      /* a bounded wait inside a kernel gave up (never in a correct run) */
  SPKV_EUNSUPPORTED = -6   /* shape outside the fixed sizes listed above */
};

/* Bits of the device error word. */
#define SPKV_DEVERR_PAGE_ID 1u      /* logical page id outside [0, np_max) or past seq_len */
#define SPKV_DEVERR_PHYS 2u         /* physical page id outside [0, n_phys_pages) */
#define SPKV_DEVERR_SLOT 4u         /* resident slot / doc slot outside its table */
#define SPKV_DEVERR_ORDER 8u        /* selected list not strictly ascending, or duplicate resident id */
#define SPKV_DEVERR_CAPACITY 16u    /* more missing pages than evictable slots */
#define SPKV_DEVERR_TIMEOUT 32u     /* a bounded intra-CTA wait gave up (reported as SPKV_ETIMEOUT) */

typedef struct spkv_cache* spkv_cache_t; /* opaque, library-owned */

/* Description of a paged KV cache.  All buffers are caller-owned device memory.
 *   k_pool, v_pool : bf16 [n_kv_heads][n_phys_pages][64][128]; one page of one head is
 *                    16 KiB contiguous ([Spin] 2B "per-head physical pages").  16-byte aligned.
 *   ksum           : fp32 [n_kv_heads][n_phys_pages][4][128]; per page and sub-block, the sum
 *                    of the valid keys (the library writes it; mean = ksum / count).  With
 *                    ksum_bf16 = 1 it is bf16 of the same shape instead: the fp32 sum, formed in
 *                    the same order, rounded once to bf16 (half the bytes for score_blocks to
 *                    read; [Spin] 2C / cheaper scoring at long context).
 *   page_cnt       : int32 [n_phys_pages]; valid tokens held by each physical page.  Read by
 *                    paged_kv_create, updated by paged_kv_append.
 *   max_units      : the largest B * n_kv_heads any call on this handle will use (sizes the
 *                    split-K workspace); 0 means 4096, larger than 4096 is SPKV_EINVAL.
 * ksum and page_cnt may both be NULL: the handle then has no summaries (for a pool of resident
 * slots that is attended but never scored, see retrieve_pages); score_blocks and
 * paged_kv_append on it return SPKV_EINVAL.
 */
typedef struct {
  int32_t n_kv_heads;
  int32_t head_dim;     /* must be 128 */
  int32_t page_tokens;  /* must be 64 */
  int32_t subblock;     /* must be 16 */
  int64_t n_phys_pages;
  void* k_pool;
  void* v_pool;
  void* ksum;
  int32_t* page_cnt;
  int32_t max_units;
  int32_t ksum_bf16;    /* 0: fp32 summaries; 1: bf16 summaries */
} spkv_desc;

/* Creates a handle for the pool described by *desc (the struct is copied; the buffers are
 * not) and builds the pooled-key summaries of every physical page from page_cnt:
 *   ksum[h][p][j][:] = sum of K[h][p][t][:] over t in [16j, min(16j+16, page_cnt[p])).
 * [NOSA] "Method 1", block-wise implementation (first pooling stage: sub-block means);
 * [NOSA] "Method 2: NOSI", kernel fusion (pooling is produced when K is written, not per step).
 * Allocates the handle, a split-K workspace and the device error word (SPKV_ENOMEM on
 * failure).  *out receives the handle.  The summary build is enqueued on `stream`. */
int paged_kv_create(const spkv_desc* desc, void* stream, spkv_cache_t* out);

/* Appends n_rows tokens.  Row i writes K and V of all heads at token slot tok_in_page[i]
 * of physical page phys_page[i]:
 *   k_new, v_new : device bf16 [n_rows][n_kv_heads][128]
 *   phys_page, tok_in_page : device int32 [n_rows]
 * then sets page_cnt[p] = max(page_cnt[p], tok + 1) and recomputes the touched sub-block
 * sums from the pool in a fixed order (bitwise the same as paged_kv_create).  Rows of one
 * call must name distinct (page, token) slots; pages are filled in token order.
 * Out-of-range ids are skipped (SPKV_DEVERR_PHYS / SPKV_DEVERR_PAGE_ID).
 * [NOSA] "Method 2: NOSI", kernel fusion; [NOSA] "Method 1", block-wise implementation. */
int paged_kv_append(spkv_cache_t cache, const int32_t* phys_page, const int32_t* tok_in_page,
                    const void* k_new, const void* v_new, int n_rows, void* stream);

/* Block scores, [NOSA] "Method 1", block-wise implementation (two-stage pooling: mean over
 * each 16-token sub-block, max over the 4 sub-blocks of the page) and dual selection
 * (query-aware part).  For unit (b, h) and every complete page p before the local page
 * l_b = (seq_len[b] - 1) / 64:
 *   scores[b][h][p] = max_j (sum_g q[b][h*G+g]) . ksum[h][page_table[b][p]][j] / (16 sqrt(128))
 * i.e. the sub-block scores of the G query heads of the group are summed before the max.
 * Entries p >= l_b are -inf.
 *   q          : device bf16 [B][Hq][128], 8-byte aligned
 *   page_table : device int32 [B][np_max], physical page of each logical page
 *   seq_len    : device int32 [B], tokens in each request's context (>= 1)
 *   scores     : device fp32 [B][n_kv_heads][np_max] (output) */
int score_blocks(spkv_cache_t cache, const void* q, int B, int Hq, const int32_t* page_table,
                 int np_max, const int32_t* seq_len, float* scores, void* stream);

/* A decode step's append and scoring in one launch: exactly paged_kv_append of each request's new
 * row at position seq_len[b] - 1 (physical page page_table[b][(seq_len[b] - 1) / 64], row
 * (seq_len[b] - 1) % 64, all kv heads), followed by score_blocks with the same arguments.  The two
 * run concurrently, which is exact because score_blocks never reads a request's local page (the
 * one holding position seq_len[b] - 1).  Requires that no two requests share that physical page
 * (the usual copy-on-write rule for the page being written).  [NOSA] "Method 2: NOSI", kernel
 * fusion: pooling produced where K is written.
 *   k_new, v_new : device bf16 [B][n_kv_heads][128], 4-byte aligned
 *   q, page_table, np_max, seq_len, scores : as score_blocks (seq_len counts the new token)
 * A local page outside [0, n_phys_pages) sets SPKV_DEVERR_PHYS and that request's row is not
 * written; (seq_len[b] - 1) / 64 >= np_max sets SPKV_DEVERR_PAGE_ID.  The handle must have
 * summaries.  B * n_kv_heads <= 65535. */
int decode_append_score(spkv_cache_t cache, const void* k_new, const void* v_new, const void* q, int B, int Hq,
                        const int32_t* page_table, int np_max, const int32_t* seq_len, float* scores,
                        void* stream);

/* Dual top-k page selection, [NOSA] "Method 1": dual selection (Gamma_q query-aware,
 * Gamma_e query-agnostic eviction head), locality guarantee, ED-DMA (pages are ranked on the
 * pre-exp eviction scores; exp is never applied).  Per unit, with candidates C = complete
 * pages 0 .. l_b - 1 (the local page l_b is always attended, outside the budget):
 *   E = top-k_e of {p in C : alive bit set} by evict_scores;
 *   every alive candidate outside E has its alive bit cleared (it can never enter E again);
 *   Q = top-k_q of C \ E by q_scores (evicted pages may enter Q);
 *   sel = ascending(E u Q), then l_b;  n_sel = |E u Q| + 1;  unused entries = -1.
 * Ranking is a total order: score descending, then page id ascending (-0.0 equals +0.0).
 *   q_scores, evict_scores : device fp32 [B][n_kv_heads][np_max]; must not be NaN
 *   alive      : device uint32 [B][n_kv_heads][ceil(np_max/32)] bitmask, bit p%32 of word
 *                p/32 (in/out); bits of non-candidate pages are left as they are, so a page
 *                becomes a candidate alive when it completes
 *   sel        : device int32 [B][n_kv_heads][k_e + k_q + 1] (output)
 *   n_sel      : device int32 [B][n_kv_heads] (output)
 * np_max <= 32768. */
int select_topk(spkv_cache_t cache, const float* q_scores, const float* evict_scores,
                uint32_t* alive, int B, int np_max, const int32_t* seq_len, int k_q, int k_e,
                int32_t* sel, int32_t* n_sel, void* stream);

/* Sparse decode attention over the selected pages (split-K flash decoding), [FA] "2.
 * Attention modification" (one-pass online softmax with rowmax / l, which are also
 * returned).  For query head g of unit (b, h):
 *   out[b][h*G+g][:] = sum_t softmax_t(q . k_t / sqrt(128)) v_t
 *   lse[b][h*G+g]    = log sum_t exp(q . k_t / sqrt(128))          (natural log)
 * over the tokens of pages sel[u][0 .. n_sel[u]); page p holds min(64, seq_len[b] - 64 p)
 * valid tokens (rows past that are never read into the result, even if they hold NaN).
 *   q          : device bf16 [B][Hq][128], 16-byte aligned
 *   page_table : device int32 [B][np_max]
 *   sel, n_sel : device int32 [B][n_kv_heads][sel_stride], [B][n_kv_heads]
 *   seq_len    : device int32 [B]
 *   out        : device fp32 [B][Hq][128];  lse: device fp32 [B][Hq]
 * A unit with no pages gets out = 0 and lse = -inf. */
int sparse_decode_attn(spkv_cache_t cache, const void* q, int B, int Hq, const int32_t* page_table,
                       int np_max, const int32_t* sel, const int32_t* n_sel, int sel_stride,
                       const int32_t* seq_len, float* out, float* lse, void* stream);

/* Decode attention with deferred RoPE, [Lazy] "Core idea" (keys are stored without their
 * placement position), "Technical implementation 2. Decoding" (the query is rotated only when
 * the relative offset changes, i.e. once per document; block id and offset bit-packed in one
 * word) and "Mathematical equivalence" (scores depend only on n - m).
 * Each page word (see spkv_pack_page_words) gives a physical page, its valid token count and
 * a document slot i; with P_i = doc_pos[b][i] and n = qpos[b] the page's keys are scored with
 * R(n - P_i) q, where R is the half-split RoPE rotation over pairs (x_j, x_{j+64}) with
 * frequencies theta^(-2j/128).  Stored keys carry only their document-local rotation.
 *   q        : device bf16 [B][Hq][128], not rotated, 16-byte aligned
 *   qpos     : device int32 [B]
 *   meta     : device uint32 [B][meta_heads][np_max]; meta_heads is 1 (one page list shared
 *              by all kv heads) or n_kv_heads
 *   n_pages  : device int32 [B], pages of each request's list
 *   doc_pos  : device int32 [B][max_docs]
 *   out, lse : as sparse_decode_attn. */
int lazy_rope_decode_attn(spkv_cache_t cache, const void* q, int B, int Hq, const int32_t* qpos,
                          const uint32_t* meta, int meta_heads, const int32_t* n_pages, int np_max,
                          const int32_t* doc_pos, int max_docs, float theta, float* out,
                          float* lse, void* stream);

/* Lazy-RoPE decode attention over shared cached documents, scheduled document by document.
 * [Lazy] "Core idea: deferred positional encoding" (a cached document, stored with only its
 * document-local rotation, is reused at any position) and "Technical implementation 2. Decoding"
 * (the query is rotated once per document by the relative offset).  The result is exactly
 * lazy_rope_decode_attn's for a request whose page list is its documents' pages in slot order:
 * request b holds document req_docs[b][i] (the plan's) in slot i, placed at token offset
 * doc_pos[b][i]; document d's pages are doc_pages[doc_first[d] .. doc_first[d+1]) (page words as
 * spkv_pack_page_words makes them; the slot field is ignored).  Each job of the plan streams one
 * document's pages of one kv head once for the query rows of up to 16 / G requests holding it,
 * each rotated by its own offset qpos[b] - doc_pos[b][i], so a document shared by many requests is
 * read once per job rather than once per request; every (request, query head) then merges the
 * partial results of its documents.
 *   plan      : from lazy_docs_plan_create on this handle (B, Hq, max_docs and req_docs come from it)
 *   q         : device bf16 [B][Hq][128], not rotated, 16-byte aligned
 *   qpos      : device int32 [B];  doc_pos: device int32 [B][max_docs]
 *   doc_pages : device uint32 page words;  doc_first: device int32 [n_docs + 1] (as given to the plan)
 *   out, lse  : as lazy_rope_decode_attn (a request without documents gets 0 and -inf).
 * A plan serves one stream at a time (its job counter and partials are reused by every call). */
typedef struct spkv_doc_plan* spkv_doc_plan_t;
int lazy_rope_decode_attn_docs(spkv_cache_t cache, spkv_doc_plan_t plan, const void* q, const int32_t* qpos,
                               const uint32_t* doc_pages, const int32_t* doc_first, const int32_t* doc_pos,
                               float theta, float* out, float* lse, void* stream);

/* Builds the document-major schedule on the host (the decode batch's document composition changes
 * far less often than every step, so one plan serves many steps):
 *   req_docs  : host int32 [B][max_docs], the document in each slot of each request, -1 for none
 *   doc_first : host int32 [n_docs + 1], the layout of the document page words (page counts)
 * Allocates the plan's device buffers (jobs, occurrences, one partial record per occurrence and
 * query head).  SPKV_EINVAL for a document id outside [-1, n_docs) or a decreasing doc_first. */
int lazy_docs_plan_create(spkv_cache_t cache, int B, int Hq, const int32_t* req_docs, int max_docs, int n_docs,
                          const int32_t* doc_first, spkv_doc_plan_t* out);
/* Number of jobs in the plan. */
int lazy_docs_plan_jobs(spkv_doc_plan_t plan);
int lazy_docs_plan_destroy(spkv_doc_plan_t plan);

/* Set-difference of selected vs GPU-resident pages, [NOSA] "Method 2: NOSI", optimised
 * memory layout (custom kernel computing set differences for block swapping).  Per unit:
 *   missing = sel[0..n_sel) \ resident (ascending), n_missing = its size;
 *   slot[i] = index s with resident[s] == sel[i], or -1.  Entries past the results are -1.
 *   resident : device int32 [n_units][n_slots], -1 = empty, no duplicate ids
 *   sel      : device int32 [n_units][sel_stride], strictly ascending in [0, n_sel)
 *   missing, slot : device int32 [n_units][sel_stride];  n_missing: device int32 [n_units]
 * n_slots <= 16384, sel_stride <= 4096. */
/* LazyAttention prefill over cached documents, on the tcgen05 tensor cores ([Lazy]
 * "Technical implementation 1. Prefilling" and "Mathematical equivalence").  Request b has T new
 * query rows at absolute positions qpos0[b] + t; they attend over the request's cached document
 * pages (page words and documents as in lazy_rope_decode_attn).  No mask is applied: every
 * cached key precedes the rows (attention of the rows among themselves, if wanted, is the
 * caller's, merged through lse).  For query head hq (kv head h = hq / G) and row t:
 *   out[b][t][hq][:] = sum_k softmax_k(q'_k . key_k / sqrt(128)) v_k
 *   lse[b][t][hq]    = log sum_k exp(q'_k . key_k / sqrt(128))                  (natural log)
 * with q'_k = R(qpos0[b] + t - doc_pos[b][slot of key k]) q[b][t][hq], the same scores as keys
 * rotated to their absolute positions.
 *   q     : device bf16 [B][T][Hq][128], unrotated, 16-byte aligned
 *   qpos0 : device int32 [B]
 *   meta, meta_heads, n_pages, np_max, doc_pos, max_docs, theta: as lazy_rope_decode_attn
 *   out   : device fp32 [B][T][Hq][128], 16-byte aligned;  lse: device fp32 [B][T][Hq]
 * The rotated query and the softmax weights enter the tensor cores as bf16 (fp32 accumulation).
 * A request with no pages gets out = 0 and lse = -inf.  B, Hq <= 65535. */
int lazy_rope_prefill_attn(spkv_cache_t cache, const void* q, int B, int T, int Hq,
                           const int32_t* qpos0, const uint32_t* meta, int meta_heads,
                           const int32_t* n_pages, int np_max, const int32_t* doc_pos,
                           int max_docs, float theta, float* out, float* lse, void* stream);

/* The whole prefill step of a prompt: lazy_rope_prefill_attn plus the new rows' causal attention
 * among themselves, in one softmax ([Lazy] "Technical implementation 1. Prefilling": the prompt's
 * tile attends to the cached documents after one relative rotation each; its own keys complete
 * the step).  Every listed key has an absolute position m = doc_pos[b][slot] + page_start[j] + t
 * (row t of listed page j), and query row t' of request b (position n = qpos0[b] + t') attends
 * to the keys with m <= n.  The caller lists the new rows' own K/V (written with paged_kv_append,
 * keys carrying the rotation of their position within the prompt, 0 .. T-1) as one more document
 * placed at doc_pos = qpos0[b], after the cached documents: cached keys all precede the rows, the
 * rows' own keys are seen causally, and out / lse are the complete prefill attention.
 *   page_start : device int32 with the shape of meta ([B][meta_heads][np_max]), the document-local
 *                position of each listed page's first token
 *   every other argument: as lazy_rope_prefill_attn (which equals this call when no key lies
 *   after any row).
 * A row that sees no key gets out = 0 and lse = -inf.  page_start NULL is SPKV_EINVAL. */
int lazy_rope_prefill_step(spkv_cache_t cache, const void* q, int B, int T, int Hq, const int32_t* qpos0,
                           const uint32_t* meta, int meta_heads, const int32_t* n_pages, int np_max,
                           const int32_t* page_start, const int32_t* doc_pos, int max_docs, float theta,
                           float* out, float* lse, void* stream);

/* The prefill above for ALiBi models ([Lazy] "Key contributions" 4: the mechanism carries over to
 * other relative position encodings, ALiBi among them).  Keys are stored with no positional
 * transform, so a cached document is reused at any offset as it is; the position enters only as
 * the bias.  The key in row t of listed page j (document slot i, page_start[j] its document-local
 * first position) sits at m = doc_pos[b][i] + page_start[j] + t, and for query row t' of request b
 * (position n = qpos0[b] + t') and query head hq:
 *   score = q . key / sqrt(128) - slopes[hq] * (n - m)
 *   out[b][t'][hq][:] = sum softmax(score) v,  lse[b][t'][hq] = log sum exp(score)   (natural log)
 * over every valid key of the request's listed pages at a position m <= n (keys after the row
 * are masked, as in lazy_rope_prefill_step: cached documents are seen whole, and the new rows'
 * own keys listed as a document placed at qpos0[b] make this the whole prefill step).
 *   page_start : device int32 with the shape of meta ([B][meta_heads][np_max])
 *   slopes     : device fp32 [Hq] (natural-log units per token of distance)
 *   q, qpos0, meta, meta_heads, n_pages, np_max, doc_pos, max_docs, out, lse: as above
 * The query and the softmax weights enter the tensor cores as bf16 (fp32 accumulation); the bias
 * is added in fp32.  Errors as lazy_rope_prefill_attn.  B, Hq <= 65535. */
int lazy_alibi_prefill_attn(spkv_cache_t cache, const void* q, int B, int T, int Hq, const int32_t* qpos0,
                            const uint32_t* meta, int meta_heads, const int32_t* n_pages, int np_max,
                            const int32_t* page_start, const int32_t* doc_pos, int max_docs,
                            const float* slopes, float* out, float* lse, void* stream);

/* The PyramidKV-style sparsification score S of a prompt's keys ([FA] "2. Attention
 * modification": the sum of the softmax probabilities the last alpha rows give each key,
 * computed from each row's maximum and sum in two passes, on the tcgen05 tensor cores).  For
 * query head hq of request b, with n = seq_len[b] prompt tokens in pages page_table[b][..] of
 * kv head hq / G, rows j < alpha at positions n - alpha + j and causal visibility:
 *   scores[b][hq][i] = sum_j softmax_{i' <= n - alpha + j}(q_j . k_i' / sqrt(128))[i]   (i < n)
 * and 0 for n <= i < 64 np_max.  The keys are read from the handle's pool; V is not used.
 *   q          : device bf16 [B][alpha][Hq][128], the prompt's last alpha query rows (RoPE
 *                already applied), 16-byte aligned
 *   page_table : device int32 [B][np_max];  seq_len: device int32 [B] (alpha <= n <= 64 np_max,
 *                else SPKV_DEVERR_PAGE_ID and the row is zeros)
 *   scores     : device fp32 [B][Hq][64 np_max] (output)
 * alpha <= 1024 (else SPKV_EUNSUPPORTED).  Two launches: the first computes each window row's
 * log-sum-exp into the handle's split-K workspace (128-row chunks in one grid), the second the
 * probabilities with a page pair's keys as the MMA's M and up to 256 window rows as N, each key's
 * sum over the rows formed by one thread in a fixed order (results are reproducible); windows of
 * more than 256 rows add later 256-row launches in order.  Past 4096 requests, or when the
 * workspace cannot hold B * alpha * Hq values, one launch runs both passes with the rows as M
 * (128-row chunks whose column sums add: up to 256 rows, both chunks in one grid adding atomically
 * onto a zeroed scores buffer, two addends onto zero giving the same sum in either order; more
 * rows, one launch per chunk, adding in order).
 * B, Hq <= 65535. */
int attn_column_scores(spkv_cache_t cache, const void* q, int B, int alpha, int Hq,
                       const int32_t* page_table, int np_max, const int32_t* seq_len,
                       float* scores, void* stream);

/* attn_column_scores with each window row's log-sum-exp supplied by the caller, as the
 * attention that already computed rowmax and l over the same keys returns it ([FA] "2. Attention
 * modification": the FlashAttention pass outputs rowmax and l, and the score adds only the
 * probability pass).  Only the probability launch runs, and it computes
 *   scores[b][hq][i] = sum over rows j with i <= n - alpha + j of exp(q_j . k_i / sqrt(128) - lse[b][j][hq])
 * which equals attn_column_scores when lse is each row's own log-sum-exp over its visible keys.
 *   lse : device fp32 [B][alpha][Hq], natural log, finite (not checked)
 * Every other argument, limit and error: as attn_column_scores; lse NULL is SPKV_EINVAL. */
int attn_column_scores_lse(spkv_cache_t cache, const void* q, const float* lse, int B, int alpha, int Hq,
                           const int32_t* page_table, int np_max, const int32_t* seq_len, float* scores,
                           void* stream);

int resident_setdiff(spkv_cache_t cache, const int32_t* resident, int n_slots, const int32_t* sel,
                     const int32_t* n_sel, int sel_stride, int n_units, int32_t* missing,
                     int32_t* n_missing, int32_t* slot, void* stream);

/* One decode step's selection and residency bookkeeping in one call: select_topk, then
 * resident_setdiff, then lru_bucket_update, with results identical to those three calls made
 * in turn with the same arguments (sel_stride = k_q + k_e + 1, n_units = B * n_kv_heads; the
 * slot argument of lru_bucket_update is the slot list resident_setdiff writes).  Sources as for
 * the three operations ([NOSA] "Method 1" and "Method 2: NOSI"; [Spin] 2B); the pages describe
 * them separately, and fusing them is this library's choice: for np_max <= 1024 the whole step
 * is one kernel (one CTA per unit, the selection in one warp's registers, the list handed over
 * in shared memory, each unit's residency rows read once); longer contexts launch the three
 * kernels in turn.  Argument rules and error behaviour: those of the three calls. */
int select_resident_update(spkv_cache_t cache, const float* q_scores, const float* evict_scores,
                           uint32_t* alive, int B, int np_max, const int32_t* seq_len, int k_q,
                           int k_e, int32_t* sel, int32_t* n_sel, int32_t* resident, int32_t* ts,
                           int n_slots, int32_t t_now, int bucket_width, int32_t* missing,
                           int32_t* n_missing, int32_t* slot, int32_t* victims, int32_t* hist,
                           void* stream);

/* Retrieve: copies the selected pages that are not resident from the host pool into the
 * resident slots the LRU update chose, and completes the slot list.  [NOSA] "Method 2: the
 * NOSI system" (the full KV cache lives in host memory; a UVA host-to-device kernel moves the
 * swapped-in blocks into their GPU slots); [Spin] 2A, the Retrieve operation.
 * `cache` is a handle over the slot pool: its k_pool / v_pool hold, for kv head h, request b
 * and slot s, the page at h * n_phys_pages + b * n_slots + s (B * n_slots <= n_phys_pages).
 * Per unit u = (b, h), for j < n_missing[u]:
 *   slot page (h, b, victims[u][j]) <- host page (h, page_table[b][missing[u][j]]), K and V;
 * then the r-th entry of slot[u][0 .. n_sel[u]) that is -1 is set to victims[u][r].
 *   k_host, v_host : bf16 [n_kv_heads][n_host_pages][64][128] in pinned host memory mapped
 *                    into the device address space (cudaHostAlloc / cudaHostRegister), read
 *                    through that address; 16-byte aligned
 *   page_table     : device int32 [B][np_max], host page of each logical page
 *   missing, n_missing : from resident_setdiff;  victims: from lru_bucket_update
 *   slot           : device int32 [B][n_kv_heads][sel_stride] (in/out): resident_setdiff's
 *                    slot list on entry, every selected page's slot on return
 *   n_sel          : device int32 [B][n_kv_heads]
 * Out-of-range ids and slots are skipped (SPKV_DEVERR_PAGE_ID / _PHYS / _SLOT); so is a slot
 * list whose -1 entries do not number n_missing (SPKV_DEVERR_SLOT).  Requires
 * B * n_kv_heads <= max_units of the handle. */
int retrieve_pages(spkv_cache_t cache, const void* k_host, const void* v_host,
                   int64_t n_host_pages, const int32_t* page_table, int np_max, int B,
                   const int32_t* missing, const int32_t* n_missing, const int32_t* victims,
                   int32_t* slot, const int32_t* n_sel, int sel_stride, int n_slots, void* stream);

/* sparse_decode_attn reading every selected page from its resident slot ([NOSA] "Method 2",
 * attention over the GPU buffer after the swap-in; [Spin] 2A, Attention on the fast tier).
 * Same result as sparse_decode_attn, with page sel[u][i] of unit u = (b, h) read from slot page
 * h * n_phys_pages + b * n_slots + slot[u][i] of the handle's pools (as retrieve_pages
 * addresses them); sel still gives the logical page, hence the valid tokens.
 *   slot : device int32 [B][n_kv_heads][sel_stride], 0 <= slot < n_slots (else the page is
 *          skipped, SPKV_DEVERR_SLOT)
 *   other arguments: as sparse_decode_attn.  B * n_slots <= n_phys_pages. */
int sparse_decode_attn_slots(spkv_cache_t cache, const void* q, int B, int Hq,
                             const int32_t* sel, const int32_t* slot, const int32_t* n_sel,
                             int sel_stride, int n_slots, const int32_t* seq_len, float* out,
                             float* lse, void* stream);

/* Bucketed LRU update, [Spin] 2B "bucketed LRU policy" (pages grouped into 64 recency
 * buckets by timestamp; eviction without a global sort).  Per unit, at time t_now:
 *   1. ts[s] = t_now for every hit slot s = slot[i] >= 0;
 *   2. bucket(s) = 63 if resident[s] < 0, else min(63, max(0, t_now - ts[s]) / bucket_width);
 *      hist[u][b] = number of slots in bucket b (all slots, after step 1);
 *   3. victims[0 .. n_missing) = untouched slots in order (bucket desc, slot asc);
 *   4. resident[victims[i]] = missing[i], ts[victims[i]] = t_now.
 *   resident, ts : device int32 [n_units][n_slots] (in/out); an empty slot's ts is ignored
 *   slot, missing: device int32 [n_units][sel_stride]; n_sel, n_missing: device int32 [n_units]
 *   victims      : device int32 [n_units][sel_stride] (output, -1 past n_missing)
 *   hist         : device int32 [n_units][64] (output)
 * bucket_width >= 1, n_slots <= 16384. */
int lru_bucket_update(spkv_cache_t cache, int32_t* resident, int32_t* ts, int n_slots,
                      const int32_t* slot, const int32_t* n_sel, const int32_t* missing,
                      const int32_t* n_missing, int sel_stride, int n_units, int32_t t_now,
                      int bucket_width, int32_t* victims, int32_t* hist, void* stream);

/* sparse_decode_attn without any allocation.  The pages this library follows have no
 * counterpart for this entry point: it exists for callers that cannot allocate device memory
 * (an engine that forbids cudaMalloc after start-up or owns all device memory through its own
 * allocator, or code that must not create a handle, since paged_kv_create allocates).  It
 * computes exactly what sparse_decode_attn computes, with the same kernel, but takes the pool
 * directly instead of a handle and keeps its split-K scratch (partial results and their
 * counters) in one fixed device array of SPKV_NOALLOC_SCRATCH_BYTES bytes that every GPU
 * loading this library holds until the process exits.  The caller passes inputs and outputs.
 *   k_pool, v_pool : device bf16 [n_kv_heads][n_phys_pages][64][128], 16-byte aligned
 *   q              : device bf16 [B][Hq][128], 16-byte aligned
 *   dev_err        : device uint32 owned by the caller (required), receives SPKV_DEVERR_* bits
 *                    (OR-ed in): out-of-range page ids and physical pages are skipped and
 *                    reported only there, so the caller reads it after the call completes
 *   other arguments: as sparse_decode_attn.
 * Every pointer above must be memory of the current device; any other (host memory, another
 * device's memory) returns SPKV_EINVAL before anything is launched.
 * Limits: B * n_kv_heads <= SPKV_NOALLOC_MAX_UNITS and Hq / n_kv_heads <= 16; larger calls
 * return SPKV_EUNSUPPORTED before anything is launched.  No cudaMalloc, cudaFree or other
 * allocating routine is called.  The first call on a device looks up the scratch's device
 * address with that device current, so make it before any stream capture.  All calls on a
 * device share the scratch, which keeps the last call's contents: each call clears the chunk
 * counter first and rewrites every per-unit record it reads, and calls whose kernels overlap
 * on the GPU (unordered streams) race on it and must not be issued. */
#define SPKV_NOALLOC_MAX_UNITS 512
#define SPKV_NOALLOC_MAX_CTAS 160
#define SPKV_NOALLOC_SCRATCH_BYTES 6926592
int sparse_decode_attn_noalloc(const void* k_pool, const void* v_pool, int n_kv_heads,
                               int64_t n_phys_pages, const void* q, int B, int Hq,
                               const int32_t* page_table, int np_max, const int32_t* sel,
                               const int32_t* n_sel, int sel_stride, const int32_t* seq_len,
                               float* out, float* lse, uint32_t* dev_err, void* stream);

/* Packs page words for lazy_rope_decode_attn on the host ([Lazy] "Technical implementation
 * 2. Decoding", bit-packed block id and offset):
 *   word = phys | (valid - 1) << 18 | doc_slot << 24,
 * with phys < 2^18, 1 <= valid <= 64, doc_slot < 256.  Host arrays of length n.
 * Returns SPKV_EINVAL (and stops) at the first field out of range. */
int spkv_pack_page_words(const int32_t* phys, const int32_t* valid, const int32_t* doc_slot,
                         int64_t n, uint32_t* words);

/* ---------------------------------------------------------------------------------------------
 * Two-level page directory ([Spin] "Unifying Sparse Attention with Hierarchical Memory for
 * Scalable Long-Context LLM Serving", section 2C "Hierarchical metadata management": a small
 * GPU-resident top-level directory points to second-level segments that are allocated on demand in
 * CPU memory, so metadata grows with the pages actually in use rather than with the logical address
 * space; latency-critical metadata stays on the GPU, bulk metadata moves to the CPU).
 *
 * The logical-to-physical page table of a request is split into segments of 2^seg_shift page ids.
 * Directory entry e = dir[b][p >> seg_shift] locates the segment holding logical page p:
 *   e >= 0   device tier: segment e of dev_segs (the GPU-resident cache of hot segments)
 *   e <= -2  host tier: host segment h = -2 - e, in pinned host memory read in place by the kernels
 *            (over NVLink-C2C on GB300): chunk h >> chunk_shift of host_chunks, segment
 *            h & (2^chunk_shift - 1) of that chunk
 *   e == -1  unmapped: no page of that range exists (a lookup there reports SPKV_DEVERR_PHYS)
 * and the physical page is entry p & (2^seg_shift - 1) of that segment.  A lookup gives exactly the
 * page a flat page_table[b][p] with the same contents gives, so the *_dir calls below return
 * bit for bit what their flat-table forms return.  (spkv_pagemap_* builds and maintains one.) */
typedef struct {
  const int32_t* dir;                 /* device int32 [B][n_dir] */
  const int32_t* dev_segs;            /* device int32 [n_dev_segs][2^seg_shift] */
  const int32_t* const* host_chunks;  /* device array of the device addresses of pinned, mapped host
                                         chunks, each int32 [2^chunk_shift][2^seg_shift] */
  int32_t n_dir;                      /* directory entries per request (>= ceil(np_max / 2^seg_shift)) */
  int32_t seg_shift;                  /* 4 .. 12 */
  int32_t n_dev_segs;
  int32_t chunk_shift;                /* 0 .. 16 */
  int64_t n_host_segs;
} spkv_page_dir;

/* score_blocks with the page table given as a two-level directory (contents as above; np_max still
 * bounds the logical pages).  Every other argument, result and error: as score_blocks. */
int score_blocks_dir(spkv_cache_t cache, const void* q, int B, int Hq, const spkv_page_dir* dir, int np_max,
                     const int32_t* seq_len, float* scores, void* stream);

/* sparse_decode_attn with the page table given as a two-level directory. */
int sparse_decode_attn_dir(spkv_cache_t cache, const void* q, int B, int Hq, const spkv_page_dir* dir, int np_max,
                           const int32_t* sel, const int32_t* n_sel, int sel_stride, const int32_t* seq_len,
                           float* out, float* lse, void* stream);

/* retrieve_pages with the (host-page) table given as a two-level directory. */
int retrieve_pages_dir(spkv_cache_t cache, const void* k_host, const void* v_host, int64_t n_host_pages,
                       const spkv_page_dir* dir, int np_max, int B, const int32_t* missing,
                       const int32_t* n_missing, const int32_t* victims, int32_t* slot, const int32_t* n_sel,
                       int sel_stride, int n_slots, void* stream);

/* A page-directory manager (host side, [Spin] 2C).  It owns the device directory, a device cache of
 * n_dev_segs hot segments and the host segments, which it allocates on demand (pinned, mapped host
 * memory, 2^chunk_shift segments per allocation) the first time a page of their range is mapped.
 * spkv_pagemap_map and spkv_pagemap_promote change the host state at once; spkv_pagemap_sync
 * enqueues on `stream` the copies that bring the device directory and the device-tier segments up to
 * date and waits for them.  Host-tier segments are read in place by the kernels, so map only pages
 * that no enqueued, unfinished kernel reads (for example between decode steps).  One thread at a time
 * per manager.  Errors: SPKV_EINVAL for bad arguments, SPKV_ENOMEM when an allocation fails,
 * SPKV_ECUDA for a failed copy. */
typedef struct spkv_pagemap* spkv_pagemap_t;

/* B requests of up to np_max logical pages, segments of 2^seg_shift ids (4 .. 12), n_dev_segs >= 0
 * device-tier slots.  Allocates the device directory (all entries unmapped) and the device slots. */
int spkv_pagemap_create(int B, int np_max, int seg_shift, int n_dev_segs, spkv_pagemap_t* out);

/* Logical pages [first_page, first_page + n) of request b get the physical ids phys[0 .. n) (host
 * int32; -1 unmaps a page).  Host segments of the range are allocated on demand. */
int spkv_pagemap_map(spkv_pagemap_t pm, int b, int first_page, int n, const int32_t* phys);

/* Moves the segment of request b that holds logical page `page` to the device tier: a free device
 * slot, else the slot promoted longest ago, whose segment returns to the host tier.  The segment
 * must be mapped (SPKV_EINVAL otherwise); promoting a device-tier segment renews it. */
int spkv_pagemap_promote(spkv_pagemap_t pm, int b, int page);

/* Brings the device directory and the device-tier segments up to date (copies on `stream`, then
 * waits for the stream). */
int spkv_pagemap_sync(spkv_pagemap_t pm, void* stream);

/* The directory view that the *_dir calls take (valid until the next map / promote / sync). */
int spkv_pagemap_view(spkv_pagemap_t pm, spkv_page_dir* out);

/* Metadata bytes: on the device (directory, device-tier slots, chunk table) and in host memory
 * (allocated host segments). */
int spkv_pagemap_bytes(spkv_pagemap_t pm, int64_t* device_bytes, int64_t* host_bytes);

/* Frees everything the manager allocated (the caller ensures no kernel still reads it). */
int spkv_pagemap_destroy(spkv_pagemap_t pm);

/* Waits for `stream`, then reads and clears the handle's device error word into *bits./* Waits for `stream`, then reads and clears the handle's device error word into *bits.
 * Returns SPKV_OK when it was zero, SPKV_EDEVICE otherwise (SPKV_ECUDA if the wait failed). */
int spkv_get_device_error(spkv_cache_t cache, void* stream, uint32_t* bits);

/* Frees the handle and what it allocated (not the caller's buffers).  The caller must make
 * sure no call on the handle is still running. */
int paged_kv_destroy(spkv_cache_t cache);

/* Number of SMs the handle's kernels size their grids for (the device's SM count). */
int spkv_sm_count(spkv_cache_t cache);

/* Sets how long each bounded hand-off wait inside this handle's attention kernels
 * (sparse_decode_attn, sparse_decode_attn_slots, lazy_rope_decode_attn) lasts before it gives up,
 * in nanoseconds; the default is 1 s, far beyond any hand-off of a correct run.  A wait that gives
 * up sets SPKV_DEVERR_TIMEOUT (reported as SPKV_ETIMEOUT by spkv_get_device_error); the CTA then
 * waits for its own copies in flight (always with the full 1 s limit) and returns, and the call's
 * outputs are undefined.  0 makes every wait that is not already complete give up at once, which
 * exercises that error path without a fault.  Applies to calls made after it; ns <= 10^10. */
int spkv_set_wait_limit(spkv_cache_t cache, uint64_t ns);

/* A static string naming a status code. */
const char* spkv_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* SPKV_H_ */
