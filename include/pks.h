/*
 * pks - top-k sparse attention decode over a paged KV cache, for GB300 (sm_103a).
 *
 * C ABI of libpks.so.  Plain integers, sizes and pointers only; every
 * function returns a pks_status and never aborts.  Device work is enqueued
 * on the caller's stream and does not synchronise; the library allocates no
 * device memory (scratch comes from a caller-owned workspace) and keeps no
 * global state.
 *
 * Sources, cited by title and section:
 *  [SA]  "Sparse Attention on GLM5.3 and HBM": introduction (top-k tokens,
 *        SDPA over only those; the selection needs the whole context in HBM),
 *        HiSparse paragraph (LRU cache of KV in HBM, load on a top-k miss,
 *        evict by least recent use), DeepSeek Sparse Attention paragraph
 *        (lightning indexer: multi-head query, single-head key, dot product,
 *        ReLU, weighted sum over heads; one top-K set shared by all heads;
 *        dense attention below K tokens).
 *  [PKV] "Paged KV cache, or why reserving for the maximum length is
 *        wasteful": "Paging" (fixed-size pages, a per-request page table,
 *        pages = ceil(len / page_size)), "Page sharing" (identical prefixes
 *        point to the same pages, only whole pages are shared), "What this
 *        table does not say" (free-page list, page tables, scattered reads).
 *  [LIN] "Why recalling an old conversation costs so much", "Three blockers":
 *        a store that takes logical slot ids must translate them to physical
 *        ids (here: token positions are always logical, only the block table
 *        maps them to pages); a pool sized outside the memory accounting
 *        crashed at start-up (here: no hidden allocation).
 *
 * Layouts (all row-major, all device pointers unless stated "host"):
 *   q            bf16  [B, Hq, D]            attention query of the decoded token
 *   q_idx        int8  [B, Hi, Di]           indexer query (Hi heads)
 *   w_idx        int32 [Hi]                  indexer head weights (or w_idx_f: float [B, Hi])
 *   kv_k, kv_v   bf16  [num_pages, page_size, Hkv, D]   paged K / V pools
 *   idx_k        int8  [num_pages, page_size, Di]       paged single-head indexer keys
 *   seq_lens     int32 [B]                   cached tokens per request (0 allowed)
 *   block_table  int32 [B, max_pages]        logical page -> physical page; entries at
 *                                            p >= ceil(len_b/page_size) are ignored
 *   topk_idx     int32 [B, k]                selected logical token positions, ascending,
 *                                            padded with -1
 *   out          bf16  [B, Hq, D]            attention output
 * Query head h reads KV head h / (Hq / Hkv) (contiguous GQA groups).
 */
#ifndef PKS_H
#define PKS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t / cudaEvent_t, passed without the CUDA headers. NULL = legacy default stream. */
typedef struct CUstream_st* pks_stream;
typedef struct CUevent_st* pks_event;

typedef int32_t pks_status;
#define PKS_OK 0
#define PKS_ERR_INVALID (-1)      /* bad argument: null pointer, negative or inconsistent size */
#define PKS_ERR_OOM (-2)          /* host page pool cannot satisfy the request (nothing taken) */
#define PKS_ERR_CUDA (-3)         /* a CUDA runtime call (launch, copy, memset) failed */
#define PKS_ERR_TIMEOUT (-4)      /* a bounded device-side wait ran out */
#define PKS_ERR_DEVICE_CHECK (-5) /* a device-side bounds check fired (see *_device_error) */
#define PKS_ERR_UNSUPPORTED (-6)  /* valid but outside the compiled shapes (see pks_decode_args) */
#define PKS_ERR_WORKSPACE (-7)    /* workspace missing, misaligned or smaller than required */
#define PKS_ERR_TOO_LARGE (-8)    /* shapes need more scratch than pks_sparse_attention_static's
                                     fixed buffer holds */

/* Static English text for a status code. */
const char* pks_status_str(pks_status status);

/* ------------------------------------------------------------------------
 * Host page allocator ([PKV] "Paging", "What this table does not say").
 * A pool of num_pages physical pages of page_size tokens with a FIFO free
 * list: pages are handed out from the front, freed pages go to the back.
 * The initial order is 0..num_pages-1, or the permutation free_order (host,
 * num_pages entries, copied).  The handle is host memory owned by the
 * library; it is not thread-safe.
 * ---------------------------------------------------------------------- */
typedef struct pks_pool pks_pool;

/* INVALID: num_pages < 1, page_size < 1, free_order not a permutation, out NULL. */
pks_status pks_pool_create(int32_t num_pages, int32_t page_size, const int32_t* free_order,
                           pks_pool** out);
void pks_pool_destroy(pks_pool* pool);
pks_status pks_pool_free_count(const pks_pool* pool, int32_t* out);

/* Take n pages from the front of the free list into out_ids (host, n entries).
 * All or nothing: OOM (and nothing taken) when fewer than n are free. */
pks_status pks_alloc_pages(pks_pool* pool, int32_t n, int32_t* out_ids);

/* Return n pages (host ids) to the back of the free list.  INVALID (and
 * nothing returned) if an id is out of range, already free, or repeated. */
pks_status pks_free_pages(pks_pool* pool, int32_t n, const int32_t* ids);

/* [PKV] "Paging" + "Page sharing": build the block table of a batch.
 * Requests are served in ascending order; request b takes ceil(len_b /
 * page_size) logical pages, in ascending order, each from pks_alloc_pages.
 * Prefix sharing: when prefix_group (host, nullable) gives request b a group
 * id >= 0, its logical page p is an alias of the page an earlier member of
 * the same group holds at p, provided the page lies wholly inside the shared
 * prefix and wholly inside request b (p < floor(prefix_len / page_size) and
 * p < floor(len_b / page_size)); otherwise a fresh page is taken.  So a group
 * of n requests at least prefix_len long saves (n-1)*floor(prefix_len/page_size)
 * pages.  Writes block_table (host, [batch, max_pages], unused entries -1) and
 * *pages_used (nullable) = fresh pages taken.  INVALID if a request needs
 * more than max_pages pages or a length is negative; OOM if the pool runs
 * out.  On any error every page this call took is returned and the table is
 * all -1. */
pks_status pks_build_block_table(pks_pool* pool, int32_t batch, const int32_t* seq_lens,
                                 const int32_t* prefix_group, int32_t prefix_len,
                                 int32_t max_pages, int32_t* block_table, int32_t* pages_used);

/* Admission on the pool's free pages ([PKV] "How many users" and "Internal
 * fragmentation").  Requests of lengths lens[i % n] (i = 0, 1, ...) arrive
 * and never finish; each takes ceil(len / page_size) pages (reserve == 0:
 * paging) or ceil(reserve / page_size) pages (reserve > 0: every request
 * reserves `reserve` tokens, and one longer than that stops admission).
 * Admission stops at the first request that does not fit.  Writes *admitted,
 * *tokens (the admitted lengths' sum) and *slots (pages taken x page_size);
 * waste = slots - tokens.  Counts only: the pool is not modified.  INVALID on
 * a negative length or when the requests take no pages (unbounded). */
pks_status pks_admission_simulate(const pks_pool* pool, int32_t n, const int32_t* lens,
                                  int32_t reserve, int64_t* admitted, int64_t* tokens,
                                  int64_t* slots);

/* ------------------------------------------------------------------------
 * Decode step ([SA] introduction and DeepSeek Sparse Attention paragraph).
 *
 * For every request b with len_b = seq_lens[b]:
 *  1. indexer scan: s[b,t] = sum_h w_idx[h] * max(0, q_idx[b,h,:] . k_idx(b,t)) in
 *     int32 for every t < len_b, k_idx(b,t) = idx_k[block_table[b][t/page_size],
 *     t % page_size, :].  The caller keeps sum_h |w_idx[h]| * Di * 128^2 < 2^31.
 *  2. top-k: if len_b <= k all tokens (dense); else the k tokens first in the
 *     order (score descending, token index ascending).  Written to topk_idx in
 *     ascending token order, -1 padded.
 *  3. attention: out[b,h] = softmax(q[b,h] . K_sel / sqrt(D)) V_sel over the
 *     selected tokens, K/V rows gathered through block_table; bf16 inputs,
 *     fp32 accumulation, bf16 output.  A request with len_b = 0 gets zeros.
 *
 * Compiled shapes (else UNSUPPORTED): D in {64, 128}; Di in {64, 128};
 * Hi in {1, 2, 4, 8}; 1 <= Hq/Hkv <= 16; B <= 4096; k <= 65536;
 * max_pages*page_size <= 2^24.  q, kv_k, kv_v, q_idx, idx_k must be 16-byte
 * aligned (INVALID otherwise).
 * ---------------------------------------------------------------------- */
typedef struct pks_decode_args {
  int32_t B, Hq, Hkv, D, Hi, Di;
  int32_t page_size, max_pages, num_pages, k;
  const int32_t* seq_lens;
  const int32_t* block_table;
  const void* q;
  const int8_t* q_idx;
  const int32_t* w_idx;
  const void* kv_k;
  const void* kv_v;
  const int8_t* idx_k;
  int32_t* topk_idx;      /* output of the step; input of pks_sparse_attention */
  void* out;
  void* workspace;        /* device scratch owned by the caller, 256-byte aligned */
  size_t workspace_bytes;
  int32_t attn_splits;    /* attention CTAs: 0 = one per resident slot on the GPU, but no
                             more than one per 32 selected positions; else this many
                             (1..1024, at most one per position), each taking an equal share
                             of all selected (KV head group, request, position) work */
  int32_t topk_mode;      /* 0 = one cooperative top-k launch when its grid fits on the GPU
                             at once, else two; 1 = always the two-kernel path */
  int32_t n_queries;      /* query tokens per request, Nq (0 or 1: one).  With Nq > 1, q is
                             [B, Nq, Hq, D], q_idx [B, Nq, Hi, Di], topk_idx [B, Nq, k] and
                             out [B, Nq, Hq, D]: every query token of request b scores the
                             request's len_b cached tokens, selects its own top-k and attends
                             over it; the indexer keys are read once for all Nq queries.
                             Nq in {1, 2, 4, 8} and Hi * Nq <= 8 (UNSUPPORTED otherwise);
                             pks_indexer_scores then writes B * Nq score rows */
  int32_t reserved[1];    /* must be 0 */
  const float* w_idx_f;   /* NULL, or real-valued indexer head weights, device float
                             [B, Hi] (one row per request; n_queries must then be 1):
                             s[b,t] = sum_h w_idx_f[b,h] * max(0, q_idx[b,h,:] . k_idx(b,t))
                             evaluated in fp32 with the heads in order, each product and
                             each sum rounded to nearest (no fused multiply-add); w_idx is
                             then not read.  The scores the scan writes (and
                             pks_indexer_scores returns) are int32 keys with the order of
                             the fp32 scores: key = bits(s) for s >= 0, bits(s) ^ 0x7fffffff
                             for s < 0 (-0 taken as +0).  Weights must keep every score
                             finite. */
  int32_t idx_fp8;        /* 0: q_idx and idx_k are int8.  1: they hold FP8 e4m3 bit
                             patterns (finite values; w_idx_f required, else INVALID); each
                             head's dot product is taken on the tensor core with fp32
                             accumulation in the hardware's order, then weighted and summed
                             over the heads as for w_idx_f */
  int32_t wait_limit;     /* polls of the top-k request barrier (a bounded device-side wait)
                             before it gives up with device error 5: 0 = the default, 2^22
                             (about half a second); >= 0 (INVALID otherwise).  Small values
                             exist to exercise the time-out path */
} pks_decode_args;

/* Workspace bytes a step with these shapes needs (pointers may be NULL). */
pks_status pks_decode_workspace_size(const pks_decode_args* args, size_t* bytes);

/* Zero the workspace's control words.  Required once before the first step on
 * a workspace (or zero the whole buffer with cudaMemset); every completed step
 * leaves them zero again, so steps can be replayed (e.g. in a CUDA graph). */
pks_status pks_decode_workspace_init(const pks_decode_args* args, pks_stream stream);

/* The whole step: scan, top-k, attention.  Four or more kernel launches:
 * scan, top-k, attention and merge; top-k is one cooperative launch when all
 * of its (4096-token chunk, request) CTAs fit on the device at once, else two
 * (three with more than 131072 tokens per request); see pks_decode_launches.
 * TIMEOUT-class failures of the top-k barrier are reported through
 * pks_decode_device_error (code 5), after which the workspace must be
 * re-initialised. */
pks_status pks_decode_step(const pks_decode_args* args, pks_stream stream);

/* Stages 1 and 2 alone (scan and top-k, writing args->topk_idx), for callers
 * that route attention elsewhere, e.g. through a residency table
 * (pks_sparse_attention_resident).  q, kv_k, kv_v and out are not used. */
pks_status pks_decode_select(const pks_decode_args* args, pks_stream stream);

/* Kernels one pks_decode_step with these shapes enqueues on the current
 * device (host only; pointers may be NULL).  INVALID: bad shapes or out NULL. */
pks_status pks_decode_launches(const pks_decode_args* args, int32_t* launches);

/* Same as pks_decode_step, recording events[0..3] (nullable entries) before the
 * scan, after the scan, after the top-k kernels and after attention. */
pks_status pks_decode_step_timed(const pks_decode_args* args, pks_stream stream,
                                 pks_event const* events);

/* Stage 1 alone, for inspection: int32 scores into scores[b * ld + t] for
 * t < len_b (device; ld >= max_pages*page_size); other entries untouched.
 * Uses no workspace. */
pks_status pks_indexer_scores(const pks_decode_args* args, int32_t* scores, int64_t ld,
                              pks_stream stream);

/* Stage 3 alone: attention over the tokens the caller put in args->topk_idx
 * (any order, -1 entries skipped, each position must be < len_b).  Writes
 * args->out; uses the workspace. */
pks_status pks_sparse_attention(const pks_decode_args* args, pks_stream stream);

/* pks_sparse_attention without a workspace, for callers that cannot allocate
 * device memory: a runtime whose memory is planned ahead and locked, or code
 * running where an allocation would synchronise or fail.  The sources have
 * no counterpart of this call; it is a deployment convenience.  Same
 * arguments, grid and results as pks_sparse_attention; args->workspace and
 * workspace_bytes are ignored.
 *
 * Scratch: one file-scope device array of 8 MiB (8388608 bytes) inside
 * libpks, holding the per-request position prefix and the split-K partials,
 * (attention CTAs + (Hkv/hg)*B) * (Hq/Hkv)*hg * (D + 2) * 4 bytes (hg = the
 * largest of 8, 4, 2, 1 dividing Hkv; CTAs = attn_splits, or the GPU's
 * resident slots when 0).  TOO_LARGE when the shapes need more (checked on
 * the host before any launch; nothing is enqueued).  The call makes no
 * cudaMalloc, cudaFree or other allocating call, and nothing in the array has
 * to start at zero: every word the merge reads is written earlier in the
 * same call.
 *
 * Set-up: the first call on each device looks up the array's address with
 * cudaGetSymbolAddress (that device current).  The attention kernel's
 * shared-memory limit is shared with pks_sparse_attention and only ever
 * raised: a call whose shapes need more shared memory than any earlier call
 * of either entry point on the device raises it first.  Neither step is a
 * stream operation; make the first call, and any call with a larger batch
 * than before, outside stream capture.
 * The array is shared by every call on a device: calls that overlap in time
 * (other streams, concurrent graph replays, other host threads) race on it.
 * Device-side bounds checks skip bad rows as in pks_sparse_attention but are
 * not reported (their flag lives in the array). */
pks_status pks_sparse_attention_static(const pks_decode_args* args, pks_stream stream);

/* Byte offset inside the workspace of the top-k request barriers' arrival
 * counters (int32, one per request and query token, zero between steps), for
 * diagnosis and for tests that make a barrier wait run out: a counter that
 * starts below zero needs more arrivals than the request's CTAs make, so its
 * CTAs give up after wait_limit polls with device error 5.  Host only;
 * pointers in args may be NULL.  INVALID: bad shapes or offset NULL. */
pks_status pks_decode_barrier_offset(const pks_decode_args* args, size_t* offset);

/* Copy the workspace's device error word to *code (host) and clear it;
 * synchronises the stream.  *code = 0 when no device check fired, else the
 * PKS_ERR_DEVICE_CHECK cause: 1 page id out of [0, num_pages), 2 selected
 * token position outside [0, len_b), 3 sequence length outside
 * [0, max_pages*page_size]. */
pks_status pks_decode_device_error(const pks_decode_args* args, int32_t* code,
                                   pks_stream stream);

/* ------------------------------------------------------------------------
 * HBM residency table ([SA] HiSparse paragraph).  A table of `capacity`
 * slots over physical pages [0, num_pages), kept in one caller-owned device
 * buffer (`state`, 256-byte aligned) with this layout (int32 unless noted):
 *   [0..15]                header: num_pages, capacity, step, n_resident,
 *                          device error word, magic, reserved
 *   page_slot[num_pages]   slot of a resident page, -1 otherwise
 *   slot_page[capacity]    page held by a slot, -1 if empty
 *   last_use[capacity]     step of the slot's last use, -1 if never
 *   lru_order[capacity]    slots ordered by (last_use ascending, slot ascending)
 *   scratch (flags and a victim list), zero between calls
 * Each section starts on a 256-byte boundary; pks_residency_offsets gives them.
 * ---------------------------------------------------------------------- */
pks_status pks_residency_state_bytes(int32_t num_pages, int32_t capacity, size_t* bytes);

/* Byte offsets of page_slot, slot_page, last_use and lru_order inside the state. */
pks_status pks_residency_offsets(int32_t num_pages, int32_t capacity, size_t* page_slot,
                                 size_t* slot_page, size_t* last_use, size_t* lru_order);

/* Fill `state`: the n_init distinct pages of init_pages (host) go to slots
 * 0..n_init-1 in ascending page order with last use 0; other slots are empty.
 * Validates on the host (INVALID on duplicates, range, n_init > capacity),
 * then copies with cudaMemcpyAsync on `stream`. */
pks_status pks_residency_init(void* state, int32_t num_pages, int32_t capacity,
                              int32_t n_init, const int32_t* init_pages, pks_stream stream);

/* One step.  A = distinct physical pages block_table[b][t / page_size] over
 * every selected t = topk_idx[b][j] >= 0.  Writes miss_list[0..n) = A minus
 * the pages resident at the start of the step, ascending, and *n_miss = n
 * (device scalar).  Pages of A already resident get last use = step; the
 * slots not holding a page of A are victims in (last use, slot) order, and
 * the i-th miss takes the i-th victim's slot (last use = step).  Misses beyond
 * the victims are reported but not admitted, so a step never evicts a page it
 * reads.  miss_list needs num_pages entries.  Two kernel launches. */
pks_status pks_residency_update(void* state, int32_t num_pages, int32_t capacity, int32_t B,
                                int32_t k, int32_t page_size, int32_t max_pages,
                                const int32_t* topk_idx, const int32_t* block_table,
                                int32_t* miss_list, int32_t* n_miss, pks_stream stream);

/* ------------------------------------------------------------------------
 * Miss fetch and attention through the residency table ([SA] HiSparse
 * paragraph: the KV cache lives in host DRAM, HBM holds an LRU cache of it,
 * a top-k miss is loaded into HBM).  The pages' K/V pools (host_k, host_v:
 * [num_pages, page_size, Hkv, D] bf16) live in device-accessible host memory
 * (pinned, read over the CPU-GPU link); the HBM slot pools (slot_k, slot_v:
 * [capacity, page_size, Hkv, D] bf16) hold the resident pages, slot s holding
 * page slot_page[s].  A step: pks_decode_select, pks_residency_update,
 * pks_residency_fetch, pks_sparse_attention_resident.
 * ---------------------------------------------------------------------- */

/* Copy the misses of the last pks_residency_update that were admitted (a
 * page of miss_list[0..*n_miss) that now has a slot) from the host pools into
 * their slots: page_bytes = page_size * Hkv * D * 2 bytes of K and of V per
 * page.  Misses that were not admitted are skipped (the attention reads them
 * from the host pools).  All pointers 16-byte aligned; page_bytes a multiple
 * of 16 (INVALID otherwise).  One kernel launch. */
pks_status pks_residency_fetch(const void* state, int32_t num_pages, int32_t capacity,
                               const int32_t* miss_list, const int32_t* n_miss,
                               const void* host_k, const void* host_v, void* slot_k,
                               void* slot_v, int64_t page_bytes, pks_stream stream);

/* pks_sparse_attention with K/V found through the residency table: args->kv_k
 * and args->kv_v are the host pools (args->num_pages pages); a token of a
 * resident page is read from its slot in slot_k / slot_v, any other from the
 * host pools.  Same grid, arithmetic and result as pks_sparse_attention on
 * the host pools.  Uses the workspace; state as for pks_residency_update. */
pks_status pks_sparse_attention_resident(const pks_decode_args* args, const void* state,
                                         int32_t capacity, const void* slot_k,
                                         const void* slot_v, pks_stream stream);

/* ----------------------------------------------------------------------
 * Sparse MLA in MQA mode ("Sparse Attention on GLM5.3 and HBM", DeepSeek
 * Sparse Attention paragraphs: the sparse MLA of DSA runs in MQA mode; the
 * pages' configuration is latent d = 512, RoPE r = 64, H = 64 or 128 query
 * heads, 2-byte values).  Every token keeps one latent row of d + r values
 * shared by all H heads:
 *   out[b,h] = sum_j softmax_j(sm_scale * q[b,h] . kv_j) kv_j[0:d]
 * j over the positions of topk_idx[b, :] holding a token (>= 0), kv_j the
 * row of token t_j found through the block table.  The pages do not give the
 * softmax scale: sm_scale 0 means 1 / sqrt(d + r).
 * ---------------------------------------------------------------------- */
typedef struct pks_mla_args {
  int32_t B;              /* requests, 0..4096 */
  int32_t H;              /* query heads, 1..128 */
  int32_t d_latent;       /* d: must be 512 */
  int32_t d_rope;         /* r: must be 64 */
  int32_t page_size, max_pages, num_pages;
  int32_t k;              /* entries per request in topk_idx, 1..65536 */
  const int32_t* seq_lens;     /* device int32 [B] */
  const int32_t* block_table;  /* device int32 [B, max_pages] */
  const int32_t* topk_idx;     /* device int32 [B, k]: token positions, -1 = none */
  const void* q;               /* device bf16 [B, H, d + r], 16-byte aligned */
  const void* kv;              /* device bf16 [num_pages, page_size, d + r], 16-byte aligned */
  void* out;                   /* device bf16 [B, H, d], 16-byte aligned (written) */
  void* workspace;             /* device scratch owned by the caller, 256-byte aligned */
  size_t workspace_bytes;
  float sm_scale;              /* softmax scale; 0 = 1 / sqrt(d + r) */
  int32_t trim;                /* 1: each list holds its selected entries first and -1
                                  after (the decode step's own top-k), so only the first
                                  min(k, len_b) positions are visited; 0: all k */
  int32_t splits;              /* CTA pairs per request: 0 = automatic (one pair per two
                                  SMs spread over the requests), else 1..64; raised to
                                  ceil(ceil(k / 64) / 32) when lower (a CTA takes at most
                                  32 tiles of 64 tokens) */
  int32_t wait_limit;          /* clock cycles a bounded mbarrier wait of the MLA kernel spins
                                  before it gives up with device error 5 (the CTA's other
                                  warps then stop too): 0 = the default, 4e9 (about 2 s);
                                  >= 0 (INVALID otherwise).  Small values exist to exercise
                                  the time-out path */
} pks_mla_args;

/* Workspace bytes pks_mla_sparse_attention needs for these shapes (pointers
 * may be NULL): a 16-byte device error word plus, with more than one split,
 * the (m, l) and fp32 output partials of every (request, split, head). */
pks_status pks_mla_workspace_size(const pks_mla_args* args, size_t* bytes);

/* Sparse MLA over the selected tokens, asynchronous on the stream.  One CTA
 * per (request, split, half of d) on the tcgen05 tensor cores (accumulators in
 * tensor memory), 230 KB of shared memory each, plus one merge launch when
 * splits > 1.  INVALID for NULL pointers (B > 0), misaligned pointers or
 * shapes outside the ranges above; UNSUPPORTED for d != 512 or r != 64;
 * WORKSPACE when the workspace is missing, misaligned or too small.  Device
 * checks (page id, token position, length out of range) skip the token and
 * set the workspace's error word, read by pks_mla_device_error.  The caller
 * zeroes the error word once (pks_mla_device_error clears it). */
pks_status pks_mla_sparse_attention(const pks_mla_args* args, pks_stream stream);

/* Copy the MLA workspace's device error word to *code and clear it (codes as
 * for pks_decode_device_error; 5: a bounded wait inside the kernel gave up).
 * Synchronises the stream. */
pks_status pks_mla_device_error(const pks_mla_args* args, int32_t* code, pks_stream stream);

/* ---- staging of a step's inputs and outputs --------------------------------
 * Not an operation of the pages: a serving convenience for moving a step's
 * small inputs (queries, lengths, block table) in and its outputs (attention
 * output, top-k) out.  On a GB300 the SMs load and store page-locked host
 * memory over the CPU-GPU link faster than the copy engines move buffers of
 * this size, and one launch replaces one copy per buffer. */

/* At most this many ranges per pks_stage_copy call. */
#define PKS_STAGE_MAX_RANGES 8

/* One byte range: dst and src are device memory or page-locked host memory
 * that the device can address (cudaHostAlloc / cudaMallocHost / registered
 * memory on a unified-address system).  Ranges of one call must not overlap. */
typedef struct pks_copy_range {
  void* dst;
  const void* src;
  size_t bytes;
} pks_copy_range;

/* Copy n (1..PKS_STAGE_MAX_RANGES) byte ranges with one kernel launch on
 * `stream`: 16-byte loads and stores where dst, src and bytes are all
 * multiples of 16, bytes otherwise.  `ranges` is a host array, read before
 * the call returns (the kernel gets the ranges as arguments, so the call can
 * be captured into a CUDA graph).  Zero-byte ranges are allowed; a null dst
 * or src with bytes > 0, n out of range or ranges null: INVALID, nothing is
 * enqueued.  Ordered like any kernel on the stream. */
pks_status pks_stage_copy(const pks_copy_range* ranges, int32_t n, pks_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* PKS_H */
