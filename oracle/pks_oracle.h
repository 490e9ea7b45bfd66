/*
 * CPU oracle for the top-k sparse attention decode step over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
 * calls this code, and this code includes nothing from the product.  It is a
 * plain, slow, obviously correct statement of what the decode step computes,
 * in int64 for integer work and double precision for floating point, used by
 * the tests and by the benchmark's CPU-baseline leg.
 *
 * Sources (cited by title and section):
 *  [SA]  "Sparse Attention on GLM5.3 and HBM" - HiSparse paragraph (LRU
 *        offload, load on top-k miss), DeepSeek Sparse Attention / lightning
 *        indexer paragraph (indexer score, top-K shared across heads, dense
 *        below K).
 *  [PKV] "Paged KV cache, or why reserving for the maximum length is wasteful"
 *        - sections "Internal fragmentation" (worked table), "Paging"
 *        (pages = ceil(len / page size), tail check rule), "How many users"
 *        (capacity), "Page sharing" (saved pages formula), "What this table
 *        does not say" (free list, page-table cost).
 *  [LIN] "Why recalling an old conversation costs so much" - "The benefit is
 *        clearly measurable" (LRU under sequential access), "Three blockers"
 *        (logical vs physical slot ids).
 *
 * Conventions: bf16 values are passed as their raw 16-bit patterns (uint16_t).
 * All arrays are dense row-major.  Functions return 0 on success and a
 * negative code on a violated precondition.
 */
#ifndef PKS_ORACLE_H
#define PKS_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* [PKV] "Paging": pages a request of len tokens holds = ceil(len / page_size). */
int64_t orc_pages_for(int64_t len, int64_t page_size);

/* [PKV] "Paging": tokens left empty in the last page = pages*page_size - len. */
int64_t orc_tail_waste(int64_t len, int64_t page_size);

/* [PKV] "Page sharing" + "Paging": build every request's block table.
 *  Requests are served in ascending order; each takes its logical pages in
 *  ascending order from the front of a FIFO free list (free_order, or
 *  0..num_pages-1 when NULL).  Prefix sharing: logical page p of request b is
 *  an alias when b belongs to a prefix group (group[b] >= 0), the page lies
 *  fully inside the shared prefix (p < floor(prefix_len / page_size)) and
 *  fully inside the request (p < floor(len_b / page_size)), and an earlier
 *  member of the group already holds such a page p; the first member needing
 *  page p allocates it.
 *  Output: block_table [B, max_pages] (unused entries -1), *pages_used.
 *  Returns 0, -1 if a request needs more than max_pages pages, -2 if the pool
 *  runs out, -3 on bad arguments. */
int orc_build_block_table(int32_t B, const int32_t* lens, const int32_t* group,
                          int32_t prefix_len, int32_t page_size, int32_t max_pages,
                          int32_t num_pages, const int32_t* free_order,
                          int32_t* block_table, int32_t* pages_used);

/* [PKV] "How many users": requests arrive cyclically in list order and never
 *  finish; admit until the next one does not fit.  Paged: a request takes
 *  ceil(len/page_size)*page_size slots.  Naive: every request takes `reserve`
 *  slots.  Return the number admitted. */
int64_t orc_capacity_paged(int32_t n, const int32_t* lens, int32_t page_size, int64_t slots);
int64_t orc_capacity_naive(int32_t n, const int32_t* lens, int32_t reserve, int64_t slots);

/* [SA] lightning indexer: for every cached token t < len_b,
 *    s[b,t] = sum_h w[h] * max(0, sum_d q_idx[b,h,d] * k_idx[phys(b,t), d])
 *  with phys(b,t) = block_table[b][t / page_size] * page_size + t % page_size,
 *  k_idx the single-head int8 indexer key pool [num_pages*page_size, Di].
 *  Scores written to scores[b*ld + t] (int64); other entries untouched. */
int orc_indexer_scores(int32_t B, const int32_t* lens, const int32_t* block_table,
                       int32_t max_pages, int32_t page_size, int32_t Hi, int32_t Di,
                       const int8_t* q_idx, const int32_t* w_idx, const int8_t* idx_k,
                       int64_t* scores, int64_t ld);

/* [SA] top-K selection shared across heads: when len_b <= k every token is
 *  kept (dense); otherwise the k tokens that come first when sorted by
 *  (score descending, token index ascending).  Output idx [B, k]: the chosen
 *  token indices in ascending order, padded with -1. */
int orc_topk(int32_t B, const int32_t* lens, const int64_t* scores, int64_t ld, int32_t k,
             int32_t* idx);

/* [SA] lightning indexer with real-valued head weights (the DSA form: a
 *  weighted sum of the heads' ReLU logits).  w_f: float [B, Hi], per request.
 *    s[b,t] = sum_h w_f[b,h] * max(0, q_idx[b,h,:] . k_idx[phys(b,t),:])
 *  evaluated in fp32 with the heads in order 0..Hi-1, each product and each
 *  sum rounded to nearest on its own (no fused multiply-add); the integer
 *  dot products are exact and below 2^24, so their conversion is exact.
 *  The pages fix no summation order: this order is the convention both sides
 *  of the parity check follow.  Scores to scores[b*ld + t] (float). */
int orc_indexer_scores_f(int32_t B, const int32_t* lens, const int32_t* block_table,
                         int32_t max_pages, int32_t page_size, int32_t Hi, int32_t Di,
                         const int8_t* q_idx, const float* w_f, const int8_t* idx_k,
                         float* scores, int64_t ld);

/* The value of an FP8 e4m3 code (NaN for 0x7f / 0xff). */
double orc_e4m3_value(uint8_t b);

/* [SA] lightning indexer on FP8 e4m3 queries and keys with real head weights
 *  (float [B, Hi]): s[b,t] = sum_h w_f[b,h] * max(0, q . k) with every dot
 *  product exact (e4m3 values are integer multiples of 2^-9, so a dot is an
 *  exact int64 count of 2^-18) and the weighted sum in float64.  This is the
 *  exact reference the kernel's fp32 tensor-core result is held against
 *  within a rounding bound; the selection is checked for validity against it.
 *  Returns -5 if a NaN code occurs. */
int orc_indexer_scores_fp8(int32_t B, const int32_t* lens, const int32_t* block_table,
                           int32_t max_pages, int32_t page_size, int32_t Hi, int32_t Di,
                           const uint8_t* q_idx, const float* w_f, const uint8_t* idx_k,
                           double* scores, int64_t ld);

/* orc_topk on float scores: (score descending, token ascending), -0 == +0. */
int orc_topk_f(int32_t B, const int32_t* lens, const float* scores, int64_t ld, int32_t k,
               int32_t* idx);

/* [SA] scaled dot-product attention over the selected tokens only:
 *    o[b,h] = sum_j softmax_j(q[b,h] . K_j / sqrt(D)) V_j,
 *  j over the tokens idx[b, :] >= 0, K_j / V_j read through the block table
 *  from pools [num_pages, page_size, Hkv, D], kv head = h / (Hq / Hkv).
 *  A request with no selected token gets o = 0.  out: double [B, Hq, D]. */
int orc_sparse_attention(int32_t B, const int32_t* block_table, int32_t max_pages,
                         int32_t page_size, int32_t Hq, int32_t Hkv, int32_t D, int32_t k,
                         const int32_t* idx, const uint16_t* q, const uint16_t* kv_k,
                         const uint16_t* kv_v, double* out);

/* [SA] DeepSeek Sparse Attention: the sparse MLA runs in MQA mode.  Every
 *  token holds one latent row of d + r values (latent part d, RoPE part r),
 *  shared by all H query heads; the key is the whole row, the value its first
 *  d values:
 *    o[b,h] = sum_j softmax_j(scale * q[b,h] . kv_j) kv_j[0:d],
 *  j over the tokens idx[b, :] >= 0, kv_j = kv[phys(b, t_j)] read through the
 *  block table from the pool [num_pages, page_size, d + r].  q: [B, H, d + r].
 *  A request with no selected token gets o = 0.  out: double [B, H, d]. */
int orc_mla_sparse_attention(int32_t B, const int32_t* block_table, int32_t max_pages,
                             int32_t page_size, int32_t H, int32_t d, int32_t r, int32_t k,
                             const int32_t* idx, const uint16_t* q, const uint16_t* kv,
                             double scale, double* out);

/* Residency table ([SA] HiSparse: LRU cache of KV pages in HBM, pages loaded on
 *  a top-k miss, evicted by least recent use).  State (caller arrays):
 *  page_slot [num_pages] (-1 = not resident), slot_page [capacity] (-1 = empty),
 *  last_use [capacity] (-1 = never), *step (0 after init). */
int orc_residency_init(int32_t num_pages, int32_t capacity, int32_t n_init,
                       const int32_t* init_pages, int32_t* page_slot, int32_t* slot_page,
                       int32_t* last_use, int32_t* step);

/* One step: A = distinct physical pages holding a selected token of any
 *  request.  miss_list = A minus the resident set, ascending; hits get
 *  last_use = step; victims = slots not holding a page of A, ordered by
 *  (last_use ascending, slot ascending); the i-th miss takes the i-th victim's
 *  slot (last_use = step); misses beyond the number of victims are reported
 *  but not admitted.  miss_list must hold num_pages entries.  n_hit counts
 *  |A intersect resident|. */
int orc_residency_step(int32_t num_pages, int32_t capacity, int32_t* page_slot,
                       int32_t* slot_page, int32_t* last_use, int32_t* step, int32_t B,
                       int32_t k, int32_t page_size, int32_t max_pages, const int32_t* idx,
                       const int32_t* block_table, int32_t* miss_list, int32_t* n_miss,
                       int32_t* n_hit);

/* Threads the OpenMP parts may use (0 = runtime default); returns the count in effect. */
int orc_set_threads(int n);

#ifdef __cplusplus
}
#endif
#endif
