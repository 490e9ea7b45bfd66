/*
 * CPU oracle - TEST INFRASTRUCTURE ONLY (see pks_oracle.h for the contract
 * and the sources).  Plain loops, int64 / double arithmetic, a library sort
 * as the only non-trivial primitive.  OpenMP only splits independent
 * requests or tokens across threads; it never changes an arithmetic order
 * that affects a result (each output element is computed by one thread in
 * the order written below).
 */
#include "pks_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

int orc_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
  return omp_get_max_threads();
#else
  (void)n;
  return 1;
#endif
}

/* ------------------------------------------------------------------ paging */

int64_t orc_pages_for(int64_t len, int64_t page_size) {
  /* [PKV] "Paging": number of pages = ceil(length / page size) */
  return (len + page_size - 1) / page_size;
}

int64_t orc_tail_waste(int64_t len, int64_t page_size) {
  /* [PKV] "Paging": only the tail of the last page is left empty */
  return orc_pages_for(len, page_size) * page_size - len;
}

int orc_build_block_table(int32_t B, const int32_t* lens, const int32_t* group,
                          int32_t prefix_len, int32_t page_size, int32_t max_pages,
                          int32_t num_pages, const int32_t* free_order,
                          int32_t* block_table, int32_t* pages_used) {
  if (B < 0 || page_size <= 0 || max_pages < 0 || num_pages < 0 || prefix_len < 0) return -3;
  for (int64_t i = 0; i < (int64_t)B * max_pages; ++i) block_table[i] = -1;

  /* [PKV] "Page sharing": only whole pages of the prefix can be shared. */
  const int32_t prefix_pages = prefix_len / page_size;

  /* group id -> the physical page each shared prefix page index was given */
  int32_t n_groups = 0;
  int32_t* group_ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)(B > 0 ? B : 1));
  int32_t* shared = (int32_t*)malloc(sizeof(int32_t) * (size_t)(B > 0 ? B : 1) *
                                     (size_t)(prefix_pages > 0 ? prefix_pages : 1));

  int32_t next_free = 0; /* FIFO free list: pop from the front */
  int rc = 0;
  for (int32_t b = 0; b < B && rc == 0; ++b) {
    const int64_t pages = orc_pages_for(lens[b], page_size);
    if (lens[b] < 0) { rc = -3; break; }
    if (pages > max_pages) { rc = -1; break; }

    int32_t gslot = -1;
    if (group != NULL && group[b] >= 0) {
      for (int32_t g = 0; g < n_groups; ++g)
        if (group_ids[g] == group[b]) gslot = g;
      if (gslot < 0) {
        gslot = n_groups++;
        group_ids[gslot] = group[b];
        for (int32_t p = 0; p < prefix_pages; ++p) shared[(int64_t)gslot * prefix_pages + p] = -1;
      }
    }
    const int32_t full_pages = lens[b] / page_size;
    for (int64_t p = 0; p < pages; ++p) {
      const int shareable = gslot >= 0 && p < prefix_pages && p < full_pages;
      if (shareable && shared[(int64_t)gslot * prefix_pages + p] >= 0) {
        block_table[(int64_t)b * max_pages + p] = shared[(int64_t)gslot * prefix_pages + p];
        continue;
      }
      if (next_free >= num_pages) { rc = -2; break; }
      const int32_t page = free_order ? free_order[next_free] : next_free;
      ++next_free;
      block_table[(int64_t)b * max_pages + p] = page;
      if (shareable) shared[(int64_t)gslot * prefix_pages + p] = page;
    }
  }
  free(group_ids);
  free(shared);
  if (pages_used) *pages_used = next_free;
  return rc;
}

int64_t orc_capacity_paged(int32_t n, const int32_t* lens, int32_t page_size, int64_t slots) {
  /* [PKV] "How many users": cyclic arrivals, never finishing, admit until the
   * next request does not fit */
  if (n <= 0 || page_size <= 0) return 0;
  int64_t cycle = 0;
  for (int32_t i = 0; i < n; ++i) cycle += orc_pages_for(lens[i], page_size) * page_size;
  if (cycle <= 0) return -1; /* requests that take no slots: unbounded */
  int64_t used = 0, admitted = 0;
  for (int64_t i = 0;; ++i) {
    const int64_t need = orc_pages_for(lens[i % n], page_size) * page_size;
    if (used + need > slots) return admitted;
    used += need;
    ++admitted;
  }
}

int64_t orc_capacity_naive(int32_t n, const int32_t* lens, int32_t reserve, int64_t slots) {
  /* [PKV] "Internal fragmentation": every request reserves the maximum length */
  if (n <= 0 || reserve <= 0) return 0;
  int64_t used = 0, admitted = 0;
  for (int64_t i = 0;; ++i) {
    if (lens[i % n] > reserve) return admitted; /* does not fit its reservation */
    if (used + reserve > slots) return admitted;
    used += reserve;
    ++admitted;
  }
}

/* ----------------------------------------------------------------- indexer */

static int64_t phys_token(const int32_t* block_table, int32_t max_pages, int32_t page_size,
                          int32_t b, int64_t t) {
  /* [PKV] "Paging": the page table says where each page lives */
  const int32_t page = block_table[(int64_t)b * max_pages + t / page_size];
  return (int64_t)page * page_size + t % page_size;
}

int orc_indexer_scores(int32_t B, const int32_t* lens, const int32_t* block_table,
                       int32_t max_pages, int32_t page_size, int32_t Hi, int32_t Di,
                       const int8_t* q_idx, const int32_t* w_idx, const int8_t* idx_k,
                       int64_t* scores, int64_t ld) {
  if (B < 0 || Hi <= 0 || Di <= 0 || page_size <= 0) return -3;
  for (int32_t b = 0; b < B; ++b) {
    if (lens[b] > (int64_t)max_pages * page_size || lens[b] > ld) return -3;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < lens[b]; ++t) {
      const int8_t* key = idx_k + phys_token(block_table, max_pages, page_size, b, t) * Di;
      int64_t s = 0;
      for (int32_t h = 0; h < Hi; ++h) {
        /* [SA] indexer: query-key dot product, then ReLU, then the weighted
         * sum over the indexer's query heads */
        const int8_t* qh = q_idx + ((int64_t)b * Hi + h) * Di;
        int64_t dot = 0;
        for (int32_t d = 0; d < Di; ++d) dot += (int64_t)qh[d] * (int64_t)key[d];
        const int64_t relu = dot > 0 ? dot : 0;
        s += (int64_t)w_idx[h] * relu;
      }
      scores[(int64_t)b * ld + t] = s;
    }
  }
  return 0;
}

/* ------------------------------------------------------------------ top-k */

typedef struct {
  int64_t score;
  int32_t t;
} scored_token;

static int by_score_desc_index_asc(const void* pa, const void* pb) {
  const scored_token* a = (const scored_token*)pa;
  const scored_token* b = (const scored_token*)pb;
  if (a->score != b->score) return a->score > b->score ? -1 : 1;
  return (a->t > b->t) - (a->t < b->t);
}

static int int32_asc(const void* pa, const void* pb) {
  const int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
  return (a > b) - (a < b);
}

int orc_topk(int32_t B, const int32_t* lens, const int64_t* scores, int64_t ld, int32_t k,
             int32_t* idx) {
  if (B < 0 || k <= 0) return -3;
  int rc = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int32_t b = 0; b < B; ++b) {
    int32_t* row = idx + (int64_t)b * k;
    for (int32_t j = 0; j < k; ++j) row[j] = -1;
    const int32_t len = lens[b];
    if (len <= k) {
      /* [SA] queries that attend to fewer than K tokens stay dense */
      for (int32_t t = 0; t < len; ++t) row[t] = t;
      continue;
    }
    scored_token* all = (scored_token*)malloc(sizeof(scored_token) * (size_t)len);
    if (!all) { rc = -4; continue; }
    for (int32_t t = 0; t < len; ++t) {
      all[t].score = scores[(int64_t)b * ld + t];
      all[t].t = t;
    }
    /* [SA] top-K by indexer score; equal scores go to the lower token index */
    qsort(all, (size_t)len, sizeof(scored_token), by_score_desc_index_asc);
    for (int32_t j = 0; j < k; ++j) row[j] = all[j].t;
    free(all);
    qsort(row, (size_t)k, sizeof(int32_t), int32_asc); /* canonical order */
  }
  return rc;
}

/* ------------------------------------------- indexer with real head weights */

int orc_indexer_scores_f(int32_t B, const int32_t* lens, const int32_t* block_table,
                         int32_t max_pages, int32_t page_size, int32_t Hi, int32_t Di,
                         const int8_t* q_idx, const float* w_f, const int8_t* idx_k,
                         float* scores, int64_t ld) {
  if (B < 0 || Hi <= 0 || Di <= 0 || page_size <= 0) return -3;
#pragma omp parallel for schedule(dynamic, 1)
  for (int32_t b = 0; b < B; ++b) {
    for (int32_t t = 0; t < lens[b]; ++t) {
      const int8_t* key = idx_k + phys_token(block_table, max_pages, page_size, b, t) * Di;
      /* [SA] weighted sum of the heads' ReLU logits, in fp32: heads in
       * order, each product and each sum rounded to nearest on its own */
      float s = 0.0f;
      for (int32_t h = 0; h < Hi; ++h) {
        const int8_t* qh = q_idx + ((int64_t)b * Hi + h) * Di;
        int64_t dot = 0;
        for (int32_t d = 0; d < Di; ++d) dot += (int64_t)qh[d] * (int64_t)key[d];
        const float relu = (float)(dot > 0 ? dot : 0); /* exact: below 2^24 */
        const float prod = w_f[(int64_t)b * Hi + h] * relu;
        s = s + prod;
      }
      scores[(int64_t)b * ld + t] = s;
    }
  }
  return 0;
}

/* FP8 e4m3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; no
 * infinities, 0x7f / 0xff are NaN) as an integer multiple of 2^-9:
 * subnormals m * 2^-9, normals (8 + m) * 2^(e - 1) * 2^-9.  Returns 0 and sets
 * *nan for a NaN code. */
static int64_t e4m3_units(uint8_t b, int* nan) {
  const int e = (b >> 3) & 15, m = b & 7;
  if (e == 15 && m == 7) {
    *nan = 1;
    return 0;
  }
  const int64_t mag = e == 0 ? (int64_t)m : (int64_t)(8 + m) << (e - 1);
  return (b & 0x80) ? -mag : mag;
}

double orc_e4m3_value(uint8_t b) {
  int nan = 0;
  const int64_t u = e4m3_units(b, &nan);
  return nan ? NAN : ldexp((double)u, -9);
}

int orc_indexer_scores_fp8(int32_t B, const int32_t* lens, const int32_t* block_table,
                           int32_t max_pages, int32_t page_size, int32_t Hi, int32_t Di,
                           const uint8_t* q_idx, const float* w_f, const uint8_t* idx_k,
                           double* scores, int64_t ld) {
  if (B < 0 || Hi <= 0 || Di <= 0 || page_size <= 0) return -3;
  int rc = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int32_t b = 0; b < B; ++b) {
    for (int32_t t = 0; t < lens[b]; ++t) {
      const uint8_t* key = idx_k + phys_token(block_table, max_pages, page_size, b, t) * Di;
      double s = 0.0;
      for (int32_t h = 0; h < Hi; ++h) {
        const uint8_t* qh = q_idx + ((int64_t)b * Hi + h) * Di;
        /* the dot product exactly: products of 2^-9 units are 2^-18 units,
         * the int64 sum is exact, and so is its conversion (below 2^53) */
        int64_t dot = 0;
        int nan = 0;
        for (int32_t d = 0; d < Di; ++d) dot += e4m3_units(qh[d], &nan) * e4m3_units(key[d], &nan);
        if (nan) rc = -5;
        const double relu = dot > 0 ? ldexp((double)dot, -18) : 0.0;
        /* [SA] weighted sum of the heads' ReLU logits (float64) */
        s += (double)w_f[(int64_t)b * Hi + h] * relu;
      }
      scores[(int64_t)b * ld + t] = s;
    }
  }
  return rc;
}

typedef struct {
  float score;
  int32_t t;
} fscored_token;

static int by_fscore_desc_index_asc(const void* x, const void* y) {
  const fscored_token* a = (const fscored_token*)x;
  const fscored_token* b = (const fscored_token*)y;
  if (a->score != b->score) return a->score > b->score ? -1 : 1;
  return (a->t > b->t) - (a->t < b->t);
}

int orc_topk_f(int32_t B, const int32_t* lens, const float* scores, int64_t ld, int32_t k,
               int32_t* idx) {
  if (B < 0 || k <= 0) return -3;
  int rc = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int32_t b = 0; b < B; ++b) {
    int32_t* row = idx + (int64_t)b * k;
    for (int32_t j = 0; j < k; ++j) row[j] = -1;
    const int32_t len = lens[b];
    if (len <= k) {
      for (int32_t t = 0; t < len; ++t) row[t] = t; /* [SA] dense below K */
      continue;
    }
    fscored_token* all = (fscored_token*)malloc(sizeof(fscored_token) * (size_t)len);
    if (!all) { rc = -4; continue; }
    for (int32_t t = 0; t < len; ++t) {
      all[t].score = scores[(int64_t)b * ld + t];
      all[t].t = t;
    }
    /* [SA] top-K by indexer score; equal scores (-0 equals +0) go to the lower index */
    qsort(all, (size_t)len, sizeof(fscored_token), by_fscore_desc_index_asc);
    for (int32_t j = 0; j < k; ++j) row[j] = all[j].t;
    free(all);
    qsort(row, (size_t)k, sizeof(int32_t), int32_asc);
  }
  return rc;
}

/* -------------------------------------------------------------- attention */

static double bf16_to_double(uint16_t bits) {
  /* bf16 is the upper half of an IEEE binary32 */
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

int orc_sparse_attention(int32_t B, const int32_t* block_table, int32_t max_pages,
                         int32_t page_size, int32_t Hq, int32_t Hkv, int32_t D, int32_t k,
                         const int32_t* idx, const uint16_t* q, const uint16_t* kv_k,
                         const uint16_t* kv_v, double* out) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || k <= 0) return -3;
  const int32_t G = Hq / Hkv;
  const double scale = 1.0 / sqrt((double)D);
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int32_t b = 0; b < B; ++b) {
    for (int32_t h = 0; h < Hq; ++h) {
      const int32_t kvh = h / G; /* query heads share a KV head in contiguous groups */
      const uint16_t* qh = q + ((int64_t)b * Hq + h) * D;
      double* o = out + ((int64_t)b * Hq + h) * D;
      for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
      double* logit = (double*)malloc(sizeof(double) * (size_t)k);
      int64_t* row = (int64_t*)malloc(sizeof(int64_t) * (size_t)k);
      int32_t n = 0;
      double m = -INFINITY;
      for (int32_t j = 0; j < k; ++j) {
        const int32_t t = idx[(int64_t)b * k + j];
        if (t < 0) continue;
        const int64_t r = (phys_token(block_table, max_pages, page_size, b, t) * Hkv + kvh) * D;
        double dot = 0.0;
        for (int32_t d = 0; d < D; ++d) dot += bf16_to_double(qh[d]) * bf16_to_double(kv_k[r + d]);
        logit[n] = dot * scale; /* [SA] scaled dot-product */
        row[n] = r;
        if (logit[n] > m) m = logit[n];
        ++n;
      }
      if (n > 0) {
        double l = 0.0;
        for (int32_t j = 0; j < n; ++j) l += exp(logit[j] - m);
        for (int32_t j = 0; j < n; ++j) {
          const double p = exp(logit[j] - m) / l; /* softmax over the selected tokens */
          for (int32_t d = 0; d < D; ++d) o[d] += p * bf16_to_double(kv_v[row[j] + d]);
        }
      }
      free(logit);
      free(row);
    }
  }
  return 0;
}

/* ------------------------------------------------- MLA in MQA mode (DSA) */

int orc_mla_sparse_attention(int32_t B, const int32_t* block_table, int32_t max_pages,
                             int32_t page_size, int32_t H, int32_t d, int32_t r, int32_t k,
                             const int32_t* idx, const uint16_t* q, const uint16_t* kv,
                             double scale, double* out) {
  if (B < 0 || H <= 0 || d <= 0 || r < 0 || k <= 0 || !(scale > 0.0)) return -3;
  const int32_t dk = d + r; /* key width: latent plus RoPE part */
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int32_t b = 0; b < B; ++b) {
    for (int32_t h = 0; h < H; ++h) {
      const uint16_t* qh = q + ((int64_t)b * H + h) * dk;
      double* o = out + ((int64_t)b * H + h) * d;
      for (int32_t c = 0; c < d; ++c) o[c] = 0.0;
      double* logit = (double*)malloc(sizeof(double) * (size_t)k);
      int64_t* row = (int64_t*)malloc(sizeof(int64_t) * (size_t)k);
      int32_t n = 0;
      double m = -INFINITY;
      for (int32_t j = 0; j < k; ++j) {
        const int32_t t = idx[(int64_t)b * k + j];
        if (t < 0) continue;
        /* [SA] MQA mode: one latent row per token, shared by every query head */
        const int64_t base = phys_token(block_table, max_pages, page_size, b, t) * dk;
        double dot = 0.0;
        for (int32_t c = 0; c < dk; ++c) dot += bf16_to_double(qh[c]) * bf16_to_double(kv[base + c]);
        logit[n] = dot * scale;
        row[n] = base;
        if (logit[n] > m) m = logit[n];
        ++n;
      }
      if (n > 0) {
        double l = 0.0;
        for (int32_t j = 0; j < n; ++j) l += exp(logit[j] - m);
        for (int32_t j = 0; j < n; ++j) {
          const double p = exp(logit[j] - m) / l;
          /* [SA] the value is the latent part only (the first d of the d + r) */
          for (int32_t c = 0; c < d; ++c) o[c] += p * bf16_to_double(kv[row[j] + c]);
        }
      }
      free(logit);
      free(row);
    }
  }
  return 0;
}

/* -------------------------------------------------------------- residency */

int orc_residency_init(int32_t num_pages, int32_t capacity, int32_t n_init,
                       const int32_t* init_pages, int32_t* page_slot, int32_t* slot_page,
                       int32_t* last_use, int32_t* step) {
  if (num_pages < 0 || capacity < 0 || n_init < 0 || n_init > capacity) return -3;
  for (int32_t p = 0; p < num_pages; ++p) page_slot[p] = -1;
  for (int32_t s = 0; s < capacity; ++s) {
    slot_page[s] = -1;
    last_use[s] = -1;
  }
  /* initial pages go to slots 0.. in ascending page order, last use 0 */
  int32_t* sorted = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n_init > 0 ? n_init : 1));
  memcpy(sorted, init_pages, sizeof(int32_t) * (size_t)n_init);
  qsort(sorted, (size_t)n_init, sizeof(int32_t), int32_asc);
  int rc = 0;
  for (int32_t i = 0; i < n_init; ++i) {
    const int32_t p = sorted[i];
    if (p < 0 || p >= num_pages || page_slot[p] >= 0) { rc = -3; break; }
    page_slot[p] = i;
    slot_page[i] = p;
    last_use[i] = 0;
  }
  free(sorted);
  *step = 0;
  return rc;
}

typedef struct {
  int32_t last_use;
  int32_t slot;
} victim;

static int by_last_use_then_slot(const void* pa, const void* pb) {
  const victim* a = (const victim*)pa;
  const victim* b = (const victim*)pb;
  if (a->last_use != b->last_use) return (a->last_use > b->last_use) - (a->last_use < b->last_use);
  return (a->slot > b->slot) - (a->slot < b->slot);
}

int orc_residency_step(int32_t num_pages, int32_t capacity, int32_t* page_slot,
                       int32_t* slot_page, int32_t* last_use, int32_t* step, int32_t B,
                       int32_t k, int32_t page_size, int32_t max_pages, const int32_t* idx,
                       const int32_t* block_table, int32_t* miss_list, int32_t* n_miss,
                       int32_t* n_hit) {
  if (num_pages < 0 || capacity < 0 || B < 0 || k <= 0 || page_size <= 0) return -3;
  const int32_t t_now = ++*step;

  /* A: the distinct physical pages that hold a selected token */
  unsigned char* accessed = (unsigned char*)calloc((size_t)(num_pages > 0 ? num_pages : 1), 1);
  for (int32_t b = 0; b < B; ++b)
    for (int32_t j = 0; j < k; ++j) {
      const int32_t t = idx[(int64_t)b * k + j];
      if (t < 0) continue;
      const int32_t page = block_table[(int64_t)b * max_pages + t / page_size];
      if (page < 0 || page >= num_pages) { free(accessed); return -3; }
      accessed[page] = 1;
    }

  /* [SA] HiSparse: selected pages not in HBM are the misses, in page order */
  int32_t misses = 0, hits = 0;
  for (int32_t p = 0; p < num_pages; ++p) {
    if (!accessed[p]) continue;
    if (page_slot[p] < 0) miss_list[misses++] = p;
    else ++hits;
  }

  /* LRU victims: slots whose page is not needed now, least recently used
   * first, ties by slot number */
  victim* v = (victim*)malloc(sizeof(victim) * (size_t)(capacity > 0 ? capacity : 1));
  int32_t n_v = 0;
  for (int32_t s = 0; s < capacity; ++s) {
    const int32_t p = slot_page[s];
    if (p >= 0 && accessed[p]) {
      last_use[s] = t_now; /* hit */
      continue;
    }
    v[n_v].last_use = last_use[s];
    v[n_v].slot = s;
    ++n_v;
  }
  qsort(v, (size_t)n_v, sizeof(victim), by_last_use_then_slot);

  const int32_t admit = misses < n_v ? misses : n_v;
  for (int32_t i = 0; i < admit; ++i) {
    const int32_t s = v[i].slot;
    if (slot_page[s] >= 0) page_slot[slot_page[s]] = -1; /* evict */
    slot_page[s] = miss_list[i];
    page_slot[miss_list[i]] = s;
    last_use[s] = t_now;
  }
  free(v);
  free(accessed);
  *n_miss = misses;
  if (n_hit) *n_hit = hits;
  return 0;
}
