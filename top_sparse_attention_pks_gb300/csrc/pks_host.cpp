// Host side of libpks: status strings, the page allocator and block-table
// builder, argument validation, workspace layout and the C entry points.
//
// "Paged KV cache, or why reserving for the maximum length is wasteful":
// "Paging" (fixed-size pages, one page table per request, ceil paging),
// "Page sharing" (aliasing whole prefix pages), "What this table does not
// say" (the allocator keeps a free-page list).  Everything here runs on the
// host; device work is only enqueued.

#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <deque>
#include <mutex>
#include <new>
#include <vector>

#include "pks_internal.h"

struct pks_pool {
  int32_t num_pages = 0;
  int32_t page_size = 0;
  std::deque<int32_t> free_list;  // FIFO: take from the front, return to the back
  std::vector<uint8_t> is_free;
};

namespace pks {

namespace {

constexpr size_t kAlign = 256;
constexpr int kMaxB = 4096;
constexpr int kMaxK = 65536;
constexpr int64_t kMaxLen = int64_t(1) << 24;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape checks shared by every decode entry point.  Pointers are checked by
// the callers that use them.
pks_status check_shapes(const pks_decode_args* a) {
  if (!a) return PKS_ERR_INVALID;
  if (a->B < 0 || a->Hq < 1 || a->Hkv < 1 || a->D < 1 || a->Hi < 1 || a->Di < 1 ||
      a->page_size < 1 || a->max_pages < 1 || a->num_pages < 1 || a->k < 1 ||
      a->attn_splits < 0 || a->attn_splits > kAttnGridMax)
    return PKS_ERR_INVALID;
  if (a->Hq % a->Hkv != 0) return PKS_ERR_INVALID;
  if (a->topk_mode < 0 || a->topk_mode > 1) return PKS_ERR_INVALID;
  if (a->reserved[0]) return PKS_ERR_INVALID;
  if (a->n_queries < 0) return PKS_ERR_INVALID;
  // compiled: Nq in {1, 2, 4, 8} with Hi * Nq <= 8
  const int nq = query_count(*a);
  if ((nq & (nq - 1)) != 0 || (int64_t)a->Hi * nq > 8) return PKS_ERR_UNSUPPORTED;
  if ((int64_t)a->B * query_count(*a) > kMaxB) return PKS_ERR_UNSUPPORTED;
  if (a->w_idx_f && nq > 1) return PKS_ERR_UNSUPPORTED;  // real weights: one query token
  if (a->idx_fp8 < 0 || a->idx_fp8 > 1 || a->wait_limit < 0) return PKS_ERR_INVALID;
  if (a->idx_fp8 && !a->w_idx_f) return PKS_ERR_INVALID;  // FP8 scores need real weights
  if ((int64_t)a->num_pages * a->page_size > INT32_MAX) return PKS_ERR_UNSUPPORTED;
  if (a->D != 64 && a->D != 128) return PKS_ERR_UNSUPPORTED;
  if (a->Di != 64 && a->Di != 128) return PKS_ERR_UNSUPPORTED;
  if (a->Hi != 1 && a->Hi != 2 && a->Hi != 4 && a->Hi != 8) return PKS_ERR_UNSUPPORTED;
  if (a->Hq / a->Hkv > 16) return PKS_ERR_UNSUPPORTED;
  if (a->B > kMaxB || a->k > kMaxK) return PKS_ERR_UNSUPPORTED;
  if ((int64_t)a->max_pages * a->page_size > kMaxLen) return PKS_ERR_UNSUPPORTED;
  return PKS_OK;
}

pks_status check_common_ptrs(const pks_decode_args* a) {
  if (a->B == 0) return PKS_OK;
  if (!a->seq_lens || !a->block_table) return PKS_ERR_INVALID;
  return PKS_OK;
}

pks_status check_scan_ptrs(const pks_decode_args* a) {
  if (a->B == 0) return PKS_OK;
  if (!a->q_idx || (!a->w_idx && !a->w_idx_f) || !a->idx_k) return PKS_ERR_INVALID;
  if (!aligned16(a->q_idx) || !aligned16(a->idx_k)) return PKS_ERR_INVALID;
  return PKS_OK;
}

pks_status check_attn_ptrs(const pks_decode_args* a) {
  if (a->B == 0) return PKS_OK;
  if (!a->q || !a->kv_k || !a->kv_v || !a->topk_idx || !a->out) return PKS_ERR_INVALID;
  if (!aligned16(a->q) || !aligned16(a->kv_k) || !aligned16(a->kv_v)) return PKS_ERR_INVALID;
  return PKS_OK;
}

pks_status check_workspace(const pks_decode_args* a, const WorkspaceLayout& L) {
  if (!a->workspace) return PKS_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(a->workspace) & (kAlign - 1)) != 0) return PKS_ERR_WORKSPACE;
  if (a->workspace_bytes < L.total) return PKS_ERR_WORKSPACE;
  return PKS_OK;
}

pks_status from_cuda(cudaError_t e) { return e == cudaSuccess ? PKS_OK : PKS_ERR_CUDA; }

}  // namespace

WorkspaceLayout workspace_layout(const pks_decode_args& a) {
  WorkspaceLayout L{};
  const int64_t B = (int64_t)a.B * query_count(a);  // one virtual request per query token
  const int G = a.Hq / a.Hkv;
  const int64_t max_len = (int64_t)a.max_pages * a.page_size;
  L.nchunks = (int)std::max<int64_t>(1, (max_len + kTopkChunk - 1) / kTopkChunk);
  // score rows padded to whole top-k chunks, so chunk loads never leave the row
  L.ld = (int64_t)L.nchunks * kTopkChunk;

  L.attn_grid_max = kAttnGridMax;
  const int hg = attn_heads_per_cta(a.Hkv);
  const int64_t nseg = (int64_t)(a.Hkv / hg) * B;  // (head group, request) segments

  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes);
    return o;
  };
  L.ctrl = off;
  L.err = take(sizeof(int32_t) * 4);
  L.hist = take(sizeof(int32_t) * (size_t)B * kScoreBins);
  L.tick_topk = take(sizeof(int32_t) * (size_t)B);
  L.depart_topk = take(sizeof(int32_t) * (size_t)B);
  L.cand_n = take(sizeof(int32_t) * (size_t)B);
  L.ctrl_end = off;
  L.scores = take(sizeof(int32_t) * (size_t)B * (size_t)L.ld);
  L.cand = take(sizeof(int32_t) * 2 * (size_t)B * (size_t)L.ld);
  L.bits = take(sizeof(uint32_t) * (size_t)B * L.nchunks * (kTopkChunk / 32));
  L.gt_cnt = take(sizeof(int32_t) * (size_t)B * L.nchunks);
  L.chunk_cnt = take(sizeof(int32_t) * 2 * (size_t)B * L.nchunks);
  L.chunk_off = take(sizeof(int32_t) * (size_t)B * L.nchunks);
  L.thresh = take(sizeof(TopkThreshold) * (size_t)B);
  // position prefix over requests, then the attention grid for the merge
  L.attn_prefix = take(sizeof(int32_t) * (size_t)(B + 2));
  // partial (m, l, o) slots: one per (CTA, segment) pair, indexed cta + segment
  const size_t nslots = (size_t)(L.attn_grid_max + nseg) * hg * G;
  L.part_ml = take(sizeof(float) * 2 * nslots);
  L.part_o = take(sizeof(float) * nslots * a.D);
  L.total = off;
  return L;
}

int device_sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
      n = 152;
    cache[dev] = n;
  }
  return cache[dev];
}

}  // namespace pks

using pks::WorkspaceLayout;

extern "C" {

const char* pks_status_str(pks_status status) {
  switch (status) {
    case PKS_OK: return "ok";
    case PKS_ERR_INVALID: return "invalid argument";
    case PKS_ERR_OOM: return "page pool exhausted";
    case PKS_ERR_CUDA: return "CUDA runtime error";
    case PKS_ERR_TIMEOUT: return "device wait timed out";
    case PKS_ERR_DEVICE_CHECK: return "device-side bounds check failed";
    case PKS_ERR_UNSUPPORTED: return "unsupported shape";
    case PKS_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case PKS_ERR_TOO_LARGE: return "shapes need more scratch than the static buffer holds";
    default: return "unknown status";
  }
}

// ----------------------------------------------------------------- pool ---

pks_status pks_pool_create(int32_t num_pages, int32_t page_size, const int32_t* free_order,
                           pks_pool** out) {
  if (!out) return PKS_ERR_INVALID;
  *out = nullptr;
  if (num_pages < 1 || page_size < 1) return PKS_ERR_INVALID;
  pks_pool* p = new (std::nothrow) pks_pool;
  if (!p) return PKS_ERR_OOM;
  p->num_pages = num_pages;
  p->page_size = page_size;
  p->is_free.assign((size_t)num_pages, 1);
  if (free_order) {
    std::vector<uint8_t> seen((size_t)num_pages, 0);
    for (int32_t i = 0; i < num_pages; ++i) {
      const int32_t id = free_order[i];
      if (id < 0 || id >= num_pages || seen[(size_t)id]) {
        delete p;
        return PKS_ERR_INVALID;
      }
      seen[(size_t)id] = 1;
      p->free_list.push_back(id);
    }
  } else {
    for (int32_t i = 0; i < num_pages; ++i) p->free_list.push_back(i);
  }
  *out = p;
  return PKS_OK;
}

void pks_pool_destroy(pks_pool* pool) { delete pool; }

pks_status pks_pool_free_count(const pks_pool* pool, int32_t* out) {
  if (!pool || !out) return PKS_ERR_INVALID;
  *out = (int32_t)pool->free_list.size();
  return PKS_OK;
}

pks_status pks_admission_simulate(const pks_pool* pool, int32_t n, const int32_t* lens,
                                  int32_t reserve, int64_t* admitted, int64_t* tokens,
                                  int64_t* slots) {
  if (!pool || n < 1 || !lens || reserve < 0 || !admitted || !tokens || !slots)
    return PKS_ERR_INVALID;
  const int64_t P = pool->page_size;
  int64_t cycle_pages = 0;
  for (int32_t i = 0; i < n; ++i) {
    if (lens[i] < 0) return PKS_ERR_INVALID;
    cycle_pages += reserve > 0 ? (reserve + P - 1) / P : (lens[i] + P - 1) / P;
  }
  if (cycle_pages == 0) return PKS_ERR_INVALID;  // requests that take no pages: unbounded
  const int64_t free_pages = (int64_t)pool->free_list.size();
  int64_t used = 0, adm = 0, tok = 0;
  for (int64_t i = 0;; ++i) {
    const int32_t len = lens[i % n];
    if (reserve > 0 && len > reserve) break;  // does not fit its reservation
    const int64_t need = reserve > 0 ? (reserve + P - 1) / P : (len + P - 1) / P;
    if (used + need > free_pages) break;
    used += need;
    tok += len;
    ++adm;
  }
  *admitted = adm;
  *tokens = tok;
  *slots = used * P;
  return PKS_OK;
}

pks_status pks_alloc_pages(pks_pool* pool, int32_t n, int32_t* out_ids) {
  if (!pool || n < 0 || (n > 0 && !out_ids)) return PKS_ERR_INVALID;
  if ((size_t)n > pool->free_list.size()) return PKS_ERR_OOM;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t id = pool->free_list.front();
    pool->free_list.pop_front();
    pool->is_free[(size_t)id] = 0;
    out_ids[i] = id;
  }
  return PKS_OK;
}

pks_status pks_free_pages(pks_pool* pool, int32_t n, const int32_t* ids) {
  if (!pool || n < 0 || (n > 0 && !ids)) return PKS_ERR_INVALID;
  std::vector<uint8_t> seen;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t id = ids[i];
    if (id < 0 || id >= pool->num_pages || pool->is_free[(size_t)id]) return PKS_ERR_INVALID;
    if (seen.empty()) seen.assign((size_t)pool->num_pages, 0);
    if (seen[(size_t)id]) return PKS_ERR_INVALID;
    seen[(size_t)id] = 1;
  }
  for (int32_t i = 0; i < n; ++i) {
    pool->is_free[(size_t)ids[i]] = 1;
    pool->free_list.push_back(ids[i]);
  }
  return PKS_OK;
}

pks_status pks_build_block_table(pks_pool* pool, int32_t batch, const int32_t* seq_lens,
                                 const int32_t* prefix_group, int32_t prefix_len,
                                 int32_t max_pages, int32_t* block_table, int32_t* pages_used) {
  if (!pool || batch < 0 || max_pages < 1 || prefix_len < 0) return PKS_ERR_INVALID;
  if (batch > 0 && (!seq_lens || !block_table)) return PKS_ERR_INVALID;
  const int64_t P = pool->page_size;
  std::fill(block_table, block_table + (int64_t)batch * max_pages, -1);
  for (int32_t b = 0; b < batch; ++b) {
    if (seq_lens[b] < 0) return PKS_ERR_INVALID;
    if ((seq_lens[b] + P - 1) / P > max_pages) return PKS_ERR_INVALID;
  }
  // "Page sharing": whole prefix pages only
  const int32_t prefix_pages = (int32_t)(prefix_len / P);
  struct Group {
    int32_t id;
    std::vector<int32_t> page;  // physical page given to each shared prefix page index
  };
  std::vector<Group> groups;
  std::vector<int32_t> taken;
  pks_status st = PKS_OK;
  for (int32_t b = 0; b < batch && st == PKS_OK; ++b) {
    Group* g = nullptr;
    if (prefix_group && prefix_group[b] >= 0) {
      for (auto& x : groups)
        if (x.id == prefix_group[b]) g = &x;
      if (!g) {
        groups.push_back(Group{prefix_group[b], std::vector<int32_t>((size_t)prefix_pages, -1)});
        g = &groups.back();
      }
    }
    const int64_t pages = (seq_lens[b] + P - 1) / P;
    const int64_t full = seq_lens[b] / P;
    for (int64_t p = 0; p < pages; ++p) {
      const bool shareable = g && p < prefix_pages && p < full;
      if (shareable && g->page[(size_t)p] >= 0) {
        block_table[(int64_t)b * max_pages + p] = g->page[(size_t)p];
        continue;
      }
      int32_t id;
      st = pks_alloc_pages(pool, 1, &id);
      if (st != PKS_OK) break;
      taken.push_back(id);
      block_table[(int64_t)b * max_pages + p] = id;
      if (shareable) g->page[(size_t)p] = id;
    }
  }
  if (st != PKS_OK) {
    pks_free_pages(pool, (int32_t)taken.size(), taken.data());
    std::fill(block_table, block_table + (int64_t)batch * max_pages, -1);
    if (pages_used) *pages_used = 0;
    return st;
  }
  if (pages_used) *pages_used = (int32_t)taken.size();
  return PKS_OK;
}

// --------------------------------------------------------------- decode ---

pks_status pks_decode_workspace_size(const pks_decode_args* args, size_t* bytes) {
  if (!bytes) return PKS_ERR_INVALID;
  const pks_status st = pks::check_shapes(args);
  if (st != PKS_OK) return st;
  *bytes = pks::workspace_layout(*args).total;
  return PKS_OK;
}

pks_status pks_decode_workspace_init(const pks_decode_args* args, pks_stream stream) {
  pks_status st = pks::check_shapes(args);
  if (st != PKS_OK) return st;
  const WorkspaceLayout L = pks::workspace_layout(*args);
  if ((st = pks::check_workspace(args, L)) != PKS_OK) return st;
  return pks::from_cuda(cudaMemsetAsync(args->workspace, 0, L.ctrl_end,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

static pks_status decode_impl(const pks_decode_args* args, pks_stream stream,
                              pks_event const* ev, bool attention = true) {
  pks_status st = pks::check_shapes(args);
  if (st != PKS_OK) return st;
  if ((st = pks::check_common_ptrs(args)) != PKS_OK) return st;
  if ((st = pks::check_scan_ptrs(args)) != PKS_OK) return st;
  if (args->B > 0 && !args->topk_idx) return PKS_ERR_INVALID;
  if (attention && (st = pks::check_attn_ptrs(args)) != PKS_OK) return st;
  const WorkspaceLayout L = pks::workspace_layout(*args);
  if ((st = pks::check_workspace(args, L)) != PKS_OK) return st;
  if (args->B == 0) return PKS_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(args->workspace);
  auto rec = [&](int i) -> cudaError_t {
    if (ev && ev[i]) return cudaEventRecord(reinterpret_cast<cudaEvent_t>(ev[i]), s);
    return cudaSuccess;
  };
  cudaError_t e = rec(0);
  if (e == cudaSuccess)
    e = pks::launch_indexer_scan(*args, reinterpret_cast<int32_t*>(ws + L.scores), L.ld,
                                 reinterpret_cast<int32_t*>(ws + L.hist),
                                 reinterpret_cast<int32_t*>(ws + L.err), s);
  if (e == cudaSuccess) e = rec(1);
  if (e == cudaSuccess) e = pks::launch_topk(*args, L, ws, s);
  if (e == cudaSuccess) e = rec(2);
  if (attention && e == cudaSuccess) e = pks::launch_attention(*args, L, ws, /*trim=*/true, s);
  if (e == cudaSuccess) e = rec(3);
  return pks::from_cuda(e);
}

pks_status pks_decode_select(const pks_decode_args* args, pks_stream stream) {
  return decode_impl(args, stream, nullptr, /*attention=*/false);
}

pks_status pks_decode_step(const pks_decode_args* args, pks_stream stream) {
  return decode_impl(args, stream, nullptr);
}

pks_status pks_decode_launches(const pks_decode_args* args, int32_t* launches) {
  if (!launches) return PKS_ERR_INVALID;
  pks_status st = pks::check_shapes(args);
  if (st != PKS_OK) return st;
  const WorkspaceLayout L = pks::workspace_layout(*args);
  *launches = args->B == 0 ? 0 : 1 + pks::topk_kernel_launches(*args, L) + 2;
  return PKS_OK;
}

pks_status pks_decode_step_timed(const pks_decode_args* args, pks_stream stream,
                                 pks_event const* events) {
  return decode_impl(args, stream, events);
}

pks_status pks_indexer_scores(const pks_decode_args* args, int32_t* scores, int64_t ld,
                              pks_stream stream) {
  pks_status st = pks::check_shapes(args);
  if (st != PKS_OK) return st;
  if ((st = pks::check_common_ptrs(args)) != PKS_OK) return st;
  if ((st = pks::check_scan_ptrs(args)) != PKS_OK) return st;
  if (ld < (int64_t)args->max_pages * args->page_size) return PKS_ERR_INVALID;
  if (args->B > 0 && !scores) return PKS_ERR_INVALID;
  if (args->B == 0) return PKS_OK;
  int32_t* err = nullptr;
  if (args->workspace) {
    const WorkspaceLayout L = pks::workspace_layout(*args);
    if (pks::check_workspace(args, L) == PKS_OK)
      err = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(args->workspace) + L.err);
  }
  return pks::from_cuda(pks::launch_indexer_scan(*args, scores, ld, nullptr, err,
                                                 reinterpret_cast<cudaStream_t>(stream)));
}

pks_status pks_sparse_attention(const pks_decode_args* args, pks_stream stream) {
  pks_status st = pks::check_shapes(args);
  if (st != PKS_OK) return st;
  if ((st = pks::check_common_ptrs(args)) != PKS_OK) return st;
  if ((st = pks::check_attn_ptrs(args)) != PKS_OK) return st;
  const WorkspaceLayout L = pks::workspace_layout(*args);
  if ((st = pks::check_workspace(args, L)) != PKS_OK) return st;
  if (args->B == 0) return PKS_OK;
  return pks::from_cuda(pks::launch_attention(*args, L, static_cast<uint8_t*>(args->workspace),
                                              /*trim=*/false,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

pks_status pks_sparse_attention_static(const pks_decode_args* args, pks_stream stream) {
  pks_status st = pks::check_shapes(args);
  if (st != PKS_OK) return st;
  if ((st = pks::check_common_ptrs(args)) != PKS_OK) return st;
  if ((st = pks::check_attn_ptrs(args)) != PKS_OK) return st;
  // reject on the host, before any CUDA call, what cannot fit even with one CTA
  if (pks::attention_static_min_bytes(*args) > pks::kAttnStaticScratchBytes)
    return PKS_ERR_TOO_LARGE;
  if (args->B == 0) return PKS_OK;
  uint8_t* scratch = nullptr;
  cudaError_t e = pks::attention_static_scratch(&scratch);
  if (e != cudaSuccess) return PKS_ERR_CUDA;
  bool too_large = false;
  e = pks::launch_attention_static(*args, scratch, reinterpret_cast<cudaStream_t>(stream),
                                   &too_large);
  if (e != cudaSuccess) return PKS_ERR_CUDA;
  return too_large ? PKS_ERR_TOO_LARGE : PKS_OK;
}

pks_status pks_decode_barrier_offset(const pks_decode_args* args, size_t* offset) {
  if (!offset) return PKS_ERR_INVALID;
  const pks_status st = pks::check_shapes(args);
  if (st != PKS_OK) return st;
  *offset = pks::workspace_layout(*args).tick_topk;
  return PKS_OK;
}

pks_status pks_decode_device_error(const pks_decode_args* args, int32_t* code,
                                   pks_stream stream) {
  if (!code) return PKS_ERR_INVALID;
  pks_status st = pks::check_shapes(args);
  if (st != PKS_OK) return st;
  const WorkspaceLayout L = pks::workspace_layout(*args);
  if ((st = pks::check_workspace(args, L)) != PKS_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t* dev = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(args->workspace) + L.err);
  int32_t host = 0;
  cudaError_t e = cudaMemcpyAsync(&host, dev, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemsetAsync(dev, 0, sizeof(int32_t), s);
  if (e != cudaSuccess) return PKS_ERR_CUDA;
  *code = host;
  return PKS_OK;
}

// ------------------------------------------------------------ residency ---

namespace {
struct ResidencyLayout {
  size_t page_slot, slot_page, last_use, lru_order, flag, slot_flag, vict, total;
};
ResidencyLayout residency_layout(int32_t num_pages, int32_t capacity) {
  ResidencyLayout R{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = pks::align_up(off + bytes);
    return o;
  };
  take(sizeof(int32_t) * 16);  // header
  R.page_slot = take(sizeof(int32_t) * (size_t)num_pages);
  R.slot_page = take(sizeof(int32_t) * (size_t)capacity);
  R.last_use = take(sizeof(int32_t) * (size_t)capacity);
  R.lru_order = take(sizeof(int32_t) * (size_t)capacity);
  R.flag = take((size_t)num_pages);
  R.slot_flag = take((size_t)capacity);
  R.vict = take(sizeof(int32_t) * (size_t)capacity);
  R.total = off;
  return R;
}
bool residency_sizes_ok(int32_t num_pages, int32_t capacity) {
  return num_pages >= 1 && capacity >= 0;
}
}  // namespace

pks_status pks_residency_state_bytes(int32_t num_pages, int32_t capacity, size_t* bytes) {
  if (!bytes || !residency_sizes_ok(num_pages, capacity)) return PKS_ERR_INVALID;
  *bytes = residency_layout(num_pages, capacity).total;
  return PKS_OK;
}

pks_status pks_residency_offsets(int32_t num_pages, int32_t capacity, size_t* page_slot,
                                 size_t* slot_page, size_t* last_use, size_t* lru_order) {
  if (!residency_sizes_ok(num_pages, capacity)) return PKS_ERR_INVALID;
  const ResidencyLayout R = residency_layout(num_pages, capacity);
  if (page_slot) *page_slot = R.page_slot;
  if (slot_page) *slot_page = R.slot_page;
  if (last_use) *last_use = R.last_use;
  if (lru_order) *lru_order = R.lru_order;
  return PKS_OK;
}

pks_status pks_residency_init(void* state, int32_t num_pages, int32_t capacity,
                              int32_t n_init, const int32_t* init_pages, pks_stream stream) {
  if (!state || !residency_sizes_ok(num_pages, capacity)) return PKS_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(state) & (pks::kAlign - 1)) != 0) return PKS_ERR_INVALID;
  if (n_init < 0 || n_init > capacity || (n_init > 0 && !init_pages)) return PKS_ERR_INVALID;
  std::vector<int32_t> pages(init_pages, init_pages + n_init);
  std::sort(pages.begin(), pages.end());
  for (int32_t i = 0; i < n_init; ++i) {
    if (pages[(size_t)i] < 0 || pages[(size_t)i] >= num_pages) return PKS_ERR_INVALID;
    if (i > 0 && pages[(size_t)i] == pages[(size_t)i - 1]) return PKS_ERR_INVALID;
  }
  const ResidencyLayout R = residency_layout(num_pages, capacity);
  std::vector<uint8_t> host(R.total, 0);
  int32_t* hdr = reinterpret_cast<int32_t*>(host.data());
  hdr[0] = num_pages;
  hdr[1] = capacity;
  hdr[2] = 0;
  hdr[3] = n_init;
  hdr[4] = 0;
  hdr[5] = pks::kResidencyMagic;
  int32_t* page_slot = reinterpret_cast<int32_t*>(host.data() + R.page_slot);
  int32_t* slot_page = reinterpret_cast<int32_t*>(host.data() + R.slot_page);
  int32_t* last_use = reinterpret_cast<int32_t*>(host.data() + R.last_use);
  int32_t* lru = reinterpret_cast<int32_t*>(host.data() + R.lru_order);
  std::fill(page_slot, page_slot + num_pages, -1);
  for (int32_t s = 0; s < capacity; ++s) {
    slot_page[s] = -1;
    last_use[s] = -1;
  }
  for (int32_t i = 0; i < n_init; ++i) {
    slot_page[i] = pages[(size_t)i];
    page_slot[pages[(size_t)i]] = i;
    last_use[i] = 0;
  }
  // (last use, slot) order: never-used empty slots first, then slots 0..n_init-1
  int32_t pos = 0;
  for (int32_t s = n_init; s < capacity; ++s) lru[pos++] = s;
  for (int32_t s = 0; s < n_init; ++s) lru[pos++] = s;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // pageable source: the call returns once the bytes are staged, so `host`
  // may go out of scope afterwards
  return pks::from_cuda(cudaMemcpyAsync(state, host.data(), R.total, cudaMemcpyHostToDevice, s));
}

pks_status pks_residency_update(void* state, int32_t num_pages, int32_t capacity, int32_t B,
                                int32_t k, int32_t page_size, int32_t max_pages,
                                const int32_t* topk_idx, const int32_t* block_table,
                                int32_t* miss_list, int32_t* n_miss, pks_stream stream) {
  if (!state || !residency_sizes_ok(num_pages, capacity)) return PKS_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(state) & (pks::kAlign - 1)) != 0) return PKS_ERR_INVALID;
  if (B < 0 || k < 1 || page_size < 1 || max_pages < 1 || !miss_list || !n_miss)
    return PKS_ERR_INVALID;
  if (B > 0 && (!topk_idx || !block_table)) return PKS_ERR_INVALID;
  const ResidencyLayout R = residency_layout(num_pages, capacity);
  return pks::from_cuda(pks::launch_residency(
      static_cast<int32_t*>(state), num_pages, capacity, B, k, page_size, max_pages, topk_idx,
      block_table, miss_list, n_miss, R.page_slot, R.slot_page, R.last_use, R.lru_order, R.flag,
      R.slot_flag, R.vict, reinterpret_cast<cudaStream_t>(stream)));
}

pks_status pks_sparse_attention_resident(const pks_decode_args* args, const void* state,
                                         int32_t capacity, const void* slot_k,
                                         const void* slot_v, pks_stream stream) {
  pks_status st = pks::check_shapes(args);
  if (st != PKS_OK) return st;
  if ((st = pks::check_common_ptrs(args)) != PKS_OK) return st;
  if ((st = pks::check_attn_ptrs(args)) != PKS_OK) return st;
  if (!state || !slot_k || !slot_v || !residency_sizes_ok(args->num_pages, capacity))
    return PKS_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(state) & (pks::kAlign - 1)) != 0) return PKS_ERR_INVALID;
  if (!pks::aligned16(slot_k) || !pks::aligned16(slot_v)) return PKS_ERR_INVALID;
  const WorkspaceLayout L = pks::workspace_layout(*args);
  if ((st = pks::check_workspace(args, L)) != PKS_OK) return st;
  if (args->B == 0) return PKS_OK;
  const ResidencyLayout R = residency_layout(args->num_pages, capacity);
  // kv_k / kv_v of the arguments are the host pools; the slots replace them
  pks_decode_args a = *args;
  a.kv_k = slot_k;
  a.kv_v = slot_v;
  pks::ResidentKv rk;
  rk.page_slot = reinterpret_cast<const int32_t*>(static_cast<const uint8_t*>(state) + R.page_slot);
  rk.capacity = capacity;
  rk.host_k = static_cast<const __nv_bfloat16*>(args->kv_k);
  rk.host_v = static_cast<const __nv_bfloat16*>(args->kv_v);
  return pks::from_cuda(pks::launch_attention(a, L, static_cast<uint8_t*>(args->workspace),
                                              /*trim=*/false,
                                              reinterpret_cast<cudaStream_t>(stream), rk));
}

pks_status pks_residency_fetch(const void* state, int32_t num_pages, int32_t capacity,
                               const int32_t* miss_list, const int32_t* n_miss,
                               const void* host_k, const void* host_v, void* slot_k,
                               void* slot_v, int64_t page_bytes, pks_stream stream) {
  if (!state || !residency_sizes_ok(num_pages, capacity)) return PKS_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(state) & (pks::kAlign - 1)) != 0) return PKS_ERR_INVALID;
  if (!miss_list || !n_miss || !host_k || !host_v || !slot_k || !slot_v) return PKS_ERR_INVALID;
  if (page_bytes < 16 || page_bytes % 16 != 0) return PKS_ERR_INVALID;
  if (!pks::aligned16(host_k) || !pks::aligned16(host_v) || !pks::aligned16(slot_k) ||
      !pks::aligned16(slot_v))
    return PKS_ERR_INVALID;
  if (capacity == 0) return PKS_OK;
  const ResidencyLayout R = residency_layout(num_pages, capacity);
  return pks::from_cuda(pks::launch_residency_fetch(
      reinterpret_cast<const int32_t*>(static_cast<const uint8_t*>(state) + R.page_slot),
      miss_list, n_miss, static_cast<const uint8_t*>(host_k), static_cast<const uint8_t*>(host_v),
      static_cast<uint8_t*>(slot_k), static_cast<uint8_t*>(slot_v), page_bytes, num_pages,
      capacity, reinterpret_cast<cudaStream_t>(stream)));
}

// ------------------------------------------------------------ sparse MLA ---

namespace {
pks_status mla_check(const pks_mla_args* a) {
  if (!a) return PKS_ERR_INVALID;
  if (a->B < 0 || a->B > pks::kMaxB || a->H < 1 || a->H > 128 || a->page_size < 1 ||
      a->max_pages < 1 || a->num_pages < 1 || a->k < 1 || a->k > pks::kMaxK ||
      a->splits < 0 || a->splits > pks::kMlaMaxSplits || a->trim < 0 || a->trim > 1 ||
      a->wait_limit < 0 || !(a->sm_scale >= 0.f))
    return PKS_ERR_INVALID;
  if (a->d_latent != pks::kMlaLatent || a->d_rope != pks::kMlaRope) return PKS_ERR_UNSUPPORTED;
  if ((int64_t)a->num_pages * a->page_size > INT32_MAX) return PKS_ERR_UNSUPPORTED;
  if ((int64_t)a->max_pages * a->page_size > pks::kMaxLen) return PKS_ERR_UNSUPPORTED;
  return PKS_OK;
}
pks_status mla_check_workspace(const pks_mla_args* a, const pks::MlaLayout& L) {
  if (!a->workspace) return PKS_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(a->workspace) & (pks::kAlign - 1)) != 0)
    return PKS_ERR_WORKSPACE;
  if (a->workspace_bytes < L.total) return PKS_ERR_WORKSPACE;
  return PKS_OK;
}
}  // namespace

pks_status pks_mla_workspace_size(const pks_mla_args* args, size_t* bytes) {
  if (!bytes) return PKS_ERR_INVALID;
  pks_status st = mla_check(args);
  if (st != PKS_OK) return st;
  *bytes = pks::mla_layout(*args).total;
  return PKS_OK;
}

pks_status pks_mla_sparse_attention(const pks_mla_args* args, pks_stream stream) {
  pks_status st = mla_check(args);
  if (st != PKS_OK) return st;
  if (args->B > 0) {
    if (!args->seq_lens || !args->block_table || !args->topk_idx || !args->q || !args->kv ||
        !args->out)
      return PKS_ERR_INVALID;
    if (!pks::aligned16(args->q) || !pks::aligned16(args->kv) || !pks::aligned16(args->out))
      return PKS_ERR_INVALID;
  }
  const pks::MlaLayout L = pks::mla_layout(*args);
  if ((st = mla_check_workspace(args, L)) != PKS_OK) return st;
  if (args->B == 0) return PKS_OK;
  return pks::from_cuda(pks::launch_mla(*args, L, reinterpret_cast<cudaStream_t>(stream)));
}

pks_status pks_mla_device_error(const pks_mla_args* args, int32_t* code, pks_stream stream) {
  if (!code) return PKS_ERR_INVALID;
  pks_status st = mla_check(args);
  if (st != PKS_OK) return st;
  const pks::MlaLayout L = pks::mla_layout(*args);
  if ((st = mla_check_workspace(args, L)) != PKS_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t* dev = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(args->workspace) + L.err);
  int32_t host = 0;
  cudaError_t e = cudaMemcpyAsync(&host, dev, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemsetAsync(dev, 0, sizeof(int32_t), s);
  if (e != cudaSuccess) return PKS_ERR_CUDA;
  *code = host;
  return PKS_OK;
}

pks_status pks_stage_copy(const pks_copy_range* ranges, int32_t n, pks_stream stream) {
  if (!ranges || n < 1 || n > PKS_STAGE_MAX_RANGES) return PKS_ERR_INVALID;
  for (int i = 0; i < n; ++i)
    if (ranges[i].bytes > 0 && (!ranges[i].dst || !ranges[i].src)) return PKS_ERR_INVALID;
  return pks::from_cuda(
      pks::launch_stage_copy(ranges, n, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
