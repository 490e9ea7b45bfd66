// Internal declarations shared by the host layer and the kernel files of libpks.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pks.h"

#include <utility>

namespace pks {

// ---- programmatic dependent launch (PDL) ----
// The kernels of a step after the first are launched with programmatic
// stream serialisation: their CTAs may be scheduled while the previous
// kernel drains, run what does not depend on it, and wait in pdl_wait()
// until it has completed and its writes are visible.  A kernel calls
// pdl_launch_dependents() once the next kernel's CTAs may take SM slots.
// Both are no-ops for a kernel launched without the attribute.
#ifdef __CUDACC__
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}
#endif

// cudaLaunchKernelEx with optional PDL and cooperative attributes.
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                      cudaStream_t s, bool pdl, bool coop, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (coop) {
    attr[n].id = cudaLaunchAttributeCooperative;
    attr[n].val.cooperative = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ---- indexer score histogram (fused into the scan, consumed by top-k) ----
// 2048 bins over int32 scores, order preserving: 0 -> bin 1024; |s| > 0 is
// binned by its leading-one position e (0..31) and the next 5 bits m, giving
// 32 bins per power of two (about 2% wide); positives above 1024, negatives
// mirrored below.
constexpr int kScoreBins = 2048;
// Tokens per top-k chunk (one CTA of the top-k kernels).
constexpr int kTopkChunk = 4096;
// Most chunks per request the single-launch top-k handles.
constexpr int kTopkCoopMaxChunks = 1024;
// Attention: tokens per pipeline tile; largest persistent grid the workspace
// holds partials for.
constexpr int kAttnTile = 16;
constexpr int kAttnGridMax = 1024;
// With an automatic grid, every attention CTA takes at least this many
// selected positions (two tiles).
constexpr int kAttnMinPositions = 2 * kAttnTile;

// KV heads handled by one attention CTA (one warp each): the largest of
// 8, 4, 2, 1 that divides Hkv.
inline int attn_heads_per_cta(int hkv) {
  for (int hg = 8; hg > 1; hg >>= 1)
    if (hkv % hg == 0) return hg;
  return 1;
}

// Device error word causes (see pks_decode_device_error).
constexpr int kErrPage = 1;
constexpr int kErrToken = 2;
constexpr int kErrLen = 3;
constexpr int kErrState = 4;
constexpr int kErrTimeout = 5;
// header word 5 of a residency state filled by pks_residency_init
constexpr int32_t kResidencyMagic = 0x504b5352;

struct TopkThreshold {
  int32_t bin;        // coarse threshold bin T1
  int32_t pad;
  uint64_t key;       // exact threshold on (score, ~token) among bin-T1 tokens
};

// Byte offsets of the workspace regions for one set of shapes.  Every region
// starts on a 256-byte boundary.  The control block (error word, histograms,
// tickets, counters) must be zero between steps; everything else is scratch.
struct WorkspaceLayout {
  size_t ctrl, err, hist, tick_topk, depart_topk, cand_n, ctrl_end;
  size_t scores, cand, bits, gt_cnt, chunk_cnt, chunk_off, thresh, attn_prefix, part_ml, part_o;
  size_t total;
  int64_t ld;          // score row stride: max_pages * page_size rounded up to kTopkChunk
  int32_t nchunks;       // top-k chunks per request
  int32_t attn_grid_max; // attention CTAs the partial slots are sized for
};

WorkspaceLayout workspace_layout(const pks_decode_args& a);

// Query tokens per request (n_queries 0 means one).  Top-k, attention and
// merge run over B * Nq virtual requests, virtual request v = b * Nq + q
// using request b's length and block table row.
inline int query_count(const pks_decode_args& a) { return a.n_queries > 1 ? a.n_queries : 1; }

// ---- kernel launchers (each returns cudaGetLastError() after launch) ----
cudaError_t launch_indexer_scan(const pks_decode_args& a, int32_t* scores, int64_t ld,
                                int32_t* hist, int32_t* err, cudaStream_t s);
cudaError_t launch_topk(const pks_decode_args& a, const WorkspaceLayout& L, uint8_t* ws,
                        cudaStream_t s);
// Top-k runs as one cooperative launch when all (chunk, request) CTAs fit on
// the device at once; otherwise as the two-kernel fallback (threshold, plus
// emit for contexts longer than the shared-memory bitmap).
bool topk_single_launch(const pks_decode_args& a, const WorkspaceLayout& L);
int topk_kernel_launches(const pks_decode_args& a, const WorkspaceLayout& L);
// trim: the top-k list holds its selected entries first (the step's own
// output), so only min(k, len_b) positions per request are visited.
// K/V through a residency table: kv_k / kv_v of the arguments are then the
// slot pools [capacity, P, Hkv, D], resident pages are read from their slot,
// other pages from the host pool (device-accessible host memory).
struct ResidentKv {
  const int32_t* page_slot = nullptr;  // nullptr: plain pool
  int capacity = 0;
  const __nv_bfloat16* host_k = nullptr;
  const __nv_bfloat16* host_v = nullptr;
};
cudaError_t launch_attention(const pks_decode_args& a, const WorkspaceLayout& L, uint8_t* ws,
                             bool trim, cudaStream_t s, const ResidentKv& rk = ResidentKv{});
// Copy the admitted misses of the last residency step (miss_list[0..*n_miss)
// with a slot in page_slot) from the host pools into the slot pools.
cudaError_t launch_residency_fetch(const int32_t* page_slot, const int32_t* miss_list,
                                   const int32_t* n_miss, const uint8_t* host_k,
                                   const uint8_t* host_v, uint8_t* slot_k, uint8_t* slot_v,
                                   int64_t page_bytes, int num_pages, int capacity,
                                   cudaStream_t s);
// Staging copy of up to kStageMaxRanges byte ranges in one launch (k_stage.cu);
// the ranges are validated by the caller.
constexpr int kStageMaxRanges = PKS_STAGE_MAX_RANGES;
cudaError_t launch_stage_copy(const pks_copy_range* ranges, int n, cudaStream_t s);
// ---- sparse MLA in MQA mode (tcgen05 kernel in k_mla.cu)
constexpr int kMlaLatent = 512;  // d: latent width, the value
constexpr int kMlaRope = 64;     // r: RoPE part of the key
constexpr int kMlaMaxSplits = 64;
// Most 64-token tiles one MLA CTA takes (its rows are resolved up front):
// the split count is raised until ceil(ceil(k / 64) / splits) fits.
constexpr int kMlaMaxCtaTiles = 32;
struct MlaLayout {
  int splits;
  size_t err, part_ml, part_o, total;
};
int mla_splits(const pks_mla_args& a);
MlaLayout mla_layout(const pks_mla_args& a);
cudaError_t launch_mla(const pks_mla_args& a, const MlaLayout& L, cudaStream_t s);
cudaError_t launch_residency(int32_t* state, int32_t num_pages, int32_t capacity, int32_t B,
                             int32_t k, int32_t page_size, int32_t max_pages,
                             const int32_t* topk_idx, const int32_t* block_table,
                             int32_t* miss_list, int32_t* n_miss, size_t off_page_slot,
                             size_t off_slot_page, size_t off_last_use, size_t off_lru,
                             size_t off_flag, size_t off_slot_flag, size_t off_vict,
                             cudaStream_t s);

// Allocation-free attention (pks_sparse_attention_static): bytes of the
// file-scope device scratch array, the least any call with these shapes
// needs (one attention CTA; host only), the array's address on the current
// device (looked up once per device), and the launcher, which sets
// *too_large instead of launching when the shapes need more than the array.
constexpr size_t kAttnStaticScratchBytes = (size_t)8 << 20;
size_t attention_static_min_bytes(const pks_decode_args& a);
cudaError_t attention_static_scratch(uint8_t** ptr);
cudaError_t launch_attention_static(const pks_decode_args& a, uint8_t* scratch, cudaStream_t s,
                                    bool* too_large);

// Number of SMs of the current device (cached per device).
int device_sm_count();

}  // namespace pks
