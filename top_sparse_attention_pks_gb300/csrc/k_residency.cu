// HBM residency table over KV pages: miss list and LRU update.
//
// "Sparse Attention on GLM5.3 and HBM", HiSparse paragraph: KV lives in an
// LRU cache in HBM backed by host DRAM; tokens chosen by the top-k selection
// that are not in HBM are loaded (a miss), and entries leave HBM by least
// recent use.  Here the cached unit is a physical KV page.  A step:
//   A      = distinct pages holding a selected token (aliased prefix pages once)
//   misses = A minus the resident set, ascending page id   -> miss list
//   hits   : last use = step
//   victims: slots not holding a page of A, least recently used first (ties by
//            slot); the i-th miss takes the i-th victim (last use = step);
//            misses beyond the victims are reported but not admitted.
//
// Instead of sorting slots by (last use, slot) every step, the table keeps
// them in that order (lru_order).  A step only appends: untouched slots keep
// their relative order, and every slot touched in the step (hits and
// admissions) takes the newest last-use value, tied among themselves, so they
// go to the back in slot order.  Both updates are order-preserving stream
// compactions.
//
// k_residency_mark (one thread per selected position) marks pages of A in a
// byte array; k_residency_update (one CTA of 1024 threads) does the rest with
// block-wide scans over tiles read with 16-byte loads, and leaves its scratch
// arrays zero again.

#include "pks_internal.h"

namespace pks {
namespace {

constexpr int kMarkThreads = 256;
constexpr int kUpdThreads = 1024;

__device__ __forceinline__ void flag_error(int32_t* err, int code) { atomicCAS(err, 0, code); }

__global__ void __launch_bounds__(kMarkThreads)
k_residency_mark(const int32_t* __restrict__ topk, const int32_t* __restrict__ block_table,
                 uint8_t* __restrict__ flag, int32_t* __restrict__ err, int B, int k,
                 int page_size, int max_pages, int num_pages) {
  const int64_t i = (int64_t)blockIdx.x * kMarkThreads + threadIdx.x;
  if (i >= (int64_t)B * k) return;
  const int t = topk[i];
  if (t < 0) return;
  const int b = (int)(i / k);
  const int lp = t / page_size;
  if (lp >= max_pages) {
    flag_error(err, kErrToken);
    return;
  }
  const int page = block_table[(int64_t)b * max_pages + lp];
  if ((unsigned)page >= (unsigned)num_pages) {
    flag_error(err, kErrPage);
    return;
  }
  flag[page] = 1;
}

__device__ __forceinline__ int block_exclusive_scan(int v, int* total, int* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    s_warp[lane] = w;  // inclusive
  }
  __syncthreads();
  *total = s_warp[31];
  return (warp > 0 ? s_warp[warp - 1] : 0) + x - v;
}

// Tiles of the three passes: a thread owns kPageTile consecutive pages,
// kSlotTile consecutive LRU positions or slots, read with 16-byte loads and
// gathered all at once, so that each tile costs about one round trip and one
// block scan.
constexpr int kPageTile = 32;
constexpr int kSlotTile = 16;

__global__ void __launch_bounds__(kUpdThreads)
k_residency_update(int32_t* __restrict__ hdr, int32_t* __restrict__ page_slot,
                   int32_t* __restrict__ slot_page, int32_t* __restrict__ last_use,
                   int32_t* __restrict__ lru_order, uint8_t* __restrict__ flag,
                   uint8_t* __restrict__ slot_flag, int32_t* __restrict__ vict,
                   int32_t* __restrict__ miss_list, int32_t* __restrict__ n_miss_out,
                   int num_pages, int capacity) {
  __shared__ int s_warp[32];
  __shared__ int s_step, s_new_resident, s_ok;
  const int tid = threadIdx.x;
  if (tid == 0) {
    s_step = hdr[2] + 1;
    s_new_resident = 0;
    // a state buffer that pks_residency_init did not fill for these sizes is
    // left untouched
    s_ok = hdr[5] == kResidencyMagic && hdr[0] == num_pages && hdr[1] == capacity;
    if (!s_ok) {
      flag_error(hdr + 4, kErrState);
      *n_miss_out = 0;
    }
  }
  __syncthreads();
  if (!s_ok) return;
  const int step = s_step;

  // ---- misses (ascending pages) and hits; every page flag is cleared
  int n_miss = 0;
  for (int p0 = 0; p0 < num_pages; p0 += kPageTile * kUpdThreads) {
    const int pb = p0 + tid * kPageTile;
    uint32_t fl = 0;  // bit j: page pb + j is in A
    int ps[kPageTile];
    if (pb + kPageTile <= num_pages) {
      const uint4* f4 = reinterpret_cast<const uint4*>(flag + pb);
      const uint4 fa = f4[0], fb = f4[1];
      const uint32_t fw[8] = {fa.x, fa.y, fa.z, fa.w, fb.x, fb.y, fb.z, fb.w};
#pragma unroll
      for (int j = 0; j < kPageTile; ++j) fl |= (uint32_t)(((fw[j >> 2] >> (8 * (j & 3))) & 0xffu) != 0) << j;
      const int4* s4 = reinterpret_cast<const int4*>(page_slot + pb);
#pragma unroll
      for (int q = 0; q < kPageTile / 4; ++q) {
        const int4 v = s4[q];
        ps[4 * q] = v.x;
        ps[4 * q + 1] = v.y;
        ps[4 * q + 2] = v.z;
        ps[4 * q + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < kPageTile; ++j) {
        const bool in = pb + j < num_pages;
        fl |= (uint32_t)(in && flag[pb + j] != 0) << j;
        ps[j] = in ? page_slot[pb + j] : -1;
      }
    }
    uint32_t missm = 0;
#pragma unroll
    for (int j = 0; j < kPageTile; ++j) missm |= (uint32_t)(((fl >> j) & 1u) && ps[j] < 0) << j;
    int tile_miss;
    int base = n_miss + block_exclusive_scan(__popc(missm), &tile_miss, s_warp);
#pragma unroll
    for (int j = 0; j < kPageTile; ++j) {
      if (!((fl >> j) & 1u)) continue;
      const int sl = ps[j];
      if (sl < 0) {
        miss_list[base++] = pb + j;
      } else if (sl < capacity) {
        slot_flag[sl] = 1;
        last_use[sl] = step;
      }
    }
    if (fl) {
      if (pb + kPageTile <= num_pages) {
        uint4* f4 = reinterpret_cast<uint4*>(flag + pb);
        f4[0] = make_uint4(0, 0, 0, 0);
        f4[1] = make_uint4(0, 0, 0, 0);
      } else {
        for (int j = 0; j < kPageTile && pb + j < num_pages; ++j) flag[pb + j] = 0;
      }
    }
    n_miss += tile_miss;
  }
  __syncthreads();  // slot flags of the hits are visible to every thread

  // ---- victims: slots not hit this step, in LRU order
  int n_v = 0;
  for (int i0 = 0; i0 < capacity; i0 += kSlotTile * kUpdThreads) {
    const int ib = i0 + tid * kSlotTile;
    int sl[kSlotTile];
    if (ib + kSlotTile <= capacity) {
      const int4* l4 = reinterpret_cast<const int4*>(lru_order + ib);
#pragma unroll
      for (int q = 0; q < kSlotTile / 4; ++q) {
        const int4 v = l4[q];
        sl[4 * q] = v.x;
        sl[4 * q + 1] = v.y;
        sl[4 * q + 2] = v.z;
        sl[4 * q + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < kSlotTile; ++j) sl[j] = ib + j < capacity ? lru_order[ib + j] : -1;
    }
    uint32_t vm = 0;  // bit j: slot sl[j] is a victim
#pragma unroll
    for (int j = 0; j < kSlotTile; ++j)
      vm |= (uint32_t)((unsigned)sl[j] < (unsigned)capacity && !slot_flag[(unsigned)sl[j] < (unsigned)capacity ? sl[j] : 0]) << j;
    int tile_v;
    int base = n_v + block_exclusive_scan(__popc(vm), &tile_v, s_warp);
#pragma unroll
    for (int j = 0; j < kSlotTile; ++j)
      if ((vm >> j) & 1u) vict[base++] = sl[j];
    n_v += tile_v;
  }
  __syncthreads();

  // ---- admission: i-th miss -> i-th victim
  const int n_admit = min(n_miss, n_v);
  int filled = 0;
  for (int i = tid; i < n_admit; i += kUpdThreads) {
    const int s = vict[i];
    const int old = slot_page[s];
    if ((unsigned)old < (unsigned)num_pages) page_slot[old] = -1;
    else ++filled;
    const int p = miss_list[i];
    slot_page[s] = p;
    page_slot[p] = s;
    last_use[s] = step;
    slot_flag[s] = 1;
  }
  if (filled) atomicAdd(&s_new_resident, filled);
  __syncthreads();

  // ---- new LRU order: untouched slots in their old order, then touched
  // slots (last use = step) by slot number; every slot flag is cleared
  const int n_keep = n_v - n_admit;
  for (int i = tid; i < n_keep; i += kUpdThreads) lru_order[i] = vict[n_admit + i];
  int n_touched = 0;
  for (int s0 = 0; s0 < capacity; s0 += kSlotTile * kUpdThreads) {
    const int sb = s0 + tid * kSlotTile;
    uint32_t tm = 0;  // bit j: slot sb + j was touched
    if (sb + kSlotTile <= capacity) {
      const uint4 f = *reinterpret_cast<const uint4*>(slot_flag + sb);
      const uint32_t fw[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
      for (int j = 0; j < kSlotTile; ++j) tm |= (uint32_t)(((fw[j >> 2] >> (8 * (j & 3))) & 0xffu) != 0) << j;
    } else {
#pragma unroll
      for (int j = 0; j < kSlotTile; ++j) tm |= (uint32_t)(sb + j < capacity && slot_flag[sb + j] != 0) << j;
    }
    int tile_t;
    int base = n_keep + n_touched + block_exclusive_scan(__popc(tm), &tile_t, s_warp);
#pragma unroll
    for (int j = 0; j < kSlotTile; ++j)
      if ((tm >> j) & 1u) lru_order[base++] = sb + j;
    if (tm) {
      if (sb + kSlotTile <= capacity) {
        *reinterpret_cast<uint4*>(slot_flag + sb) = make_uint4(0, 0, 0, 0);
      } else {
        for (int j = 0; j < kSlotTile && sb + j < capacity; ++j) slot_flag[sb + j] = 0;
      }
    }
    n_touched += tile_t;
  }
  if (tid == 0) {
    hdr[2] = step;
    hdr[3] += s_new_resident;
    *n_miss_out = n_miss;
  }
}

}  // namespace

cudaError_t launch_residency(int32_t* state, int32_t num_pages, int32_t capacity, int32_t B,
                             int32_t k, int32_t page_size, int32_t max_pages,
                             const int32_t* topk_idx, const int32_t* block_table,
                             int32_t* miss_list, int32_t* n_miss, size_t off_page_slot,
                             size_t off_slot_page, size_t off_last_use, size_t off_lru,
                             size_t off_flag, size_t off_slot_flag, size_t off_vict,
                             cudaStream_t s) {
  uint8_t* base = reinterpret_cast<uint8_t*>(state);
  uint8_t* flag = base + off_flag;
  const int64_t n = (int64_t)B * k;
  if (n > 0) {
    const int64_t grid = (n + kMarkThreads - 1) / kMarkThreads;
    k_residency_mark<<<(unsigned)grid, kMarkThreads, 0, s>>>(topk_idx, block_table, flag,
                                                             state + 4, B, k, page_size,
                                                             max_pages, num_pages);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  k_residency_update<<<1, kUpdThreads, 0, s>>>(
      state, reinterpret_cast<int32_t*>(base + off_page_slot),
      reinterpret_cast<int32_t*>(base + off_slot_page), reinterpret_cast<int32_t*>(base + off_last_use),
      reinterpret_cast<int32_t*>(base + off_lru), flag, base + off_slot_flag,
      reinterpret_cast<int32_t*>(base + off_vict), miss_list, n_miss, num_pages, capacity);
  return cudaGetLastError();
}

}  // namespace pks
