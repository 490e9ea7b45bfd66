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
// k_residency_mark (one thread per selected position, across the GPU) marks
// the pages of A in a byte array and gives every hit its new last use and
// slot flag (idempotent writes); k_residency_update (one CTA of 1024 threads)
// does the ordered part — miss list, victims, admissions, the new LRU order —
// as coalesced order-preserving compactions, and leaves its scratch arrays
// zero again.

#include "pks_internal.h"

namespace pks {
namespace {

constexpr int kMarkThreads = 256;
constexpr int kUpdThreads = 1024;

__device__ __forceinline__ void flag_error(int32_t* err, int code) { atomicCAS(err, 0, code); }

__global__ void __launch_bounds__(kMarkThreads)
k_residency_mark(const int32_t* __restrict__ topk, const int32_t* __restrict__ block_table,
                 int32_t* __restrict__ hdr, const int32_t* __restrict__ page_slot,
                 uint8_t* __restrict__ flag, uint8_t* __restrict__ slot_flag,
                 int32_t* __restrict__ last_use, int B, int k, int page_size, int max_pages,
                 int num_pages, int capacity) {
  const int64_t i = (int64_t)blockIdx.x * kMarkThreads + threadIdx.x;
  if (i >= (int64_t)B * k) return;
  // a state buffer that pks_residency_init did not fill for these sizes is
  // left untouched (the update kernel reports it)
  if (hdr[5] != kResidencyMagic || hdr[0] != num_pages || hdr[1] != capacity) return;
  const int t = topk[i];
  if (t < 0) return;
  const int b = (int)(i / k);
  const int lp = t / page_size;
  if (lp >= max_pages) {
    flag_error(hdr + 4, kErrToken);
    return;
  }
  const int page = block_table[(int64_t)b * max_pages + lp];
  if ((unsigned)page >= (unsigned)num_pages) {
    flag_error(hdr + 4, kErrPage);
    return;
  }
  flag[page] = 1;
  // a hit: the slot's last use becomes this step (the same values from every
  // thread that selected a token of the page)
  const int sl = page_slot[page];
  if ((unsigned)sl < (unsigned)capacity) {
    slot_flag[sl] = 1;
    last_use[sl] = hdr[2] + 1;
  }
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

// Order-preserving compaction of n items in CTA-wide rounds of 32 per thread:
// item (round r, thread t) is index base + r * 1024 + t, so every warp load
// and store is coalesced.  keep(i) says whether item i is kept; emit(i, pos)
// writes it at position pos of the output.  Warp ballots give the counts of
// each (round, warp), one block scan over those 1024 counts gives every
// warp's output offset.  Returns the number kept.
template <typename Keep, typename Emit>
__device__ __forceinline__ int compact(int n, int* s_cnt, int* s_warp, Keep keep, Emit emit) {
  constexpr int kRounds = 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int kept = 0;
  for (int base = 0; base < n; base += kRounds * kUpdThreads) {
    uint32_t mine = 0;  // bit r: this thread's item of round r is kept
    // keep() is evaluated on a clamped index so that every round's loads are
    // unconditional and go out together
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
      const int idx = base + r * kUpdThreads + tid;
      const bool k = keep(idx < n ? idx : n - 1);
      mine |= (uint32_t)(idx < n && k) << r;
    }
    // counts of (round, warp) in round-major order: entry r * 32 + warp
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
      const uint32_t m = __ballot_sync(0xffffffffu, (mine >> r) & 1u);
      if (lane == 0) s_cnt[r * 32 + warp] = __popc(m);
    }
    __syncthreads();
    int total;
    const int v = s_cnt[tid];  // entry tid = (round tid / 32, warp tid % 32)
    const int off = block_exclusive_scan(v, &total, s_warp);
    s_cnt[tid] = off;
    __syncthreads();
    const uint32_t lt = (1u << lane) - 1u;
#pragma unroll 8
    for (int r = 0; r < kRounds; ++r) {
      const uint32_t m = __ballot_sync(0xffffffffu, (mine >> r) & 1u);
      if ((mine >> r) & 1u)
        emit(base + r * kUpdThreads + tid, kept + s_cnt[r * 32 + warp] + __popc(m & lt));
    }
    kept += total;
    __syncthreads();  // s_cnt is reused by the next tile
  }
  return kept;
}

__global__ void __launch_bounds__(kUpdThreads)
k_residency_update(int32_t* __restrict__ hdr, int32_t* __restrict__ page_slot,
                   int32_t* __restrict__ slot_page, int32_t* __restrict__ last_use,
                   int32_t* __restrict__ lru_order, uint8_t* __restrict__ flag,
                   uint8_t* __restrict__ slot_flag, int32_t* __restrict__ vict,
                   int32_t* __restrict__ miss_list, int32_t* __restrict__ n_miss_out,
                   int num_pages, int capacity) {
  __shared__ int s_warp[32];
  __shared__ int s_cnt[kUpdThreads];
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

  // ---- misses: pages of A without a slot, ascending (the mark kernel has
  // already given the hits their new last use and slot flag)
  const int n_miss = compact(
      num_pages, s_cnt, s_warp, [&](int p) { return (flag[p] != 0) & (page_slot[p] < 0); },
      [&](int p, int pos) { miss_list[pos] = p; });
  // every page flag is cleared for the next step
  for (int i = tid * 16; i < num_pages; i += kUpdThreads * 16) {
    if (i + 16 <= num_pages) *reinterpret_cast<uint4*>(flag + i) = make_uint4(0, 0, 0, 0);
    else for (int j = i; j < num_pages; ++j) flag[j] = 0;
  }

  // ---- victims: slots not hit this step, in LRU order
  const int n_v = compact(
      capacity, s_cnt, s_warp,
      [&](int i) {
        const int sl = lru_order[i];
        const bool in = (unsigned)sl < (unsigned)capacity;
        return in & (slot_flag[in ? sl : 0] == 0);
      },
      [&](int i, int pos) { vict[pos] = lru_order[i]; });
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
  compact(
      capacity, s_cnt, s_warp, [&](int sl) { return slot_flag[sl] != 0; },
      [&](int sl, int pos) { lru_order[n_keep + pos] = sl; });
  __syncthreads();
  for (int i = tid * 16; i < capacity; i += kUpdThreads * 16) {
    if (i + 16 <= capacity) *reinterpret_cast<uint4*>(slot_flag + i) = make_uint4(0, 0, 0, 0);
    else for (int j = i; j < capacity; ++j) slot_flag[j] = 0;
  }
  if (tid == 0) {
    hdr[2] = step;
    hdr[3] += s_new_resident;
    *n_miss_out = n_miss;
  }
}

// Miss fetch ([SA] HiSparse paragraph: a top-k miss is loaded into HBM).
// One CTA per admitted miss page at a time (grid-stride over the miss list):
// the page's K and V bytes are read from the host pools (device-accessible
// host memory, over the CPU-GPU link) with 16-byte loads, eight in flight per
// thread, and written to the page's slot in the HBM slot pools.
constexpr int kFetchThreads = 256;

__global__ void __launch_bounds__(kFetchThreads)
k_residency_fetch(const int32_t* __restrict__ page_slot, const int32_t* __restrict__ miss_list,
                  const int32_t* __restrict__ n_miss, const int4* __restrict__ host_k,
                  const int4* __restrict__ host_v, int4* __restrict__ slot_k,
                  int4* __restrict__ slot_v, int64_t page_vec, int num_pages, int capacity) {
  const int n = min(*n_miss, num_pages);
  for (int i = blockIdx.x; i < n; i += gridDim.x) {
    const int p = miss_list[i];
    if ((unsigned)p >= (unsigned)num_pages) continue;
    const int sl = page_slot[p];
    if ((unsigned)sl >= (unsigned)capacity) continue;  // reported, not admitted
    const int4* sk = host_k + (int64_t)p * page_vec;
    const int4* sv = host_v + (int64_t)p * page_vec;
    int4* dk = slot_k + (int64_t)sl * page_vec;
    int4* dv = slot_v + (int64_t)sl * page_vec;
    constexpr int U = 4;
    for (int64_t j0 = threadIdx.x; j0 < page_vec; j0 += (int64_t)kFetchThreads * U) {
      int4 a[U], b[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t j = j0 + (int64_t)u * kFetchThreads;
        if (j < page_vec) {
          a[u] = __ldcs(sk + j);
          b[u] = __ldcs(sv + j);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t j = j0 + (int64_t)u * kFetchThreads;
        if (j < page_vec) {
          dk[j] = a[u];
          dv[j] = b[u];
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_residency_fetch(const int32_t* page_slot, const int32_t* miss_list,
                                   const int32_t* n_miss, const uint8_t* host_k,
                                   const uint8_t* host_v, uint8_t* slot_k, uint8_t* slot_v,
                                   int64_t page_bytes, int num_pages, int capacity,
                                   cudaStream_t s) {
  const int grid = device_sm_count() * 4;
  k_residency_fetch<<<grid, kFetchThreads, 0, s>>>(
      page_slot, miss_list, n_miss, reinterpret_cast<const int4*>(host_k),
      reinterpret_cast<const int4*>(host_v), reinterpret_cast<int4*>(slot_k),
      reinterpret_cast<int4*>(slot_v), page_bytes / 16, num_pages, capacity);
  return cudaGetLastError();
}

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
    k_residency_mark<<<(unsigned)grid, kMarkThreads, 0, s>>>(
        topk_idx, block_table, state, reinterpret_cast<const int32_t*>(base + off_page_slot), flag,
        base + off_slot_flag, reinterpret_cast<int32_t*>(base + off_last_use), B, k, page_size,
        max_pages, num_pages, capacity);
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
