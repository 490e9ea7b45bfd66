// Staging copies of a step's inputs and outputs: up to eight byte ranges in
// one launch, moved by SM loads and stores.
//
// Not part of the sparse-attention method: on a Grace-Blackwell node the SMs
// read and write page-locked host memory over the CPU-GPU link, and for the
// few hundred kilobytes of a decode step's queries, block table, output and
// top-k list they do so faster than the copy engines, with one launch instead
// of one copy per buffer.  Each range moves as 16-byte vectors when its two
// pointers and its size are multiples of 16, else byte by byte.  Every thread
// takes up to four units of the concatenated ranges per pass, all loads
// before the stores, so that many link round trips are in flight at once.

#include "pks_internal.h"

namespace pks {
namespace {

constexpr int kStageThreads = 256;
constexpr int kStageUnroll = 4;

struct StageRanges {
  void* dst[kStageMaxRanges];
  const void* src[kStageMaxRanges];
  int64_t units[kStageMaxRanges];  // 16-byte vectors or bytes
  int64_t first[kStageMaxRanges];  // first unit of the range in the concatenation
  int wide[kStageMaxRanges];       // 1: 16-byte units
  int n;
  int64_t total;
};

__device__ __forceinline__ int range_of(const StageRanges& r, int64_t u) {
  int i = 0;
  while (i + 1 < r.n && r.first[i + 1] <= u) ++i;
  return i;
}

__global__ void __launch_bounds__(kStageThreads)
k_stage_copy(const StageRanges r) {
  // launched with programmatic serialization: the next kernel may launch now
  // and wait for this one; this one waits for the kernel before it
  pdl_launch_dependents();
  pdl_wait();
  const int64_t stride = (int64_t)gridDim.x * kStageThreads;
  for (int64_t u0 = (int64_t)blockIdx.x * kStageThreads + threadIdx.x; u0 < r.total;
       u0 += stride * kStageUnroll) {
    int4 v[kStageUnroll];
    int which[kStageUnroll];
#pragma unroll
    for (int j = 0; j < kStageUnroll; ++j) {
      const int64_t u = u0 + (int64_t)j * stride;
      which[j] = -1;
      if (u < r.total) {
        const int i = range_of(r, u);
        const int64_t e = u - r.first[i];
        which[j] = i;
        if (r.wide[i])
          v[j] = __ldcs(reinterpret_cast<const int4*>(r.src[i]) + e);
        else
          v[j].x = reinterpret_cast<const uint8_t*>(r.src[i])[e];
      }
    }
#pragma unroll
    for (int j = 0; j < kStageUnroll; ++j) {
      const int i = which[j];
      if (i < 0) continue;
      const int64_t e = u0 + (int64_t)j * stride - r.first[i];
      if (r.wide[i])
        __stcs(reinterpret_cast<int4*>(r.dst[i]) + e, v[j]);
      else
        reinterpret_cast<uint8_t*>(r.dst[i])[e] = (uint8_t)v[j].x;
    }
  }
}

}  // namespace

cudaError_t launch_stage_copy(const pks_copy_range* ranges, int n, cudaStream_t s) {
  StageRanges r{};
  r.n = n;
  int64_t total = 0;
  for (int i = 0; i < n; ++i) {
    const bool wide = ((reinterpret_cast<uintptr_t>(ranges[i].dst) |
                        reinterpret_cast<uintptr_t>(ranges[i].src) | ranges[i].bytes) &
                       15) == 0;
    r.dst[i] = ranges[i].dst;
    r.src[i] = ranges[i].src;
    r.wide[i] = wide ? 1 : 0;
    r.units[i] = wide ? (int64_t)(ranges[i].bytes / 16) : (int64_t)ranges[i].bytes;
    r.first[i] = total;
    total += r.units[i];
  }
  r.total = total;
  if (total == 0) return cudaSuccess;
  const int64_t per_cta = (int64_t)kStageThreads * kStageUnroll;
  int64_t grid = (total + per_cta - 1) / per_cta;
  const int64_t cap = (int64_t)device_sm_count() * 8;
  if (grid > cap) grid = cap;
  return launch_ex(k_stage_copy, dim3((unsigned)grid), dim3(kStageThreads), 0, s, /*pdl=*/true,
                   /*coop=*/false, r);
}

}  // namespace pks
