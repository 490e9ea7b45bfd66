// Exact top-k selection shared across heads, on int32 indexer scores.
//
// "Sparse Attention on GLM5.3 and HBM", DeepSeek Sparse Attention paragraph:
// the top-K tokens by indexer score are selected once per query and shared by
// all attention heads; a query that attends to fewer than K tokens stays
// dense.  Ties are broken towards the lower token index, so the selected set
// is unique: the k largest of the composite key (score, -index).
//
// Three passes, none of which sorts:
//  1. (fused into the indexer scan) a 2048-bin histogram of the scores of
//     every request, bins ordered like the scores.
//  2. k_topk_threshold, one CTA per (4096-token chunk, request): every CTA
//     finds the threshold bin T1 (the bin holding the k-th largest score)
//     from the histogram, counts its tokens above T1 and appends its tokens in
//     T1 (the candidates) to a per-request list.  The last CTA of a request
//     to finish (atomic ticket, no waiting) radix-selects the exact threshold
//     key among the candidates, 8 bits at a time, and turns the per-chunk
//     counts into output offsets.  It then zeroes the histogram and counters.
//  3. k_topk_emit, one CTA per (chunk, request): re-reads the scores and
//     writes the selected token indices in ascending order (ballot + block
//     scan) at the chunk's offset.
// Scores of one step (4 bytes per token) stay in L2 between the passes.

#include "pks_internal.h"

namespace pks {
namespace {

constexpr int kTopkThreads = 256;

__device__ __forceinline__ int score_bin(int s) {
  if (s == 0) return kScoreBins / 2;
  const unsigned a = s > 0 ? (unsigned)s : 0u - (unsigned)s;
  const int e = 31 - __clz(a);
  const unsigned m = e >= 5 ? (a >> (e - 5)) & 31u : (a << (5 - e)) & 31u;
  const int v = e * 32 + (int)m;
  return s > 0 ? kScoreBins / 2 + 1 + v : kScoreBins / 2 - 1 - v;
}

// Larger key = earlier in the (score descending, index ascending) order.
__device__ __forceinline__ uint64_t order_key(int score, int t) {
  return ((uint64_t)((uint32_t)score ^ 0x80000000u) << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)t);
}

__device__ __forceinline__ int clamp_len(int len, int max_len) {
  return (len < 0 || len > max_len) ? 0 : len;
}

template <int NT>
__device__ __forceinline__ int block_sum(int v, int* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if (lane == 0) s_warp[warp] = v;
  __syncthreads();
  int t = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) t += s_warp[w];
  return t;
}

template <int NT>
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
  int before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    const int s = s_warp[w];
    if (w < warp) before += s;
    tot += s;
  }
  *total = tot;
  return before + x - v;
}

__global__ void __launch_bounds__(kTopkThreads)
k_topk_threshold(const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ scores,
                 int64_t ld, int32_t* __restrict__ hist, int32_t* __restrict__ tick,
                 int32_t* __restrict__ cand_n, int2* __restrict__ cand,
                 int32_t* __restrict__ gt_cnt, int32_t* __restrict__ chunk_off,
                 TopkThreshold* __restrict__ thr, int32_t* __restrict__ err, int k, int max_len,
                 int nchunks_max) {
  extern __shared__ int s_cnt[];  // [nchunks_max] selected candidates per chunk
  __shared__ int s_warp[kTopkThreads / 32];
  __shared__ int s_bins[kTopkThreads];
  __shared__ int s_T1, s_above, s_last, s_cand_base[kTopkThreads / 32];
  __shared__ int s_digit, s_digit_above, s_digit_count;

  const int b = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int len = clamp_len(seq_lens[b], max_len);
  if (len <= k) return;
  const int nch = (len + kTopkChunk - 1) / kTopkChunk;
  if (c >= nch) return;

  // ---- 1. threshold bin: the bin where the count from the top reaches k
  const int32_t* hb = hist + (int64_t)b * kScoreBins;
  constexpr int kPer = kScoreBins / kTopkThreads;
  int h[kPer];
  int local = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    h[i] = __ldcg(hb + tid * kPer + i);
    local += h[i];
  }
  if (tid == 0) {
    s_T1 = -1;
    s_above = 0;
  }
  // suffix sums: scan in reversed thread order
  s_bins[kTopkThreads - 1 - tid] = local;
  __syncthreads();
  int total;
  const int rev_before = block_exclusive_scan<kTopkThreads>(s_bins[tid], &total, s_warp);
  __syncthreads();
  s_bins[kTopkThreads - 1 - tid] = rev_before;  // tokens in bins above this thread's bins
  __syncthreads();
  {
    int run = s_bins[tid];
#pragma unroll
    for (int i = kPer - 1; i >= 0; --i) {
      if (run < k && run + h[i] >= k) {
        s_T1 = tid * kPer + i;
        s_above = run;
      }
      run += h[i];
    }
  }
  __syncthreads();
  const int T1 = s_T1;
  if (T1 < 0) {
    // fewer than k tokens counted: the workspace was not initialised
    if (tid == 0 && c == 0) atomicCAS(err, 0, kErrState);
    return;
  }

  // ---- 2. count tokens above T1, append the T1 tokens as candidates
  const int start = c * kTopkChunk, stop = min(len, start + kTopkChunk);
  const int32_t* sb = scores + (int64_t)b * ld;
  int2* cb = cand + (int64_t)b * max_len;
  int gt = 0;
  for (int base = start; base < stop; base += kTopkThreads) {
    const int t = base + tid;
    const bool valid = t < stop;
    const int s = valid ? sb[t] : 0;
    const int bin = score_bin(s);
    gt += (valid && bin > T1) ? 1 : 0;
    const bool eq = valid && bin == T1;
    const unsigned m = __ballot_sync(0xffffffffu, eq);
    if (m) {
      if (lane == 0) s_cand_base[warp] = atomicAdd(cand_n + b, __popc(m));
      __syncwarp();
      const int slot = s_cand_base[warp] + __popc(m & ((1u << lane) - 1u));
      if (eq && slot < max_len) cb[slot] = make_int2(s, t);
      __syncwarp();
    }
  }
  const int gt_total = block_sum<kTopkThreads>(gt, s_warp);
  if (tid == 0) gt_cnt[(int64_t)b * nchunks_max + c] = gt_total;

  // ---- ticket: the last chunk CTA of this request refines
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    s_last = atomicAdd(tick + b, 1) == nch - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  const int n = min(__ldcg(cand_n + b), max_len);
  int need = k - s_above;  // 1 <= need <= n when the workspace is consistent
  uint64_t prefix = 0;
  int bits = 0;
  for (;;) {
    const int shift = 56 - bits;
    s_bins[tid] = 0;
    if (tid == 0) {
      s_digit = 0;
      s_digit_above = 0;
      s_digit_count = 0;
    }
    __syncthreads();
    for (int i = tid; i < n; i += kTopkThreads) {
      const int2 e = __ldcg(cb + i);
      const uint64_t key = order_key(e.x, e.y);
      if (bits == 0 || (key >> (64 - bits)) == prefix)
        atomicAdd(&s_bins[(int)((key >> shift) & 255u)], 1);
    }
    __syncthreads();
    if (warp == 0) {
      // lane owns digits [8*lane, 8*lane+8); find the digit where the count
      // from the top reaches `need`
      int d[8], sum = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        d[i] = s_bins[lane * 8 + i];
        sum += d[i];
      }
      // suffix sum over lanes: tokens with a larger digit than this lane's
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32) incl += y;
      }
      const int above = incl - sum;
      int run = above;
#pragma unroll
      for (int i = 7; i >= 0; --i) {
        if (run < need && run + d[i] >= need) {
          s_digit = lane * 8 + i;
          s_digit_above = run;
          s_digit_count = d[i];
        }
        run += d[i];
      }
    }
    __syncthreads();
    need -= s_digit_above;
    prefix = (prefix << 8) | (uint64_t)s_digit;
    bits += 8;
    const bool done = s_digit_count == need || bits == 64;
    __syncthreads();
    if (done) break;
  }
  const uint64_t kstar = bits == 64 ? prefix : (prefix << (64 - bits));

  // ---- per-chunk selected counts -> output offsets
  for (int i = tid; i < nchunks_max; i += kTopkThreads) s_cnt[i] = 0;
  __syncthreads();
  for (int i = tid; i < n; i += kTopkThreads) {
    const int2 e = __ldcg(cb + i);
    if (order_key(e.x, e.y) >= kstar && (unsigned)e.y < (unsigned)len)
      atomicAdd(&s_cnt[e.y / kTopkChunk], 1);
  }
  __syncthreads();
  const int per = (nch + kTopkThreads - 1) / kTopkThreads;
  int mine = 0;
  for (int i = 0; i < per; ++i) {
    const int cc = tid * per + i;
    if (cc < nch) mine += s_cnt[cc] + __ldcg(gt_cnt + (int64_t)b * nchunks_max + cc);
  }
  int tot;
  int off = block_exclusive_scan<kTopkThreads>(mine, &tot, s_warp);
  for (int i = 0; i < per; ++i) {
    const int cc = tid * per + i;
    if (cc < nch) {
      chunk_off[(int64_t)b * nchunks_max + cc] = off;
      off += s_cnt[cc] + __ldcg(gt_cnt + (int64_t)b * nchunks_max + cc);
    }
  }
  if (tid == 0) {
    TopkThreshold t;
    t.bin = T1;
    t.pad = 0;
    t.key = kstar;
    thr[b] = t;
    tick[b] = 0;
    cand_n[b] = 0;
  }
  // leave the histogram zero for the next step
  for (int i = tid; i < kScoreBins; i += kTopkThreads) hist[(int64_t)b * kScoreBins + i] = 0;
}

__global__ void __launch_bounds__(kTopkThreads)
k_topk_emit(const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ scores, int64_t ld,
            const int32_t* __restrict__ chunk_off, const TopkThreshold* __restrict__ thr,
            int32_t* __restrict__ topk, int k, int max_len, int nchunks_max) {
  __shared__ int s_warp[kTopkThreads / 32];
  const int b = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
  const int lane = tid & 31;
  const int len = clamp_len(seq_lens[b], max_len);
  int32_t* row = topk + (int64_t)b * k;
  if (len <= k) {
    // dense: every token, then -1 padding
    const int nch = max(1, (len + kTopkChunk - 1) / kTopkChunk);
    if (c >= nch) return;
    const int start = c * kTopkChunk, stop = min(len, start + kTopkChunk);
    for (int t = start + tid; t < stop; t += kTopkThreads) row[t] = t;
    if (c == 0)
      for (int j = len + tid; j < k; j += kTopkThreads) row[j] = -1;
    return;
  }
  const int nch = (len + kTopkChunk - 1) / kTopkChunk;
  if (c >= nch) return;
  const TopkThreshold th = thr[b];
  int off = chunk_off[(int64_t)b * nchunks_max + c];
  const int start = c * kTopkChunk, stop = min(len, start + kTopkChunk);
  const int32_t* sb = scores + (int64_t)b * ld;
  for (int base = start; base < stop; base += kTopkThreads) {
    const int t = base + tid;
    bool sel = false;
    if (t < stop) {
      const int s = sb[t];
      const int bin = score_bin(s);
      sel = bin > th.bin || (bin == th.bin && order_key(s, t) >= th.key);
    }
    const unsigned m = __ballot_sync(0xffffffffu, sel);
    int tile_total;
    const int wbase = block_exclusive_scan<kTopkThreads>(lane == 0 ? __popc(m) : 0, &tile_total,
                                                         s_warp);
    const int warp_off = __shfl_sync(0xffffffffu, wbase, 0);
    const int pos = off + warp_off + __popc(m & ((1u << lane) - 1u));
    if (sel && pos < k) row[pos] = t;
    off += tile_total;
  }
}

}  // namespace

cudaError_t launch_topk(const pks_decode_args& a, const WorkspaceLayout& L, uint8_t* ws,
                        cudaStream_t s) {
  const int max_len = a.max_pages * a.page_size;
  dim3 grid(L.nchunks, a.B);
  const size_t smem = sizeof(int) * (size_t)L.nchunks;
  k_topk_threshold<<<grid, kTopkThreads, smem, s>>>(
      a.seq_lens, reinterpret_cast<const int32_t*>(ws + L.scores), L.ld,
      reinterpret_cast<int32_t*>(ws + L.hist), reinterpret_cast<int32_t*>(ws + L.tick_topk),
      reinterpret_cast<int32_t*>(ws + L.cand_n), reinterpret_cast<int2*>(ws + L.cand),
      reinterpret_cast<int32_t*>(ws + L.gt_cnt), reinterpret_cast<int32_t*>(ws + L.chunk_off),
      reinterpret_cast<TopkThreshold*>(ws + L.thresh), reinterpret_cast<int32_t*>(ws + L.err),
      a.k, max_len, L.nchunks);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  k_topk_emit<<<grid, kTopkThreads, 0, s>>>(
      a.seq_lens, reinterpret_cast<const int32_t*>(ws + L.scores), L.ld,
      reinterpret_cast<const int32_t*>(ws + L.chunk_off),
      reinterpret_cast<const TopkThreshold*>(ws + L.thresh), a.topk_idx, a.k, max_len,
      L.nchunks);
  return cudaGetLastError();
}

}  // namespace pks
