// Exact top-k selection shared across heads, on int32 indexer scores.
//
// "Sparse Attention on GLM5.3 and HBM", DeepSeek Sparse Attention paragraph:
// the top-K tokens by indexer score are selected once per query and shared by
// all attention heads; a query that attends to fewer than K tokens stays
// dense.  Ties are broken towards the lower token index, so the selected set
// is unique: the k largest of the composite key (score, -index).
//
// No sort.  The indexer scan leaves a 2048-bin histogram of each request's
// scores (bins ordered like the scores).  k_topk_threshold runs one CTA per
// (4096-token chunk, request):
//  * every CTA finds the threshold bin T1 (the bin holding the k-th largest
//    score), writes the bits of its tokens above T1 into the request's token
//    bitmap (one warp ballot = one 32-token word, no atomics) and appends its
//    tokens in T1 to the candidate list (one atomic per CTA);
//  * the last CTA of a request to finish (atomic ticket, no CTA ever waits)
//    radix-selects, 8 bits at a time and starting after the bits all
//    candidates share, the exact threshold key among the candidates (a few
//    hundred in practice) and adds the selected candidates to the bitmap.
//    For requests up to 131072 tokens it then copies the bitmap to shared
//    memory and writes the k selected indices in ascending order with one
//    block scan; for longer requests it computes per-chunk offsets and
//    k_topk_emit writes each chunk's indices from its 128 bitmap words.
//    It leaves the histogram and counters zero for the next step.
// Dense requests (len <= k) are written directly.

#include "pks_internal.h"

namespace pks {
namespace {

constexpr int kTopkThreads = 256;
constexpr int kPerThread = kTopkChunk / kTopkThreads;
// candidates staged in shared memory for the exact select (more go through L2)
constexpr int kCandCap = 2048;
// requests up to this many tokens are emitted through the shared bitmap
constexpr int kBitmapTokens = 131072;

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
__device__ __forceinline__ int key_token(uint64_t key) {
  return (int)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFu));
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

struct TopkWs {
  int32_t* hist;       // [B][kScoreBins]   control
  int32_t* tick;       // [B]               control
  int32_t* cand_n;     // [B]               control
  int2* cand;          // [B][max_len]      (score, token) of bin-T1 tokens
  uint32_t* bits;      // [B][nchunks*128]  selected-token bitmap, 32 tokens a word
  int32_t* gt_cnt;     // [B][nchunks]      tokens above T1 per chunk
  int32_t* chunk_off;  // [B][nchunks]      output offset per chunk (long requests)
  TopkThreshold* thr;  // [B]
  int32_t* err;
};

__global__ void __launch_bounds__(kTopkThreads)
k_topk_threshold(const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ scores,
                 int64_t ld, TopkWs w, int32_t* __restrict__ topk, int k, int max_len,
                 int nchunks_max) {
  extern __shared__ __align__(16) uint8_t dsm[];
  // [kCandCap] staged candidate keys | [kBitmapTokens/32] bitmap | [nchunks] counts
  uint64_t* s_key = reinterpret_cast<uint64_t*>(dsm);
  uint32_t* s_bm = reinterpret_cast<uint32_t*>(dsm + sizeof(uint64_t) * kCandCap);
  int* s_cnt = reinterpret_cast<int*>(dsm + sizeof(uint64_t) * kCandCap + kBitmapTokens / 8);
  __shared__ int s_warp[kTopkThreads / 32];
  __shared__ int s_bins[kTopkThreads];
  __shared__ int s_T1, s_above, s_last;
  __shared__ int s_digit, s_digit_above, s_digit_count;
  __shared__ unsigned long long s_and[kTopkThreads / 32], s_or[kTopkThreads / 32];

  const int b = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
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

  // ---- chunk scores first (independent of the histogram): one L2 latency
  const int start = c * kTopkChunk, stop = min(len, start + kTopkChunk);
  const int32_t* sb = scores + (int64_t)b * ld;
  int sc[kPerThread];
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) {
    const int t = start + j * kTopkThreads + tid;
    sc[j] = t < stop ? sb[t] : 0;
  }

  // ---- threshold bin: the bin where the count from the top reaches k
  const int32_t* hb = w.hist + (int64_t)b * kScoreBins;
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
  s_bins[kTopkThreads - 1 - tid] = local;  // suffix sums = scan in reversed order
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
    if (tid == 0 && c == 0) atomicCAS(w.err, 0, kErrState);
    return;
  }

  // ---- tokens above T1 (bitmap words) and candidates (tokens in T1)
  int2* cb = w.cand + (int64_t)b * max_len;
  uint32_t* bw = w.bits + (int64_t)b * nchunks_max * (kTopkChunk / 32);
  int gt = 0, n_eq = 0;
  unsigned eqm = 0;  // bit j: this thread's token of slice j is a candidate
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) {
    const int t = start + j * kTopkThreads + tid;
    const bool valid = t < stop;
    const int bin = score_bin(sc[j]);
    // slice j of warp `warp` is the aligned 32-token word at t - lane
    const unsigned m = __ballot_sync(0xffffffffu, valid && bin > T1);
    if (lane == 0) {
      bw[(start + j * kTopkThreads + warp * 32) >> 5] = m;
      gt += __popc(m);
    }
    if (valid && bin == T1) {
      eqm |= 1u << j;
      ++n_eq;
    }
  }
  // one atomic per CTA reserves the candidates' slots
  int n_eq_total;
  int eq_base = block_exclusive_scan<kTopkThreads>(n_eq, &n_eq_total, s_warp);
  __shared__ int s_cand_base;
  if (tid == 0) s_cand_base = n_eq_total ? atomicAdd(w.cand_n + b, n_eq_total) : 0;
  __syncthreads();
  eq_base += s_cand_base;
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) {
    if (eqm & (1u << j)) {
      if (eq_base < max_len) cb[eq_base] = make_int2(sc[j], start + j * kTopkThreads + tid);
      ++eq_base;
    }
  }
  const int gt_total = block_sum<kTopkThreads>(gt, s_warp);
  if (tid == 0) w.gt_cnt[(int64_t)b * nchunks_max + c] = gt_total;

  // ---- ticket: the last chunk CTA of this request finishes the selection
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    s_last = atomicAdd(w.tick + b, 1) == nch - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  const int n = min(__ldcg(w.cand_n + b), max_len);
  int need = k - s_above;  // 1 <= need <= n when the workspace is consistent
  const bool staged = n <= kCandCap;
  uint64_t kand = ~0ull, kor = 0ull;
  for (int i = tid; i < n; i += kTopkThreads) {
    const int2 e = __ldcg(cb + i);
    const uint64_t key = order_key(e.x, e.y);
    if (staged) s_key[i] = key;
    kand &= key;
    kor |= key;
  }
  // leading bits shared by every candidate need no pass
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    kand &= __shfl_xor_sync(0xffffffffu, kand, o);
    kor |= __shfl_xor_sync(0xffffffffu, kor, o);
  }
  if (lane == 0) {
    s_and[warp] = kand;
    s_or[warp] = kor;
  }
  __syncthreads();
  kand = ~0ull;
  kor = 0ull;
#pragma unroll
  for (int i = 0; i < kTopkThreads / 32; ++i) {
    kand &= s_and[i];
    kor |= s_or[i];
  }
  const int common = n > 0 ? __clzll((long long)(kand ^ kor)) : 64;  // 64 when all equal
  int bits = (common / 8) * 8;
  uint64_t prefix = bits == 0 ? 0ull : (bits == 64 ? kand : (kand >> (64 - bits)));
  while (bits < 64) {
    const int shift = 56 - bits;
    s_bins[tid] = 0;
    if (tid == 0) {
      s_digit = 0;
      s_digit_above = 0;
      s_digit_count = 0;
    }
    __syncthreads();
    for (int i = tid; i < n; i += kTopkThreads) {
      uint64_t key;
      if (staged) {
        key = s_key[i];
      } else {
        const int2 e = __ldcg(cb + i);
        key = order_key(e.x, e.y);
      }
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
      int incl = sum;  // suffix sum over lanes
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32) incl += y;
      }
      int run = incl - sum;
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
    const bool done = s_digit_count == need;
    __syncthreads();
    if (done) break;
  }
  const uint64_t kstar = bits == 64 ? prefix : (prefix << (64 - bits));

  if (len <= kBitmapTokens) {
    // ---- ordered output through the bitmap, staged in shared memory
    const int words = (len + 31) >> 5;
    for (int i = tid; i < words; i += kTopkThreads) s_bm[i] = __ldcg(bw + i);
    __syncthreads();
    for (int i = tid; i < n; i += kTopkThreads) {
      uint64_t key;
      if (staged) {
        key = s_key[i];
      } else {
        const int2 e = __ldcg(cb + i);
        key = order_key(e.x, e.y);
      }
      const int t = key_token(key);
      if (key >= kstar && (unsigned)t < (unsigned)len) atomicOr(&s_bm[t >> 5], 1u << (t & 31));
    }
    __syncthreads();
    const int per = (words + kTopkThreads - 1) / kTopkThreads;
    const int w0 = min(words, tid * per), w1 = min(words, w0 + per);
    int cnt = 0;
    for (int i = w0; i < w1; ++i) cnt += __popc(s_bm[i]);
    int tot;
    int pos = block_exclusive_scan<kTopkThreads>(cnt, &tot, s_warp);
    for (int i = w0; i < w1; ++i) {
      uint32_t bits_w = s_bm[i];
      while (bits_w) {
        const int bit = __ffs(bits_w) - 1;
        bits_w &= bits_w - 1u;
        if (pos < k) row[pos] = i * 32 + bit;
        ++pos;
      }
    }
  } else {
    // ---- long request: per-chunk output offsets for k_topk_emit
    for (int i = tid; i < nchunks_max; i += kTopkThreads) s_cnt[i] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += kTopkThreads) {
      uint64_t key;
      if (staged) {
        key = s_key[i];
      } else {
        const int2 e = __ldcg(cb + i);
        key = order_key(e.x, e.y);
      }
      const int t = key_token(key);
      if (key >= kstar && (unsigned)t < (unsigned)len) {
        atomicAdd(&s_cnt[t / kTopkChunk], 1);
        atomicOr(bw + (t >> 5), 1u << (t & 31));
      }
    }
    __syncthreads();
    const int per = (nch + kTopkThreads - 1) / kTopkThreads;
    int mine = 0;
    for (int i = 0; i < per; ++i) {
      const int cc = tid * per + i;
      if (cc < nch) mine += s_cnt[cc] + __ldcg(w.gt_cnt + (int64_t)b * nchunks_max + cc);
    }
    int tot;
    int off = block_exclusive_scan<kTopkThreads>(mine, &tot, s_warp);
    for (int i = 0; i < per; ++i) {
      const int cc = tid * per + i;
      if (cc < nch) {
        w.chunk_off[(int64_t)b * nchunks_max + cc] = off;
        off += s_cnt[cc] + __ldcg(w.gt_cnt + (int64_t)b * nchunks_max + cc);
      }
    }
  }
  if (tid == 0) {
    TopkThreshold t;
    t.bin = T1;
    t.pad = 0;
    t.key = kstar;
    w.thr[b] = t;
    w.tick[b] = 0;
    w.cand_n[b] = 0;
  }
  // leave the histogram zero for the next step
  for (int i = tid; i < kScoreBins; i += kTopkThreads) w.hist[(int64_t)b * kScoreBins + i] = 0;
}

__global__ void __launch_bounds__(kTopkThreads)
k_topk_emit(const int32_t* __restrict__ seq_lens, const uint32_t* __restrict__ bits,
            const int32_t* __restrict__ chunk_off, int32_t* __restrict__ topk, int k,
            int max_len, int nchunks_max) {
  __shared__ int s_warp[kTopkThreads / 32];
  constexpr int kWords = kTopkChunk / 32;  // 128 words per chunk
  const int b = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
  const int len = clamp_len(seq_lens[b], max_len);
  if (len <= k || len <= kBitmapTokens) return;  // written by the threshold kernel
  const int nch = (len + kTopkChunk - 1) / kTopkChunk;
  if (c >= nch) return;
  int32_t* row = topk + (int64_t)b * k;
  const uint32_t word =
      tid < kWords ? __ldcg(bits + (int64_t)b * nchunks_max * kWords + c * kWords + tid) : 0u;
  int tot;
  int pos = chunk_off[(int64_t)b * nchunks_max + c] +
            block_exclusive_scan<kTopkThreads>(__popc(word), &tot, s_warp);
  uint32_t w = word;
  while (w) {
    const int bit = __ffs(w) - 1;
    w &= w - 1u;
    if (pos < k) row[pos] = c * kTopkChunk + tid * 32 + bit;
    ++pos;
  }
}

}  // namespace

cudaError_t launch_topk(const pks_decode_args& a, const WorkspaceLayout& L, uint8_t* ws,
                        cudaStream_t s) {
  const int max_len = a.max_pages * a.page_size;
  dim3 grid(L.nchunks, a.B);
  TopkWs w;
  w.hist = reinterpret_cast<int32_t*>(ws + L.hist);
  w.tick = reinterpret_cast<int32_t*>(ws + L.tick_topk);
  w.cand_n = reinterpret_cast<int32_t*>(ws + L.cand_n);
  w.cand = reinterpret_cast<int2*>(ws + L.cand);
  w.bits = reinterpret_cast<uint32_t*>(ws + L.bits);
  w.gt_cnt = reinterpret_cast<int32_t*>(ws + L.gt_cnt);
  w.chunk_off = reinterpret_cast<int32_t*>(ws + L.chunk_off);
  w.thr = reinterpret_cast<TopkThreshold*>(ws + L.thresh);
  w.err = reinterpret_cast<int32_t*>(ws + L.err);
  const size_t smem = sizeof(uint64_t) * kCandCap + kBitmapTokens / 8 + sizeof(int) * L.nchunks;
  static size_t configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  size_t& done = configured[dev & 63];
  if (smem > done) {
    cudaError_t e = cudaFuncSetAttribute(k_topk_threshold,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    done = smem;
  }
  k_topk_threshold<<<grid, kTopkThreads, smem, s>>>(
      a.seq_lens, reinterpret_cast<const int32_t*>(ws + L.scores), L.ld, w, a.topk_idx, a.k,
      max_len, L.nchunks);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || max_len <= kBitmapTokens) return e;
  k_topk_emit<<<grid, kTopkThreads, 0, s>>>(
      a.seq_lens, reinterpret_cast<const uint32_t*>(ws + L.bits),
      reinterpret_cast<const int32_t*>(ws + L.chunk_off), a.topk_idx, a.k, max_len, L.nchunks);
  return cudaGetLastError();
}

int topk_kernel_launches(const pks_decode_args& a) {
  return (int64_t)a.max_pages * a.page_size > kBitmapTokens ? 2 : 1;
}

}  // namespace pks
