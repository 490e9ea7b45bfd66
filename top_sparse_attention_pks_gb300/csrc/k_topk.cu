// Exact top-k selection shared across heads, on int32 indexer scores.
//
// "Sparse Attention on GLM5.3 and HBM", DeepSeek Sparse Attention paragraph:
// the top-K tokens by indexer score are selected once per query and shared by
// all attention heads; a query that attends to fewer than K tokens stays
// dense.  Ties are broken towards the lower token index, so the selected set
// is unique: the k largest of the composite key (score, -index).
//
// No sort.  The indexer scan leaves a 2048-bin histogram of each request's
// scores (bins ordered like the scores).  One CTA per (4096-token chunk,
// request) runs the chunk phase: it finds the threshold bin T1 (the bin
// holding the k-th largest score), counts its tokens above T1 and appends its
// tokens in T1 to the request's candidate list (one atomic per CTA).  The
// exact threshold key among the candidates (a few hundred in practice) is
// then radix-selected 8 bits at a time, starting after the bits all
// candidates share.
//
// k_topk_select (one cooperative launch, used whenever the grid fits on the
// GPU at once): the CTAs of a request meet at a counter barrier after the
// chunk phase; each then selects the threshold itself and writes its own
// chunk's indices at the chunk's output offset, so no CTA runs a serial tail.
//
// k_topk_threshold (+ k_topk_emit), the fallback for larger grids: no CTA
// waits; the last CTA of a request to finish (atomic ticket) selects the
// threshold, merges the selected candidates into the request's token bitmap
// and writes the indices, or, beyond 131072 tokens, per-chunk offsets that
// k_topk_emit turns into indices.
//
// Dense requests (len <= k) are written directly.  Both paths leave the
// histogram and counters zero for the next step.

#include "pks_internal.h"

namespace pks {
namespace {

constexpr int kTopkThreads = 256;
constexpr int kPerThread = kTopkChunk / kTopkThreads;
// candidates staged in shared memory for the exact select (more go through L2)
constexpr int kCandCap = 2048;
// requests up to this many tokens are emitted through the shared bitmap
constexpr int kBitmapTokens = 131072;
// polls of a request barrier before it gives up (about 0.4 s), unless the
// caller sets wait_limit
constexpr int kBarrierSpins = 1 << 22;

__device__ __forceinline__ int score_bin(int s) {
  if (s == 0) return kScoreBins / 2;
  const unsigned a = s > 0 ? (unsigned)s : 0u - (unsigned)s;
  const int e = 31 - __clz(a);
  const unsigned m = e >= 5 ? (a >> (e - 5)) & 31u : (a << (5 - e)) & 31u;
  const int v = e * 32 + (int)m;
  return s > 0 ? kScoreBins / 2 + 1 + v : kScoreBins / 2 - 1 - v;
}

// Scores from real-valued head weights are order-preserving int32 keys of the
// fp32 score (the scan bins them the same way).
__device__ __forceinline__ int key_bin(int key) {
  // the fp32 score's magnitude bits a: exact zero alone in the middle bin;
  // |score| < 1 one bin per octave down to 2^-32; from 1 up 32 bins per
  // octave (exponent and top five mantissa bits), the top bin from 2^30 up
  const uint32_t a = (uint32_t)(key >= 0 ? key : key ^ 0x7fffffff) & 0x7fffffffu;
  if (a == 0) return kScoreBins / 2;
  const int e = (int)(a >> 23) - 127;
  int v;
  if (e < 0) v = e < -32 ? 0 : 32 + e;
  else v = 32 + (e > 29 ? 29 * 32 + 31 : e * 32 + (int)((a >> 18) & 31u));
  return key >= 0 ? kScoreBins / 2 + 1 + v : kScoreBins / 2 - 1 - v;
}
__device__ __forceinline__ int score_bin_m(int s, bool fkey) {
  return fkey ? key_bin(s) : score_bin(s);
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
  int32_t* tick;       // [B]               control: ticket / barrier arrivals
  int32_t* depart;     // [B]               control: barrier departures
  int32_t* cand_n;     // [B]               control
  int2* cand;          // [B][max_len]      (score, token) of bin-T1 tokens
  uint32_t* bits;      // [B][nchunks*128]  selected-token bitmap, 32 tokens a word
  int32_t* gt_cnt;     // [B][nchunks]      tokens above T1 per chunk
  int32_t* chunk_off;  // [B][nchunks]      output offset per chunk (long requests)
  TopkThreshold* thr;  // [B]
  int32_t* err;
  int fkey;            // scores are keys of fp32 scores (real-valued head weights)
};

// Shared memory of the chunk phase and the exact select.
template <int NT>
struct TopkSmemT {
  int warp[NT / 32];
  int bins[NT > 256 ? NT : 256];  // threshold-bin scan (NT), radix digits (256)
  int T1, above, flag;
  int digit, digit_above, digit_count;
  int cand_base;
  int tied;  // select_threshold took the one-score shortcut
  unsigned long long kand[NT / 32], kor[NT / 32];
};
using TopkSmem = TopkSmemT<kTopkThreads>;

// Chunk phase, run by every CTA of a request: load the chunk's scores, find
// the threshold bin T1 from the request's histogram, count the chunk's tokens
// above T1 and append its bin-T1 tokens to the candidate list.  Returns false
// (and flags kErrState once) when the histogram counts fewer than k tokens.
// With `bitmap` it also writes the chunk's above-T1 bitmap words.
__device__ __forceinline__ bool chunk_phase(const int32_t* __restrict__ sb, const int32_t* hb,
                                            int start, int stop, int k, int2* cb, int cand_cap,
                                            int32_t* cand_n,
                                            uint32_t* bw, bool bitmap, int32_t* err, bool report,
                                            int (&sc)[kPerThread], int& T1, int& above,
                                            int& gt_total, TopkSmem& sm, bool fkey) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // chunk scores first (independent of the histogram): one L2 latency
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) {
    const int t = start + j * kTopkThreads + tid;
    sc[j] = t < stop ? sb[t] : 0;
  }
  // threshold bin: the bin where the count from the top reaches k
  constexpr int kPer = kScoreBins / kTopkThreads;
  int h[kPer];
  int local = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    h[i] = __ldcg(hb + tid * kPer + i);
    local += h[i];
  }
  if (tid == 0) {
    sm.T1 = -1;
    sm.above = 0;
  }
  sm.bins[kTopkThreads - 1 - tid] = local;  // suffix sums = scan in reversed order
  __syncthreads();
  int total;
  const int rev_before = block_exclusive_scan<kTopkThreads>(sm.bins[tid], &total, sm.warp);
  __syncthreads();
  sm.bins[kTopkThreads - 1 - tid] = rev_before;  // tokens in bins above this thread's bins
  __syncthreads();
  {
    int run = sm.bins[tid];
#pragma unroll
    for (int i = kPer - 1; i >= 0; --i) {
      if (run < k && run + h[i] >= k) {
        sm.T1 = tid * kPer + i;
        sm.above = run;
      }
      run += h[i];
    }
  }
  __syncthreads();
  T1 = sm.T1;
  above = sm.above;
  if (T1 < 0) {
    // fewer than k tokens counted: the workspace was not initialised
    if (tid == 0 && report) atomicCAS(err, 0, kErrState);
    return false;
  }
  int gt = 0, n_eq = 0;
  unsigned eqm = 0;  // bit j: this thread's token of slice j is a candidate
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) {
    const int t = start + j * kTopkThreads + tid;
    const bool valid = t < stop;
    const int bin = score_bin_m(sc[j], fkey);
    // slice j of warp `warp` is the aligned 32-token word at t - lane
    const unsigned m = __ballot_sync(0xffffffffu, valid && bin > T1);
    if (lane == 0) {
      if (bitmap) bw[(start + j * kTopkThreads + warp * 32) >> 5] = m;
      gt += __popc(m);
    }
    if (valid && bin == T1) {
      eqm |= 1u << j;
      ++n_eq;
    }
  }
  // one atomic per CTA reserves the candidates' slots
  int n_eq_total;
  int eq_base = block_exclusive_scan<kTopkThreads>(n_eq, &n_eq_total, sm.warp);
  if (tid == 0) sm.cand_base = n_eq_total ? atomicAdd(cand_n, n_eq_total) : 0;
  __syncthreads();
  eq_base += sm.cand_base;
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) {
    if (eqm & (1u << j)) {
      if (eq_base < cand_cap) cb[eq_base] = make_int2(sc[j], start + j * kTopkThreads + tid);
      ++eq_base;
    }
  }
  gt_total = block_sum<kTopkThreads>(gt, sm.warp);
  return true;
}

// Arrival at a request barrier, by one thread after the CTA's writes are
// ordered by __syncthreads.
__device__ __forceinline__ void request_arrive(int32_t* arrive) {
  __threadfence();
  atomicAdd(arrive, 1);
}

// Bounded wait until `count` CTAs of a request have arrived (one thread).
// Every arrival is a fence and an atomic add (a release), so the acquire load
// that sees the full count orders this thread's later reads after all the
// arrivers' writes; the CTA's other threads follow it through __syncthreads.
__device__ __forceinline__ bool request_wait(int32_t* arrive, int count, int spins) {
  for (int it = 0; it < spins; ++it) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];\n" : "=r"(v) : "l"(arrive) : "memory");
    if (v >= count) return true;
    if (it >= 32) __nanosleep(64);
  }
  return false;
}

// Dense request (len <= k): every token, then -1 padding.
__device__ __forceinline__ void write_dense(int32_t* row, int len, int k, int c) {
  const int start = c * kTopkChunk, stop = min(len, start + kTopkChunk);
  for (int t = start + threadIdx.x; t < stop; t += kTopkThreads) row[t] = t;
  if (c == 0)
    for (int j = len + threadIdx.x; j < k; j += kTopkThreads) row[j] = -1;
}

// Single-launch selection for grids that fit on the GPU at once (launched
// cooperatively, so all CTAs of a request are resident together).  One CTA
// per (4096-token chunk, request); thread i owns the 16 consecutive tokens
// 16i..16i+15 of the chunk, read with four 16-byte loads (score rows are
// padded to whole chunks).
//  1. Chunk phase: threshold bin T1 from the histogram and the score range
//     [lo, hi] of that bin; per-thread masks of the tokens above hi and in
//     [lo, hi]; the chunk's T1 tokens go to the chunk's own region of the
//     candidate buffer and its two counts to chunk_cnt (no atomics).
//  2. Counter barrier of the request's CTAs.
//  3. Every CTA reads all chunks' counts together with the first candidates
//     of every chunk (one round trip), selects the same exact threshold key,
//     and writes its own chunk's selected tokens in ascending order at the
//     chunk's output offset: tokens above T1 in earlier chunks plus selected
//     candidates of earlier chunks.
// CTA 0 clears the histogram once every CTA has read it; the last CTA to
// leave resets the request's barrier counters.
constexpr int kTokPerThread = kTopkChunk / kTopkThreads;  // 16
constexpr int kSpecSlots = 2 * kTopkThreads;              // candidates read with the counts

// Score range [lo, hi] of a non-empty histogram bin (the inverse of
// score_bin on the scores that reach the bin).
__device__ __forceinline__ void bin_range(int bin, int& lo, int& hi, bool fkey) {
  if (fkey) {  // the keys of the fp32 scores that key_bin puts in `bin`
    if (bin == kScoreBins / 2) {  // exact zero (-0 is stored as +0)
      lo = hi = 0;
      return;
    }
    const bool pos = bin > kScoreBins / 2;
    const int v = pos ? bin - (kScoreBins / 2 + 1) : (kScoreBins / 2 - 1) - bin;
    uint32_t alo, ahi;
    if (v < 32) {  // one octave of |score| < 1 (v = 0: everything below 2^-31)
      alo = v == 0 ? 1u : (uint32_t)(v - 32 + 127) << 23;
      ahi = ((uint32_t)(v - 32 + 128) << 23) - 1u;
    } else {
      const int u = v - 32;
      alo = ((uint32_t)((u >> 5) + 127) << 23) | ((uint32_t)(u & 31) << 18);
      ahi = u == 29 * 32 + 31 ? 0x7fffffffu : alo | 0x3ffffu;
    }
    if (pos) {
      lo = (int)alo;
      hi = (int)ahi;
    } else {  // key = ~magnitude bits for negative scores: larger magnitude, smaller key
      lo = (int)(0xffffffffu - ahi);
      hi = (int)(0xffffffffu - alo);
    }
    return;
  }
  if (bin == kScoreBins / 2) {
    lo = hi = 0;
    return;
  }
  const bool pos = bin > kScoreBins / 2;
  const int v = pos ? bin - (kScoreBins / 2 + 1) : (kScoreBins / 2 - 1) - bin;
  const int e = v >> 5, m = v & 31;
  int64_t alo, ahi;
  if (e >= 5) {
    alo = (int64_t)(32 + m) << (e - 5);
    ahi = ((int64_t)(33 + m) << (e - 5)) - 1;
  } else {
    alo = (32 + m) >> (5 - e);
    ahi = alo;
  }
  if (pos) {
    lo = (int)alo;
    hi = (int)(ahi > INT32_MAX ? (int64_t)INT32_MAX : ahi);
  } else {
    lo = (int)(-ahi < (int64_t)INT32_MIN ? (int64_t)INT32_MIN : -ahi);
    hi = (int)(-alo);
  }
}

// Exact threshold key among the n candidates: the need-th largest
// (score, ~token) key, radix-selected 8 bits at a time after the leading bits
// that every candidate shares.  Block-wide (NT threads); every thread returns
// the key.  `ordered`: key_at(0..n-1) lists the candidates in ascending token
// order, so when they all share one score the need-th largest key is simply
// the need-th candidate (many exact ties, e.g. at score 0).
template <int NT, typename KeyAt>
__device__ __forceinline__ uint64_t select_threshold(int n, int need, KeyAt key_at,
                                                     TopkSmemT<NT>& sm, bool ordered = false) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint64_t kand = ~0ull, kor = 0ull;
  for (int i = tid; i < n; i += NT) {
    const uint64_t key = key_at(i);
    kand &= key;
    kor |= key;
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    kand &= __shfl_xor_sync(0xffffffffu, kand, o);
    kor |= __shfl_xor_sync(0xffffffffu, kor, o);
  }
  if (lane == 0) {
    sm.kand[warp] = kand;
    sm.kor[warp] = kor;
  }
  __syncthreads();
  kand = ~0ull;
  kor = 0ull;
#pragma unroll
  for (int i = 0; i < NT / 32; ++i) {
    kand &= sm.kand[i];
    kor |= sm.kor[i];
  }
  const int common = n > 0 ? __clzll((long long)(kand ^ kor)) : 64;  // 64 when all equal
  const bool tied = ordered && common >= 32 && need >= 1 && need <= n;
  if (tid == 0) sm.tied = tied ? 1 : 0;  // read by the caller after its next barrier
  if (tied) return key_at(need - 1);
  int bits = (common / 8) * 8;
  uint64_t prefix = bits == 0 ? 0ull : (bits == 64 ? kand : (kand >> (64 - bits)));
  while (bits < 64) {
    const int shift = 56 - bits;
    if (tid < 256) sm.bins[tid] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += NT) {
      const uint64_t key = key_at(i);
      if (bits == 0 || (key >> (64 - bits)) == prefix)
        atomicAdd(&sm.bins[(int)((key >> shift) & 255u)], 1);
    }
    __syncthreads();
    if (warp == 0) {
      // lane owns digits [8*lane, 8*lane+8); find the digit where the count
      // from the top reaches `need`
      int d[8], sum = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        d[i] = sm.bins[lane * 8 + i];
        sum += d[i];
      }
      int incl = sum;  // suffix sum over lanes
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32) incl += y;
      }
      int run = incl - sum;
      int digit = 0, above = 0, count = 0;
      bool hit = false;
#pragma unroll
      for (int i = 7; i >= 0; --i) {
        if (run < need && run + d[i] >= need) {
          digit = lane * 8 + i;
          above = run;
          count = d[i];
          hit = true;
        }
        run += d[i];
      }
      const unsigned who = __ballot_sync(0xffffffffu, hit);
      if (who == 0u) {
        if (lane == 0) {  // inconsistent counts: settle on the lowest digit
          sm.digit = 0;
          sm.digit_above = 0;
          sm.digit_count = 0;
        }
      } else if (lane == __ffs(who) - 1) {
        sm.digit = digit;
        sm.digit_above = above;
        sm.digit_count = count;
      }
    }
    __syncthreads();
    need -= sm.digit_above;
    prefix = (prefix << 8) | (uint64_t)sm.digit;
    bits += 8;
    const bool done = sm.digit_count == need;
    __syncthreads();
    if (done) break;
  }
  return bits == 64 ? prefix : (prefix << (64 - bits));
}

// four CTAs an SM (64 registers): 608 resident CTAs on 152 SMs
__global__ void __launch_bounds__(kTopkThreads, 4)
k_topk_select(const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ scores,
              int64_t ld, TopkWs w, int2* __restrict__ chunk_cnt, int32_t* __restrict__ topk,
              int k, int max_len, int nchunks_max, int nq, int spins) {
  __shared__ uint64_t s_key[kCandCap];
  __shared__ int s_eqoff[kTopkCoopMaxChunks + 1];  // candidates before each chunk
  __shared__ int s_before, s_lo, s_hi;
  __shared__ TopkSmem sm;
  const int b = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
  const int start = c * kTopkChunk;
  const int len = clamp_len(seq_lens[b / nq], max_len);  // b: virtual request
  pdl_wait();  // scores and histogram come from the scan

  // all loads of the chunk phase at once: this thread's 16 scores (rows
  // padded to whole chunks, so always in bounds) and 8 histogram bins
  int4 v[4];
  {
    const int4* sp = reinterpret_cast<const int4*>(scores + (int64_t)b * ld + start) + 4 * tid;
#pragma unroll
    for (int r = 0; r < 4; ++r) v[r] = __ldcg(sp + r);
  }
  int32_t* hb = w.hist + (int64_t)b * kScoreBins;
  constexpr int kPer = kScoreBins / kTopkThreads;  // 8 bins a thread
  int h[kPer];
  {
    const int4 h0 = __ldcg(reinterpret_cast<const int4*>(hb) + 2 * tid);
    const int4 h1 = __ldcg(reinterpret_cast<const int4*>(hb) + 2 * tid + 1);
    h[0] = h0.x; h[1] = h0.y; h[2] = h0.z; h[3] = h0.w;
    h[4] = h1.x; h[5] = h1.y; h[6] = h1.z; h[7] = h1.w;
  }
  int32_t* row = topk + (int64_t)b * k;
  if (len <= k) {
    const int nch = max(1, (len + kTopkChunk - 1) / kTopkChunk);
    if (c < nch) write_dense(row, len, k, c);
    return;
  }
  const int nch = (len + kTopkChunk - 1) / kTopkChunk;
  if (c >= nch) return;
  const int stop = min(len, start + kTopkChunk);

  // ---- threshold bin: the bin where the count from the top reaches k
  int local = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) local += h[i];
  if (tid == 0) sm.T1 = -1;
  sm.bins[kTopkThreads - 1 - tid] = local;  // suffix sums = scan in reversed order
  __syncthreads();
  int total;
  const int rev_before = block_exclusive_scan<kTopkThreads>(sm.bins[tid], &total, sm.warp);
  __syncthreads();
  sm.bins[kTopkThreads - 1 - tid] = rev_before;  // tokens in bins above this thread's bins
  __syncthreads();
  {
    int run = sm.bins[tid];
#pragma unroll
    for (int i = kPer - 1; i >= 0; --i) {
      if (run < k && run + h[i] >= k) {
        sm.T1 = tid * kPer + i;
        sm.above = run;
        int lo, hi;
        bin_range(tid * kPer + i, lo, hi, w.fkey != 0);
        s_lo = lo;
        s_hi = hi;
      }
      run += h[i];
    }
  }
  __syncthreads();
  const int T1 = sm.T1, above = sm.above;
  if (T1 < 0) {
    // fewer than k tokens counted: the workspace was not initialised (every
    // CTA of the request reads the same histogram, so all return here)
    if (tid == 0 && c == 0) atomicCAS(w.err, 0, kErrState);
    return;
  }
  const int lo = s_lo, hi = s_hi;

  // ---- masks of this thread's tokens above T1 (gtm) and in T1 (eqm); bit j
  // is token start + 16 * tid + j
  unsigned gtm = 0, eqm = 0;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int sv[4] = {v[r].x, v[r].y, v[r].z, v[r].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int bit = 4 * r + e;
      const bool valid = start + kTokPerThread * tid + bit < stop;
      gtm |= (unsigned)(valid && sv[e] > hi) << bit;
      eqm |= (unsigned)(valid && sv[e] >= lo && sv[e] <= hi) << bit;
    }
  }
  // one scan of both counts: above-T1 in the high half, candidates in the low
  int packed_total;
  const int packed_before = block_exclusive_scan<kTopkThreads>(
      (__popc(gtm) << 16) | __popc(eqm), &packed_total, sm.warp);
  const int eq_before = packed_before & 0xffff;
  int2* cregion = w.cand + ((int64_t)b * nchunks_max + c) * kTopkChunk;
  if (eqm) {
    int pos = eq_before;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int sv[4] = {v[r].x, v[r].y, v[r].z, v[r].w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if ((eqm >> (4 * r + e)) & 1u)
          cregion[pos++] = make_int2(sv[e], start + kTokPerThread * tid + 4 * r + e);
    }
  }
  if (tid == 0)
    chunk_cnt[(int64_t)b * nchunks_max + c] = make_int2(packed_total >> 16, packed_total & 0xffff);

  // ---- barrier of the request's CTAs (a request of one chunk is one CTA:
  // its own writes are visible to it after __syncthreads)
  __syncthreads();
  if (nch > 1) {
    if (tid == 0) request_arrive(w.tick + b);
    if (tid == 0) sm.flag = request_wait(w.tick + b, nch, spins);
    __syncthreads();
    if (!sm.flag) {
      if (tid == 0) atomicCAS(w.err, 0, kErrTimeout);
      return;
    }
  }
  // every CTA of the request is resident: the attention grid may now take
  // SM slots without keeping a CTA of this grid from its barrier
  pdl_launch_dependents();
  // every CTA has read the histogram: clear it for the next step
  if (c == 0)
    for (int i = tid; i < kScoreBins; i += kTopkThreads) hb[i] = 0;

  // ---- per-chunk counts, read together with the first `win` candidates of
  // every chunk (slots tid and tid + kTopkThreads)
  const int2* cbase = w.cand + (int64_t)b * nchunks_max * kTopkChunk;
  const int win = kSpecSlots / nch;  // 0 when there are more chunks than slots
  int2 spec[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int slot = tid + u * kTopkThreads;
    spec[u] = make_int2(0, -1);
    if (win > 0 && slot / win < nch)
      spec[u] = __ldcg(cbase + (int64_t)(slot / win) * kTopkChunk + slot % win);
  }
  {
    // nch <= kTopkCoopMaxChunks = 4 * kTopkThreads: up to 4 chunks a thread,
    // their candidate counts parked in s_eqoff across the scan
    const int per = (nch + kTopkThreads - 1) / kTopkThreads;
    int eq_sum = 0, gt_before = 0;
    for (int i = 0; i < per; ++i) {
      const int cc = tid * per + i;
      if (cc < nch) {
        const int2 cnt = __ldcg(chunk_cnt + (int64_t)b * nchunks_max + cc);
        s_eqoff[cc] = cnt.y;
        eq_sum += cnt.y;
        if (cc < c) gt_before += cnt.x;
      }
    }
    int n_total;
    int off = block_exclusive_scan<kTopkThreads>(eq_sum, &n_total, sm.warp);
    for (int i = 0; i < per; ++i) {
      const int cc = tid * per + i;
      if (cc < nch) {
        const int cnt = s_eqoff[cc];
        s_eqoff[cc] = off;
        off += cnt;
      }
    }
    if (tid == 0) s_eqoff[nch] = n_total;
    gt_before = block_sum<kTopkThreads>(gt_before, sm.warp);
    if (tid == 0) s_before = gt_before;
    __syncthreads();
  }
  const int n = s_eqoff[nch];
  // candidate i of the request, in chunk order, from L2
  auto cand_at = [&](int i) -> int2 {
    int l = 0, h2 = nch - 1;  // last chunk with s_eqoff <= i
    while (l < h2) {
      const int mid = (l + h2 + 1) >> 1;
      if (s_eqoff[mid] <= i) l = mid; else h2 = mid - 1;
    }
    return __ldcg(cbase + (int64_t)l * kTopkChunk + (i - s_eqoff[l]));
  };
  const bool staged = n <= kCandCap;
  if (staged) {
    // the speculatively read candidates, then the rest of any chunk with more
    // than `win` of them
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int slot = tid + u * kTopkThreads;
      if (win > 0 && slot / win < nch) {
        const int ch = slot / win, jj = slot % win;
        if (jj < s_eqoff[ch + 1] - s_eqoff[ch]) s_key[s_eqoff[ch] + jj] = order_key(spec[u].x, spec[u].y);
      }
    }
    for (int i = tid; i < n; i += kTopkThreads) {
      int l = 0, h2 = nch - 1;
      while (l < h2) {
        const int mid = (l + h2 + 1) >> 1;
        if (s_eqoff[mid] <= i) l = mid; else h2 = mid - 1;
      }
      if (i - s_eqoff[l] >= win) {
        const int2 e = __ldcg(cbase + (int64_t)l * kTopkChunk + (i - s_eqoff[l]));
        s_key[i] = order_key(e.x, e.y);
      }
    }
    __syncthreads();
  }
  auto key_at = [&](int i) -> uint64_t {
    if (staged) return s_key[i];
    const int2 e = cand_at(i);
    return order_key(e.x, e.y);
  };
  // candidates are in token order (chunk regions in chunk order)
  const int need = k - above;
  const uint64_t kstar = select_threshold(n, need, key_at, sm, /*ordered=*/true);
  __syncthreads();
  // one score among all candidates: the selected ones are the first `need`
  // in token order, so positions decide without reading the keys again
  const bool tied = sm.tied != 0;

  // ---- output offset: above-T1 tokens and selected candidates of earlier chunks
  int before = 0;
  if (!tied)
    for (int i = tid; i < s_eqoff[c]; i += kTopkThreads) before += key_at(i) >= kstar;
  before = s_before + (tied ? min(s_eqoff[c], need) : block_sum<kTopkThreads>(before, sm.warp));

  // ---- this chunk's selected tokens, ascending: this thread's candidates sit
  // in the request's list in token order from its chunk's offset plus its
  // scan position
  unsigned selm = gtm;
  if (eqm) {
    int i = s_eqoff[c] + eq_before;
#pragma unroll
    for (int bit = 0; bit < kTokPerThread; ++bit)
      if ((eqm >> bit) & 1u) {
        if (tied ? i < need : key_at(i) >= kstar) selm |= 1u << bit;
        ++i;
      }
  }
  int sel_total;
  int pos = before + block_exclusive_scan<kTopkThreads>(__popc(selm), &sel_total, sm.warp);
  while (selm) {
    const int bit = __ffs(selm) - 1;
    selm &= selm - 1u;
    if (pos < k) row[pos] = start + kTokPerThread * tid + bit;
    ++pos;
  }

  // the last CTA to leave resets the request's barrier counters
  __syncthreads();
  if (tid == 0) {
    // no fence: the departures only order the reset below after every CTA's
    // last read of the arrival counter, which was an acquire load that this
    // CTA's atomic cannot pass; the outputs are published by the kernel's end
    if (nch > 1 && atomicAdd(w.depart + b, 1) == nch - 1) {
      w.tick[b] = 0;
      w.depart[b] = 0;
    }
  }
}

// Two-launch fallback for grids too large to be resident at once.  One CTA
// per (chunk, request) runs the chunk phase and writes above-T1 bitmap words;
// the last CTA of a request to finish (atomic ticket, no CTA ever waits)
// selects the exact threshold, adds the selected candidates to the bitmap and
// either emits the k indices itself through a shared-memory copy of the
// bitmap (requests up to 131072 tokens) or computes per-chunk offsets for
// k_topk_emit.
__global__ void __launch_bounds__(kTopkThreads)
k_topk_threshold(const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ scores,
                 int64_t ld, TopkWs w, int32_t* __restrict__ topk, int k, int max_len,
                 int nchunks_max, int nq) {
  extern __shared__ __align__(16) uint8_t dsm[];
  // [kCandCap] staged candidate keys | [kBitmapTokens/32] bitmap | [nchunks] counts
  uint64_t* s_key = reinterpret_cast<uint64_t*>(dsm);
  uint32_t* s_bm = reinterpret_cast<uint32_t*>(dsm + sizeof(uint64_t) * kCandCap);
  int* s_cnt = reinterpret_cast<int*>(dsm + sizeof(uint64_t) * kCandCap + kBitmapTokens / 8);
  __shared__ TopkSmem sm;
  __shared__ int s_last;

  const int b = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
  const int len = clamp_len(seq_lens[b / nq], max_len);  // b: virtual request
  pdl_wait();  // scores and histogram come from the scan
  pdl_launch_dependents();
  int32_t* row = topk + (int64_t)b * k;
  if (len <= k) {
    const int nch = max(1, (len + kTopkChunk - 1) / kTopkChunk);
    if (c < nch) write_dense(row, len, k, c);
    return;
  }
  const int nch = (len + kTopkChunk - 1) / kTopkChunk;
  if (c >= nch) return;
  const int start = c * kTopkChunk, stop = min(len, start + kTopkChunk);
  int2* cb = w.cand + (int64_t)b * max_len;
  uint32_t* bw = w.bits + (int64_t)b * nchunks_max * (kTopkChunk / 32);
  int sc[kPerThread];
  int T1, above, gt_total;
  if (!chunk_phase(scores + (int64_t)b * ld, w.hist + (int64_t)b * kScoreBins, start, stop, k,
                   cb, max_len, w.cand_n + b, bw, true, w.err, c == 0, sc, T1, above, gt_total, sm,
                   w.fkey != 0))
    return;
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
  const bool staged = n <= kCandCap;
  if (staged) {
    for (int i = tid; i < n; i += kTopkThreads) {
      const int2 e = __ldcg(cb + i);
      s_key[i] = order_key(e.x, e.y);
    }
    __syncthreads();
  }
  auto key_at = [&](int i) -> uint64_t {
    if (staged) return s_key[i];
    const int2 e = __ldcg(cb + i);
    return order_key(e.x, e.y);
  };
  const uint64_t kstar = select_threshold(n, k - above, key_at, sm);

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
    int pos = block_exclusive_scan<kTopkThreads>(cnt, &tot, sm.warp);
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
    int off = block_exclusive_scan<kTopkThreads>(mine, &tot, sm.warp);
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
            int max_len, int nchunks_max, int nq) {
  __shared__ int s_warp[kTopkThreads / 32];
  constexpr int kWords = kTopkChunk / 32;  // 128 words per chunk
  const int b = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
  const int len = clamp_len(seq_lens[b / nq], max_len);  // b: virtual request
  pdl_wait();  // bitmap and offsets come from k_topk_threshold
  pdl_launch_dependents();
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

namespace {

TopkWs topk_ws(const WorkspaceLayout& L, uint8_t* ws) {
  TopkWs w;
  w.hist = reinterpret_cast<int32_t*>(ws + L.hist);
  w.tick = reinterpret_cast<int32_t*>(ws + L.tick_topk);
  w.depart = reinterpret_cast<int32_t*>(ws + L.depart_topk);
  w.cand_n = reinterpret_cast<int32_t*>(ws + L.cand_n);
  w.cand = reinterpret_cast<int2*>(ws + L.cand);
  w.bits = reinterpret_cast<uint32_t*>(ws + L.bits);
  w.gt_cnt = reinterpret_cast<int32_t*>(ws + L.gt_cnt);
  w.chunk_off = reinterpret_cast<int32_t*>(ws + L.chunk_off);
  w.thr = reinterpret_cast<TopkThreshold*>(ws + L.thresh);
  w.err = reinterpret_cast<int32_t*>(ws + L.err);
  w.fkey = 0;
  return w;
}

// CTAs of k_topk_select the current device holds at once (cached per device).
int64_t select_capacity() {
  static int64_t cache[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  int64_t& cap = cache[dev & 63];
  if (cap == 0) {
    int coop = 0, bps = 0;
    if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, k_topk_select, kTopkThreads, 0) !=
            cudaSuccess)
      bps = 0;
    cap = coop ? (int64_t)bps * device_sm_count() : 0;
    if (cap == 0) cap = -1;
  }
  return cap;
}

}  // namespace

bool topk_single_launch(const pks_decode_args& a, const WorkspaceLayout& L) {
  return a.topk_mode == 0 && L.nchunks <= kTopkCoopMaxChunks &&
         (int64_t)L.nchunks * a.B * query_count(a) <= select_capacity();
}

cudaError_t launch_topk(const pks_decode_args& a, const WorkspaceLayout& L, uint8_t* ws,
                        cudaStream_t s) {
  const int max_len = a.max_pages * a.page_size;
  const int nq = query_count(a);
  const dim3 grid(L.nchunks, a.B * nq);  // virtual requests
  TopkWs w = topk_ws(L, ws);
  w.fkey = a.w_idx_f != nullptr ? 1 : 0;
  const int32_t* scores = reinterpret_cast<const int32_t*>(ws + L.scores);
  if (topk_single_launch(a, L)) {
    // cooperative: the launch fails rather than run with CTAs of a request
    // that cannot all be resident
    return launch_ex(k_topk_select, grid, dim3(kTopkThreads), 0, s, /*pdl=*/true, /*coop=*/true,
                     a.seq_lens, scores, L.ld, w, reinterpret_cast<int2*>(ws + L.chunk_cnt),
                     a.topk_idx, a.k, max_len, (int)L.nchunks, nq,
                     a.wait_limit > 0 ? a.wait_limit : kBarrierSpins);
  }
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
  cudaError_t e = launch_ex(k_topk_threshold, grid, dim3(kTopkThreads), smem, s, true, false,
                            a.seq_lens, scores, L.ld, w, a.topk_idx, a.k, max_len,
                            (int)L.nchunks, nq);
  if (e != cudaSuccess || max_len <= kBitmapTokens) return e;
  return launch_ex(k_topk_emit, grid, dim3(kTopkThreads), 0, s, true, false, a.seq_lens,
                   reinterpret_cast<const uint32_t*>(ws + L.bits),
                   reinterpret_cast<const int32_t*>(ws + L.chunk_off), a.topk_idx, a.k, max_len,
                   (int)L.nchunks, nq);
}

int topk_kernel_launches(const pks_decode_args& a, const WorkspaceLayout& L) {
  if (topk_single_launch(a, L)) return 1;
  return (int64_t)a.max_pages * a.page_size > kBitmapTokens ? 2 : 1;
}

}  // namespace pks
