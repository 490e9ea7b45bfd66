// Indexer scan: int8 lightning-indexer scores of every cached token, with the
// per-request score histogram that seeds the top-k radix select fused in.
//
// "Sparse Attention on GLM5.3 and HBM", DeepSeek Sparse Attention paragraph:
// the indexer query is multi-headed, the key single-headed; a token's score is
// the weighted sum over query heads of ReLU(query . key).  The introduction
// notes that selection needs the whole context resident in HBM: this kernel
// streams every indexer key once and is bound by HBM bandwidth.
//
// Work split: the tokens of all requests are cut into rounds of 256 tokens of
// one request; a persistent grid gives each CTA a contiguous range of rounds.
// In a round each warp handles 32 consecutive tokens.  A token's Di-byte key
// is read by Di/16 lanes with one 16-byte load each (a warp load covers 512
// contiguous bytes when the tokens share a page), the next round's keys are
// loaded before the current round is reduced.  Per lane: dp4a over its
// 16-byte slice for every head, then a transposed shuffle reduction that
// halves the per-lane head vector at each step, so that after log2(Di/16)
// steps every lane of the token holds full dot products, followed by ReLU,
// head weights and a short cross-lane sum.  After Di/16 warp steps each lane
// holds one token's score, so score stores are one 128-byte line per warp.

#include "pks_internal.h"

namespace pks {
namespace {

constexpr int kScanThreads = 256;
constexpr int kRoundTokens = kScanThreads;

__device__ __forceinline__ int score_bin(int s) {
  if (s == 0) return kScoreBins / 2;
  const unsigned a = s > 0 ? (unsigned)s : 0u - (unsigned)s;
  const int e = 31 - __clz(a);
  const unsigned m = e >= 5 ? (a >> (e - 5)) & 31u : (a << (5 - e)) & 31u;
  const int v = e * 32 + (int)m;  // 0 .. 1023
  return s > 0 ? kScoreBins / 2 + 1 + v : kScoreBins / 2 - 1 - v;
}

__device__ __forceinline__ void flag_error(int32_t* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// Exclusive scan over the block of one int per thread; returns this thread's
// prefix and writes the block total to *total.
template <int NT>
__device__ __forceinline__ int block_exclusive_scan(int v, int* total, int* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < NT / 32 ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < NT / 32) s_warp[lane] = w;  // inclusive warp totals
  }
  __syncthreads();
  const int before = (warp > 0 ? s_warp[warp - 1] : 0) + x - v;
  *total = s_warp[NT / 32 - 1];
  __syncthreads();
  return before;
}

// Reduce the per-lane head partials of one token across its LANES lanes.
// v: HI partial dot products over this lane's 16-byte slice.  wk: the head
// weights of the heads this lane ends up holding (see lane_heads).
template <int HI, int LANES>
struct TokenReduce {
  static constexpr int n_after(int st_count) { return HI; }
  // number of heads a lane holds after the halving steps
  static constexpr int kFinal = HI >= LANES ? HI / LANES : 1;

  // first head held by lane j after the halving steps
  __device__ static int head_base(int j) {
    int n = HI, base = 0;
#pragma unroll
    for (int st = LANES / 2; st >= 1; st >>= 1) {
      if (n >= 2) {
        n >>= 1;
        if (j & st) base += n;
      }
    }
    return base;
  }

  __device__ static int run(int (&v)[HI], int j, const int (&wk)[kFinal]) {
    int cur[HI];
#pragma unroll
    for (int i = 0; i < HI; ++i) cur[i] = v[i];
    int n = HI;
    unsigned halving = 0;
#pragma unroll
    for (int st = LANES / 2; st >= 1; st >>= 1) {
      if (n >= 2) {
        const int h = n >> 1;
        const bool up = (j & st) != 0;
#pragma unroll
        for (int i = 0; i < HI / 2; ++i) {
          if (i < h) {
            const int keep = up ? cur[i + h] : cur[i];
            const int send = up ? cur[i] : cur[i + h];
            cur[i] = keep + __shfl_xor_sync(0xffffffffu, send, st);
          }
        }
        n = h;
        halving |= (unsigned)st;
      } else {
        cur[0] += __shfl_xor_sync(0xffffffffu, cur[0], st);
      }
    }
    int s = 0;
#pragma unroll
    for (int i = 0; i < kFinal; ++i) s += wk[i] * max(cur[i], 0);
#pragma unroll
    for (int st = LANES / 2; st >= 1; st >>= 1)
      if (halving & (unsigned)st) s += __shfl_xor_sync(0xffffffffu, s, st);
    return s;
  }
};

template <int HI, int DI>
__global__ void __launch_bounds__(kScanThreads, HI >= 8 ? 1 : 2)
k_indexer_scan(const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ block_table,
               const int8_t* __restrict__ q_idx, const int32_t* __restrict__ w_idx,
               const int8_t* __restrict__ idx_k, int32_t* __restrict__ scores, int64_t ld,
               int32_t* __restrict__ hist, int32_t* __restrict__ err, int B, int max_pages,
               int page_size, int num_pages, int k) {
  constexpr int LANES = DI / 16;  // lanes per token
  constexpr int TPW = 32 / LANES;  // tokens per warp step
  using R = TokenReduce<HI, LANES>;

  extern __shared__ int s_prefix[];  // [B + 1] rounds prefix
  __shared__ int s_hist[kScoreBins];
  __shared__ int s_warp[kScanThreads / 32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane / LANES, j = lane % LANES;
  const int max_len = max_pages * page_size;

  // rounds per request -> exclusive prefix in shared memory
  const int per = (B + kScanThreads - 1) / kScanThreads;
  int local = 0;
  for (int i = 0; i < per; ++i) {
    const int b = tid * per + i;
    if (b < B) {
      int len = seq_lens[b];
      if (len < 0 || len > max_len) {
        if (blockIdx.x == 0) flag_error(err, kErrLen);
        len = 0;
      }
      local += (len + kRoundTokens - 1) / kRoundTokens;
    }
  }
  int total_rounds;
  int run = block_exclusive_scan<kScanThreads>(local, &total_rounds, s_warp);
  for (int i = 0; i < per; ++i) {
    const int b = tid * per + i;
    if (b < B) {
      s_prefix[b] = run;
      int len = seq_lens[b];
      if (len < 0 || len > max_len) len = 0;
      run += (len + kRoundTokens - 1) / kRoundTokens;
    }
  }
  if (tid == 0) s_prefix[B] = total_rounds;
  for (int i = tid; i < kScoreBins; i += kScanThreads) s_hist[i] = 0;
  __syncthreads();

  const int64_t G = gridDim.x;
  const int begin = (int)((int64_t)blockIdx.x * total_rounds / G);
  const int end = (int)((int64_t)(blockIdx.x + 1) * total_rounds / G);
  if (begin >= end) return;

  // first request with rounds at or after `begin`
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_prefix[mid] <= begin) lo = mid; else hi = mid - 1;
  }
  int b = lo;
  int item = begin;
  while (item < end) {
    while (s_prefix[b + 1] <= item) ++b;
    int len = seq_lens[b];
    if (len < 0 || len > max_len) len = 0;
    const int r0 = item - s_prefix[b];
    const int r1 = min(end, s_prefix[b + 1]) - s_prefix[b];
    item = s_prefix[b] + r1;
    const bool do_hist = hist != nullptr && len > k;

    // this lane's 16-byte slice of every indexer query head, and the weights
    // of the heads it holds after the reduction
    int4 qv[HI];
#pragma unroll
    for (int h = 0; h < HI; ++h)
      qv[h] = __ldg(reinterpret_cast<const int4*>(q_idx + ((int64_t)b * HI + h) * DI) + j);
    int wk[R::kFinal];
    {
      const int base = R::head_base(j);
#pragma unroll
      for (int i = 0; i < R::kFinal; ++i) {
        int w = 0;
#pragma unroll
        for (int h = 0; h < HI; ++h)
          if (h == base + i) w = __ldg(w_idx + h);
        wk[i] = w;
      }
    }
    const int32_t* bt = block_table + (int64_t)b * max_pages;

    auto load_round = [&](int r, int4 (&keys)[LANES]) {
#pragma unroll
      for (int u = 0; u < LANES; ++u) {
        const int t = r * kRoundTokens + warp * 32 + u * TPW + g;
        int4 v = make_int4(0, 0, 0, 0);
        if (t < len) {
          const int page = __ldg(bt + t / page_size);
          if ((unsigned)page < (unsigned)num_pages) {
            const int8_t* p = idx_k + ((int64_t)page * page_size + t % page_size) * DI;
            v = __ldcs(reinterpret_cast<const int4*>(p) + j);
          } else {
            flag_error(err, kErrPage);
          }
        }
        keys[u] = v;
      }
    };

    int4 cur[LANES];
    load_round(r0, cur);
    for (int r = r0; r < r1; ++r) {
      int4 nxt[LANES];
      if (r + 1 < r1) load_round(r + 1, nxt);
      int mine = 0;
#pragma unroll
      for (int u = 0; u < LANES; ++u) {
        int part[HI];
#pragma unroll
        for (int h = 0; h < HI; ++h) {
          int acc = __dp4a(cur[u].x, qv[h].x, 0);
          acc = __dp4a(cur[u].y, qv[h].y, acc);
          acc = __dp4a(cur[u].z, qv[h].z, acc);
          acc = __dp4a(cur[u].w, qv[h].w, acc);
          part[h] = acc;
        }
        const int s = R::run(part, j, wk);
        if (j == u) mine = s;
      }
      const int t = r * kRoundTokens + warp * 32 + j * TPW + g;
      const bool valid = t < len;
      if (valid) scores[(int64_t)b * ld + t] = mine;
      if (do_hist) {
        const unsigned vmask = __ballot_sync(0xffffffffu, valid);
        if (valid) {
          const int bin = score_bin(mine);
          const unsigned peers = __match_any_sync(vmask, bin);
          if (lane == __ffs(peers) - 1) atomicAdd(&s_hist[bin], __popc(peers));
        }
      }
#pragma unroll
      for (int u = 0; u < LANES; ++u) cur[u] = nxt[u];
    }
    if (do_hist) {
      __syncthreads();
      int32_t* gh = hist + (int64_t)b * kScoreBins;
      for (int i = tid; i < kScoreBins; i += kScanThreads) {
        const int c = s_hist[i];
        if (c) {
          atomicAdd(gh + i, c);
          s_hist[i] = 0;
        }
      }
      __syncthreads();
    }
  }
}

template <int HI, int DI>
cudaError_t launch_scan_t(const pks_decode_args& a, int32_t* scores, int64_t ld, int32_t* hist,
                          int32_t* err, cudaStream_t s) {
  auto kern = k_indexer_scan<HI, DI>;
  const size_t smem = sizeof(int) * (size_t)(a.B + 1);
  static int blocks_per_sm[2] = {0, 0};
  int dev = 0;
  cudaGetDevice(&dev);
  int& bps = blocks_per_sm[dev & 1];
  if (bps == 0) {
    if (smem > 48 * 1024)
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, kern, kScanThreads, smem);
    if (bps < 1) bps = 1;
  }
  const int grid = device_sm_count() * bps;
  kern<<<grid, kScanThreads, smem, s>>>(a.seq_lens, a.block_table, a.q_idx, a.w_idx, a.idx_k,
                                        scores, ld, hist, err, a.B, a.max_pages, a.page_size,
                                        a.num_pages, a.k);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_indexer_scan(const pks_decode_args& a, int32_t* scores, int64_t ld,
                                int32_t* hist, int32_t* err, cudaStream_t s) {
#define PKS_SCAN_CASE(HI_, DI_) \
  if (a.Hi == HI_ && a.Di == DI_) return launch_scan_t<HI_, DI_>(a, scores, ld, hist, err, s);
  PKS_SCAN_CASE(1, 64)
  PKS_SCAN_CASE(2, 64)
  PKS_SCAN_CASE(4, 64)
  PKS_SCAN_CASE(8, 64)
  PKS_SCAN_CASE(1, 128)
  PKS_SCAN_CASE(2, 128)
  PKS_SCAN_CASE(4, 128)
  PKS_SCAN_CASE(8, 128)
#undef PKS_SCAN_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pks
