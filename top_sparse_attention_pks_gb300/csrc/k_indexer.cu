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
// one request; a persistent grid (one CTA per SM) gives each CTA a contiguous
// range of rounds, and each of its 8 warps owns 32 tokens of every round.
// A warp streams its tokens' keys with 16-byte cp.async (each warp-wide copy
// covers 512 contiguous bytes when the tokens share a page) into its own
// slice of a shared-memory ring several rounds deep, so HBM reads run well
// ahead of the arithmetic and no block-wide barrier is needed in the loop.
// Every lane then scores one token: it reads its key back from shared memory
// (rows XOR-swizzled by 16-byte chunk, so the reads are conflict-free), runs
// dp4a against the indexer query held in registers, applies ReLU and the
// head weights.  Score stores are one 128-byte line per warp.

#include <cuda.h>

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

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// Pipeline depth in rounds: 4 rounds of 32 KB (Di = 128) or 8 of 16 KB in
// flight per CTA, enough to cover HBM latency at full bandwidth with one
// CTA per SM.
template <int DI>
struct ScanCfg {
  static constexpr int kStages = DI == 128 ? 5 : 9;
  static constexpr int kStageBytes = kRoundTokens * DI;
  static constexpr size_t smem_bytes(int B, int HI) {
    return (size_t)kStages * kStageBytes + sizeof(int) * kScoreBins + 16 * (size_t)HI * (DI / 16) +
           sizeof(int) * (size_t)(B + 1);
  }
};

template <int HI, int DI>
__global__ void __launch_bounds__(kScanThreads, 1)
k_indexer_scan(const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ block_table,
               const int8_t* __restrict__ q_idx, const int32_t* __restrict__ w_idx,
               const int8_t* __restrict__ idx_k, int32_t* __restrict__ scores, int64_t ld,
               int32_t* __restrict__ hist, int32_t* __restrict__ err, int B, int max_pages,
               int page_size, int page_shift, int num_pages, int k) {
  constexpr int CH = DI / 16;       // 16-byte chunks per key
  constexpr int TPI = 32 / CH;      // tokens covered by one warp-wide load instruction
  constexpr int SWZ_DIV = 8 / CH;   // chunk c of token r is stored at c ^ ((r / SWZ_DIV) % CH)
  constexpr bool kQInRegs = HI <= 4;
  constexpr int kStages = ScanCfg<DI>::kStages;
  constexpr int kStageBytes = ScanCfg<DI>::kStageBytes;
  constexpr int kWarpBytes = 32 * DI;

  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;  // [kStages][8 warps][32 tokens][DI], rows swizzled by 16-byte chunk
  int* s_hist = reinterpret_cast<int*>(smem + (size_t)kStages * kStageBytes);
  int4* s_q = reinterpret_cast<int4*>(s_hist + kScoreBins);  // [HI][CH] when q is not in registers
  int* s_prefix = reinterpret_cast<int*>(s_q + HI * CH);      // [B + 1] rounds prefix
  __shared__ int s_warp[kScanThreads / 32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
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

  // first request holding round `begin`
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_prefix[mid] <= begin) lo = mid; else hi = mid - 1;
  }

  // ---- loader.  Page lookups run two rounds ahead of the copies that use
  // them (a dependent block-table read would otherwise stall the warp once
  // per round).  lookup(item) returns this lane's physical token row, or -1.
  int lk_b = lo, lk_len = 0;
  {
    const int len = seq_lens[lk_b];
    lk_len = (len < 0 || len > max_len) ? 0 : len;
  }
  auto lookup_page = [&](int item, int& slot) -> int {
    // advance to the request holding `item` (items only increase)
    while (s_prefix[lk_b + 1] <= item) {
      ++lk_b;
      const int len = seq_lens[lk_b];
      lk_len = (len < 0 || len > max_len) ? 0 : len;
    }
    const int t = (item - s_prefix[lk_b]) * kRoundTokens + warp * 32 + lane;
    slot = -1;
    if (t >= lk_len) return -1;
    const int lp = page_shift >= 0 ? (t >> page_shift) : t / page_size;
    slot = page_shift >= 0 ? (t & (page_size - 1)) : t % page_size;
    return __ldg(block_table + (int64_t)lk_b * max_pages + lp);
  };
  auto issue = [&](int page, int slot, int stage) {
    int row = -1;
    if (slot >= 0) {
      if ((unsigned)page < (unsigned)num_pages) row = page * page_size + slot;
      else flag_error(err, kErrPage);
    }
    uint8_t* wbase = ring + (size_t)stage * kStageBytes + warp * kWarpBytes;
    const int c = lane % CH;
#pragma unroll
    for (int i = 0; i < CH; ++i) {
      const int tt = i * TPI + lane / CH;  // token of this warp's slice
      const int rr = __shfl_sync(0xffffffffu, row, tt);
      if (rr >= 0)
        cp_async16(smem_u32(wbase + tt * DI + ((c ^ ((tt / SWZ_DIV) % CH)) << 4)),
                   idx_k + (int64_t)rr * DI + c * 16);
    }
  };

  // prologue: copies for the first kStages-1 rounds, lookups for the next two
#pragma unroll
  for (int st = 0; st < kStages - 1; ++st) {
    if (begin + st < end) {
      int slot;
      const int page = lookup_page(begin + st, slot);
      issue(page, slot, st);
    }
    cp_async_commit();
  }
  int pg0 = -1, sl0 = -1, pg1 = -1, sl1 = -1;  // lookups of rounds begin+S-1, begin+S
  if (begin + kStages - 1 < end) pg0 = lookup_page(begin + kStages - 1, sl0);
  if (begin + kStages < end) pg1 = lookup_page(begin + kStages, sl1);

  // ---- consumer: every lane scores one token per round
  int4 q[kQInRegs ? HI : 1][kQInRegs ? CH : 1];
  int w[HI];
  int cb = -1, cb_len = 0;
  bool do_hist = false;
  int b = lo;
  const int swz = (lane / SWZ_DIV) % CH;
  for (int item = begin; item < end; ++item) {
    const int rel = item - begin;
    {
      int pg2 = -1, sl2 = -1;
      if (item + kStages + 1 < end) pg2 = lookup_page(item + kStages + 1, sl2);
      if (item + kStages - 1 < end) issue(pg0, sl0, (rel + kStages - 1) % kStages);
      pg0 = pg1;
      sl0 = sl1;
      pg1 = pg2;
      sl1 = sl2;
    }
    cp_async_commit();

    while (s_prefix[b + 1] <= item) ++b;
    if (b != cb) {
      // request switch (uniform across the CTA): flush the histogram, load q
      if (do_hist) {
        __syncthreads();
        int32_t* gh = hist + (int64_t)cb * kScoreBins;
        for (int i = tid; i < kScoreBins; i += kScanThreads) {
          const int cnt = s_hist[i];
          if (cnt) {
            atomicAdd(gh + i, cnt);
            s_hist[i] = 0;
          }
        }
      }
      __syncthreads();
      cb = b;
      const int len = seq_lens[b];
      cb_len = (len < 0 || len > max_len) ? 0 : len;
      do_hist = hist != nullptr && cb_len > k;
      const int4* qg = reinterpret_cast<const int4*>(q_idx + (int64_t)b * HI * DI);
      if constexpr (kQInRegs) {
#pragma unroll
        for (int h = 0; h < HI; ++h)
#pragma unroll
          for (int cc = 0; cc < CH; ++cc) q[h][cc] = __ldg(qg + h * CH + cc);
      } else {
        for (int i = tid; i < HI * CH; i += kScanThreads) s_q[i] = __ldg(qg + i);
        __syncthreads();
      }
#pragma unroll
      for (int h = 0; h < HI; ++h) w[h] = __ldg(w_idx + h);
    }

    cp_async_wait<kStages - 1>();
    __syncwarp();
    const uint8_t* rowp = ring + (size_t)(rel % kStages) * kStageBytes + warp * kWarpBytes + lane * DI;
    int acc[HI];
#pragma unroll
    for (int h = 0; h < HI; ++h) acc[h] = 0;
#pragma unroll
    for (int cc = 0; cc < CH; ++cc) {
      const int4 kv = *reinterpret_cast<const int4*>(rowp + ((cc ^ swz) << 4));
#pragma unroll
      for (int h = 0; h < HI; ++h) {
        int4 qv;
        if constexpr (kQInRegs) qv = q[h][cc];
        else qv = s_q[h * CH + cc];
        acc[h] = __dp4a(kv.x, qv.x, acc[h]);
        acc[h] = __dp4a(kv.y, qv.y, acc[h]);
        acc[h] = __dp4a(kv.z, qv.z, acc[h]);
        acc[h] = __dp4a(kv.w, qv.w, acc[h]);
      }
    }
    int score = 0;
#pragma unroll
    for (int h = 0; h < HI; ++h) score += w[h] * max(acc[h], 0);

    const int t = (item - s_prefix[b]) * kRoundTokens + warp * 32 + lane;
    const bool valid = t < cb_len;
    if (valid) scores[(int64_t)b * ld + t] = score;
    if (do_hist) {
      const unsigned vmask = __ballot_sync(0xffffffffu, valid);
      if (valid) {
        const int bin = score_bin(score);
        const unsigned peers = __match_any_sync(vmask, bin);
        if (lane == __ffs(peers) - 1) atomicAdd(&s_hist[bin], __popc(peers));
      }
    }
    __syncwarp();
  }
  cp_async_wait<0>();
  if (do_hist) {
    __syncthreads();
    int32_t* gh = hist + (int64_t)cb * kScoreBins;
    for (int i = tid; i < kScoreBins; i += kScanThreads) {
      const int cnt = s_hist[i];
      if (cnt) atomicAdd(gh + i, cnt);
    }
  }
}

// ---------------------------------------------------------------------------
// Register-streaming variant.  Keys go from HBM straight into registers with
// coalesced 16-byte loads (each warp-wide load covers Di/16 lanes x 32/(Di/16)
// tokens = 512 contiguous bytes), double-buffered one round ahead, 16 warps
// per SM.  Lane (g, j) holds chunk j of the tokens j' * (32 / (Di/16)) + g of
// its round and multiplies it with chunk j of every indexer head (query
// chunks live in registers).  A transposed butterfly across the Di/16 lanes of
// a token then halves the token slots at each step, so that after log2(Di/16)
// steps lane (g, j) holds the full head dot products of token j*(32/(Di/16))+g
// and finishes its score alone.  Shared memory holds only the histogram and
// the round prefix; the loop has no block-wide barrier.

constexpr int kRegWarps = 16;
constexpr int kRegThreads = kRegWarps * 32;
constexpr int kRegRound = kRegThreads;  // tokens per CTA round (32 per warp)

template <int HI, int DI>
__global__ void __launch_bounds__(kRegThreads, 1)
k_indexer_scan_reg(const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ block_table,
                   const int8_t* __restrict__ q_idx, const int32_t* __restrict__ w_idx,
                   const int8_t* __restrict__ idx_k, int32_t* __restrict__ scores, int64_t ld,
                   int32_t* __restrict__ hist, int32_t* __restrict__ err, int B, int max_pages,
                   int page_size, int page_shift, int num_pages, int k) {
  constexpr int LPT = DI / 16;  // lanes per token (one 16-byte chunk each)
  constexpr int TPI = 32 / LPT;  // tokens per warp-wide load
  constexpr int NI = LPT;        // loads per lane per round (32 tokens)

  extern __shared__ int smem_i[];
  int* s_hist = smem_i;                 // [kScoreBins]
  int* s_prefix = smem_i + kScoreBins;  // [B + 1]
  __shared__ int s_warp[kRegThreads / 32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane / LPT, j = lane % LPT;
  const int max_len = max_pages * page_size;

  // rounds per request -> exclusive prefix in shared memory
  const int per = (B + kRegThreads - 1) / kRegThreads;
  int local = 0;
  for (int i = 0; i < per; ++i) {
    const int b = tid * per + i;
    if (b < B) {
      int len = seq_lens[b];
      if (len < 0 || len > max_len) {
        if (blockIdx.x == 0) flag_error(err, kErrLen);
        len = 0;
      }
      local += (len + kRegRound - 1) / kRegRound;
    }
  }
  int total_rounds;
  int run = block_exclusive_scan<kRegThreads>(local, &total_rounds, s_warp);
  for (int i = 0; i < per; ++i) {
    const int b = tid * per + i;
    if (b < B) {
      s_prefix[b] = run;
      int len = seq_lens[b];
      if (len < 0 || len > max_len) len = 0;
      run += (len + kRegRound - 1) / kRegRound;
    }
  }
  if (tid == 0) s_prefix[B] = total_rounds;
  for (int i = tid; i < kScoreBins; i += kRegThreads) s_hist[i] = 0;
  __syncthreads();

  const int64_t G = gridDim.x;
  const int begin = (int)((int64_t)blockIdx.x * total_rounds / G);
  const int end = (int)((int64_t)(blockIdx.x + 1) * total_rounds / G);
  if (begin >= end) return;
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_prefix[mid] <= begin) lo = mid; else hi = mid - 1;
  }

  // ---- page lookups, one token per lane, issued two rounds ahead
  int lk_b = lo, lk_len = 0, lk_next = s_prefix[lo + 1];
  {
    const int len = seq_lens[lk_b];
    lk_len = (len < 0 || len > max_len) ? 0 : len;
  }
  // -> physical key row of this lane's token of round `item` (page id still
  // to be checked), or -1; `slot` receives the row within the page
  auto lookup = [&](int item, int& slot) -> int {
    while (lk_next <= item) {
      ++lk_b;
      lk_next = s_prefix[lk_b + 1];
      const int len = seq_lens[lk_b];
      lk_len = (len < 0 || len > max_len) ? 0 : len;
    }
    const int t = (item - s_prefix[lk_b]) * kRegRound + warp * 32 + lane;
    slot = -1;
    if (t >= lk_len) return -1;
    const int lp = page_shift >= 0 ? (t >> page_shift) : t / page_size;
    slot = page_shift >= 0 ? (t & (page_size - 1)) : t % page_size;
    return __ldg(block_table + (int64_t)lk_b * max_pages + lp);
  };
  auto to_row = [&](int page, int slot) -> int {
    if (slot < 0) return -1;
    if ((unsigned)page < (unsigned)num_pages) return page * page_size + slot;
    flag_error(err, kErrPage);
    return -1;
  };
  auto load_round = [&](int row, int4 (&buf)[NI]) {
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const int rr = __shfl_sync(0xffffffffu, row, i * TPI + g);
      buf[i] = rr >= 0 ? __ldcs(reinterpret_cast<const int4*>(idx_k + (int64_t)rr * DI) + j)
                       : make_int4(0, 0, 0, 0);
    }
  };

  int4 cur[NI], nxt[NI];
  int pg1, sl1, pg2, sl2;  // lookups of rounds item+1 and item+2
  {
    int sl0;
    const int pg0 = lookup(begin, sl0);
    load_round(to_row(pg0, sl0), cur);
    pg1 = begin + 1 < end ? lookup(begin + 1, sl1) : (sl1 = -1, -1);
    pg2 = begin + 2 < end ? lookup(begin + 2, sl2) : (sl2 = -1, -1);
  }

  int4 qv[HI];
  int w[HI];
  int cb = -1, cb_len = 0, cb_first = 0, cb_next = 0;
  bool do_hist = false;
  for (int item = begin; item < end; ++item) {
    if (item + 1 < end) load_round(to_row(pg1, sl1), nxt);
    {
      int sl3 = -1;
      const int pg3 = item + 3 < end ? lookup(item + 3, sl3) : -1;
      pg1 = pg2;
      sl1 = sl2;
      pg2 = pg3;
      sl2 = sl3;
    }
    if (item >= cb_next) {
      // request switch (uniform across the CTA): flush the histogram, load q
      int b = cb < 0 ? lo : cb;
      while (s_prefix[b + 1] <= item) ++b;
      if (do_hist) {
        __syncthreads();
        int32_t* gh = hist + (int64_t)cb * kScoreBins;
        for (int i = tid; i < kScoreBins; i += kRegThreads) {
          const int cnt = s_hist[i];
          if (cnt) {
            atomicAdd(gh + i, cnt);
            s_hist[i] = 0;
          }
        }
      }
      __syncthreads();
      cb = b;
      cb_first = s_prefix[b];
      cb_next = s_prefix[b + 1];
      const int len = seq_lens[b];
      cb_len = (len < 0 || len > max_len) ? 0 : len;
      do_hist = hist != nullptr && cb_len > k;
#pragma unroll
      for (int h = 0; h < HI; ++h) {
        qv[h] = __ldg(reinterpret_cast<const int4*>(q_idx + ((int64_t)b * HI + h) * DI) + j);
        w[h] = __ldg(w_idx + h);
      }
    }

    // partial dot products: p[i][h] over this lane's chunk of token slot i
    int p[NI][HI];
#pragma unroll
    for (int i = 0; i < NI; ++i)
#pragma unroll
      for (int h = 0; h < HI; ++h) {
        int a = __dp4a(cur[i].x, qv[h].x, 0);
        a = __dp4a(cur[i].y, qv[h].y, a);
        a = __dp4a(cur[i].z, qv[h].z, a);
        p[i][h] = __dp4a(cur[i].w, qv[h].w, a);
      }
    // transposed butterfly: at stride s the lane keeps the upper half of its
    // slots when (j & s) is set, and adds its partner's copy of them
#pragma unroll
    for (int s = LPT / 2, n = NI; s >= 1; s >>= 1, n >>= 1) {
      const bool up = (j & s) != 0;
#pragma unroll
      for (int m = 0; m < n / 2; ++m)
#pragma unroll
        for (int h = 0; h < HI; ++h) {
          const int keep = up ? p[m + n / 2][h] : p[m][h];
          const int send = up ? p[m][h] : p[m + n / 2][h];
          p[m][h] = keep + __shfl_xor_sync(0xffffffffu, send, s);
        }
    }
    int score = 0;
#pragma unroll
    for (int h = 0; h < HI; ++h) score += w[h] * max(p[0][h], 0);

    // lane (g, j) now holds token slot j, i.e. token j * TPI + g of the round
    const int t = (item - cb_first) * kRegRound + warp * 32 + j * TPI + g;
    const bool valid = t < cb_len;
    if (valid) scores[(int64_t)cb * ld + t] = score;
    if (do_hist) {
      const unsigned vmask = __ballot_sync(0xffffffffu, valid);
      if (valid) {
        const int bin = score_bin(score);
        const unsigned peers = __match_any_sync(vmask, bin);
        if (lane == __ffs(peers) - 1) atomicAdd(&s_hist[bin], __popc(peers));
      }
    }
#pragma unroll
    for (int i = 0; i < NI; ++i) cur[i] = nxt[i];
  }
  if (do_hist) {
    __syncthreads();
    int32_t* gh = hist + (int64_t)cb * kScoreBins;
    for (int i = tid; i < kScoreBins; i += kRegThreads) {
      const int cnt = s_hist[i];
      if (cnt) atomicAdd(gh + i, cnt);
    }
  }
}

// ---------------------------------------------------------------------------
// Tensor-core variant for 4 or 8 indexer heads.  The head dot products of 16
// tokens are one int8 MMA tile per 32 key bytes: m16n8k32 with the tokens as
// M, the (zero-padded to 8) heads as N and the key bytes as K, int32
// accumulate - exact, like dp4a, but the cross-lane sum happens inside the
// tensor core, so a 32-token round costs 8 MMAs instead of ~100 dp4a and
// shuffles per lane.  Keys stream from HBM straight into the A fragments: lane
// (g, t) loads bytes [16t, 16t+16) and [64+16t, 64+16t+16) of tokens g and
// g+8 of each 16-token tile (each warp-wide load reads 8 rows x 64 contiguous
// bytes); the K order inside a tile is permuted identically in the key and
// query fragments, which leaves every dot product unchanged.

template <int DI>
__device__ __forceinline__ void imma_16832(int (&c)[4], int a0, int a1, int a2, int a3, int b0,
                                           int b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int HI, int DI, int NT>
__global__ void __launch_bounds__(NT, 1)
k_indexer_scan_mma(const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ block_table,
                   const int8_t* __restrict__ q_idx, const int32_t* __restrict__ w_idx,
                   const int8_t* __restrict__ idx_k, int32_t* __restrict__ scores, int64_t ld,
                   int32_t* __restrict__ hist, int32_t* __restrict__ err, int B, int max_pages,
                   int page_size, int page_shift, int num_pages, int k) {
  static_assert(HI <= 8, "N = 8 heads per MMA");
  constexpr int HALVES = DI / 64;      // 64-byte halves of a key (2 or 1)
  constexpr int NLD = 2 * 2 * HALVES;  // loads per lane per 32-token round

  extern __shared__ int smem_i[];
  int* s_hist = smem_i;                 // [kScoreBins]
  int* s_prefix = smem_i + kScoreBins;  // [B + 1]
  __shared__ int s_warp[NT / 32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gq = lane >> 2, tq = lane & 3;  // MMA group and thread-in-group
  const int max_len = max_pages * page_size;

  const int per = (B + NT - 1) / NT;
  int local = 0;
  for (int i = 0; i < per; ++i) {
    const int b = tid * per + i;
    if (b < B) {
      int len = seq_lens[b];
      if (len < 0 || len > max_len) {
        if (blockIdx.x == 0) flag_error(err, kErrLen);
        len = 0;
      }
      local += (len + NT - 1) / NT;
    }
  }
  int total_rounds;
  int run = block_exclusive_scan<NT>(local, &total_rounds, s_warp);
  for (int i = 0; i < per; ++i) {
    const int b = tid * per + i;
    if (b < B) {
      s_prefix[b] = run;
      int len = seq_lens[b];
      if (len < 0 || len > max_len) len = 0;
      run += (len + NT - 1) / NT;
    }
  }
  if (tid == 0) s_prefix[B] = total_rounds;
  for (int i = tid; i < kScoreBins; i += NT) s_hist[i] = 0;
  __syncthreads();

  const int64_t G = gridDim.x;
  const int begin = (int)((int64_t)blockIdx.x * total_rounds / G);
  const int end = (int)((int64_t)(blockIdx.x + 1) * total_rounds / G);
  if (begin >= end) return;
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_prefix[mid] <= begin) lo = mid; else hi = mid - 1;
  }

  int lk_b = lo, lk_len = 0, lk_next = s_prefix[lo + 1];
  {
    const int len = seq_lens[lk_b];
    lk_len = (len < 0 || len > max_len) ? 0 : len;
  }
  // page of this lane's token (token `lane` of the warp's 32) of round `item`
  auto lookup = [&](int item, int& slot) -> int {
    while (lk_next <= item) {
      ++lk_b;
      lk_next = s_prefix[lk_b + 1];
      const int len = seq_lens[lk_b];
      lk_len = (len < 0 || len > max_len) ? 0 : len;
    }
    const int t = (item - s_prefix[lk_b]) * NT + warp * 32 + lane;
    slot = -1;
    if (t >= lk_len) return -1;
    const int lp = page_shift >= 0 ? (t >> page_shift) : t / page_size;
    slot = page_shift >= 0 ? (t & (page_size - 1)) : t % page_size;
    return __ldg(block_table + (int64_t)lk_b * max_pages + lp);
  };
  auto to_row = [&](int page, int slot) -> int {
    if (slot < 0) return -1;
    if ((unsigned)page < (unsigned)num_pages) return page * page_size + slot;
    flag_error(err, kErrPage);
    return -1;
  };
  // loads of a round: [tile u][half hv][row g or g+8]
  auto load_round = [&](int row, int4 (&buf)[NLD]) {
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
      for (int r8 = 0; r8 < 2; ++r8) {
        const int rr = __shfl_sync(0xffffffffu, row, u * 16 + gq + 8 * r8);
#pragma unroll
        for (int hv = 0; hv < HALVES; ++hv)
          buf[(u * HALVES + hv) * 2 + r8] =
              rr >= 0 ? __ldcs(reinterpret_cast<const int4*>(idx_k + (int64_t)rr * DI) + 4 * hv + tq)
                      : make_int4(0, 0, 0, 0);
      }
  };

  // single-buffered: the other warps of the SM overlap a warp's load latency
  int4 cur[NLD];
  int pg0, sl0, pg1, sl1;  // lookups of rounds item and item+1
  pg0 = lookup(begin, sl0);
  pg1 = begin + 1 < end ? lookup(begin + 1, sl1) : (sl1 = -1, -1);

  int4 qf[HALVES];  // chunks 4*hv + tq of head gq (zero for padded heads)
  int w0 = 0, w1 = 0;  // weights of heads 2tq and 2tq+1
  int cb = -1, cb_len = 0, cb_first = 0, cb_next = 0;
  bool do_hist = false;
  // output token of this lane: tile (tq >> 1), row gq + 8 * (tq & 1)
  const int my_tok = (tq >> 1) * 16 + gq + 8 * (tq & 1);
  for (int item = begin; item < end; ++item) {
    load_round(to_row(pg0, sl0), cur);
    {
      int sl2 = -1;
      const int pg2 = item + 2 < end ? lookup(item + 2, sl2) : -1;
      pg0 = pg1;
      sl0 = sl1;
      pg1 = pg2;
      sl1 = sl2;
    }
    if (item >= cb_next) {
      int b = cb < 0 ? lo : cb;
      while (s_prefix[b + 1] <= item) ++b;
      if (do_hist) {
        __syncthreads();
        int32_t* gh = hist + (int64_t)cb * kScoreBins;
        for (int i = tid; i < kScoreBins; i += NT) {
          const int cnt = s_hist[i];
          if (cnt) {
            atomicAdd(gh + i, cnt);
            s_hist[i] = 0;
          }
        }
      }
      __syncthreads();
      cb = b;
      cb_first = s_prefix[b];
      cb_next = s_prefix[b + 1];
      const int len = seq_lens[b];
      cb_len = (len < 0 || len > max_len) ? 0 : len;
      do_hist = hist != nullptr && cb_len > k;
#pragma unroll
      for (int hv = 0; hv < HALVES; ++hv)
        qf[hv] = gq < HI ? __ldg(reinterpret_cast<const int4*>(q_idx + ((int64_t)b * HI + gq) * DI) +
                                 4 * hv + tq)
                         : make_int4(0, 0, 0, 0);
      w0 = 2 * tq < HI ? __ldg(w_idx + 2 * tq) : 0;
      w1 = 2 * tq + 1 < HI ? __ldg(w_idx + 2 * tq + 1) : 0;
    }

    int sc[2][2];  // [tile][row g / g+8]
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      int c[4] = {0, 0, 0, 0};
#pragma unroll
      for (int hv = 0; hv < HALVES; ++hv) {
        const int4 r0 = cur[(u * HALVES + hv) * 2 + 0];  // token row gq
        const int4 r1 = cur[(u * HALVES + hv) * 2 + 1];  // token row gq + 8
        imma_16832<DI>(c, r0.x, r1.x, r0.y, r1.y, qf[hv].x, qf[hv].y);
        imma_16832<DI>(c, r0.z, r1.z, r0.w, r1.w, qf[hv].z, qf[hv].w);
      }
      // c0, c1: heads 2tq, 2tq+1 of row gq; c2, c3: the same for row gq+8
      int pa = w0 * max(c[0], 0) + w1 * max(c[1], 0);
      int pb = w0 * max(c[2], 0) + w1 * max(c[3], 0);
      pa += __shfl_xor_sync(0xffffffffu, pa, 1);
      pa += __shfl_xor_sync(0xffffffffu, pa, 2);
      pb += __shfl_xor_sync(0xffffffffu, pb, 1);
      pb += __shfl_xor_sync(0xffffffffu, pb, 2);
      sc[u][0] = pa;
      sc[u][1] = pb;
    }
    const int score = (tq >> 1) ? ((tq & 1) ? sc[1][1] : sc[1][0])
                                : ((tq & 1) ? sc[0][1] : sc[0][0]);  // no local-memory indexing
    const int t = (item - cb_first) * NT + warp * 32 + my_tok;
    const bool valid = t < cb_len;
    if (valid) scores[(int64_t)cb * ld + t] = score;
    // plain shared atomics: colliding lanes of a warp are serialised by the
    // hardware, which costs less than aggregating them first
    if (do_hist && valid) atomicAdd(&s_hist[score_bin(score)], 1);
  }
  if (do_hist) {
    __syncthreads();
    int32_t* gh = hist + (int64_t)cb * kScoreBins;
    for (int i = tid; i < kScoreBins; i += NT) {
      const int cnt = s_hist[i];
      if (cnt) atomicAdd(gh + i, cnt);
    }
  }
}

// ---------------------------------------------------------------------------
// TMA variant (page sizes that are powers of two >= 8).  Same work split; the
// copies are tiled cp.async.bulk.tensor loads of one box of min(64, page_size)
// key rows, issued by one lane per box, completing on a per-warp, per-stage
// mbarrier.  The 128-byte (Di = 128) or 64-byte (Di = 64) swizzle of the
// tensor map puts chunk c of row r at c ^ (r % 8) or c ^ ((r / 2) % 4): the
// layout the readers use.  8 warps per CTA (one CTA per SM); a warp round is
// 64 tokens and every lane scores two of them (rows lane and lane + 32), so
// each indexer-query load and all per-round bookkeeping serve two tokens.

constexpr int kTmaWarps = 8;
constexpr int kTmaThreads = kTmaWarps * 32;
constexpr int kWarpTokens = 64;
constexpr int kTmaRound = kTmaWarps * kWarpTokens;  // tokens per CTA round
constexpr uint32_t kWaitLimit = 1u << 24;           // bounded mbarrier wait (polls)

template <int DI>
struct TmaCfg {
  static constexpr int kStages = DI == 128 ? 3 : 6;
  static constexpr int kWarpStage = kWarpTokens * DI;  // bytes of one warp's round
  static size_t smem_bytes(int B, int HI) {
    return 1024 + (size_t)kTmaWarps * kStages * kWarpStage + sizeof(int) * kScoreBins +
           (size_t)HI * DI + sizeof(uint64_t) * kTmaWarps * kStages + sizeof(int) * (size_t)(B + 1);
  }
};

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: false if the phase did not complete within kWaitLimit polls.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

template <int HI, int DI>
__global__ void __launch_bounds__(kTmaThreads, 1)
k_indexer_scan_tma(const __grid_constant__ CUtensorMap keys, const int32_t* __restrict__ seq_lens,
                   const int32_t* __restrict__ block_table, const int8_t* __restrict__ q_idx,
                   const int32_t* __restrict__ w_idx, int32_t* __restrict__ scores, int64_t ld,
                   int32_t* __restrict__ hist, int32_t* __restrict__ err, int B, int max_pages,
                   int page_size, int page_shift, int num_pages, int k) {
  constexpr int CH = DI / 16;
  constexpr int SWZ_DIV = 8 / CH;
  constexpr int kStages = TmaCfg<DI>::kStages;
  constexpr int kWarpStage = TmaCfg<DI>::kWarpStage;
  constexpr bool kQInRegs = HI * CH <= 16;

  extern __shared__ uint8_t smem_raw[];
  // the swizzle pattern is taken from address bits: align the ring to 1 KB
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* ring = smem;  // [warps][kStages][64 rows][DI]
  int* s_hist = reinterpret_cast<int*>(ring + (size_t)kTmaWarps * kStages * kWarpStage);
  int4* s_q = reinterpret_cast<int4*>(s_hist + kScoreBins);                // [HI][CH]
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(s_q + HI * CH);           // [warps][kStages]
  int* s_prefix = reinterpret_cast<int*>(s_bar + kTmaWarps * kStages);    // [B + 1]
  __shared__ int s_warp[kTmaThreads / 32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int max_len = max_pages * page_size;
  const int box_rows = page_size < kWarpTokens ? page_size : kWarpTokens;
  const int nbox = kWarpTokens / box_rows;  // boxes per warp round (<= 8)

  // rounds per request -> exclusive prefix in shared memory
  const int per = (B + kTmaThreads - 1) / kTmaThreads;
  int local = 0;
  for (int i = 0; i < per; ++i) {
    const int b = tid * per + i;
    if (b < B) {
      int len = seq_lens[b];
      if (len < 0 || len > max_len) {
        if (blockIdx.x == 0) flag_error(err, kErrLen);
        len = 0;
      }
      local += (len + kTmaRound - 1) / kTmaRound;
    }
  }
  int total_rounds;
  int run = block_exclusive_scan<kTmaThreads>(local, &total_rounds, s_warp);
  for (int i = 0; i < per; ++i) {
    const int b = tid * per + i;
    if (b < B) {
      s_prefix[b] = run;
      int len = seq_lens[b];
      if (len < 0 || len > max_len) len = 0;
      run += (len + kTmaRound - 1) / kTmaRound;
    }
  }
  if (tid == 0) s_prefix[B] = total_rounds;
  for (int i = tid; i < kScoreBins; i += kTmaThreads) s_hist[i] = 0;
  if (lane == 0)
    for (int st = 0; st < kStages; ++st) mbar_init(smem_u32(&s_bar[warp * kStages + st]), 1);
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  __syncthreads();

  const int64_t G = gridDim.x;
  const int begin = (int)((int64_t)blockIdx.x * total_rounds / G);
  const int end = (int)((int64_t)(blockIdx.x + 1) * total_rounds / G);
  if (begin >= end) return;

  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_prefix[mid] <= begin) lo = mid; else hi = mid - 1;
  }

  // ---- producer side.  Lane i < nbox owns box i of the warp's 64 tokens;
  // page lookups run two rounds ahead of the copies.
  int lk_b = lo, lk_len = 0, lk_next = s_prefix[lo + 1];
  {
    const int len = seq_lens[lk_b];
    lk_len = (len < 0 || len > max_len) ? 0 : len;
  }
  // -> first row of this lane's box in the key pool, or -1 (no box)
  auto lookup_box = [&](int item) -> int {
    while (lk_next <= item) {
      ++lk_b;
      lk_next = s_prefix[lk_b + 1];
      const int len = seq_lens[lk_b];
      lk_len = (len < 0 || len > max_len) ? 0 : len;
    }
    const int t0 = (item - s_prefix[lk_b]) * kTmaRound + warp * kWarpTokens + lane * box_rows;
    if (lane >= nbox || t0 >= lk_len) return -1;
    const int page = __ldg(block_table + (int64_t)lk_b * max_pages + (t0 >> page_shift));
    if ((unsigned)page >= (unsigned)num_pages) {
      flag_error(err, kErrPage);
      return -1;
    }
    return page * page_size + (t0 & (page_size - 1));
  };
  uint8_t* wring = ring + (size_t)warp * kStages * kWarpStage;
  const uint32_t bar0 = smem_u32(&s_bar[warp * kStages]);
  auto produce = [&](int row, int stage) {
    const uint32_t bar = bar0 + 8u * stage;
    const unsigned have = __ballot_sync(0xffffffffu, row >= 0);
    if (lane == 0) mbar_arrive_tx(bar, (uint32_t)__popc(have) * box_rows * DI);
    __syncwarp();
    if (row >= 0)
      tma_load_2d(smem_u32(wring + (size_t)stage * kWarpStage + (size_t)lane * box_rows * DI),
                  &keys, 0, row, bar);
  };

  int pst = 0;  // stage the next produce goes to
#pragma unroll
  for (int st = 0; st < kStages - 1; ++st) {
    if (begin + st < end) produce(lookup_box(begin + st), pst);
    pst = pst + 1 == kStages ? 0 : pst + 1;
  }
  int rw0 = -1, rw1 = -1;  // looked-up boxes of rounds begin+S-1 and begin+S
  if (begin + kStages - 1 < end) rw0 = lookup_box(begin + kStages - 1);
  if (begin + kStages < end) rw1 = lookup_box(begin + kStages);

  // ---- consumer side: every lane scores rows lane and lane + 32 of a round
  int4 q[kQInRegs ? HI : 1][kQInRegs ? CH : 1];
  int w[HI];
  int cb = -1, cb_len = 0, cb_first = 0, cb_next = 0;
  bool do_hist = false, dead = false;
  int cst = 0;       // stage being consumed
  uint32_t par = 0;  // its mbarrier phase parity
  const int swz = (lane / SWZ_DIV) % CH;  // same for rows lane and lane + 32
  for (int item = begin; item < end; ++item) {
    {
      const int rw2 = item + kStages + 1 < end ? lookup_box(item + kStages + 1) : -1;
      if (item + kStages - 1 < end && !dead) produce(rw0, pst);
      pst = pst + 1 == kStages ? 0 : pst + 1;
      rw0 = rw1;
      rw1 = rw2;
    }

    if (item >= cb_next) {
      // request switch (uniform across the CTA): flush the histogram, load q
      int b = cb < 0 ? lo : cb;
      while (s_prefix[b + 1] <= item) ++b;
      if (do_hist) {
        __syncthreads();
        int32_t* gh = hist + (int64_t)cb * kScoreBins;
        for (int i = tid; i < kScoreBins; i += kTmaThreads) {
          const int cnt = s_hist[i];
          if (cnt) {
            atomicAdd(gh + i, cnt);
            s_hist[i] = 0;
          }
        }
      }
      __syncthreads();
      cb = b;
      cb_first = s_prefix[b];
      cb_next = s_prefix[b + 1];
      const int len = seq_lens[b];
      cb_len = (len < 0 || len > max_len) ? 0 : len;
      do_hist = hist != nullptr && cb_len > k;
      const int4* qg = reinterpret_cast<const int4*>(q_idx + (int64_t)b * HI * DI);
      if constexpr (kQInRegs) {
#pragma unroll
        for (int h = 0; h < HI; ++h)
#pragma unroll
          for (int cc = 0; cc < CH; ++cc) q[h][cc] = __ldg(qg + h * CH + cc);
      } else {
        for (int i = tid; i < HI * CH; i += kTmaThreads) s_q[i] = __ldg(qg + i);
        __syncthreads();
      }
#pragma unroll
      for (int h = 0; h < HI; ++h) w[h] = __ldg(w_idx + h);
    }

    if (!dead && !mbar_wait(bar0 + 8u * cst, par)) {
      flag_error(err, kErrTimeout);
      dead = true;
    }
    __syncwarp();
    const uint8_t* row0 = wring + (size_t)cst * kWarpStage + lane * DI;
    const uint8_t* row1 = row0 + 32 * DI;
    int acc0[HI], acc1[HI];
#pragma unroll
    for (int h = 0; h < HI; ++h) acc0[h] = acc1[h] = 0;
#pragma unroll
    for (int cc = 0; cc < CH; ++cc) {
      const int4 k0 = *reinterpret_cast<const int4*>(row0 + ((cc ^ swz) << 4));
      const int4 k1 = *reinterpret_cast<const int4*>(row1 + ((cc ^ swz) << 4));
#pragma unroll
      for (int h = 0; h < HI; ++h) {
        int4 qv;
        if constexpr (kQInRegs) qv = q[h][cc];
        else qv = s_q[h * CH + cc];
        acc0[h] = __dp4a(k0.x, qv.x, acc0[h]);
        acc1[h] = __dp4a(k1.x, qv.x, acc1[h]);
        acc0[h] = __dp4a(k0.y, qv.y, acc0[h]);
        acc1[h] = __dp4a(k1.y, qv.y, acc1[h]);
        acc0[h] = __dp4a(k0.z, qv.z, acc0[h]);
        acc1[h] = __dp4a(k1.z, qv.z, acc1[h]);
        acc0[h] = __dp4a(k0.w, qv.w, acc0[h]);
        acc1[h] = __dp4a(k1.w, qv.w, acc1[h]);
      }
    }
    int s0 = 0, s1 = 0;
#pragma unroll
    for (int h = 0; h < HI; ++h) {
      s0 += w[h] * max(acc0[h], 0);
      s1 += w[h] * max(acc1[h], 0);
    }
    cst = cst + 1 == kStages ? 0 : cst + 1;
    par ^= cst == 0 ? 1u : 0u;

    const int t0 = (item - cb_first) * kTmaRound + warp * kWarpTokens + lane;
    const bool v0 = t0 < cb_len && !dead, v1 = t0 + 32 < cb_len && !dead;
    int32_t* srow = scores + (int64_t)cb * ld;
    if (v0) srow[t0] = s0;
    if (v1) srow[t0 + 32] = s1;
    if (do_hist) {
      const unsigned m0 = __ballot_sync(0xffffffffu, v0);
      if (v0) {
        const int bin = score_bin(s0);
        const unsigned peers = __match_any_sync(m0, bin);
        if (lane == __ffs(peers) - 1) atomicAdd(&s_hist[bin], __popc(peers));
      }
      const unsigned m1 = __ballot_sync(0xffffffffu, v1);
      if (v1) {
        const int bin = score_bin(s1);
        const unsigned peers = __match_any_sync(m1, bin);
        if (lane == __ffs(peers) - 1) atomicAdd(&s_hist[bin], __popc(peers));
      }
    }
    __syncwarp();
  }
  if (dead) {
    // let this warp's copies still in flight land before the CTA exits
    for (int st = 0; st < kStages; ++st) (void)mbar_wait(bar0 + 8u * st, 0);
  }
  if (do_hist) {
    __syncthreads();
    int32_t* gh = hist + (int64_t)cb * kScoreBins;
    for (int i = tid; i < kScoreBins; i += kTmaThreads) {
      const int cnt = s_hist[i];
      if (cnt) atomicAdd(gh + i, cnt);
    }
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// Tensor map over the key pool viewed as [num_pages * page_size rows, Di bytes].
bool make_key_map(const pks_decode_args& a, CUtensorMap* map) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)a.Di, (cuuint64_t)a.num_pages * a.page_size};
  const cuuint64_t strides[1] = {(cuuint64_t)a.Di};
  const cuuint32_t box[2] = {(cuuint32_t)a.Di,
                             (cuuint32_t)(a.page_size < kWarpTokens ? a.page_size : kWarpTokens)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(a.idx_k), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            a.Di == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Raise a kernel's dynamic shared-memory limit once per device to the
// largest size seen.  `configured` must belong to that one kernel.  Not a
// stream operation, so after the first call it stays out of graph capture.
template <typename K>
cudaError_t raise_smem(K kern, size_t smem, size_t (&configured)[64]) {
  int dev = 0;
  cudaGetDevice(&dev);
  size_t& done = configured[dev & 63];
  if (smem > done) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    done = smem;
  }
  return cudaSuccess;
}

template <int HI, int DI>
cudaError_t launch_scan_t(const pks_decode_args& a, int32_t* scores, int64_t ld, int32_t* hist,
                          int32_t* err, cudaStream_t s) {
  int shift = -1;
  if ((a.page_size & (a.page_size - 1)) == 0) {
    shift = 0;
    while ((1 << shift) < a.page_size) ++shift;
  }
  static size_t configured[64] = {0};  // per instantiation
  // 4 or 8 heads: int8 MMA; 1 or 2 heads: dp4a
  constexpr int kMmaThreads = 1024;
  auto kern = HI >= 4 ? k_indexer_scan_mma<(HI >= 4 ? HI : 4), DI, kMmaThreads>
                      : k_indexer_scan_reg<HI, DI>;
  const int threads = HI >= 4 ? kMmaThreads : kRegThreads;
  const size_t smem = sizeof(int) * ((size_t)kScoreBins + a.B + 1);
  cudaError_t e = raise_smem(kern, smem, configured);
  if (e != cudaSuccess) return e;
  kern<<<device_sm_count(), threads, smem, s>>>(a.seq_lens, a.block_table, a.q_idx, a.w_idx,
                                                    a.idx_k, scores, ld, hist, err, a.B,
                                                    a.max_pages, a.page_size, shift, a.num_pages,
                                                    a.k);
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
