// Indexer scan: int8 lightning-indexer scores of every cached token, with the
// per-request score histogram that seeds the top-k radix select fused in.
//
// "Sparse Attention on GLM5.3 and HBM", DeepSeek Sparse Attention paragraph:
// the indexer query is multi-headed, the key single-headed; a token's score is
// the weighted sum over query heads of ReLU(query . key).  The introduction
// notes that selection needs the whole context resident in HBM: this kernel
// streams every indexer key once and is bound by HBM bandwidth.
//
// Work split: the tokens of all requests are cut into CTA rounds of 1024
// tokens of one request; a persistent grid (one 1024-thread CTA per SM) gives
// each CTA a contiguous range of rounds.  Keys stream from HBM straight into
// registers with coalesced 16-byte loads (no shared-memory staging: on GB300
// register loads with 32 warps an SM reach a higher read bandwidth than
// cp.async or TMA fills of shared memory); the head dot products are int8
// tensor-core MMAs for any number of heads up to 8.  Each score is binned into
// the request's shared-memory histogram, which is added to the global one when
// the CTA leaves the request (it seeds the top-k selection).

#include "pks_internal.h"

namespace pks {
namespace {

__device__ __forceinline__ int score_bin(int s) {
  if (s == 0) return kScoreBins / 2;
  const unsigned a = s > 0 ? (unsigned)s : 0u - (unsigned)s;
  const int e = 31 - __clz(a);
  const unsigned m = e >= 5 ? (a >> (e - 5)) & 31u : (a << (5 - e)) & 31u;
  const int v = e * 32 + (int)m;  // 0 .. 1023
  return s > 0 ? kScoreBins / 2 + 1 + v : kScoreBins / 2 - 1 - v;
}

// Real-valued head weights: the fp32 score is stored as an int32 key with the
// same order (negative scores have their magnitude bits flipped; -0 becomes
// +0 first, so equal scores give equal keys).
__device__ __forceinline__ int float_key(float f) {
  const int b = __float_as_int(__fadd_rn(f, 0.f));
  return b >= 0 ? b : b ^ 0x7fffffff;
}
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

// Score store with an L2 evict-last policy: the top-k reads the scores right
// after the scan, while the keys stream through L2 with evict-first loads.
__device__ __forceinline__ void store_score_keep(int32_t* p, int v) {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;\n" : "=l"(pol));
  asm volatile("st.global.L2::cache_hint.s32 [%0], %1, %2;\n" ::"l"(p), "r"(v), "l"(pol) : "memory");
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

// ---------------------------------------------------------------------------
// The head dot products of 16 tokens are one int8 MMA tile per 32 key bytes:
// m16n8k32 with the tokens as M, the (zero-padded to 8) heads as N and the key
// bytes as K, int32 accumulate - exact, like dp4a, but the cross-lane sum
// happens inside the tensor core, so a 32-token round costs 8 MMAs instead of
// ~100 dp4a and shuffles per lane, whatever the number of heads.  Keys stream
// from HBM straight into the A fragments: lane
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

// FP8 (e4m3) queries and keys: D = A.B + C with fp32 accumulation
__device__ __forceinline__ void fmma_e4m3_16832(float (&c)[4], int a0, int a1, int a2, int a3,
                                                int b0, int b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// FW: real-valued head weights w_f [B * NQ, HI] instead of the integer w_idx
// [HI]; the score of a (token, query) is then the fp32 sum over the heads in
// order of w * ReLU(dot), each product and sum rounded to nearest.
// F8 (with FW): q_idx and idx_k hold FP8 e4m3 values; each head's dot product
// comes from the tensor core in fp32 (its accumulation order is the
// hardware's), the weighted sum over heads as for FW.
template <int HI, int DI, int NT, int NQ, bool FW, bool F8 = false>
__global__ void __launch_bounds__(NT, 1)
k_indexer_scan_mma(const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ block_table,
                   const int8_t* __restrict__ q_idx, const int32_t* __restrict__ w_idx,
                   const float* __restrict__ w_f,
                   const int8_t* __restrict__ idx_k, int32_t* __restrict__ scores, int64_t ld,
                   int32_t* __restrict__ hist, int32_t* __restrict__ err, int B, int max_pages,
                   int page_size, int page_shift, int num_pages, int k) {
  static_assert(HI * NQ <= 8, "N = 8 query heads per MMA");
  constexpr int HALVES = DI / 64;      // 64-byte halves of a key (2 or 1)
  constexpr int NLD = 2 * 2 * HALVES;  // loads per lane per 32-token round

  extern __shared__ int smem_i[];
  // the top-k grid may take SM slots as soon as this grid's CTAs retire
  pdl_launch_dependents();
  // launched with programmatic serialization: inputs staged by the kernel
  // before this one (if any) are visible after the wait
  pdl_wait();
  int* s_hist = smem_i;                      // [NQ][kScoreBins]
  int* s_prefix = smem_i + NQ * kScoreBins;  // [B + 1]
  // NQ > 1 or FW: (weighted) ReLU of each (token, query head) of a warp's round
  constexpr bool kTile = NQ > 1 || FW;
  __shared__ int s_ep[kTile ? NT / 32 : 1][32][8];
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
  for (int i = tid; i < NQ * kScoreBins; i += NT) s_hist[i] = 0;
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

  // page lookups run two rounds ahead of the loads that use them
  int pg0, sl0, pg1, sl1;  // lookups of the next two rounds to load
  int next_lookup = begin;
  pg0 = lookup(next_lookup, sl0);
  ++next_lookup;
  pg1 = next_lookup < end ? lookup(next_lookup, sl1) : (sl1 = -1, -1);
  ++next_lookup;
  // row of this lane's token in the next round to load
  auto next_row = [&]() -> int {
    const int row = to_row(pg0, sl0);
    int sl2 = -1;
    const int pg2 = next_lookup < end ? lookup(next_lookup, sl2) : -1;
    ++next_lookup;
    pg0 = pg1;
    sl0 = sl1;
    pg1 = pg2;
    sl1 = sl2;
    return row;
  };

  // query head n of the MMA's N = 8 columns: query n / HI, indexer head n % HI
  int4 qf[HALVES];  // chunks 4*hv + tq of query head gq (zero for padding)
  int w0 = 0, w1 = 0;  // weights of query heads 2tq and 2tq+1
  float wf[FW ? HI * NQ : 1];  // FW: the request's real weights, query-major
  int cb = -1, cb_len = 0, cb_first = 0, cb_next = 0;
  bool do_hist = false;
  // output token of this lane: tile (tq >> 1), row gq + 8 * (tq & 1)
  const int my_tok = (tq >> 1) * 16 + gq + 8 * (tq & 1);
  // scores of round `item` from its keys in buf
  auto process = [&](int item, const int4 (&buf)[NLD]) {
    if (item >= cb_next) {
      int b = cb < 0 ? lo : cb;
      while (s_prefix[b + 1] <= item) ++b;
      if (do_hist) {
        __syncthreads();
        // request cb's queries are virtual requests cb * NQ .. cb * NQ + NQ - 1
        int32_t* gh = hist + (int64_t)cb * NQ * kScoreBins;
        for (int i = tid; i < NQ * kScoreBins; i += NT) {
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
      // q_idx is [B, NQ, HI, DI]: query head n of request b is row b * NQ * HI + n
#pragma unroll
      for (int hv = 0; hv < HALVES; ++hv)
        qf[hv] = gq < HI * NQ
                     ? __ldg(reinterpret_cast<const int4*>(q_idx + ((int64_t)b * NQ * HI + gq) * DI) +
                             4 * hv + tq)
                     : make_int4(0, 0, 0, 0);
      if constexpr (FW) {
        w0 = w1 = 1;  // the tile keeps the plain ReLU; the real weights come after
#pragma unroll
        for (int i = 0; i < HI * NQ; ++i) wf[i] = __ldg(w_f + (int64_t)b * NQ * HI + i);
      } else {
        w0 = 2 * tq < HI * NQ ? __ldg(w_idx + (2 * tq) % HI) : 0;
        w1 = 2 * tq + 1 < HI * NQ ? __ldg(w_idx + (2 * tq + 1) % HI) : 0;
      }
    }

    if constexpr (kTile) {
      // weighted ReLU of every (token, query head) into the warp's tile; then
      // lane L sums the HI heads of each query for token L of the round
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        if constexpr (F8) {
          // fp32 ReLU of each head's dot product, kept as bits in the tile
          float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int hv = 0; hv < HALVES; ++hv) {
            const int4 r0 = buf[(u * HALVES + hv) * 2 + 0];
            const int4 r1 = buf[(u * HALVES + hv) * 2 + 1];
            fmma_e4m3_16832(c, r0.x, r1.x, r0.y, r1.y, qf[hv].x, qf[hv].y);
            fmma_e4m3_16832(c, r0.z, r1.z, r0.w, r1.w, qf[hv].z, qf[hv].w);
          }
          s_ep[warp][u * 16 + gq][2 * tq] = __float_as_int(fmaxf(c[0], 0.f));
          s_ep[warp][u * 16 + gq][2 * tq + 1] = __float_as_int(fmaxf(c[1], 0.f));
          s_ep[warp][u * 16 + gq + 8][2 * tq] = __float_as_int(fmaxf(c[2], 0.f));
          s_ep[warp][u * 16 + gq + 8][2 * tq + 1] = __float_as_int(fmaxf(c[3], 0.f));
        } else {
          int c[4] = {0, 0, 0, 0};
#pragma unroll
          for (int hv = 0; hv < HALVES; ++hv) {
            const int4 r0 = buf[(u * HALVES + hv) * 2 + 0];
            const int4 r1 = buf[(u * HALVES + hv) * 2 + 1];
            imma_16832<DI>(c, r0.x, r1.x, r0.y, r1.y, qf[hv].x, qf[hv].y);
            imma_16832<DI>(c, r0.z, r1.z, r0.w, r1.w, qf[hv].z, qf[hv].w);
          }
          s_ep[warp][u * 16 + gq][2 * tq] = w0 * max(c[0], 0);
          s_ep[warp][u * 16 + gq][2 * tq + 1] = w1 * max(c[1], 0);
          s_ep[warp][u * 16 + gq + 8][2 * tq] = w0 * max(c[2], 0);
          s_ep[warp][u * 16 + gq + 8][2 * tq + 1] = w1 * max(c[3], 0);
        }
      }
      __syncwarp();
      const int t = (item - cb_first) * NT + warp * 32 + lane;
      const bool valid = t < cb_len;
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        int score = 0;
        if constexpr (FW) {
          float sf = 0.f;
#pragma unroll
          for (int h = 0; h < HI; ++h) {
            const int r = s_ep[warp][lane][q * HI + h];
            sf = __fadd_rn(sf, __fmul_rn(wf[q * HI + h], F8 ? __int_as_float(r) : (float)r));
          }
          score = float_key(sf);
        } else {
#pragma unroll
          for (int h = 0; h < HI; ++h) score += s_ep[warp][lane][q * HI + h];
        }
        if (valid) store_score_keep(scores + ((int64_t)cb * NQ + q) * ld + t, score);
        if (do_hist && valid)
          atomicAdd(&s_hist[q * kScoreBins + (FW ? key_bin(score) : score_bin(score))], 1);
      }
      __syncwarp();  // the tile is rewritten next round
      return;
    }
    int sc[2][2];  // [tile][row g / g+8]
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      int c[4] = {0, 0, 0, 0};
#pragma unroll
      for (int hv = 0; hv < HALVES; ++hv) {
        const int4 r0 = buf[(u * HALVES + hv) * 2 + 0];  // token row gq
        const int4 r1 = buf[(u * HALVES + hv) * 2 + 1];  // token row gq + 8
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
    if (valid) store_score_keep(scores + (int64_t)cb * ld + t, score);
    // plain shared atomics: colliding lanes of a warp are serialised by the
    // hardware, which costs less than aggregating them first
    if (do_hist && valid) atomicAdd(&s_hist[score_bin(score)], 1);
  };

  // single-buffered: the other warps of the SM overlap a warp's load latency
  // (double-buffering the key registers measured slower on GB300)
  int4 cur[NLD];
  for (int item = begin; item < end; ++item) {
    load_round(next_row(), cur);
    process(item, cur);
  }
  if (do_hist) {
    __syncthreads();
    int32_t* gh = hist + (int64_t)cb * NQ * kScoreBins;
    for (int i = tid; i < NQ * kScoreBins; i += NT) {
      const int cnt = s_hist[i];
      if (cnt) atomicAdd(gh + i, cnt);
    }
  }
}

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

// threads a CTA (one CTA an SM)
constexpr int kMmaThreads = 1024;

template <int HI, int DI, int NQ, bool FW = false, bool F8 = false>
cudaError_t launch_scan_t(const pks_decode_args& a, int32_t* scores, int64_t ld, int32_t* hist,
                          int32_t* err, cudaStream_t s) {
  int shift = -1;
  if ((a.page_size & (a.page_size - 1)) == 0) {
    shift = 0;
    while ((1 << shift) < a.page_size) ++shift;
  }
  static size_t configured[64] = {0};  // per instantiation
  const size_t smem = sizeof(int) * ((size_t)NQ * kScoreBins + a.B + 1);
  auto kern = k_indexer_scan_mma<HI, DI, kMmaThreads, NQ, FW, F8>;
  cudaError_t e = raise_smem(kern, smem, configured);
  if (e != cudaSuccess) return e;
  return launch_ex(kern, dim3(device_sm_count()), dim3(kMmaThreads), smem, s, /*pdl=*/true,
                   /*coop=*/false, a.seq_lens, a.block_table, a.q_idx, a.w_idx, a.w_idx_f, a.idx_k,
                   scores, ld, hist, err, a.B, a.max_pages, a.page_size, shift, a.num_pages, a.k);
}

}  // namespace

cudaError_t launch_indexer_scan(const pks_decode_args& a, int32_t* scores, int64_t ld,
                                int32_t* hist, int32_t* err, cudaStream_t s) {
  const int nq = query_count(a);
  if (a.w_idx_f && a.idx_fp8) {  // FP8 e4m3 queries and keys, real weights
#define PKS_SCAN_F8(HI_, DI_) \
  if (a.Hi == HI_ && a.Di == DI_)  \
    return launch_scan_t<HI_, DI_, 1, true, true>(a, scores, ld, hist, err, s);
    PKS_SCAN_F8(1, 64)
    PKS_SCAN_F8(2, 64)
    PKS_SCAN_F8(4, 64)
    PKS_SCAN_F8(8, 64)
    PKS_SCAN_F8(1, 128)
    PKS_SCAN_F8(2, 128)
    PKS_SCAN_F8(4, 128)
    PKS_SCAN_F8(8, 128)
#undef PKS_SCAN_F8
    return cudaErrorInvalidValue;
  }
  if (a.w_idx_f) {  // real-valued head weights: one query token per request
#define PKS_SCAN_FW(HI_, DI_) \
  if (a.Hi == HI_ && a.Di == DI_) return launch_scan_t<HI_, DI_, 1, true>(a, scores, ld, hist, err, s);
    PKS_SCAN_FW(1, 64)
    PKS_SCAN_FW(2, 64)
    PKS_SCAN_FW(4, 64)
    PKS_SCAN_FW(8, 64)
    PKS_SCAN_FW(1, 128)
    PKS_SCAN_FW(2, 128)
    PKS_SCAN_FW(4, 128)
    PKS_SCAN_FW(8, 128)
#undef PKS_SCAN_FW
    return cudaErrorInvalidValue;
  }
#define PKS_SCAN_CASE(HI_, DI_, NQ_)                       \
  if (a.Hi == HI_ && a.Di == DI_ && nq == NQ_)             \
    return launch_scan_t<HI_, DI_, NQ_>(a, scores, ld, hist, err, s);
  PKS_SCAN_CASE(1, 64, 1)
  PKS_SCAN_CASE(2, 64, 1)
  PKS_SCAN_CASE(4, 64, 1)
  PKS_SCAN_CASE(8, 64, 1)
  PKS_SCAN_CASE(1, 128, 1)
  PKS_SCAN_CASE(2, 128, 1)
  PKS_SCAN_CASE(4, 128, 1)
  PKS_SCAN_CASE(8, 128, 1)
  // several query tokens per request (Hi * Nq <= 8)
  PKS_SCAN_CASE(1, 64, 2)
  PKS_SCAN_CASE(1, 64, 4)
  PKS_SCAN_CASE(1, 64, 8)
  PKS_SCAN_CASE(2, 64, 2)
  PKS_SCAN_CASE(2, 64, 4)
  PKS_SCAN_CASE(4, 64, 2)
  PKS_SCAN_CASE(1, 128, 2)
  PKS_SCAN_CASE(1, 128, 4)
  PKS_SCAN_CASE(1, 128, 8)
  PKS_SCAN_CASE(2, 128, 2)
  PKS_SCAN_CASE(2, 128, 4)
  PKS_SCAN_CASE(4, 128, 2)
#undef PKS_SCAN_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pks
