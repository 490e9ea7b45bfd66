// Sparse scaled dot-product attention over the selected tokens, split-K.
//
// "Sparse Attention on GLM5.3 and HBM", introduction: attention runs over
// only the top-k tokens, which cuts the bytes SDPA reads; "Paged KV cache",
// "Paging" and "What this table does not say": K/V are found through the
// page table, so the reads are scattered rows that the kernel must gather
// efficiently.
//
// Persistent stream-K over the flattened (KV-head group, request, selected
// position) space: every CTA (one per SM) takes an equal contiguous range of
// it.  A CTA first turns its positions into physical token rows (block table
// lookup, bounds checked), then streams 16-token tiles of K and V rows for
// its head group (HG heads x D x 2 bytes, contiguous) with 16-byte cp.async
// into a 3-stage shared-memory ring; rows are stored XOR-swizzled by 16-byte
// chunk so that ldmatrix reads are free of bank conflicts.  Each warp owns one
// KV head and keeps an online-softmax state for the G query heads that share
// it.  Both products run transposed on the tensor cores (bf16 in, fp32
// accumulate), with the G heads as the 8-wide N dimension of m16n8k16 (one
// column tile for G <= 8, two for G <= 16): S^T = K Q^T takes the 16 tokens
// of a tile as M, and O^T += V^T P^T the head dimension as M, so no MMA
// carries padding rows and O^T needs D / 4 accumulators a thread per column
// tile.  P^T moves from the accumulator layout of S^T to the B-operand layout
// with one movmatrix transpose per 8x8 block.  A CTA that owns a whole
// (group, request) segment writes its bf16 output; otherwise it writes a
// partial (m, l, o) to a slot indexed by (CTA + segment), and
// k_attention_merge combines the partials of each split segment by
// log-sum-exp rescaling.
//
// At G = 8 query heads per KV head the work is about 8 FLOP per byte of K/V,
// far below the tensor-core ridge: the MMAs only keep the arithmetic off the
// critical path.  What bounds the kernel is the rate at which an SM streams
// gathered rows through the ring (a 64 KB tile about every 1.5 us, 6.3 TB/s
// over 152 SMs, measured), so the compute between a tile's arrival and its
// release is kept short.

#include <cuda_bf16.h>

#include "pks_internal.h"

namespace pks {
namespace {

constexpr int kAttnStages = 3;      // shared-memory ring depth in tiles
constexpr int kAttnRowCap = 2048;   // positions whose rows are resolved at once

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// transpose of an 8x8 bf16 matrix held one pair a thread in the mma layout
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
  return y;
}

// D += A(16x16, row) * B(16x8, col), bf16 inputs, fp32 accumulators
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void flag_error(int32_t* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// Decode flattened position f (head group major, then request, then top-k
// position) of a CTA's range into its segment (group, request) and position.
struct SegCursor {
  int g, b, p;      // head group, request, position within the request's list
  int seg_end;      // flattened end of the current segment
};

__device__ __forceinline__ int64_t lmin(int64_t a, int64_t b) { return a < b ? a : b; }

// CTAs that take part for T positions: at most the grid and T, and with an
// automatic grid (min_per_cta > 0) at most one per min_per_cta positions, so
// that small steps are not cut into one-position pieces.
__device__ __forceinline__ int64_t attn_effective_grid(int64_t T, int64_t grid, int min_per_cta) {
  int64_t g = T < grid ? T : grid;
  if (min_per_cta > 0) {
    const int64_t cap = (T + min_per_cta - 1) / min_per_cta;
    if (cap < g) g = cap;
  }
  return g < 1 ? 1 : g;
}

// With an automatic grid, every segment (head group, request) of the same
// size and at least four CTAs a segment, round the grid down to a whole number of
// CTAs per segment when that keeps three quarters of it: no CTA then straddles
// two segments.  (Measured: 16 segments of 2048 positions take 2 us less on
// 144 or 128 CTAs than on 152 or 136; with 2.4 CTAs a segment the lost CTAs
// cost more than the straddles.)
__device__ __forceinline__ int64_t attn_aligned_grid(int64_t g, int64_t nseg, bool uniform,
                                                     int min_per_cta) {
  if (min_per_cta <= 0 || !uniform || nseg <= 0 || g < 4 * nseg) return g;
  const int64_t a = (g / nseg) * nseg;
  return 4 * a >= 3 * g ? a : g;
}

// CTA that owns flattened position f when [0, T) is cut into G equal ranges.
__device__ __forceinline__ int owner_cta(int64_t f, int64_t T, int64_t G) {
  return (int)(((f + 1) * G + T - 1) / T - 1);
}

// RES: K/V through a residency table (slot pools plus the host pool); the
// plain instantiation keeps the host-row select out of the copy loop.
template <int D, int HG, bool RES, int NGT>
__global__ void __launch_bounds__(HG * 32, 1)
k_sparse_attention(const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ block_table,
                   const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kv_k,
                   const __nv_bfloat16* __restrict__ kv_v, const int32_t* __restrict__ topk,
                   int32_t* __restrict__ prefix_out, float2* __restrict__ part_ml,
                   float* __restrict__ part_o, __nv_bfloat16* __restrict__ out,
                   int32_t* __restrict__ err, int B, int Hq, int Hkv, int G, int page_size,
                   int max_pages, int num_pages, int k, int trim, int min_per_cta,
                   float scale_log2, ResidentKv rk, int nq) {
  constexpr int NT = HG * 32;
  constexpr int CH = D / 8;   // 16-byte chunks per head row
  constexpr int KS = D / 16;  // k-steps of S^T = K Q^T
  constexpr int MT = D / 16;  // 16-row tiles of O^T (head dimension)
  constexpr int TILE = kAttnTile;
  constexpr int STAGE_ELEMS = TILE * HG * D;  // one of K or V
  const float kNegInf = __int_as_float(0xff800000);

  extern __shared__ __align__(128) uint8_t smem[];
  __nv_bfloat16* s_kv = reinterpret_cast<__nv_bfloat16*>(smem);  // [stages][K|V][TILE][HG][D]
  int32_t* s_row = reinterpret_cast<int32_t*>(smem + (size_t)kAttnStages * 2 * STAGE_ELEMS * 2);
  int32_t* s_prefix = s_row + kAttnRowCap;  // [B + 1] top-k positions per request, prefix
  __shared__ int s_warp[NT / 32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int max_len = max_pages * page_size;
  const int ngroups = Hkv / HG;

  // ---- prefix over requests of the positions to visit: k_b = min(k, len_b)
  // when the list is the step's own top-k (selected entries first, -1 after),
  // else all k positions (entries may sit anywhere)
  {
    const int per = (B + NT - 1) / NT;
    int local = 0;
    for (int i = 0; i < per; ++i) {
      const int b = tid * per + i;
      if (b < B) {
        const int len = seq_lens[b / nq];  // b: virtual request
        local += (len < 0 || len > max_len) ? 0 : (trim ? min(len, k) : k);
      }
    }
    int x = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    int before = x - local;
    for (int w = 0; w < warp; ++w) before += s_warp[w];
    for (int i = 0; i < per; ++i) {
      const int b = tid * per + i;
      if (b < B) {
        s_prefix[b] = before;
        const int len = seq_lens[b / nq];  // b: virtual request
        before += (len < 0 || len > max_len) ? 0 : (trim ? min(len, k) : k);
      }
    }
    if (tid == NT - 1) s_prefix[B] = before;
    __syncthreads();
  }
  // the merge grid may take the SM slots this grid leaves free
  pdl_launch_dependents();
  pdl_wait();  // the selection comes from the top-k kernel
  const int64_t Treq = s_prefix[B];
  const int64_t T = Treq * ngroups;
  // with fewer positions than CTAs only the first T CTAs take part, so every
  // participating CTA owns at least one position and the contributors of a
  // segment are exactly the CTAs from its first to its last owner
  // every request visits exactly k positions when the total is B * k (no
  // request visits more), so all segments have the same size
  const int64_t GRID = attn_aligned_grid(attn_effective_grid(T, gridDim.x, min_per_cta),
                                         (int64_t)ngroups * B, Treq == (int64_t)B * k, min_per_cta);
  const int cta = blockIdx.x;

  // requests with no position to visit (length 0) get zero outputs; CTA 0
  // also publishes the position prefix and the grid for the merge kernel
  if (cta == 0) {
    for (int i = tid; i <= B; i += NT) prefix_out[i] = s_prefix[i];
    if (tid == 0) prefix_out[B + 1] = (int32_t)GRID;
    // a thread a request finds the empty ones; the CTA zeroes them together
    // (normally there are none, and the check costs one barrier per NT requests)
    for (int b0 = 0; b0 < B; b0 += NT) {
      const int b = b0 + tid;
      if (!__syncthreads_or(b < B && s_prefix[b + 1] == s_prefix[b])) continue;
      for (int bb = b0; bb < B && bb < b0 + NT; ++bb) {
        if (s_prefix[bb + 1] != s_prefix[bb]) continue;
        for (int i = tid; i < Hq * D; i += NT) out[(int64_t)bb * Hq * D + i] = __float2bfloat16(0.f);
      }
    }
  }
  if (T == 0 || cta >= GRID) return;
  const int64_t lo = cta * T / GRID, hi = (cta + 1) * T / GRID;
  if (lo >= hi) return;

  auto locate = [&](int64_t f) {
    SegCursor c;
    c.g = (int)(f / Treq);
    const int fb = (int)(f - (int64_t)c.g * Treq);
    int l = 0, h = B - 1;  // last request with prefix <= fb
    while (l < h) {
      const int mid = (l + h + 1) >> 1;
      if (s_prefix[mid] <= fb) l = mid; else h = mid - 1;
    }
    c.b = l;
    c.p = fb - s_prefix[l];
    c.seg_end = (int)((int64_t)c.g * Treq + s_prefix[l + 1]);
    return c;
  };

  // mma fragment coordinates: g8 = lane / 4 (row group), t4 = lane % 4;
  // column tile nt covers query heads nt * 8 + 2 * t4 + {0, 1} of the group
  const int g8 = lane >> 2, t4 = lane & 3;
  uint32_t qb[NGT][KS][2];   // Q^T as the B operand (dims x heads)
  float o[NGT][MT][4];       // O^T accumulators (dims x heads)
  float m_h[NGT][2], l_h[NGT][2];  // running max (log2 units) and partial sum per head
  auto reset_state = [&]() {
#pragma unroll
    for (int nt = 0; nt < NGT; ++nt) {
#pragma unroll
      for (int i = 0; i < MT; ++i) o[nt][i][0] = o[nt][i][1] = o[nt][i][2] = o[nt][i][3] = 0.f;
      m_h[nt][0] = m_h[nt][1] = kNegInf;
      l_h[nt][0] = l_h[nt][1] = 0.f;
    }
  };
  auto load_q = [&](int g, int b) {
    const int head = g * HG + warp;  // this warp's KV head
    const __nv_bfloat16* qb0 = q + ((int64_t)b * Hq + (int64_t)head * G) * D;
#pragma unroll
    for (int nt = 0; nt < NGT; ++nt) {
      const int j = nt * 8 + g8;  // query head of the group (B column)
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const __nv_bfloat16* src = qb0 + (int64_t)j * D + ks * 16 + t4 * 2;
        qb[nt][ks][0] = j < G ? *reinterpret_cast<const uint32_t*>(src) : 0u;
        qb[nt][ks][1] = j < G ? *reinterpret_cast<const uint32_t*>(src + 8) : 0u;
      }
    }
  };

  // write this CTA's share of segment (g, b): the whole output when it owns
  // the whole segment, else a partial (m, l, o) that k_attention_merge combines
  auto finish_segment = [&](int g, int b, int64_t seg_lo, int64_t seg_hi) {
    float l_t[NGT][2];
#pragma unroll
    for (int nt = 0; nt < NGT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float l = l_h[nt][e];  // sum over the 16 token rows: lanes of equal t4
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        l_t[nt][e] = l;
      }
    const int head = g * HG + warp;
    const int c_first = owner_cta(seg_lo, T, GRID), c_last = owner_cta(seg_hi - 1, T, GRID);
    if (c_first == c_last) {
      __nv_bfloat16* ob = out + ((int64_t)b * Hq + (int64_t)head * G) * D;
#pragma unroll
      for (int nt = 0; nt < NGT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int j = nt * 8 + 2 * t4 + e;
          if (j >= G) continue;
          const float il = l_t[nt][e] > 0.f ? 1.f / l_t[nt][e] : 0.f;
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            ob[(int64_t)j * D + mt * 16 + g8] = __float2bfloat16(o[nt][mt][e] * il);
            ob[(int64_t)j * D + mt * 16 + g8 + 8] = __float2bfloat16(o[nt][mt][e + 2] * il);
          }
        }
      return;
    }
    const int seg = g * B + b;
    const int64_t slot = (int64_t)cta + seg;
    const int64_t base = (slot * HG + warp) * G;
#pragma unroll
    for (int nt = 0; nt < NGT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int j = nt * 8 + 2 * t4 + e;
        if (j >= G) continue;
        float* po = part_o + (base + j) * D;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          po[mt * 16 + g8] = o[nt][mt][e];
          po[mt * 16 + g8 + 8] = o[nt][mt][e + 2];
        }
        if (g8 == 0) part_ml[base + j] = make_float2(m_h[nt][e], l_t[nt][e]);
      }
  };

  // consumer cursor: segment whose state the warps hold
  int64_t cs_pos = lo;
  SegCursor csc{0, 0, 0, 0};
  bool have_state = false;
  for (int64_t chunk_lo = lo; chunk_lo < hi; chunk_lo += kAttnRowCap) {
    const int64_t chunk_hi = lmin(hi, chunk_lo + kAttnRowCap);
    // ---- physical token rows of the chunk's positions: those of the first
    // tiles first, so their copies start while the rest are looked up
    auto resolve_rows = [&](int64_t f0, int64_t f1) {
      for (int64_t f = f0 + tid; f < f1; f += NT) {
        const SegCursor c = locate(f);
        int len = seq_lens[c.b / nq];
        if (len < 0 || len > max_len) len = 0;
        const int t = topk[(int64_t)c.b * k + c.p];
        int row = -1;
        if (t >= 0) {
          if (t >= len) {
            flag_error(err, kErrToken);
          } else {
            const int page = block_table[(int64_t)(c.b / nq) * max_pages + t / page_size];
            if ((unsigned)page < (unsigned)num_pages) {
              row = page * page_size + t % page_size;
              if (RES) {
                // resident page: its slot's row; otherwise the host pool's
                // row, encoded as -(row) - 2 (-1 stays "no token")
                const int sl = rk.page_slot[page];
                row = (unsigned)sl < (unsigned)rk.capacity ? sl * page_size + t % page_size
                                                           : -row - 2;
              }
            }
            else flag_error(err, kErrPage);
          }
        }
        s_row[f - chunk_lo] = row;
      }
    };
    // the first pass takes one position a thread (at least the ring's first
    // tiles): as many rows resolve in one dependent round trip as in fewer
    constexpr int kFirstPass = NT > (kAttnStages - 1) * TILE ? NT : (kAttnStages - 1) * TILE;
    const int64_t early_hi = lmin(chunk_hi, chunk_lo + kFirstPass);
    resolve_rows(chunk_lo, early_hi);
    __syncthreads();

    // ---- tiles: runs of up to TILE positions inside one segment
    int64_t ld_pos = chunk_lo;  // flattened position of the next tile to load
    int ld_seg_end = locate(chunk_lo).seg_end;
    auto load_next = [&](int stage) {
      if (ld_pos >= chunk_hi) return;
      if (ld_pos >= ld_seg_end) ld_seg_end = locate(ld_pos).seg_end;
      const int n = (int)lmin(TILE, lmin(ld_seg_end, chunk_hi) - ld_pos);
      const int g = (int)(ld_pos / Treq);
      __nv_bfloat16* sk = s_kv + (size_t)stage * 2 * STAGE_ELEMS;
      __nv_bfloat16* sv = sk + STAGE_ELEMS;
      const int rbase = (int)(ld_pos - chunk_lo);
#pragma unroll 4
      for (int idx = tid; idx < TILE * HG * CH; idx += NT) {
        const int r = idx / (HG * CH), rem = idx % (HG * CH);
        const int hh = rem / CH, c = rem % CH;
        const int row = r < n ? s_row[rbase + r] : -1;
        const int off = (r * HG + hh) * D + ((c ^ (r & 7)) << 3);
        // row >= 0: kv_k / kv_v (the pool, or the resident slots); row <= -2:
        // the host pool's row -row - 2; -1: no token (zero fill)
        const bool host = RES && row < -1;
        const int64_t prow = host ? -(int64_t)row - 2 : (int64_t)row;
        const int64_t src = row != -1 ? (prow * Hkv + g * HG + hh) * D + c * 8 : 0;
        const int bytes = row != -1 ? 16 : 0;  // 0 bytes: zero fill
        if (RES) {
          cp_async16(smem_u32(sk + off), (host ? rk.host_k : kv_k) + src, bytes);
          cp_async16(smem_u32(sv + off), (host ? rk.host_v : kv_v) + src, bytes);
        } else {
          cp_async16(smem_u32(sk + off), kv_k + src, bytes);
          cp_async16(smem_u32(sv + off), kv_v + src, bytes);
        }
      }
      ld_pos += n;
    };

    int n_tiles = 0;
    {
      // count tiles of the chunk (uniform across the CTA)
      int64_t f = chunk_lo;
      int se = ld_seg_end;
      while (f < chunk_hi) {
        if (f >= se) se = locate(f).seg_end;
        f += lmin(TILE, lmin(se, chunk_hi) - f);
        ++n_tiles;
      }
    }
#pragma unroll
    for (int st = 0; st < kAttnStages - 1; ++st) {
      if (st < n_tiles) load_next(st);
      cp_async_commit();
    }
    resolve_rows(early_hi, chunk_hi);
    __syncthreads();
    for (int tile = 0; tile < n_tiles; ++tile) {
      if (tile + kAttnStages - 1 < n_tiles) load_next((tile + kAttnStages - 1) % kAttnStages);
      cp_async_commit();
      if (!have_state || cs_pos >= csc.seg_end) {
        csc = locate(cs_pos);
        load_q(csc.g, csc.b);
        reset_state();
        have_state = true;
      }
      const int n = (int)lmin(TILE, lmin(csc.seg_end, chunk_hi) - cs_pos);
      const int rbase = (int)(cs_pos - chunk_lo);
      cp_async_wait<kAttnStages - 1>();
      __syncthreads();

      const __nv_bfloat16* sk = s_kv + (size_t)(tile % kAttnStages) * 2 * STAGE_ELEMS;
      const __nv_bfloat16* sv = sk + STAGE_ELEMS;
      // S^T = K Q^T: 16 tokens (M) x 8 heads (N) per column tile, two
      // accumulator chains (even and odd k-steps) for latency
      float sacc[2][NGT][4];
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int nt = 0; nt < NGT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) sacc[c][nt][i] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const int row = (lane & 7) + (((lane >> 3) & 1) << 3);  // token
        const int chunk = 2 * ks + (lane >> 4);
        uint32_t a[4];
        ldsm_x4(smem_u32(sk + (row * HG + warp) * D + ((chunk ^ (row & 7)) << 3)), a[0], a[1],
                a[2], a[3]);
#pragma unroll
        for (int nt = 0; nt < NGT; ++nt)
          mma_bf16(sacc[ks & 1][nt], a, qb[nt][ks][0], qb[nt][ks][1]);
      }
      // rows g8 and g8 + 8 of the tile; masked tokens score -inf
      const bool v0 = g8 < n && s_row[rbase + g8] != -1;
      const bool v1 = g8 + 8 < n && s_row[rbase + g8 + 8] != -1;
      uint32_t pb[NGT][2];  // P^T as the B operand (tokens x heads)
#pragma unroll
      for (int nt = 0; nt < NGT; ++nt) {
        float x[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float sv_ = sacc[0][nt][i] + sacc[1][nt][i];
          x[i] = (i < 2 ? v0 : v1) ? sv_ * scale_log2 : kNegInf;
        }
        float al[2], p[4];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          // column max over the 16 tokens: own two rows, then lanes of equal t4
          float mx = fmaxf(x[e], x[e + 2]);
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float mn = fmaxf(m_h[nt][e], mx);
          al[e] = mn == kNegInf ? 1.f : exp2f(m_h[nt][e] - mn);
          p[e] = x[e] == kNegInf ? 0.f : exp2f(x[e] - mn);
          p[e + 2] = x[e + 2] == kNegInf ? 0.f : exp2f(x[e + 2] - mn);
          l_h[nt][e] = l_h[nt][e] * al[e] + (p[e] + p[e + 2]);
          m_h[nt][e] = mn;
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          o[nt][mt][0] *= al[0];
          o[nt][mt][1] *= al[1];
          o[nt][mt][2] *= al[0];
          o[nt][mt][3] *= al[1];
        }
        // (token g8, heads 2 t4 + {0,1}) -> (tokens 2 t4 + {0,1}, head g8)
        pb[nt][0] = movmatrix_t(pack_bf16(p[0], p[1]));
        pb[nt][1] = movmatrix_t(pack_bf16(p[2], p[3]));
      }
      // O^T += V^T P^T: 16 dims (M) x 8 heads (N), k = the 16 tokens
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const int row = (lane & 7) + ((lane >> 4) << 3);  // token
        const int chunk = 2 * mt + ((lane >> 3) & 1);
        uint32_t a[4];
        ldsm_x4_t(smem_u32(sv + (row * HG + warp) * D + ((chunk ^ (row & 7)) << 3)), a[0], a[1],
                  a[2], a[3]);
#pragma unroll
        for (int nt = 0; nt < NGT; ++nt) mma_bf16(o[nt][mt], a, pb[nt][0], pb[nt][1]);
      }
      __syncthreads();
      cs_pos += n;
      if (cs_pos == csc.seg_end || cs_pos == hi) {
        const int64_t seg_lo = (int64_t)csc.g * Treq + s_prefix[csc.b];
        finish_segment(csc.g, csc.b, seg_lo, csc.seg_end);
        have_state = false;
      }
    }
    cp_async_wait<0>();
    __syncthreads();
  }
}

// Combine the partial (m, l, o) of a segment's contributing CTAs: one warp per
// (query head, request); segments that one attention CTA owned whole are
// skipped (it wrote the output itself).  Two dependent L2 round trips: the
// position prefix, then every contributor's (m, l) (one lane each) together
// with the o rows of up to 16 contributors (lanes own float4 columns); more
// contributors take further batches.
template <int D>
__global__ void __launch_bounds__(128)
k_attention_merge(const int32_t* __restrict__ prefix, const float2* __restrict__ part_ml,
                  const float* __restrict__ part_o, __nv_bfloat16* __restrict__ out, int B,
                  int Hq, int Hkv, int HG, int G) {
  constexpr int DV4 = D / 4;  // float4 columns of a row (32 or 16)
  constexpr int kBatch = 16;  // contributors' o rows in flight per lane
  const float kNegInf = __int_as_float(0xff800000);
  const int lane = threadIdx.x & 31;
  const int qh = blockIdx.x * 4 + (threadIdx.x >> 5);  // query head
  const int b = blockIdx.y;
  pdl_launch_dependents();  // a following kernel may launch and wait for this grid
  pdl_wait();  // prefix and partials come from the attention kernel
  if (qh >= Hq) return;
  const int h = qh / G, gg = qh % G;  // KV head and row within its group
  const int g = h / HG, hh = h % HG;
  const int64_t Treq = prefix[B];
  const int p0 = prefix[b], p1 = prefix[b + 1];
  const int64_t T = Treq * (Hkv / HG);
  if (T == 0 || p1 == p0) return;
  const int64_t GRID = prefix[B + 1];  // CTAs that took part, as the attention kernel chose
  const int64_t seg_lo = (int64_t)g * Treq + p0;
  const int c_first = owner_cta(seg_lo, T, GRID), c_last = owner_cta(seg_lo + (p1 - p0) - 1, T, GRID);
  if (c_first == c_last) return;
  const int seg = g * B + b;
  const int64_t pstride = (int64_t)HG * G;
  auto pidx = [&](int c) { return ((int64_t)c + seg) * pstride + (int64_t)hh * G + gg; };
  const int nc = c_last - c_first + 1;

  // (m, l) of contributors lane, lane + 32, ... and the first batch of o rows
  float2 ml = nc > lane ? __ldcg(&part_ml[pidx(c_first + lane)]) : make_float2(kNegInf, 0.f);
  float4 v[kBatch];
#pragma unroll
  for (int u = 0; u < kBatch; ++u)
    v[u] = (u < nc && lane < DV4)
               ? __ldcg(reinterpret_cast<const float4*>(part_o + pidx(c_first + u) * D) + lane)
               : make_float4(0.f, 0.f, 0.f, 0.f);
  float M = ml.x;
  for (int c = c_first + 32 + lane; c <= c_last; c += 32) M = fmaxf(M, __ldcg(&part_ml[pidx(c)].x));
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float L = ml.x == kNegInf ? 0.f : ml.y * exp2f(ml.x - M);
  for (int c = c_first + 32 + lane; c <= c_last; c += 32) {
    const float2 e = __ldcg(&part_ml[pidx(c)]);
    if (e.x != kNegInf) L += e.y * exp2f(e.x - M);
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  const float il = L > 0.f ? 1.f / L : 0.f;
  // weight of contributor c_first + u (u < 32) from the lane holding its (m, l)
  const float f_mine = ml.x == kNegInf ? 0.f : exp2f(ml.x - M);

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int u = 0; u < kBatch; ++u) {
    const float f = __shfl_sync(0xffffffffu, f_mine, u);
    acc.x += f * v[u].x;
    acc.y += f * v[u].y;
    acc.z += f * v[u].z;
    acc.w += f * v[u].w;
  }
  for (int c0 = c_first + kBatch; c0 <= c_last; c0 += kBatch) {
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int c = c0 + u;
      v[u] = (c <= c_last && lane < DV4)
                 ? __ldcg(reinterpret_cast<const float4*>(part_o + pidx(c) * D) + lane)
                 : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int c = c0 + u;
      float m = kNegInf;
      if (c <= c_last) m = __ldcg(&part_ml[pidx(c)].x);
      const float f = m == kNegInf ? 0.f : exp2f(m - M);
      acc.x += f * v[u].x;
      acc.y += f * v[u].y;
      acc.z += f * v[u].z;
      acc.w += f * v[u].w;
    }
  }
  if (lane >= DV4) return;
  __nv_bfloat16* dst = out + ((int64_t)b * Hq + qh) * D + lane * 4;
  *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(acc.x * il, acc.y * il);
  *reinterpret_cast<__nv_bfloat162*>(dst + 2) = __floats2bfloat162_rn(acc.z * il, acc.w * il);
}

template <int D, int HG>
size_t attn_smem_bytes(int B) {
  return (size_t)kAttnStages * 2 * kAttnTile * HG * D * sizeof(__nv_bfloat16) +
         sizeof(int32_t) * (size_t)(kAttnRowCap + B + 1);
}

// Dynamic shared-memory limit of one attention instantiation on the current
// device, raised to `smem` when it is lower and never lowered, with the
// resident CTAs an SM it allows at that limit (cached with it).  Every
// launcher of the instantiation goes through here, so a call with a small
// batch cannot undo the limit that a larger one set.  Attribute calls are not
// stream operations: after the first call at a size they stay out of any
// graph capture.
template <int D, int HG, bool RES, int NGT>
cudaError_t attn_configure(size_t smem, int* blocks_per_sm) {
  static size_t configured[64] = {0};
  static int per_sm[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (smem > configured[dev]) {
    auto kern = k_sparse_attention<D, HG, RES, NGT>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int bps = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, kern, HG * 32, smem);
    if (e != cudaSuccess) return e;
    configured[dev] = smem;
    per_sm[dev] = bps < 1 ? 1 : bps;
  }
  *blocks_per_sm = per_sm[dev];
  return cudaSuccess;
}

template <int D, int HG, bool RES, int NGT>
cudaError_t launch_attn_t(const pks_decode_args& a, const WorkspaceLayout& L, uint8_t* ws,
                          bool trim, const ResidentKv& rk, cudaStream_t s) {
  auto kern = k_sparse_attention<D, HG, RES, NGT>;
  const int nq = query_count(a);
  const int Bv = a.B * nq;  // virtual requests
  const size_t smem = attn_smem_bytes<D, HG>(Bv);
  int bps = 1;
  {
    cudaError_t e = attn_configure<D, HG, RES, NGT>(smem, &bps);
    if (e != cudaSuccess) return e;
  }
  int grid = a.attn_splits > 0 ? a.attn_splits : device_sm_count() * bps;
  if (grid > L.attn_grid_max) grid = L.attn_grid_max;
  const int G = a.Hq / a.Hkv;
  const int min_per_cta = a.attn_splits > 0 ? 0 : kAttnMinPositions;
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)a.D);
  cudaError_t e = launch_ex(
      kern, dim3(grid), dim3(HG * 32), smem, s, /*pdl=*/true, /*coop=*/false, a.seq_lens,
      a.block_table, reinterpret_cast<const __nv_bfloat16*>(a.q),
      reinterpret_cast<const __nv_bfloat16*>(a.kv_k), reinterpret_cast<const __nv_bfloat16*>(a.kv_v),
      (const int32_t*)a.topk_idx, reinterpret_cast<int32_t*>(ws + L.attn_prefix),
      reinterpret_cast<float2*>(ws + L.part_ml), reinterpret_cast<float*>(ws + L.part_o),
      reinterpret_cast<__nv_bfloat16*>(a.out), reinterpret_cast<int32_t*>(ws + L.err), Bv, a.Hq,
      a.Hkv, G, a.page_size, a.max_pages, a.num_pages, a.k, trim ? 1 : 0, min_per_cta,
      scale_log2, rk, nq);
  if (e != cudaSuccess) return e;
  return launch_ex(k_attention_merge<D>, dim3((a.Hq + 3) / 4, Bv), dim3(128), 0, s, true, false,
                   reinterpret_cast<const int32_t*>(ws + L.attn_prefix),
                   reinterpret_cast<const float2*>(ws + L.part_ml),
                   reinterpret_cast<const float*>(ws + L.part_o),
                   reinterpret_cast<__nv_bfloat16*>(a.out), Bv, a.Hq, a.Hkv, (int)HG, G);
}

// ---- allocation-free variant: scratch in a fixed device array -------------
// The attention scratch (the per-request position prefix, the device check
// word and the split-K partials) lives in one file-scope device array instead
// of a caller workspace.  Its size bounds the shapes: the partial slots grow
// with (attention CTAs + head-group segments) x heads x D.
__device__ __align__(256) uint8_t g_attn_static_scratch[kAttnStaticScratchBytes];

// Scratch offsets inside the static array for `grid` attention CTAs.
struct StaticAttnLayout {
  size_t err, attn_prefix, part_ml, part_o, total;
};
StaticAttnLayout static_attn_layout(const pks_decode_args& a, int64_t grid) {
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const int hg = attn_heads_per_cta(a.Hkv);
  const int G = a.Hq / a.Hkv;
  const int64_t Bv = (int64_t)a.B * query_count(a);
  const int64_t nseg = (int64_t)(a.Hkv / hg) * Bv;
  const size_t nslots = (size_t)(grid + nseg) * hg * G;
  StaticAttnLayout L{};
  size_t off = 0;
  L.err = off;
  off = up(off + sizeof(int32_t) * 4);
  L.attn_prefix = off;
  off = up(off + sizeof(int32_t) * (size_t)(Bv + 2));
  L.part_ml = off;
  off = up(off + sizeof(float) * 2 * nslots);
  L.part_o = off;
  off = up(off + sizeof(float) * nslots * a.D);
  L.total = off;
  return L;
}

template <int D, int HG, int NGT>
cudaError_t launch_attn_static_t(const pks_decode_args& a, uint8_t* scratch, cudaStream_t s,
                                 bool* too_large) {
  auto kern = k_sparse_attention<D, HG, false, NGT>;
  const int nq = query_count(a);
  const int Bv = a.B * nq;
  const size_t smem = attn_smem_bytes<D, HG>(Bv);
  int bps = 1;
  cudaError_t e = attn_configure<D, HG, false, NGT>(smem, &bps);
  if (e != cudaSuccess) return e;
  // the same grid pks_sparse_attention uses for these arguments
  int grid = a.attn_splits > 0 ? a.attn_splits : device_sm_count() * bps;
  if (grid > kAttnGridMax) grid = kAttnGridMax;
  const StaticAttnLayout L = static_attn_layout(a, grid);
  if (L.total > kAttnStaticScratchBytes) {
    *too_large = true;
    return cudaSuccess;
  }
  const int G = a.Hq / a.Hkv;
  const int min_per_cta = a.attn_splits > 0 ? 0 : kAttnMinPositions;
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)a.D);
  kern<<<grid, HG * 32, smem, s>>>(
      a.seq_lens, a.block_table, reinterpret_cast<const __nv_bfloat16*>(a.q),
      reinterpret_cast<const __nv_bfloat16*>(a.kv_k), reinterpret_cast<const __nv_bfloat16*>(a.kv_v),
      a.topk_idx, reinterpret_cast<int32_t*>(scratch + L.attn_prefix),
      reinterpret_cast<float2*>(scratch + L.part_ml), reinterpret_cast<float*>(scratch + L.part_o),
      reinterpret_cast<__nv_bfloat16*>(a.out), reinterpret_cast<int32_t*>(scratch + L.err), Bv,
      a.Hq, a.Hkv, G, a.page_size, a.max_pages, a.num_pages, a.k, /*trim=*/0, min_per_cta,
      scale_log2, ResidentKv{}, nq);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  k_attention_merge<D><<<dim3((a.Hq + 3) / 4, Bv), 128, 0, s>>>(
      reinterpret_cast<const int32_t*>(scratch + L.attn_prefix),
      reinterpret_cast<const float2*>(scratch + L.part_ml),
      reinterpret_cast<const float*>(scratch + L.part_o), reinterpret_cast<__nv_bfloat16*>(a.out),
      Bv, a.Hq, a.Hkv, HG, G);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(const pks_decode_args& a, const WorkspaceLayout& L, uint8_t* ws,
                             bool trim, cudaStream_t s, const ResidentKv& rk) {
  const int hg = attn_heads_per_cta(a.Hkv);
  const bool wide = a.Hq / a.Hkv > 8;  // two 8-head column tiles
#define PKS_ATTN_CASE(D_, HG_)                                                             \
  if (a.D == D_ && hg == HG_) {                                                            \
    if (wide)                                                                              \
      return rk.page_slot ? launch_attn_t<D_, HG_, true, 2>(a, L, ws, trim, rk, s)          \
                          : launch_attn_t<D_, HG_, false, 2>(a, L, ws, trim, rk, s);        \
    return rk.page_slot ? launch_attn_t<D_, HG_, true, 1>(a, L, ws, trim, rk, s)            \
                        : launch_attn_t<D_, HG_, false, 1>(a, L, ws, trim, rk, s);          \
  }
  PKS_ATTN_CASE(64, 1)
  PKS_ATTN_CASE(64, 2)
  PKS_ATTN_CASE(64, 4)
  PKS_ATTN_CASE(64, 8)
  PKS_ATTN_CASE(128, 1)
  PKS_ATTN_CASE(128, 2)
  PKS_ATTN_CASE(128, 4)
  PKS_ATTN_CASE(128, 8)
#undef PKS_ATTN_CASE
  return cudaErrorInvalidValue;
}

size_t attention_static_min_bytes(const pks_decode_args& a) {
  return static_attn_layout(a, 1).total;
}

cudaError_t attention_static_scratch(uint8_t** ptr) {
  static void* cache[64] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!cache[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attn_static_scratch);
    if (e != cudaSuccess) return e;
    cache[dev] = p;
  }
  *ptr = static_cast<uint8_t*>(cache[dev]);
  return cudaSuccess;
}

cudaError_t launch_attention_static(const pks_decode_args& a, uint8_t* scratch, cudaStream_t s,
                                    bool* too_large) {
  *too_large = false;
  const int hg = attn_heads_per_cta(a.Hkv);
  const bool wide = a.Hq / a.Hkv > 8;
#define PKS_ATTN_STATIC_CASE(D_, HG_)                                                       \
  if (a.D == D_ && hg == HG_)                                                              \
    return wide ? launch_attn_static_t<D_, HG_, 2>(a, scratch, s, too_large)               \
                : launch_attn_static_t<D_, HG_, 1>(a, scratch, s, too_large);
  PKS_ATTN_STATIC_CASE(64, 1)
  PKS_ATTN_STATIC_CASE(64, 2)
  PKS_ATTN_STATIC_CASE(64, 4)
  PKS_ATTN_STATIC_CASE(64, 8)
  PKS_ATTN_STATIC_CASE(128, 1)
  PKS_ATTN_STATIC_CASE(128, 2)
  PKS_ATTN_STATIC_CASE(128, 4)
  PKS_ATTN_STATIC_CASE(128, 8)
#undef PKS_ATTN_STATIC_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pks
