// Sparse scaled dot-product attention over the selected tokens, split-K.
//
// "Sparse Attention on GLM5.3 and HBM", introduction: attention runs over
// only the top-k tokens, which cuts the bytes SDPA reads; "Paged KV cache",
// "Paging" and "What this table does not say": K/V are found through the
// page table, so the reads are scattered rows that the kernel must gather
// efficiently.
//
// One CTA per (split, KV head, request).  A split is a contiguous range of
// top-k positions.  The CTA first turns its positions into physical token rows
// (block table lookup, bounds checked), then streams 64-token tiles of K and V
// rows for its KV head (D*2 bytes each, contiguous) with 16-byte cp.async into
// a 3-stage shared-memory ring; rows are stored XOR-swizzled by 16-byte chunk
// so that ldmatrix reads are free of bank conflicts.  Each of the 4 warps owns
// 16 tokens of every tile and keeps its own online-softmax state for the G
// query heads of the group: S = Q K^T and O += P V run on the tensor cores
// (bf16 in, fp32 accumulate) with the G heads as the 16-row M dimension,
// padded with zero rows.  The warps' states are merged in shared memory, and
// the splits of one (request, KV head) are merged by the last CTA to finish
// (log-sum-exp rescaling), which writes the bf16 output.
//
// At G = 8 query heads per KV head the work is about 8 FLOP per byte of K/V,
// far below the tensor-core ridge: the kernel is bound by HBM bandwidth, and
// the MMAs only keep the arithmetic off the critical path.

#include <cuda_bf16.h>

#include "pks_internal.h"

namespace pks {
namespace {

constexpr int kAttnThreads = 128;
constexpr int kStages = 3;

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

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 2)
k_sparse_attention(const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ block_table,
                   const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kv_k,
                   const __nv_bfloat16* __restrict__ kv_v, const int32_t* __restrict__ topk,
                   int32_t* __restrict__ tick, float2* __restrict__ part_ml,
                   float* __restrict__ part_o, __nv_bfloat16* __restrict__ out,
                   int32_t* __restrict__ err, int Hq, int Hkv, int G, int page_size,
                   int max_pages, int num_pages, int k, int split_len, float scale_log2) {
  constexpr int CH = D / 8;   // 16-byte chunks per row
  constexpr int KS = D / 16;  // k-steps of S = Q K^T
  constexpr int ND = D / 8;   // 8-wide column tiles of O
  constexpr int TILE = kAttnTile;
  const float kNegInf = __int_as_float(0xff800000);

  extern __shared__ __align__(128) uint8_t smem[];
  int32_t* s_row = reinterpret_cast<int32_t*>(smem);
  const int row_bytes = (split_len * 4 + 127) & ~127;
  __nv_bfloat16* s_kv = reinterpret_cast<__nv_bfloat16*>(smem + row_bytes);
  __shared__ int s_last;

  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z, splits = gridDim.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int max_len = max_pages * page_size;
  int len = seq_lens[b];
  if (len < 0 || len > max_len) {
    if (h == 0 && split == 0 && tid == 0) flag_error(err, kErrLen);
    len = 0;
  }
  const int p0 = split * split_len;
  const int n_pos = max(0, min(k, p0 + split_len) - p0);

  // ---- selected positions -> physical token rows (page * page_size + slot)
  const int32_t* bt = block_table + (int64_t)b * max_pages;
  for (int i = tid; i < n_pos; i += kAttnThreads) {
    const int t = topk[(int64_t)b * k + p0 + i];
    int row = -1;
    if (t >= 0) {
      if (t >= len) {
        flag_error(err, kErrToken);
      } else {
        const int page = bt[t / page_size];
        if ((unsigned)page < (unsigned)num_pages) row = page * page_size + t % page_size;
        else flag_error(err, kErrPage);
      }
    }
    s_row[i] = row;
  }

  // ---- Q fragments of the G heads (rows >= G are zero)
  const int ra = lane >> 2, rb = ra + 8, cq = (lane & 3) * 2;
  uint32_t qa[KS][4];
  {
    const __nv_bfloat16* qb = q + ((int64_t)b * Hq + (int64_t)h * G) * D;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int col = ks * 16 + cq;
      qa[ks][0] = ra < G ? *reinterpret_cast<const uint32_t*>(qb + ra * D + col) : 0u;
      qa[ks][1] = rb < G ? *reinterpret_cast<const uint32_t*>(qb + rb * D + col) : 0u;
      qa[ks][2] = ra < G ? *reinterpret_cast<const uint32_t*>(qb + ra * D + col + 8) : 0u;
      qa[ks][3] = rb < G ? *reinterpret_cast<const uint32_t*>(qb + rb * D + col + 8) : 0u;
    }
  }
  __syncthreads();

  const int n_tiles = (n_pos + TILE - 1) / TILE;
  auto load_tile = [&](int tile, int stage) {
    __nv_bfloat16* sk = s_kv + (size_t)stage * 2 * TILE * D;
    __nv_bfloat16* sv = sk + TILE * D;
#pragma unroll 4
    for (int idx = tid; idx < TILE * CH; idx += kAttnThreads) {
      const int r = idx / CH, c = idx % CH;
      const int pos = tile * TILE + r;
      const int row = pos < n_pos ? s_row[pos] : -1;
      const int off = r * D + ((c ^ (r & 7)) << 3);
      const int64_t src = row >= 0 ? ((int64_t)row * Hkv + h) * D + c * 8 : 0;
      const int bytes = row >= 0 ? 16 : 0;  // 0 bytes: zero fill
      cp_async16(smem_u32(sk + off), kv_k + src, bytes);
      cp_async16(smem_u32(sv + off), kv_v + src, bytes);
    }
  };

  float o[ND][4];
#pragma unroll
  for (int i = 0; i < ND; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_a = kNegInf, m_b = kNegInf, l_a = 0.f, l_b = 0.f;

#pragma unroll
  for (int st = 0; st < kStages - 1; ++st) {
    if (st < n_tiles) load_tile(st, st);
    cp_async_commit();
  }

  const int r0 = warp * 16;
  for (int tile = 0; tile < n_tiles; ++tile) {
    {
      const int nt = tile + kStages - 1;
      if (nt < n_tiles) load_tile(nt, nt % kStages);
      cp_async_commit();
    }
    cp_async_wait<kStages - 1>();
    __syncthreads();

    const __nv_bfloat16* sk = s_kv + (size_t)(tile % kStages) * 2 * TILE * D;
    const __nv_bfloat16* sv = sk + TILE * D;

    // S^T fragments: 16 heads (rows) x 16 tokens (2 column tiles)
    float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int row = r0 + ((lane >> 4) << 3) + (lane & 7);
      const int chunk = 2 * ks + ((lane >> 3) & 1);
      uint32_t b0, b1, b2, b3;
      ldsm_x4(smem_u32(sk + row * D + ((chunk ^ (row & 7)) << 3)), b0, b1, b2, b3);
      mma_bf16(sacc[0], qa[ks], b0, b1);
      mma_bf16(sacc[1], qa[ks], b2, b3);
    }

    // online softmax (log2 domain) for rows ra and rb
    float x[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int pos = tile * TILE + r0 + nt * 8 + cq + e;
        const bool valid = pos < n_pos && s_row[pos] >= 0;
        x[nt][e] = valid ? sacc[nt][e] * scale_log2 : kNegInf;
        x[nt][e + 2] = valid ? sacc[nt][e + 2] * scale_log2 : kNegInf;
      }
    }
    float mx_a = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
    float mx_b = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
    mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
    mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
    mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
    mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
    const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
    const float al_a = mn_a == kNegInf ? 1.f : exp2f(m_a - mn_a);
    const float al_b = mn_b == kNegInf ? 1.f : exp2f(m_b - mn_b);
    float p[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      p[nt][0] = x[nt][0] == kNegInf ? 0.f : exp2f(x[nt][0] - mn_a);
      p[nt][1] = x[nt][1] == kNegInf ? 0.f : exp2f(x[nt][1] - mn_a);
      p[nt][2] = x[nt][2] == kNegInf ? 0.f : exp2f(x[nt][2] - mn_b);
      p[nt][3] = x[nt][3] == kNegInf ? 0.f : exp2f(x[nt][3] - mn_b);
    }
    l_a = l_a * al_a + (p[0][0] + p[0][1] + p[1][0] + p[1][1]);
    l_b = l_b * al_b + (p[0][2] + p[0][3] + p[1][2] + p[1][3]);
    m_a = mn_a;
    m_b = mn_b;
#pragma unroll
    for (int i = 0; i < ND; ++i) {
      o[i][0] *= al_a;
      o[i][1] *= al_a;
      o[i][2] *= al_b;
      o[i][3] *= al_b;
    }
    const uint32_t pa[4] = {pack_bf16(p[0][0], p[0][1]), pack_bf16(p[0][2], p[0][3]),
                            pack_bf16(p[1][0], p[1][1]), pack_bf16(p[1][2], p[1][3])};
#pragma unroll
    for (int nd = 0; nd < ND; nd += 2) {
      const int row = r0 + (((lane >> 3) & 1) << 3) + (lane & 7);
      const int chunk = nd + (lane >> 4);
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(smem_u32(sv + row * D + ((chunk ^ (row & 7)) << 3)), b0, b1, b2, b3);
      mma_bf16(o[nd], pa, b0, b1);
      mma_bf16(o[nd + 1], pa, b2, b3);
    }
    __syncthreads();
  }
  cp_async_wait<0>();
  __syncthreads();

  // ---- merge the 4 warps' states in shared memory (reusing the ring)
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
  float* s_o = reinterpret_cast<float*>(s_kv);  // [4][16][D]
  float* s_m = s_o + 4 * 16 * D;                // [4][16]
  float* s_l = s_m + 4 * 16;                    // [4][16]
#pragma unroll
  for (int nd = 0; nd < ND; ++nd) {
    const int d = nd * 8 + cq;
    s_o[(warp * 16 + ra) * D + d] = o[nd][0];
    s_o[(warp * 16 + ra) * D + d + 1] = o[nd][1];
    s_o[(warp * 16 + rb) * D + d] = o[nd][2];
    s_o[(warp * 16 + rb) * D + d + 1] = o[nd][3];
  }
  if ((lane & 3) == 0) {
    s_m[warp * 16 + ra] = m_a;
    s_l[warp * 16 + ra] = l_a;
    s_m[warp * 16 + rb] = m_b;
    s_l[warp * 16 + rb] = l_b;
  }
  __syncthreads();

  const int64_t bh = (int64_t)b * Hkv + h;
  for (int idx = tid; idx < G * D; idx += kAttnThreads) {
    const int g = idx / D, d = idx % D;
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, s_m[w * 16 + g]);
    float L = 0.f, O = 0.f;
    if (M != kNegInf) {
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float mw = s_m[w * 16 + g];
        if (mw == kNegInf) continue;
        const float f = exp2f(mw - M);
        L += s_l[w * 16 + g] * f;
        O += s_o[(w * 16 + g) * D + d] * f;
      }
    }
    if (splits == 1) {
      out[((int64_t)b * Hq + (int64_t)h * G + g) * D + d] = __float2bfloat16(L > 0.f ? O / L : 0.f);
    } else {
      const int64_t slot = (bh * splits + split) * G + g;
      part_o[slot * D + d] = O;
      if (d == 0) part_ml[slot] = make_float2(M, L);
    }
  }
  if (splits == 1) return;

  // ---- the last split CTA of (request, KV head) merges the splits
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    s_last = atomicAdd(tick + bh, 1) == splits - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int idx = tid; idx < G * D; idx += kAttnThreads) {
    const int g = idx / D, d = idx % D;
    float M = kNegInf;
    for (int s = 0; s < splits; ++s) M = fmaxf(M, __ldcg(&part_ml[(bh * splits + s) * G + g].x));
    float L = 0.f, O = 0.f;
    if (M != kNegInf) {
      for (int s = 0; s < splits; ++s) {
        const int64_t slot = (bh * splits + s) * G + g;
        const float2 ml = __ldcg(&part_ml[slot]);
        if (ml.x == kNegInf) continue;
        const float f = exp2f(ml.x - M);
        L += ml.y * f;
        O += __ldcg(&part_o[slot * D + d]) * f;
      }
    }
    out[((int64_t)b * Hq + (int64_t)h * G + g) * D + d] = __float2bfloat16(L > 0.f ? O / L : 0.f);
  }
  if (tid == 0) tick[bh] = 0;
}

template <int D>
cudaError_t launch_attn_t(const pks_decode_args& a, const WorkspaceLayout& L, uint8_t* ws,
                          cudaStream_t s) {
  auto kern = k_sparse_attention<D>;
  const size_t row_bytes = ((size_t)L.split_len * 4 + 127) & ~(size_t)127;
  const size_t ring = (size_t)kStages * 2 * kAttnTile * D * sizeof(__nv_bfloat16);
  const size_t merge = (4 * 16 * D + 2 * 4 * 16) * sizeof(float);
  const size_t smem = row_bytes + (ring > merge ? ring : merge);
  // raise the dynamic shared-memory limit once per device and size (not a
  // stream operation, so it stays out of any graph capture after the first call)
  static size_t configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  size_t& done = configured[dev & 63];
  if (smem > done) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    done = smem;
  }
  const int G = a.Hq / a.Hkv;
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)a.D);
  dim3 grid(L.splits, a.Hkv, a.B);
  kern<<<grid, kAttnThreads, smem, s>>>(
      a.seq_lens, a.block_table, reinterpret_cast<const __nv_bfloat16*>(a.q),
      reinterpret_cast<const __nv_bfloat16*>(a.kv_k), reinterpret_cast<const __nv_bfloat16*>(a.kv_v),
      a.topk_idx, reinterpret_cast<int32_t*>(ws + L.tick_attn),
      reinterpret_cast<float2*>(ws + L.part_ml), reinterpret_cast<float*>(ws + L.part_o),
      reinterpret_cast<__nv_bfloat16*>(a.out), reinterpret_cast<int32_t*>(ws + L.err), a.Hq, a.Hkv,
      G, a.page_size, a.max_pages, a.num_pages, a.k, L.split_len, scale_log2);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(const pks_decode_args& a, const WorkspaceLayout& L, uint8_t* ws,
                             cudaStream_t s) {
  if (a.D == 64) return launch_attn_t<64>(a, L, ws, s);
  if (a.D == 128) return launch_attn_t<128>(a, L, ws, s);
  return cudaErrorInvalidValue;
}

}  // namespace pks
