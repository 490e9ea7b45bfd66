// Sparse MLA decode in MQA mode on the fifth-generation tensor cores.
//
// "Sparse Attention on GLM5.3 and HBM", DeepSeek Sparse Attention paragraphs:
// the sparse MLA runs in MQA mode.  Every token keeps one latent row of d + r
// values (d = 512 latent, r = 64 RoPE) shared by all H query heads; a head's
// scores use the whole row and its output is the softmax-weighted sum of the
// latent part.  The pages' intensity model, 2H(2d + r) FLOP per (d + r) * 2
// bytes, is about 1.89 H FLOP/B: with 64-128 heads both products are real
// dense contractions with the heads as the M dimension, which is what the
// tcgen05 MMA with its accumulator in tensor memory is for.
//
// One CTA per (request, split of its selected tokens, half of the latent
// value width), 512 threads: warps 0-7 are the softmax threads, two per row of
// the MMA (query heads, zero rows above H; row h is tensor-memory lane h, read
// by warps h / 32 and h / 32 + 4, each for half of the row's columns); warp 8
// is the producer (MMA issue); warps 9-14 gather the K/V rows; warp 15 issues
// the second half of S.
// Per 64-token tile:
//   S[128 x 64]   = Q[128 x 576] . K^T          tcgen05.mma, fp32 in TMEM
//   P             = exp2(S * scale - m)         two threads per head row
//   O[128 x 256] += P[128 x 64] . V[64 x 256]   tcgen05.mma, fp32 in TMEM
// A tcgen05.mma costs about the same time for N = 32 or 64 and M = 64 or
// 128 (measured): the cost is the issue, so S is computed 64 tokens at a
// time, as two N = 32 halves issued side by side by two threads.  Tensor memory holds
// O (256 columns: this CTA's half of the value width; all of O would fill
// it, hence the two halves, which both compute S), S (64 columns) and Q's
// values 0..383 (192 columns, the A operand of 24 of the 36 k-steps of S);
// Q's values 384..575 stay in shared memory (48 KiB, 128-byte swizzled,
// K-major).  K/V tiles are gathered through the block table with cp.async
// into a two-stage ring (72 KiB each); the same tile is the K operand
// (K-major) and the V operand (MN-major).  P goes through shared memory
// (128-byte swizzled, K-major).  The running max moves only when a tile's
// max exceeds it by more than 8 (log2 units), so O is rarely rescaled in
// TMEM.
//
// Roles and hand-offs (mbarriers, every wait bounded):
//   all threads, once: the physical row of every position of the CTA's tiles
//     (top-k entry, then block table) into a shared table;
//   gather warps: tile t into stage t & 1 once the O update of tile t - 2 has
//     released the stage (bar_free), then publish it (bar_full);
//   producer warp: issues O += P.V of tile t - 1 once its P is written (bar_p,
//     commit -> bar_o and bar_free) and then S = Q.K^T of tile t's tokens
//     0..31 once its gathers have landed (bar_full, commit -> bar_s[0]);
//   issuer warp: S of tile t's tokens 32..63 on the same conditions
//     (commit -> bar_s[1]);
//   softmax warps: after the O update of tile t - 1 (bar_o) take their half
//     of S of tile t (bar_s[half]), exchange each row's max and sum between
//     its two threads (bar_mx, bar_ps), rescale O if the max moved, write P
//     (bar_p).
// So the tensor pipe runs O(t - 1) before S(t), and the next tile's gathers
// run beside the softmax instead of in front of it.  With several splits per
// request the CTAs write (m, l, O) partials that k_mla_merge combines.

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pks_internal.h"

namespace pks {
namespace {

constexpr int kDL = kMlaLatent;             // latent width d (the value)
constexpr int kDK = kMlaLatent + kMlaRope;  // key width d + r
constexpr int kTile = 64;                   // tokens per tile (MMA N of S)
constexpr int kRows = 128;                  // MMA M: query heads, zero padded
constexpr int kHalf = kDL / 2;              // value columns per CTA
constexpr int kCons = 2 * kRows;            // softmax threads: two per head row
constexpr int kProdWarp = kCons / 32;       // warp 8: the producer
constexpr int kGather = 192;                 // gather threads: warps 9-14
constexpr int kIssueWarp = kProdWarp + 1 + kGather / 32;  // warp 15: issues S for tokens 32..63
constexpr int kThreads = kCons + 32 + kGather + 32;  // 512: softmax, producer, gather, issuer
constexpr int kBlk = kDK / 64;              // 64-value (128-byte) column blocks
constexpr int kQTmemDims = 384;             // Q values 0..383 live in tensor memory
constexpr int kQSmemBlk = (kDK - kQTmemDims) / 64;  // the rest: 3 column blocks in smem
constexpr uint32_t kQBlockBytes = kRows * 128;
constexpr uint32_t kKBlockBytes = kTile * 128;
constexpr uint32_t kQBytes = kQSmemBlk * kQBlockBytes;
constexpr uint32_t kKStageBytes = kBlk * kKBlockBytes;
constexpr uint32_t kPBytes = kRows * kTile * 2;  // 128-byte rows
constexpr uint32_t kSmemBytes = kQBytes + 2 * kKStageBytes + kPBytes + 1024;
constexpr uint32_t kTmemCols = 512;
// tensor-memory columns: O (fp32), S (fp32), Q values 0..383 (two bf16 a column)
constexpr uint32_t kTmemO = 0, kTmemS = kHalf, kTmemQ = kHalf + kTile;
static_assert(kTmemQ + kQTmemDims / 2 == kTmemCols, "O, S and Q fill the tensor memory");
constexpr long long kWaitCycles = 4000000000LL;  // about 2 s at 2 GHz, unless wait_limit is set
// tiles of one CTA whose rows are resolved up front (the host picks enough
// splits that no CTA has more)
constexpr int kMaxCtaTiles = kMlaMaxCtaTiles;

static_assert(kDK % 64 == 0 && kDL % 64 == 0, "latent and key widths in 64-value blocks");
static_assert(kSmemBytes <= 232448, "shared memory of one CTA");
static_assert(kRows * (kHalf + 4) * 4 <= 2 * kKStageBytes, "O staged in the K stages");

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void flag_error(int32_t* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

// generic-proxy writes of this thread to shared memory become visible to the
// tensor core's (async proxy) reads
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// ---- mbarrier (completion of committed MMAs) ------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// bounded wait for the phase with the given parity; false when it gave up
// or when another warp of the CTA has given up (*abort set)
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          const volatile int* abort, long long budget) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (*abort || clock64() - t0 > budget) return false;
  return true;
}
// bounded wait that ignores the abort flag: the producer waits for its own
// MMAs to complete before the tensor memory they write is freed
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > kWaitCycles) return;
}

// ---- tcgen05: tensor memory, MMA, commit ----------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                   smem_u32(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

// 2^x with the hardware's approximate exponential (ex2.approx: a few ulp in
// fp32); the probabilities it gives are rounded to bf16 for the P.V product
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// D[tmem] (+)= A[smem] . B[smem], bf16 inputs, fp32 accumulator
__device__ __forceinline__ void mma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] . B[smem]: A's rows in the D lanes, two bf16 a column
__device__ __forceinline__ void mma_bf16_ta(uint32_t d, uint32_t a_tmem, uint64_t b,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// arrive once on bar when every MMA this thread issued so far has completed
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
          smem_u32(bar))
      : "memory");
}

// 32 consecutive fp32 columns of this thread's lane (warp w reads lanes
// 32w .. 32w + 31); the wait is inside the same statement so no use of the
// values can be scheduled before it
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
      "%29, %30, %31, %32};\n"
      "tcgen05.wait::st.sync.aligned;\n" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

// barrier `id` among `n` threads that also ANDs a predicate over them
__device__ __forceinline__ bool bar_and(uint32_t id, uint32_t n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, %2, %3, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
// Shared-memory operand descriptor: start address, leading and stride byte
// offsets (16-byte units), descriptor version 1, swizzle mode in bits 61-63
// (2: 128-byte swizzle, 4: 64-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo,
                                              uint32_t swizzle) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) |
         ((uint64_t)(sbo >> 4) << 32) | (1ull << 46) | ((uint64_t)swizzle << 61);
}
constexpr uint32_t kSw128 = 2;

// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5 = 1), bf16
// A and B (bits 7-9, 10-12 = 1), B major-ness in bit 16 (1: MN-major), N / 8
// in bits 17-22, M / 16 in bits 24-28; A is K-major.
constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
constexpr uint32_t kIdescS = idesc_bf16(kRows, kTile / 2, false);  // S = Q . K^T, half the tokens
constexpr uint32_t kIdescO = idesc_bf16(kRows, kHalf, true);    // O += P . V

__global__ void __launch_bounds__(kThreads, 1)
k_mla_attention(const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ block_table,
                const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kv,
                const int32_t* __restrict__ topk, float2* __restrict__ part_ml,
                float* __restrict__ part_o, __nv_bfloat16* __restrict__ out,
                int32_t* __restrict__ err, int B, int H, int page_size, int max_pages,
                int num_pages, int k, int trim, int splits, float scale_log2,
                long long budget) {
  extern __shared__ uint8_t smem_raw[];
  // bar_full[i]: stage i gathered (one arrival a gather warp); bar_s[h]: S of
  // the tile's tokens 32h .. 32h + 31 ready (two issuing threads);
  // bar_p: P written (one arrival a softmax warp); bar_o: O update done;
  // bar_mx / bar_ps: every softmax warp has posted its rows' half max / sum
  // bar_free[i]: the O update of the last tile in stage i is done (the stage
  // may be refilled)
  __shared__ __align__(8) uint64_t bar_full[2], bar_free[2], bar_s[2], bar_p, bar_o, bar_mx, bar_ps;
  __shared__ uint32_t s_tmem;
  __shared__ int32_t s_row[kMaxCtaTiles][kTile];         // physical row of each position
  __shared__ uint32_t s_mask[kMaxCtaTiles][kTile / 32];  // positions with a row
  __shared__ int s_abort;
  __shared__ float s_mx[2][kRows], s_ps[2][kRows];  // a row's two halves: tile max, sum

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the merge kernel may take SM slots now (it waits for this grid to finish)
  pdl_launch_dependents();
  const int half = blockIdx.x & 1;
  const int split = (blockIdx.x >> 1) % splits;
  const int b = (blockIdx.x >> 1) / splits;
  if (b >= B) return;
  const float kNegInf = __int_as_float(0xff800000);

  const int max_len = max_pages * page_size;
  int len = seq_lens[b];
  if (len < 0 || len > max_len) {
    if (tid == 0) flag_error(err, kErrLen);
    len = -1;
  }
  // positions of the request's list to visit: its own top-k list holds the
  // selected entries first (trim: min(k, len) of them), any other list is
  // visited in full
  const int npos = len < 0 ? 0 : (trim ? min(len, k) : k);
  const int ntiles_req = (npos + kTile - 1) / kTile;
  const int t_lo = (int)((int64_t)split * ntiles_req / splits);
  const int t_hi = (int)((int64_t)(split + 1) * ntiles_req / splits);
  const int ntiles = t_hi - t_lo;
  const int64_t slot = (int64_t)b * splits + split;  // partial slot of this CTA
  const int h = tid % kRows;                           // head row of a softmax thread

  if (ntiles > kMaxCtaTiles) {  // more than the row table holds: the host rules this out
    if (tid == 0) flag_error(err, kErrState);
    return;
  }
  if (ntiles == 0) {  // nothing selected in this range
    pdl_wait();  // the previous kernel may still read the outputs
    if (tid < kRows && h < H) {
      if (splits > 1) {
        if (half == 0) part_ml[slot * H + h] = make_float2(kNegInf, 0.f);
      } else {
        __nv_bfloat16* ob = out + ((int64_t)b * H + h) * kDL + half * kHalf;
        for (int c = 0; c < kHalf; ++c) ob[c] = __float2bfloat16(0.f);
      }
    }
    return;
  }

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = base, sK = base + kQBytes, sP = sK + 2 * kKStageBytes;

  if (warp == 0) tmem_alloc(&s_tmem, kTmemCols);
  if (tid == kCons) {
    // one arrival a warp (after the warp's own fences and a __syncwarp)
    mbar_init(&bar_full[0], kGather / 32);
    mbar_init(&bar_full[1], kGather / 32);
    mbar_init(&bar_free[0], 1);
    mbar_init(&bar_free[1], 1);
    mbar_init(&bar_s[0], 1);
    mbar_init(&bar_s[1], 1);
    mbar_init(&bar_p, kCons / 32);
    mbar_init(&bar_o, 1);
    mbar_init(&bar_mx, kCons / 32);
    mbar_init(&bar_ps, kCons / 32);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    s_abort = 0;
  }
  // Q rows (heads; zero rows from H to 128).  Values 384..575: 128-byte
  // swizzled K-major in shared memory (16-byte chunk c of row r in column
  // block j at chunk c ^ (r & 7)).  Values 0..383: staged row by row in the
  // K stages (rows padded to 784 bytes), then copied by each head's thread
  // into its tensor-memory lane.
  constexpr uint32_t kQStageRow = kQTmemDims * 2 + 16;
  {
    const __nv_bfloat16* qb = q + (int64_t)b * H * kDK;
    for (int id = tid; id < kRows * kBlk * 8; id += kThreads) {
      const int r = id / (kBlk * 8), cc = id % (kBlk * 8);
      const __nv_bfloat16* src = qb + (r < H ? (int64_t)r * kDK + cc * 8 : 0);
      uint32_t dst;
      if (cc < kQTmemDims / 8) {
        dst = sK + r * kQStageRow + cc * 16;
      } else {
        const int j = (cc - kQTmemDims / 8) >> 3, c = cc & 7;
        dst = sQ + j * kQBlockBytes + r * 128 + ((c ^ (r & 7)) << 4);
      }
      cp_async16(dst, src, r < H ? 16 : 0);
    }
    cp_async_commit();
    cp_async_wait_all();
    fence_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  if (tid < kRows) {
    const uint32_t lo = (uint32_t)(warp * 32) << 16;
    const uint32_t src = sK + (uint32_t)tid * kQStageRow;
#pragma unroll 1
    for (int c = 0; c < kQTmemDims / 64; ++c) {
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        uint32_t x0, x1, x2, x3;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];\n"
                     : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3)
                     : "r"(src + (uint32_t)(c * 128 + i * 4)));
        v[i] = __uint_as_float(x0);
        v[i + 1] = __uint_as_float(x1);
        v[i + 2] = __uint_as_float(x2);
        v[i + 3] = __uint_as_float(x3);
      }
      tmem_st32(tmem + lo + kTmemQ + c * 32, v);
    }
  }
  // the selection comes from the top-k kernel: everything above (tensor
  // memory, barriers, Q) overlapped its tail.  Then every thread helps to
  // resolve the physical row of each position of this CTA's tiles (-1: none),
  // one 32-position group a warp at a time
  pdl_wait();
  for (int g = warp; g < ntiles * (kTile / 32); g += kThreads / 32) {
    const int tile = g / (kTile / 32), w = g % (kTile / 32);
    const int p = (t_lo + tile) * kTile + w * 32 + lane;
    int row = -1;
    if (p < npos) {
      const int t = topk[(int64_t)b * k + p];
      if (t >= 0) {
        if (t >= len) {
          flag_error(err, kErrToken);
        } else {
          const int page = block_table[(int64_t)b * max_pages + t / page_size];
          if ((unsigned)page < (unsigned)num_pages) row = page * page_size + t % page_size;
          else flag_error(err, kErrPage);
        }
      }
    }
    s_row[tile][w * 32 + lane] = row;
    const uint32_t m = __ballot_sync(0xffffffffu, row >= 0);
    if (lane == 0) s_mask[tile][w] = m;
  }
  // the staging area becomes the K stages: every thread is done reading it,
  // and the rows are in place
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint64_t dq0 = smem_desc(sQ, 16, 1024, kSw128);
  const uint64_t dp0 = smem_desc(sP, 16, 1024, kSw128);
  // S = Q . K^T of local tile tt for its tokens 32 h2 .. 32 h2 + 31 (one
  // thread): 36 k-steps of N = 32.  Two threads in two warps issue the two
  // halves side by side; their rows start 32 rows (4 KiB, whole swizzle
  // atoms) into every column block of the stage.
  auto issue_s = [&](int tt, int h2) {
    const uint64_t dk0 = smem_desc(sK + (uint32_t)(tt & 1) * kKStageBytes + (uint32_t)h2 * 32 * 128,
                                   16, 1024, kSw128);
    const uint32_t d = tmem + kTmemS + (uint32_t)h2 * (kTile / 2);
#pragma unroll
    for (int kk = 0; kk < kDK / 16; ++kk) {
      const uint64_t db = dk0 + (uint64_t)(((kk >> 2) * kKBlockBytes + (kk & 3) * 32) >> 4);
      if (kk < kQTmemDims / 16) {
        mma_bf16_ta(d, tmem + kTmemQ + kk * 8, db, kIdescS, kk > 0 ? 1u : 0u);
      } else {
        const int qk = kk - kQTmemDims / 16;
        mma_bf16(d, dq0 + (uint64_t)(((qk >> 2) * kQBlockBytes + (qk & 3) * 32) >> 4), db,
                 kIdescS, 1u);
      }
    }
    mma_commit(&bar_s[h2]);
  };

  if (warp == kProdWarp || warp == kIssueWarp) {
    // ================= MMA issue: producer warp and second S issuer ========
    auto issue_pv = [&](int tt) {  // O += P . V(tile tt)
      const uint32_t vst = sK + (uint32_t)(tt & 1) * kKStageBytes +
                           (uint32_t)half * (kHalf / 64) * kKBlockBytes;
      const uint64_t dv0 = smem_desc(vst, kKBlockBytes, 1024, kSw128);
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk)
        mma_bf16(tmem + kTmemO, dp0 + (uint64_t)((kk * 32) >> 4),
                 dv0 + (uint64_t)((kk * 16 * 128) >> 4), kIdescO, (tt > 0 || kk > 0) ? 1u : 0u);
      mma_commit(&bar_o);
      mma_commit(&bar_free[tt & 1]);
    };
    // lane 0 waits, the warp follows: control flow stays warp-uniform
    auto wait0 = [&](uint64_t* bar, uint32_t parity) -> bool {
      bool w = lane == 0 ? mbar_wait(bar, parity, &s_abort, budget) : true;
      __syncwarp();
      return __shfl_sync(0xffffffffu, w ? 1 : 0, 0) != 0;
    };
    const bool prod = warp == kProdWarp;  // the producer also issues every O update
    const int h2 = prod ? 0 : 1;
    bool ok = true;
    int last_s = -1, last_pv = -1;  // the last tiles whose S / O update was issued
    for (int t = 0; t < ntiles && ok; ++t) {
      // 1. the previous tile's P is written: its O update (producer), and the
      //    S accumulator may be rewritten (both issuers).  The O update's
      //    completion frees P and, on bar_free, the previous tile's stage.
      if (t > 0) {
        if (!wait0(&bar_p, (t - 1) & 1)) { ok = false; break; }
        if (prod && lane == 0) {
          tc_fence_after();
          issue_pv(t - 1);
          last_pv = t - 1;
        }
        __syncwarp();
      }
      // 2. this thread's half of S = Q . K^T once the tile's gathers landed
      if (!wait0(&bar_full[t & 1], (t >> 1) & 1)) { ok = false; break; }
      if (lane == 0) {
        tc_fence_after();
        issue_s(t, h2);
        last_s = t;
      }
      __syncwarp();
    }
    if (ok && prod) {
      if (!wait0(&bar_p, (ntiles - 1) & 1)) ok = false;
      else if (lane == 0) {
        tc_fence_after();
        issue_pv(ntiles - 1);
        last_pv = ntiles - 1;
      }
    }
    if (!ok && lane == 0) {
      flag_error(err, kErrTimeout);
      s_abort = 1;
    }
    // every MMA this thread issued completes before the tensor memory is
    // freed, also when another warp gave up (normally these have completed)
    if (lane == 0) {
      if (last_s >= 0) mbar_drain(&bar_s[h2], last_s & 1);
      if (last_pv >= 0) mbar_drain(&bar_o, last_pv & 1);
    }
    __syncwarp();
  } else if (warp < kProdWarp) {
    // ================= softmax warps: two threads per head row =============
    // thread tid: row h = tid % 128 (warps w and w + 4 share TMEM lanes), half
    // ch = tid / 128 of the row's S columns (32 of 64) and O columns (128 of 256)
    const int ch = tid / kRows;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;  // this warp's TMEM lanes
    // every lane waits; a vote keeps control flow warp-uniform (the TMEM
    // accesses are warp-collective)
    auto waitw = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, &s_abort, budget)) != 0;
    };
    float m_run = kNegInf, l_run = 0.f;
    bool ok = true;
    for (int t = 0; t < ntiles && ok; ++t) {
      // the O update of tile t - 1 is done: O may be rescaled and P rewritten
      if (t > 0) {
        if (!waitw(&bar_o, (t - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      if (!waitw(&bar_s[ch], t & 1)) {  // this thread's 32 columns
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t mask = s_mask[t][ch];
      float sv[32];
      tmem_ld32(tmem + lane_off + kTmemS + ch * 32, sv);
      float mh = kNegInf;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        sv[j] = (mask >> j) & 1u ? sv[j] * scale_log2 : kNegInf;
        mh = fmaxf(mh, sv[j]);
      }
      // the row's max over both halves (both threads get the same value)
      s_mx[ch][h] = mh;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_mx);
      if (!waitw(&bar_mx, t & 1)) {
        ok = false;
        break;
      }
      const float mt = fmaxf(s_mx[0][h], s_mx[1][h]);
      const bool move = mt > m_run + 8.f;  // also true on the first valid tile
      const float m_new = move ? mt : m_run;
      const float alpha = move ? exp2f(m_run - m_new) : 1.f;  // 0 when m_run = -inf
      float ph = 0.f;
      uint32_t pk[16];
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const float p0 = sv[j] == kNegInf ? 0.f : ex2_approx(sv[j] - m_new);
        const float p1 = sv[j + 1] == kNegInf ? 0.f : ex2_approx(sv[j + 1] - m_new);
        const __nv_bfloat162 pp = __floats2bfloat162_rn(p0, p1);
        ph += __low2float(pp) + __high2float(pp);
        pk[j / 2] = *reinterpret_cast<const uint32_t*>(&pp);
      }
      // the row's sum, added in the same order by both threads
      s_ps[ch][h] = ph;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_ps);
      if (!waitw(&bar_ps, t & 1)) {
        ok = false;
        break;
      }
      l_run = l_run * alpha + (s_ps[0][h] + s_ps[1][h]);
      m_run = m_new;
      // rescale the O accumulated so far (warp-wide: TMEM access is collective)
      if (__any_sync(0xffffffffu, move && t > 0)) {
        const float a = (move && t > 0) ? alpha : 1.f;
#pragma unroll 1
        for (int c = ch * 4; c < ch * 4 + 4; ++c) {  // this thread's 128 O columns
          float ov[32];
          tmem_ld32(tmem + lane_off + kTmemO + c * 32, ov);
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] *= a;
          tmem_st32(tmem + lane_off + kTmemO + c * 32, ov);
        }
      }
      // P row h: 64 bf16 = eight 16-byte chunks, 128-byte swizzle (chunk c of
      // row h at chunk c ^ (h & 7)); this thread writes chunks 4ch .. 4ch + 3
      const uint32_t prow = sP + (uint32_t)h * 128;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int c = ch * 4 + i;
        const uint32_t dst = prow + ((c ^ (h & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(dst), "r"(pk[4 * i]),
                     "r"(pk[4 * i + 1]), "r"(pk[4 * i + 2]), "r"(pk[4 * i + 3])
                     : "memory");
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_p);
    }
    // ---- O of this CTA's half: to the output, or to the partial slot.  A
    // thread's row is 512 contiguous bytes, so the rows go through shared
    // memory (the K stages: every gather and MMA has completed once the last
    // O update has) and leave as whole rows, 512 bytes a warp instruction,
    // instead of 32 rows' 16-byte pieces
    const bool have_o = ok && waitw(&bar_o, (ntiles - 1) & 1);
    float* stage = reinterpret_cast<float*>(smem_raw + (sK - smem_u32(smem_raw)));
    constexpr int kStageRow = kHalf + 4;  // floats; 16 bytes of padding spread the banks
    if (have_o) {
      tc_fence_after();
      // the output is normalised here; partials keep (m, l) apart
      const float scale = splits == 1 ? (l_run > 0.f ? 1.f / l_run : 0.f) : 1.f;
#pragma unroll 1
      for (int c = ch * 4; c < ch * 4 + 4; ++c) {
        float ov[32];
        tmem_ld32(tmem + lane_off + kTmemO + c * 32, ov);
        float* dst = stage + h * kStageRow + c * 32;
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          *reinterpret_cast<float4*>(dst + i) =
              make_float4(ov[i] * scale, ov[i + 1] * scale, ov[i + 2] * scale, ov[i + 3] * scale);
      }
      if (splits > 1 && half == 0 && ch == 0 && h < H)
        part_ml[slot * H + h] = make_float2(m_run, l_run);
    }
    // the 256 softmax threads: every row staged, unless a warp gave up
    if (bar_and(1, kCons, have_o)) {
      constexpr int kQ = kHalf / 4;  // float4 columns of a row
      for (int idx = tid; idx < H * kQ; idx += kCons) {
        const int r = idx / kQ, q4 = idx % kQ;
        const float4 v = *reinterpret_cast<const float4*>(stage + r * kStageRow + q4 * 4);
        if (splits == 1) {
          __nv_bfloat16* ob = out + ((int64_t)b * H + r) * kDL + half * kHalf + q4 * 4;
          __nv_bfloat162 p0 = __floats2bfloat162_rn(v.x, v.y);
          __nv_bfloat162 p1 = __floats2bfloat162_rn(v.z, v.w);
          uint2 w;
          w.x = *reinterpret_cast<uint32_t*>(&p0);
          w.y = *reinterpret_cast<uint32_t*>(&p1);
          *reinterpret_cast<uint2*>(ob) = w;
        } else {
          *reinterpret_cast<float4*>(part_o + (slot * H + r) * kDL + half * kHalf + q4 * 4) = v;
        }
      }
    }
    if (!have_o) ok = false;
    if (!ok && lane == 0) {
      flag_error(err, kErrTimeout);
      s_abort = 1;
    }
  } else {
    // ================= gather warps: K/V rows of every tile =================
    // tile t goes to stage t & 1 once the O update of tile t - 2 (the stage's
    // last reader) is done; its 64 rows x 72 16-byte chunks, 128-byte swizzle
    // (chunk c of row r in column block j at chunk c ^ (r & 7))
    const int gt = tid - (kCons + 32);
    bool ok = true;
    for (int t = 0; t < ntiles && ok; ++t) {
      const int st = t & 1;
      if (t >= 2) {
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&bar_free[st], ((t - 2) >> 1) & 1, &s_abort, budget))) {
          ok = false;
          break;
        }
      }
      const uint32_t dst0 = sK + (uint32_t)st * kKStageBytes;
#pragma unroll 2
      for (int id = gt; id < kTile * kBlk * 8; id += kGather) {
        const int r = id / (kBlk * 8), cc = id % (kBlk * 8);
        const int j = cc >> 3, c = cc & 7;
        const int row = s_row[t][r];
        const __nv_bfloat16* src = kv + (row >= 0 ? (int64_t)row * kDK + cc * 8 : 0);
        cp_async16(dst0 + j * kKBlockBytes + r * 128 + ((c ^ (r & 7)) << 4), src,
                   row >= 0 ? 16 : 0);
      }
      cp_async_commit();
      // this thread's copies have landed: visible to the tensor core, counted
      cp_async_wait_all();
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_full[st]);
    }
    if (!ok && lane == 0) {
      flag_error(err, kErrTimeout);
      s_abort = 1;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// out[b, h] from the splits' partials: softmax-weighted by exp2(m_s - M)
__global__ void __launch_bounds__(128)
k_mla_merge(const float2* __restrict__ part_ml, const float* __restrict__ part_o,
            __nv_bfloat16* __restrict__ out, int H, int splits) {
  const int h = blockIdx.x, b = blockIdx.y;
  pdl_launch_dependents();  // a following kernel may launch and wait for this grid
  pdl_wait();  // the partials come from k_mla_attention
  const float kNegInf = __int_as_float(0xff800000);
  float M = kNegInf;
  for (int s = 0; s < splits; ++s) {
    const float2 e = part_ml[((int64_t)b * splits + s) * H + h];
    if (e.y > 0.f) M = fmaxf(M, e.x);
  }
  float L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < splits; ++s) {
    const int64_t sl = ((int64_t)b * splits + s) * H + h;
    const float2 e = part_ml[sl];
    if (!(e.y > 0.f)) continue;
    const float w = exp2f(e.x - M);
    L += w * e.y;
    const float4 v = reinterpret_cast<const float4*>(part_o + sl * kDL)[threadIdx.x];
    acc.x += w * v.x;
    acc.y += w * v.y;
    acc.z += w * v.z;
    acc.w += w * v.w;
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  __nv_bfloat16* ob = out + ((int64_t)b * H + h) * kDL + threadIdx.x * 4;
  *reinterpret_cast<__nv_bfloat162*>(ob) = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  *reinterpret_cast<__nv_bfloat162*>(ob + 2) = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
}

}  // namespace

int mla_splits(const pks_mla_args& a) {
  const int tiles = (a.k + kTile - 1) / kTile;
  // no CTA takes more tiles than its row table holds
  const int least = (tiles + kMaxCtaTiles - 1) / kMaxCtaTiles;
  int s = a.splits;
  if (s <= 0) {
    const int per = a.B > 0 ? device_sm_count() / (2 * a.B) : 1;
    s = per < 1 ? 1 : per;
    if (s > tiles) s = tiles;
  }
  if (s < least) s = least;
  return s < 1 ? 1 : s;
}

MlaLayout mla_layout(const pks_mla_args& a) {
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  MlaLayout L{};
  L.splits = mla_splits(a);
  size_t off = 0;
  L.err = off;
  off = up(off + 16);
  const size_t nslot = (size_t)a.B * (size_t)L.splits * (size_t)a.H;
  L.part_ml = off;
  off = up(off + (L.splits > 1 ? sizeof(float2) * nslot : 0));
  L.part_o = off;
  off = up(off + (L.splits > 1 ? sizeof(float) * nslot * kDL : 0));
  L.total = off;
  return L;
}

cudaError_t launch_mla(const pks_mla_args& a, const MlaLayout& L, cudaStream_t s) {
  static bool configured[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (!configured[dev & 63]) {
    e = cudaFuncSetAttribute(k_mla_attention, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    configured[dev & 63] = true;
  }
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  const float scale = a.sm_scale > 0.f ? a.sm_scale : 1.f / sqrtf((float)kDK);
  const float scale_log2 = scale * 1.4426950408889634f;
  const int grid = a.B * L.splits * 2;
  // programmatic dependent launches: the MLA kernel's set-up overlaps the
  // previous kernel (the top-k of the step), the merge's launch the MLA tail
  e = launch_ex(k_mla_attention, dim3(grid), dim3(kThreads), kSmemBytes, s, /*pdl=*/true,
                /*coop=*/false, a.seq_lens, a.block_table,
                static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.kv),
                a.topk_idx, reinterpret_cast<float2*>(ws + L.part_ml),
                reinterpret_cast<float*>(ws + L.part_o), static_cast<__nv_bfloat16*>(a.out),
                reinterpret_cast<int32_t*>(ws + L.err), a.B, a.H, a.page_size, a.max_pages,
                a.num_pages, a.k, a.trim ? 1 : 0, L.splits, scale_log2,
                a.wait_limit > 0 ? (long long)a.wait_limit : kWaitCycles);
  if (e != cudaSuccess || L.splits == 1) return e;
  return launch_ex(k_mla_merge, dim3(a.H, a.B), dim3(128), 0, s, /*pdl=*/true, /*coop=*/false,
                   reinterpret_cast<const float2*>(ws + L.part_ml),
                   reinterpret_cast<const float*>(ws + L.part_o),
                   static_cast<__nv_bfloat16*>(a.out), a.H, L.splits);
}

}  // namespace pks
