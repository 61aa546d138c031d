// Batch-invariant GEMM on the 5th-generation tensor cores
// ("Deterministic and bit-exact inference", *technical*: matrix
// multiplication made batch-invariant by fixing each output element's
// reduction order regardless of batch size).
//
// C[M][N] = A[M][K] . W[N][K]^T, bf16 inputs, fp32 accumulation in tensor
// memory (TMEM), one rounding at the store.
//
// Per output element the arithmetic is fixed by (N, K) alone:
//  * every tile is 128 rows of A by BN rows of W; each K step is one
//    tcgen05.mma of shape 128 x BN x 16 (kind::f16, bf16 in, fp32 accumulate),
//    four per 64-wide K block, K blocks in ascending order;
//  * one pipeline stage carries j consecutive 64-wide K blocks of A and W,
//    each brought by a single 3-D TMA copy (a CTA keeps only a few copies in
//    flight, so each copy must be large for the weight stream to keep up);
//  * K is cut into `splits` equal, contiguous ranges (splits depends on N and
//    K only); the CTAs of one cluster compute one range each.  Row m belongs
//    to rank m % splits, which adds the fp32 partials of its rows in rank
//    order p0 + p1 + ...: for tiles of up to kPushMaxRows rows every rank
//    pushes them into the owner's shared memory, for taller tiles every rank
//    stages its own and the owners read them over DSMEM -- no atomics, no
//    batch-dependent split;
//  * TMA brings in the rows of A that exist (M rounded up to 8, at most 128);
//    the tile rows beyond them feed accumulator rows that are never stored.
// Row i therefore meets the same instructions in the same order for every M,
// at whichever lane of the tile it lands.
//
// Roles inside a 128-thread CTA: thread 0 issues TMA loads into a ring of
// shared-memory stages (mbarrier full/empty pairs), thread 32 issues the MMAs
// and commits each stage back to the producer, and all four warps read the
// accumulator out of TMEM (warp w owns TMEM lanes 32w..32w+31 = tile rows).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "rope.cuh"

namespace kinv {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;  // one 128-byte swizzle row of bf16
constexpr int kGemmThreads = 128;
constexpr int A_STAGE = BM * BK * 2;
constexpr int kRopeTabRows = 4;  // owned rows up to which the RoPE angles are formed ahead
constexpr int kPushMaxRows = 8;  // split-K tiles of more rows have the owners pull the partials
constexpr int kMaxSplits = 8;     // K splits (cluster size) at most
// mbarriers after the ring: full and empty per stage, done, recv, one
// "ready" per K-split rank (push path), "read" (pull path) and a spare that
// keeps the count even (what follows them must stay 16-byte aligned)
__host__ __device__ constexpr int bar_count(int stages) { return 2 * stages + 4 + kMaxSplits; }
static_assert(bar_count(1) % 2 == 0 && bar_count(2) % 2 == 0, "an even barrier count keeps the tables 16-byte aligned");

// tcgen05 instruction descriptor, kind::f16: fp32 accumulate (bits 4-5 = 1),
// A and B bf16 (bits 7-9 = 1, bits 10-12 = 1), both K-major, N >> 3 at bits
// 17-22, M >> 4 at bits 24-28.
template <int BN>
__device__ constexpr uint32_t instr_desc() {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(BN >> 3) << 17) |
         (static_cast<uint32_t>(BM >> 4) << 24);
}

// Shared-memory matrix descriptor for a K-major tile written by TMA with
// 128-byte swizzling: start address >> 4, leading offset 1 (unused for this
// layout), stride between 8-row groups 1024 bytes, descriptor version 1,
// layout type 2 (128-byte swizzle).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t addr) {
  return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (1ull << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ float silu_times(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// bf16(x + v) for a bf16 x given by its bits and the projection's fp32
// result v: the residual stream is the stored tensor, the projection's output
// is never stored, so the sum is rounded once
__device__ __forceinline__ float residual_add(uint32_t x_bits, float v) {
  const float x = __uint_as_float((x_bits & 0xFFFFu) << 16);
  return __bfloat162float(__float2bfloat16_rn(__fadd_rn(x, v)));
}

__host__ __device__ constexpr int rope_pre_bytes(int own_rows, int D, int BN) {
  return own_rows * (8 + (D / 2) * 8) + BN * 2;
}

// The QKV projection's epilogue: the bf16 result rows (as a plain store would
// round them) go through RoPE with the optional QK-norm (the same per-head
// arithmetic as kinv_rope_append) straight into q and the KV cache.
struct RopeEpilogue {
  int on;
  int D, Hq, Hkv;
  __nv_bfloat16* q_out;  // [M][Hq][D]
  __nv_bfloat16* k_cache;
  __nv_bfloat16* v_cache;
  int64_t seq_stride, tok_stride;
  const int32_t* seq;
  const int32_t* pos;
  const __nv_bfloat16* q_norm;
  const __nv_bfloat16* k_norm;
  float eps;
  RopeFreqs freqs;
};

struct GemmArgs {
  void* C;
  int64_t ldc;
  int M, N;
  int k_stages;  // pipeline stages per split (each j K blocks)
  int j;         // 64-wide K blocks per stage
  int a_rows;    // rows of A that TMA brings in per tile (the rest of the 128 are never stored)
  int a_blk;     // bytes of one K block of A in shared memory (a_rows * 128)
  int c_f32;
  int swiglu;    // output silu(gate) * up: tile columns [0, BN/2) gate, [BN/2, BN) up
  int stages;
  int splits;
  int own_rows;  // split-K: rows a rank owns at most (ceil(a_rows / splits))
  int pull;      // split-K with more than kPushMaxRows rows: owners read the partials instead of receiving them
  int ring_bytes;  // the stage ring, or more when the epilogue's receive slots need it
  int* status;
  RopeEpilogue rope;
  // RMSNorm folded in (kinv_gemm_fusion): scale row m by 1/rms from the
  // partial sums of squares row_ss[m][0 .. row_ss_tiles)
  const float* row_ss;
  int row_ss_tiles;
  int norm_dim;
  float eps;
  // residual: resid[m][n] = bf16(resid[m][n] + product), and the new
  // row's sum of squares over this tile's 128 columns -> ss_out[m][n0 / 128]
  __nv_bfloat16* resid;
  int64_t ld_resid;
  float* ss_out;
  // the large-M tile kernel's schedule
  int kb_per_split;  // 64-wide K blocks of one K range
  int tiles_m, tiles_n;
  int n_tail;        // the last n_tail tiles (M fastest) run as two 128-wide halves each
};

// Rows [0, n) of a staged tile (bf16, row stride BN) are rows row_of(r) of the
// QKV projection; each warp takes (row, head) items of the tile.
// What the RoPE epilogue needs besides the staged rows, gathered ahead of the
// epilogue into shared memory (decode: few owned rows): each row's position
// and sequence, the cos and sin of its angles, and the norm gains of the
// tile's heads.
struct RopePre {
  int* pos;             // [n]
  int* seq;             // [n]
  float* cs;            // [n][D/2][2]
  __nv_bfloat16* nw;    // [BN / D][D]: the gains of the tile's q/k heads
};

// `pre` (nullable): RopePre for the staged rows; otherwise everything is read
// or formed here.
template <int D, int BN, typename RowOf>
__device__ __forceinline__ void rope_rows(const __nv_bfloat16* stage, const RopePre* pre, int n,
                                          int n0, int M, const RopeEpilogue& e, RowOf row_of) {
  constexpr int HALF = D / 2;
  constexpr int P = D / 64;
  constexpr int HPT = BN / D;  // heads per tile
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int idx = warp; idx < n * HPT; idx += kGemmThreads / 32) {
    const int r = idx / HPT, j = idx % HPT;
    const int m = row_of(r);
    if (m >= M) continue;
    const int h = n0 / D + j;
    const int p = pre ? pre->pos[r] : e.pos[m];
    const int sq = pre ? pre->seq[r] : e.seq[m];
    const int64_t tok = static_cast<int64_t>(sq) * e.seq_stride + static_cast<int64_t>(p) * e.tok_stride;
    const __nv_bfloat16* src = stage + r * BN + j * D;
    if (h >= e.Hq + e.Hkv) {  // value head: the bits as stored
      __nv_bfloat16* dst = e.v_cache + tok + (h - e.Hq - e.Hkv) * D;
      for (int c = lane; c < D / 8; c += 32)
        reinterpret_cast<uint4*>(dst)[c] = reinterpret_cast<const uint4*>(src)[c];
      continue;
    }
    float a[P], b[P], c[P], sn[P];
#pragma unroll
    for (int q = 0; q < P; ++q) {
      a[q] = __bfloat162float(src[lane * P + q]);
      b[q] = __bfloat162float(src[HALF + lane * P + q]);
      if (pre) {
        c[q] = pre->cs[(r * HALF + lane * P + q) * 2];
        sn[q] = pre->cs[(r * HALF + lane * P + q) * 2 + 1];
      } else {
        rope_angle(p, e.freqs.inv_freq[lane * P + q], c[q], sn[q]);
      }
    }
    const __nv_bfloat16* g = h < e.Hq ? e.q_norm : e.k_norm;
    if (g && pre) g = pre->nw + j * D;
    __nv_bfloat16* dst = h < e.Hq ? e.q_out + (static_cast<int64_t>(m) * e.Hq + h) * D
                                  : e.k_cache + tok + (h - e.Hq) * D;
    rope_norm_rotate<D>(a, b, c, sn, g, e.eps, lane, dst);
  }
}

// Head size dispatch (a tile holds whole heads: the plan's tiles are 128 wide).
template <int BN, typename RowOf>
__device__ __forceinline__ void rope_dispatch(const __nv_bfloat16* stage, const RopePre* pre, int n,
                                              int n0, int M, const RopeEpilogue& e, RowOf row_of) {
  if constexpr (BN % 128 == 0) {
    if (e.D == 128) {
      rope_rows<128, BN>(stage, pre, n, n0, M, e, row_of);
      return;
    }
  }
  if constexpr (BN % 64 == 0) rope_rows<64, BN>(stage, pre, n, n0, M, e, row_of);
}

template <int BN>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                const GemmArgs args) {
  constexpr int W_BLK = BN * BK * 2;  // one K block of W
  constexpr uint32_t TMEM_COLS = BN < 32 ? 32 : BN;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int stages = args.stages;
  const int jb = args.j;
  const int W_STAGE = W_BLK * jb;
  // A stages first, then W stages; a stage holds j K blocks back to back.
  // An MMA reads 128 rows (16 KB) from the start of an A block; when a block
  // holds fewer rows the extra rows come from the memory that follows
  // (inside this block's shared memory) and only feed accumulator rows that
  // are never stored.
  const int a_blk = args.a_blk;
  const int a_stride = a_blk * jb;
  unsigned char* a_st = base;
  unsigned char* w_st = base + stages * a_stride;
  // split-K partials received from every rank, [splits][own_rows][BN] fp32,
  // over the stage ring (idle by then in every rank of the cluster)
  float* recv = reinterpret_cast<float*>(base);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + args.ring_bytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + bar_count(stages));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // split-K RoPE epilogue with few owned rows (decode): what it needs is
  // gathered by the otherwise idle warps 2 and 3 while the weights stream
  const bool use_pre = args.rope.on && args.splits > 1 && args.own_rows <= kRopeTabRows;
  RopePre pre{};
  // the tables after the barriers take 16-byte vector accesses
  unsigned char* tail = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(tmem_slot + 4) + 15) & ~static_cast<uintptr_t>(15));
  if (use_pre) {
    pre.pos = reinterpret_cast<int*>(tail);
    pre.seq = pre.pos + args.own_rows;
    pre.cs = reinterpret_cast<float*>(pre.seq + args.own_rows);
    pre.nw = reinterpret_cast<__nv_bfloat16*>(pre.cs + args.own_rows * args.rope.D);
    tail += rope_pre_bytes(args.own_rows, args.rope.D, BN);
  }
  float* row_inv = reinterpret_cast<float*>(tail);  // [BM] when row_ss is given
  if (args.row_ss) tail += BM * 4;
  float* red4 = reinterpret_cast<float*>(tail);     // [own_rows][4] for the split residual
  const bool push = args.splits > 1 && !args.pull;
  // the residual rows a rank owns ([own_rows][BN] bf16, either split-K
  // path), read while the weights stream
  const bool use_resid_pre = args.splits > 1 && args.resid != nullptr;
  uint16_t* resid_pre = reinterpret_cast<uint16_t*>(red4 + (use_resid_pre ? args.own_rows * 4 : 0));
  auto full_bar = [&](int s) { return smem_addr(bars + s); };
  auto empty_bar = [&](int s) { return smem_addr(bars + stages + s); };
  const uint32_t done_bar = smem_addr(bars + 2 * stages);
  const uint32_t recv_bar = smem_addr(bars + 2 * stages + 1);
  // ready_bar(q) completes when rank q's MMAs are done (its ring may take partials)
  auto ready_bar = [&](int q) { return smem_addr(bars + 2 * stages + 2 + q); };
  // read_bar completes when every rank has read this rank's staged rows (pull path)
  const uint32_t read_bar = smem_addr(bars + 2 * stages + 2 + kMaxSplits);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int splits = args.splits;
  const int rank = splits > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int m0 = blockIdx.y * BM;  // M tiles of one N tile are launch neighbours: W is read once
  const int n0 = blockIdx.z * BN;
  const int rows_here = args.M - m0 < BM ? args.M - m0 : BM;
  const uint32_t stage_bytes = static_cast<uint32_t>(a_stride + W_STAGE);
  const int k_stages = args.k_stages;
  const int kb0 = rank * k_stages * jb;  // first K block of this split

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(done_bar, 1);
    mbar_init(recv_bar, 1);
    if (push)
      for (int q = 0; q < splits; ++q) mbar_init(ready_bar(q), 1);
    if (splits > 1 && args.pull) mbar_init(read_bar, splits);
    *abort_flag = 0;
    fence_mbar_init();
    if (splits > 1) {
      // the partial rows this rank owns arrive from every other rank
      const int owned = rank < rows_here ? (rows_here - rank + splits - 1) / splits : 0;
      mbar_arrive_expect_tx(recv_bar, static_cast<uint32_t>((splits - 1) * owned * BN * 4));
    }
  }
  if (warp == 0) tmem_alloc(smem_addr(tmem_slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // dependents are released once this block holds its tensor memory (a
  // dependent block that allocated first would wait on this grid)
  pdl_launch_dependents();
  // push path: the peers' barriers are initialised before any remote arrive
  // or store reaches them (the matching wait comes at the epilogue)
  if (push) cluster_arrive_relaxed();

  int issued = 0;
  if (warp == 0) {
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmW)) : "memory");
      const uint64_t pol_a = l2_policy_evict_last();   // A is re-read by every N tile
      const uint64_t pol_w = l2_policy_evict_first();  // each W tile is read once
      // The weights do not depend on the kernel before this one: the first
      // ring's worth of W tiles is requested before waiting for it; A (its
      // output) only after.  Fresh stages need no empty-barrier wait.
      const int pre = k_stages < stages ? k_stages : stages;
      for (int kt = 0; kt < pre; ++kt) {
        mbar_arrive_expect_tx(full_bar(kt), stage_bytes);
        tma_load_3d(smem_addr(w_st + kt * W_STAGE), &tmW, 0, n0, kb0 + kt * jb, full_bar(kt), pol_w);
      }
      pdl_wait();
      for (int kt = 0; kt < pre; ++kt)
        tma_load_3d(smem_addr(a_st + kt * a_stride), &tmA, 0, m0, kb0 + kt * jb, full_bar(kt), pol_a);
      issued = pre;
      for (int kt = pre; kt < k_stages; ++kt) {
        const int s = kt % stages;
        const uint32_t ph = (kt / stages) & 1u;
        if (*abort_flag ||
            !mbar_wait_bounded(empty_bar(s), ph ^ 1u, args.status, DEV_TIMEOUT_GEMM_PRODUCER)) {
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(full_bar(s), stage_bytes);
        const int kb = kb0 + kt * jb;
        tma_load_3d(smem_addr(a_st + s * a_stride), &tmA, 0, m0, kb, full_bar(s), pol_a);
        tma_load_3d(smem_addr(w_st + s * W_STAGE), &tmW, 0, n0, kb, full_bar(s), pol_w);
        ++issued;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = instr_desc<BN>();
      for (int kt = 0; kt < k_stages; ++kt) {
        const int s = kt % stages;
        const uint32_t ph = (kt / stages) & 1u;
        if (*abort_flag ||
            !mbar_wait_bounded(full_bar(s), ph, args.status, DEV_TIMEOUT_GEMM_MMA)) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int jj = 0; jj < jb; ++jj) {
          const uint32_t a_addr = smem_addr(a_st + s * a_stride + jj * a_blk);
          const uint32_t w_addr = smem_addr(w_st + s * W_STAGE + jj * W_BLK);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            umma_bf16(tmem, sdesc_sw128(a_addr + kk * 32), sdesc_sw128(w_addr + kk * 32), idesc,
                      (kt | jj | kk) != 0 ? 1u : 0u);
          }
        }
        umma_commit(empty_bar(s));  // the stage is free once these MMAs have read it
      }
      umma_commit(done_bar);
    }
    __syncwarp();
  }

  if (use_pre && warp >= 2) {
    const RopeEpilogue& e = args.rope;
    const int t2 = threadIdx.x - 64;
    // the gains of the tile's q and k heads (weights: no dependency wait)
    for (int idx = t2; idx < BN; idx += 64) {
      const int h = n0 / e.D + idx / e.D;
      const __nv_bfloat16* g = h < e.Hq ? e.q_norm : (h < e.Hq + e.Hkv ? e.k_norm : nullptr);
      pre.nw[idx] = g ? g[idx % e.D] : __float2bfloat16_rn(0.f);
    }
    pdl_wait();  // positions are written by earlier kernels
    const int half = e.D / 2;
    const int owned = rank < rows_here ? (rows_here - rank + splits - 1) / splits : 0;
    for (int i = t2; i < owned; i += 64) {
      pre.pos[i] = e.pos[m0 + i * splits + rank];
      pre.seq[i] = e.seq[m0 + i * splits + rank];
    }
    for (int idx = t2; idx < owned * half; idx += 64) {
      const int i = idx / half, jj = idx % half;
      rope_angle(e.pos[m0 + i * splits + rank], e.freqs.inv_freq[jj], pre.cs[idx * 2], pre.cs[idx * 2 + 1]);
    }
  }

  if (args.row_ss && warp >= 2) {
    // 1 / rms of this tile's rows from the partial sums of squares (written by
    // the kernel that produced A), tiles added in ascending order
    pdl_wait();
    for (int r = threadIdx.x - 64; r < rows_here; r += 64) {
      const float* ss = args.row_ss + static_cast<int64_t>(m0 + r) * args.row_ss_tiles;
      float acc = ss[0];
      for (int q = 1; q < args.row_ss_tiles; ++q) acc = __fadd_rn(acc, ss[q]);
      row_inv[r] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(acc, static_cast<float>(args.norm_dim)),
                                                       args.eps)));
    }
  }

  if (use_resid_pre && warp >= 2) {
    // the residual rows this rank owns (written by earlier kernels)
    pdl_wait();
    constexpr int CH = BN / 8;  // 16-byte chunks per row
    const int owned = rank < rows_here ? (rows_here - rank + splits - 1) / splits : 0;
    for (int idx = threadIdx.x - 64; idx < owned * CH; idx += 64) {
      const int i = idx / CH, c = idx % CH;
      const __nv_bfloat16* src = args.resid + static_cast<int64_t>(m0 + i * splits + rank) * args.ld_resid + n0 + c * 8;
      *reinterpret_cast<uint4*>(resid_pre + i * BN + c * 8) = *reinterpret_cast<const uint4*>(src);
    }
  }

  // push path: the peers' barriers are initialised (every rank arrived at its
  // start), waited for here, before the MMAs finish
  if (push) {
    __syncwarp();
    cluster_wait();
  }

  // ---- epilogue
  const bool ok = mbar_wait_bounded(done_bar, 0, args.status, DEV_TIMEOUT_GEMM_EPILOGUE);
  __syncwarp();
  tc_fence_after();
  const int row_local = warp * 32 + lane;
  const int m = m0 + row_local;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  const bool good = ok && !*abort_flag && k_stages > 0;
  constexpr int HALF = BN / 2;
  if (args.row_ss) __syncthreads();  // row_inv is complete
  const float inv_here = args.row_ss && row_local < rows_here ? row_inv[row_local] : 1.0f;
  auto scale32 = [&](uint32_t (&v)[32]) {
    if (args.row_ss) {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__fmul_rn(__uint_as_float(v[j]), inv_here));
    }
  };

  if (splits == 1 && args.swiglu) {
    // columns [0, BN/2) of the tile are gate features n0/2 .. n0/2 + BN/2 - 1,
    // columns [BN/2, BN) the up features for the same ids
#pragma unroll 1
    for (int c0 = 0; c0 < HALF && good; c0 += 32) {
      uint32_t gv[32], uv[32];
      tmem_ld32(lane_base + c0, gv);
      tmem_ld32(lane_base + HALF + c0, uv);
      scale32(gv);
      scale32(uv);
      if (m < args.M) {
        __nv_bfloat16* crow = static_cast<__nv_bfloat16*>(args.C) + m * args.ldc + n0 / 2 + c0;
#pragma unroll
        for (int j = 0; j < 32; j += 8) {
          uint4 o;
          o.x = pack_bf16(silu_times(__uint_as_float(gv[j + 0]), __uint_as_float(uv[j + 0])),
                          silu_times(__uint_as_float(gv[j + 1]), __uint_as_float(uv[j + 1])));
          o.y = pack_bf16(silu_times(__uint_as_float(gv[j + 2]), __uint_as_float(uv[j + 2])),
                          silu_times(__uint_as_float(gv[j + 3]), __uint_as_float(uv[j + 3])));
          o.z = pack_bf16(silu_times(__uint_as_float(gv[j + 4]), __uint_as_float(uv[j + 4])),
                          silu_times(__uint_as_float(gv[j + 5]), __uint_as_float(uv[j + 5])));
          o.w = pack_bf16(silu_times(__uint_as_float(gv[j + 6]), __uint_as_float(uv[j + 6])),
                          silu_times(__uint_as_float(gv[j + 7]), __uint_as_float(uv[j + 7])));
          *reinterpret_cast<uint4*>(crow + j) = o;
        }
      }
    }
  } else if (splits == 1) {
    __nv_bfloat16* stage = reinterpret_cast<__nv_bfloat16*>(base);  // rope: the ring is idle now
    float ss_row = 0.f;  // residual: the new row's sum of squares over the tile, in column order
    if (good) {
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(lane_base + c0, r);
        scale32(r);
        if (args.resid) {
          if (m < args.M) {
            __nv_bfloat16* xrow = args.resid + m * args.ld_resid + n0 + c0;
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
              const uint4 xv = *reinterpret_cast<const uint4*>(xrow + j);
              const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
              uint32_t ow[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const float s0 = residual_add(xw[q] & 0xFFFFu, __uint_as_float(r[j + 2 * q]));
                const float s1 = residual_add(xw[q] >> 16, __uint_as_float(r[j + 2 * q + 1]));
                ss_row = fmaf(s0, s0, ss_row);
                ss_row = fmaf(s1, s1, ss_row);
                ow[q] = pack_bf16(s0, s1);
              }
              *reinterpret_cast<uint4*>(xrow + j) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
            }
          }
        } else if (args.rope.on) {
          if (m < args.M) {
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
              uint4 o;
              o.x = pack_bf16(__uint_as_float(r[j + 0]), __uint_as_float(r[j + 1]));
              o.y = pack_bf16(__uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
              o.z = pack_bf16(__uint_as_float(r[j + 4]), __uint_as_float(r[j + 5]));
              o.w = pack_bf16(__uint_as_float(r[j + 6]), __uint_as_float(r[j + 7]));
              *reinterpret_cast<uint4*>(stage + row_local * BN + c0 + j) = o;
            }
          }
        } else if (m < args.M) {
          if (args.c_f32) {
            float* crow = static_cast<float*>(args.C) + m * args.ldc + n0 + c0;
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              if (n0 + c0 + j < args.N)
                *reinterpret_cast<uint4*>(crow + j) = make_uint4(r[j], r[j + 1], r[j + 2], r[j + 3]);
            }
          } else {
            __nv_bfloat16* crow = static_cast<__nv_bfloat16*>(args.C) + m * args.ldc + n0 + c0;
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
              if (n0 + c0 + j < args.N) {
                uint4 o;
                o.x = pack_bf16(__uint_as_float(r[j + 0]), __uint_as_float(r[j + 1]));
                o.y = pack_bf16(__uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
                o.z = pack_bf16(__uint_as_float(r[j + 4]), __uint_as_float(r[j + 5]));
                o.w = pack_bf16(__uint_as_float(r[j + 6]), __uint_as_float(r[j + 7]));
                *reinterpret_cast<uint4*>(crow + j) = o;
              }
            }
          }
        }
      }
    }
    if (args.resid && good && m < args.M)
      args.ss_out[static_cast<int64_t>(m) * (args.N / BN) + n0 / BN] = ss_row;
    if (args.rope.on) {
      __syncthreads();
      if (good) {
        auto row_of = [&](int r) { return m0 + r; };
        rope_dispatch<BN>(stage, nullptr, rows_here, n0, args.M, args.rope, row_of);
      }
    }
  } else if (args.pull) {
    // Constant split-K, more than kPushMaxRows rows: every rank stages its fp32 partial rows in
    // its own (idle) ring; after a cluster barrier the owner of row m (rank
    // m % splits) reads that row from every rank -- a warp per row, lane l
    // taking columns 4l .. 4l + 3 -- and adds them in rank order.  The
    // arithmetic of every output is the push path's below, so a row's bits do
    // not depend on which path its M took.
    if constexpr (BN == kGemmThreads) {
      constexpr int LDP = BN + 4;  // padded row of the staged partials (floats)
      float* part = reinterpret_cast<float*>(base);  // this rank's MMAs are done: its ring is idle
      if (warp * 32 < rows_here) {
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(lane_base + c0, r);
          if (row_local < rows_here) {
#pragma unroll
            for (int q = 0; q < 32; q += 4)
              *reinterpret_cast<uint4*>(part + row_local * LDP + c0 + q) = make_uint4(r[q], r[q + 1], r[q + 2], r[q + 3]);
          }
        }
      }
      cluster_sync();  // every rank's partials are staged
      const int owned = rank < rows_here ? (rows_here - rank + splits - 1) / splits : 0;
      __nv_bfloat16* stage = reinterpret_cast<__nv_bfloat16*>(part + args.a_rows * LDP);  // rope rows
      // The output of owned row i from a4, its sum over the ranks (warp-wide:
      // lane l holds columns 4l .. 4l + 3).
      auto emit = [&](int i, float (&a4)[4]) {
        const int ml = i * splits + rank;
        const int mm = m0 + ml;
        if (args.row_ss) {
          const float inv = row_inv[ml];
#pragma unroll
          for (int e = 0; e < 4; ++e) a4[e] = __fmul_rn(a4[e], inv);
        }
        if (args.swiglu) {
          // lanes 0..15 hold gate columns 4l.., lanes 16..31 the matching up columns
          float u4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) u4[e] = __shfl_down_sync(0xffffffffu, a4[e], 16);
          if (lane < 16) {
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(args.C) + mm * args.ldc + n0 / 2 + 4 * lane;
            *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16(silu_times(a4[0], u4[0]), silu_times(a4[1], u4[1])),
                                                        pack_bf16(silu_times(a4[2], u4[2]), silu_times(a4[3], u4[3])));
          }
        } else if (args.resid) {
          __nv_bfloat16* xp = args.resid + mm * args.ld_resid + n0 + 4 * lane;
          const uint2 xv = *reinterpret_cast<const uint2*>(resid_pre + i * BN + 4 * lane);
          float sv[4];
          sv[0] = residual_add(xv.x & 0xFFFFu, a4[0]);
          sv[1] = residual_add(xv.x >> 16, a4[1]);
          sv[2] = residual_add(xv.y & 0xFFFFu, a4[2]);
          sv[3] = residual_add(xv.y >> 16, a4[3]);
          *reinterpret_cast<uint2*>(xp) = make_uint2(pack_bf16(sv[0], sv[1]), pack_bf16(sv[2], sv[3]));
          // the push path's per-warp butterfly over columns 32w .. 32w + 31
          // (xor 16, 8, 4, 2, 1 on the column index) in this layout: column
          // 4l + e -> lane bits 2..0 and element bits 1..0
          float q4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) q4[e] = __fmul_rn(sv[e], sv[e]);
#pragma unroll
          for (int o = 4; o > 0; o >>= 1) {
#pragma unroll
            for (int e = 0; e < 4; ++e) q4[e] = __fadd_rn(q4[e], __shfl_xor_sync(0xffffffffu, q4[e], o));
          }
          {
            const float t0 = __fadd_rn(q4[0], q4[2]), t1 = __fadd_rn(q4[1], q4[3]);
            q4[0] = __fadd_rn(t0, t1);
          }
          // group totals at lanes 0, 8, 16, 24; then the four groups in order
          const float g1 = __shfl_sync(0xffffffffu, q4[0], 8);
          const float g2 = __shfl_sync(0xffffffffu, q4[0], 16);
          const float g3 = __shfl_sync(0xffffffffu, q4[0], 24);
          if (lane == 0)
            args.ss_out[static_cast<int64_t>(mm) * (args.N / BN) + n0 / BN] =
                __fadd_rn(__fadd_rn(__fadd_rn(q4[0], g1), g2), g3);
        } else if (args.rope.on) {
          *reinterpret_cast<uint2*>(stage + i * BN + 4 * lane) =
              make_uint2(pack_bf16(a4[0], a4[1]), pack_bf16(a4[2], a4[3]));
        } else if (args.c_f32) {
          if (n0 + 4 * lane < args.N)
            *reinterpret_cast<float4*>(static_cast<float*>(args.C) + mm * args.ldc + n0 + 4 * lane) =
                make_float4(a4[0], a4[1], a4[2], a4[3]);
        } else {
          if (n0 + 4 * lane < args.N)
            *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(args.C) + mm * args.ldc + n0 + 4 * lane) =
                make_uint2(pack_bf16(a4[0], a4[1]), pack_bf16(a4[2], a4[3]));
        }
      };
      // Warp w takes the owned rows i = w (mod 4).  DSMEM reads are long
      // latency, so a warp requests the partials of a batch of rows (16 reads
      // per lane) before it adds any; each row's sum is still formed in rank
      // order.  The split count is a power of two up to kMaxSplits.
      auto pull_rows = [&](auto splits_c) {
        constexpr int S = decltype(splits_c)::value;
        constexpr int RB = 16 / S;  // rows per batch
        for (int i0 = warp; i0 < owned && good; i0 += 4 * RB) {
          float4 v[RB][S];
#pragma unroll
          for (int u = 0; u < RB; ++u) {
            if (i0 + 4 * u < owned) {
              const uint32_t off = smem_addr(part + ((i0 + 4 * u) * S + rank) * LDP + 4 * lane);
#pragma unroll
              for (int q = 0; q < S; ++q) v[u][q] = ld_dsmem_v4(map_to_rank(off, q));
            }
          }
#pragma unroll
          for (int u = 0; u < RB; ++u) {
            if (i0 + 4 * u < owned) {
              float4 acc = v[u][0];
#pragma unroll
              for (int q = 1; q < S; ++q) {
                acc.x = __fadd_rn(acc.x, v[u][q].x);
                acc.y = __fadd_rn(acc.y, v[u][q].y);
                acc.z = __fadd_rn(acc.z, v[u][q].z);
                acc.w = __fadd_rn(acc.w, v[u][q].w);
              }
              float a4[4] = {acc.x, acc.y, acc.z, acc.w};
              emit(i0 + 4 * u, a4);
            }
          }
        }
      };
      if (splits == 2)
        pull_rows(std::integral_constant<int, 2>{});
      else if (splits == 4)
        pull_rows(std::integral_constant<int, 4>{});
      else
        pull_rows(std::integral_constant<int, kMaxSplits>{});
      __syncthreads();  // this rank's reads of the peers' rows are done
      if (warp == 0 && lane < splits) mbar_arrive_cluster_relaxed(map_to_rank(read_bar, lane));
      if (args.rope.on && good) {
        auto row_of = [&](int r) { return m0 + r * splits + rank; };
        rope_dispatch<BN>(stage, use_pre ? &pre : nullptr, owned, n0, args.M, args.rope, row_of);
      }
    }
  } else {
    // Constant split-K.  Rank r pushes row m of its partial tile into slot r of
    // the owner rank m % splits (row index m / splits there; the owner's own
    // rows are plain local stores); once all slots of its rows are in, the
    // owner adds them in rank order and stores.  The slots overlay the
    // owner's ring: a row goes out once the owner has announced (ready_bar)
    // that its MMAs are done.
    if (warp == 0 && lane < splits) mbar_arrive_cluster_relaxed(map_to_rank(ready_bar(rank), lane));
    const int own_rows = args.own_rows;
    if (warp * 32 < rows_here) {
      const bool row_ok = row_local < rows_here;
      const int owner = row_ok ? row_local % splits : rank;
      float* dst_local = recv + (rank * own_rows + (row_ok ? row_local / splits : 0)) * BN;
      const uint32_t dst_base = map_to_rank(smem_addr(dst_local), owner);
      const uint32_t dst_bar = map_to_rank(recv_bar, owner);
      bool can = true;
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 64) {
        uint32_t r[64];
        tmem_ld64(lane_base + c0, r);
        if (c0 == 0 && row_ok && owner != rank)
          can = mbar_wait_cluster_relaxed_bounded(ready_bar(owner), 0, args.status, DEV_TIMEOUT_GEMM_EPILOGUE);
        if (!can) continue;
        if (row_ok && owner == rank) {
#pragma unroll
          for (int q = 0; q < 64; q += 4)
            *reinterpret_cast<uint4*>(dst_local + c0 + q) = make_uint4(r[q], r[q + 1], r[q + 2], r[q + 3]);
        } else if (row_ok) {
#pragma unroll
          for (int q = 0; q < 64; q += 4)
            st_async_v4(dst_base + (c0 + q) * 4, r[q], r[q + 1], r[q + 2], r[q + 3], dst_bar);
        }
      }
    }
    __syncthreads();  // this rank's own rows are in place
    const int owned = rank < rows_here ? (rows_here - rank + splits - 1) / splits : 0;
    const bool got =
        __syncthreads_and(mbar_wait_bounded(recv_bar, 0, args.status, DEV_TIMEOUT_GEMM_EPILOGUE));
    if (good && got) {
      const int slot = own_rows * BN;
      if (args.swiglu) {
        // gate column f and up column HALF + f of each owned row
        for (int idx = threadIdx.x; idx < owned * HALF; idx += kGemmThreads) {
          const int i = idx / HALF, f = idx % HALF;
          const float* src = recv + i * BN + f;
          float g = src[0], u = src[HALF];
          for (int q = 1; q < splits; ++q) {
            g = __fadd_rn(g, src[q * slot]);
            u = __fadd_rn(u, src[q * slot + HALF]);
          }
          if (args.row_ss) {
            const float inv = row_inv[i * splits + rank];
            g = __fmul_rn(g, inv);
            u = __fmul_rn(u, inv);
          }
          const int mm = m0 + i * splits + rank;
          static_cast<__nv_bfloat16*>(args.C)[mm * args.ldc + n0 / 2 + f] =
              __float2bfloat16_rn(silu_times(g, u));
        }
      } else if (args.resid) {
        if constexpr (BN == kGemmThreads) {
          // thread t takes column t of each owned row in turn; the row's sum of
          // squares: a fixed butterfly in each warp, then the four warps in order
          for (int i = 0; i < owned; ++i) {
            const int col = threadIdx.x;
            const float* src = recv + i * BN + col;
            float acc = src[0];
            for (int q = 1; q < splits; ++q) acc = __fadd_rn(acc, src[q * slot]);
            const int mm = m0 + i * splits + rank;
            __nv_bfloat16* xp = args.resid + mm * args.ld_resid + n0 + col;
            const float sv = residual_add(resid_pre[i * BN + col], acc);
            *xp = __float2bfloat16_rn(sv);
            float sq = __fmul_rn(sv, sv);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sq = __fadd_rn(sq, __shfl_xor_sync(0xffffffffu, sq, o));
            if (lane == 0) red4[i * 4 + warp] = sq;
          }
          __syncthreads();
          for (int i = threadIdx.x; i < owned; i += kGemmThreads) {
            const float sq = __fadd_rn(__fadd_rn(__fadd_rn(red4[i * 4], red4[i * 4 + 1]), red4[i * 4 + 2]),
                                       red4[i * 4 + 3]);
            args.ss_out[static_cast<int64_t>(m0 + i * splits + rank) * (args.N / BN) + n0 / BN] = sq;
          }
        }
      } else {
        // rope: the owned rows are staged after the receive slots
        __nv_bfloat16* stage = reinterpret_cast<__nv_bfloat16*>(recv + splits * slot);
        for (int idx = threadIdx.x; idx < owned * BN; idx += kGemmThreads) {
          const int i = idx / BN, col = idx % BN;
          const int nn = n0 + col;
          if (nn >= args.N) continue;
          const float* src = recv + i * BN + col;
          float acc = src[0];
          for (int q = 1; q < splits; ++q) acc = __fadd_rn(acc, src[q * slot]);
          if (args.row_ss) acc = __fmul_rn(acc, row_inv[i * splits + rank]);
          const int mm = m0 + i * splits + rank;
          if (args.rope.on)
            stage[i * BN + col] = __float2bfloat16_rn(acc);
          else if (args.c_f32)
            static_cast<float*>(args.C)[mm * args.ldc + nn] = acc;
          else
            static_cast<__nv_bfloat16*>(args.C)[mm * args.ldc + nn] = __float2bfloat16_rn(acc);
        }
        if (args.rope.on) {
          __syncthreads();
          auto row_of = [&](int r) { return m0 + r * splits + rank; };
          rope_dispatch<BN>(stage, use_pre ? &pre : nullptr, owned, n0, args.M, args.rope, row_of);
        }
      }
    }
  }

  // ---- teardown
  if (push && warp == 0 && lane < splits) {
    // no peer may still be about to arrive on this block's barriers
    mbar_wait_cluster_relaxed_bounded(ready_bar(lane), 0, args.status, DEV_TIMEOUT_GEMM_EPILOGUE);
  }
  if (splits > 1 && args.pull && threadIdx.x == 0) {
    // every rank has read this block's staged rows (and will not touch it again)
    mbar_wait_cluster_relaxed_bounded(read_bar, 0, args.status, DEV_TIMEOUT_GEMM_EPILOGUE);
  }
  if (*abort_flag && warp == 0 && lane == 0) {
    // give loads still in flight a bounded chance to land before the block exits
    for (int kt = issued - stages > 0 ? issued - stages : 0; kt < issued; ++kt)
      mbar_wait_bounded(full_bar(kt % stages), (kt / stages) & 1u, nullptr, 0);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// The large-M schedule: gemm_kernel's per-element arithmetic, laid out for the
// tensor cores instead of the weight stream.
//
// For an output element gemm_kernel forms, for each of the plan's `splits`
// contiguous K ranges r, a partial p_r accumulated from zero over the range's
// 64-wide K blocks in ascending order (16-deep bf16 MMA steps, fp32 in TMEM),
// then ((p_0 + p_1) + p_2) + ... in fp32 in rank order, then the epilogue.
// With many rows the K split only costs: every 128-row tile goes through a
// cluster reduction whose epilogue does not overlap the MMAs.  Here one CTA
// per SM walks a static list of 128 x 256 output tiles (row tiles fastest, so
// the CTAs in flight share a few weight tiles in L2); for each tile it forms
// the K ranges one after another in two TMEM accumulators used in turn, and
// eight epilogue warps fold each finished range into a running sum held in
// registers while the tensor cores work on the next range (or the next
// tile).  The sums are the same fp32 operations in the same order as
// gemm_kernel's, and so are the epilogues (row scale, SwiGLU, residual add and
// its sums of squares, bf16 / fp32 store), so a row has the same bits through
// either kernel.
//
// Roles (320 threads): warps 0-7 fold and store (warp w reads TMEM lanes
// 32 (w % 4) .. + 31 = tile rows, columns 128 (w / 4) .. + 127), warp 8 lane 0
// issues the TMA loads, warp 9 lane 0 the MMAs (warp 9 also owns the TMEM
// allocation: two accumulators of 256 columns).
constexpr int kTilesBN = 256;
constexpr int kTilesThreads = 320;
constexpr int kTilesEpiWarps = 8;
constexpr int kTilesABytes = BM * BK * 2;        // 16 KB
constexpr int kTilesBBytes = kTilesBN * BK * 2;  // 32 KB
constexpr int kTilesStage = kTilesABytes + kTilesBBytes;  // per K block of a stage
__host__ __device__ constexpr int tiles_bar_count(int stages) { return 2 * stages + 5; }

// The push path's sum of squares of a 128-column tile (per warp a fixed xor
// butterfly over 32 columns, then the four warps in order), formed by one
// thread that holds the tile's 128 values: the same pairs in the same order.
__device__ __forceinline__ float sumsq_butterfly128(const float (&v)[128]) {
  float g4[4];
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    float t[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      t[i] = __fadd_rn(__fmul_rn(v[32 * g + i], v[32 * g + i]), __fmul_rn(v[32 * g + i + 16], v[32 * g + i + 16]));
#pragma unroll
    for (int i = 0; i < 8; ++i) t[i] = __fadd_rn(t[i], t[i + 8]);
#pragma unroll
    for (int i = 0; i < 4; ++i) t[i] = __fadd_rn(t[i], t[i + 4]);
#pragma unroll
    for (int i = 0; i < 2; ++i) t[i] = __fadd_rn(t[i], t[i + 2]);
    g4[g] = __fadd_rn(t[0], t[1]);
  }
  return __fadd_rn(__fadd_rn(__fadd_rn(g4[0], g4[1]), g4[2]), g4[3]);
}

template <int J>
__global__ void __launch_bounds__(kTilesThreads, 1)
    gemm_tiles_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                      const __grid_constant__ CUtensorMap tmW_half, const GemmArgs args) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int stages = args.stages;
  // a stage holds J consecutive K blocks (one TMA copy of A and one of W):
  // [J][128][64] of A, then [J][256][64] of W
  constexpr int j = J;
  constexpr int stage_bytes = J * kTilesStage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + stages * stage_bytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + tiles_bar_count(stages));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  auto full_bar = [&](int st) { return smem_addr(bars + st); };
  auto empty_bar = [&](int st) { return smem_addr(bars + stages + st); };
  auto acc_full = [&](int b) { return smem_addr(bars + 2 * stages + b); };
  auto acc_empty = [&](int b) { return smem_addr(bars + 2 * stages + 2 + b); };
  const uint32_t done_bar = smem_addr(bars + 2 * stages + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles_m = args.tiles_m;
  // the work list: whole 128 x 256 tiles, then the last n_tail tiles as
  // 128 x 128 halves, so the last round over the SMs is a short one (a
  // 128 x 128 MMA gives each element the bits of the 128 x 256 one)
  const int tiles_full = tiles_m * args.tiles_n - args.n_tail;
  const int n_tiles = tiles_full + 2 * args.n_tail;
  auto tile_at = [&](int v, int& m0, int& n0) -> bool {  // true: a 128-wide half
    int t = v, hf = 0;
    const bool narrow = v >= tiles_full;
    if (narrow) {
      t = tiles_full + ((v - tiles_full) >> 1);
      hf = (v - tiles_full) & 1;
    }
    m0 = (t % tiles_m) * BM;
    n0 = (t / tiles_m) * kTilesBN + hf * 128;
    return narrow;
  };
  const int splits = args.splits, kbs = args.kb_per_split;

  if (threadIdx.x == 0) {
    for (int st = 0; st < stages; ++st) {
      mbar_init(full_bar(st), 1);
      mbar_init(empty_bar(st), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full(b), 1);
      mbar_init(acc_empty(b), kTilesEpiWarps);
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) tmem_alloc(smem_addr(tmem_slot), 2 * kTilesBN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Dependent kernels may be scheduled only once every block of this grid
  // holds its tensor memory: a dependent block that took the columns first
  // would wait for this grid while this block waited for the columns.
  pdl_launch_dependents();
  // everything this kernel reads may come from the kernels before it
  pdl_wait();

  if (warp == 8) {
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmW)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmW_half)) : "memory");
      const uint64_t pol_a = l2_policy_evict_last();
      const uint64_t pol_w = l2_policy_evict_last();  // a weight tile serves every row tile
      int it = 0;
      bool stop = false;
      for (int t = blockIdx.x; t < n_tiles && !stop; t += gridDim.x) {
        int m0, n0;
        const bool narrow = tile_at(t, m0, n0);
        for (int kb = 0; kb < splits * kbs; kb += j, ++it) {
          const int st = it % stages;
          const uint32_t ph = (it / stages) & 1u;
          if (*abort_flag ||
              !mbar_wait_bounded(empty_bar(st), ph ^ 1u, args.status, DEV_TIMEOUT_GEMM_PRODUCER)) {
            *abort_flag = 1;
            stop = true;
            break;
          }
          mbar_arrive_expect_tx(full_bar(st), narrow ? J * (kTilesABytes + kTilesBBytes / 2) : stage_bytes);
          unsigned char* sa = base + st * stage_bytes;
          tma_load_3d(smem_addr(sa), &tmA, 0, m0, kb, full_bar(st), pol_a);
          tma_load_3d(smem_addr(sa + j * kTilesABytes), narrow ? &tmW_half : &tmW, 0, n0, kb, full_bar(st), pol_w);
        }
      }
      // loads still in flight (only after an abort) land before the block exits
      for (int q = it - stages > 0 ? it - stages : 0; q < it; ++q)
        mbar_wait_bounded(full_bar(q % stages), (q / stages) & 1u, nullptr, 0);
    }
    __syncwarp();
  } else if (warp == 9) {
    if (lane == 0) {
      int it = 0, seq = 0;
      bool stop = false;
      for (int t = blockIdx.x; t < n_tiles && !stop; t += gridDim.x) {
        int m0, n0;
        // one 128 x 256 MMA per 16-deep step, or 128 x 128 for a half tile
        // (whose W blocks, 128 rows each, lie 16 KB apart in the stage)
        const bool narrow = tile_at(t, m0, n0);
        const uint32_t idesc = narrow ? instr_desc<128>() : instr_desc<kTilesBN>();
        const uint32_t w_blk = narrow ? kTilesBBytes / 2 : kTilesBBytes;
        for (int r = 0; r < splits && !stop; ++r, ++seq) {
          const int b = seq & 1;
          const uint32_t aph = (seq >> 1) & 1u;
          if (*abort_flag ||
              !mbar_wait_bounded(acc_empty(b), aph ^ 1u, args.status, DEV_TIMEOUT_GEMM_MMA)) {
            *abort_flag = 1;
            stop = true;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + static_cast<uint32_t>(b * kTilesBN);
          for (int k = 0; k < kbs; k += j, ++it) {
            const int st = it % stages;
            const uint32_t ph = (it / stages) & 1u;
            if (*abort_flag || !mbar_wait_bounded(full_bar(st), ph, args.status, DEV_TIMEOUT_GEMM_MMA)) {
              *abort_flag = 1;
              stop = true;
              break;
            }
            tc_fence_after();
            const uint32_t a0 = smem_addr(base + st * stage_bytes);
            const uint32_t b0 = a0 + j * kTilesABytes;
#pragma unroll
            for (int h = 0; h < J; ++h) {  // the stage's K blocks, ascending
              const uint32_t a_addr = a0 + h * kTilesABytes, b_addr = b0 + h * w_blk;
#pragma unroll
              for (int kk = 0; kk < BK / 16; ++kk) {
                const uint32_t accum = (k | h | kk) != 0 ? 1u : 0u;
                umma_bf16(d, sdesc_sw128(a_addr + kk * 32), sdesc_sw128(b_addr + kk * 32), idesc, accum);
              }
            }
            umma_commit(empty_bar(st));
          }
          if (!stop) umma_commit(acc_full(b));
        }
      }
      // every MMA issued has completed before the TMEM is released
      umma_commit(done_bar);
      mbar_wait_bounded(done_bar, 0, args.status, DEV_TIMEOUT_GEMM_MMA);
    }
    __syncwarp();
  } else {
    const int lg = warp & 3;       // TMEM lane group: tile rows 32 lg .. 32 lg + 31
    const int half = warp >> 2;    // tile columns 128 half .. 128 half + 127
    const int row = lg * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(lg * 32) << 16) + half * 128;
    int seq = 0;
    bool stop = false;
    for (int t = blockIdx.x; t < n_tiles && !stop; t += gridDim.x) {
      int m0, n0;
      const bool narrow = tile_at(t, m0, n0);
      const int m = m0 + row;
      const int nc0 = n0 + half * 128;  // this thread's first column
      const bool cols = !narrow || half == 0;  // a half tile has columns for warps 0-3 only
      float acc[128];
      for (int r = 0; r < splits; ++r, ++seq) {
        const int b = seq & 1;
        const uint32_t aph = (seq >> 1) & 1u;
        const bool ok = mbar_wait_bounded(acc_full(b), aph, args.status, DEV_TIMEOUT_GEMM_EPILOGUE);
        if (__any_sync(0xffffffffu, !ok || *abort_flag)) {
          *abort_flag = 1;
          stop = true;
          break;
        }
        tc_fence_after();
        if (cols) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t v[32];
            tmem_ld32(lane_base + b * kTilesBN + c * 32, v);
#pragma unroll
            for (int j = 0; j < 32; ++j)
              acc[c * 32 + j] = r == 0 ? __uint_as_float(v[j]) : __fadd_rn(acc[c * 32 + j], __uint_as_float(v[j]));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(acc_empty(b)) : "memory");
      }
      if (stop || !cols || m >= args.M || nc0 >= args.N) continue;
      if (args.row_ss) {
        // 1 / rms of the row from its partial sums of squares, tiles in order
        const float* ss = args.row_ss + static_cast<int64_t>(m) * args.row_ss_tiles;
        float sacc = ss[0];
        for (int q = 1; q < args.row_ss_tiles; ++q) sacc = __fadd_rn(sacc, ss[q]);
        const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(sacc, static_cast<float>(args.norm_dim)),
                                                              args.eps)));
#pragma unroll
        for (int j = 0; j < 128; ++j) acc[j] = __fmul_rn(acc[j], inv);
      }
      if (args.swiglu) {
        // columns 0..63 of this half are gate features nc0/2 .. nc0/2 + 63,
        // columns 64..127 the up features for the same ids
        __nv_bfloat16* crow = static_cast<__nv_bfloat16*>(args.C) + m * args.ldc + nc0 / 2;
#pragma unroll
        for (int j = 0; j < 64; j += 8) {
          uint4 o;
          o.x = pack_bf16(silu_times(acc[j + 0], acc[64 + j + 0]), silu_times(acc[j + 1], acc[64 + j + 1]));
          o.y = pack_bf16(silu_times(acc[j + 2], acc[64 + j + 2]), silu_times(acc[j + 3], acc[64 + j + 3]));
          o.z = pack_bf16(silu_times(acc[j + 4], acc[64 + j + 4]), silu_times(acc[j + 5], acc[64 + j + 5]));
          o.w = pack_bf16(silu_times(acc[j + 6], acc[64 + j + 6]), silu_times(acc[j + 7], acc[64 + j + 7]));
          *reinterpret_cast<uint4*>(crow + j) = o;
        }
      } else if (args.resid) {
        __nv_bfloat16* xrow = args.resid + m * args.ld_resid + nc0;
        float ss_seq = 0.f;  // one range: the column-order FMA chain of the unsplit epilogue
#pragma unroll
        for (int j = 0; j < 128; j += 8) {
          const uint4 xv = *reinterpret_cast<const uint4*>(xrow + j);
          const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
          uint32_t ow[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float s0 = residual_add(xw[q] & 0xFFFFu, acc[j + 2 * q]);
            const float s1 = residual_add(xw[q] >> 16, acc[j + 2 * q + 1]);
            acc[j + 2 * q] = s0;
            acc[j + 2 * q + 1] = s1;
            ss_seq = fmaf(s0, s0, ss_seq);
            ss_seq = fmaf(s1, s1, ss_seq);
            ow[q] = pack_bf16(s0, s1);
          }
          *reinterpret_cast<uint4*>(xrow + j) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
        }
        args.ss_out[static_cast<int64_t>(m) * (args.N / 128) + nc0 / 128] =
            splits > 1 ? sumsq_butterfly128(acc) : ss_seq;
      } else if (args.c_f32) {
        float* crow = static_cast<float*>(args.C) + m * args.ldc + nc0;
#pragma unroll
        for (int j = 0; j < 128; j += 4)
          if (nc0 + j < args.N)
            *reinterpret_cast<float4*>(crow + j) = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
      } else {
        __nv_bfloat16* crow = static_cast<__nv_bfloat16*>(args.C) + m * args.ldc + nc0;
#pragma unroll
        for (int j = 0; j < 128; j += 8) {
          if (nc0 + j < args.N) {
            uint4 o;
            o.x = pack_bf16(acc[j + 0], acc[j + 1]);
            o.y = pack_bf16(acc[j + 2], acc[j + 3]);
            o.z = pack_bf16(acc[j + 4], acc[j + 5]);
            o.w = pack_bf16(acc[j + 6], acc[j + 7]);
            *reinterpret_cast<uint4*>(crow + j) = o;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * kTilesBN);
  }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// A row-major [rows][cols] bf16 matrix seen as 3-D (64 columns, rows,
// cols / 64 K blocks): one box is box_rows rows by kblocks K blocks, landing
// in shared memory as kblocks consecutive [box_rows][64] swizzled blocks.
bool make_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int64_t ld,
              int box_rows, int kblocks) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(BK), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(cols / BK)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2, BK * 2};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows),
                             static_cast<cuuint32_t>(kblocks)};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct Plan {
  int bn, splits;
  int j;            // K blocks per pipeline stage
  int smem_budget;  // bytes of stage ring per block (sets blocks per SM)
};

// The tile width and the K split depend on (N, K) only -- never on M -- so
// every row meets the same reduction order whatever the batch.  Decode GEMMs
// stream the weights once and are bound by how many bytes are in flight: a
// CTA keeps only a few TMA copies outstanding, so there are many CTAs (a K
// split bringing the count to at least 256) and each copy carries two K
// blocks (32 KB of W).  How many K blocks a copy carries and how deep the
// ring is do not change the order of the MMAs; they are set per launch.
Plan plan_for(int N, int K) {
  const int kb = K / BK;
  Plan p{128, 1, 2, 112 * 1024};
  const int tiles = (N + p.bn - 1) / p.bn;
  int s = 1;
  while (s < 8 && tiles * s < 256 && kb % (4 * s) == 0) s *= 2;
  p.splits = s;
  if ((kb / s) % 2) p.j = 1;
  return p;
}

// Shared memory a block may use so that `ctas` blocks are resident at once
// (at most four per SM: four 128-column TMEM tiles).
int ring_cap(long long ctas) {
  const int sms = sm_count() > 0 ? sm_count() : 1;
  long long per_sm = (ctas + sms - 1) / sms;
  per_sm = per_sm < 1 ? 1 : (per_sm > 4 ? 4 : per_sm);
  return static_cast<int>(smem_per_sm() / per_sm) - smem_reserved_per_block() - 1024 - 256;
}

size_t smem_bytes(int stages, int ring_bytes, int tab_bytes) {
  return 1024 + static_cast<size_t>(ring_bytes) + bar_count(stages) * 8 + 16 + 16 + tab_bytes;
}

template <int BN>
kinv_status launch_gemm(const CUtensorMap& ta, const CUtensorMap& tw, GemmArgs a, int budget,
                        int grid_y, int grid_z, cudaStream_t stream) {
  // The ring is sized so that the whole grid is resident at once (a second
  // wave would double the time of a weight stream): at most the SM's shared
  // memory divided by the blocks each SM must hold, within the plan's budget
  // and 2..8 stages.  It must also hold the split-K receive slots (they reuse
  // it), and the 128 rows one MMA reads from the start of the last A block
  // must stay inside the block's shared memory.
  a.own_rows = (a.a_rows + a.splits - 1) / a.splits;
  // split-K with more than kPushMaxRows rows: owners pull the partials (coalesced reads) from
  // rows staged in each rank's ring; otherwise ranks push into receive slots
  a.pull = a.splits > 1 && a.a_rows > kPushMaxRows && BN == kGemmThreads ? 1 : 0;
  // split-K receive slots (or the staged partial rows), plus the staged bf16
  // rows of the RoPE epilogue
  const int recv_bytes = a.pull ? a.a_rows * (BN + 4) * 4 + (a.rope.on ? a.own_rows * BN * 2 : 0)
                         : a.splits > 1 ? a.splits * a.own_rows * BN * 4 +
                                            (a.rope.on ? a.own_rows * BN * 2 : 0)
                                        : (a.rope.on ? a.a_rows * BN * 2 : 0);
  // what the block keeps after the ring and its barriers: the RoPE inputs,
  // 1/rms per row, the split residual's partial sums and its residual rows
  const bool split = a.splits > 1;
  const int tab_bytes = (a.rope.on && split && a.own_rows <= kRopeTabRows
                             ? rope_pre_bytes(a.own_rows, a.rope.D, BN)
                             : 0) +
                        (a.row_ss ? BM * 4 : 0) +
                        (a.resid && split ? a.own_rows * 16 + a.own_rows * BN * 2 : 0);
  const int cap = ring_cap(static_cast<long long>(a.splits) * grid_y * grid_z) - tab_bytes;
  const int limit = budget < cap ? budget : cap;
  const int stage = a.a_blk * a.j + BN * BK * 2 * a.j;
  int stages = limit / stage;
  stages = stages < 2 ? 2 : (stages > 8 ? 8 : stages);
  while ((stages - 1) * a.a_blk * a.j + (a.j - 1) * a.a_blk + A_STAGE > stages * stage) ++stages;
  a.stages = stages;
  // the epilogue's receive slots reuse the ring and may run past it
  a.ring_bytes = stages * stage > recv_bytes ? stages * stage : (recv_bytes + 15) / 16 * 16;
  const size_t smem = smem_bytes(stages, a.ring_bytes, tab_bytes);
  if (smem > static_cast<size_t>(max_smem_optin())) return KINV_ERR_UNSUPPORTED;
  // the opt-in limit is raised (once per context) to the largest request seen
  const kinv_status attr = ensure_smem(reinterpret_cast<const void*>(gemm_kernel<BN>), smem);
  if (attr != KINV_OK) return attr;
  return launch_kernel(gemm_kernel<BN>, dim3(a.splits, grid_y, grid_z), dim3(kGemmThreads), smem,
                       stream, static_cast<unsigned>(a.splits), ta, tw, a);
}

// The large-M schedule: one CTA per SM (at most one per tile), the stage ring
// as deep as shared memory allows.
template <int J>
kinv_status launch_gemm_tiles_j(const void* A, int64_t lda, const void* W, int64_t ldw, int K, GemmArgs a,
                              cudaStream_t stream) {
  a.kb_per_split = K / BK / a.splits;
  a.tiles_m = (a.M + BM - 1) / BM;
  a.tiles_n = (a.N + kTilesBN - 1) / kTilesBN;
  a.j = J;
  CUtensorMap ta, tw, tw_half;
  if (!make_map(&ta, A, a.M, K, lda, BM, a.j) || !make_map(&tw, W, a.N, K, ldw, kTilesBN, a.j) ||
      !make_map(&tw_half, W, a.N, K, ldw, kTilesBN / 2, a.j))
    return KINV_ERR_CUDA;
  const int stage = a.j * kTilesStage;
  const int avail = max_smem_optin() - 1024 - 256;
  int stages = avail / stage;
  stages = stages > 6 ? 6 : stages;
  if (stages < 2) return KINV_ERR_UNSUPPORTED;
  a.stages = stages;
  const size_t smem = 1024 + static_cast<size_t>(stages) * stage + tiles_bar_count(stages) * 8 + 16;
  const kinv_status attr = ensure_smem(reinterpret_cast<const void*>(gemm_tiles_kernel<J>), smem);
  if (attr != KINV_OK) return attr;
  const long long tiles = static_cast<long long>(a.tiles_m) * a.tiles_n;
  const int sms = sm_count() > 0 ? sm_count() : 1;
  // a partial last round over the SMs (at least one full round before it)
  // runs its tiles as halves when they fit one round: it then takes about
  // as long as half a tile's operands take to stream in
  const long long rem = tiles % sms;
  a.n_tail = tiles >= sms && rem > 0 && 2 * rem <= sms ? static_cast<int>(rem) : 0;
  const long long work = tiles + a.n_tail;
  const int grid = static_cast<int>(work < sms ? work : sms);
  return launch_kernel(gemm_tiles_kernel<J>, dim3(grid), dim3(kTilesThreads), smem, stream, 1, ta, tw, tw_half,
                       a);
}

// Two K blocks per TMA copy: a CTA keeps only a few copies in flight, and
// larger copies (measured, per launch) took the 4096-row projections 7-12 %
// faster, and the shapes with at most about one tile per CTA (QKV and O at
// 512-1024 rows) 9-14 %; with a few tiles per CTA at 512-1024 rows (gate/up,
// and down with K = 12288) the deeper ring of single blocks was 2-5 %
// faster.  The MMAs keep their order.
kinv_status launch_gemm_tiles(const void* A, int64_t lda, const void* W, int64_t ldw, int K, GemmArgs a,
                              cudaStream_t stream) {
  const long long tiles_m = (a.M + BM - 1) / BM;
  const long long tiles = tiles_m * ((a.N + kTilesBN - 1) / kTilesBN);
  const int sms = sm_count() > 0 ? sm_count() : 1;
  const bool two = (K / BK / a.splits) % 2 == 0 && (tiles_m >= 16 || (2 * tiles <= 3LL * sms && K < 8192));
  return two ? launch_gemm_tiles_j<2>(A, lda, W, ldw, K, a, stream)
             : launch_gemm_tiles_j<1>(A, lda, W, ldw, K, a, stream);
}

// Whether the tile schedule runs a call (else the cluster split-K schedule).
// Either gives a row the same bits, so this is a speed choice.  Measured on
// the GB300 (cold L2, per launch): with one K range per tile the tile
// schedule is faster from 129 rows; with a K split, from 384 rows (768 for
// K >= 8192, whose tiles' K loops are long and few at that size).
#ifndef KINV_TILES_MIN_ROWS
#define KINV_TILES_MIN_ROWS 129
#endif
bool use_tiles(int M, int K, int splits) {
  if (M < KINV_TILES_MIN_ROWS) return false;
  if (splits == 1) return true;
  return M >= (K >= 8192 ? 768 : 384);
}

}  // namespace
}  // namespace kinv

using namespace kinv;

namespace kinv {
namespace {
kinv_status gemm_impl(const void* A, int64_t lda, const void* W, int64_t ldw, void* C, int64_t ldc,
                      kinv_dtype c_dtype, int M, int N, int K, bool swiglu, const RopeEpilogue* rope,
                      const kinv_gemm_fusion* fu, cudaStream_t stream) {
  if (M < 0 || N <= 0 || K <= 0) return KINV_ERR_INVALID_ARG;
  if (c_dtype != KINV_BF16 && c_dtype != KINV_F32) return KINV_ERR_INVALID_ARG;
  if (M == 0) return KINV_OK;
  const bool resid = fu && fu->resid;
  if (fu && fu->row_ss && (fu->row_ss_tiles <= 0 || fu->norm_dim <= 0 || !(fu->eps >= 0.f)))
    return KINV_ERR_INVALID_ARG;
  if (resid) {
    // the residual stream is the only output; a producing projection takes no row scale
    if (!fu->ss_out || swiglu || rope || fu->ld_resid < N || fu->row_ss) return KINV_ERR_INVALID_ARG;
    if (N % 128) return KINV_ERR_UNSUPPORTED;
    if (!aligned16(fu->resid) || fu->ld_resid % 8) return KINV_ERR_ALIGNMENT;
    rope = nullptr;
  }
  const bool no_c = rope || resid;
  if (!A || !W || (!C && !no_c)) return KINV_ERR_INVALID_ARG;
  if (K % BK || N % 16 || ((swiglu || rope) && (N % 128 || c_dtype != KINV_BF16)))
    return KINV_ERR_UNSUPPORTED;
  if (lda < K || ldw < K || (!no_c && ldc < (swiglu ? N / 2 : N))) return KINV_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(W) || (!no_c && !aligned16(C)) || lda % 8 || ldw % 8 ||
      (!no_c && (c_dtype == KINV_BF16 ? ldc % 8 : ldc % 4)))
    return KINV_ERR_ALIGNMENT;
  const Plan p = plan_for(N, K);  // 128-wide tiles: 64 gate and the matching 64 up columns
  const int grid_y = (M + BM - 1) / BM;
  const int grid_z = (N + p.bn - 1) / p.bn;
  if (grid_y > 65535 || grid_z > 65535) return KINV_ERR_UNSUPPORTED;
  // A tiles carry only the rows that exist (a multiple of 8 up to 128): zero
  // fill of a mostly empty box is slow, and the tile rows beyond M feed only
  // accumulator rows that are never stored.
  const int a_rows = M >= BM ? BM : ((M + 7) / 8) * 8;
  // K blocks per stage only set how the loads are grouped, not the order of
  // the MMAs: two per stage when two such stages fit the one-wave ring
  const long long ctas = static_cast<long long>(p.splits) * grid_y * grid_z;
  const int two_stages = 2 * (a_rows * BK * 2 + p.bn * BK * 2) * p.j;
  const int j = two_stages <= ring_cap(ctas) && two_stages <= p.smem_budget ? p.j : 1;
  CUtensorMap ta, tw;
  if (!make_map(&ta, A, M, K, lda, a_rows, j) || !make_map(&tw, W, N, K, ldw, p.bn, j))
    return KINV_ERR_CUDA;
  GemmArgs a;
  a.C = C;
  a.ldc = ldc;
  a.M = M;
  a.N = N;
  a.k_stages = K / BK / p.splits / j;
  a.j = j;
  a.a_rows = a_rows;
  a.a_blk = a_rows * BK * 2;
  a.c_f32 = c_dtype == KINV_F32;
  a.swiglu = swiglu ? 1 : 0;
  a.stages = 0;
  a.splits = p.splits;
  a.own_rows = 0;
  a.pull = 0;
  a.ring_bytes = 0;
  a.status = device_status_word();
  a.rope = rope ? *rope : RopeEpilogue{};
  a.rope.on = rope ? 1 : 0;
  a.row_ss = fu ? fu->row_ss : nullptr;
  a.row_ss_tiles = fu ? fu->row_ss_tiles : 0;
  a.norm_dim = fu ? fu->norm_dim : 0;
  a.eps = fu ? fu->eps : 0.f;
  a.resid = resid ? static_cast<__nv_bfloat16*>(fu->resid) : nullptr;
  a.ld_resid = resid ? fu->ld_resid : 0;
  a.ss_out = resid ? fu->ss_out : nullptr;
  a.kb_per_split = 0;
  a.tiles_m = a.tiles_n = 0;
  a.n_tail = 0;
  if (!rope && use_tiles(M, K, p.splits))
    return launch_gemm_tiles(A, lda, W, ldw, K, a, stream);
  switch (p.bn) {
    case 128: return launch_gemm<128>(ta, tw, a, p.smem_budget, grid_y, grid_z, stream);
    default: return KINV_ERR_UNSUPPORTED;
  }
}
}  // namespace
}  // namespace kinv

extern "C" kinv_status kinv_gemm(const void* A, int64_t lda, const void* W, int64_t ldw, void* C,
                                 int64_t ldc, kinv_dtype c_dtype, int M, int N, int K,
                                 kinv_stream stream) {
  return kinv::gemm_impl(A, lda, W, ldw, C, ldc, c_dtype, M, N, K, false, nullptr, nullptr, stream);
}

extern "C" kinv_status kinv_gemm_fused(const void* A, int64_t lda, const void* W, int64_t ldw, void* C,
                                       int64_t ldc, kinv_dtype c_dtype, int M, int N, int K,
                                       const kinv_gemm_fusion* fusion, kinv_stream stream) {
  return kinv::gemm_impl(A, lda, W, ldw, C, ldc, c_dtype, M, N, K, false, nullptr, fusion, stream);
}

extern "C" kinv_status kinv_gemm_swiglu(const void* A, int64_t lda, const void* W_gu, int64_t ldw,
                                        void* act, int64_t ld_act, int M, int F, int K,
                                        const kinv_gemm_fusion* fusion, kinv_stream stream) {
  if (F <= 0 || F % 64) return F <= 0 ? KINV_ERR_INVALID_ARG : KINV_ERR_UNSUPPORTED;
  if (fusion && fusion->resid) return KINV_ERR_INVALID_ARG;
  return kinv::gemm_impl(A, lda, W_gu, ldw, act, ld_act, KINV_BF16, M, 2 * F, K, true, nullptr, fusion,
                         stream);
}

extern "C" kinv_status kinv_gemm_qkv_rope(const void* A, int64_t lda, const void* W_qkv, int64_t ldw,
                                          void* q_out, void* k_cache, void* v_cache,
                                          int64_t seq_stride, int64_t tok_stride, const int32_t* seq,
                                          const int32_t* pos, const void* q_norm, const void* k_norm,
                                          float eps, int M, int Hq, int Hkv, int D, int K,
                                          float rope_base, const kinv_gemm_fusion* fusion,
                                          kinv_stream stream) {
  if (M < 0 || Hq <= 0 || Hkv <= 0 || K <= 0 || !(rope_base > 0.f) || !(eps >= 0.f))
    return KINV_ERR_INVALID_ARG;
  if (M == 0) return KINV_OK;
  if (!q_out || !k_cache || !v_cache || !seq || !pos) return KINV_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return KINV_ERR_UNSUPPORTED;
  if (tok_stride < static_cast<int64_t>(Hkv) * D || seq_stride < 0) return KINV_ERR_INVALID_ARG;
  if (!aligned16(q_out) || !aligned16(k_cache) || !aligned16(v_cache) || seq_stride % 8 ||
      tok_stride % 8)
    return KINV_ERR_ALIGNMENT;
  kinv::RopeEpilogue e{};
  e.D = D;
  e.Hq = Hq;
  e.Hkv = Hkv;
  e.q_out = static_cast<__nv_bfloat16*>(q_out);
  e.k_cache = static_cast<__nv_bfloat16*>(k_cache);
  e.v_cache = static_cast<__nv_bfloat16*>(v_cache);
  e.seq_stride = seq_stride;
  e.tok_stride = tok_stride;
  e.seq = seq;
  e.pos = pos;
  e.q_norm = static_cast<const __nv_bfloat16*>(q_norm);
  e.k_norm = static_cast<const __nv_bfloat16*>(k_norm);
  e.eps = eps;
  for (int i = 0; i < D / 2; ++i)
    e.freqs.inv_freq[i] = std::pow(static_cast<double>(rope_base), -2.0 * i / D);
  const int N = (Hq + 2 * Hkv) * D;
  if (fusion && fusion->resid) return KINV_ERR_INVALID_ARG;
  return kinv::gemm_impl(A, lda, W_qkv, ldw, nullptr, N, KINV_BF16, M, N, K, false, &e, fusion, stream);
}
