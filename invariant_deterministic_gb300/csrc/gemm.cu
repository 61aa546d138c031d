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
//  * K is cut into `splits` equal, contiguous ranges (splits depends on N and
//    K only); the CTAs of one cluster compute one range each, and the partial
//    sums are added in rank order p0 + p1 + ... through distributed shared
//    memory -- no atomics, no batch-dependent split;
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

#include <mutex>

#include "common.cuh"

namespace kinv {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;  // one 128-byte swizzle row of bf16
constexpr int kGemmThreads = 128;
constexpr int A_STAGE = BM * BK * 2;

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

struct GemmArgs {
  void* C;
  int64_t ldc;
  int M, N;
  int k_tiles;  // 64-wide K blocks per split
  int a_rows;   // rows of A that TMA brings in per tile (the rest of the 128 are never stored)
  int a_stride; // bytes between A stages (a_rows * 128)
  int c_f32;
  int swiglu;   // output silu(gate) * up: tile columns [0, 32) gate, [32, 64) up
  int stages;
  int splits;
  int* status;
};

template <int BN>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                const GemmArgs args) {
  constexpr int W_STAGE = BN * BK * 2;
  constexpr uint32_t TMEM_COLS = BN < 32 ? 32 : BN;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int stages = args.stages;
  // A stages first, then W stages.  An MMA reads 128 rows (16 KB) from the
  // start of an A stage; when a stage holds fewer rows the extra rows come
  // from the following stages (inside this block's shared memory) and only
  // feed accumulator rows that are never stored.
  const int a_stride = args.a_stride;
  unsigned char* a_st = base;
  unsigned char* w_st = base + stages * a_stride;
  uint64_t* bars = reinterpret_cast<uint64_t*>(w_st + stages * W_STAGE);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * stages + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  auto full_bar = [&](int s) { return smem_addr(bars + s); };
  auto empty_bar = [&](int s) { return smem_addr(bars + stages + s); };
  const uint32_t done_bar = smem_addr(bars + 2 * stages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int splits = args.splits;
  const int rank = splits > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int m0 = blockIdx.y * BM;  // M tiles of one N tile are launch neighbours: W is read once
  const int n0 = blockIdx.z * BN;
  const uint32_t stage_bytes = static_cast<uint32_t>(args.a_rows * BK * 2 + W_STAGE);
  const int k_tiles = args.k_tiles;
  const int kt0 = rank * k_tiles;

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(smem_addr(tmem_slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

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
      const int pre = k_tiles < stages ? k_tiles : stages;
      for (int kt = 0; kt < pre; ++kt) {
        mbar_arrive_expect_tx(full_bar(kt), stage_bytes);
        tma_load_2d(smem_addr(w_st + kt * W_STAGE), &tmW, (kt0 + kt) * BK, n0, full_bar(kt), pol_w);
      }
      pdl_wait();
      for (int kt = 0; kt < pre; ++kt)
        tma_load_2d(smem_addr(a_st + kt * a_stride), &tmA, (kt0 + kt) * BK, m0, full_bar(kt), pol_a);
      issued = pre;
      for (int kt = pre; kt < k_tiles; ++kt) {
        const int s = kt % stages;
        const uint32_t ph = (kt / stages) & 1u;
        if (*abort_flag ||
            !mbar_wait_bounded(empty_bar(s), ph ^ 1u, args.status, DEV_TIMEOUT_GEMM_PRODUCER)) {
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(full_bar(s), stage_bytes);
        const int kx = (kt0 + kt) * BK;
        tma_load_2d(smem_addr(a_st + s * a_stride), &tmA, kx, m0, full_bar(s), pol_a);
        tma_load_2d(smem_addr(w_st + s * W_STAGE), &tmW, kx, n0, full_bar(s), pol_w);
        ++issued;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = instr_desc<BN>();
      for (int kt = 0; kt < k_tiles; ++kt) {
        const int s = kt % stages;
        const uint32_t ph = (kt / stages) & 1u;
        if (*abort_flag ||
            !mbar_wait_bounded(full_bar(s), ph, args.status, DEV_TIMEOUT_GEMM_MMA)) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t a_addr = smem_addr(a_st + s * a_stride);
        const uint32_t w_addr = smem_addr(w_st + s * W_STAGE);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          umma_bf16(tmem, sdesc_sw128(a_addr + kk * 32), sdesc_sw128(w_addr + kk * 32), idesc,
                    (kt | kk) != 0 ? 1u : 0u);
        }
        umma_commit(empty_bar(s));  // the stage is free once these MMAs have read it
      }
      umma_commit(done_bar);
    }
    __syncwarp();
  }

  // ---- epilogue
  const bool ok = mbar_wait_bounded(done_bar, 0, args.status, DEV_TIMEOUT_GEMM_EPILOGUE);
  __syncwarp();
  tc_fence_after();
  const int row_local = warp * 32 + lane;
  const int m = m0 + row_local;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  const bool good = ok && !*abort_flag && k_tiles > 0;

  if (splits == 1 && args.swiglu) {
    // columns [0, 32) of the tile are gate features n0/2 .. n0/2 + 31, columns
    // [32, 64) the up features for the same ids
    if (good) {
      uint32_t gv[32], uv[32];
      tmem_ld32(lane_base, gv);
      tmem_ld32(lane_base + 32, uv);
      if (m < args.M) {
        __nv_bfloat16* crow = static_cast<__nv_bfloat16*>(args.C) + m * args.ldc + n0 / 2;
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
    if (good) {
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(lane_base + c0, r);
        if (m < args.M) {
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
  } else {
    // Constant split-K: park this CTA's fp32 partial tile in its own shared
    // memory (the stage ring is idle now), then rank q reduces columns
    // [q * BN / splits, (q + 1) * BN / splits) of every row present, over all
    // ranks in rank order p0 + p1 + ...
    constexpr int LDR = BN + 1;
    float* red = reinterpret_cast<float*>(base);
    const int rows_here = args.M - m0 < BM ? args.M - m0 : BM;
    if (good && warp * 32 < rows_here) {
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(lane_base + c0, r);
#pragma unroll
        for (int j = 0; j < 32; ++j) red[row_local * LDR + c0 + j] = __uint_as_float(r[j]);
      }
    }
    cluster_sync();
    const int cols_per = BN / splits;
    const int cbase = rank * cols_per;
    if (good && args.swiglu) {
      // rank q forms features [q * 32 / splits, (q + 1) * 32 / splits): their
      // gate column f and up column 32 + f, each summed in rank order
      const int feats_per = 32 / splits;
      const int fbase = rank * feats_per;
      for (int idx = threadIdx.x; idx < rows_here * feats_per; idx += kGemmThreads) {
        const int rl = idx / feats_per;
        const int f = fbase + idx % feats_per;
        const int mm = m0 + rl;
        const uint32_t lg = smem_addr(red + rl * LDR + f);
        const uint32_t lu = smem_addr(red + rl * LDR + 32 + f);
        float pg[8], pu[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (q < splits) {
            pg[q] = ld_dsmem_f32(map_to_rank(lg, q));
            pu[q] = ld_dsmem_f32(map_to_rank(lu, q));
          }
        float g = pg[0], u = pu[0];
#pragma unroll
        for (int q = 1; q < 8; ++q)
          if (q < splits) {
            g = __fadd_rn(g, pg[q]);
            u = __fadd_rn(u, pu[q]);
          }
        static_cast<__nv_bfloat16*>(args.C)[mm * args.ldc + n0 / 2 + f] =
            __float2bfloat16_rn(silu_times(g, u));
      }
    } else if (good) {
      for (int idx = threadIdx.x; idx < rows_here * cols_per; idx += kGemmThreads) {
        const int rl = idx / cols_per;
        const int col = cbase + idx % cols_per;
        const int mm = m0 + rl, nn = n0 + col;
        if (nn >= args.N) continue;
        const uint32_t local = smem_addr(red + rl * LDR + col);
        float part[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (q < splits) part[q] = ld_dsmem_f32(map_to_rank(local, q));
        float acc = part[0];
#pragma unroll
        for (int q = 1; q < 8; ++q)
          if (q < splits) acc = __fadd_rn(acc, part[q]);
        if (args.c_f32)
          static_cast<float*>(args.C)[mm * args.ldc + nn] = acc;
        else
          static_cast<__nv_bfloat16*>(args.C)[mm * args.ldc + nn] = __float2bfloat16_rn(acc);
      }
    }
    cluster_sync();  // no CTA leaves while another still reads its partial
  }

  // ---- teardown
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

bool make_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int64_t ld,
              int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct Plan {
  int bn, splits;
  int smem_budget;  // bytes of stage ring per block (sets blocks per SM)
};

// The tile width and the K split depend on (N, K) only -- never on M -- so
// every row meets the same reduction order whatever the batch.  Measured on
// the decode shapes: three 24 KB stages (three CTAs per SM) beat deeper rings,
// and a split of K into up to four ranks that brings the CTA count to about
// 256 beats both no split and eight ranks.  Wide outputs (the LM head) take
// 128-wide tiles and no split.
Plan plan_for(int N, int K) {
  const int kt = K / BK;
  Plan p{64, 1, 72 * 1024};
  if (N >= 37888) p = Plan{128, 1, 96 * 1024};
  const int tiles = (N + p.bn - 1) / p.bn;
  // a long K (the down projection) takes up to eight ranks and a 48 KB ring
  const bool long_k = K >= 8192;
  const int max_s = long_k ? 8 : 4;
  const int want = long_k ? 512 : 256;
  int s = 1;
  while (s < max_s && tiles * s < want && kt % (2 * s) == 0 && kt / (2 * s) >= 4) s *= 2;
  p.splits = s;
  if (s == 8) p.smem_budget = 48 * 1024;
  return p;
}

template <int BN>
size_t smem_bytes(int stages, int a_stride) {
  return 1024 + static_cast<size_t>(stages) * (a_stride + BN * BK * 2) + (2 * stages + 1) * 8 + 16;
}

template <int BN>
kinv_status launch_gemm(const CUtensorMap& ta, const CUtensorMap& tw, GemmArgs a, int budget,
                        int grid_y, int grid_z, cudaStream_t stream) {
  // As many stages as the budget holds (2..8): small M leaves room for more
  // weight tiles in flight.  The ring must also hold the split-K partial tile
  // and the 128 rows one MMA reads from the start of the last A stage.
  const int stage = a.a_stride + BN * BK * 2;
  int stages = budget / stage;
  stages = stages < 2 ? 2 : (stages > 8 ? 8 : stages);
  while (static_cast<size_t>(stages) * stage < static_cast<size_t>(BM) * (BN + 1) * 4 ||
         (stages - 1) * a.a_stride + A_STAGE > stages * stage)
    ++stages;
  a.stages = stages;
  const size_t smem = smem_bytes<BN>(stages, a.a_stride);
  if (smem > static_cast<size_t>(max_smem_optin())) return KINV_ERR_UNSUPPORTED;
  // the opt-in limit is raised once per device to the largest request seen
  static size_t configured[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return KINV_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (configured[dev] < smem) {
      if (cudaFuncSetAttribute(gemm_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem)) != cudaSuccess)
        return KINV_ERR_CUDA;
      configured[dev] = smem;
    }
  }
  return launch_kernel(gemm_kernel<BN>, dim3(a.splits, grid_y, grid_z), dim3(kGemmThreads), smem,
                       stream, static_cast<unsigned>(a.splits), ta, tw, a);
}

}  // namespace
}  // namespace kinv

using namespace kinv;

namespace kinv {
namespace {
kinv_status gemm_impl(const void* A, int64_t lda, const void* W, int64_t ldw, void* C, int64_t ldc,
                      kinv_dtype c_dtype, int M, int N, int K, bool swiglu, cudaStream_t stream) {
  if (M < 0 || N <= 0 || K <= 0) return KINV_ERR_INVALID_ARG;
  if (c_dtype != KINV_BF16 && c_dtype != KINV_F32) return KINV_ERR_INVALID_ARG;
  if (M == 0) return KINV_OK;
  if (!A || !W || !C) return KINV_ERR_INVALID_ARG;
  if (K % BK || N % 16 || (swiglu && (N % 64 || c_dtype != KINV_BF16))) return KINV_ERR_UNSUPPORTED;
  if (lda < K || ldw < K || ldc < (swiglu ? N / 2 : N)) return KINV_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(W) || !aligned16(C) || lda % 8 || ldw % 8 ||
      (c_dtype == KINV_BF16 ? ldc % 8 : ldc % 4))
    return KINV_ERR_ALIGNMENT;
  Plan p = plan_for(N, K);
  if (swiglu) p.bn = 64;  // a tile holds 32 gate and the matching 32 up columns
  const int grid_y = (M + BM - 1) / BM;
  const int grid_z = (N + p.bn - 1) / p.bn;
  if (grid_y > 65535 || grid_z > 65535) return KINV_ERR_UNSUPPORTED;
  // A tiles carry only the rows that exist (a multiple of 8 up to 128): zero
  // fill of a mostly empty box is slow, and the tile rows beyond M feed only
  // accumulator rows that are never stored.
  const int a_rows = M >= BM ? BM : ((M + 7) / 8) * 8;
  CUtensorMap ta, tw;
  if (!make_map(&ta, A, M, K, lda, a_rows) || !make_map(&tw, W, N, K, ldw, p.bn)) return KINV_ERR_CUDA;
  GemmArgs a;
  a.C = C;
  a.ldc = ldc;
  a.M = M;
  a.N = N;
  a.k_tiles = K / BK / p.splits;
  a.a_rows = a_rows;
  a.a_stride = a_rows * BK * 2;
  a.c_f32 = c_dtype == KINV_F32;
  a.swiglu = swiglu ? 1 : 0;
  a.stages = 0;
  a.splits = p.splits;
  a.status = device_status_word();
  switch (p.bn) {
    case 64: return launch_gemm<64>(ta, tw, a, p.smem_budget, grid_y, grid_z, stream);
    case 128: return launch_gemm<128>(ta, tw, a, p.smem_budget, grid_y, grid_z, stream);
    default: return KINV_ERR_UNSUPPORTED;
  }
}
}  // namespace
}  // namespace kinv

extern "C" kinv_status kinv_gemm(const void* A, int64_t lda, const void* W, int64_t ldw, void* C,
                                 int64_t ldc, kinv_dtype c_dtype, int M, int N, int K,
                                 kinv_stream stream) {
  return kinv::gemm_impl(A, lda, W, ldw, C, ldc, c_dtype, M, N, K, false, stream);
}

extern "C" kinv_status kinv_gemm_swiglu(const void* A, int64_t lda, const void* W_gu, int64_t ldw,
                                        void* act, int64_t ld_act, int M, int F, int K,
                                        kinv_stream stream) {
  if (F <= 0 || F % 32) return F <= 0 ? KINV_ERR_INVALID_ARG : KINV_ERR_UNSUPPORTED;
  return kinv::gemm_impl(A, lda, W_gu, ldw, act, ld_act, KINV_BF16, M, 2 * F, K, true, stream);
}
