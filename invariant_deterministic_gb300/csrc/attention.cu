// Batch-invariant split-KV attention for decode and prefill
// ("Deterministic and bit-exact inference", *technical*: attention made
// batch-invariant "with a fixed split size for the key-value dimension rather
// than a fixed number of splits").
//
// A query row with L visible keys cuts them into splits of 256 keys at
// absolute offsets 0, 256, 512, ...; the cut depends only on L.  Split kernel:
// one thread block (eight warps) per (split, kv head, group of query rows of
// one sequence); up to 16 (row, query head) pairs form the 16 rows of
// warp-level tensor-core MMAs (m16n8k16, bf16 inputs, fp32 accumulation).
// K, then V, arrive in shared memory through cp.async.  For every pair:
//   s_t  = (q . k_t) * scale   warp w forms keys 32w..32w+31: eight 16-wide
//                              k steps of d, ascending, accumulated in fp32
//   m    = max_t s_t           (max is exact in any order)
//   e_t  = exp(s_t - m)        in fp32, then carried as the bf16 pair
//   hi_t = bf16(e_t), lo_t = bf16(e_t - hi_t)   (about 16 significant bits)
//   l    = sum_t (hi_t + lo_t) a lane's eight keys in order, a fixed
//                              butterfly over four lanes, warps in order
//   o[d] = sum_t hi_t v_t[d] + sum_t lo_t v_t[d]
//                              each sum sixteen 16-key k steps, ascending,
//                              in fp32; the two sums added once at the end
// and (m, l, o) is stored as the split's fp32 partial.  The tensor cores take
// P one bf16 half at a time: P's tile holds hi for the first pass and lo for
// the second (the lo values wait in registers).  A key a pair cannot
// see (beyond its count) gets p_t = 0; keys past the split's end read zero V.
// An MMA row depends only on its own q row and weights, so a pair's bits are
// the same whichever pairs share the block.
// Merge kernel: per (row, query head), fold the partials in ascending split
// order with the log-sum-exp update, then o / l -> bf16.
//
// Decode is the case of one row per block with L = kv_len[b]; prefill groups
// up to 32 / (Hq/Hkv) consecutive rows of one sequence per block (they share
// the split's K and V tiles in shared memory) with L = position + 1.  Both run
// the same compiled kernels, so a decode step equals a one-row prefill bit for
// bit, and a prompt's rows have the same bits for every chunking.
#include <math.h>

#include "common.cuh"

namespace kinv {
namespace {

constexpr int kSplit = 256;      // keys per split (the fixed split size)
constexpr int kThreads = 256;    // eight warps, 32 keys each for the scores
constexpr int kRowsMma = 16;     // (row, head) pairs of one block: the MMA's 16 rows
constexpr int kMaxG = 8;         // query heads per kv head
constexpr int kPrefillTiles = 4; // prefill: 16-row MMA tiles of (row, head) pairs per block

struct AttnParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  int64_t seq_stride, tok_stride;
  const int32_t* kv_len;    // decode
  const int32_t* q_start;   // prefill
  const int32_t* q_len;
  const int32_t* q_offset;
  __nv_bfloat16* out;
  float* ws_o;              // [rows][Hq][S][D]
  float* ws_ml;             // [rows][Hq][S][2]
  int prefill;
  int Hq, Hkv, G, R;
  int S;                    // splits per row in the workspace
  int groups_per_seq;       // prefill: ceil(max_q_len / R)
  int rg_cap;               // R * G: sizes the query and weight buffers
  float scale;
  // bounds the device-side lengths must keep (the host cannot read them):
  // decode 0 <= kv_len[b] <= max_len; prefill 0 <= q_len[b] <= max_q_len,
  // 0 <= q_start[b] <= max_len - q_len[b], 0 <= q_offset[b] <= total_rows - q_len[b]
  int max_len;              // decode: Lmax; prefill: max_kv
  int max_q_len;
  int total_rows;
  int* status;              // device status word (a sequence outside the bounds)
};

// A sequence whose device-side lengths break the bounds above is left out
// (decode writes zeros for it, prefill leaves its rows untouched) and the call
// records DEV_ATTN_BAD_LENGTH, so no access leaves the caller's buffers.
__device__ __forceinline__ bool seq_ok(const AttnParams& p, int b) {
  if (!p.prefill) {
    const int n = p.kv_len[b];
    return n >= 0 && n <= p.max_len;
  }
  const int n = p.q_len[b], st = p.q_start[b], off = p.q_offset[b];
  return n >= 0 && n <= p.max_q_len && st >= 0 && st <= p.max_len - n && off >= 0 &&
         off <= p.total_rows - n;
}

__device__ __forceinline__ void report_bad_length(const AttnParams& p) {
  if (threadIdx.x == 0 && p.status) atomicExch(p.status, DEV_ATTN_BAD_LENGTH);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Rows handled by this block: their q/out row indices and visible key counts.
struct RowSet {
  int nrows;
  int seq;
  int row0;     // q/out row of the first row (rows are consecutive)
  int len0;     // visible keys of the first row (row r sees len0 + r)
};

__device__ __forceinline__ bool block_rows(const AttnParams& p, RowSet& rs) {
  const int bq = p.prefill ? static_cast<int>(blockIdx.z) / p.groups_per_seq : static_cast<int>(blockIdx.z);
  if (!seq_ok(p, bq)) {
    report_bad_length(p);
    return false;
  }
  if (!p.prefill) {
    const int b = blockIdx.z;
    rs.nrows = 1;
    rs.seq = b;
    rs.row0 = b;
    rs.len0 = p.kv_len[b];
    return rs.len0 > 0;
  }
  const int b = blockIdx.z / p.groups_per_seq;
  const int j = blockIdx.z % p.groups_per_seq;
  const int first = j * p.R;
  const int n = p.q_len[b];
  if (first >= n) return false;
  rs.nrows = min(p.R, n - first);
  rs.seq = b;
  rs.row0 = p.q_offset[b] + first;
  rs.len0 = p.q_start[b] + first + 1;
  return true;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// D = A . B + D, one 16 x 8 x 16 warp MMA, bf16 inputs, fp32 accumulation.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// A softmax weight as the pair hi + lo of bf16 values: hi = bf16(x) and
// lo = bf16(x - hi) (x - hi is exact in fp32), so hi + lo carries x to about
// 16 significant bits where bf16 alone keeps 8.
__device__ __forceinline__ void split_bf16(float x, float& hi, float& lo) {
  hi = __bfloat162float(__float2bfloat16_rn(x));
  lo = __bfloat162float(__float2bfloat16_rn(__fsub_rn(x, hi)));
}

template <int D>
__global__ void __launch_bounds__(kThreads) attn_split_kernel(const AttnParams p) {
  constexpr int C8 = D / 8;               // 16-byte chunks per key row
  constexpr int SUB = 64;                 // keys per load stage
  constexpr int NSUB = kSplit / SUB;      // the K stages are reused for V
  constexpr int KS = D / 16;              // 16-wide k steps of q . k
  // Tiles in shared memory, rows of 16-byte chunks; chunk c of row r is
  // stored at chunk c ^ (r & 7), so the eight row addresses of every ldmatrix
  // phase fall in eight different bank groups.
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __nv_bfloat16* kv = reinterpret_cast<__nv_bfloat16*>(smem_raw);                 // [256][D]
  __nv_bfloat16* pt = reinterpret_cast<__nv_bfloat16*>(smem_raw + kSplit * D * 2);  // P [16][256]
  __shared__ float wmax[kThreads / 32][kRowsMma];
  __shared__ float wsum[kThreads / 32][kRowsMma];

  pdl_launch_dependents();
  pdl_wait();
  RowSet rs;
  if (!block_rows(p, rs)) return;
  // kv heads are the fastest grid index: the blocks reading the 256-byte
  // slices of the same token rows run side by side
  const int g = blockIdx.x;
  const int s = blockIdx.y;
  const int k0 = s * kSplit;
  const int lenmax = rs.len0 + rs.nrows - 1;           // the last row sees the most keys
  const int nmax = min(kSplit, lenmax - k0);
  if (nmax <= 0) return;
  const int G = p.G;
  const int RG = rs.nrows * G;                         // (row, head) pairs: MMA rows 0..RG-1
  const int t = threadIdx.x;
  const int lane = t & 31, warp = t >> 5;
  const int gq = lane >> 2, tq = lane & 3;             // fragment row / column group
  const int64_t seq_off = rs.seq * p.seq_stride + static_cast<int64_t>(k0) * p.tok_stride + g * D;
  const uint32_t kv_base = smem_addr(kv);
  const uint32_t pt_base = smem_addr(pt);
  auto count = [&](int r) { return r < RG ? min(kSplit, rs.len0 + r / G - k0) : 0; };

  auto load_sub = [&](const __nv_bfloat16* src, int j) {
    const int rows = min(SUB, nmax - j * SUB);
    for (int idx = t; idx < rows * C8; idx += kThreads) {
      const int r = idx / C8, c = idx % C8;
      const int key = j * SUB + r;
      cp_async16(kv_base + static_cast<uint32_t>(key * D * 2 + ((c ^ (key & 7)) << 4)),
                 src + seq_off + static_cast<int64_t>(key) * p.tok_stride + c * 8);
    }
  };
#pragma unroll
  for (int j = 0; j < NSUB; ++j) load_sub(p.k, j);
  cp_async_commit();

  // q fragments (A operand, rows = (row, head) pairs), straight from global
  uint32_t qa[KS][4];
  {
    const int r_lo = gq, r_hi = gq + 8;
    const __nv_bfloat16* q_lo = r_lo < RG
        ? p.q + (static_cast<int64_t>(rs.row0 + r_lo / G) * p.Hq + g * G + r_lo % G) * D : nullptr;
    const __nv_bfloat16* q_hi = r_hi < RG
        ? p.q + (static_cast<int64_t>(rs.row0 + r_hi / G) * p.Hq + g * G + r_hi % G) * D : nullptr;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int d0 = ks * 16 + 2 * tq;
      qa[ks][0] = q_lo ? *reinterpret_cast<const uint32_t*>(q_lo + d0) : 0u;
      qa[ks][1] = q_hi ? *reinterpret_cast<const uint32_t*>(q_hi + d0) : 0u;
      qa[ks][2] = q_lo ? *reinterpret_cast<const uint32_t*>(q_lo + d0 + 8) : 0u;
      qa[ks][3] = q_hi ? *reinterpret_cast<const uint32_t*>(q_hi + d0 + 8) : 0u;
    }
  }
  cp_async_wait<0>();
  __syncthreads();

  // --- scores: warp w owns keys 32w .. 32w + 31 (four 8-key n blocks)
  float sc[4][4];
#pragma unroll
  for (int nb = 0; nb < 4; ++nb) {
#pragma unroll
    for (int i = 0; i < 4; ++i) sc[nb][i] = 0.f;
    const int key = warp * 32 + nb * 8 + (lane & 7);
#pragma unroll
    for (int kp = 0; kp < KS / 2; ++kp) {
      const int c = kp * 4 + (lane >> 3);
      uint32_t b0, b1, b2, b3;
      ldsm_x4(kv_base + static_cast<uint32_t>(key * D * 2 + ((c ^ (key & 7)) << 4)), b0, b1, b2, b3);
      mma_bf16_16816(sc[nb], qa[2 * kp], b0, b1);
      mma_bf16_16816(sc[nb], qa[2 * kp + 1], b2, b3);
    }
  }
  __syncthreads();  // every warp is done with K: the stages take V now
#pragma unroll
  for (int j = 0; j < NSUB; ++j) load_sub(p.v, j);
  // keys the split does not hold read as zero (their weights are zero, and a
  // stale NaN times zero would not be)
  for (int idx = t; idx < (kSplit - nmax) * C8; idx += kThreads) {
    const int key = nmax + idx / C8, c = idx % C8;
    *reinterpret_cast<uint4*>(kv + key * D + ((c ^ (key & 7)) << 3)) = make_uint4(0, 0, 0, 0);
  }
  cp_async_commit();

  // --- softmax statistics.  A lane holds rows gq and gq + 8, keys
  // 32w + 8nb + 2tq (+1).  Maxima: lane, then the four lanes of a row
  // (exact), then the eight warps.  Weights are rounded to bf16 once; the sum
  // adds the rounded weights: a lane's eight in (nb, pair) order, a fixed
  // butterfly over the four lanes, the eight warps in ascending order.
  const int cnt_lo = count(gq), cnt_hi = count(gq + 8);
  float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
  for (int nb = 0; nb < 4; ++nb) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int key = warp * 32 + nb * 8 + 2 * tq + e;
      sc[nb][e] = key < cnt_lo ? __fmul_rn(sc[nb][e], p.scale) : -INFINITY;
      sc[nb][2 + e] = key < cnt_hi ? __fmul_rn(sc[nb][2 + e], p.scale) : -INFINITY;
      mx_lo = fmaxf(mx_lo, sc[nb][e]);
      mx_hi = fmaxf(mx_hi, sc[nb][2 + e]);
    }
  }
#pragma unroll
  for (int o = 1; o <= 2; o <<= 1) {
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, o));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, o));
  }
  if (tq == 0) {
    wmax[warp][gq] = mx_lo;
    wmax[warp][gq + 8] = mx_hi;
  }
  __syncthreads();
  float m_lo = wmax[0][gq], m_hi = wmax[0][gq + 8];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) {
    m_lo = fmaxf(m_lo, wmax[w][gq]);
    m_hi = fmaxf(m_hi, wmax[w][gq + 8]);
  }
  float sum_lo = 0.f, sum_hi = 0.f;
  // writes the weights held in w[nb][0..3] (rows gq and gq + 8) into P's tile
  auto write_p = [&](const float (&w)[4][4]) {
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) {
      const int kc = warp * 4 + nb;                       // 8-key chunk of P
      const uint32_t off_lo = static_cast<uint32_t>(gq * kSplit * 2 + ((kc ^ (gq & 7)) << 4) + 4 * tq);
      const uint32_t off_hi = static_cast<uint32_t>((gq + 8) * kSplit * 2 + ((kc ^ (gq & 7)) << 4) + 4 * tq);
      *reinterpret_cast<uint32_t*>(reinterpret_cast<unsigned char*>(pt) + off_lo) = pack_bf16(w[nb][0], w[nb][1]);
      *reinterpret_cast<uint32_t*>(reinterpret_cast<unsigned char*>(pt) + off_hi) = pack_bf16(w[nb][2], w[nb][3]);
    }
  };
  float hi[4][4];  // the high halves; sc keeps the low halves for the second pass
#pragma unroll
  for (int nb = 0; nb < 4; ++nb) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float xl = sc[nb][e] == -INFINITY ? 0.f : expf(__fsub_rn(sc[nb][e], m_lo));
      const float xh = sc[nb][2 + e] == -INFINITY ? 0.f : expf(__fsub_rn(sc[nb][2 + e], m_hi));
      split_bf16(xl, hi[nb][e], sc[nb][e]);
      split_bf16(xh, hi[nb][2 + e], sc[nb][2 + e]);
      sum_lo = __fadd_rn(sum_lo, __fadd_rn(hi[nb][e], sc[nb][e]));
      sum_hi = __fadd_rn(sum_hi, __fadd_rn(hi[nb][2 + e], sc[nb][2 + e]));
    }
  }
  write_p(hi);
#pragma unroll
  for (int o = 1; o <= 2; o <<= 1) {
    sum_lo = __fadd_rn(sum_lo, __shfl_xor_sync(0xffffffffu, sum_lo, o));
    sum_hi = __fadd_rn(sum_hi, __shfl_xor_sync(0xffffffffu, sum_hi, o));
  }
  if (tq == 0) {
    wsum[warp][gq] = sum_lo;
    wsum[warp][gq + 8] = sum_hi;
  }
  cp_async_wait<0>();
  __syncthreads();

  // --- o = P . V: warp w owns columns 16w .. 16w + 15 (two 8-wide n
  // blocks) over all 256 keys, sixteen k steps of 16 keys in ascending order;
  // once over the high halves of P, once over the low halves.
  auto pv = [&](float (&acc)[2][4]) {
#pragma unroll
    for (int nb = 0; nb < 2; ++nb)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[nb][i] = 0.f;
    if (warp >= D / 16) return;
#pragma unroll 4
    for (int kk = 0; kk < kSplit / 16; ++kk) {
      uint32_t a[4];
      {
        const int prow = lane & 15;
        const int kc = 2 * kk + (lane >> 4);
        ldsm_x4(pt_base + static_cast<uint32_t>(prow * kSplit * 2 + ((kc ^ (prow & 7)) << 4)), a[0], a[1],
                a[2], a[3]);
      }
      uint32_t b0, b1, b2, b3;
      {
        const int key = kk * 16 + (lane & 15);
        const int c = warp * 2 + (lane >> 4);
        ldsm_x4_t(kv_base + static_cast<uint32_t>(key * D * 2 + ((c ^ (key & 7)) << 4)), b0, b1, b2, b3);
      }
      mma_bf16_16816(acc[0], a, b0, b1);
      mma_bf16_16816(acc[1], a, b2, b3);
    }
  };
  float oc[2][4], ol[2][4];
  pv(oc);
  __syncthreads();  // every warp is done with the high halves
  write_p(sc);
  __syncthreads();
  pv(ol);
  if (warp < D / 16) {
    // rows gq and gq + 8, columns 16w + 8nb + 2tq (+1)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = gq + 8 * h;
      if (r < RG && count(r) > 0) {
        const int row = r / G, i = r % G;
        const int64_t base = (static_cast<int64_t>(rs.row0 + row) * p.Hq + g * G + i) * p.S + s;
#pragma unroll
        for (int nb = 0; nb < 2; ++nb)
          *reinterpret_cast<float2*>(p.ws_o + base * D + warp * 16 + nb * 8 + 2 * tq) =
              make_float2(__fadd_rn(oc[nb][2 * h], ol[nb][2 * h]), __fadd_rn(oc[nb][2 * h + 1], ol[nb][2 * h + 1]));
        if (warp == 0 && tq == 0) {
          float l = wsum[0][r];
#pragma unroll
          for (int w = 1; w < kThreads / 32; ++w) l = __fadd_rn(l, wsum[w][r]);
          p.ws_ml[base * 2 + 0] = h ? m_hi : m_lo;
          p.ws_ml[base * 2 + 1] = l;
        }
      }
    }
  }
}

// The split kernel for prefill: MT 16-row MMA tiles of (row, head) pairs per
// block, sharing the block's K and V tiles (so each tile load serves MT times
// the rows).  Every pair is one MMA row and meets exactly the arithmetic of
// attn_split_kernel (the same MMAs in the same order, the same softmax, sums
// and rounding), so a prefill row has the bits of the decode row.
template <int D, int MT>
__global__ void __launch_bounds__(kThreads, 2) attn_split_tiles_kernel(const AttnParams p) {
  constexpr int C8 = D / 8;               // 16-byte chunks per key row
  constexpr int SUB = 64;                 // keys per load stage
  constexpr int NSUB = kSplit / SUB;      // the K stages are reused for V
  constexpr int KS = D / 16;              // 16-wide k steps of q . k
  constexpr int PR = kRowsMma * MT;       // (row, head) pairs of a block
  // Tiles in shared memory, rows of 16-byte chunks; chunk c of row r is
  // stored at chunk c ^ (r & 7), so the eight row addresses of every ldmatrix
  // phase fall in eight different bank groups.
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __nv_bfloat16* kv = reinterpret_cast<__nv_bfloat16*>(smem_raw);                 // [256][D]
  __nv_bfloat16* pt = reinterpret_cast<__nv_bfloat16*>(smem_raw + kSplit * D * 2);  // P [PR][256]
  // the block's q rows [PR][D] (swizzled like K) live where P goes, until the scores are done
  __nv_bfloat16* qs = pt;
  static_assert(kRowsMma * MT * D <= kRowsMma * MT * kSplit, "q rows fit in the P tile");
  __shared__ float wmax[kThreads / 32][PR];
  __shared__ float wsum[kThreads / 32][PR];

  pdl_launch_dependents();
  pdl_wait();
  RowSet rs;
  if (!block_rows(p, rs)) return;
  // kv heads are the fastest grid index: the blocks reading the 256-byte
  // slices of the same token rows run side by side
  const int g = blockIdx.x;
  const int s = blockIdx.y;
  const int k0 = s * kSplit;
  const int lenmax = rs.len0 + rs.nrows - 1;           // the last row sees the most keys
  const int nmax = min(kSplit, lenmax - k0);
  if (nmax <= 0) return;
  const int G = p.G;
  const int RG = rs.nrows * G;                         // (row, head) pairs: MMA rows 0..RG-1
  const int t = threadIdx.x;
  const int lane = t & 31, warp = t >> 5;
  const int gq = lane >> 2, tq = lane & 3;             // fragment row / column group
  const int64_t seq_off = rs.seq * p.seq_stride + static_cast<int64_t>(k0) * p.tok_stride + g * D;
  const uint32_t kv_base = smem_addr(kv);
  const uint32_t pt_base = smem_addr(pt);
  auto count = [&](int r) { return r < RG ? min(kSplit, rs.len0 + r / G - k0) : 0; };

  auto load_sub = [&](const __nv_bfloat16* src, int j) {
    const int rows = min(SUB, nmax - j * SUB);
    for (int idx = t; idx < rows * C8; idx += kThreads) {
      const int r = idx / C8, c = idx % C8;
      const int key = j * SUB + r;
      cp_async16(kv_base + static_cast<uint32_t>(key * D * 2 + ((c ^ (key & 7)) << 4)),
                 src + seq_off + static_cast<int64_t>(key) * p.tok_stride + c * 8);
    }
  };
#pragma unroll
  for (int j = 0; j < NSUB; ++j) load_sub(p.k, j);
  cp_async_commit();

  // the q rows of the block's pairs, once (pair r: row r / G, head g * G + r % G);
  // rows of pairs past RG, in a tile that has pairs, read as zero
  const uint32_t qs_base = smem_addr(qs);
  const int tiles = (RG + kRowsMma - 1) / kRowsMma;
  for (int idx = t; idx < tiles * kRowsMma * C8; idx += kThreads) {
    const int r = idx / C8, c = idx % C8;
    if (r < RG)
      cp_async16(qs_base + static_cast<uint32_t>(r * D * 2 + ((c ^ (r & 7)) << 4)),
                 p.q + (static_cast<int64_t>(rs.row0 + r / G) * p.Hq + g * G + r % G) * D + c * 8);
    else
      *reinterpret_cast<uint4*>(qs + r * D + ((c ^ (r & 7)) << 3)) = make_uint4(0, 0, 0, 0);
  }
  cp_async_commit();
  uint32_t qa[KS][4];
  cp_async_wait<0>();
  __syncthreads();

  // --- scores: warp w owns keys 32w .. 32w + 31 (four 8-key n blocks), for
  // every tile of pairs
  float sc[MT][4][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
    for (int nb = 0; nb < 4; ++nb)
#pragma unroll
      for (int i = 0; i < 4; ++i) sc[mt][nb][i] = 0.f;
    if (mt * kRowsMma >= RG) continue;  // (block-uniform)
    // q fragments (A operand) of tile mt: lane l gives row mt * 16 + (l & 15),
    // 8-column block 2 ks + (l >> 4) -- the MMA's a0..a3
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int qrow = mt * kRowsMma + (lane & 15);
      const int c = 2 * ks + (lane >> 4);
      ldsm_x4(qs_base + static_cast<uint32_t>(qrow * D * 2 + ((c ^ (qrow & 7)) << 4)), qa[ks][0], qa[ks][1],
              qa[ks][2], qa[ks][3]);
    }
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) {
      const int key = warp * 32 + nb * 8 + (lane & 7);
#pragma unroll
      for (int kp = 0; kp < KS / 2; ++kp) {
        const int c = kp * 4 + (lane >> 3);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kv_base + static_cast<uint32_t>(key * D * 2 + ((c ^ (key & 7)) << 4)), b0, b1, b2, b3);
        mma_bf16_16816(sc[mt][nb], qa[2 * kp], b0, b1);
        mma_bf16_16816(sc[mt][nb], qa[2 * kp + 1], b2, b3);
      }
    }
  }
  __syncthreads();  // every warp is done with K: the stages take V now
#pragma unroll
  for (int j = 0; j < NSUB; ++j) load_sub(p.v, j);
  // keys the split does not hold read as zero (their weights are zero, and a
  // stale NaN times zero would not be)
  for (int idx = t; idx < (kSplit - nmax) * C8; idx += kThreads) {
    const int key = nmax + idx / C8, c = idx % C8;
    *reinterpret_cast<uint4*>(kv + key * D + ((c ^ (key & 7)) << 3)) = make_uint4(0, 0, 0, 0);
  }
  cp_async_commit();

  // --- softmax statistics.  A lane holds rows gq and gq + 8 of each tile,
  // keys 32w + 8nb + 2tq (+1).  Maxima: lane, then the four lanes of a row
  // (exact), then the eight warps.  Weights are rounded to bf16 once; the sum
  // adds the rounded weights: a lane's eight in (nb, pair) order, a fixed
  // butterfly over the four lanes, the eight warps in ascending order.
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    if (mt * kRowsMma >= RG) continue;
    const int r_lo = mt * kRowsMma + gq, r_hi = r_lo + 8;
    const int cnt_lo = count(r_lo), cnt_hi = count(r_hi);
    float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = warp * 32 + nb * 8 + 2 * tq + e;
        sc[mt][nb][e] = key < cnt_lo ? __fmul_rn(sc[mt][nb][e], p.scale) : -INFINITY;
        sc[mt][nb][2 + e] = key < cnt_hi ? __fmul_rn(sc[mt][nb][2 + e], p.scale) : -INFINITY;
        mx_lo = fmaxf(mx_lo, sc[mt][nb][e]);
        mx_hi = fmaxf(mx_hi, sc[mt][nb][2 + e]);
      }
    }
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, o));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, o));
    }
    if (tq == 0) {
      wmax[warp][r_lo] = mx_lo;
      wmax[warp][r_hi] = mx_hi;
    }
  }
  __syncthreads();
  // writes the weights held in w[nb][0..3] (rows gq and gq + 8 of tile mt)
  // into P's tile
  auto write_p = [&](int mt, const float (&w)[4][4]) {
    const int r_lo = mt * kRowsMma + gq, r_hi = r_lo + 8;
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) {
      const int kc = warp * 4 + nb;                       // 8-key chunk of P
      const uint32_t off_lo = static_cast<uint32_t>(r_lo * kSplit * 2 + ((kc ^ (gq & 7)) << 4) + 4 * tq);
      const uint32_t off_hi = static_cast<uint32_t>(r_hi * kSplit * 2 + ((kc ^ (gq & 7)) << 4) + 4 * tq);
      *reinterpret_cast<uint32_t*>(reinterpret_cast<unsigned char*>(pt) + off_lo) = pack_bf16(w[nb][0], w[nb][1]);
      *reinterpret_cast<uint32_t*>(reinterpret_cast<unsigned char*>(pt) + off_hi) = pack_bf16(w[nb][2], w[nb][3]);
    }
  };
  float m_lo[MT], m_hi[MT];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    m_lo[mt] = m_hi[mt] = -INFINITY;
    if (mt * kRowsMma >= RG) continue;
    const int r_lo = mt * kRowsMma + gq, r_hi = r_lo + 8;
    m_lo[mt] = wmax[0][r_lo];
    m_hi[mt] = wmax[0][r_hi];
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w) {
      m_lo[mt] = fmaxf(m_lo[mt], wmax[w][r_lo]);
      m_hi[mt] = fmaxf(m_hi[mt], wmax[w][r_hi]);
    }
    float sum_lo = 0.f, sum_hi = 0.f;
    float hi[4][4];  // the high halves; sc keeps the low halves for the second pass
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float xl = sc[mt][nb][e] == -INFINITY ? 0.f : expf(__fsub_rn(sc[mt][nb][e], m_lo[mt]));
        const float xh = sc[mt][nb][2 + e] == -INFINITY ? 0.f : expf(__fsub_rn(sc[mt][nb][2 + e], m_hi[mt]));
        split_bf16(xl, hi[nb][e], sc[mt][nb][e]);
        split_bf16(xh, hi[nb][2 + e], sc[mt][nb][2 + e]);
        sum_lo = __fadd_rn(sum_lo, __fadd_rn(hi[nb][e], sc[mt][nb][e]));
        sum_hi = __fadd_rn(sum_hi, __fadd_rn(hi[nb][2 + e], sc[mt][nb][2 + e]));
      }
    }
    write_p(mt, hi);
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      sum_lo = __fadd_rn(sum_lo, __shfl_xor_sync(0xffffffffu, sum_lo, o));
      sum_hi = __fadd_rn(sum_hi, __shfl_xor_sync(0xffffffffu, sum_hi, o));
    }
    if (tq == 0) {
      wsum[warp][r_lo] = sum_lo;
      wsum[warp][r_hi] = sum_hi;
    }
  }
  cp_async_wait<0>();
  __syncthreads();

  // --- o = P . V: warp w owns columns 16w .. 16w + 15 (two 8-wide n
  // blocks) over all 256 keys, sixteen k steps of 16 keys in ascending order;
  // each V fragment serves every tile.  Once over the high halves of P, once
  // over the low halves, the two sums added at the end.
  auto pv = [&](float (&acc)[MT][2][4]) {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[mt][nb][i] = 0.f;
    if (warp >= D / 16) return;
#pragma unroll 4
    for (int kk = 0; kk < kSplit / 16; ++kk) {
      uint32_t b0, b1, b2, b3;
      {
        const int key = kk * 16 + (lane & 15);
        const int c = warp * 2 + (lane >> 4);
        ldsm_x4_t(kv_base + static_cast<uint32_t>(key * D * 2 + ((c ^ (key & 7)) << 4)), b0, b1, b2, b3);
      }
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        if (mt >= tiles) continue;
        uint32_t a[4];
        const int prow = mt * kRowsMma + (lane & 15);
        const int kc = 2 * kk + (lane >> 4);
        ldsm_x4(pt_base + static_cast<uint32_t>(prow * kSplit * 2 + ((kc ^ (prow & 7)) << 4)), a[0], a[1],
                a[2], a[3]);
        mma_bf16_16816(acc[mt][0], a, b0, b1);
        mma_bf16_16816(acc[mt][1], a, b2, b3);
      }
    }
  };
  float oc[MT][2][4], ol[MT][2][4];
  pv(oc);
  __syncthreads();  // every warp is done with the high halves
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
    if (mt * kRowsMma < RG) write_p(mt, sc[mt]);
  __syncthreads();
  pv(ol);
  if (warp < D / 16) {
    // rows gq and gq + 8 of each tile, columns 16w + 8nb + 2tq (+1)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r = mt * kRowsMma + gq + 8 * h;
        if (r < RG && count(r) > 0) {
          const int row = r / G, i = r % G;
          const int64_t base = (static_cast<int64_t>(rs.row0 + row) * p.Hq + g * G + i) * p.S + s;
#pragma unroll
          for (int nb = 0; nb < 2; ++nb)
            *reinterpret_cast<float2*>(p.ws_o + base * D + warp * 16 + nb * 8 + 2 * tq) =
                make_float2(__fadd_rn(oc[mt][nb][2 * h], ol[mt][nb][2 * h]),
                            __fadd_rn(oc[mt][nb][2 * h + 1], ol[mt][nb][2 * h + 1]));
          if (warp == 0 && tq == 0) {
            float l = wsum[0][r];
#pragma unroll
            for (int w = 1; w < kThreads / 32; ++w) l = __fadd_rn(l, wsum[w][r]);
            p.ws_ml[base * 2 + 0] = h ? m_hi[mt] : m_lo[mt];
            p.ws_ml[base * 2 + 1] = l;
          }
        }
      }
    }
  }
}

// One block per (query head, row); thread d folds column d.
template <int D>
__global__ void attn_merge_kernel(const AttnParams p) {
  pdl_launch_dependents();
  pdl_wait();
  int row, len;
  if (!p.prefill) {
    row = blockIdx.y;
    if (!seq_ok(p, row)) {
      report_bad_length(p);
      len = 0;  // zeros
    } else {
      len = p.kv_len[row];
    }
  } else {
    const int b = blockIdx.z;
    const int i = blockIdx.y;
    if (!seq_ok(p, b)) {
      if (i == 0) report_bad_length(p);
      return;
    }
    if (i >= p.q_len[b]) return;
    row = p.q_offset[b] + i;
    len = p.q_start[b] + i + 1;
  }
  const int h = blockIdx.x;
  const int d = threadIdx.x;
  __nv_bfloat16* dst = p.out + (static_cast<int64_t>(row) * p.Hq + h) * D + d;
  if (len <= 0) {
    *dst = __float2bfloat16_rn(0.f);
    return;
  }
  const int ns = min((len + kSplit - 1) / kSplit, p.S);
  const int64_t base = (static_cast<int64_t>(row) * p.Hq + h) * p.S;
  float m_acc = -INFINITY, l_acc = 0.f, o_acc = 0.f;
  constexpr int CH = 8;  // partials loaded ahead of the (sequential) fold
  for (int s0 = 0; s0 < ns; s0 += CH) {
    float mv[CH], lv[CH], ov[CH];
#pragma unroll
    for (int i = 0; i < CH; ++i) {
      if (s0 + i < ns) {
        const float2 ml = *reinterpret_cast<const float2*>(p.ws_ml + (base + s0 + i) * 2);
        mv[i] = ml.x;
        lv[i] = ml.y;
        ov[i] = p.ws_o[(base + s0 + i) * D + d];
      }
    }
#pragma unroll
    for (int i = 0; i < CH; ++i) {
      if (s0 + i < ns) {
        const float m_new = fmaxf(m_acc, mv[i]);
        const float a = expf(__fsub_rn(m_acc, m_new));
        const float c = expf(__fsub_rn(mv[i], m_new));
        l_acc = __fadd_rn(__fmul_rn(l_acc, a), __fmul_rn(lv[i], c));
        o_acc = __fadd_rn(__fmul_rn(o_acc, a), __fmul_rn(ov[i], c));
        m_acc = m_new;
      }
    }
  }
  *dst = __float2bfloat16_rn(__fdiv_rn(o_acc, l_acc));
}

template <int D, int MT>
size_t split_smem_bytes() {
  return static_cast<size_t>(kSplit) * D * 2 + static_cast<size_t>(kRowsMma) * MT * kSplit * 2;
}

// MT == 1: attn_split_kernel (decode); otherwise attn_split_tiles_kernel.
template <int D, int MT>
kinv_status launch(const AttnParams& p, dim3 split_grid, dim3 merge_grid, cudaStream_t stream) {
  void (*kernel)(const AttnParams);
  if constexpr (MT == 1)
    kernel = attn_split_kernel<D>;
  else
    kernel = attn_split_tiles_kernel<D, MT>;
  const size_t smem = split_smem_bytes<D, MT>();
  const kinv_status attr = ensure_smem(reinterpret_cast<const void*>(kernel), smem);
  if (attr != KINV_OK) return attr;
  const kinv_status st = launch_kernel(kernel, split_grid, dim3(kThreads), smem, stream, 1, p);
  if (st != KINV_OK) return st;
  return launch_kernel(attn_merge_kernel<D>, merge_grid, dim3(D), 0, stream, 1, p);
}

kinv_status check_common(const void* q, const void* k, const void* v, int64_t seq_stride,
                         int64_t tok_stride, const void* out, int Hq, int Hkv, int D,
                         int split_len, const void* ws) {
  if (!q || !k || !v || !out || !ws) return KINV_ERR_INVALID_ARG;
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv) return KINV_ERR_INVALID_ARG;
  const int G = Hq / Hkv;
  if (G != 1 && G != 2 && G != 4 && G != kMaxG) return KINV_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return KINV_ERR_UNSUPPORTED;
  if (split_len != kSplit) return KINV_ERR_UNSUPPORTED;
  if (tok_stride < static_cast<int64_t>(Hkv) * D || seq_stride < 0) return KINV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(ws) ||
      seq_stride % 8 || tok_stride % 8)
    return KINV_ERR_ALIGNMENT;
  return KINV_OK;
}

size_t workspace_bytes(int64_t rows, int Hq, int D, int S) {
  const size_t o = static_cast<size_t>(rows) * Hq * S * D * 4;
  const size_t ml = static_cast<size_t>(rows) * Hq * S * 2 * 4;
  return ((o + 255) / 256) * 256 + ml;
}

}  // namespace
}  // namespace kinv

using namespace kinv;

extern "C" size_t kinv_attn_decode_workspace(int B, int Hq, int D, int Lmax, int split_len) {
  if (B <= 0 || Hq <= 0 || D <= 0 || Lmax <= 0 || split_len <= 0) return 0;
  return workspace_bytes(B, Hq, D, (Lmax + split_len - 1) / split_len);
}

namespace kinv {
namespace {
// Host-side checks of a decode call (no CUDA call is made): the same order for
// kinv_attn_decode and kinv_attn_decode_noalloc.
kinv_status decode_check(const void* q, const void* k_cache, const void* v_cache, int64_t seq_stride,
                         int64_t tok_stride, const int32_t* kv_len, const void* out, int B, int Hq,
                         int Hkv, int D, int Lmax, int split_len, const void* workspace,
                         size_t ws_bytes) {
  if (B < 0 || Lmax < 0) return KINV_ERR_INVALID_ARG;
  if (B == 0) return KINV_OK;
  if (!kv_len) return KINV_ERR_INVALID_ARG;
  const kinv_status st = check_common(q, k_cache, v_cache, seq_stride, tok_stride, out, Hq, Hkv, D,
                                      split_len, workspace);
  if (st != KINV_OK) return st;
  if (B > 65535) return KINV_ERR_UNSUPPORTED;
  const int S = Lmax > 0 ? (Lmax + kSplit - 1) / kSplit : 1;
  if (ws_bytes < workspace_bytes(B, Hq, D, S)) return KINV_ERR_WORKSPACE;
  return KINV_OK;
}

// Enqueues a checked decode call with its partials in `workspace`.
kinv_status decode_launch(const void* q, const void* k_cache, const void* v_cache, int64_t seq_stride,
                          int64_t tok_stride, const int32_t* kv_len, void* out, int B, int Hq, int Hkv,
                          int D, int Lmax, float scale, void* workspace, cudaStream_t stream) {
  const int S = Lmax > 0 ? (Lmax + kSplit - 1) / kSplit : 1;
  AttnParams p{};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k_cache);
  p.v = static_cast<const __nv_bfloat16*>(v_cache);
  p.seq_stride = seq_stride;
  p.tok_stride = tok_stride;
  p.kv_len = kv_len;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.ws_o = static_cast<float*>(workspace);
  const size_t o_bytes = static_cast<size_t>(B) * Hq * S * D * 4;
  p.ws_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) + ((o_bytes + 255) / 256) * 256);
  p.prefill = 0;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.R = 1;
  p.S = S;
  p.groups_per_seq = 1;
  p.rg_cap = ((p.G + 3) / 4) * 4;
  p.scale = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(D));
  p.max_len = Lmax;
  p.max_q_len = 0;
  p.total_rows = B;
  p.status = device_status_word();
  const dim3 split_grid(Hkv, S, B), merge_grid(Hq, B, 1);
  return D == 128 ? launch<128, 1>(p, split_grid, merge_grid, stream)
                  : launch<64, 1>(p, split_grid, merge_grid, stream);
}
}  // namespace
}  // namespace kinv

extern "C" kinv_status kinv_attn_decode(const void* q, const void* k_cache, const void* v_cache,
                                        int64_t seq_stride, int64_t tok_stride,
                                        const int32_t* kv_len, void* out, int B, int Hq, int Hkv,
                                        int D, int Lmax, int split_len, float scale,
                                        void* workspace, size_t ws_bytes, kinv_stream stream) {
  const kinv_status st = decode_check(q, k_cache, v_cache, seq_stride, tok_stride, kv_len, out, B, Hq, Hkv,
                                      D, Lmax, split_len, workspace, ws_bytes);
  if (st != KINV_OK || B == 0) return st;
  return decode_launch(q, k_cache, v_cache, seq_stride, tok_stride, kv_len, out, B, Hq, Hkv, D, Lmax, scale,
                       workspace, stream);
}

extern "C" size_t kinv_attn_prefill_workspace(int total_rows, int Hq, int D, int max_kv,
                                              int split_len) {
  if (total_rows <= 0 || Hq <= 0 || D <= 0 || max_kv <= 0 || split_len <= 0) return 0;
  return workspace_bytes(total_rows, Hq, D, (max_kv + split_len - 1) / split_len);
}

extern "C" kinv_status kinv_attn_prefill(const void* q, const void* k_cache, const void* v_cache,
                                         int64_t seq_stride, int64_t tok_stride,
                                         const int32_t* q_start, const int32_t* q_len,
                                         const int32_t* q_offset, void* out, int B,
                                         int total_rows, int max_q_len, int max_kv, int Hq,
                                         int Hkv, int D, int split_len, float scale,
                                         void* workspace, size_t ws_bytes, kinv_stream stream) {
  if (B < 0 || total_rows < 0 || max_q_len < 0 || max_kv < 0) return KINV_ERR_INVALID_ARG;
  if (B == 0 || total_rows == 0 || max_q_len == 0) return KINV_OK;
  if (!q_start || !q_len || !q_offset || max_kv <= 0) return KINV_ERR_INVALID_ARG;
  kinv_status st = check_common(q, k_cache, v_cache, seq_stride, tok_stride, out, Hq, Hkv, D,
                                split_len, workspace);
  if (st != KINV_OK) return st;
  const int S = (max_kv + kSplit - 1) / kSplit;
  if (ws_bytes < workspace_bytes(total_rows, Hq, D, S)) return KINV_ERR_WORKSPACE;
  AttnParams p{};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k_cache);
  p.v = static_cast<const __nv_bfloat16*>(v_cache);
  p.seq_stride = seq_stride;
  p.tok_stride = tok_stride;
  p.q_start = q_start;
  p.q_len = q_len;
  p.q_offset = q_offset;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.ws_o = static_cast<float*>(workspace);
  const size_t o_bytes = static_cast<size_t>(total_rows) * Hq * S * D * 4;
  p.ws_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) + ((o_bytes + 255) / 256) * 256);
  p.prefill = 1;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.R = kRowsMma * kPrefillTiles / p.G;
  p.S = S;
  p.groups_per_seq = (max_q_len + p.R - 1) / p.R;
  p.rg_cap = p.R * p.G;
  p.scale = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(D));
  p.max_len = max_kv;
  p.max_q_len = max_q_len;
  p.total_rows = total_rows;
  p.status = device_status_word();
  const int64_t groups = static_cast<int64_t>(B) * p.groups_per_seq;
  if (groups > 65535 || max_q_len > 65535 || B > 65535) return KINV_ERR_UNSUPPORTED;
  const dim3 split_grid(Hkv, S, static_cast<unsigned>(groups)), merge_grid(Hq, max_q_len, B);
  return D == 128 ? launch<128, kPrefillTiles>(p, split_grid, merge_grid, stream)
                  : launch<64, kPrefillTiles>(p, split_grid, merge_grid, stream);
}

// ---------------------------------------------------------------------------
// kinv_attn_decode_noalloc: decode attention for callers that cannot allocate
// device memory.  The split partials go to a scratch array compiled into the
// library instead of a caller-provided workspace.

#include <map>
#include <mutex>

// Scratch shared by every kinv_attn_decode_noalloc call on a device (held by
// each GPU that loads the library until the process exits).
static __device__ __align__(256) unsigned char kinv_noalloc_scratch[KINV_NOALLOC_SCRATCH_BYTES];

namespace kinv {
namespace {

// In host code the array's name is a host-side stand-in, not a device
// address: the device address is looked up with the device current, checked,
// and cached per CUDA context (a context created again after cudaDeviceReset
// loads the module afresh and gets its own lookup).
void* noalloc_scratch_address() {
  static std::mutex mu;
  static std::map<unsigned long long, void*> addr;
  std::lock_guard<std::mutex> lock(mu);
  unsigned long long ctx = context_id();
  if (ctx != 0) {
    auto it = addr.find(ctx);
    if (it != addr.end()) return it->second;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, kinv_noalloc_scratch) != cudaSuccess || !p) return nullptr;
  ctx = context_id();  // the lookup makes the primary context current if none was
  if (ctx != 0) addr[ctx] = p;
  return p;
}

}  // namespace
}  // namespace kinv

extern "C" kinv_status kinv_attn_decode_noalloc(const void* q, const void* k_cache,
                                                const void* v_cache, int64_t seq_stride,
                                                int64_t tok_stride, const int32_t* kv_len,
                                                void* out, int B, int Hq, int Hkv, int D, int Lmax,
                                                int split_len, float scale, kinv_stream stream) {
  // the checks of kinv_attn_decode, in its order, with an aligned stand-in
  // for the workspace and the scratch array's size as its size
  const void* aligned_placeholder = reinterpret_cast<const void*>(static_cast<uintptr_t>(256));
  const kinv_status st = decode_check(q, k_cache, v_cache, seq_stride, tok_stride, kv_len, out, B, Hq, Hkv,
                                      D, Lmax, split_len, aligned_placeholder,
                                      static_cast<size_t>(KINV_NOALLOC_SCRATCH_BYTES));
  if (st != KINV_OK || B == 0) return st;
  void* scratch = noalloc_scratch_address();
  if (!scratch) return KINV_ERR_CUDA;
  return decode_launch(q, k_cache, v_cache, seq_stride, tok_stride, kv_len, out, B, Hq, Hkv, D, Lmax, scale,
                       scratch, stream);
}
