// Batch-invariant split-KV attention for decode and prefill
// ("Deterministic and bit-exact inference", *technical*: attention is made
// batch-invariant by cutting the keys into splits of one fixed length, not
// into a fixed number of splits).
//
// A query row with L visible keys cuts them into splits of 256 keys at
// absolute offsets 0, 256, 512, ...; the cut depends only on L.  The softmax
// is taken in base 2 (2^(x log2 e) = e^x, the form FlashAttention uses), with
// c = fp32(scale * log2 e).  For every (row, query head) pair and split:
//   r_t  = q . k_t             sixteen-deep tensor-core steps over d,
//                              ascending, accumulated in fp32
//   m    = fp32(max_t r_t * c) (max is exact in any order, and rounding a
//                              product by c > 0 keeps the order)
//   e_t  = 2^fma(r_t, c, -m)   ex2.approx; then carried as the bf16 pair
//   hi_t = bf16(e_t), lo_t = bf16(e_t - hi_t)   (about 16 significant bits)
//   l    = sum_t e_t           in 32-key groups: within a group key
//                              8nb + 2tq + e is added to partial tq in (nb, e)
//                              order, the partials (0 + 1) + (2 + 3), the
//                              groups in order
//   o[d] = one fp32 chain over sixteen 16-key steps, ascending; each step
//          adds its hi . v, then its lo . v
// and the splits are folded in ascending order with the log-sum-exp update
// (factors 2^(m_old - m_new), 2^(m_split - m_new)), then o / l -> bf16.  A key
// a pair cannot see gets weight 0; keys past the split's end read zero V.  A
// pair's bits depend only on its own q row and its sequence's keys and values.
//
// Decode (one new row per sequence): the split kernel, one block (eight
// warps, warp-level mma.sync m16n8k16) per (split, kv head, sequence), stores
// each split's (m, l, o) partial; the merge kernel folds them.  Prefill (rows
// of a prompt chunk): one tcgen05 block per (sequence, kv head, 128 pairs)
// folds the splits on chip.  A 16-deep tcgen05 step gives each element the
// bits of the mma.sync step, and both take the sums above in the same order,
// so a decode step equals a one-row prefill bit for bit and a prompt's rows
// have the same bits for every chunking.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <cmath>

#include <mutex>
#include <type_traits>

#include "common.cuh"

namespace kinv {
namespace {

constexpr int kSplit = 256;      // keys per split (the fixed split size)
constexpr int kThreads = 256;    // eight warps, 32 keys each for the scores
constexpr int kMaxG = 8;         // query heads per kv head
constexpr int kRowsP = 8;        // P rows kept in shared memory (G <= 8); the rest read a zero row

struct AttnParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  int64_t seq_stride, tok_stride;
  const int32_t* kv_len;
  __nv_bfloat16* out;
  float* ws_o;              // [B][Hq][S][D]
  float* ws_ml;             // [B][Hq][S][2]
  int Hq, Hkv, G;
  int S;                    // splits per row in the workspace
  float c2;                 // fp32(scale * log2 e) > 0
  int max_len;              // Lmax: the bound 0 <= kv_len[b] <= Lmax (the host cannot read kv_len)
  int* status;              // device status word (a sequence outside the bound)
};

// A sequence whose kv_len breaks the bound gets zeros and the call records
// DEV_ATTN_BAD_LENGTH, so no access leaves the caller's buffers.
__device__ __forceinline__ bool seq_ok(const AttnParams& p, int b) {
  const int n = p.kv_len[b];
  return n >= 0 && n <= p.max_len;
}

__device__ __forceinline__ void report_bad_length(const AttnParams& p) {
  if (threadIdx.x == 0 && p.status) atomicExch(p.status, DEV_ATTN_BAD_LENGTH);
}

// A 16-byte cp.async with an L2 eviction policy (createpolicy).
__device__ __forceinline__ void cp_async16_hint(uint32_t dst, const void* src, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "l"(policy)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
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
  // P_hi and P_lo [8][256]: the MMA's rows 8-15 (no (row, head) pair when
  // G <= 8) read a row of zeros
  __nv_bfloat16* pt = reinterpret_cast<__nv_bfloat16*>(smem_raw + kSplit * D * 2);
  __nv_bfloat16* pt_lo = pt + kRowsP * kSplit;
  unsigned char* zrow = reinterpret_cast<unsigned char*>(pt_lo + kRowsP * kSplit);  // [256] zeros
  __shared__ float wmax[kThreads / 32][kRowsP];
  __shared__ float wsum[kThreads / 32][kRowsP];

  pdl_launch_dependents();
  pdl_wait();
  // kv heads are the fastest grid index: the blocks reading the 256-byte
  // slices of the same token rows run side by side
  const int g = blockIdx.x;
  const int s = blockIdx.y;
  const int b = blockIdx.z;
  if (!seq_ok(p, b)) {
    report_bad_length(p);
    return;
  }
  const int len = p.kv_len[b];
  const int k0 = s * kSplit;
  const int nmax = min(kSplit, len - k0);              // keys of this split
  if (nmax <= 0) return;
  const int G = p.G;                                   // (row, head) pairs: MMA rows 0..G-1
  const int t = threadIdx.x;
  const int lane = t & 31, warp = t >> 5;
  const int gq = lane >> 2, tq = lane & 3;             // fragment row / column group
  const int64_t seq_off = b * p.seq_stride + static_cast<int64_t>(k0) * p.tok_stride + g * D;
  const uint32_t kv_base = smem_addr(kv);
  const uint32_t pt_base = smem_addr(pt), pt_lo_base = smem_addr(pt_lo), zrow_base = smem_addr(zrow);

  // each K/V row is read once per step: it should not push the partials
  // (read back by the merge) out of L2
  const uint64_t kv_policy = l2_policy_evict_first();
  auto load_sub = [&](const __nv_bfloat16* src, int j) {
    const int rows = min(SUB, nmax - j * SUB);
    for (int idx = t; idx < rows * C8; idx += kThreads) {
      const int r = idx / C8, c = idx % C8;
      const int key = j * SUB + r;
      cp_async16_hint(kv_base + static_cast<uint32_t>(key * D * 2 + ((c ^ (key & 7)) << 4)),
                      src + seq_off + static_cast<int64_t>(key) * p.tok_stride + c * 8, kv_policy);
    }
  };
#pragma unroll
  for (int j = 0; j < NSUB; ++j) load_sub(p.k, j);
  cp_async_commit();

  // q fragments (A operand, rows = (row, head) pairs), straight from global
  uint32_t qa[KS][4];
  {
    const int r_lo = gq, r_hi = gq + 8;
    const __nv_bfloat16* q_lo = r_lo < G ? p.q + (static_cast<int64_t>(b) * p.Hq + g * G + r_lo) * D : nullptr;
    const __nv_bfloat16* q_hi = r_hi < G ? p.q + (static_cast<int64_t>(b) * p.Hq + g * G + r_hi) * D : nullptr;
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

  // --- softmax statistics.  A lane holds row gq (pair gq < G; the
  // fragment's rows gq + 8 hold no pair), keys 32w + 8nb + 2tq (+1).  Maxima
  // of the raw scores: lane, then the four lanes of a row (exact), then the
  // eight warps; m = fp32(max * c).  The sum adds the weights e: a lane's
  // eight in (nb, pair) order, a fixed butterfly over the four lanes, the
  // eight warps in ascending order.
  const int cnt = gq < G ? nmax : 0;
  float mx = -INFINITY;
#pragma unroll
  for (int nb = 0; nb < 4; ++nb) {
#pragma unroll
    for (int e = 0; e < 2; ++e)
      if (warp * 32 + nb * 8 + 2 * tq + e < cnt) mx = fmaxf(mx, sc[nb][e]);
  }
#pragma unroll
  for (int o = 1; o <= 2; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (tq == 0) wmax[warp][gq] = mx;
  __syncthreads();
  float m = wmax[0][gq];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) m = fmaxf(m, wmax[w][gq]);
  m = __fmul_rn(m, p.c2);
  float sum = 0.f;
  uint32_t hp[4], lp[4];  // bf16 pairs of the high and the low halves
#pragma unroll
  for (int nb = 0; nb < 4; ++nb) {
    float x[2], h[2], l[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      x[e] = warp * 32 + nb * 8 + 2 * tq + e < cnt ? ex2_approx(__fmaf_rn(sc[nb][e], p.c2, -m)) : 0.f;
      split_bf16(x[e], h[e], l[e]);
      sum = __fadd_rn(sum, x[e]);
    }
    hp[nb] = pack_bf16(h[0], h[1]);
    lp[nb] = pack_bf16(l[0], l[1]);
  }
  // row gq of the P tiles (8-key chunk kc at chunk kc ^ gq)
#pragma unroll
  for (int nb = 0; nb < 4; ++nb) {
    const int kc = warp * 4 + nb;
    const uint32_t off = static_cast<uint32_t>(gq * kSplit * 2 + ((kc ^ gq) << 4) + 4 * tq);
    *reinterpret_cast<uint32_t*>(reinterpret_cast<unsigned char*>(pt) + off) = hp[nb];
    *reinterpret_cast<uint32_t*>(reinterpret_cast<unsigned char*>(pt_lo) + off) = lp[nb];
  }
  if (t < kSplit * 2 / 16) *reinterpret_cast<uint4*>(zrow + 16 * t) = make_uint4(0, 0, 0, 0);
#pragma unroll
  for (int o = 1; o <= 2; o <<= 1) sum = __fadd_rn(sum, __shfl_xor_sync(0xffffffffu, sum, o));
  if (tq == 0) wsum[warp][gq] = sum;
  cp_async_wait<0>();
  __syncthreads();

  // --- o = P . V: warp w owns columns 16w .. 16w + 15 (two 8-wide n
  // blocks) over all 256 keys: sixteen k steps of 16 keys in ascending order,
  // each adding its high halves, then its low halves, to one fp32 chain.
  float oc[2][4];
#pragma unroll
  for (int nb = 0; nb < 2; ++nb)
#pragma unroll
    for (int i = 0; i < 4; ++i) oc[nb][i] = 0.f;
  if (warp < D / 16) {
    const int prow = lane & 15;
#pragma unroll 4
    for (int kk = 0; kk < kSplit / 16; ++kk) {
      uint32_t ah[4], al[4];
      {
        const int kc = 2 * kk + (lane >> 4);
        const uint32_t chunk = static_cast<uint32_t>((kc ^ (prow & 7)) << 4);
        const uint32_t off = static_cast<uint32_t>(prow * kSplit * 2) + chunk;
        ldsm_x4(prow < kRowsP ? pt_base + off : zrow_base + chunk, ah[0], ah[1], ah[2], ah[3]);
        ldsm_x4(prow < kRowsP ? pt_lo_base + off : zrow_base + chunk, al[0], al[1], al[2], al[3]);
      }
      uint32_t b0, b1, b2, b3;
      {
        const int key = kk * 16 + (lane & 15);
        const int c = warp * 2 + (lane >> 4);
        ldsm_x4_t(kv_base + static_cast<uint32_t>(key * D * 2 + ((c ^ (key & 7)) << 4)), b0, b1, b2, b3);
      }
      mma_bf16_16816(oc[0], ah, b0, b1);
      mma_bf16_16816(oc[1], ah, b2, b3);
      mma_bf16_16816(oc[0], al, b0, b1);
      mma_bf16_16816(oc[1], al, b2, b3);
    }
    // row gq = query head g G + gq of sequence b, columns 16w + 8nb + 2tq (+1)
    if (gq < G) {
      const int64_t base = (static_cast<int64_t>(b) * p.Hq + g * G + gq) * p.S + s;
#pragma unroll
      for (int nb = 0; nb < 2; ++nb)
        *reinterpret_cast<float2*>(p.ws_o + base * D + warp * 16 + nb * 8 + 2 * tq) =
            make_float2(oc[nb][0], oc[nb][1]);
      if (warp == 0 && tq == 0) {
        float l = wsum[0][gq];
#pragma unroll
        for (int w = 1; w < kThreads / 32; ++w) l = __fadd_rn(l, wsum[w][gq]);
        p.ws_ml[base * 2 + 0] = m;
        p.ws_ml[base * 2 + 1] = l;
      }
    }
  }
}

// One block per (query head, row); thread d folds column d.
template <int D>
__global__ void attn_merge_kernel(const AttnParams p) {
  pdl_launch_dependents();
  pdl_wait();
  const int row = blockIdx.y;
  int len = 0;  // a sequence outside the bound gets zeros
  if (!seq_ok(p, row))
    report_bad_length(p);
  else
    len = p.kv_len[row];
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
        const float a = ex2_approx(__fsub_rn(m_acc, m_new));
        const float c = ex2_approx(__fsub_rn(mv[i], m_new));
        l_acc = __fadd_rn(__fmul_rn(l_acc, a), __fmul_rn(lv[i], c));
        o_acc = __fadd_rn(__fmul_rn(o_acc, a), __fmul_rn(ov[i], c));
        m_acc = m_new;
      }
    }
  }
  *dst = __float2bfloat16_rn(__fdiv_rn(o_acc, l_acc));
}

// ---------------------------------------------------------------------------
// Prefill on the tcgen05 tensor cores.  One block per (sequence, kv head,
// tile of 128 (row, head) pairs: 128 / G consecutive rows, each with its G
// query heads); it walks the 256-key splits the tile's rows can see in
// ascending order and folds each split into a running (m, l, o) per pair in
// registers with the merge kernel's arithmetic, so no partial goes to memory.
// Per pair and split it computes what attn_split_kernel computes:
//   R = Q . K^T         tcgen05 128 x 128 x 16 steps over the head dimension,
//                       ascending, fp32 in tensor memory (the per-element
//                       result of a 16-deep step equals mma.sync's), two
//                       128-key halves
//   max, e = 2^fma(r, c, -m), hi / lo, l in the decode kernel's order
//   O = P . V           one chain of sixteen 16-key steps, each the hi step
//                       then the lo step, P read from tensor memory
// and then folds as the merge kernel does; out = bf16(o / l).  So a prompt
// row has the bits of the decode step at its position.
// Roles (320 threads): warps 0-7 take the pairs (TMEM lane = pair), two
// threads per pair: warp w handles keys 128 (w / 4) .. + 127 of each split
// (chunks 2 (w / 4) and 2 (w / 4) + 1) and output columns D/2 (w / 4) ..
// + D/2 - 1 of the fold; the two exchange their maxima and 32-key group sums
// through shared memory, so the sums keep their order.  Warp 8 lane 0 issues
// the MMAs; warp 9 issues the TMA loads of Q, K and V and zeroes V rows past
// the tile's last visible key.
// Tensor memory: R of a split in columns 0-255 (chunk j at 64 j); once a
// thread has read its chunk it writes the chunk's P there as packed bf16
// pairs (32-key group h of the chunk: hi at 64 j + 32 h, lo 16 columns
// further), which the PV MMAs read as their A operand; O in two buffers after
// it, so split s + 1's PV runs while split s is folded.  The MMA thread
// issues split s + 1's R half h right after split s's PV chunks 2h and
// 2h + 1 (the MMAs run in issue order, so their P is read before R
// overwrites it), and the softmax threads fold split s after writing split
// s + 1's P.
constexpr int kTcThreads = 320;
constexpr int kTcPairs = 128;
constexpr int kTcBars = 17;

struct PrefillTcArgs {
  const int32_t* q_start;
  const int32_t* q_len;
  const int32_t* q_offset;
  __nv_bfloat16* out;
  int Hq, Hkv, G, RT;  // RT rows per tile (128 / G)
  int tiles_per_seq;
  int max_len, max_q_len, total_rows;
  float c2;            // fp32(scale * log2 e) > 0
  int* status;
};

// tcgen05 instruction descriptor, kind::f16: fp32 accumulate, bf16 A and B,
// A K-major, B K-major (b_mn = 0) or MN-major (b_mn = 1), N, M = 128.
__host__ __device__ constexpr uint32_t tc_idesc(int n, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(b_mn) << 16) |
         (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(128 >> 4) << 24);
}
// Shared-memory descriptors, 128-byte swizzle, version 1.  K-major: rows of
// 128 bytes (64 bf16 of K), 8-row groups 1024 bytes apart.  MN-major: rows of
// 128 bytes along MN (64 bf16) per K index, 8 K rows 1024 bytes apart (stride
// field), the next 64 MN elements `mn_stride` bytes further (leading field).
__device__ __forceinline__ uint64_t desc_k_sw128(uint32_t addr) {
  return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (1ull << 16) | (64ull << 32) | (1ull << 46) |
         (2ull << 61);
}
__device__ __forceinline__ uint64_t desc_mn_sw128(uint32_t addr, uint32_t mn_stride) {
  return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>((mn_stride >> 4) & 0x3FFFu) << 16) |
         (64ull << 32) | (1ull << 46) | (2ull << 61);
}

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    attn_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV, const PrefillTcArgs a) {
  constexpr int DS = D / 64;                   // 64-wide slices of the head dimension
  constexpr int Q_SLICE = kTcPairs * 128;      // [128 pairs][64]
  constexpr int Q_BYTES = DS * Q_SLICE;
  constexpr int KV_SLICE = kSplit * 128;       // [256 keys][64] per slice
  constexpr int KV_BYTES = DS * KV_SLICE;
  constexpr int DH = D / 2;                    // output columns per thread
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char* q_s = base;
  unsigned char* k_s = q_s + Q_BYTES;
  unsigned char* v_s = k_s + KV_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(v_s + KV_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kTcBars + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // the two threads of a pair exchange their raw maxima [2][128] and their
  // 32-key group sums [8][128]
  float* x_max = reinterpret_cast<float*>(tmem_slot + 4);
  float* x_w = x_max + 2 * kTcPairs;
  const uint32_t q_full = smem_addr(bars + 0), k_full = smem_addr(bars + 1), k_empty = smem_addr(bars + 2);
  const uint32_t v_full = smem_addr(bars + 3), v_ready = smem_addr(bars + 4), v_empty = smem_addr(bars + 5);
  auto s_full = [&](int h) { return smem_addr(bars + 6 + h); };     // R chunks 2h, 2h + 1 written
  auto p_full = [&](int j) { return smem_addr(bars + 8 + j); };     // P chunk j written
  auto o_full = [&](int i) { return smem_addr(bars + 12 + i); };    // O buffer i complete
  auto o_empty = [&](int i) { return smem_addr(bars + 14 + i); };   // O buffer i read
  const uint32_t done_bar = smem_addr(bars + 16);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, t = threadIdx.x;
  const int g = blockIdx.y;
  const int b = blockIdx.z;
  const int tile = a.tiles_per_seq - 1 - static_cast<int>(blockIdx.x);  // the longest tiles first
  pdl_wait();
  // the sequence's device-side lengths within the stated bounds, else left out
  const int n = a.q_len[b], st0 = a.q_start[b], off = a.q_offset[b];
  if (!(n >= 0 && n <= a.max_q_len && st0 >= 0 && st0 <= a.max_len - n && off >= 0 && off <= a.total_rows - n)) {
    if (t == 0 && tile == 0 && a.status) atomicExch(a.status, DEV_ATTN_BAD_LENGTH);
    return;
  }
  const int first = tile * a.RT;
  if (first >= n) return;
  const int nrows = min(a.RT, n - first);
  const int row0 = off + first;           // q / out row of the tile's first row
  const int len0 = st0 + first + 1;       // keys the first row sees (row r: len0 + r)
  const int len_last = len0 + nrows - 1;
  const int ns = (len_last + kSplit - 1) / kSplit;

  if (t == 0) {
    for (int i = 0; i < kTcBars; ++i) {
      // p_full: the 128 threads of the half that writes the chunk; o_empty:
      // all 256 softmax threads; the rest one arrival (a thread or a commit)
      const int count = (i >= 8 && i < 12) ? kTcPairs : (i == 14 || i == 15) ? 2 * kTcPairs : 1;
      mbar_init(smem_addr(bars + i), count);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 8) tmem_alloc(smem_addr(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();  // after the TMEM allocation (see the GEMM kernels)
  int* status = a.status;

  if (warp == 9) {
    // ---- TMA: Q once; K of split s + 1 as soon as split s's R MMAs are
    // done, V of split s + 1 as soon as split s's PV MMAs are done.  V rows
    // past the tile's last visible key are zeroed (stale cache rows may hold
    // anything, and their weight 0 times a NaN would not be 0).
    const uint64_t pol = l2_policy_evict_last();
    bool stop = false;
    int k_issued = 0, v_issued = 0;  // splits whose K / V loads were issued
    auto load_k = [&](int s) {
      mbar_arrive_expect_tx(k_full, KV_BYTES);
      for (int ds = 0; ds < DS; ++ds)
        tma_load_4d(smem_addr(k_s + ds * KV_SLICE), &tmK, 64 * ds, g, s * kSplit, b, k_full, pol);
      k_issued = s + 1;
    };
    auto load_v = [&](int s) {
      mbar_arrive_expect_tx(v_full, KV_BYTES);
      for (int ds = 0; ds < DS; ++ds)
        tma_load_4d(smem_addr(v_s + ds * KV_SLICE), &tmV, 64 * ds, g, s * kSplit, b, v_full, pol);
      v_issued = s + 1;
    };
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmQ)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmK)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmV)) : "memory");
      mbar_arrive_expect_tx(q_full, Q_BYTES);
      for (int ds = 0; ds < DS; ++ds)
        tma_load_3d(smem_addr(q_s + ds * Q_SLICE), &tmQ, 64 * ds, g * a.G, row0, q_full, pol);
      load_k(0);
      load_v(0);
    }
    for (int s = 0; s < ns && !stop; ++s) {
      const uint32_t ph = s & 1;
      if (lane == 0) {
        bool ok = true;
        if (s + 1 < ns) {
          ok = !*abort_flag && mbar_wait_bounded(k_empty, ph, status, DEV_TIMEOUT_ATTN);
          if (ok) load_k(s + 1);
        }
        if (ok) ok = mbar_wait_bounded(v_full, ph, status, DEV_TIMEOUT_ATTN);
        if (!ok) *abort_flag = 1;
      }
      stop = __shfl_sync(0xffffffffu, *abort_flag, 0) != 0;
      if (stop) break;
      const int nmax = min(kSplit, len_last - s * kSplit);
      for (int idx = lane; idx < (kSplit - nmax) * DS * 8; idx += 32) {
        const int key = nmax + idx / (DS * 8), rest = idx % (DS * 8);
        *reinterpret_cast<uint4*>(v_s + (rest / 8) * KV_SLICE + key * 128 + (rest % 8) * 16) = make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(v_ready);
        if (s + 1 < ns) {
          const bool ok = !*abort_flag && mbar_wait_bounded(v_empty, ph, status, DEV_TIMEOUT_ATTN);
          if (ok) load_v(s + 1);
          else *abort_flag = 1;
        }
      }
    }
    if (lane == 0) {
      // loads still in flight (only after an abort) land before the block exits
      mbar_wait_bounded(q_full, 0, nullptr, 0);
      if (k_issued > 0) mbar_wait_bounded(k_full, (k_issued - 1) & 1u, nullptr, 0);
      if (v_issued > 0) mbar_wait_bounded(v_full, (v_issued - 1) & 1u, nullptr, 0);
    }
    __syncwarp();
  } else if (warp == 8) {
    // ---- MMA issue: iteration s issues split s - 1's PV chunks and split
    // s's R chunks, interleaved
    if (lane == 0) {
      constexpr uint32_t idesc_r = tc_idesc(128, 0);
      constexpr uint32_t idesc_o = tc_idesc(D, 1);
      bool ok = mbar_wait_bounded(q_full, 0, status, DEV_TIMEOUT_ATTN);
      // base descriptors; an operand at byte offset b from a base adds b / 16
      // to the start-address field (shared addresses stay below 256 KB, so
      // the field never carries into the next)
      const uint64_t qd = desc_k_sw128(smem_addr(q_s)), kd = desc_k_sw128(smem_addr(k_s));
      const uint64_t vd = desc_mn_sw128(smem_addr(v_s), KV_SLICE);
      for (int s = 0; s <= ns && ok; ++s) {
        const bool has_r = s < ns, has_pv = s > 0;
        const int sp = s - 1;
        const uint32_t o_col = tmem + 256 + static_cast<uint32_t>((sp & 1) * D);
        if (has_pv)
          ok = !*abort_flag && mbar_wait_bounded(v_ready, sp & 1, status, DEV_TIMEOUT_ATTN) &&
               mbar_wait_bounded(o_empty(sp & 1), ((sp >> 1) & 1) ^ 1, status, DEV_TIMEOUT_ATTN);
        if (ok && has_r) ok = !*abort_flag && mbar_wait_bounded(k_full, s & 1, status, DEV_TIMEOUT_ATTN);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (has_pv) {
            ok = !*abort_flag && mbar_wait_bounded(p_full(j), sp & 1, status, DEV_TIMEOUT_ATTN);
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t vdesc = vd + static_cast<uint64_t>(((4 * j + kk) * 2048) >> 4);
              const uint32_t p_hi = tmem + static_cast<uint32_t>(64 * j + 32 * (kk >> 1) + 8 * (kk & 1));
              umma_bf16_tmem_a(o_col, p_hi, vdesc, idesc_o, (j | kk) != 0 ? 1u : 0u);
              umma_bf16_tmem_a(o_col, p_hi + 16, vdesc, idesc_o, 1u);
            }
          }
          if (has_r && (j & 1)) {
            // R of chunks j - 1 and j (keys 128 h .. + 127, h = j / 2): one
            // 128 x 128 MMA per 16-deep step
            const int h = j >> 1;
#pragma unroll
            for (int ds = 0; ds < DS; ++ds)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                umma_bf16(tmem + static_cast<uint32_t>(128 * h),
                          qd + static_cast<uint64_t>((ds * Q_SLICE + kk * 32) >> 4),
                          kd + static_cast<uint64_t>((ds * KV_SLICE + h * 128 * 128 + kk * 32) >> 4), idesc_r,
                          (ds | kk) != 0 ? 1u : 0u);
            umma_commit(s_full(h));
          }
        }
        if (!ok) break;
        if (has_pv) {
          umma_commit(v_empty);
          umma_commit(o_full(sp & 1));
        }
        if (has_r) umma_commit(k_empty);
      }
      if (!ok) *abort_flag = 1;
      umma_commit(done_bar);
      mbar_wait_bounded(done_bar, 0, status, DEV_TIMEOUT_ATTN);
    }
    __syncwarp();
  } else {
    // ---- two threads per (row, head) pair
    const int pr = t & (kTcPairs - 1);                   // pair = TMEM lane
    const int half = t >> 7;                             // keys 128 half .., columns D/2 half ..
    const int r = pr / a.G, hi_head = g * a.G + pr % a.G;
    const int len = len0 + r;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const float c2 = a.c2;
    float o_acc[DH];
#pragma unroll
    for (int d = 0; d < DH; ++d) o_acc[d] = 0.f;
    float m_acc = -INFINITY, l_acc = 0.f;
    bool ok = true;
    auto softmax_sync = []() { asm volatile("bar.sync 1, 256;" ::: "memory"); };
    // named barrier 1 over the 256 softmax threads, returning whether `v`
    // holds for any of them
    auto softmax_sync_or = [](bool v) {
      uint32_t r;
      asm volatile(
          "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
          "bar.red.or.pred p, 1, 256, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
          : "=r"(r)
          : "r"(static_cast<uint32_t>(v))
          : "memory");
      return r != 0;
    };
    auto check = [&](bool waited) {
      if (__any_sync(0xffffffffu, !waited || *abort_flag)) {
        *abort_flag = 1;
        ok = false;
      }
    };
    // folds split sf (maximum mf, sum lf, visible keys or not) into the
    // running state, this thread's D/2 output columns of O buffer sf & 1
    auto fold = [&](int sf, float mf, float lf, bool in) {
      check(mbar_wait_bounded(o_full(sf & 1), (sf >> 1) & 1, status, DEV_TIMEOUT_ATTN));
      tc_fence_after();
      const float m_new = fmaxf(m_acc, mf);
      const float fa = ex2_approx(__fsub_rn(m_acc, m_new));
      const float fc = ex2_approx(__fsub_rn(mf, m_new));
      // o * 1 = o exactly: where no pair of the warp moves its maximum the
      // update drops that product
      const bool unit = __all_sync(0xffffffffu, !in || fa == 1.f);
      if (in) l_acc = __fadd_rn(__fmul_rn(l_acc, fa), __fmul_rn(lf, fc));
      const uint32_t col = lane_base + 256 + static_cast<uint32_t>((sf & 1) * D + half * DH);
#pragma unroll
      for (int c = 0; c < DH / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(col + 32 * c, v);
        // the same roundings on pairs of columns (packed fp32x2 multiply and add)
        if (in) {
          const float2 fc2 = make_float2(fc, fc), fa2 = make_float2(fa, fa);
#pragma unroll
          for (int jj = 0; jj < 32; jj += 2) {
            float2 o = make_float2(o_acc[32 * c + jj], o_acc[32 * c + jj + 1]);
            const float2 t = __fmul2_rn(make_float2(__uint_as_float(v[jj]), __uint_as_float(v[jj + 1])), fc2);
            o = __fadd2_rn(unit ? o : __fmul2_rn(o, fa2), t);
            o_acc[32 * c + jj] = o.x;
            o_acc[32 * c + jj + 1] = o.y;
          }
        }
      }
      if (in) m_acc = m_new;
      tc_fence_before();
      mbar_arrive(o_empty(sf & 1));
    };
    float m_prev = 0.f, l_prev = 0.f;
    bool in_prev = false;
    for (int s = 0; s < ns; ++s) {
      const uint32_t ph = s & 1;
      const int cnt = min(kSplit, len - s * kSplit);
      // every pair of the tile sees the whole split: no key is masked
      const bool whole = len0 - s * kSplit >= kSplit;
      check(mbar_wait_bounded(s_full(half), ph, status, DEV_TIMEOUT_ATTN));
      tc_fence_after();
      // the raw maximum (exact in any order): this thread's 128 keys, four
      // chains, then the pair's
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
      for (int c = 4 * half; c < 4 * half + 4; ++c) {
        uint32_t v[32];
        tmem_ld32(lane_base + 32 * c, v);
        if (whole) {
#pragma unroll
          for (int jj = 0; jj < 32; jj += 8) {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              mx[e] = fmax3(mx[e], __uint_as_float(v[jj + 2 * e]), __uint_as_float(v[jj + 2 * e + 1]));
          }
        } else {
#pragma unroll
          for (int jj = 0; jj < 32; jj += 4) {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (32 * c + jj + e < cnt) mx[e] = fmaxf(mx[e], __uint_as_float(v[jj + e]));
          }
        }
      }
      x_max[half * kTcPairs + pr] = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      // the exchange's barrier also takes one decision for all 256 threads:
      // leave if any of them has given up (a flag read after a plain barrier
      // could change between two threads' reads)
      if (softmax_sync_or(!ok || *abort_flag)) {
        ok = false;
        break;
      }
      const float m = __fmul_rn(fmaxf(x_max[pr], x_max[kTcPairs + pr]), c2);
      const float2 c2x2 = make_float2(c2, c2), neg_m2 = make_float2(-m, -m);
      // weights, their group sums (to x_w), and this half's two P chunks in place of R
#pragma unroll 1
      for (int jh = 0; jh < 2; ++jh) {
        const int j = 2 * half + jh;  // 64-key chunk of the split
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int c = 2 * j + h;  // 32-key group c
          uint32_t v[32];
          tmem_ld32(lane_base + 32 * c, v);
          uint32_t hp[16], lp[16];  // bf16 pairs of the high and the low halves
          // (two copies of the loop: without and with the mask test)
          auto weights = [&](auto masked) {
#pragma unroll
            for (int jj = 0; jj < 32; jj += 2) {
              // fma(r, c, -m) and x - hi on pairs (packed fp32x2; x - hi as
              // fma(hi, -1, x), the same single rounding)
              const float2 arg = __ffma2_rn(make_float2(__uint_as_float(v[jj]), __uint_as_float(v[jj + 1])), c2x2,
                                            neg_m2);
              float x[2] = {ex2_approx(arg.x), ex2_approx(arg.y)};
              if (decltype(masked)::value) {
#pragma unroll
                for (int e = 0; e < 2; ++e) x[e] = 32 * c + jj + e < cnt ? x[e] : 0.f;
              }
              const __nv_bfloat162 h2 = __float22bfloat162_rn(make_float2(x[0], x[1]));
              const __nv_bfloat162 l2 = __float22bfloat162_rn(
                  __ffma2_rn(__bfloat1622float2(h2), make_float2(-1.f, -1.f), make_float2(x[0], x[1])));
              hp[jj / 2] = *reinterpret_cast<const uint32_t*>(&h2);
              lp[jj / 2] = *reinterpret_cast<const uint32_t*>(&l2);
              v[jj] = __float_as_uint(x[0]);
              v[jj + 1] = __float_as_uint(x[1]);
            }
          };
          if (whole)
            weights(std::false_type{});
          else
            weights(std::true_type{});
          tmem_st16(lane_base + 64 * j + 32 * h, hp);
          tmem_st16(lane_base + 64 * j + 32 * h + 16, lp);
          // the decode kernel's order: key 8nb + 2tq + e into partial tq in
          // (nb, e) order, then (0 + 1) + (2 + 3)
          float sq[4];
#pragma unroll
          for (int tq = 0; tq < 4; ++tq) {
            float acc = 0.f;
#pragma unroll
            for (int nb = 0; nb < 4; ++nb)
#pragma unroll
              for (int e = 0; e < 2; ++e) acc = __fadd_rn(acc, __uint_as_float(v[8 * nb + 2 * tq + e]));
            sq[tq] = acc;
          }
          x_w[(2 * j + h) * kTcPairs + pr] = __fadd_rn(__fadd_rn(sq[0], sq[1]), __fadd_rn(sq[2], sq[3]));
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(p_full(j));
      }
      // l: the groups 0 .. 7 in order
      softmax_sync();
      float l = x_w[pr];
#pragma unroll
      for (int q = 1; q < 8; ++q) l = __fadd_rn(l, x_w[q * kTcPairs + pr]);
      if (s > 0) fold(s - 1, m_prev, l_prev, in_prev);
      m_prev = m;
      l_prev = l;
      in_prev = cnt > 0;
    }
    if (ok && ns > 0) fold(ns - 1, m_prev, l_prev, in_prev);
    if (ok && r < nrows) {
      __nv_bfloat16* dst = a.out + (static_cast<int64_t>(row0 + r) * a.Hq + hi_head) * D + half * DH;
#pragma unroll
      for (int d = 0; d < DH; d += 8) {
        uint4 o;
        o.x = pack_bf16(__fdiv_rn(o_acc[d + 0], l_acc), __fdiv_rn(o_acc[d + 1], l_acc));
        o.y = pack_bf16(__fdiv_rn(o_acc[d + 2], l_acc), __fdiv_rn(o_acc[d + 3], l_acc));
        o.z = pack_bf16(__fdiv_rn(o_acc[d + 4], l_acc), __fdiv_rn(o_acc[d + 5], l_acc));
        o.w = pack_bf16(__fdiv_rn(o_acc[d + 6], l_acc), __fdiv_rn(o_acc[d + 7], l_acc));
        *reinterpret_cast<uint4*>(dst + d) = o;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
size_t prefill_tc_smem_bytes() {
  return 1024 + static_cast<size_t>(D / 64) * kTcPairs * 128 + 2 * static_cast<size_t>(D / 64) * kSplit * 128 +
         (kTcBars + 1) * 8 + 16 + 10 * kTcPairs * 4;
}

template <int D>
size_t split_smem_bytes() {
  return static_cast<size_t>(kSplit) * D * 2 + (2 * kRowsP + 1) * static_cast<size_t>(kSplit) * 2;
}

// Decode: attn_split_kernel, then the merge.
template <int D>
kinv_status launch(const AttnParams& p, dim3 split_grid, dim3 merge_grid, cudaStream_t stream) {
  void (*kernel)(const AttnParams) = attn_split_kernel<D>;
  const size_t smem = split_smem_bytes<D>();
  const kinv_status attr = ensure_smem(reinterpret_cast<const void*>(kernel), smem);
  if (attr != KINV_OK) return attr;
  const kinv_status st = launch_kernel(kernel, split_grid, dim3(kThreads), smem, stream, 1, p);
  if (st != KINV_OK) return st;
  return launch_kernel(attn_merge_kernel<D>, merge_grid, dim3(D), 0, stream, 1, p);
}

PFN_cuTensorMapEncodeTiled_v12000 tma_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// A bf16 tensor of rank `r` (dims innermost first, byte strides of dims 1..),
// boxes of `box` elements, 128-byte swizzle, out-of-range elements zero.
bool encode_map(CUtensorMap* map, const void* ptr, int r, const uint64_t* dims, const uint64_t* strides,
                const uint32_t* box) {
  auto fn = tma_encoder();
  if (!fn) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < r; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < r) st[i] = strides[i];
  }
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, r, const_cast<void*>(ptr), d, st, bx, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Prefill with the tcgen05 kernel: one block per (sequence, kv head, tile of
// 128 (row, head) pairs).
template <int D>
kinv_status launch_prefill_tc(const void* q, const void* k_cache, const void* v_cache, int64_t seq_stride,
                              int64_t tok_stride, PrefillTcArgs a, int B, cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  const uint64_t qd[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(a.Hq), static_cast<uint64_t>(a.total_rows)};
  const uint64_t qs[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(a.Hq) * D * 2};
  const uint32_t qb[3] = {64, static_cast<uint32_t>(a.G), static_cast<uint32_t>(a.RT)};
  const uint64_t kd[4] = {static_cast<uint64_t>(D), static_cast<uint64_t>(a.Hkv), static_cast<uint64_t>(a.max_len),
                          static_cast<uint64_t>(B)};
  // one sequence: any sequence stride describes it (the coordinate is 0)
  const int64_t sst = B > 1 ? seq_stride : static_cast<int64_t>(a.max_len) * tok_stride;
  const uint64_t ks[3] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(tok_stride) * 2,
                          static_cast<uint64_t>(sst) * 2};
  const uint32_t kb[4] = {64, 1, static_cast<uint32_t>(kSplit), 1};
  if (!encode_map(&mq, q, 3, qd, qs, qb) || !encode_map(&mk, k_cache, 4, kd, ks, kb) ||
      !encode_map(&mv, v_cache, 4, kd, ks, kb))
    return KINV_ERR_UNSUPPORTED;
  const size_t smem = prefill_tc_smem_bytes<D>();
  if (smem > static_cast<size_t>(max_smem_optin())) return KINV_ERR_UNSUPPORTED;
  const kinv_status attr = ensure_smem(reinterpret_cast<const void*>(attn_prefill_tc_kernel<D>), smem);
  if (attr != KINV_OK) return attr;
  return launch_kernel(attn_prefill_tc_kernel<D>, dim3(a.tiles_per_seq, a.Hkv, B), dim3(kTcThreads), smem, stream, 1,
                       mq, mk, mv, a);
}

// c = fp32(scale * log2 e), the scores' factor in the base-2 softmax; a
// scale that is not a positive finite number means 1 / sqrt(D).
float base2_factor(float scale, int D) {
  const float s = (scale > 0.f && std::isfinite(scale)) ? scale : 1.0f / sqrtf(static_cast<float>(D));
  return static_cast<float>(static_cast<double>(s) * 1.4426950408889634074);
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
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.S = S;
  p.c2 = base2_factor(scale, D);
  p.max_len = Lmax;
  p.status = device_status_word();
  const dim3 split_grid(Hkv, S, B), merge_grid(Hq, B, 1);
  return D == 128 ? launch<128>(p, split_grid, merge_grid, stream)
                  : launch<64>(p, split_grid, merge_grid, stream);
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
  // the splits are folded on chip: no workspace
  (void)total_rows;
  (void)Hq;
  (void)D;
  (void)max_kv;
  (void)split_len;
  return 0;
}

extern "C" kinv_status kinv_attn_prefill(const void* q, const void* k_cache, const void* v_cache,
                                         int64_t seq_stride, int64_t tok_stride,
                                         const int32_t* q_start, const int32_t* q_len,
                                         const int32_t* q_offset, void* out, int B,
                                         int total_rows, int max_q_len, int max_kv, int Hq,
                                         int Hkv, int D, int split_len, float scale,
                                         void* workspace, size_t ws_bytes, kinv_stream stream) {
  (void)ws_bytes;
  if (B < 0 || total_rows < 0 || max_q_len < 0 || max_kv < 0) return KINV_ERR_INVALID_ARG;
  if (B == 0 || total_rows == 0 || max_q_len == 0) return KINV_OK;
  if (!q_start || !q_len || !q_offset || max_kv <= 0) return KINV_ERR_INVALID_ARG;
  // no workspace is used; an aligned stand-in keeps the shared checks
  const void* aligned_placeholder = reinterpret_cast<const void*>(static_cast<uintptr_t>(256));
  kinv_status st = check_common(q, k_cache, v_cache, seq_stride, tok_stride, out, Hq, Hkv, D, split_len,
                                workspace ? workspace : aligned_placeholder);
  if (st != KINV_OK) return st;
  PrefillTcArgs a{};
  a.q_start = q_start;
  a.q_len = q_len;
  a.q_offset = q_offset;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.G = Hq / Hkv;
  a.RT = kTcPairs / a.G;
  a.tiles_per_seq = (max_q_len + a.RT - 1) / a.RT;
  a.max_len = max_kv;
  a.max_q_len = max_q_len;
  a.total_rows = total_rows;
  a.c2 = base2_factor(scale, D);
  a.status = device_status_word();
  if (a.tiles_per_seq > 65535 || B > 65535) return KINV_ERR_UNSUPPORTED;
  if (B > 1 && seq_stride <= 0) return KINV_ERR_INVALID_ARG;
  return D == 128 ? launch_prefill_tc<128>(q, k_cache, v_cache, seq_stride, tok_stride, a, B, stream)
                  : launch_prefill_tc<64>(q, k_cache, v_cache, seq_stride, tok_stride, a, B, stream);
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
