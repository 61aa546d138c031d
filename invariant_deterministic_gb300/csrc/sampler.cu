// Seeded, batch-invariant sampler (Kinetic "Receipts", *Making a receipt*:
// the receipt records temperature, top_k, top_p, min_p, the repeat, presence
// and frequency penalties, repeat_last_n and the seed, so the same settings
// must give the same token).
//
// Eight thread blocks (one cluster) per row, each owning a contiguous eighth
// of the vocabulary; they exchange the row maximum, threshold counts, radix
// histograms and their candidates through distributed shared memory, and
// rank 0 of the cluster finishes the row.  Nothing is shared between rows,
// and every quantity exchanged is an exact maximum, an integer count or a set
// of candidates, so the result does not depend on how the row is divided.
//  1. Logit bias and penalties: a shared-memory bitmap marks the distinct
//     ids among the row's last repeat_last_n history tokens and the ids of
//     its logit-bias list.  A marked logit first gets its bias entries added
//     (list order); then, if the id is in the window, z becomes z / r
//     (z > 0) or z * r, and, when a presence (p) or frequency (f) penalty is
//     set, z - (c * f + p) with c the id's count in the window; every
//     operation a correctly rounded fp32 one.  Each block computes the final
//     value of every marked id once, stored by the id's rank among the marked
//     ids (a per-word prefix count of the bitmap), so a visit of a marked id
//     is one table read.
//  2. Ranking uses the order-preserving 32-bit key of each penalised fp32
//     value and, for equal keys, the lower id first: a strict total order.
//     Greedy (temperature <= 0) takes its maximum.  Otherwise radix passes over
//     the key (11, 11, 10 bits) narrow a threshold until at most kCap ids lie
//     at or above it; those are gathered (slots come from an atomic counter,
//     which only decides where a candidate is parked) and bitonic-sorted by the
//     total order, so the candidate list does not depend on the parking order.
//     If more than kCap ids tie exactly at the threshold, the ties are taken
//     lowest id first by an ordered block-wide scan.
//  3. s_i = z_i / T; e_i = exp(s_i - s_0); the running sums in candidate
//     order (a fixed-order warp scan) give top-p, min-p and the draw.
//  4. The draw: u = (Philox4x32-10(counter = (step lo, step hi, 0, 0),
//     key = (seed lo, seed hi)).word0 >> 8) * 2^-24 (Salmon et al., SC'11,
//     restated here from the published round function and constants).
// Over the whole vocabulary (no top-k) nothing is gathered: every mass the
// filters and the draw need -- the total, the entropy of typical-p, the mass
// of the ids at or above a key -- is a masked sum over the whole row in one
// fixed order (4 ids in order per lane of a 128-id block, a butterfly over the
// lanes, a butterfly over the 32 blocks of a 4096-id group, the groups in
// order), and the cuts are found by searching the 32-bit keys, seven
// thresholds per pass, for where that mass crosses the target; ties at the cut
// key are taken lowest id first (equal keys, equal weights).  Counts and
// maxima are exact.
#include <math.h>

#include <mutex>

#include "common.cuh"

namespace kinv {
namespace {

constexpr int kThreadsS = 512;
constexpr int kMaxCluster = 8;  // blocks sharing one row, at most
constexpr int kMaxTopK = 1024;
constexpr int kCap = 4096;  // candidates gathered before sorting
constexpr int kMaxBlocks = 2048;  // full-vocabulary mode: 128-id blocks of the row (V <= 262144)
constexpr int kRounds = 10;  // 16-byte vectors of the row each thread keeps in registers
constexpr int kMaxHist = 1024;  // history row length (the penalty window) at most
constexpr int kMaxBias = 1024;  // logit-bias entries per row at most
constexpr int kMaxMarked = kMaxHist + kMaxBias;  // ids a row's bias and penalties can touch
constexpr int kRegSpan = kThreadsS * 4 * kRounds;  // ids a block holds in registers

__device__ __forceinline__ uint32_t ordered_key(float z) {
  if (isnan(z)) z = -INFINITY;
  const uint32_t u = __float_as_uint(z);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  const uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(u);
}

struct Philox4 {
  uint32_t x, y, z, w;
};

__device__ __forceinline__ Philox4 philox4x32_10(Philox4 c, uint32_t k0, uint32_t k1) {
  constexpr uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  constexpr uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += W0;
      k1 += W1;
    }
    const uint32_t hi0 = __umulhi(M0, c.x), lo0 = M0 * c.x;
    const uint32_t hi1 = __umulhi(M1, c.z), lo1 = M1 * c.z;
    c = Philox4{hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0};
  }
  return c;
}

struct Smem {
  unsigned long long cand[kCap];  // this block's candidates (rank 0: all of them)
  uint32_t hist[2048];            // this block's radix histogram (read by the peers)
  uint32_t comb[2048];            // the cluster's histogram
  float e[kMaxTopK];
  uint32_t warp_cnt[32];
  float wmax[32];
  int wcnt[32][8];
  unsigned long long wbest[32];
  int cnt[8];
  uint32_t offs[kMaxCluster + 1];
  // read by the peers
  float x_max;
  int x_cnt[8];
  unsigned long long x_best;
  uint32_t n_cand;
  // this block's copy of the cluster-wide decisions
  float m_all;
  // whole vocabulary: sums of one pass, per 128-id block of a group, per
  // 4096-id group of this block's share, and (rank 0) every group's
  float psum[16][32];
  float gsum[16][kMaxBlocks / 32];
  float gall[16][kMaxBlocks / 32];
  float res[16];          // the pass results (rank 0's, copied to every block)
  long long xi[2];        // this block's integer partials (counts, first ids)
  long long ires[2];      // the cluster's (copied to every block)
  uint32_t eq_taken;
  uint32_t thresh;
  int k_rem;
  int ok;
  int fast;
  float thresh_f;
  float typ_h;               // typical-p: -(entropy) of the candidates
  float mk_val[kMaxMarked];  // the final logit of each marked id, by rank
  int mk_cnt[kMaxMarked];    // its count in the penalty window
};

// The penalties of one row (step 1 above).
struct Penalty {
  const uint32_t* bitmap;   // marked ids: the window's and the bias list's
  const uint16_t* mk_base;  // marked ids in the words before each word
  const float* mk_val;      // the final logit of each marked id, by rank
};

__device__ __forceinline__ float penalise(float z, int id, const Penalty& pe) {
  const uint32_t word = pe.bitmap[id >> 5];
  const uint32_t below = (1u << (id & 31)) - 1u;
  if ((word >> (id & 31)) & 1u) z = pe.mk_val[pe.mk_base[id >> 5] + __popc(word & below)];
  return z;
}

// The final logit of a marked id with window count c: its bias entries in
// list order, then, if it is in the window (c > 0), the repeat penalty and the
// presence and frequency penalties.
__device__ float marked_value(float z, int id, const kinv_logit_bias* bias, int nb, int c, float r, float f,
                              float p, bool additive) {
  for (int j = 0; j < nb; ++j)
    if (bias[j].id == id) z = __fadd_rn(z, bias[j].bias);
  if (c > 0) {
    z = z > 0.f ? __fdiv_rn(z, r) : __fmul_rn(z, r);
    if (additive) z = __fsub_rn(z, __fadd_rn(__fmul_rn(static_cast<float>(c), f), p));
  }
  return z;
}

__device__ __forceinline__ float penalised(const float* __restrict__ row, int i, const Penalty& pe) {
  return penalise(row[i], i, pe);
}

// Visits every id in [v0, v1) once, in rounds in which each thread loads
// four 16-byte vectors (16 logits) before using any of them, so a pass keeps
// many loads in flight.  f(valid, id, value) sees the penalised logit (NaN as
// -inf); every lane runs the same number of rounds (f may use warp votes).
template <typename F>
__device__ __forceinline__ void for_each_value(const float* __restrict__ row, int v0, int v1,
                                               const Penalty& pe, F&& f) {
  constexpr int U = 4;
  const int t = threadIdx.x;
  const int n = v1 > v0 ? v1 - v0 : 0;
  const float* seg = row + v0;
  const bool vec = (reinterpret_cast<uintptr_t>(seg) & 15u) == 0;
  const int n4 = vec ? (n >> 2) : 0;
  const float4* seg4 = reinterpret_cast<const float4*>(seg);
  for (int base = 0; base < n4; base += kThreadsS * U) {
    float4 x[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i4 = base + u * kThreadsS + t;
      x[u] = i4 < n4 ? seg4[i4] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i4 = base + u * kThreadsS + t;
      const bool valid = i4 < n4;
      const float xv[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = v0 + 4 * i4 + e;
        float z = xv[e];
        if (valid) z = penalise(z, i, pe);
        f(valid, i, isnan(z) ? -INFINITY : z);
      }
    }
  }
  // the ids not covered by whole vectors, one per thread and round
  for (int base = 4 * n4; base < n; base += kThreadsS) {
    const int i = v0 + base + t;
    const bool valid = base + t < n;
    const float z = valid ? penalised(row, i, pe) : 0.f;
    f(valid, i, isnan(z) ? -INFINITY : z);
  }
}

__device__ __forceinline__ unsigned long long composite(uint32_t key, int id) {
  return (static_cast<unsigned long long>(key) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(id));
}

// Bitonic sort of n (power of two) composites, descending.
__device__ void bitonic_desc(unsigned long long* a, int n) {
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int j = i ^ stride;
        if (j > i) {
          const bool desc = (i & size) == 0;
          const unsigned long long x = a[i], y = a[j];
          if (desc ? (x < y) : (x > y)) {
            a[i] = y;
            a[j] = x;
          }
        }
      }
      __syncthreads();
    }
  }
}

template <bool kRegs>
__global__ void __launch_bounds__(kThreadsS) sample_kernel(
    const float* __restrict__ logits, int64_t ld, int V, const kinv_sampling_params* __restrict__ params,
    const int32_t* __restrict__ history, int hist_ld, const int32_t* __restrict__ hist_len,
    const int64_t* __restrict__ step, int32_t* __restrict__ out, int* status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(smem_raw + sizeof(Smem));
  uint16_t* mk_base = reinterpret_cast<uint16_t*>(bitmap + ((V + 31) >> 5));
  pdl_launch_dependents();
  pdl_wait();
  const int b = blockIdx.y;
  const int rank = static_cast<int>(cluster_ctarank());
  const int C = static_cast<int>(gridDim.x);  // the cluster: all blocks of this row
  const int t = threadIdx.x;
  const int lane = t & 31, warp = t >> 5;
  constexpr int kWarps = kThreadsS / 32;
  const float* row = logits + b * ld;
  const kinv_sampling_params prm = params[b];
  const int words = (V + 31) >> 5;
  // this block's ids: a multiple of 128 per rank (whole vectors, whole bitmap
  // words); over the whole vocabulary a multiple of 4096 (whole groups of its
  // sums)
  const bool whole_row = (prm.top_k <= 0 || prm.top_k >= V) && V > kMaxTopK && prm.temperature > 0.f;
  const int quantum = whole_row ? 4096 : 128;
  const int chunk = ((V + C - 1) / C + quantum - 1) / quantum * quantum;
  const int v0 = min(V, rank * chunk), v1 = min(V, v0 + chunk);
  auto peer = [](const void* p, int q) { return map_to_rank(smem_addr(p), static_cast<uint32_t>(q)); };

  // This block's logits, read once into registers when its share of the row
  // fits (thread t holds ids v0 + 2048 q + 4 t .. + 3 for round q); the loads
  // are in flight while the penalty tables below are built, and the penalties
  // are applied after.  Otherwise every pass streams the row from memory.
  const bool in_regs = kRegs && v1 - v0 <= kRegSpan;
  const bool vec = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
  float4 vr[kRegs ? kRounds : 1];
  if (in_regs) {
#pragma unroll
    for (int q = 0; q < (kRegs ? kRounds : 1); ++q) {
      const int i = v0 + q * kThreadsS * 4 + 4 * t;
      float x[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if (vec && i + 3 < v1) {
        const float4 f = *reinterpret_cast<const float4*>(row + i);
        x[0] = f.x; x[1] = f.y; x[2] = f.z; x[3] = f.w;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (i + e < v1) x[e] = row[i + e];
      }
      vr[q] = make_float4(x[0], x[1], x[2], x[3]);
    }
  }

  // 1. penalty bitmap (the whole row, in every block)
  for (int i = t; i < words; i += kThreadsS) bitmap[i] = 0u;
  __syncthreads();
  const float r = prm.repeat_penalty;
  const bool additive = prm.frequency_penalty != 0.f || prm.presence_penalty != 0.f;
  const int nb = prm.logit_bias ? min(max(prm.n_logit_bias, 0), kMaxBias) : 0;
  const int hl = hist_len ? min(max(hist_len[b], 0), hist_ld) : 0;
  int n_pen = prm.repeat_last_n < 0 ? hl : min(prm.repeat_last_n, hl);
  if (r == 1.0f && !additive) n_pen = 0;
  const int32_t* win_g = n_pen > 0 ? history + static_cast<int64_t>(b) * hist_ld + hl - n_pen : nullptr;
  for (int i = t; i < n_pen; i += kThreadsS) {
    const int id = win_g[i];
    if (id >= 0 && id < V) atomicOr(&bitmap[id >> 5], 1u << (id & 31));  // idempotent bit set
  }
  for (int i = t; i < nb; i += kThreadsS) {
    const int id = prm.logit_bias[i].id;
    if (id >= 0 && id < V) atomicOr(&bitmap[id >> 5], 1u << (id & 31));
  }
  __syncthreads();
  for (int i = t; i < kMaxMarked; i += kThreadsS) sm.mk_cnt[i] = 0;
  // rank of the marked ids: thread t takes words [t * per, (t + 1) * per),
  // a block-wide exclusive scan of their bit counts gives its first rank
  {
    const int per = (words + kThreadsS - 1) / kThreadsS;
    const int w0 = min(words, t * per), w1 = min(words, w0 + per);
    int cnt = 0;
    for (int w = w0; w < w1; ++w) cnt += __popc(bitmap[w]);
    int x = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) sm.warp_cnt[warp] = static_cast<uint32_t>(x);
    __syncthreads();
    int run = x - cnt;
    for (int w2 = 0; w2 < warp; ++w2) run += static_cast<int>(sm.warp_cnt[w2]);
    for (int w = w0; w < w1; ++w) {
      mk_base[w] = static_cast<uint16_t>(run);
      run += __popc(bitmap[w]);
    }
  }
  __syncthreads();
  // window counts by rank, then each marked id's final logit
  auto rank_of = [&](int id) {
    return mk_base[id >> 5] + __popc(bitmap[id >> 5] & ((1u << (id & 31)) - 1u));
  };
  for (int i = t; i < n_pen; i += kThreadsS) {
    const int id = win_g[i];
    if (id >= 0 && id < V) atomicAdd(&sm.mk_cnt[rank_of(id)], 1);
  }
  __syncthreads();
  {
    const int per = (words + kThreadsS - 1) / kThreadsS;
    const int w0 = min(words, t * per), w1 = min(words, w0 + per);
    for (int w = w0; w < w1; ++w) {
      uint32_t bits = bitmap[w];
      int k = mk_base[w];
      while (bits) {
        const int id = w * 32 + __ffs(bits) - 1;
        bits &= bits - 1u;
        sm.mk_val[k] = marked_value(row[id], id, prm.logit_bias, nb, sm.mk_cnt[k], r, prm.frequency_penalty,
                                    prm.presence_penalty, additive);
        ++k;
      }
    }
  }
  __syncthreads();
  const Penalty pe{bitmap, mk_base, sm.mk_val};

  if (in_regs) {
    // the penalties and NaN as -inf, on the values loaded at the start
#pragma unroll
    for (int q = 0; q < (kRegs ? kRounds : 1); ++q) {
      const int i = v0 + q * kThreadsS * 4 + 4 * t;
      float x[4] = {vr[q].x, vr[q].y, vr[q].z, vr[q].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float z = x[e];
        if (i + e < v1) z = penalise(z, i + e, pe);
        x[e] = isnan(z) ? -INFINITY : z;
      }
      vr[q] = make_float4(x[0], x[1], x[2], x[3]);
    }
  }
  // f(valid, id, value) over this block's ids; every lane makes the same calls
  auto visit = [&](auto&& f) {
    if (in_regs) {
#pragma unroll
      for (int q = 0; q < (kRegs ? kRounds : 1); ++q) {
        const int i = v0 + q * kThreadsS * 4 + 4 * t;
        f(i < v1, i, vr[q].x);
        f(i + 1 < v1, i + 1, vr[q].y);
        f(i + 2 < v1, i + 2, vr[q].z);
        f(i + 3 < v1, i + 3, vr[q].w);
      }
    } else {
      for_each_value(row, v0, v1, pe, f);
    }
  };
  auto visit_key = [&](auto&& f) {
    visit([&](bool valid, int i, float z) { f(valid, i, valid ? ordered_key(z) : 0u); });
  };

  const float temp = prm.temperature;

  // ---- the whole vocabulary (no top-k): masked sums and key searches
  auto whole_vocabulary = [&]() {
    constexpr int NS = 15;  // thresholds per search pass
    // the row maximum (exact, any order)
    {
      float mx = -INFINITY;
      visit([&](bool valid, int, float z) {
        if (valid) mx = fmaxf(mx, z);
      });
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      if (lane == 0) sm.wmax[warp] = mx;
      __syncthreads();
      if (t == 0) {
        float m = sm.wmax[0];
        for (int w = 1; w < kWarps; ++w) m = fmaxf(m, sm.wmax[w]);
        sm.x_max = m;
      }
      cluster_sync();
      if (warp == 0) {
        float m = lane < C ? ld_dsmem_f32(peer(&sm.x_max, lane)) : -INFINITY;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) sm.m_all = m;
      }
      __syncthreads();
    }
    const float s0 = __fdiv_rn(sm.m_all, temp);
    const uint32_t key_hi = ordered_key(sm.m_all);
    auto weight = [&](float z) { return expf(__fsub_rn(__fdiv_rn(z, temp), s0)); };
    const int groups = (V + 4095) / 4096;
    const int g0 = v1 > v0 ? v0 / 4096 : 0, g1 = v1 > v0 ? (v1 + 4095) / 4096 : 0;

    // nt sums of term(j, id, z, e) over the whole row in the fixed order (4
    // ids per lane of a 128-id block, a butterfly over the lanes, a butterfly
    // over the group's 32 blocks, the groups in order); every block gets
    // them in sm.res
    auto pass_sums = [&](int nt, auto&& term) {
      for (int g = g0; g < g1; ++g) {
        for (int bb = warp; bb < 32; bb += kWarps) {
          float acc[NS];
#pragma unroll
          for (int j = 0; j < NS; ++j) acc[j] = 0.f;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int i = (32 * g + bb) * 128 + 4 * lane + q;
            if (i < V) {
              float z = penalised(row, i, pe);
              if (isnan(z)) z = -INFINITY;
              const float e = weight(z);
#pragma unroll
              for (int j = 0; j < NS; ++j)
                if (j < nt) acc[j] = __fadd_rn(acc[j], term(j, i, z, e));
            }
          }
#pragma unroll
          for (int j = 0; j < NS; ++j) {
            if (j < nt) {
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) acc[j] = __fadd_rn(acc[j], __shfl_xor_sync(0xffffffffu, acc[j], o));
              if (lane == 0) sm.psum[j][bb] = acc[j];
            }
          }
        }
        __syncthreads();
        if (warp < nt) {
          float v = sm.psum[warp][lane];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
          if (lane == 0) sm.gsum[warp][g - g0] = v;
        }
        __syncthreads();
      }
      cluster_sync();  // every block's group sums are in place
      if (rank == 0) {
        for (int idx = t; idx < nt * groups; idx += kThreadsS) {
          const int j = idx / groups, g = idx % groups;
          const int q = g * 4096 / chunk;  // the block holding group g
          const int gl = g - q * (chunk / 4096);
          sm.gall[j][g] = q == 0 ? sm.gsum[j][gl] : ld_dsmem_f32(peer(&sm.gsum[j][gl], q));
        }
        __syncthreads();
        if (t < nt) {
          float acc = 0.f;
          for (int g = 0; g < groups; ++g) acc = __fadd_rn(acc, sm.gall[t][g]);
          sm.res[t] = acc;
        }
      }
      cluster_sync();  // rank 0's sums are in place
      if (rank != 0 && t < nt) sm.res[t] = ld_dsmem_f32(peer(&sm.res[t], 0));
      __syncthreads();
    };
    // over the ids with pred(id, z): the count (sm.ires[0]) and, with
    // `largest` false, the smallest composite (key, id) (the last in
    // candidate order), else the largest (the first), in sm.ires[1]
    auto pass_count = [&](bool largest, auto&& pred) {
      long long c = 0;
      unsigned long long best = largest ? 0ull : ~0ull;
      visit([&](bool valid, int i, float z) {
        if (valid && pred(i, z)) {
          ++c;
          const unsigned long long x = composite(ordered_key(z), i);
          best = largest ? (x > best ? x : best) : (x < best ? x : best);
        }
      });
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        c += __shfl_xor_sync(0xffffffffu, c, o);
        const unsigned long long y = __shfl_xor_sync(0xffffffffu, best, o);
        best = largest ? (y > best ? y : best) : (y < best ? y : best);
      }
      if (lane == 0) {
        sm.wcnt[warp][0] = static_cast<int>(c);
        sm.wbest[warp] = best;
      }
      __syncthreads();
      if (t == 0) {
        long long tc = 0;
        unsigned long long tb = largest ? 0ull : ~0ull;
        for (int w = 0; w < kWarps; ++w) {
          tc += sm.wcnt[w][0];
          tb = largest ? (sm.wbest[w] > tb ? sm.wbest[w] : tb) : (sm.wbest[w] < tb ? sm.wbest[w] : tb);
        }
        sm.xi[0] = tc;
        sm.xi[1] = static_cast<long long>(tb);
      }
      cluster_sync();
      if (t == 0) {
        long long tc = 0;
        unsigned long long tb = largest ? 0ull : ~0ull;
        for (int q = 0; q < C; ++q) {
          tc += static_cast<long long>(ld_dsmem_u64(peer(&sm.xi[0], q)));
          const unsigned long long y = ld_dsmem_u64(peer(&sm.xi[1], q));
          tb = largest ? (y > tb ? y : tb) : (y < tb ? y : tb);
        }
        sm.ires[0] = tc;
        sm.ires[1] = static_cast<long long>(tb);
      }
      cluster_sync();  // every block has read the partials
    };
    // the n-th smallest id (n >= 1) with pred(id, z), or -1
    auto pass_nth = [&](long long n, auto&& pred) {
      pass_count(true, pred);
      // the ids per block are in sm.xi[0] of each block (kept until the next
      // pass): the block holding the n-th one finds it by an ordered scan
      long long before = 0;
      int owner = -1;
      for (int q = 0; q < C; ++q) {
        const long long cq = static_cast<long long>(ld_dsmem_u64(peer(&sm.xi[0], q)));
        if (owner < 0 && n <= before + cq) owner = q;
        else if (owner < 0) before += cq;
      }
      __syncthreads();
      if (t == 0) sm.thresh = 0xFFFFFFFFu;
      __syncthreads();
      if (owner == rank) {
        long long run = before;
        for (int base = v0; base < v1; base += kThreadsS) {
          const int i = base + t;
          bool hit = false;
          if (i < v1) {
            float z = penalised(row, i, pe);
            if (isnan(z)) z = -INFINITY;
            hit = pred(i, z);
          }
          const unsigned bal = __ballot_sync(0xffffffffu, hit);
          if (lane == 0) sm.warp_cnt[warp] = __popc(bal);
          __syncthreads();
          long long r = run + __popc(bal & ((1u << lane) - 1u)) + 1;
          for (int w2 = 0; w2 < warp; ++w2) r += sm.warp_cnt[w2];
          if (hit && r == n) sm.thresh = static_cast<uint32_t>(i);
          long long tot = 0;
          for (int w2 = 0; w2 < kWarps; ++w2) tot += sm.warp_cnt[w2];
          __syncthreads();
          run += tot;
          if (run >= n) break;
        }
      }
      cluster_sync();
      int id = -1;
      if (owner >= 0) {
        const uint32_t x = ld_dsmem_u32(peer(&sm.thresh, owner));
        id = x == 0xFFFFFFFFu ? -1 : static_cast<int>(x);
      }
      cluster_sync();  // every block has read it
      return id;
    };
    // the largest key k with F(k) >= target (strict: > target), F(k) the sum
    // of e over the ids with in(id, z) and key >= k, F(0) meeting the target
    auto search_max = [&](auto&& in, float target, bool strict) {
      uint32_t lo = 0, hi = key_hi;
      while (lo < hi) {
        const unsigned long long span = static_cast<unsigned long long>(hi) - lo;
        uint32_t th[NS];
#pragma unroll
        for (int j = 0; j < NS; ++j)
          th[j] = lo + static_cast<uint32_t>((span * static_cast<unsigned long long>(j + 1) + NS) / (NS + 1));
        pass_sums(NS, [&](int j, int i, float z, float e) {
          return (ordered_key(z) >= th[j] && in(i, z)) ? e : 0.f;
        });
        int best = -1;
        for (int j = 0; j < NS; ++j)
          if (strict ? sm.res[j] > target : sm.res[j] >= target) best = j;
        if (best < 0) {
          hi = th[0] - 1;
        } else {
          lo = th[best];
          if (best < NS - 1) hi = th[best + 1] - 1;
        }
      }
      return lo;
    };
    // at the cut key kc (ties there have one weight e_t): how many of them,
    // lowest id first, the kept prefix takes: the first j whose running sum
    // from the mass above reaches the target (strict: passes it)
    auto tie_take = [&](auto&& in, uint32_t kc, float target, bool strict) {
      pass_sums(1, [&](int, int i, float z, float e) {
        return (ordered_key(z) > kc && in(i, z)) ? e : 0.f;
      });
      float acc = sm.res[0];
      pass_count(true, [&](int i, float z) { return ordered_key(z) == kc && in(i, z); });
      const long long n_t = sm.ires[0];
      const float e_t = weight(key_value(kc));
      long long j = 0;
      while (j < n_t) {
        acc = __fadd_rn(acc, e_t);
        ++j;
        if (strict ? acc > target : acc >= target) break;
      }
      return pass_nth(j > 0 ? j : 1, [&](int i, float z) { return ordered_key(z) == kc && in(i, z); });
    };

    // the total
    pass_sums(1, [&](int, int, float, float e) { return e; });
    const float total = sm.res[0];
    // typical-p: the shortest set by (|-log p - H|, candidate order) whose p
    // reaches typical_p
    const bool typical = prm.typical_p > 0.f && prm.typical_p < 1.0f;
    float h = 0.f;
    uint32_t th_eps = 0xFFFFFFFFu;
    unsigned long long c_typ = 0ull;
    auto eps_key = [&](float e) {
      const float pi = __fdiv_rn(e, total);
      return pi > 0.f ? ordered_key(fabsf(__fsub_rn(-logf(pi), h))) : ordered_key(INFINITY);
    };
    if (typical) {
      pass_sums(1, [&](int, int, float, float e) {
        const float pi = __fdiv_rn(e, total);
        return pi > 0.f ? __fmul_rn(pi, logf(pi)) : 0.f;
      });
      h = -sm.res[0];
      const float tp = prm.typical_p;
      // the smallest eps key E with sum of p over the ids with eps key <= E
      // reaching typical_p (every id if rounding keeps the sum below it)
      uint32_t lo = 0, hi = 0xFFFFFFFFu;
      while (lo < hi) {
        const unsigned long long span = static_cast<unsigned long long>(hi) - lo;
        uint32_t th[NS];
#pragma unroll
        for (int j = 0; j < NS; ++j)
          th[j] = lo + static_cast<uint32_t>((span * static_cast<unsigned long long>(j + 1)) / (NS + 1));
        pass_sums(NS, [&](int j, int, float, float e) {
          return eps_key(e) <= th[j] ? __fdiv_rn(e, total) : 0.f;
        });
        int best = NS;
        for (int j = NS - 1; j >= 0; --j)
          if (sm.res[j] >= tp) best = j;
        if (best == NS) {
          lo = th[NS - 1] + 1;
        } else {
          hi = th[best];
          if (best > 0) lo = th[best - 1] + 1;
        }
      }
      th_eps = lo;
      // ties at that eps key, in candidate order: the shortest prefix that
      // reaches typical_p from the mass below
      pass_sums(1, [&](int, int, float, float e) { return eps_key(e) < th_eps ? __fdiv_rn(e, total) : 0.f; });
      const float below = sm.res[0];
      pass_count(true, [&](int, float z) { return eps_key(weight(z)) == th_eps; });
      const long long n_t = sm.ires[0];
      if (n_t > kCap) {
        if (rank == 0 && t == 0) {
          out[b] = -1;
          if (status) atomicExch(status, DEV_SAMPLER_UNSUPPORTED);
        }
        return;
      }
      if (t == 0) sm.n_cand = 0;
      __syncthreads();
      visit([&](bool valid, int i, float z) {
        if (valid && eps_key(weight(z)) == th_eps) {
          const uint32_t slot = atomicAdd(&sm.n_cand, 1u);  // parking slot only
          sm.cand[slot] = composite(ordered_key(z), i);
        }
      });
      cluster_sync();
      if (rank == 0) {
        if (t == 0) {
          uint32_t off = sm.n_cand;
          for (int q = 1; q < C; ++q) {
            sm.offs[q] = off;
            off += ld_dsmem_u32(peer(&sm.n_cand, q));
          }
          sm.offs[C] = off;
          sm.offs[0] = 0;
        }
        __syncthreads();
        for (int q = 1; q < C; ++q) {
          const int n_q = static_cast<int>(sm.offs[q + 1] - sm.offs[q]);
          const uint32_t src = peer(&sm.cand[0], q);
          for (int i = t; i < n_q; i += kThreadsS) sm.cand[sm.offs[q] + i] = ld_dsmem_u64(src + 8u * i);
        }
        __syncthreads();
        const int n = static_cast<int>(sm.offs[C]);
        int n2 = 1;
        while (n2 < n) n2 <<= 1;
        for (int i = n + t; i < n2; i += kThreadsS) sm.cand[i] = 0ull;
        __syncthreads();
        bitonic_desc(sm.cand, n2);
        if (t == 0) {
          float acc = below;
          unsigned long long last = sm.cand[0];
          for (int j = 0; j < n; ++j) {
            last = sm.cand[j];
            acc = __fadd_rn(acc, __fdiv_rn(weight(key_value(static_cast<uint32_t>(last >> 32))), total));
            if (acc >= tp) break;
          }
          sm.xi[1] = static_cast<long long>(last);
        }
      }
      cluster_sync();
      c_typ = ld_dsmem_u64(peer(&sm.xi[1], 0));
      cluster_sync();  // every block has read it
    }
    auto in_typ = [&](int i, float z) {
      if (!typical) return true;
      const uint32_t ek = eps_key(weight(z));
      return ek < th_eps || (ek == th_eps && composite(ordered_key(z), i) >= c_typ);
    };
    // top-p over the typical set, in candidate order
    uint32_t k_tp = 0;
    int tie_tp = V;
    if (prm.top_p < 1.0f) {
      float tot = total;
      if (typical) {
        pass_sums(1, [&](int, int i, float z, float e) { return in_typ(i, z) ? e : 0.f; });
        tot = sm.res[0];
      }
      const float target = __fmul_rn(prm.top_p, tot);
      k_tp = search_max(in_typ, target, false);
      tie_tp = tie_take(in_typ, k_tp, target, false);
    }
    auto in_tp = [&](int i, float z) {
      const uint32_t kz = ordered_key(z);
      return in_typ(i, z) && (kz > k_tp || (kz == k_tp && i <= tie_tp));
    };
    // the first candidate of the typical set (it is always kept), and min-p
    // relative to its weight
    pass_count(true, in_typ);
    const unsigned long long first_c = static_cast<unsigned long long>(sm.ires[1]);
    const int first_id = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(first_c & 0xFFFFFFFFull));
    const float thr = prm.min_p > 0.0f ? __fmul_rn(prm.min_p, weight(key_value(static_cast<uint32_t>(first_c >> 32))))
                                       : -INFINITY;
    auto in_kept = [&](int i, float z) { return i == first_id || (in_tp(i, z) && weight(z) >= thr); };
    pass_sums(1, [&](int, int i, float z, float e) { return in_kept(i, z) ? e : 0.f; });
    const float kept = sm.res[0];
    // the draw: the first kept candidate whose running sum passes u * kept
    const uint64_t stp = static_cast<uint64_t>(step[b]);
    const Philox4 w = philox4x32_10(
        Philox4{static_cast<uint32_t>(stp), static_cast<uint32_t>(stp >> 32), 0u, 0u},
        static_cast<uint32_t>(prm.seed), static_cast<uint32_t>(prm.seed >> 32));
    const float u = static_cast<float>(w.x >> 8) * (1.0f / 16777216.0f);
    const float target = __fmul_rn(u, kept);
    int pick;
    if (kept > target) {
      const uint32_t k_d = search_max(in_kept, target, true);
      pick = tie_take(in_kept, k_d, target, true);
    } else {
      pass_count(false, in_kept);  // (u < 1 never gets here) the last kept candidate
      pick = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(static_cast<unsigned long long>(sm.ires[1]) & 0xFFFFFFFFull));
    }
    if (rank == 0 && t == 0) out[b] = pick;
  };

  if (!(temp > 0.f)) {
    // greedy: maximum of the strict total order
    unsigned long long best = 0ull;
    visit([&](bool valid, int i, float z) {
      const unsigned long long c = valid ? composite(ordered_key(z), i) : 0ull;
      best = c > best ? c : best;
    });
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long x = __shfl_xor_sync(0xffffffffu, best, o);
      best = x > best ? x : best;
    }
    if (lane == 0) sm.wbest[warp] = best;
    __syncthreads();
    if (t == 0) {
      unsigned long long m = sm.wbest[0];
      for (int w = 1; w < kWarps; ++w) m = sm.wbest[w] > m ? sm.wbest[w] : m;
      sm.x_best = m;
    }
    cluster_sync();
    if (rank == 0 && t == 0) {
      unsigned long long m = 0ull;
      for (int q = 0; q < C; ++q) {
        const unsigned long long x = ld_dsmem_u64(peer(&sm.x_best, q));
        m = x > m ? x : m;
      }
      out[b] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(m & 0xFFFFFFFFull));
    }
    cluster_sync();  // the peers stay until rank 0 has read them
    return;
  }
  // Whole vocabulary (no top-k) over more than kMaxTopK ids: the searches
  // below; otherwise the top k are gathered and sorted.
  const bool full = (prm.top_k <= 0 || prm.top_k >= V) && V > kMaxTopK;
  const int k = full ? kMaxTopK : ((prm.top_k <= 0 || prm.top_k >= V) ? V : prm.top_k);
  if (k > kMaxTopK || (full && (V + 127) / 128 > kMaxBlocks)) {
    if (rank == 0 && t == 0) {
      out[b] = -1;
      if (status) atomicExch(status, DEV_SAMPLER_UNSUPPORTED);
    }
    return;
  }
  if (full) {
    whole_vocabulary();
    return;
  }

  // 2a. Fast path: the row maximum M, then how many ids have a value of at
  // least M - delta for eight deltas (integer counts, exact maximum: nothing
  // depends on the order of the sums).  The smallest delta that holds at
  // least k ids, if it holds at most kCap, gives the gathering threshold; the
  // set gathered is every id at or above it, which contains the top k.
  constexpr float kDeltas[8] = {0.5f, 1.f, 2.f, 4.f, 8.f, 16.f, 32.f, 64.f};
  {
    float mx = -INFINITY;
    visit([&](bool valid, int, float z) {
      if (valid) mx = fmaxf(mx, z);
    });
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) sm.wmax[warp] = mx;
    __syncthreads();
    if (t == 0) {
      float m = sm.wmax[0];
      for (int w = 1; w < kWarps; ++w) m = fmaxf(m, sm.wmax[w]);
      sm.x_max = m;
    }
    cluster_sync();
    if (warp == 0) {
      float m = lane < C ? ld_dsmem_f32(peer(&sm.x_max, lane)) : -INFINITY;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == 0) sm.m_all = m;
    }
    __syncthreads();
    const float m = sm.m_all;
    float th[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) th[j] = __fsub_rn(m, kDeltas[j]);
    int c[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    visit([&](bool valid, int, float z) {
#pragma unroll
      for (int j = 0; j < 8; ++j) c[j] += (valid && z >= th[j]) ? 1 : 0;
    });
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) c[j] += __shfl_xor_sync(0xffffffffu, c[j], o);
      if (lane == 0) sm.wcnt[warp][j] = c[j];
    }
    __syncthreads();
    if (t < 8) {
      int tot = 0;
      for (int w = 0; w < kWarps; ++w) tot += sm.wcnt[w][t];
      sm.x_cnt[t] = tot;
    }
    cluster_sync();
    if (t < 8) {
      int tot = 0;
      for (int q = 0; q < C; ++q) tot += static_cast<int>(ld_dsmem_u32(peer(&sm.x_cnt[t], q)));
      sm.cnt[t] = tot;
    }
    __syncthreads();
    if (t == 0) {
      sm.fast = 0;
      for (int j = 0; j < 8; ++j) {
        if (sm.cnt[j] >= k) {
          if (sm.cnt[j] <= kCap && m > -INFINITY) {
            sm.fast = 1;
            sm.thresh_f = th[j];
          }
          break;
        }
      }
    }
    __syncthreads();
  }
  const bool fast = sm.fast != 0;

  // 2b. Otherwise, radix narrowing of the threshold over the cluster's
  // summed histograms (every block takes the same decision)
  uint32_t prefix = 0;  // fixed high bits of the threshold
  int fixed = 0;        // how many high bits are fixed
  int k_rem = k;        // how many ids are still needed at or below the prefix
  int above = 0;        // ids strictly above the prefix region (all taken)
  bool exact_ties = false;
  const int widths[3] = {11, 11, 10};
  for (int pass = 0; pass < 3 && !fast; ++pass) {
    const int w = widths[pass];
    const int shift = 32 - fixed - w;
    const int nb = 1 << w;
    for (int i = t; i < nb; i += kThreadsS) sm.hist[i] = 0u;
    __syncthreads();
    visit_key([&](bool valid, int, uint32_t key) {
      const bool in = valid && (fixed == 0 || (key >> (32 - fixed)) == prefix);
      const uint32_t digit = in ? (key >> shift) & (nb - 1) : 0xFFFFFFFFu;
      const unsigned peers = __match_any_sync(0xffffffffu, digit);
      if (in && lane == __ffs(peers) - 1) atomicAdd(&sm.hist[digit], __popc(peers));
    });
    cluster_sync();  // every block's histogram is complete
    for (int i = t; i < nb; i += kThreadsS) {
      uint32_t tot = 0;
      for (int q = 0; q < C; ++q) tot += ld_dsmem_u32(peer(&sm.hist[i], q));
      sm.comb[i] = tot;
    }
    cluster_sync();  // every block has read the histograms (the next pass reuses them)
    if (warp == 0) {
      // lane l sums bins [nb - (l + 1) * nb / 32, nb - l * nb / 32) (lane 0 the
      // top block); an exclusive scan from the top finds the block holding
      // the k_rem-th id, whose lane then walks its bins downwards
      const int per = nb / 32;
      const int hi = nb - lane * per;
      int bsum = 0;
      for (int d = hi - 1; d >= hi - per; --d) bsum += static_cast<int>(sm.comb[d]);
      int incl = bsum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const int excl = incl - bsum;
      const unsigned hit = __ballot_sync(0xffffffffu, incl >= k_rem);
      const int owner = hit ? __ffs(hit) - 1 : 31;
      if (lane == owner) {
        int cum = excl, d = hi - 1;
        for (; d > hi - per; --d) {
          if (cum + static_cast<int>(sm.comb[d]) >= k_rem) break;
          cum += sm.comb[d];
        }
        // ids with digit > d are all in; ids with digit == d hold the k_rem-th
        const int at_or_above = above + cum + static_cast<int>(sm.comb[d]);
        sm.thresh = ((prefix << w) | static_cast<uint32_t>(d)) << shift;
        sm.k_rem = k_rem - cum;
        sm.ok = at_or_above <= kCap ? 1 : 0;
        sm.warp_cnt[0] = static_cast<uint32_t>(above + cum);
      }
    }
    __syncthreads();
    const uint32_t th = sm.thresh;
    prefix = th >> shift;
    fixed += w;
    if (sm.ok) break;
    above = static_cast<int>(sm.warp_cnt[0]);
    k_rem = sm.k_rem;
    __syncthreads();
    if (pass == 2) exact_ties = true;
  }
  const uint32_t thresh = sm.thresh;
  if (t == 0) {
    sm.n_cand = 0;
    sm.eq_taken = 0;
  }
  __syncthreads();
  if (fast) {
    const float tf = sm.thresh_f;
    visit([&](bool valid, int i, float z) {
      if (valid && z >= tf) {
        const uint32_t slot = atomicAdd(&sm.n_cand, 1u);  // parking slot only
        sm.cand[slot] = composite(ordered_key(z), i);
      }
    });
  } else if (!exact_ties) {
    visit_key([&](bool valid, int i, uint32_t key) {
      if (valid && key >= thresh) {
        const uint32_t slot = atomicAdd(&sm.n_cand, 1u);  // parking slot only
        sm.cand[slot] = composite(key, i);
      }
    });
  } else if (rank == 0) {
    // More than kCap ids tie exactly at the threshold (rare): rank 0 takes
    // every id above it plus the lowest-id ties, scanning the whole row in id
    // order.
    const int need_eq = k_rem;
    for (int base = 0; base < V; base += kThreadsS) {
      const int i = base + t;
      uint32_t key = 0;
      if (i < V) key = ordered_key(penalised(row, i, pe));
      const bool gt = i < V && key > thresh;
      const bool eq = i < V && key == thresh;
      if (gt) {
        const uint32_t slot = atomicAdd(&sm.n_cand, 1u);
        sm.cand[slot] = composite(key, i);
      }
      const unsigned ballot = __ballot_sync(0xffffffffu, eq);
      if (!__syncthreads_or(ballot != 0u)) continue;
      if (lane == 0) sm.warp_cnt[warp] = __popc(ballot);
      __syncthreads();
      uint32_t before = sm.eq_taken;
      for (int w2 = 0; w2 < warp; ++w2) before += sm.warp_cnt[w2];
      before += __popc(ballot & ((1u << lane) - 1u));
      if (eq && static_cast<int>(before) < need_eq) {
        const uint32_t slot = atomicAdd(&sm.n_cand, 1u);
        sm.cand[slot] = composite(key, i);
      }
      __syncthreads();
      if (t == 0) {
        uint32_t tot = 0;
        for (int w2 = 0; w2 < kWarps; ++w2) tot += sm.warp_cnt[w2];
        sm.eq_taken += tot;
      }
      __syncthreads();
    }
  }
  cluster_sync();  // every block's candidates are parked
  if (rank == 0) {
    // rank 0 appends the peers' candidates after its own
    if (t == 0) {
      uint32_t off = sm.n_cand;
      sm.offs[0] = 0;
      for (int q = 1; q < C; ++q) {
        sm.offs[q] = off;
        off += ld_dsmem_u32(peer(&sm.n_cand, q));
      }
      sm.offs[C] = off;
    }
    __syncthreads();
    for (int q = 1; q < C; ++q) {
      const int n_q = static_cast<int>(sm.offs[q + 1] - sm.offs[q]);
      const uint32_t src = peer(&sm.cand[0], q);
      for (int i = t; i < n_q; i += kThreadsS) sm.cand[sm.offs[q] + i] = ld_dsmem_u64(src + 8u * i);
    }
  }
  cluster_sync();  // the peers stay until rank 0 has read them
  if (rank != 0) return;
  const int n_cand = static_cast<int>(sm.offs[C]);
  const int kk = min(k, n_cand);
  // The first kk candidates in the strict total order (composites are
  // distinct).  Up to 1024 candidates: each one's position is the number of
  // candidates above it; more: a bitonic sort.
  unsigned long long* top = reinterpret_cast<unsigned long long*>(sm.hist);  // room for kMaxTopK
  if (n_cand <= kMaxTopK) {
    for (int i = t; i < n_cand; i += kThreadsS) {
      const unsigned long long x = sm.cand[i];
      int pos = 0;
      for (int j = 0; j < n_cand; ++j) pos += sm.cand[j] > x ? 1 : 0;
      if (pos < kk) top[pos] = x;
    }
  } else {
    int n2 = 1;
    while (n2 < n_cand) n2 <<= 1;
    for (int i = n_cand + t; i < n2; i += kThreadsS) sm.cand[i] = 0ull;
    __syncthreads();
    bitonic_desc(sm.cand, n2);
    for (int i = t; i < kk; i += kThreadsS) top[i] = sm.cand[i];
  }
  __syncthreads();

  // 3. exponentials in candidate order, then warp 0 forms the prefix sums
  // P[i] = e_0 + ... + e_i (32 at a time: a warp scan with a fixed shuffle
  // pattern plus the total of the chunks before) and applies top-p, min-p
  // and the draw on them.
  const float s0 = __fdiv_rn(key_value(static_cast<uint32_t>(top[0] >> 32)), temp);
  for (int i = t; i < kk; i += kThreadsS) {
    const float si = __fdiv_rn(key_value(static_cast<uint32_t>(top[i] >> 32)), temp);
    sm.e[i] = expf(__fsub_rn(si, s0));
  }
  __syncthreads();
  float* P = reinterpret_cast<float*>(sm.comb);  // room for kMaxTopK
  // P[i] = v(0) + ... + v(i) over the candidates, by warp 0
  auto prefix_sums = [&](auto&& v_of) {
    float carry = 0.f;
    for (int c0 = 0; c0 < kk; c0 += 32) {
      const int i = c0 + lane;
      float v = i < kk ? v_of(i) : 0.f;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v = __fadd_rn(v, y);
      }
      v = __fadd_rn(v, carry);
      if (i < kk) P[i] = v;
      carry = __shfl_sync(0xffffffffu, v, 31);
    }
    __syncwarp();
  };
  if (warp == 0) prefix_sums([&](int i) { return sm.e[i]; });
  // Typical-p (0 < typical_p < 1): p_i = e_i / P[kk-1], H = -sum p_i log p_i
  // (lane l adds terms l, l + 32, ... in order, then a fixed butterfly); the
  // candidates sorted by (|-log p_i - H|, i) ascending; the shortest such
  // prefix whose p (a fixed-order warp scan) reaches typical_p is kept.
  const bool typical = prm.typical_p > 0.f && prm.typical_p < 1.0f;
  uint32_t* kmask = reinterpret_cast<uint32_t*>(sm.cand + 3072);  // kept candidates (typical-p)
  if (typical) {
    __syncthreads();  // P
    const float total = P[kk - 1];
    float* lp = reinterpret_cast<float*>(sm.cand + 2048);
    for (int i = t; i < kk; i += kThreadsS) {
      const float pi = __fdiv_rn(sm.e[i], total);
      lp[i] = pi > 0.f ? logf(pi) : 0.f;
    }
    for (int i = t; i < 32; i += kThreadsS) kmask[i] = 0u;
    __syncthreads();
    if (warp == 0) {
      float acc = 0.f;
      for (int i = lane; i < kk; i += 32) acc = __fadd_rn(acc, __fmul_rn(__fdiv_rn(sm.e[i], total), lp[i]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, o));
      if (lane == 0) sm.typ_h = acc;
    }
    __syncthreads();
    const float h = -sm.typ_h;
    int n2 = 1;
    while (n2 < kk) n2 <<= 1;
    for (int i = t; i < n2; i += kThreadsS) {
      unsigned long long key = 0ull;  // padding sorts last
      if (i < kk) {
        const float pi = __fdiv_rn(sm.e[i], total);
        const float eps = pi > 0.f ? fabsf(__fsub_rn(-lp[i], h)) : INFINITY;
        key = composite(~ordered_key(eps), i);  // descending order = (eps, i) ascending
      }
      sm.cand[i] = key;
    }
    __syncthreads();
    bitonic_desc(sm.cand, n2);
    if (warp == 0) {
      auto idx_at = [&](int i) { return static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(sm.cand[i] & 0xFFFFFFFFull)); };
      int m = kk;
      float carry = 0.f;
      for (int c0 = 0; c0 < kk; c0 += 32) {
        const int i = c0 + lane;
        float v = i < kk ? __fdiv_rn(sm.e[idx_at(i)], total) : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, v, o);
          if (lane >= o) v = __fadd_rn(v, y);
        }
        v = __fadd_rn(v, carry);
        const unsigned hit = __ballot_sync(0xffffffffu, i < kk && v >= prm.typical_p);
        if (hit) {
          m = c0 + __ffs(hit);
          break;
        }
        carry = __shfl_sync(0xffffffffu, v, 31);
      }
      for (int i = lane; i < m; i += 32) {
        const int j = idx_at(i);
        atomicOr(&kmask[j >> 5], 1u << (j & 31));
      }
      __syncwarp();
      prefix_sums([&](int i) { return (kmask[i >> 5] >> (i & 31)) & 1u ? sm.e[i] : 0.f; });
    }
  }
  if (warp != 0) return;
  auto kept_at = [&](int j) { return !typical || ((kmask[j >> 5] >> (j & 31)) & 1u); };
  // first i < n with pred(i), else n (warp-uniform)
  auto first = [&](int n, auto&& pred) {
    for (int c0 = 0; c0 < n; c0 += 32) {
      const int i = c0 + lane;
      const unsigned hit = __ballot_sync(0xffffffffu, i < n && pred(i));
      if (hit) return c0 + __ffs(hit) - 1;
    }
    return n;
  };
  const float total = P[kk - 1];
  int keep = kk;
  if (prm.top_p < 1.0f) {
    const float target = __fmul_rn(prm.top_p, total);
    const int i = first(kk, [&](int j) { return P[j] >= target; });
    keep = i < kk ? i + 1 : kk;
  }
  const int j0 = first(kk, kept_at);  // the first kept candidate (the largest kept e)
  if (prm.min_p > 0.0f) {
    const float thr = __fmul_rn(prm.min_p, sm.e[j0]);
    const int n = first(keep, [&](int j) { return kept_at(j) && !(sm.e[j] >= thr); });
    keep = n > j0 ? n : j0 + 1;
  }
  const float kept = P[keep - 1];
  const uint64_t st = static_cast<uint64_t>(step[b]);
  const Philox4 w = philox4x32_10(
      Philox4{static_cast<uint32_t>(st), static_cast<uint32_t>(st >> 32), 0u, 0u},
      static_cast<uint32_t>(prm.seed), static_cast<uint32_t>(prm.seed >> 32));
  const float u = static_cast<float>(w.x >> 8) * (1.0f / 16777216.0f);
  const float target = __fmul_rn(u, kept);
  int pick = first(keep, [&](int j) { return P[j] > target; });
  if (pick >= keep) {  // (u < 1 never gets here) the last kept candidate
    pick = keep - 1;
    while (pick > 0 && !kept_at(pick)) --pick;
  }
  if (lane == 0)
    out[b] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(top[pick] & 0xFFFFFFFFull));
}

}  // namespace
}  // namespace kinv

using namespace kinv;

extern "C" size_t kinv_sample_workspace(int B, int V) {
  (void)B;
  (void)V;
  return 0;
}

// Smem, the bitmap of marked ids ((V + 31) / 32 words) and the rank of each
// word's first marked id (uint16 per word)
static size_t sampler_smem_bytes(int V) {
  const size_t words = (static_cast<size_t>(V) + 31) / 32;
  return sizeof(Smem) + words * 4 + (words * 2 + 15) / 16 * 16;
}

extern "C" kinv_status kinv_sample(const float* logits, int64_t ld, int B, int V,
                                   const kinv_sampling_params* params, const int32_t* history,
                                   int hist_ld, const int32_t* hist_len, const int64_t* step,
                                   int32_t* out_tokens, void* workspace, size_t ws_bytes,
                                   kinv_stream stream) {
  (void)workspace;
  (void)ws_bytes;
  if (B < 0 || V <= 0 || ld < V || hist_ld < 0) return KINV_ERR_INVALID_ARG;
  if (B == 0) return KINV_OK;
  if (!logits || !params || !step || !out_tokens) return KINV_ERR_INVALID_ARG;
  if (hist_len && (!history || hist_ld <= 0)) return KINV_ERR_INVALID_ARG;
  if (hist_ld > kMaxHist) return KINV_ERR_UNSUPPORTED;
  const size_t smem = sampler_smem_bytes(V);
  if (smem > static_cast<size_t>(max_smem_optin())) return KINV_ERR_UNSUPPORTED;
  if (B > 65535) return KINV_ERR_UNSUPPORTED;
  // Blocks per row: up to eight while the grid stays within one block per
  // SM.  The token does not depend on this choice (every exchanged quantity
  // is exact and the candidate set is the same), only the speed does.
  int C = kMaxCluster;
  while (C > 1 && static_cast<long long>(B) * C > sm_count()) C >>= 1;
  const int chunk = ((V + C - 1) / C + 127) / 128 * 128;
  const bool regs = chunk <= kRegSpan;
  const kinv_status attr = ensure_smem(reinterpret_cast<const void*>(regs ? sample_kernel<true> : sample_kernel<false>),
                                       static_cast<size_t>(max_smem_optin()));
  if (attr != KINV_OK) return attr;
  if (regs)
    return launch_kernel(sample_kernel<true>, dim3(C, B), dim3(kThreadsS), smem, stream,
                         static_cast<unsigned>(C), logits, ld, V, params, history, hist_ld, hist_len,
                         step, out_tokens, device_status_word());
  return launch_kernel(sample_kernel<false>, dim3(C, B), dim3(kThreadsS), smem, stream,
                       static_cast<unsigned>(C), logits, ld, V, params, history, hist_ld, hist_len, step,
                       out_tokens, device_status_word());
}
