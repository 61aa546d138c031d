// Seeded, batch-invariant sampler (Kinetic "Receipts", *Making a receipt*:
// the receipt records temperature, top_k, top_p, min_p, repeat_penalty,
// repeat_last_n and the seed, so the same settings must give the same token).
//
// One thread block per row; nothing is shared between rows.
//  1. Repeat penalty: a shared-memory bitmap marks the distinct ids among the
//     row's last repeat_last_n history tokens; a marked logit z becomes z / r
//     (z > 0) or z * r, both correctly rounded fp32 operations.
//  2. Ranking uses the order-preserving 32-bit key of each penalised fp32
//     value and, for equal keys, the lower id first: a strict total order.
//     Greedy (temperature <= 0) takes its maximum.  Otherwise radix passes over
//     the key (11, 11, 10 bits) narrow a threshold until at most kCap ids lie
//     at or above it; those are gathered (slots come from an atomic counter,
//     which only decides where a candidate is parked) and bitonic-sorted by the
//     total order, so the candidate list does not depend on the parking order.
//     If more than kCap ids tie exactly at the threshold, the ties are taken
//     lowest id first by an ordered block-wide scan.
//  3. s_i = z_i / T; e_i = exp(s_i - s_0); one thread forms the running sums in
//     candidate order and applies top-p, min-p and the draw.
//  4. The draw: u = (Philox4x32-10(counter = (step lo, step hi, 0, 0),
//     key = (seed lo, seed hi)).word0 >> 8) * 2^-24 (Salmon et al., SC'11,
//     restated here from the published round function and constants).
#include <math.h>

#include "common.cuh"

namespace kinv {
namespace {

constexpr int kThreadsS = 1024;
constexpr int kMaxTopK = 1024;
constexpr int kCap = 4096;  // candidates gathered before sorting

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
  uint32_t hist[2048];
  unsigned long long cand[kCap];
  float e[kMaxTopK];
  uint32_t warp_cnt[32];
  uint32_t n_cand;
  uint32_t eq_taken;
  uint32_t thresh;      // gather ids whose key >= thresh
  int k_rem;
  int ok;
  int result;
  float wmax[32];
  int wcnt[32][8];
  int cnt[8];
  float thresh_f;       // fast path: gather ids whose value >= thresh_f
  int fast;
};

__device__ __forceinline__ float penalised(const float* __restrict__ row, int i,
                                           const uint32_t* bitmap, float r) {
  float z = row[i];
  if ((bitmap[i >> 5] >> (i & 31)) & 1u) z = z > 0.f ? __fdiv_rn(z, r) : __fmul_rn(z, r);
  return z;
}

// Visits every id of the row once, in rounds in which each thread loads
// four 16-byte vectors (16 logits) before using any of them, so a pass keeps
// many loads in flight.  f(valid, id, key) sees the key of the penalised
// logit; every lane runs the same number of rounds (f may use warp votes).
template <typename F>
__device__ __forceinline__ void for_each_value(const float* __restrict__ row, int V,
                                               const uint32_t* bitmap, float r, F&& f) {
  constexpr int U = 4;
  const int t = threadIdx.x;
  const bool vec = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
  const int V4 = vec ? (V >> 2) : 0;
  const float4* row4 = reinterpret_cast<const float4*>(row);
  for (int base = 0; base < V4; base += kThreadsS * U) {
    float4 x[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i4 = base + u * kThreadsS + t;
      x[u] = i4 < V4 ? row4[i4] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i4 = base + u * kThreadsS + t;
      const bool valid = i4 < V4;
      const float xv[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = 4 * i4 + e;
        float z = xv[e];
        if (valid && ((bitmap[i >> 5] >> (i & 31)) & 1u)) z = z > 0.f ? __fdiv_rn(z, r) : __fmul_rn(z, r);
        f(valid, i, isnan(z) ? -INFINITY : z);
      }
    }
  }
  // the ids not covered by whole vectors, one per thread and round
  for (int base = 4 * V4; base < V; base += kThreadsS) {
    const int i = base + t;
    const bool valid = i < V;
    const float z = valid ? penalised(row, i, bitmap, r) : 0.f;
    f(valid, i, isnan(z) ? -INFINITY : z);
  }
}

template <typename F>
__device__ __forceinline__ void for_each_key(const float* __restrict__ row, int V,
                                             const uint32_t* bitmap, float r, F&& f) {
  for_each_value(row, V, bitmap, r,
                 [&](bool valid, int i, float z) { f(valid, i, valid ? ordered_key(z) : 0u); });
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

__global__ void __launch_bounds__(kThreadsS) sample_kernel(
    const float* __restrict__ logits, int64_t ld, int V, const kinv_sampling_params* __restrict__ params,
    const int32_t* __restrict__ history, int hist_ld, const int32_t* __restrict__ hist_len,
    const int64_t* __restrict__ step, int32_t* __restrict__ out, int* status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(smem_raw + sizeof(Smem));
  pdl_launch_dependents();
  pdl_wait();
  const int b = blockIdx.x;
  const int t = threadIdx.x;
  const int lane = t & 31, warp = t >> 5;
  const float* row = logits + b * ld;
  const kinv_sampling_params prm = params[b];
  const int words = (V + 31) >> 5;

  // 1. penalty bitmap
  for (int i = t; i < words; i += kThreadsS) bitmap[i] = 0u;
  __syncthreads();
  const float r = prm.repeat_penalty;
  const int hl = hist_len ? min(max(hist_len[b], 0), hist_ld) : 0;
  int n_pen = prm.repeat_last_n < 0 ? hl : min(prm.repeat_last_n, hl);
  if (r == 1.0f) n_pen = 0;
  for (int i = t; i < n_pen; i += kThreadsS) {
    const int id = history[static_cast<int64_t>(b) * hist_ld + hl - n_pen + i];
    if (id >= 0 && id < V) atomicOr(&bitmap[id >> 5], 1u << (id & 31));  // idempotent bit set
  }
  __syncthreads();

  const float temp = prm.temperature;
  if (!(temp > 0.f)) {
    // greedy: maximum of the strict total order
    unsigned long long best = 0ull;
    for (int i = t; i < V; i += kThreadsS) {
      const unsigned long long c = composite(ordered_key(penalised(row, i, bitmap, r)), i);
      best = c > best ? c : best;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long x = __shfl_xor_sync(0xffffffffu, best, o);
      best = x > best ? x : best;
    }
    if (lane == 0) sm.cand[warp] = best;
    __syncthreads();
    if (t == 0) {
      unsigned long long m = sm.cand[0];
      for (int w = 1; w < kThreadsS / 32; ++w) m = sm.cand[w] > m ? sm.cand[w] : m;
      out[b] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(m & 0xFFFFFFFFull));
    }
    return;
  }
  const int k = (prm.top_k <= 0 || prm.top_k >= V) ? V : prm.top_k;
  if (k > kMaxTopK) {
    if (t == 0) {
      out[b] = -1;
      if (status) atomicExch(status, DEV_SAMPLER_UNSUPPORTED);
    }
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
    for_each_value(row, V, bitmap, r, [&](bool valid, int, float z) {
      if (valid) mx = fmaxf(mx, z);
    });
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) sm.wmax[warp] = mx;
    __syncthreads();
    float m = sm.wmax[0];
    for (int w = 1; w < kThreadsS / 32; ++w) m = fmaxf(m, sm.wmax[w]);
    float th[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) th[j] = __fsub_rn(m, kDeltas[j]);
    int c[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for_each_value(row, V, bitmap, r, [&](bool valid, int, float z) {
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
      for (int w = 0; w < kThreadsS / 32; ++w) tot += sm.wcnt[w][t];
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
      sm.n_cand = 0;
    }
    __syncthreads();
  }
  const bool fast = sm.fast != 0;

  // 2b. Otherwise, radix narrowing of the threshold
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
    for_each_key(row, V, bitmap, r, [&](bool valid, int, uint32_t key) {
      const bool in = valid && (fixed == 0 || (key >> (32 - fixed)) == prefix);
      const uint32_t digit = in ? (key >> shift) & (nb - 1) : 0xFFFFFFFFu;
      const unsigned peers = __match_any_sync(0xffffffffu, digit);
      if (in && lane == __ffs(peers) - 1) atomicAdd(&sm.hist[digit], __popc(peers));
    });
    __syncthreads();
    if (warp == 0) {
      // lane l sums bins [nb - (l + 1) * nb / 32, nb - l * nb / 32) (lane 0 the
      // top block); an exclusive scan from the top finds the block holding
      // the k_rem-th id, whose lane then walks its bins downwards
      const int per = nb / 32;
      const int hi = nb - lane * per;
      int bsum = 0;
      for (int d = hi - 1; d >= hi - per; --d) bsum += static_cast<int>(sm.hist[d]);
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
          if (cum + static_cast<int>(sm.hist[d]) >= k_rem) break;
          cum += sm.hist[d];
        }
        // ids with digit > d are all in; ids with digit == d hold the k_rem-th
        const int at_or_above = above + cum + static_cast<int>(sm.hist[d]);
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
    for_each_value(row, V, bitmap, r, [&](bool valid, int i, float z) {
      if (valid && z >= tf) {
        const uint32_t slot = atomicAdd(&sm.n_cand, 1u);  // parking slot only
        sm.cand[slot] = composite(ordered_key(z), i);
      }
    });
  } else if (!exact_ties) {
    for_each_key(row, V, bitmap, r, [&](bool valid, int i, uint32_t key) {
      if (valid && key >= thresh) {
        const uint32_t slot = atomicAdd(&sm.n_cand, 1u);  // parking slot only
        sm.cand[slot] = composite(key, i);
      }
    });
  } else {
    // every id above the threshold, plus the lowest-id ties, in id order
    const int need_eq = k_rem;
    for (int base = 0; base < V; base += kThreadsS) {
      const int i = base + t;
      uint32_t key = 0;
      if (i < V) key = ordered_key(penalised(row, i, bitmap, r));
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
        for (int w2 = 0; w2 < kThreadsS / 32; ++w2) tot += sm.warp_cnt[w2];
        sm.eq_taken += tot;
      }
      __syncthreads();
    }
  }
  __syncthreads();
  const int n_cand = static_cast<int>(sm.n_cand);
  int n2 = 1;
  while (n2 < n_cand) n2 <<= 1;
  for (int i = n_cand + t; i < n2; i += kThreadsS) sm.cand[i] = 0ull;
  __syncthreads();
  bitonic_desc(sm.cand, n2);
  const int kk = min(k, n_cand);

  // 3. exponentials in candidate order
  const float s0 = __fdiv_rn(key_value(static_cast<uint32_t>(sm.cand[0] >> 32)), temp);
  for (int i = t; i < kk; i += kThreadsS) {
    const float si = __fdiv_rn(key_value(static_cast<uint32_t>(sm.cand[i] >> 32)), temp);
    sm.e[i] = expf(__fsub_rn(si, s0));
  }
  __syncthreads();
  if (t == 0) {
    float total = 0.f;
    for (int i = 0; i < kk; ++i) total = __fadd_rn(total, sm.e[i]);
    int keep = kk;
    if (prm.top_p < 1.0f) {
      const float target = __fmul_rn(prm.top_p, total);
      float cum = 0.f;
      keep = kk;
      for (int i = 0; i < kk; ++i) {
        cum = __fadd_rn(cum, sm.e[i]);
        if (cum >= target) {
          keep = i + 1;
          break;
        }
      }
    }
    if (prm.min_p > 0.0f) {
      int n = 0;
      while (n < keep && sm.e[n] >= prm.min_p) ++n;
      keep = n > 0 ? n : 1;
    }
    float kept = 0.f;
    for (int i = 0; i < keep; ++i) kept = __fadd_rn(kept, sm.e[i]);
    const uint64_t st = static_cast<uint64_t>(step[b]);
    const Philox4 w = philox4x32_10(
        Philox4{static_cast<uint32_t>(st), static_cast<uint32_t>(st >> 32), 0u, 0u},
        static_cast<uint32_t>(prm.seed), static_cast<uint32_t>(prm.seed >> 32));
    const float u = static_cast<float>(w.x >> 8) * (1.0f / 16777216.0f);
    const float target = __fmul_rn(u, kept);
    int pick = keep - 1;
    float cum = 0.f;
    for (int i = 0; i < keep; ++i) {
      cum = __fadd_rn(cum, sm.e[i]);
      if (cum > target) {
        pick = i;
        break;
      }
    }
    out[b] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(sm.cand[pick] & 0xFFFFFFFFull));
  }
}

}  // namespace
}  // namespace kinv

using namespace kinv;

extern "C" size_t kinv_sample_workspace(int B, int V) {
  (void)B;
  (void)V;
  return 0;
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
  const size_t smem = sizeof(Smem) + static_cast<size_t>((V + 31) / 32) * 4;
  if (smem > static_cast<size_t>(max_smem_optin())) return KINV_ERR_UNSUPPORTED;
  static bool configured[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KINV_ERR_CUDA;
  if (dev < 64 && !configured[dev]) {
    if (cudaFuncSetAttribute(sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             max_smem_optin()) != cudaSuccess)
      return KINV_ERR_CUDA;
    configured[dev] = true;
  }
  return launch_kernel(sample_kernel, dim3(B), dim3(kThreadsS), smem, stream, 1, logits, ld, V, params,
                       history, hist_ld, hist_len, step, out_tokens, device_status_word());
}
