// Batch-invariant split-KV attention for decode and prefill
// ("Deterministic and bit-exact inference", *technical*: attention made
// batch-invariant "with a fixed split size for the key-value dimension rather
// than a fixed number of splits").
//
// A query row with L visible keys cuts them into splits of 256 keys at
// absolute offsets 0, 256, 512, ...; the cut depends only on L.  Split kernel:
// one thread block per (split, kv head, group of query rows of one sequence);
// K and then V stream through a ring of four 64-key stages (cp.async), so
// loads stay in flight while the scores are formed.  For every query row r and
// query head i of the kv head's group (a "pair"):
//   s_t  = (q . k_t) * scale   four partial dot products over interleaved
//                              16-byte chunks of d (fp32 FMAs, chunks
//                              ascending), added by a fixed two-step butterfly
//   m    = max_t s_t           (max is exact in any order)
//   e_t  = exp(s_t - m)
//   l    = sum_t e_t           lane l sums keys l, l+32, ..., l+224 in order,
//                              then a fixed butterfly over the 32 lanes
//   o[d] = sum_t e_t v_t[d]    four key groups (t mod 4) each summed with FMAs
//                              over t ascending, then a fixed butterfly
// and (m, l, o) is stored as the split's fp32 partial.  A key a row cannot see
// (beyond its count) gets e_t = 0 in l and is skipped in o, so a row's
// arithmetic is the same whichever rows share the block.
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
constexpr int kThreads = 256;    // four per key of a 64-key stage
constexpr int kMaxRG = 32;       // rows x query heads handled by one block
constexpr int kMaxG = 8;         // query heads per kv head

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
};

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

template <int D>
__global__ void __launch_bounds__(kThreads) attn_split_kernel(const AttnParams p) {
  constexpr int C8 = D / 8;               // 16-byte chunks per key row
  constexpr int SUB = 64;                 // keys per pipeline stage
  constexpr int NSUB = kSplit / SUB;      // 4 stages: the ring holds the whole split
  // Ring of NSUB stages, each [SUB][D] bf16.  Chunk c of key row k sits at
  // chunk c ^ swz(k), swz(k) = 4 (k & 1) | (k & 2): the score phase (two keys
  // x four chunk lanes per 8-thread phase) and the o phase (four keys x eight
  // column pairs per warp) both hit distinct bank groups.
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __nv_bfloat16* ring = reinterpret_cast<__nv_bfloat16*>(smem_raw);
  float* qs = reinterpret_cast<float*>(smem_raw + kSplit * D * 2);        // [rg_cap][D]
  float* es = qs + p.rg_cap * D;                                          // [rg_cap/4][256][4]
  __shared__ float mrow[kMaxRG];
  __shared__ float lrow[kMaxRG];

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
  const int RG = rs.nrows * G;                         // (row, head) pairs of this block
  const int RB = (RG + 3) >> 2;                        // handled in blocks of four
  const int t = threadIdx.x;
  const int lane = t & 31, warp = t >> 5;
  const int64_t seq_off = rs.seq * p.seq_stride + static_cast<int64_t>(k0) * p.tok_stride + g * D;
  auto swz = [](int key) { return ((key & 1) << 2) | (key & 2); };
  // keys visible to (row, head) pair r (rows of one block see consecutive lengths)
  auto count = [&](int r) { return r < RG ? min(kSplit, rs.len0 + r / G - k0) : 0; };

  auto load_sub = [&](const __nv_bfloat16* src, int j) {
    const int rows = min(SUB, nmax - j * SUB);
    __nv_bfloat16* dst = ring + j * SUB * D;
    for (int idx = t; idx < rows * C8; idx += kThreads) {
      const int r = idx / C8, c = idx % C8;
      const int key = j * SUB + r;
      cp_async16(smem_addr(dst + r * D + ((c ^ swz(key)) << 3)),
                 src + seq_off + static_cast<int64_t>(key) * p.tok_stride + c * 8);
    }
    cp_async_commit();  // an empty group when the sub-tile holds no key keeps the count
  };

#pragma unroll
  for (int j = 0; j < NSUB; ++j) load_sub(p.k, j);
  for (int idx = t; idx < RB * 4 * D; idx += kThreads) {
    const int rg = idx / D, d = idx % D;
    float v = 0.f;
    if (rg < RG) {
      const int r = rg / G, i = rg % G;
      v = __bfloat162float(p.q[(static_cast<int64_t>(rs.row0 + r) * p.Hq + g * G + i) * D + d]);
    }
    qs[idx] = v;
  }

  // --- scores.  Four threads per key; lane q4 of a quad sums chunks q4,
  // q4 + 4, ... of d with FMAs, then two xor-shuffles add the quad's partials
  // (the same bits in all four lanes); lane q4 stores pair q4 of the block.
  const int kq = t >> 2, q4 = t & 3;
#pragma unroll
  for (int j = 0; j < NSUB; ++j) {
    cp_async_wait<3>();  // groups after K_j: K_{j+1..3} and V_{0..j-1}, three in all
    __syncthreads();
    if (j * SUB < nmax) {
      const int key = j * SUB + kq;
      const __nv_bfloat16* kr = ring + j * SUB * D + kq * D;
      uint4 kc[C8 / 4];
#pragma unroll
      for (int m = 0; m < C8 / 4; ++m)
        kc[m] = *reinterpret_cast<const uint4*>(kr + (((q4 + 4 * m) ^ swz(key)) << 3));
      for (int rb = 0; rb < RB; ++rb) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int m = 0; m < C8 / 4; ++m) {
          const int c = q4 + 4 * m;
          const float kf[8] = {bf16_lo(kc[m].x), bf16_hi(kc[m].x), bf16_lo(kc[m].y), bf16_hi(kc[m].y),
                               bf16_lo(kc[m].z), bf16_hi(kc[m].z), bf16_lo(kc[m].w), bf16_hi(kc[m].w)};
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const float4 qa = *reinterpret_cast<const float4*>(qs + (rb * 4 + r) * D + c * 8);
            const float4 qb = *reinterpret_cast<const float4*>(qs + (rb * 4 + r) * D + c * 8 + 4);
            float a = acc[r];
            a = fmaf(qa.x, kf[0], a); a = fmaf(qa.y, kf[1], a);
            a = fmaf(qa.z, kf[2], a); a = fmaf(qa.w, kf[3], a);
            a = fmaf(qb.x, kf[4], a); a = fmaf(qb.y, kf[5], a);
            a = fmaf(qb.z, kf[6], a); a = fmaf(qb.w, kf[7], a);
            acc[r] = a;
          }
        }
        float mine = 0.f;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          float a = acc[r];
          a = __fadd_rn(a, __shfl_xor_sync(0xffffffffu, a, 1));
          a = __fadd_rn(a, __shfl_xor_sync(0xffffffffu, a, 2));
          if (r == q4) mine = a;
        }
        const int pr = rb * 4 + q4;
        es[(rb * kSplit + key) * 4 + q4] = key < count(pr) ? __fmul_rn(mine, p.scale) : -INFINITY;
      }
    }
    __syncthreads();           // stage j is free
    if (j * SUB < nmax) load_sub(p.v, j);
    else cp_async_commit();
  }

  // --- softmax statistics: warp w takes block w (four pairs); lane l owns
  // keys l, l + 32, ..., l + 224 (sequential), then a butterfly per pair.
  for (int rb = warp; rb < RB; rb += kThreads / 32) {
    float4* e4 = reinterpret_cast<float4*>(es) + rb * kSplit;
    int cnt[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) cnt[r] = count(rb * 4 + r);
    float m[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
    for (int i = 0; i < kSplit / 32; ++i) {
      const int key = lane + 32 * i;
      const float4 x = e4[key];
      const float xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int r = 0; r < 4; ++r)
        if (key < cnt[r]) m[r] = fmaxf(m[r], xv[r]);
    }
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m[r] = fmaxf(m[r], __shfl_xor_sync(0xffffffffu, m[r], o));
    float l[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < kSplit / 32; ++i) {
      const int key = lane + 32 * i;
      const float4 x = e4[key];
      float xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        xv[r] = key < cnt[r] ? expf(__fsub_rn(xv[r], m[r])) : 0.f;
        l[r] = __fadd_rn(l[r], xv[r]);
      }
      e4[key] = make_float4(xv[0], xv[1], xv[2], xv[3]);
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) l[r] = __fadd_rn(l[r], __shfl_xor_sync(0xffffffffu, l[r], o));
      if (lane == 0) {
        mrow[rb * 4 + r] = m[r];
        lrow[rb * 4 + r] = l[r];
      }
    }
  }

  // --- o = sum_t e_t v_t.  Warp w owns column pairs dp = 8w .. 8w + 7; lane
  // = 8 kg + (dp - 8w): key group kg sums keys kg, kg + 4, ... ascending with
  // FMAs, and a butterfly over the four key groups (xor 8, 16) adds them.
  constexpr int DP_WARPS = D / 16;
  const int kg = lane >> 3;
  const int dp = warp * 8 + (lane & 7);
  const int col = 2 * dp;
  for (int rb = 0; rb < RB; ++rb) {
    int cnt[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) cnt[r] = count(rb * 4 + r);
    float2 o[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                   make_float2(0.f, 0.f)};
    const float4* e4 = reinterpret_cast<const float4*>(es) + rb * kSplit;
#pragma unroll
    for (int j = 0; j < NSUB; ++j) {
      if (rb == 0) {
        if (j == 0) cp_async_wait<3>();
        else if (j == 1) cp_async_wait<2>();
        else if (j == 2) cp_async_wait<1>();
        else cp_async_wait<0>();
        __syncthreads();
      }
      if (warp < DP_WARPS) {
        const int kend = min(SUB, nmax - j * SUB);
        const __nv_bfloat16* vt = ring + j * SUB * D;
        for (int kk = kg; kk < kend; kk += 4) {
          const int key = j * SUB + kk;
          const uint32_t vv = *reinterpret_cast<const uint32_t*>(
              vt + kk * D + (((col >> 3) ^ swz(key)) << 3) + (col & 7));
          const float v0 = bf16_lo(vv), v1 = bf16_hi(vv);
          const float4 e = e4[key];
          const float ev[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            if (key < cnt[r]) {
              o[r].x = fmaf(ev[r], v0, o[r].x);
              o[r].y = fmaf(ev[r], v1, o[r].y);
            }
          }
        }
      }
    }
    if (warp < DP_WARPS) {
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        o[r].x = __fadd_rn(o[r].x, __shfl_xor_sync(0xffffffffu, o[r].x, 8));
        o[r].y = __fadd_rn(o[r].y, __shfl_xor_sync(0xffffffffu, o[r].y, 8));
        o[r].x = __fadd_rn(o[r].x, __shfl_xor_sync(0xffffffffu, o[r].x, 16));
        o[r].y = __fadd_rn(o[r].y, __shfl_xor_sync(0xffffffffu, o[r].y, 16));
        const int pr = rb * 4 + r;
        if (kg == 0 && pr < RG && cnt[r] > 0) {
          const int row = pr / G, i = pr % G;
          const int64_t base = (static_cast<int64_t>(rs.row0 + row) * p.Hq + g * G + i) * p.S + s;
          *reinterpret_cast<float2*>(p.ws_o + base * D + col) = o[r];
          if (dp == 0) {
            p.ws_ml[base * 2 + 0] = mrow[pr];
            p.ws_ml[base * 2 + 1] = lrow[pr];
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
    len = p.kv_len[row];
  } else {
    const int b = blockIdx.z;
    const int i = blockIdx.y;
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
  const int ns = (len + kSplit - 1) / kSplit;
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

template <int D>
size_t split_smem_bytes(int rg_cap) {
  return static_cast<size_t>(kSplit) * D * 2 + static_cast<size_t>(rg_cap) * D * 4 +
         static_cast<size_t>(rg_cap) * kSplit * 4;
}

template <int D>
kinv_status launch(const AttnParams& p, dim3 split_grid, dim3 merge_grid, cudaStream_t stream) {
  const size_t smem = split_smem_bytes<D>(p.rg_cap);
  static bool configured[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KINV_ERR_CUDA;
  if (dev < 64 && !configured[dev]) {
    if (cudaFuncSetAttribute(attn_split_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(split_smem_bytes<D>(kMaxRG))) != cudaSuccess)
      return KINV_ERR_CUDA;
    configured[dev] = true;
  }
  const kinv_status st = launch_kernel(attn_split_kernel<D>, split_grid, dim3(kThreads), smem, stream, 1, p);
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

extern "C" kinv_status kinv_attn_decode(const void* q, const void* k_cache, const void* v_cache,
                                        int64_t seq_stride, int64_t tok_stride,
                                        const int32_t* kv_len, void* out, int B, int Hq, int Hkv,
                                        int D, int Lmax, int split_len, float scale,
                                        void* workspace, size_t ws_bytes, kinv_stream stream) {
  if (B < 0 || Lmax < 0) return KINV_ERR_INVALID_ARG;
  if (B == 0) return KINV_OK;
  if (!kv_len) return KINV_ERR_INVALID_ARG;
  kinv_status st = check_common(q, k_cache, v_cache, seq_stride, tok_stride, out, Hq, Hkv, D,
                                split_len, workspace);
  if (st != KINV_OK) return st;
  if (B > 65535) return KINV_ERR_UNSUPPORTED;
  const int S = Lmax > 0 ? (Lmax + kSplit - 1) / kSplit : 1;
  if (ws_bytes < workspace_bytes(B, Hq, D, S)) return KINV_ERR_WORKSPACE;
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
  const dim3 split_grid(Hkv, S, B), merge_grid(Hq, B, 1);
  return D == 128 ? launch<128>(p, split_grid, merge_grid, stream)
                  : launch<64>(p, split_grid, merge_grid, stream);
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
  p.R = kMaxRG / p.G < 8 ? kMaxRG / p.G : 8;
  p.S = S;
  p.groups_per_seq = (max_q_len + p.R - 1) / p.R;
  p.rg_cap = ((p.R * p.G + 3) / 4) * 4;
  p.scale = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(D));
  const int64_t groups = static_cast<int64_t>(B) * p.groups_per_seq;
  if (groups > 65535 || max_q_len > 65535 || B > 65535) return KINV_ERR_UNSUPPORTED;
  const dim3 split_grid(Hkv, S, static_cast<unsigned>(groups)), merge_grid(Hq, max_q_len, B);
  return D == 128 ? launch<128>(p, split_grid, merge_grid, stream)
                  : launch<64>(p, split_grid, merge_grid, stream);
}

// ---------------------------------------------------------------------------
// kinv_attn_decode_noalloc: decode attention for callers that cannot allocate
// device memory.  The split partials go to a scratch array compiled into the
// library instead of a caller-provided workspace.

#include <mutex>

// Scratch shared by every kinv_attn_decode_noalloc call on a device (held by
// each GPU that loads the library until the process exits).
static __device__ __align__(256) unsigned char kinv_noalloc_scratch[KINV_NOALLOC_SCRATCH_BYTES];

namespace kinv {
namespace {

// In host code the array's name is a host-side stand-in, not a device
// address: the device address is looked up once per device, with that device
// current, and cached.
void* noalloc_scratch_address() {
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, kinv_noalloc_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace
}  // namespace kinv

extern "C" kinv_status kinv_attn_decode_noalloc(const void* q, const void* k_cache,
                                                const void* v_cache, int64_t seq_stride,
                                                int64_t tok_stride, const int32_t* kv_len,
                                                void* out, int B, int Hq, int Hkv, int D, int Lmax,
                                                int split_len, float scale, kinv_stream stream) {
  if (B < 0 || Lmax < 0) return KINV_ERR_INVALID_ARG;
  if (B == 0) return KINV_OK;
  if (!kv_len || Hq <= 0 || D <= 0) return KINV_ERR_INVALID_ARG;
  if (B > 65535) return KINV_ERR_UNSUPPORTED;
  if (split_len != kSplit) return KINV_ERR_UNSUPPORTED;
  const int S = Lmax > 0 ? (Lmax + kSplit - 1) / kSplit : 1;
  const size_t need = workspace_bytes(B, Hq, D, S);
  if (need > static_cast<size_t>(KINV_NOALLOC_SCRATCH_BYTES)) return KINV_ERR_WORKSPACE;
  // shape and alignment checks first (no CUDA call), with a stand-in pointer
  const void* aligned_placeholder = reinterpret_cast<const void*>(static_cast<uintptr_t>(256));
  kinv_status st = check_common(q, k_cache, v_cache, seq_stride, tok_stride, out, Hq, Hkv, D,
                                split_len, aligned_placeholder);
  if (st != KINV_OK) return st;
  void* scratch = noalloc_scratch_address();
  if (!scratch) return KINV_ERR_CUDA;
  AttnParams p{};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k_cache);
  p.v = static_cast<const __nv_bfloat16*>(v_cache);
  p.seq_stride = seq_stride;
  p.tok_stride = tok_stride;
  p.kv_len = kv_len;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.ws_o = static_cast<float*>(scratch);
  const size_t o_bytes = static_cast<size_t>(B) * Hq * S * D * 4;
  p.ws_ml = reinterpret_cast<float*>(static_cast<char*>(scratch) + ((o_bytes + 255) / 256) * 256);
  p.prefill = 0;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.R = 1;
  p.S = S;
  p.groups_per_seq = 1;
  p.rg_cap = ((p.G + 3) / 4) * 4;
  p.scale = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(D));
  const dim3 split_grid(Hkv, S, B), merge_grid(Hq, B, 1);
  return D == 128 ? launch<128>(p, split_grid, merge_grid, stream)
                  : launch<64>(p, split_grid, merge_grid, stream);
}
