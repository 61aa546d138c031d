// Element-wise glue of the decoder block: embedding gather, residual add,
// SwiGLU, rotary embedding with the key/value append, and the per-step
// bookkeeping of a decode loop.  None of these sums across elements except
// the optional per-head RMSNorm in kinv_rope_append, whose order is fixed
// per head exactly as in kinv_rmsnorm's scheme (per-lane, butterfly, lane 0).
#include <math.h>

#include <cmath>

#include "common.cuh"
#include "rope.cuh"

namespace kinv {
namespace {

__global__ void embed_kernel(const uint4* __restrict__ table, int vocab, int dim8,
                             const int32_t* __restrict__ ids, uint4* __restrict__ out) {
  pdl_launch_dependents();
  pdl_wait();
  const int r = blockIdx.x;
  const int id = ids[r];
  for (int c = threadIdx.x; c < dim8; c += blockDim.x) {
    uint4 v = make_uint4(0, 0, 0, 0);
    if (id >= 0 && id < vocab) v = table[static_cast<int64_t>(id) * dim8 + c];
    out[static_cast<int64_t>(r) * dim8 + c] = v;
  }
}

// out may alias x or y: each element is read before it is written, by the
// same thread.
__global__ void add_kernel(const uint4* x, const uint4* y, uint4* out, int64_t n8) {
  pdl_launch_dependents();
  pdl_wait();
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4 a = x[i], b = y[i];
    uint4 o;
    o.x = pack_bf16(bf16_lo(a.x) + bf16_lo(b.x), bf16_hi(a.x) + bf16_hi(b.x));
    o.y = pack_bf16(bf16_lo(a.y) + bf16_lo(b.y), bf16_hi(a.y) + bf16_hi(b.y));
    o.z = pack_bf16(bf16_lo(a.z) + bf16_lo(b.z), bf16_hi(a.z) + bf16_hi(b.z));
    o.w = pack_bf16(bf16_lo(a.w) + bf16_lo(b.w), bf16_hi(a.w) + bf16_hi(b.w));
    out[i] = o;
  }
}

// out[n][k] = bf16(w[n][k] * g[k]), fp32 product: an RMSNorm gain moved into
// the columns of the projection it feeds.  One thread per 8 columns.
__global__ void scale_columns_kernel(const __nv_bfloat16* __restrict__ w, int64_t ldw,
                                     const uint4* __restrict__ g, __nv_bfloat16* __restrict__ out,
                                     int64_t ldo, int K8) {
  pdl_launch_dependents();
  pdl_wait();
  const int n = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= K8) return;
  const uint4 a = *reinterpret_cast<const uint4*>(w + n * ldw + c * 8);
  const uint4 b = g[c];
  uint4 o;
  o.x = pack_bf16(__fmul_rn(bf16_lo(a.x), bf16_lo(b.x)), __fmul_rn(bf16_hi(a.x), bf16_hi(b.x)));
  o.y = pack_bf16(__fmul_rn(bf16_lo(a.y), bf16_lo(b.y)), __fmul_rn(bf16_hi(a.y), bf16_hi(b.y)));
  o.z = pack_bf16(__fmul_rn(bf16_lo(a.z), bf16_lo(b.z)), __fmul_rn(bf16_hi(a.z), bf16_hi(b.z)));
  o.w = pack_bf16(__fmul_rn(bf16_lo(a.w), bf16_lo(b.w)), __fmul_rn(bf16_hi(a.w), bf16_hi(b.w)));
  *reinterpret_cast<uint4*>(out + n * ldo + c * 8) = o;
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

__global__ void swiglu_kernel(const __nv_bfloat16* __restrict__ gu, int64_t ld_gu,
                              __nv_bfloat16* __restrict__ out, int64_t ld_out, int F) {
  pdl_launch_dependents();
  pdl_wait();
  const int r = blockIdx.y;
  const int c = (blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (c >= F) return;
  const uint4 g = *reinterpret_cast<const uint4*>(gu + r * ld_gu + c);
  const uint4 u = *reinterpret_cast<const uint4*>(gu + r * ld_gu + F + c);
  uint4 o;
  o.x = pack_bf16(silu_mul(bf16_lo(g.x), bf16_lo(u.x)), silu_mul(bf16_hi(g.x), bf16_hi(u.x)));
  o.y = pack_bf16(silu_mul(bf16_lo(g.y), bf16_lo(u.y)), silu_mul(bf16_hi(g.y), bf16_hi(u.y)));
  o.z = pack_bf16(silu_mul(bf16_lo(g.z), bf16_lo(u.z)), silu_mul(bf16_hi(g.z), bf16_hi(u.z)));
  o.w = pack_bf16(silu_mul(bf16_lo(g.w), bf16_lo(u.w)), silu_mul(bf16_hi(g.w), bf16_hi(u.w)));
  *reinterpret_cast<uint4*>(out + r * ld_out + c) = o;
}

// Inverse frequencies base^(-2i/D), formed once per call on the host in fp64.
// One block per row.  The first D/2 threads compute this row's rotation
// angles in fp64 (theta_i = p * inv_freq_i, then sin and cos) into shared
// memory; then each warp takes one head (grid.y picks eight of the row's
// heads).  Lane l of a warp holds the pairs
// (i, i + D/2) for i in {l * P .. l * P + P - 1}, P = D / 64.
template <int D>
__global__ void rope_append_kernel(const __nv_bfloat16* __restrict__ qkv, int64_t ld_qkv,
                                   __nv_bfloat16* __restrict__ q_out,
                                   __nv_bfloat16* __restrict__ k_cache,
                                   __nv_bfloat16* __restrict__ v_cache, int64_t seq_stride,
                                   int64_t tok_stride, const int32_t* __restrict__ seq,
                                   const int32_t* __restrict__ pos,
                                   const __nv_bfloat16* __restrict__ q_norm,
                                   const __nv_bfloat16* __restrict__ k_norm, float eps, int Hq,
                                   int Hkv, int heads_per_block, const RopeFreqs freqs) {
  constexpr int HALF = D / 2;
  constexpr int P = D / 64;  // pairs per lane
  __shared__ float cs[HALF], sn[HALF];
  pdl_launch_dependents();
  pdl_wait();
  const int r = blockIdx.x;
  const int p = pos[r];
  const int s = seq[r];
  for (int i = threadIdx.x; i < HALF; i += blockDim.x) rope_angle(p, freqs.inv_freq[i], cs[i], sn[i]);
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  const __nv_bfloat16* row = qkv + r * ld_qkv;
  __nv_bfloat16* kdst_row = k_cache + s * seq_stride + p * tok_stride;
  __nv_bfloat16* vdst_row = v_cache + s * seq_stride + p * tok_stride;
  const int heads = Hq + 2 * Hkv;
  // block y takes heads [y hpb, (y + 1) hpb) of the row, the warps in turn
  const int h_end = min(heads, (static_cast<int>(blockIdx.y) + 1) * heads_per_block);
  for (int h = blockIdx.y * heads_per_block + warp; h < h_end; h += nwarps) {
    const __nv_bfloat16* src = row + h * D;
    if (h >= Hq + Hkv) {  // value head: copy bits
      const int g = h - Hq - Hkv;
      for (int c = lane; c < D / 8; c += 32)
        reinterpret_cast<uint4*>(vdst_row + g * D)[c] = reinterpret_cast<const uint4*>(src)[c];
      continue;
    }
    float a[P], b[P], c[P], sv[P];
#pragma unroll
    for (int j = 0; j < P; ++j) {
      a[j] = __bfloat162float(src[lane * P + j]);
      b[j] = __bfloat162float(src[HALF + lane * P + j]);
      c[j] = cs[lane * P + j];
      sv[j] = sn[lane * P + j];
    }
    __nv_bfloat16* dst = h < Hq ? q_out + (static_cast<int64_t>(r) * Hq + h) * D
                                : kdst_row + (h - Hq) * D;
    rope_norm_rotate<D>(a, b, c, sv, h < Hq ? q_norm : k_norm, eps, lane, dst);
  }
}

__global__ void decode_advance_kernel(const int32_t* __restrict__ tokens, int32_t* history,
                                      int hist_ld, int32_t* hist_len, int64_t* step, int32_t* pos,
                                      int32_t* kv_len, int B) {
  pdl_launch_dependents();
  pdl_wait();
  // one warp per request: the warp shifts the history row in chunks of 32
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= B) return;
  int32_t* h = history + static_cast<int64_t>(b) * hist_ld;
  int n = hist_len[b];
  if (n >= hist_ld) {
    for (int i0 = 1; i0 < hist_ld; i0 += 32) {
      const int i = i0 + lane;
      const int32_t v = i < hist_ld ? h[i] : 0;
      __syncwarp();
      if (i < hist_ld) h[i - 1] = v;
      __syncwarp();
    }
    n = hist_ld - 1;
  }
  if (lane == 0) {
    h[n] = tokens[b];
    hist_len[b] = n + 1;
    step[b] += 1;
    if (pos) pos[b] += 1;
    if (kv_len) kv_len[b] += 1;
  }
}

}  // namespace
}  // namespace kinv

using namespace kinv;

extern "C" kinv_status kinv_embed(const void* table, int vocab, int dim, const int32_t* ids,
                                  void* out, int rows, kinv_stream stream) {
  if (rows < 0 || vocab <= 0 || dim <= 0) return KINV_ERR_INVALID_ARG;
  if (rows == 0) return KINV_OK;
  if (!table || !ids || !out) return KINV_ERR_INVALID_ARG;
  if (dim % 8) return KINV_ERR_UNSUPPORTED;
  if (!aligned16(table) || !aligned16(out)) return KINV_ERR_ALIGNMENT;
  const int dim8 = dim / 8;
  return launch_kernel(embed_kernel, dim3(rows), dim3(dim8 < 256 ? 32 * ((dim8 + 31) / 32) : 256), 0,
                       stream, 1, static_cast<const uint4*>(table), vocab, dim8, ids,
                       static_cast<uint4*>(out));
}

extern "C" kinv_status kinv_add(const void* x, const void* y, void* out, int64_t n,
                                kinv_stream stream) {
  if (n < 0) return KINV_ERR_INVALID_ARG;
  if (n == 0) return KINV_OK;
  if (!x || !y || !out) return KINV_ERR_INVALID_ARG;
  if (n % 8) return KINV_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(y) || !aligned16(out)) return KINV_ERR_ALIGNMENT;
  const int64_t n8 = n / 8;
  const int64_t blocks = (n8 + 255) / 256;
  const int grid = static_cast<int>(blocks < 4096 ? blocks : 4096);
  return launch_kernel(add_kernel, dim3(grid), dim3(256), 0, stream, 1, static_cast<const uint4*>(x),
                       static_cast<const uint4*>(y), static_cast<uint4*>(out), n8);
}

extern "C" kinv_status kinv_scale_columns(const void* w, int64_t ldw, const void* g, void* out,
                                          int64_t ldo, int N, int K, kinv_stream stream) {
  if (N < 0 || K <= 0) return KINV_ERR_INVALID_ARG;
  if (N == 0) return KINV_OK;
  if (!w || !g || !out || ldw < K || ldo < K) return KINV_ERR_INVALID_ARG;
  if (K % 8) return KINV_ERR_UNSUPPORTED;
  if (!aligned16(w) || !aligned16(g) || !aligned16(out) || ldw % 8 || ldo % 8) return KINV_ERR_ALIGNMENT;
  if (N > 65535 * 4) return KINV_ERR_UNSUPPORTED;
  const int K8 = K / 8;
  // rows in chunks of at most 65535 grid rows
  for (int n0 = 0; n0 < N; n0 += 65535) {
    const int rows = N - n0 < 65535 ? N - n0 : 65535;
    const kinv_status st = launch_kernel(
        scale_columns_kernel, dim3((K8 + 127) / 128, rows), dim3(128), 0, stream, 1,
        static_cast<const __nv_bfloat16*>(w) + static_cast<int64_t>(n0) * ldw, ldw,
        static_cast<const uint4*>(g), static_cast<__nv_bfloat16*>(out) + static_cast<int64_t>(n0) * ldo, ldo,
        K8);
    if (st != KINV_OK) return st;
  }
  return KINV_OK;
}

extern "C" kinv_status kinv_swiglu(const void* gu, int64_t ld_gu, void* out, int64_t ld_out,
                                   int rows, int F, kinv_stream stream) {
  if (rows < 0 || F <= 0) return KINV_ERR_INVALID_ARG;
  if (rows == 0) return KINV_OK;
  if (!gu || !out) return KINV_ERR_INVALID_ARG;
  if (F % 8) return KINV_ERR_UNSUPPORTED;
  if (ld_gu < 2 * static_cast<int64_t>(F) || ld_out < F) return KINV_ERR_INVALID_ARG;
  if (!aligned16(gu) || !aligned16(out) || ld_gu % 8 || ld_out % 8) return KINV_ERR_ALIGNMENT;
  if (rows > 65535) return KINV_ERR_UNSUPPORTED;
  dim3 grid((F / 8 + 127) / 128, rows);
  return launch_kernel(swiglu_kernel, grid, dim3(128), 0, stream, 1,
                       static_cast<const __nv_bfloat16*>(gu), ld_gu, static_cast<__nv_bfloat16*>(out),
                       ld_out, F);
}

extern "C" kinv_status kinv_rope_append(const void* qkv, int64_t ld_qkv, void* q_out,
                                        void* k_cache, void* v_cache, int64_t seq_stride,
                                        int64_t tok_stride, const int32_t* seq,
                                        const int32_t* pos, const void* q_norm,
                                        const void* k_norm, float eps, int rows, int Hq, int Hkv,
                                        int D, float rope_base, kinv_stream stream) {
  if (rows < 0 || Hq <= 0 || Hkv <= 0 || !(rope_base > 0.f) || !(eps >= 0.f))
    return KINV_ERR_INVALID_ARG;
  if (rows == 0) return KINV_OK;
  if (!qkv || !q_out || !k_cache || !v_cache || !seq || !pos) return KINV_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return KINV_ERR_UNSUPPORTED;
  if (ld_qkv < static_cast<int64_t>(Hq + 2 * Hkv) * D || tok_stride < static_cast<int64_t>(Hkv) * D ||
      seq_stride < 0)
    return KINV_ERR_INVALID_ARG;
  if (!aligned16(qkv) || !aligned16(q_out) || !aligned16(k_cache) || !aligned16(v_cache) ||
      ld_qkv % 8 || seq_stride % 8 || tok_stride % 8)
    return KINV_ERR_ALIGNMENT;
  RopeFreqs freqs;
  for (int i = 0; i < D / 2; ++i) freqs.inv_freq[i] = std::pow(static_cast<double>(rope_base), -2.0 * i / D);
  const int heads = Hq + 2 * Hkv;
  // eight warps; a block takes eight heads of a row (few rows: more blocks in
  // flight) or, from 512 rows, every head of it (the angles formed once per
  // row, a sixth of the blocks: measured 1.8 times as fast at 4096 rows of
  // the 8B shape, 1.2 times at 512)
  const int threads = 256;
  const int hpb = rows >= 512 ? heads : 8;
  const dim3 grid(rows, (heads + hpb - 1) / hpb);
  auto* k = static_cast<__nv_bfloat16*>(k_cache);
  auto* v = static_cast<__nv_bfloat16*>(v_cache);
  auto* src = static_cast<const __nv_bfloat16*>(qkv);
  auto* qo = static_cast<__nv_bfloat16*>(q_out);
  auto* qn = static_cast<const __nv_bfloat16*>(q_norm);
  auto* kn = static_cast<const __nv_bfloat16*>(k_norm);
  if (D == 128)
    return launch_kernel(rope_append_kernel<128>, grid, dim3(threads), 0, stream, 1, src,
                         ld_qkv, qo, k, v, seq_stride, tok_stride, seq, pos, qn, kn, eps, Hq, Hkv,
                         hpb, freqs);
  return launch_kernel(rope_append_kernel<64>, grid, dim3(threads), 0, stream, 1, src, ld_qkv,
                       qo, k, v, seq_stride, tok_stride, seq, pos, qn, kn, eps, Hq, Hkv,
                       hpb, freqs);
}

extern "C" kinv_status kinv_decode_advance(const int32_t* tokens, int32_t* history, int hist_ld,
                                           int32_t* hist_len, int64_t* step, int32_t* pos,
                                           int32_t* kv_len, int B, kinv_stream stream) {
  if (B < 0 || hist_ld <= 0) return KINV_ERR_INVALID_ARG;
  if (B == 0) return KINV_OK;
  if (!tokens || !history || !hist_len || !step) return KINV_ERR_INVALID_ARG;
  return launch_kernel(decode_advance_kernel, dim3((B + 3) / 4), dim3(128), 0, stream, 1, tokens,
                       history, hist_ld, hist_len, step, pos, kv_len, B);
}
