// Batch-invariant RMSNorm ("Deterministic and bit-exact inference",
// *technical*: RMSNorm made batch-invariant by fixing each row's reduction
// order).
//
// One thread block per row.  The block size depends only on `dim`; thread t
// owns the 8-element chunks t, t + T, t + 2T, ... and sums their squares in
// that order with fused multiply-adds; the 32 lane sums of a warp meet in a
// fixed xor-butterfly whose lane-0 result is taken; the warp sums are added by
// one thread in ascending warp order.  Nothing depends on the number of rows,
// so a row's bits are the same in any batch.
#include "common.cuh"

namespace kinv {
namespace {

constexpr int kMaxChunksPerThread = 8;  // dim <= 256 threads * 8 chunks * 8

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x);
  f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
  f[4] = bf16_lo(u.z); f[5] = bf16_hi(u.z);
  f[6] = bf16_lo(u.w); f[7] = bf16_hi(u.w);
}

__global__ void rmsnorm_kernel(__nv_bfloat16* __restrict__ x, int64_t ldx,
                               const __nv_bfloat16* __restrict__ residual,
                               const __nv_bfloat16* __restrict__ w,
                               __nv_bfloat16* __restrict__ y, int64_t ldy, int dim, float eps) {
  __shared__ float warp_sums[8];
  __shared__ float row_inv;
  pdl_launch_dependents();
  pdl_wait();
  const int row = blockIdx.x;
  const int t = threadIdx.x;
  const int T = blockDim.x;
  const int chunks = dim >> 3;
  __nv_bfloat16* xr = x + row * ldx;
  const __nv_bfloat16* rr = residual ? residual + row * ldx : nullptr;

  float v[kMaxChunksPerThread][8];
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < kMaxChunksPerThread; ++i) {
    const int c = t + i * T;
    if (c < chunks) {
      uint4 u = *reinterpret_cast<const uint4*>(xr + c * 8);
      unpack8(u, v[i]);
      if (rr) {
        float r8[8];
        unpack8(*reinterpret_cast<const uint4*>(rr + c * 8), r8);
        // new residual stream s = bf16(x + r), kept in registers as bf16 values
#pragma unroll
        for (int e = 0; e < 8; ++e) v[i][e] = __bfloat162float(__float2bfloat16_rn(v[i][e] + r8[e]));
        uint4 o;
        o.x = pack_bf16(v[i][0], v[i][1]);
        o.y = pack_bf16(v[i][2], v[i][3]);
        o.z = pack_bf16(v[i][4], v[i][5]);
        o.w = pack_bf16(v[i][6], v[i][7]);
        *reinterpret_cast<uint4*>(xr + c * 8) = o;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) acc = fmaf(v[i][e], v[i][e], acc);
    }
  }
  // fixed butterfly inside the warp; lane 0's value is the warp's sum
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((t & 31) == 0) warp_sums[t >> 5] = acc;
  __syncthreads();
  if (t == 0) {
    float ss = 0.f;
    for (int i = 0; i < (T >> 5); ++i) ss += warp_sums[i];
    row_inv = 1.0f / sqrtf(ss / static_cast<float>(dim) + eps);
  }
  __syncthreads();
  const float inv = row_inv;
  __nv_bfloat16* yr = y + row * ldy;
#pragma unroll
  for (int i = 0; i < kMaxChunksPerThread; ++i) {
    const int c = t + i * T;
    if (c < chunks) {
      float g[8];
      unpack8(*reinterpret_cast<const uint4*>(w + c * 8), g);
      uint4 o;
      o.x = pack_bf16(v[i][0] * inv * g[0], v[i][1] * inv * g[1]);
      o.y = pack_bf16(v[i][2] * inv * g[2], v[i][3] * inv * g[3]);
      o.z = pack_bf16(v[i][4] * inv * g[4], v[i][5] * inv * g[5]);
      o.w = pack_bf16(v[i][6] * inv * g[6], v[i][7] * inv * g[7]);
      *reinterpret_cast<uint4*>(yr + c * 8) = o;
    }
  }
}

}  // namespace
}  // namespace kinv

extern "C" kinv_status kinv_rmsnorm(void* x, int64_t ldx, const void* residual, const void* w,
                                    void* y, int64_t ldy, int rows, int dim, float eps,
                                    kinv_stream stream) {
  using namespace kinv;
  if (rows < 0 || dim <= 0 || !(eps >= 0.f)) return KINV_ERR_INVALID_ARG;
  if (rows == 0) return KINV_OK;
  if (!x || !w || !y) return KINV_ERR_INVALID_ARG;
  if (dim % 8 != 0 || dim > 256 * 8 * kMaxChunksPerThread) return KINV_ERR_UNSUPPORTED;
  if (ldx < dim || ldy < dim) return KINV_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w) || !aligned16(y) || (residual && !aligned16(residual)) ||
      ldx % 8 || ldy % 8)
    return KINV_ERR_ALIGNMENT;
  const int chunks = dim / 8;
  int threads = chunks < 256 ? ((chunks + 31) / 32) * 32 : 256;
  return launch_kernel(rmsnorm_kernel, dim3(rows), dim3(threads), 0, stream, 1,
                       static_cast<__nv_bfloat16*>(x), ldx, static_cast<const __nv_bfloat16*>(residual),
                       static_cast<const __nv_bfloat16*>(w), static_cast<__nv_bfloat16*>(y), ldy, dim,
                       eps);
}
