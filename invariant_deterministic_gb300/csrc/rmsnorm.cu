// Batch-invariant RMSNorm ("Deterministic and bit-exact inference",
// *technical*: RMSNorm made batch-invariant by fixing each row's reduction
// order).
//
// One warp per row (eight rows per 256-thread block; which block a row lands
// in does not touch its arithmetic).  Lane l owns the 8-element chunks
// l, l + 32, l + 64, ... of the row and sums their squares in that order with
// fused multiply-adds; a fixed xor butterfly over the 32 lanes adds the lane
// sums (every lane ends with the same bits).  Nothing depends on the number
// of rows, so a row's bits are the same in any batch.  With a residual, the
// first pass also forms and stores s = bf16(x + r); the second pass re-reads
// the lane's own chunks of s (written by the same lane).
#include "common.cuh"

namespace kinv {
namespace {

constexpr int kRowsPerBlock = 8;

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x);
  f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
  f[4] = bf16_lo(u.z); f[5] = bf16_hi(u.z);
  f[6] = bf16_lo(u.w); f[7] = bf16_hi(u.w);
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint4 o;
  o.x = pack_bf16(f[0], f[1]);
  o.y = pack_bf16(f[2], f[3]);
  o.z = pack_bf16(f[4], f[5]);
  o.w = pack_bf16(f[6], f[7]);
  return o;
}

__global__ void __launch_bounds__(32 * kRowsPerBlock)
    rmsnorm_kernel(__nv_bfloat16* x, int64_t ldx, const __nv_bfloat16* __restrict__ residual,
                   const __nv_bfloat16* __restrict__ w, __nv_bfloat16* __restrict__ y, int64_t ldy,
                   int rows, int dim, float eps) {
  pdl_launch_dependents();
  pdl_wait();
  const int row = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int chunks = dim >> 3;
  __nv_bfloat16* xr = x + row * ldx;
  const __nv_bfloat16* rr = residual ? residual + row * ldx : nullptr;

  float acc = 0.f;
  for (int c = lane; c < chunks; c += 32) {
    float v[8];
    unpack8(*reinterpret_cast<const uint4*>(xr + c * 8), v);
    if (rr) {
      float r8[8];
      unpack8(*reinterpret_cast<const uint4*>(rr + c * 8), r8);
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = __bfloat162float(__float2bfloat16_rn(v[e] + r8[e]));
      *reinterpret_cast<uint4*>(xr + c * 8) = pack8(v);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) acc = fmaf(v[e], v[e], acc);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, o));
  const float inv = 1.0f / sqrtf(acc / static_cast<float>(dim) + eps);
  __nv_bfloat16* yr = y + row * ldy;
  for (int c = lane; c < chunks; c += 32) {
    float v[8], g[8];
    unpack8(*reinterpret_cast<const uint4*>(xr + c * 8), v);
    unpack8(*reinterpret_cast<const uint4*>(w + c * 8), g);
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = v[e] * inv * g[e];
    *reinterpret_cast<uint4*>(yr + c * 8) = pack8(v);
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
  if (dim % 8 != 0 || dim > 16384) return KINV_ERR_UNSUPPORTED;
  if (ldx < dim || ldy < dim) return KINV_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w) || !aligned16(y) || (residual && !aligned16(residual)) ||
      ldx % 8 || ldy % 8)
    return KINV_ERR_ALIGNMENT;
  const int blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
  return launch_kernel(rmsnorm_kernel, dim3(blocks), dim3(32 * kRowsPerBlock), 0, stream, 1,
                       static_cast<__nv_bfloat16*>(x), ldx, static_cast<const __nv_bfloat16*>(residual),
                       static_cast<const __nv_bfloat16*>(w), static_cast<__nv_bfloat16*>(y), ldy, rows,
                       dim, eps);
}
