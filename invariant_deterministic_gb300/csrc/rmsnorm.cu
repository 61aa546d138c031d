// Batch-invariant RMSNorm ("Deterministic and bit-exact inference",
// *technical*: RMSNorm made batch-invariant by fixing each row's reduction
// order).
//
// One thread block per row.  The block size depends only on `dim`; thread t
// owns the 8-element chunks t, t + T, t + 2T, ... (all loaded up front) and
// sums their squares in that order with fused multiply-adds; a fixed xor
// butterfly adds the 32 lane sums of a warp (every lane ends with the same
// bits); the warp sums are added in ascending warp order.  Nothing depends on
// the number of rows, so a row's bits are the same in any batch.
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

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint4 o;
  o.x = pack_bf16(f[0], f[1]);
  o.y = pack_bf16(f[2], f[3]);
  o.z = pack_bf16(f[4], f[5]);
  o.w = pack_bf16(f[6], f[7]);
  return o;
}

__global__ void __launch_bounds__(256)
    rmsnorm_kernel(__nv_bfloat16* x, int64_t ldx, const __nv_bfloat16* __restrict__ residual,
                   const __nv_bfloat16* __restrict__ w, __nv_bfloat16* __restrict__ y, int64_t ldy,
                   int dim, float eps) {
  __shared__ float warp_sums[8];
  pdl_launch_dependents();
  pdl_wait();
  const int row = blockIdx.x;
  const int t = threadIdx.x;
  const int T = blockDim.x;
  const int lane = t & 31;
  const int chunks = dim >> 3;
  __nv_bfloat16* xr = x + row * ldx;
  const __nv_bfloat16* rr = residual ? residual + row * ldx : nullptr;

  uint4 raw[kMaxChunksPerThread];
  uint4 rraw[kMaxChunksPerThread];
#pragma unroll
  for (int i = 0; i < kMaxChunksPerThread; ++i) {
    const int c = t + i * T;
    if (c < chunks) {
      raw[i] = *reinterpret_cast<const uint4*>(xr + c * 8);
      if (rr) rraw[i] = *reinterpret_cast<const uint4*>(rr + c * 8);
    }
  }
  float v[kMaxChunksPerThread][8];
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < kMaxChunksPerThread; ++i) {
    const int c = t + i * T;
    if (c < chunks) {
      unpack8(raw[i], v[i]);
      if (rr) {
        float r8[8];
        unpack8(rraw[i], r8);
        // the new residual stream s = bf16(x + r), kept as bf16 values
#pragma unroll
        for (int e = 0; e < 8; ++e) v[i][e] = __bfloat162float(__float2bfloat16_rn(v[i][e] + r8[e]));
        *reinterpret_cast<uint4*>(xr + c * 8) = pack8(v[i]);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) acc = fmaf(v[i][e], v[i][e], acc);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, o));
  if (lane == 0) warp_sums[t >> 5] = acc;
  __syncthreads();
  float ss = warp_sums[0];
  for (int i = 1; i < (T >> 5); ++i) ss = __fadd_rn(ss, warp_sums[i]);
  const float inv = 1.0f / sqrtf(ss / static_cast<float>(dim) + eps);
  __nv_bfloat16* yr = y + row * ldy;
#pragma unroll
  for (int i = 0; i < kMaxChunksPerThread; ++i) {
    const int c = t + i * T;
    if (c < chunks) {
      float g[8];
      unpack8(*reinterpret_cast<const uint4*>(w + c * 8), g);
#pragma unroll
      for (int e = 0; e < 8; ++e) v[i][e] = v[i][e] * inv * g[e];
      *reinterpret_cast<uint4*>(yr + c * 8) = pack8(v[i]);
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
  if (rows > 2147483647 / 2) return KINV_ERR_UNSUPPORTED;
  const int chunks = dim / 8;
  const int threads = chunks < 256 ? ((chunks + 31) / 32) * 32 : 256;
  return launch_kernel(rmsnorm_kernel, dim3(rows), dim3(threads), 0, stream, 1,
                       static_cast<__nv_bfloat16*>(x), ldx, static_cast<const __nv_bfloat16*>(residual),
                       static_cast<const __nv_bfloat16*>(w), static_cast<__nv_bfloat16*>(y), ldy, dim,
                       eps);
}

// ------------------------------------------------------------ row_sumsq
namespace kinv {
namespace {

// One warp per (row, 128-column tile): lane l squares columns 4l .. 4l + 3 in
// order (FMA), then a fixed butterfly adds the lanes.
__global__ void row_sumsq_kernel(const __nv_bfloat16* __restrict__ x, int64_t ldx, int rows, int tiles,
                                 float* __restrict__ ss) {
  pdl_launch_dependents();
  pdl_wait();
  const int item = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (item >= rows * tiles) return;
  const int r = item / tiles, t = item % tiles;
  const uint2 v = *reinterpret_cast<const uint2*>(x + r * ldx + t * 128 + lane * 4);
  const float a0 = __uint_as_float(v.x << 16), a1 = __uint_as_float(v.x & 0xFFFF0000u);
  const float a2 = __uint_as_float(v.y << 16), a3 = __uint_as_float(v.y & 0xFFFF0000u);
  float acc = 0.f;
  acc = fmaf(a0, a0, acc);
  acc = fmaf(a1, a1, acc);
  acc = fmaf(a2, a2, acc);
  acc = fmaf(a3, a3, acc);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, o));
  if (lane == 0) ss[static_cast<int64_t>(r) * tiles + t] = acc;
}

}  // namespace
}  // namespace kinv

extern "C" kinv_status kinv_row_sumsq(const void* x, int64_t ldx, int rows, int dim, float* ss_out,
                                      kinv_stream stream) {
  if (rows < 0 || dim <= 0 || ldx < dim) return KINV_ERR_INVALID_ARG;
  if (rows == 0) return KINV_OK;
  if (!x || !ss_out) return KINV_ERR_INVALID_ARG;
  if (dim % 128) return KINV_ERR_UNSUPPORTED;
  if (!kinv::aligned16(x) || ldx % 8) return KINV_ERR_ALIGNMENT;
  const int tiles = dim / 128;
  const int64_t items = static_cast<int64_t>(rows) * tiles;
  if (items > (int64_t(1) << 30)) return KINV_ERR_UNSUPPORTED;
  const int warps = 8;
  return kinv::launch_kernel(kinv::row_sumsq_kernel, dim3(static_cast<unsigned>((items + warps - 1) / warps)),
                             dim3(32 * warps), 0, stream, 1, static_cast<const __nv_bfloat16*>(x), ldx,
                             rows, tiles, ss_out);
}
