// Rotary position embedding with the optional per-head RMSNorm (QK-norm), as
// one warp per head.  Shared by the stand-alone kernel (kinv_rope_append) and
// the epilogue of the fused QKV projection (kinv_gemm_qkv_rope), so both
// produce the same bits for the same bf16 inputs.
//
// Rotate-half pairs (i, i + D/2), theta_i = p * base^(-2i/D) for absolute
// position p: (a, b) -> (a cos - b sin, b cos + a sin).
#pragma once

#include "common.cuh"

namespace kinv {

struct RopeFreqs {
  double inv_freq[64];  // base^(-2i/D), formed on the host in fp64
};

// cos and sin of theta = p * inv_freq: theta in fp64, reduced to [-pi, pi] in
// fp64 (2 pi split into a head and a tail), then sin and cos in fp32.
__device__ __forceinline__ void rope_angle(int p, double inv_freq, float& c, float& s) {
  const double theta = static_cast<double>(p) * inv_freq;
  const double k = rint(theta * 0.15915494309189535);  // 1 / (2 pi)
  double red = fma(-k, 6.283185307179586, theta);
  red = fma(-k, 2.4492935982947064e-16, red);
  sincosf(static_cast<float>(red), &s, &c);
}

// One head of D values held by a warp: lane l holds the pairs (i, i + D/2) for
// i in {l * P .. l * P + P - 1}, P = D / 64, as a[] and b[]; c[] and s[] are
// the cos and sin of those i.  With a norm weight nw the head is first scaled
// by 1 / sqrt(mean of squares + eps) (per lane: the a's then the b's by FMA,
// then a butterfly over the 32 lanes) and by nw.  Writes the rotated head to
// dst (bf16).
template <int D>
__device__ __forceinline__ void rope_norm_rotate(float (&a)[D / 64], float (&b)[D / 64],
                                                 const float (&c)[D / 64], const float (&s)[D / 64],
                                                 const __nv_bfloat16* __restrict__ nw, float eps,
                                                 int lane, __nv_bfloat16* __restrict__ dst) {
  constexpr int HALF = D / 2;
  constexpr int P = D / 64;
  if (nw) {
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < P; ++j) acc = fmaf(a[j], a[j], acc);
#pragma unroll
    for (int j = 0; j < P; ++j) acc = fmaf(b[j], b[j], acc);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, o));
    acc = __shfl_sync(0xffffffffu, acc, 0);
    const float inv =
        __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(acc, static_cast<float>(D)), eps)));
#pragma unroll
    for (int j = 0; j < P; ++j) {
      a[j] = __fmul_rn(__fmul_rn(a[j], inv), __bfloat162float(nw[lane * P + j]));
      b[j] = __fmul_rn(__fmul_rn(b[j], inv), __bfloat162float(nw[HALF + lane * P + j]));
    }
  }
  // every operation rounded on its own (no contraction), wherever this is inlined
#pragma unroll
  for (int j = 0; j < P; ++j) {
    const int i = lane * P + j;
    dst[i] = __float2bfloat16_rn(__fsub_rn(__fmul_rn(a[j], c[j]), __fmul_rn(b[j], s[j])));
    dst[HALF + i] = __float2bfloat16_rn(__fadd_rn(__fmul_rn(b[j], c[j]), __fmul_rn(a[j], s[j])));
  }
}

}  // namespace kinv
