// rope.cuh — RMSNorm + RoPE row helpers shared by the prologue kernel and by the attention
// kernel's Q and own-row preparation (device code).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "internal.cuh"
#include "ptx.cuh"

namespace ea {

// 2*pi as an fp32 head plus an fp32 tail, for a two-step Cody-Waite reduction.
constexpr float kTwoPiHi = 6.28318548202514648438f;
constexpr float kTwoPiLo = -1.74845553146951715e-07f;
constexpr float kInvTwoPi = 0.159154943091895335768f;

// cos and sin of pos * inv where inv = inv_hi + inv_lo. The product is formed as an exact fp32
// pair (fma residual) and reduced modulo 2*pi (the first step is exact because |a| < 2^13 keeps
// a - k*2pi_hi within 23 bits), so that the angle keeps about 1e-6 rad accuracy up to the 8K
// positions of a long cache; the reduced angle, within [-pi, pi], goes to the hardware sine and
// cosine (__sincosf: absolute error about 2^-21 there, far below a bf16 step, and no branch,
// so that many angles are evaluated side by side).
__device__ __forceinline__ void rope_cos_sin(int pos, float inv_hi, float inv_lo, float& c,
                                             float& s) {
  const float p = static_cast<float>(pos);
  const float a_hi = p * inv_hi;
  const float a_lo = fmaf(p, inv_hi, -a_hi) + p * inv_lo;
  const float k = rintf(a_hi * kInvTwoPi);
  float r = fmaf(-k, kTwoPiHi, a_hi);
  r = fmaf(-k, kTwoPiLo, r);
  r += a_lo;
  __sincosf(r, &s, &c);
}

// The eight inverse frequencies [dl, dl + 8) of the RoPE table (hi and lo parts), read as
// 16-byte vectors (dl a multiple of 8). The lanes of a warp read different entries, so that one
// vector read per four values keeps the table traffic low.
__device__ __forceinline__ void load_inv8(const float* hi, const float* lo, int dl, float (&ih)[8],
                                          float (&il)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(hi + dl), b = *reinterpret_cast<const float4*>(hi + dl + 4);
  const float4 c = *reinterpret_cast<const float4*>(lo + dl), d = *reinterpret_cast<const float4*>(lo + dl + 4);
  ih[0] = a.x; ih[1] = a.y; ih[2] = a.z; ih[3] = a.w; ih[4] = b.x; ih[5] = b.y; ih[6] = b.z; ih[7] = b.w;
  il[0] = c.x; il[1] = c.y; il[2] = c.z; il[3] = c.w; il[4] = d.x; il[5] = d.y; il[6] = d.z; il[7] = d.w;
}

__device__ __forceinline__ void unpack_bf16x8(const uint4 v, float (&x)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    x[2 * e] = __uint_as_float(w[e] << 16);
    x[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint4 pack8(const float (&y)[8], bool f16) {
  uint32_t w[4];
#pragma unroll
  for (int e = 0; e < 4; ++e)
    w[e] = f16 ? pack_f16x2(y[2 * e], y[2 * e + 1]) : pack_bf16x2(y[2 * e], y[2 * e + 1]);
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// RMSNorm over the 128 channels of one row held by an octet (lane i: channels [8i, 8i+8) in lo
// and their RoPE partners [64+8i, 64+8i+8) in hi), then rotate_half RoPE, all in-thread:
//   y[d] = n[d] cos - n[d+64] sin,   y[d+64] = n[d+64] cos + n[d] sin   (d < 64).
__device__ __forceinline__ void norm_rope(const float (&xl)[8], const float (&xh)[8],
                                          const float (&gl)[8], const float (&gh)[8],
                                          const float (&cs)[8], const float (&sn)[8],
                                          float (&yl)[8], float (&yh)[8]) {
  // sum of squares in two independent chains (a single chain of 16 dependent FMAs is the
  // longest latency of the row)
  float s2[2] = {0.f, 0.f};
#pragma unroll
  for (int e = 0; e < 8; ++e) s2[e & 1] = fmaf(xl[e], xl[e], fmaf(xh[e], xh[e], s2[e & 1]));
  float ss = s2[0] + s2[1];
#pragma unroll
  for (int m = 4; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
  const float rs = rsqrtf(ss * (1.0f / kD) + 1e-6f);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float nl = xl[e] * rs * gl[e];
    const float nh = xh[e] * rs * gh[e];
    yl[e] = fmaf(nl, cs[e], -nh * sn[e]);
    yh[e] = fmaf(nh, cs[e], nl * sn[e]);
  }
}

// Byte offset of the 16-byte chunk holding channels [8i, 8i+8) of row r in a swizzled tile
// whose two 64-channel atoms are `atom_bytes` apart.
__device__ __forceinline__ uint32_t swz_off(int r, int i, uint32_t atom_bytes) {
  return static_cast<uint32_t>(i >> 3) * atom_bytes + static_cast<uint32_t>(r) * 128u +
         (static_cast<uint32_t>((i & 7) ^ (r & 7)) << 4);
}

}  // namespace ea
