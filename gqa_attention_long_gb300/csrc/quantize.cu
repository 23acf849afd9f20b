// quantize.cu — producer of the FP8 (OCP E4M3) cache variant: rows [0, n_rows) of a bf16 cache
// [8][Smax][128] become e4m3 codes with one fp32 scale amax/448 per (kv head, 128-row block).
//
// The pages keep the cache in bf16 or Tenstorrent block-float8 and cast the expert's own rows
// to the cache dtype before writing them (alpamayo_tt/expert.py, TTExpert.layer: typecast then
// fill_cache; alpamayo_tt/EXPERT_NOTES.md, "Timing": bfp8 cache). Block-float8 has no GPU
// counterpart; e4m3 codes with per-block fp32 scales take its place.
//
// One CTA per (kv head, 128-row block): pass 1 finds the block's amax, pass 2 encodes. The
// scale and the quotient x / scale are formed with IEEE round-to-nearest division, and the
// encode is cvt.rn.satfinite.e4m3x2.f32, so the codes are a deterministic function of the
// bf16 input.
#include <cuda_fp8.h>

#include "internal.cuh"
#include "ptx.cuh"

namespace ea {

__global__ void __launch_bounds__(256) quantize_cache_kernel(const __nv_bfloat16* __restrict__ src,
                                                             uint8_t* __restrict__ dst,
                                                             float* __restrict__ scales,
                                                             int n_rows, int Smax) {
  __shared__ float red[8];
  const int nb = Smax / kScaleBlock;
  const int g = blockIdx.x / nb, b = blockIdx.x % nb;
  const int r0 = b * kScaleBlock;
  const int r1 = min(r0 + kScaleBlock, n_rows);
  if (r0 >= r1) return;  // uniform per CTA
  const int n_chunks = (r1 - r0) * (kD / 8);  // 8-channel chunks in the block
  const size_t base = (static_cast<size_t>(g) * Smax + r0) * kD;

  float v[8][8];
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int c = threadIdx.x + 256 * k;
    if (c < n_chunks) {
      const uint4 w = *reinterpret_cast<const uint4*>(src + base + static_cast<size_t>(c) * 8);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v[k][2 * e] = __uint_as_float(ws[e] << 16);
        v[k][2 * e + 1] = __uint_as_float(ws[e] & 0xFFFF0000u);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(v[k][e]));
    }
  }
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) amax = fmaxf(amax, red[w]);
  const float sc = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  if (threadIdx.x == 0) scales[g * (nb + 1) + b] = sc;

#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int c = threadIdx.x + 256 * k;
    if (c < n_chunks) {
      uint32_t q[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = make_float2(__fdiv_rn(v[k][2 * e], sc), __fdiv_rn(v[k][2 * e + 1], sc));
        q[e] = __nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
      }
      *reinterpret_cast<uint2*>(dst + base + static_cast<size_t>(c) * 8) =
          make_uint2(q[0] | (q[1] << 16), q[2] | (q[3] << 16));
    }
  }
}

}  // namespace ea
