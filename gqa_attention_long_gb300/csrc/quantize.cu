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


// ------------------------------------------------------------------------------ MXFP4 cache
// The 4-bit cache variant: OCP MX v1.0 MXFP4, E2M1 codes with one power-of-two (E8M0) scale per
// 32 consecutive channels of a row (the block-scaled 4-bit type of the sm_103a tensor cores).
// One warp per cache row: lane l holds channels 4 l .. 4 l + 3, so block j (channels
// [32 j, 32 j + 32)) is lanes 8 j .. 8 j + 7 and its amax takes three shuffles. The block's
// exponent is e = floor(log2(amax)) - 2 (2: the exponent of E2M1's largest value, 6 = 1.5 * 2^2),
// clamped to [-127, 127], 0 for an all-zero block; x * 2^-e is exact, and rounding to E2M1 is
// done with the format's midpoints, each tie going to the code with mantissa bit 0:
//   magnitude 0 0.5 1 1.5 2 3 4 6 = codes 0..7; bit 3 = the sign of x.
// Output: codes packed two per byte (the lower channel in the low nibble), 64 bytes per row, and
// one scale byte e + 127 per block, 4 per row.
__device__ __forceinline__ uint32_t e2m1_code(float x) {
  const float r = fabsf(x);
  uint32_t c = (r > 0.25f) + (r >= 0.75f) + (r > 1.25f) + (r >= 1.75f) + (r > 2.5f) + (r >= 3.5f) +
               (r > 5.0f);
  return c | (signbit(x) ? 8u : 0u);
}

__global__ void __launch_bounds__(256) quantize_mxfp4_kernel(const __nv_bfloat16* __restrict__ src,
                                                             uint8_t* __restrict__ codes,
                                                             uint8_t* __restrict__ scales,
                                                             int n_rows, int Smax) {
  const int lane = threadIdx.x & 31;
  const long long w = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (w >= static_cast<long long>(kHkv) * n_rows) return;  // uniform per warp
  const long long g = w / n_rows, r = w % n_rows;
  const size_t row = static_cast<size_t>(g) * Smax + static_cast<size_t>(r);
  const uint2 raw = *reinterpret_cast<const uint2*>(src + row * kD + 4 * lane);
  const float x[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                      __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u)};
  float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
  for (int m = 1; m < 8; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
  int e = 0;
  if (amax > 0.f) e = min(max(ilogbf(amax) - 2, -127), 127);
  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) c[i] = e2m1_code(ldexpf(x[i], -e));
  const uint16_t packed = static_cast<uint16_t>(c[0] | (c[1] << 4) | (c[2] << 8) | (c[3] << 12));
  *reinterpret_cast<uint16_t*>(codes + row * (kD / 2) + 2 * lane) = packed;
  if ((lane & 7) == 0) scales[row * (kD / 32) + (lane >> 3)] = static_cast<uint8_t>(e + 127);
}

cudaError_t launch_quantize_mxfp4(const __nv_bfloat16* src, uint8_t* codes, uint8_t* scales, int n_rows,
                                  int Smax, cudaStream_t stream) {
  const long long rows = static_cast<long long>(kHkv) * n_rows;
  quantize_mxfp4_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, stream>>>(src, codes, scales,
                                                                                 n_rows, Smax);
  return cudaGetLastError();
}

}  // namespace ea
