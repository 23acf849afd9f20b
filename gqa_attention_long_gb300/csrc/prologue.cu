// prologue.cu — K1: fused per-head RMSNorm + HF rotate_half RoPE of the 64 expert tokens, the
// own-row write into the cache tail, and the staging of the roped Q (and a swizzled copy of the
// own K/V rows) in the workspace in the shared-memory layout the attention kernel consumes.
//
// alpamayo_tt/expert.py, TTExpert.layer (rms_norm of q and k with the q_norm / k_norm gains,
// rotary_embedding_hf, typecast to the cache dtype, fill_cache at row Smax-64) and
// TTExpert.set_context (positions i + rope_delta + S); alpamayo_tt/EXPERT_NOTES.md, "Layouts".
//
// A CTA handles q heads 2g and 2g+1, k head g and v head g of one layer, for 16 tokens (bf16
// cache) or all 64 (FP8 cache). A half-warp owns one token at a time; lane i of the half-warp
// holds channels [8i, 8i+8), so a RoPE pair (d, d+64) sits in lanes i and i+8 and is exchanged
// with one shuffle. Every global access is a 16-byte vector access. It also zeroes the unit's
// per-row arrival counters used by the attention kernel's merge.
#include <cuda_fp8.h>

#include "internal.cuh"
#include "ptx.cuh"

namespace ea {

namespace {

// 2*pi as an fp32 head plus an fp32 tail, for a two-step Cody-Waite reduction.
constexpr float kTwoPiHi = 6.28318548202514648438f;
constexpr float kTwoPiLo = -1.74845553146951715e-07f;
constexpr float kInvTwoPi = 0.159154943091895335768f;

// cos and sin of pos * inv where inv = inv_hi + inv_lo. The product is formed as an exact fp32
// pair (fma residual), reduced modulo 2*pi (the first step is exact because |a| < 2^13 keeps
// a - k*2pi_hi within 23 bits), and only then handed to sincosf, so that the angle keeps about
// 1e-6 rad accuracy up to the 8K positions of a long cache.
__device__ __forceinline__ void rope_cos_sin(int pos, float inv_hi, float inv_lo, float& c,
                                             float& s) {
  const float p = static_cast<float>(pos);
  const float a_hi = p * inv_hi;
  const float a_lo = fmaf(p, inv_hi, -a_hi) + p * inv_lo;
  const float k = rintf(a_hi * kInvTwoPi);
  float r = fmaf(-k, kTwoPiHi, a_hi);
  r = fmaf(-k, kTwoPiLo, r);
  r += a_lo;
  sincosf(r, &s, &c);
}

__device__ __forceinline__ void unpack_bf16x8(const uint4 v, float (&x)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    x[2 * e] = __uint_as_float(w[e] << 16);
    x[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ void load_bf16x8(const __nv_bfloat16* src, float (&x)[8]) {
  unpack_bf16x8(*reinterpret_cast<const uint4*>(src), x);
}

__device__ __forceinline__ uint4 pack8(const float (&y)[8], bool f16) {
  uint32_t w[4];
#pragma unroll
  for (int e = 0; e < 4; ++e)
    w[e] = f16 ? pack_f16x2(y[2 * e], y[2 * e + 1]) : pack_bf16x2(y[2 * e], y[2 * e + 1]);
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// RMSNorm over the 128 channels held by a half-warp (8 per lane), then rotate_half RoPE.
__device__ __forceinline__ void norm_rope(const float (&x)[8], const float (&gam)[8],
                                          const float (&cs)[8], const float (&sn)[8], bool upper,
                                          float (&y)[8]) {
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
#pragma unroll
  for (int m = 8; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
  const float rs = rsqrtf(ss * (1.0f / kD) + 1e-6f);
  float n[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) n[e] = x[e] * rs * gam[e];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float partner = __shfl_xor_sync(0xffffffffu, n[e], 8);
    // d < 64:  y[d] = n[d] cos - n[d+64] sin;   d >= 64: y[d] = n[d] cos + n[d-64] sin
    y[e] = upper ? fmaf(n[e], cs[e], partner * sn[e]) : fmaf(n[e], cs[e], -partner * sn[e]);
  }
}

// Byte offset of the 16-byte chunk holding channels [8i, 8i+8) of row r in a swizzled tile
// whose two 64-channel atoms are `atom_bytes` apart.
__device__ __forceinline__ uint32_t swz_off(int r, int i, uint32_t atom_bytes) {
  return static_cast<uint32_t>(i >> 3) * atom_bytes + static_cast<uint32_t>(r) * 128u +
         (static_cast<uint32_t>((i & 7) ^ (r & 7)) << 4);
}

__device__ __forceinline__ float block_max_256(float v, float* red) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) r = fmaxf(r, red[w]);
  return r;
}

// 8 fp32 values / scale -> 8 e4m3 codes (RNE, satfinite) and their exact f16 widening.
__device__ __forceinline__ void quant8(const float (&y)[8], float scale, uint2& codes, uint4& wide) {
  uint32_t c[4];
  uint32_t h[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 q = make_float2(__fdiv_rn(y[2 * e], scale), __fdiv_rn(y[2 * e + 1], scale));
    const __nv_fp8x2_storage_t s = __nv_cvt_float2_to_fp8x2(q, __NV_SATFINITE, __NV_E4M3);
    c[e] = s;
    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(s, __NV_E4M3);
    h[e] = static_cast<uint32_t>(hr.x) | (static_cast<uint32_t>(hr.y) << 16);
  }
  codes = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
  wide = make_uint4(h[0], h[1], h[2], h[3]);
}

}  // namespace

// TPH = tokens per half-warp: 1 for bf16 caches (four light CTAs per unit, so that many CTAs
// are resident per SM), 4 for FP8 caches (one CTA per unit: the own-row scale needs the amax
// over all 64 tokens of the head).
template <int TPH>
__global__ void __launch_bounds__(256) prologue_kernel_t(const __grid_constant__ PrologueParams p) {
  // Launched programmatically after the previous kernel in the stream: wait for it (it may have
  // produced q/k/v, or still read the workspace), then let the attention kernel's CTAs start
  // their set-up; they wait for this grid before reading anything written here.
  pdl_wait_primary();
  pdl_launch_dependents();
  __shared__ float red[8];

  constexpr int kCtasPerUnit = 4 / TPH;
  const int unit_id = blockIdx.x / kCtasPerUnit;
  const int quarter = blockIdx.x % kCtasPerUnit;
  const int l = unit_id / kHkv, g = unit_id % kHkv;
  const PrologueLayer& L = p.layer[l];
  const int hw = threadIdx.x >> 4;   // half-warp: tokens t0 + hw + 16 tt
  const int t0 = quarter * 16;
  const int i = threadIdx.x & 15;    // channels [8i, 8i+8)
  const int d0 = 8 * i;
  const bool upper = i >= 8;
  const bool fp8 = p.fp8 != 0;
  const int Smax = p.Smax;

  float gq[8], gk[8], ih[8], il[8];
  load_bf16x8(L.q_gamma + d0, gq);
  load_bf16x8(L.k_gamma + d0, gk);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    ih[e] = p.inv_hi[(d0 & 63) + e];
    il[e] = p.inv_lo[(d0 & 63) + e];
  }
  const size_t unit = static_cast<size_t>(l) * kHkv + g;
  if (quarter == 0 && threadIdx.x < kRows) p.row_cnt[unit * kRows + threadIdx.x] = 0u;
  uint8_t* qdst = p.q_ws + unit * kQTileBytes;
  uint8_t* tdst = p.tail_ws + unit * kTailUnitBytes;

  float kr[TPH][8], vr[TPH][8];  // kept for the FP8 path, whose scale needs all 64 rows first
  float kmax = 0.f, vmax = 0.f;

  // All raw rows of this thread's 4 tokens are requested before any arithmetic, so that the
  // loads overlap instead of paying one memory latency per token.
  uint4 rq[TPH][2], rk[TPH], rv[TPH];
#pragma unroll
  for (int tt = 0; tt < TPH; ++tt) {
    const int t = t0 + hw + 16 * tt;
    rq[tt][0] = *reinterpret_cast<const uint4*>(L.q_raw + (static_cast<size_t>(2 * g) * kTok + t) * kD + d0);
    rq[tt][1] = *reinterpret_cast<const uint4*>(L.q_raw + (static_cast<size_t>(2 * g + 1) * kTok + t) * kD + d0);
    rk[tt] = *reinterpret_cast<const uint4*>(L.k_raw + (static_cast<size_t>(g) * kTok + t) * kD + d0);
    rv[tt] = *reinterpret_cast<const uint4*>(L.v_raw + (static_cast<size_t>(g) * kTok + t) * kD + d0);
  }

#pragma unroll
  for (int tt = 0; tt < TPH; ++tt) {
    const int t = t0 + hw + 16 * tt;
    const int pos = t + p.rope_delta + p.S;
    float cs[8], sn[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) rope_cos_sin(pos, ih[e], il[e], cs[e], sn[e]);

#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int h = 2 * g + hh;
      float x[8], y[8];
      unpack_bf16x8(rq[tt][hh], x);
      norm_rope(x, gq, cs, sn, upper, y);
      const int r = hh * kTok + t;
      *reinterpret_cast<uint4*>(qdst + swz_off(r, i, kQTileBytes / 2)) = pack8(y, fp8);
      if (L.q_rope != nullptr)
        *reinterpret_cast<uint4*>(L.q_rope + (static_cast<size_t>(h) * kTok + t) * kD + d0) =
            pack8(y, false);
    }
    float x[8];
    unpack_bf16x8(rk[tt], x);
    norm_rope(x, gk, cs, sn, upper, kr[tt]);
    const uint4 vraw = rv[tt];
    const size_t row = static_cast<size_t>(g) * Smax + (Smax - kTok) + t;
    const uint32_t so = swz_off(t, i, kTailHalfBytes / 2);
    if (!fp8) {
      const uint4 kb = pack8(kr[tt], false);
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(L.k_cache) + row * kD + d0) = kb;
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(L.v_cache) + row * kD + d0) = vraw;
      *reinterpret_cast<uint4*>(tdst + so) = kb;
      *reinterpret_cast<uint4*>(tdst + kTailHalfBytes + so) = vraw;
    } else {
      unpack_bf16x8(vraw, vr[tt]);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        kmax = fmaxf(kmax, fabsf(kr[tt][e]));
        vmax = fmaxf(vmax, fabsf(vr[tt][e]));
      }
    }
  }
  if (TPH != 4 || !fp8) return;

  // FP8 cache: the 64 own rows of this head share one scale slot, column Smax/128.
  kmax = block_max_256(kmax, red);
  vmax = block_max_256(vmax, red);
  const float ksc = kmax > 0.f ? __fdiv_rn(kmax, 448.0f) : 1.0f;
  const float vsc = vmax > 0.f ? __fdiv_rn(vmax, 448.0f) : 1.0f;
  const int ncol = Smax / kScaleBlock + 1;
  if (threadIdx.x == 0) {
    L.k_scale[g * ncol + ncol - 1] = ksc;
    L.v_scale[g * ncol + ncol - 1] = vsc;
  }
#pragma unroll
  for (int tt = 0; tt < TPH; ++tt) {
    const int t = t0 + hw + 16 * tt;
    const size_t row = static_cast<size_t>(g) * Smax + (Smax - kTok) + t;
    const uint32_t so = swz_off(t, i, kTailHalfBytes / 2);
    uint2 c;
    uint4 w;
    quant8(kr[tt], ksc, c, w);
    *reinterpret_cast<uint2*>(static_cast<uint8_t*>(L.k_cache) + row * kD + d0) = c;
    *reinterpret_cast<uint4*>(tdst + so) = w;
    quant8(vr[tt], vsc, c, w);
    *reinterpret_cast<uint2*>(static_cast<uint8_t*>(L.v_cache) + row * kD + d0) = c;
    *reinterpret_cast<uint4*>(tdst + kTailHalfBytes + so) = w;
  }
}

// Host-side launcher (the kernel template is instantiated and launched in this file).
cudaError_t launch_prologue_kernel(const PrologueParams& pp, bool fp8, cudaLaunchConfig_t cfg) {
  cfg.gridDim = dim3(pp.n_layers * kHkv * (fp8 ? 1 : 4));  // FP8: one CTA per unit; bf16: four
  cfg.blockDim = dim3(256);
  return fp8 ? cudaLaunchKernelEx(&cfg, prologue_kernel_t<4>, pp)
             : cudaLaunchKernelEx(&cfg, prologue_kernel_t<1>, pp);
}

}  // namespace ea
