// linear.cu — the projections of the expert's decoder layer for its 64 tokens (Y = X W^T with
// weights stored [out_features, in_features]) on the sm_103a tensor cores, and the small
// kernels that finish the layer around them: RMSNorm, head split, residual adds, SwiGLU.
//
// alpamayo_tt/expert.py, TTExpert.layer: rms_norm(x, ln1); the fused wqkv projection and
// nlp_create_qkv_heads; after the attention, nlp_concat_heads, wo and the residual add;
// rms_norm(x1, ln2); w1 with silu, w3, their product, w2 and the second residual add.
//
// The activation operand is tiny (64 x K) and the weights are large (N x K) and read once, so
// a projection is HBM-bound on its weights. It is computed transposed, D[n][t] = sum_k W[n][k]
// X[t][k]: 128 weight rows form the M = 128 operand A and the 64 tokens the N = 64 operand B of
// tcgen05.mma (kind::f16, bf16 in, fp32 accumulator in 64 TMEM columns). To spread the weights
// over every SM the K dimension is split: CTA (tile, split) streams weight rows [128 tile,
// 128 tile + 128) over its range of 64-channel k-steps, and writes its fp32 partial
// D[t][n] into part[split][t][n]; a finishing kernel sums the splits and applies the layer's
// epilogue. Two CTAs fit on an SM (96 KB ring, 64 TMEM columns each).
#include "internal.cuh"
#include "ptx.cuh"

namespace ea {

namespace lin {
constexpr int kThreads = 192;  // warps 0-3: epilogue (TMEM lanes 0-127); warp 4: TMA; warp 5: MMA
constexpr int kStages = 4;
constexpr uint32_t kWTile = 128 * 64 * 2;  // 128 weight rows x 64 channels, bf16, 128-byte rows
constexpr uint32_t kXTile = 64 * 64 * 2;   // 64 tokens x 64 channels
constexpr uint32_t kStage = kWTile + kXTile;
constexpr uint32_t SM_BAR = kStages * kStage;          // full[kStages], empty[kStages], done
constexpr uint32_t SM_TMEM = SM_BAR + (2 * kStages + 1) * 8;
constexpr uint32_t SM_ABORT = SM_TMEM + 4;
constexpr uint32_t kSmemBytes = SM_ABORT + 4 + 1024;   // + slack to align the base to 1 KB
constexpr uint32_t kTmemCols = 64;
}  // namespace lin

__global__ void __launch_bounds__(lin::kThreads, 2) linear_kernel(const __grid_constant__ LinearParams p) {
  using namespace lin;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + SM_BAR;
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (kStages + s); };
  const uint32_t done = bar0 + 8u * (2 * kStages);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + SM_ABORT);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x, split = blockIdx.y;
  const int k0 = split * p.kps;
  const int nk = min(p.kps, p.ksteps - k0);  // >= 1 by the host's choice of the split count

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(done, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(sbase + SM_TMEM, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    prefetch_tensormap(&p.wmap[tile < p.tiles0 ? 0 : 1]);
    prefetch_tensormap(&p.xmap);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + SM_TMEM);

  if (warp == 4) {
    if (lane == 0) {
      const uint64_t pol_w = l2_policy_evict_first();  // weights: read once
      const uint64_t pol_x = l2_policy_evict_last();   // activations: read by every CTA
      const CUtensorMap* wm = &p.wmap[tile < p.tiles0 ? 0 : 1];
      const int row0 = (tile < p.tiles0 ? tile : tile - p.tiles0) * 128;
      // The weights do not depend on the previous kernel in the stream (no kernel of this
      // library writes them): their first ring stages are loaded, and the rest of this CTA's
      // weight slice prefetched into L2, while that kernel may still run. The activations
      // are its output: they are loaded only after griddepcontrol.wait.
      const int pre = nk < kStages ? nk : kStages;
      for (int i = 0; i < pre; ++i) {
        mbar_expect_tx(full(i), kStage);
        tma_load_2d(sbase + i * kStage, wm, full(i), (k0 + i) * 64, row0, pol_w);
      }
      for (int i = pre; i < nk; ++i) tma_prefetch_2d(wm, (k0 + i) * 64, row0);
      pdl_wait_primary();
      for (int i = 0; i < pre; ++i) {
        const int kk = k0 + i;
        tma_load_4d(sbase + i * kStage + kWTile, &p.xmap, full(i), 0, kk % p.c1, 0, kk / p.c1, pol_x);
      }
      bool ok = true;
      int i = pre;
      for (; i < nk; ++i) {
        const int s = i % kStages;
        ok = bounded_wait(empty(s), ((i / kStages) - 1) & 1, abort_flag, p.status, kErrLinearWait);
        if (!ok) break;
        const int kk = k0 + i;
        const uint32_t dst = sbase + s * kStage;
        mbar_expect_tx(full(s), kStage);
        tma_load_2d(dst, wm, full(s), kk * 64, row0, pol_w);
        tma_load_4d(dst + kWTile, &p.xmap, full(s), 0, kk % p.c1, 0, kk / p.c1, pol_x);
      }
      pdl_launch_dependents();
      if (!ok) {  // let the copies already issued land before the CTA gives its shared memory back
        for (int j = (i > kStages ? i - kStages : 0); j < i; ++j)
          if (!drain_wait(full(j % kStages), (j / kStages) & 1)) atomicOr(p.status, kErrDrain);
      }
    }
  } else if (warp == 5) {
    if (lane == 0) {
      constexpr uint32_t kIdesc = umma_idesc_f16(128, 64, true, false, false);
      bool ok = true;
      for (int i = 0; i < nk && ok; ++i) {
        const int s = i % kStages;
        ok = bounded_wait(full(s), (i / kStages) & 1, abort_flag, p.status, kErrLinearWait);
        if (!ok) break;
        tc_fence_after();
        const uint32_t wa = sbase + s * kStage, xa = wa + kWTile;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // 16 channels (32 bytes of the 128-byte row) per MMA
          umma_f16_ss(tmem, sw128_desc(wa + kk * 32, 16, 1024), sw128_desc(xa + kk * 32, 16, 1024),
                      kIdesc, i > 0 || kk > 0);
        umma_commit(empty(s));
      }
      // every MMA issued so far completes before `done` (and before TMEM is released)
      umma_commit(done);
      if (!drain_wait(done, 0)) atomicOr(p.status, kErrDrain);
    }
  } else {
    // epilogue: thread r of warps 0-3 owns TMEM lane r = weight row 128 tile + r; its 64 columns
    // are the 64 tokens. part[split][t][n]: for a fixed token a warp's stores are 128
    // contiguous bytes. (The partial buffer may still be read by the previous kernel in the
    // stream until griddepcontrol.wait returns.)
    pdl_wait_primary();
    const bool ok = bounded_wait(done, 0, abort_flag, p.status, kErrLinearWait);
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
      const int r = warp * 32 + lane;
      float* dst = p.part + static_cast<size_t>(split) * kTok * p.N + static_cast<size_t>(tile) * 128 + r;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t v[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + 32 * h, v);
        tmem_wait_ld();
        reg_fence32(v);
#pragma unroll
        for (int e = 0; e < 32; ++e) dst[static_cast<size_t>(32 * h + e) * p.N] = __uint_as_float(v[e]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, kTmemCols);
}

// ----------------------------------------------------------------------- finishing kernels
// Sum over the K splits of part[s][t][n .. n+3] (fp32, 16-byte aligned), eight splits' loads
// in flight at a time (the adds in split order).
__device__ __forceinline__ float4 split_sum4(const float* part, int splits, int N, int t, int n) {
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
  const size_t stride = static_cast<size_t>(kTok) * N;
  const float* p0 = part + static_cast<size_t>(t) * N + n;
  for (int s0 = 0; s0 < splits; s0 += 8) {
    float4 v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)  // unconditional loads (index clamped), so all eight are in flight
      v[e] = __ldcg(reinterpret_cast<const float4*>(p0 + min(s0 + e, splits - 1) * stride));
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if (s0 + e < splits) {
        a.x += v[e].x;
        a.y += v[e].y;
        a.z += v[e].z;
        a.w += v[e].w;
      }
    }
  }
  return a;
}

__device__ __forceinline__ float bf16_val(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// One CTA per token row: y = x (+ the split sum of part, if given), rounded to bf16 and stored
// to y_out (if given); then, if gamma is given, h = gamma * y / sqrt(mean(y^2) + eps) over the
// row's `width` channels, rounded to bf16 and stored to h_out. The layer's first RMSNorm
// (no part), the wo finish (part, residual, norm) and the w2 finish (part, residual) use it.
__global__ void __launch_bounds__(384) residual_norm_kernel(const float* part, int splits,
                                                           const __nv_bfloat16* x, int width,
                                                           __nv_bfloat16* y_out,
                                                           const __nv_bfloat16* gamma,
                                                           __nv_bfloat16* h_out) {
  pdl_launch_dependents();
  pdl_wait_primary();
  __shared__ float red[32];
  __shared__ float row_y[kMaxHidden];
  const int t = blockIdx.x;
  float ss = 0.f;
  for (int n = 4 * threadIdx.x; n < width; n += 4 * blockDim.x) {
    const uint2 xv = *reinterpret_cast<const uint2*>(x + static_cast<size_t>(t) * width + n);
    float y[4] = {__uint_as_float(xv.x << 16), __uint_as_float(xv.x & 0xFFFF0000u),
                  __uint_as_float(xv.y << 16), __uint_as_float(xv.y & 0xFFFF0000u)};
    if (part != nullptr) {
      const float4 a = split_sum4(part, splits, width, t, n);
      y[0] = bf16_val(y[0] + a.x);
      y[1] = bf16_val(y[1] + a.y);
      y[2] = bf16_val(y[2] + a.z);
      y[3] = bf16_val(y[3] + a.w);
    }
    if (y_out != nullptr) {
      uint2 o;
      o.x = pack_bf16x2(y[0], y[1]);
      o.y = pack_bf16x2(y[2], y[3]);
      *reinterpret_cast<uint2*>(y_out + static_cast<size_t>(t) * width + n) = o;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      row_y[n + e] = y[e];
      ss = fmaf(y[e], y[e], ss);
    }
  }
  if (gamma == nullptr) return;
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) tot += red[w];
  const float rs = rsqrtf(tot / static_cast<float>(width) + 1e-6f);
  for (int n = 4 * threadIdx.x; n < width; n += 4 * blockDim.x) {
    const uint2 gv = *reinterpret_cast<const uint2*>(gamma + n);
    const float g[4] = {__uint_as_float(gv.x << 16), __uint_as_float(gv.x & 0xFFFF0000u),
                        __uint_as_float(gv.y << 16), __uint_as_float(gv.y & 0xFFFF0000u)};
    uint2 o;
    o.x = pack_bf16x2(g[0] * (row_y[n] * rs), g[1] * (row_y[n + 1] * rs));
    o.y = pack_bf16x2(g[2] * (row_y[n + 2] * rs), g[3] * (row_y[n + 3] * rs));
    *reinterpret_cast<uint2*>(h_out + static_cast<size_t>(t) * width + n) = o;
  }
}

// The fused projection's split sums -> bf16 q [16][64][128], k and v [8][64][128]: feature
// 128 h + d of the q (k, v) block is channel d of head h (nlp_create_qkv_heads).
__global__ void __launch_bounds__(256) qkv_heads_kernel(const float* part, int splits,
                                                       __nv_bfloat16* q, __nv_bfloat16* k,
                                                       __nv_bfloat16* v) {
  pdl_launch_dependents();
  pdl_wait_primary();
  constexpr int kN = (kHq + 2 * kHkv) * kD;  // 4096
  const int t = blockIdx.y;
  const int n = 4 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (n >= kN) return;
  const float4 a = split_sum4(part, splits, kN, t, n);
  uint2 o;
  o.x = pack_bf16x2(a.x, a.y);
  o.y = pack_bf16x2(a.z, a.w);
  const int head = n / kD, d = n % kD;
  __nv_bfloat16* dst = head < kHq ? q + (static_cast<size_t>(head) * kTok + t) * kD
                       : head < kHq + kHkv ? k + (static_cast<size_t>(head - kHq) * kTok + t) * kD
                                           : v + (static_cast<size_t>(head - kHq - kHkv) * kTok + t) * kD;
  *reinterpret_cast<uint2*>(dst + d) = o;
}

// SwiGLU: gu[t][j] = silu(gate) * up, where gate and up are the split sums of features j and
// inter + j (the gate projection w1 fills the first `inter` features of the GEMM, the up
// projection w3 the rest); silu(g) = g / (1 + e^-g).
__global__ void __launch_bounds__(256) swiglu_kernel(const float* part, int splits, int inter,
                                                    __nv_bfloat16* gu) {
  pdl_launch_dependents();
  pdl_wait_primary();
  const int t = blockIdx.y;
  const int j = 4 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (j >= inter) return;
  const float4 g = split_sum4(part, splits, 2 * inter, t, j);
  const float4 u = split_sum4(part, splits, 2 * inter, t, inter + j);
  auto sw = [](float a, float b) { return a * __frcp_rn(1.0f + expf(-a)) * b; };
  uint2 o;
  o.x = pack_bf16x2(sw(g.x, u.x), sw(g.y, u.y));
  o.y = pack_bf16x2(sw(g.z, u.z), sw(g.w, u.w));
  *reinterpret_cast<uint2*>(gu + static_cast<size_t>(t) * inter + j) = o;
}

// Plain projection output: y[t][n] = bf16(split sum of part[.][t][n]), y row-major [64][N].
__global__ void __launch_bounds__(256) split_sum_bf16_kernel(const float* part, int splits, int N,
                                                            __nv_bfloat16* y) {
  pdl_launch_dependents();
  pdl_wait_primary();
  const int t = blockIdx.y;
  const int n = 4 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (n >= N) return;
  const float4 a = split_sum4(part, splits, N, t, n);
  uint2 o;
  o.x = pack_bf16x2(a.x, a.y);
  o.y = pack_bf16x2(a.z, a.w);
  *reinterpret_cast<uint2*>(y + static_cast<size_t>(t) * N + n) = o;
}

// ------------------------------------------------------------------------------ launchers
cudaError_t linear_set_attributes() {
  return cudaFuncSetAttribute(linear_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(lin::kSmemBytes));
}

cudaError_t launch_linear(const LinearParams& lp, int tiles, int splits, cudaLaunchConfig_t cfg) {
  cfg.gridDim = dim3(tiles, splits);
  cfg.blockDim = dim3(lin::kThreads);
  cfg.dynamicSmemBytes = lin::kSmemBytes;
  return cudaLaunchKernelEx(&cfg, linear_kernel, lp);
}

cudaError_t launch_residual_norm(const float* part, int splits, const __nv_bfloat16* x, int width,
                                 __nv_bfloat16* y_out, const __nv_bfloat16* gamma,
                                 __nv_bfloat16* h_out, cudaLaunchConfig_t cfg) {
  cfg.gridDim = dim3(kTok);
  cfg.blockDim = dim3(384);  // one float4 of a 1536-wide row per thread
  cfg.dynamicSmemBytes = 0;
  return cudaLaunchKernelEx(&cfg, residual_norm_kernel, part, splits, x, width, y_out, gamma, h_out);
}

cudaError_t launch_qkv_heads(const float* part, int splits, __nv_bfloat16* q, __nv_bfloat16* k,
                             __nv_bfloat16* v, cudaLaunchConfig_t cfg) {
  constexpr int kN = (kHq + 2 * kHkv) * kD;
  cfg.gridDim = dim3(kN / 4 / 256, kTok);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  return cudaLaunchKernelEx(&cfg, qkv_heads_kernel, part, splits, q, k, v);
}

cudaError_t launch_swiglu(const float* part, int splits, int inter, __nv_bfloat16* gu,
                          cudaLaunchConfig_t cfg) {
  cfg.gridDim = dim3((inter / 4 + 255) / 256, kTok);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  return cudaLaunchKernelEx(&cfg, swiglu_kernel, part, splits, inter, gu);
}

}  // namespace ea

namespace ea {
cudaError_t launch_split_sum_bf16(const float* part, int splits, int N, __nv_bfloat16* y,
                                  cudaLaunchConfig_t cfg) {
  cfg.gridDim = dim3((N / 4 + 255) / 256, kTok);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  return cudaLaunchKernelEx(&cfg, split_sum_bf16_kernel, part, splits, N, y);
}
}  // namespace ea
