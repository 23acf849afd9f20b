// linear.cu — the projections of the expert's decoder layer for its 64 tokens (Y = X W^T with
// weights stored [out_features, in_features]) on the sm_103a tensor cores, with the layer's
// RMSNorms of the residual stream fused into the projections that consume them.
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
// 128 tile + 128) over its range of 64-channel k-steps. The splits of a tile form one thread-
// block cluster, which sums its fp32 partials through distributed shared memory and writes
// the projection's output with its epilogue (head split, residual add, SwiGLU) applied, so no
// partial sum travels through global memory. Two CTAs fit on an SM (96 KB ring, 64 TMEM
// columns each).
#include "internal.cuh"
#include "cluster_exit.cuh"
#include "ptx.cuh"

namespace ea {

namespace lin {
constexpr int kThreads = 192;  // warps 0-3: epilogue (TMEM lanes 0-127); warp 4: TMA; warp 5: MMA
constexpr int kStages = 4;
constexpr uint32_t kWTile = 128 * 64 * 2;  // 128 weight rows x 64 channels, bf16, 128-byte rows
constexpr uint32_t kXTile = 64 * 64 * 2;   // 64 tokens x 64 channels
constexpr uint32_t kStage = kWTile + kXTile;
// barriers: full[kStages], empty[kStages], done, and (fused RMSNorm) xrdy[kStages], gains
constexpr uint32_t SM_BAR = kStages * kStage;
constexpr uint32_t SM_TMEM = SM_BAR + (3 * kStages + 2) * 8;
constexpr uint32_t SM_ABORT = SM_TMEM + 4;
// fused RMSNorm: per-token sums of squares of this CTA's channels, then 1 / rms; the gains of
// this CTA's channels (at most kNormMaxSteps k-steps, a split-planning constraint)
constexpr uint32_t SM_SSQ = (SM_ABORT + 4 + 15) & ~15u;
constexpr uint32_t SM_INV = SM_SSQ + kTok * 4;
constexpr uint32_t SM_GAMMA = SM_INV + kTok * 4;
constexpr uint32_t kSmemBytes = SM_GAMMA + kNormMaxSteps * 128 + 1024;  // + slack to align the base
static_assert(2 * (kSmemBytes + 1024) <= 228 * 1024, "two CTAs per SM");
constexpr uint32_t kTmemCols = 64;
constexpr int kMaxCluster = 16;                         // K splits of one tile = one cluster
static_assert(kTok * 128 * 4 <= kStages * kStage, "the fp32 tile fits in the drained ring");
}  // namespace lin

// Sum over the cluster's S CTAs (in rank order) of the float4 at shared address `addr` of each,
// up to four loads in flight at a time. The CTA's own partial (rank q) is read with a local
// shared-memory load: a load through the cluster window costs the same distributed-shared-memory
// bandwidth whichever CTA it names.
__device__ __forceinline__ float4 cluster_sum4(uint32_t addr, uint32_t S, uint32_t q) {
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
  for (uint32_t p0 = 0; p0 < S; p0 += 4) {
    float4 v[4];
#pragma unroll
    for (uint32_t e = 0; e < 4; ++e) {
      const uint32_t pe = p0 + e;  // the same for every thread of the CTA
      if (pe == q) {
        const uint4 u = ld_shared_v4(addr);
        v[e] = make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z),
                           __uint_as_float(u.w));
      } else if (pe < S) {
        v[e] = ld_shared_cluster_v4(mapa_shared(addr, pe));
      }
    }
#pragma unroll
    for (uint32_t e = 0; e < 4; ++e) {
      if (p0 + e < S) {
        a.x += v[e].x;
        a.y += v[e].y;
        a.z += v[e].z;
        a.w += v[e].w;
      }
    }
  }
  return a;
}

__device__ __forceinline__ uint2 pack_bf16x4(float a, float b, float c, float d) {
  uint2 o;
  o.x = pack_bf16x2(a, b);
  o.y = pack_bf16x2(c, d);
  return o;
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g * __frcp_rn(1.0f + expf(-g)) * u; }

// One projection tile: CTA (tile, split) of a cluster of the tile's S splits. Its MMAs leave the
// split's fp32 partial D[row][token] in TMEM; the epilogue warps move it into the (drained)
// ring as [token][row]; after a cluster barrier every CTA sums, for its share of the tile, the
// S partials read from the cluster's shared memory (in split order, so the result does not
// depend on timing), and applies the projection's epilogue:
//   kLinPlain     y[t][n] = sum                      (y row-major [64][N])
//   kLinResidual  y[t][n] = res[t][n] + sum          (rounded once, to bf16)
//   kLinQkvHeads  tile h = features [128 h, 128 h + 128): q head h (h < 16), k head h - 16
//                 (h < 24) or v head h - 24, written head-major [head][t][d]
//   kLinSwiglu    the tile's rows are 64 gate rows (wmap[0]) then the same 64 up rows
//                 (wmap[1]); y[t][64 tile + j] = silu(gate_j) * up_j
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
  auto xrdy = [&](int s) { return bar0 + 8u * (2 * kStages + 1 + s); };
  const uint32_t gbar = bar0 + 8u * (3 * kStages + 1);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + SM_ABORT);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x, split = blockIdx.y;
  const bool pair = p.mode == kLinSwiglu;
  const bool norm = p.norm_gamma != nullptr;  // the X operand is rms_norm(X) * norm_gamma
  const int k0 = split * p.kps;
  const int nk = min(p.kps, p.ksteps - k0);  // >= 1 by the host's choice of the split count

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(done, 1);
    for (int s = 0; s < kStages; ++s) mbar_init(xrdy(s), 128);
    mbar_init(gbar, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(sbase + SM_TMEM, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    prefetch_tensormap(&p.wmap[0]);
    if (pair) prefetch_tensormap(&p.wmap[1]);
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
      const int row0 = tile * (pair ? 64 : 128);
      auto load_w = [&](int s, int kk) {  // one stage's weight rows (two 64-row boxes for a pair)
        const uint32_t dst = sbase + s * kStage;
        tma_load_2d(dst, &p.wmap[0], full(s), kk * 64, row0, pol_w);
        if (pair) tma_load_2d(dst + kWTile / 2, &p.wmap[1], full(s), kk * 64, row0, pol_w);
      };
      // The weights do not depend on the previous kernel in the stream (no kernel of this
      // library writes them): their first ring stages are loaded, and the rest of this CTA's
      // weight slice prefetched into L2, while that kernel may still run. The activations
      // are its output: they are loaded only after griddepcontrol.wait.
      const int pre = nk < kStages ? nk : kStages;
      if (norm) {  // the gains of this CTA's channels, one contiguous bulk copy
        mbar_expect_tx(gbar, static_cast<uint32_t>(nk) * 128u);
        bulk_load(sbase + SM_GAMMA, p.norm_gamma + static_cast<size_t>(k0) * 64, static_cast<uint32_t>(nk) * 128u,
                  gbar, pol_x);
      }
      for (int i = 0; i < pre; ++i) {
        mbar_expect_tx(full(i), kStage);
        load_w(i, k0 + i);
      }
      for (int i = pre; i < nk; ++i) {
        tma_prefetch_2d(&p.wmap[0], (k0 + i) * 64, row0);
        if (pair) tma_prefetch_2d(&p.wmap[1], (k0 + i) * 64, row0);
      }
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
        mbar_expect_tx(full(s), kStage);
        load_w(s, kk);
        tma_load_4d(sbase + s * kStage + kWTile, &p.xmap, full(s), 0, kk % p.c1, 0, kk / p.c1, pol_x);
      }
      pdl_launch_dependents();
      if (!ok) {  // let the copies already issued land before the ring is reused or released
        for (int j = (i > kStages ? i - kStages : 0); j < i; ++j)
          if (!drain_wait(full(j % kStages), (j / kStages) & 1)) atomicOr(p.status, kErrDrain);
      }
      // the gains' copy has landed before the CTA can leave (normally long since)
      if (norm && !drain_wait(gbar, 0)) atomicOr(p.status, kErrDrain);
    }
  } else if (warp == 5) {
    if (lane == 0) {
      constexpr uint32_t kIdesc = umma_idesc_f16(128, 64, true, false, false);
      bool ok = true;
      for (int i = 0; i < nk && ok; ++i) {
        const int s = i % kStages;
        ok = bounded_wait(full(s), (i / kStages) & 1, abort_flag, p.status, kErrLinearWait);
        if (ok && norm) ok = bounded_wait(xrdy(s), (i / kStages) & 1, abort_flag, p.status, kErrLinearWait);
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
    if (norm) {
      // Fused RMSNorm of the X operand. Y = rms_norm(X) diag(g) W^T is computed as
      // diag(1 / rms) ((X diag(g)) W^T): while the MMAs run, warps 0-3 scale each landed X tile
      // by the gains of its 64 channels in place (token t = thread / 2, one half of the row
      // each) and sum the squares of X over this CTA's channels; the cluster's CTAs cover all K
      // channels, so after the first cluster barrier every CTA sums those per-token partials in
      // rank order and applies 1 / rms to the reduced tile.
      const int t = threadIdx.x >> 1, half = threadIdx.x & 1;
      float2 ss2 = make_float2(0.f, 0.f);
      const bool gok = bounded_wait(gbar, 0, abort_flag, p.status, kErrLinearWait);
      for (int i = 0; i < nk && gok; ++i) {
        const int s = i % kStages;
        if (!bounded_wait(full(s), (i / kStages) & 1, abort_flag, p.status, kErrLinearWait)) break;
        uint4 gc[4];  // gains of channels 64 (k0 + i) + 32 half .. + 31
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) gc[jj] = ld_shared_v4(sbase + SM_GAMMA + i * 128 + 16 * (4 * half + jj));
        // row t of the tile: 128 bytes, 16-byte chunk j stored at position j ^ (t % 8)
        const uint32_t row = sbase + s * kStage + kWTile + t * 128;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int j = 4 * half + jj;
          const uint32_t a = row + 16 * (j ^ (t & 7));
          const uint4 xv = ld_shared_v4(a);
          const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
          const uint32_t gw[4] = {gc[jj].x, gc[jj].y, gc[jj].z, gc[jj].w};
          uint32_t o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 xf = make_float2(__uint_as_float(xw[e] << 16), __uint_as_float(xw[e] & 0xFFFF0000u));
            ss2 = __ffma2_rn(xf, xf, ss2);
            // g * x of two bf16 values is exact in fp32, so one bf16x2 multiply (round to
            // nearest) gives the same bits as the fp32 product rounded to bf16
            asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(o[e]) : "r"(xw[e]), "r"(gw[e]));
          }
          st_shared_v4(a, o[0], o[1], o[2], o[3]);
        }
        fence_proxy_async_smem();  // the scaled tile is read by the tensor core
        mbar_arrive(xrdy(s));
      }
      float ss = ss2.x + ss2.y;
      ss += __shfl_xor_sync(0xffffffffu, ss, 1);
      if (half == 0) st_shared_f32(sbase + SM_SSQ + 4u * t, ss);
    }
    // thread r of warps 0-3 owns TMEM lane r (tile row r); its 64 columns are the 64 tokens.
    // The split's partial goes to shared memory as [token][row] (conflict-free stores).
    const bool ok = bounded_wait(done, 0, abort_flag, p.status, kErrLinearWait);
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
      const int r = warp * 32 + lane;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t v[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + 32 * h, v);
        tmem_wait_ld();
        reg_fence32(v);
#pragma unroll
        for (int e = 0; e < 32; ++e)
          st_shared_f32(sbase + static_cast<uint32_t>((32 * h + e) * 128 + r) * 4u, __uint_as_float(v[e]));
      }
    }
  }
  // every CTA of the cluster has its partial in shared memory
  cluster_sync();
  if (warp < 4) {
    // outputs are written, and the residual read, only after the previous kernel has finished
    pdl_wait_primary();
    const uint32_t S = gridDim.y, q = cluster_ctarank();
    const int i = threadIdx.x;
    if (norm) {
      if (i < kTok) {  // 1 / rms of token i: its sums of squares over the cluster, in rank order
        const uint32_t a = sbase + SM_SSQ + 4u * i;
        float v[kMaxCluster];
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r) {
          v[r] = 0.f;
          if (r < static_cast<int>(S))
            v[r] = r == static_cast<int>(q) ? reinterpret_cast<const float*>(smem + SM_SSQ)[i]
                                            : ld_shared_cluster_f32(mapa_shared(a, r));
        }
        float ssq = 0.f;
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r)
          if (r < static_cast<int>(S)) ssq += v[r];
        st_shared_f32(sbase + SM_INV + 4u * i, rsqrtf(ssq / static_cast<float>(p.ksteps * 64) + 1e-6f));
      }
      bar_sync(1, 128);
    }
    const int per_t = pair ? 16 : 32;  // float4 items per token: (gate) rows of the tile / 4
    const int n_items = kTok * per_t;
    for (int item = static_cast<int>(q) * 128 + i; item < n_items; item += static_cast<int>(S) * 128) {
      const int t = item / per_t, c = 4 * (item % per_t);  // token, first row of the float4
      float4 a = cluster_sum4(sbase + static_cast<uint32_t>(t * 128 + c) * 4u, S, q);
      const float inv = norm ? reinterpret_cast<const float*>(smem + SM_INV)[t] : 1.f;
      if (norm) a = make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv);
      if (p.mode == kLinSwiglu) {
        float4 u = cluster_sum4(sbase + static_cast<uint32_t>(t * 128 + 64 + c) * 4u, S, q);
        if (norm) u = make_float4(u.x * inv, u.y * inv, u.z * inv, u.w * inv);
        *reinterpret_cast<uint2*>(p.y + static_cast<size_t>(t) * p.N + tile * 64 + c) =
            pack_bf16x4(silu_mul(a.x, u.x), silu_mul(a.y, u.y), silu_mul(a.z, u.z), silu_mul(a.w, u.w));
      } else if (p.mode == kLinQkvHeads) {
        __nv_bfloat16* dst = tile < kHq ? p.q + static_cast<size_t>(tile) * kTok * kD
                             : tile < kHq + kHkv ? p.k + static_cast<size_t>(tile - kHq) * kTok * kD
                                                 : p.v + static_cast<size_t>(tile - kHq - kHkv) * kTok * kD;
        *reinterpret_cast<uint2*>(dst + static_cast<size_t>(t) * kD + c) = pack_bf16x4(a.x, a.y, a.z, a.w);
      } else {
        const size_t o = static_cast<size_t>(t) * p.N + tile * 128 + c;
        float4 b = a;
        if (p.mode == kLinResidual) {
          const uint2 rv = *reinterpret_cast<const uint2*>(p.res + o);
          b.x += __uint_as_float(rv.x << 16);
          b.y += __uint_as_float(rv.x & 0xFFFF0000u);
          b.z += __uint_as_float(rv.y << 16);
          b.w += __uint_as_float(rv.y & 0xFFFF0000u);
        }
        *reinterpret_cast<uint2*>(p.y + o) = pack_bf16x4(b.x, b.y, b.z, b.w);
      }
    }
  }
  // no CTA leaves (or reuses its shared memory) while a peer may still read it
  cluster_sync_exit();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------------------ launchers
cudaError_t linear_set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(linear_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(lin::kSmemBytes));
  if (e == cudaSuccess) e = cudaFuncSetAttribute(linear_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

// grid (tiles, splits) in clusters of (1, splits); cfg carries the PDL attribute in attrs[0] and
// has room for the cluster attribute in attrs[1]
cudaError_t launch_linear(const LinearParams& lp, int tiles, int splits, cudaLaunchConfig_t cfg) {
  cfg.gridDim = dim3(tiles, splits);
  cfg.blockDim = dim3(lin::kThreads);
  cfg.dynamicSmemBytes = lin::kSmemBytes;
  cudaLaunchAttribute* attr = cfg.attrs;
  attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
  attr[cfg.numAttrs].val.clusterDim.x = 1;
  attr[cfg.numAttrs].val.clusterDim.y = static_cast<unsigned>(splits);
  attr[cfg.numAttrs].val.clusterDim.z = 1;
  cfg.numAttrs += 1;
  return cudaLaunchKernelEx(&cfg, linear_kernel, lp);
}

}  // namespace ea
