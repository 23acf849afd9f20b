// merge.cu — K3: log-sum-exp merge of the (layer, kv head) units that the attention kernel split
// across CTAs (the reduction that follows the split-KV decode of alpamayo_tt/expert.py,
// TTExpert.attention_core, where each KV head's keys are spread over several cores).
//
// For a split unit, CTA part s left a normalised partial O_s[128][128] (fp32) and, per folded
// row, lse_s = m_s + log2(l_s) in log2-scaled score units. The merged row is
//   M = max_s lse_s,   w_s = 2^(lse_s - M) / sum_t 2^(lse_t - M),   out = sum_s w_s O_s,
// written as bf16 to out[layer][2g + r/64][r%64][:] (folded row r of kv head g).
//
// One warp per folded row; lane j owns columns [4j, 4j+4). Parts are taken kBatch at a time
// (8, or 24 when a unit has more than 8 parts): every lane requests the batch's lse values
// (broadcast loads) together with its float4s, so a row costs one round trip to L2 per batch,
// and the running max and weight sum are carried across batches (a unit has at most as many
// parts as there are CTAs: a single layer spread over every SM has ~20, one batch of 24).
#include "internal.cuh"
#include "ptx.cuh"

namespace ea {

constexpr int kMergeWarps = 4;  // rows per CTA

template <int CAP, int kBatch>
__global__ void __launch_bounds__(kMergeWarps * 32) merge_kernel(const __grid_constant__ MergeParams<CAP> p) {
  // Launched programmatically after the attention kernel: let the next kernel in the stream set
  // up, then wait until every partial of the attention grid is written and visible.
  pdl_launch_dependents();
  pdl_wait_primary();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x / (kRows / kMergeWarps);
  const int r = (blockIdx.x % (kRows / kMergeWarps)) * kMergeWarps + warp;
  if (split >= p.n_split) return;
  const SplitUnit su = p.unit[split];
  const int u = su.u, c0 = su.c0, nparts = su.nparts;

  float M = -INFINITY, L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int q0 = 0; q0 < nparts; q0 += kBatch) {
    float lse[kBatch];
    float4 o[kBatch];
#pragma unroll
    for (int e = 0; e < kBatch; ++e) {
      if (q0 + e < nparts) {
        const int q = q0 + e;
        const size_t pr = (static_cast<size_t>(c0 + q) * 2 + (q == 0 ? su.slot0 : 0)) * kRows + r;
        lse[e] = __ldcg(p.part_lse + pr);
        o[e] = __ldcg(reinterpret_cast<const float4*>(p.part_o + pr * kD) + lane);
      } else {
        lse[e] = -INFINITY;
        o[e] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    float mb = lse[0];
#pragma unroll
    for (int e = 1; e < kBatch; ++e) mb = fmaxf(mb, lse[e]);
    const float Mn = fmaxf(M, mb);
    const float alpha = ex2_approx(M - Mn);  // 0 on the first batch (M = -inf)
    L *= alpha;
    acc.x *= alpha;
    acc.y *= alpha;
    acc.z *= alpha;
    acc.w *= alpha;
#pragma unroll
    for (int e = 0; e < kBatch; ++e) {
      const float w = ex2_approx(lse[e] - Mn);  // 0 for the padding entries
      L += w;
      acc.x = fmaf(w, o[e].x, acc.x);
      acc.y = fmaf(w, o[e].y, acc.y);
      acc.z = fmaf(w, o[e].z, acc.z);
      acc.w = fmaf(w, o[e].w, acc.w);
    }
    M = Mn;
  }
  const float invL = 1.0f / L;
  acc.x *= invL;
  acc.y *= invL;
  acc.z *= invL;
  acc.w *= invL;
  __nv_bfloat16* orow = p.out[u / kHkv] + (static_cast<size_t>(u % kHkv) * kRows + r) * kD;
  uint2 v;
  v.x = pack_bf16x2(acc.x, acc.y);
  v.y = pack_bf16x2(acc.z, acc.w);
  *reinterpret_cast<uint2*>(orow + 4 * lane) = v;
}

// Host-side launcher (the kernel template is instantiated and launched in this file).
template <int CAP>
cudaError_t launch_merge_kernel(const MergeParams<CAP>& mp, cudaLaunchConfig_t cfg) {
  cfg.gridDim = dim3(mp.n_split * (kRows / kMergeWarps));
  cfg.blockDim = dim3(kMergeWarps * 32);
  int max_parts = 0;
  for (int i = 0; i < mp.n_split; ++i) max_parts = mp.unit[i].nparts > max_parts ? mp.unit[i].nparts : max_parts;
  return max_parts <= 8 ? cudaLaunchKernelEx(&cfg, merge_kernel<CAP, 8>, mp)
                        : cudaLaunchKernelEx(&cfg, merge_kernel<CAP, 24>, mp);
}
template cudaError_t launch_merge_kernel<kSmallCap>(const MergeParams<kSmallCap>&, cudaLaunchConfig_t);
template cudaError_t launch_merge_kernel<kMaxLayersPerLaunch>(const MergeParams<kMaxLayersPerLaunch>&,
                                                               cudaLaunchConfig_t);

}  // namespace ea
