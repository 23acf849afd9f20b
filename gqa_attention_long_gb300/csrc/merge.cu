// merge.cu — K3: log-sum-exp merge of the split-KV partial outputs.
//
// The pages' flash-decode kernel splits each KV head's keys over ~16 cores and reduces the
// partial results (alpamayo_tt/expert.py, module docstring and TTExpert.attention_core;
// alpamayo_tt/EXPERT_NOTES.md, "Attention over the VLM cache: masking approach"). Here the key
// tiles of all (layer, kv head) units are cut into one contiguous range per attention CTA; a
// unit whose tiles fall into several ranges leaves one normalised fp32 partial O_s and one
// log2-sum-exp lse_s per range and row, and this kernel combines them:
//   M = max_s lse_s,  w_s = 2^(lse_s - M),  out = sum_s w_s O_s / sum_s w_s.
// Units covered by a single range were written by the attention kernel itself; the host passes
// the list of split units.
//
// Grid: (split units) x (128 / 8) CTAs of 8 warps; one warp per folded row. Lane k holds segment
// k's weight (max and sum are warp-shuffle reductions); the weights are broadcast by shuffle
// while every lane accumulates 4 of the 128 channels with float4 loads issued 4 segments at a
// time.
#include "internal.cuh"
#include "ptx.cuh"

namespace ea {

namespace {

__device__ __forceinline__ int cta_of_tile(long long x, long long W, int n) {
  int c = static_cast<int>((x * n) / W);
  while (c + 1 < n && cta_tile_start(c + 1, W, n) <= x) ++c;
  while (c > 0 && cta_tile_start(c, W, n) > x) --c;
  return c;
}

// Partial slot of CTA c for the unit starting at tile `first`: slot 0 if the unit's part is
// the CTA's first segment (the CTA starts inside or at the start of the unit), else slot 1.
__device__ __forceinline__ size_t part_index(int c, long long first, long long W, int n) {
  return static_cast<size_t>(c) * 2 + (cta_tile_start(c, W, n) >= first ? 0 : 1);
}

}  // namespace

__global__ void __launch_bounds__(32 * kMergeRowsPerCta) merge_kernel(const __grid_constant__ MergeParams p) {
  pdl_wait_primary();      // partials come from the attention kernel
  pdl_launch_dependents();  // the next prologue may start: nothing it writes is read here
  if (p.n_split == 0) return;
  const int u = p.split_unit[blockIdx.x / (kRows / kMergeRowsPerCta)];
  const int r = (blockIdx.x % (kRows / kMergeRowsPerCta)) * kMergeRowsPerCta + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const long long first = static_cast<long long>(u) * p.T;
  const int c0 = cta_of_tile(first, p.W, p.n_ctas);
  const int c1 = cta_of_tile(first + p.T - 1, p.W, p.n_ctas);
  const int nseg = c1 - c0 + 1;
  const int l = u / kHkv, g = u % kHkv;

  float M = -INFINITY;
  for (int k = lane; k < nseg; k += 32)
    M = fmaxf(M, p.part_lse[part_index(c0 + k, first, p.W, p.n_ctas) * kRows + r]);
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, m));

  float Lsum = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int kc = 0; kc < nseg; kc += 32) {
    const int k = kc + lane;
    const float wk = k < nseg
        ? ex2_approx(p.part_lse[part_index(c0 + k, first, p.W, p.n_ctas) * kRows + r] - M) : 0.f;
    float ws = wk;
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, m);
    Lsum += ws;
    const int cnt = min(32, nseg - kc);
    for (int q0 = 0; q0 < cnt; q0 += 4) {
      float4 o[4];
      float w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        w[q] = __shfl_sync(0xffffffffu, wk, (q0 + q) & 31);
        o[q] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (q0 + q < cnt)
          o[q] = *reinterpret_cast<const float4*>(
              p.part_o + (part_index(c0 + kc + q0 + q, first, p.W, p.n_ctas) * kRows + r) * kD + lane * 4);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (q0 + q < cnt) {
          acc.x = fmaf(w[q], o[q].x, acc.x);
          acc.y = fmaf(w[q], o[q].y, acc.y);
          acc.z = fmaf(w[q], o[q].z, acc.z);
          acc.w = fmaf(w[q], o[q].w, acc.w);
        }
      }
    }
  }
  const float inv = 1.0f / Lsum;
  // folded row r of kv head g is output row g*128 + r = (q head 2g + r/64, token r%64)
  *reinterpret_cast<uint2*>(p.out[l] + (static_cast<size_t>(g) * kRows + r) * kD + lane * 4) =
      make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
}

}  // namespace ea
