// merge.cu — K3: log-sum-exp merge of the split-KV partial outputs.
//
// The pages' flash-decode kernel splits each KV head's keys over ~16 cores and reduces the
// partial results (alpamayo_tt/expert.py, module docstring and TTExpert.attention_core;
// alpamayo_tt/EXPERT_NOTES.md, "Attention over the VLM cache: masking approach"). Here the key
// tiles of all (layer, kv head) units are cut into one contiguous range per attention CTA; a
// unit whose tiles fall into several ranges leaves one normalised fp32 partial O_s and one
// log2-sum-exp lse_s per range and row, and this kernel combines them:
//   M = max_s lse_s,  w_s = 2^(lse_s - M),  out = sum_s w_s O_s / sum_s w_s.
// Units covered by a single range were written by the attention kernel itself.
//
// One CTA per unit, one warp per row at a time; lane k holds segment k's weight, max and sum
// are warp-shuffle reductions, and the weights are broadcast by shuffle while every lane
// accumulates 4 of the 128 channels (float4 loads, coalesced).
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

}  // namespace

__global__ void __launch_bounds__(128) merge_kernel(const __grid_constant__ MergeParams p) {
  pdl_wait_primary();  // partials come from the attention kernel
  const int u = blockIdx.x;
  const long long first = static_cast<long long>(u) * p.T;
  const long long last = first + p.T - 1;
  const int c0 = cta_of_tile(first, p.W, p.n_ctas);
  const int c1 = cta_of_tile(last, p.W, p.n_ctas);
  if (c0 == c1) return;
  const int nseg = c1 - c0 + 1;
  const int l = u / kHkv, g = u % kHkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  for (int r = warp; r < kRows; r += 4) {
    // pass 1: max and sum of the weights (segments strided over the lanes)
    float M = -INFINITY;
    for (int k = lane; k < nseg; k += 32) {
      const int c = c0 + k;
      const int slot = cta_tile_start(c, p.W, p.n_ctas) >= first ? 0 : 1;
      M = fmaxf(M, p.part_lse[(static_cast<size_t>(c) * 2 + slot) * kRows + r]);
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, m));
    float Lsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int kc = 0; kc < nseg; kc += 32) {
      const int k = kc + lane;
      float wk = 0.f;
      if (k < nseg) {
        const int c = c0 + k;
        const int slot = cta_tile_start(c, p.W, p.n_ctas) >= first ? 0 : 1;
        wk = ex2_approx(p.part_lse[(static_cast<size_t>(c) * 2 + slot) * kRows + r] - M);
      }
      float ws = wk;
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, m);
      Lsum += ws;
      const int cnt = min(32, nseg - kc);
      for (int q = 0; q < cnt; ++q) {
        const float w = __shfl_sync(0xffffffffu, wk, q);
        const int c = c0 + kc + q;
        const int slot = cta_tile_start(c, p.W, p.n_ctas) >= first ? 0 : 1;
        const float4 o = *reinterpret_cast<const float4*>(
            p.part_o + ((static_cast<size_t>(c) * 2 + slot) * kRows + r) * kD + lane * 4);
        acc.x = fmaf(w, o.x, acc.x);
        acc.y = fmaf(w, o.y, acc.y);
        acc.z = fmaf(w, o.z, acc.z);
        acc.w = fmaf(w, o.w, acc.w);
      }
    }
    const float inv = 1.0f / Lsum;
    const uint32_t lo = pack_bf16x2(acc.x * inv, acc.y * inv);
    const uint32_t hi = pack_bf16x2(acc.z * inv, acc.w * inv);
    // folded row r of kv head g is output row g*128 + r = (q head 2g + r/64, token r%64)
    *reinterpret_cast<uint2*>(p.out[l] + (static_cast<size_t>(g) * kRows + r) * kD + lane * 4) =
        make_uint2(lo, hi);
  }
}

}  // namespace ea
