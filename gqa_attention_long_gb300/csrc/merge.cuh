// merge.cuh — log-sum-exp merge of the (layer, kv head) units that the attention kernel split
// across more than two CTAs (the reduction that follows the split-KV decode of
// alpamayo_tt/expert.py, TTExpert.attention_core, where each KV head's keys are spread over
// several cores). Run by the attention kernel itself once every CTA has written its partials.
//
// For a split unit, CTA part s left a normalised partial O_s[128][128] and, per folded row,
// lse_s = m_s + log2(l_s) in log2-scaled score units. The merged row is
//   M = max_s lse_s,   w_s = 2^(lse_s - M) / sum_t 2^(lse_t - M),   out = sum_s w_s O_s,
// written as bf16 to out[layer][2g + r/64][r%64][:] (folded row r of kv head g).
//
// Partials are f16, each half row (64 columns) stored times a power of two whose inverse sits
// beside the lse, and chunk-major (16-byte chunk c, columns 8c .. 8c+7, of row r at c * 128 + r).
// One thread merges one row's chunk c (8 output columns); the 128 threads of a group take the
// 128 rows of one chunk, so that every load instruction of a warp reads 512 contiguous bytes.
// Parts are taken kBatch at a time, each thread requesting a batch's lse values, scales and
// chunks together (indices past the last part are clamped to it and weighted 0), so that a row
// costs one round trip to L2 per batch; the running max and weight sum are carried across
// batches (a single layer spread over every SM has ~20 parts per unit, one batch of 20).
#pragma once

#include "internal.cuh"
#include "ptx.cuh"

namespace ea {

template <int kBatch>
__device__ __forceinline__ void merge_row_chunk(const uint4* part_o, const float* part_lse,
                                                const SplitUnit& su, int c, int r,
                                                __nv_bfloat16* out_layer) {
  const int u = su.u, nparts = su.nparts;
  float M = -INFINITY, L = 0.f;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  for (int q0 = 0; q0 < nparts; q0 += kBatch) {
    float lse[kBatch], isc[kBatch];
    uint4 o[kBatch];
#pragma unroll
    for (int e = 0; e < kBatch; ++e) {
      const int q = min(q0 + e, nparts - 1);
      // part q's slot: 2 (c0 + q), except the first part's, which is 2 c0 + slot0
      const size_t sl = static_cast<size_t>(su.c0 + q) * 2 + (q == 0 ? su.slot0 : 0);
      lse[e] = __ldcg(part_lse + sl * 3 * kRows + r);
      isc[e] = __ldcg(part_lse + (sl * 3 + 1 + (c >> 3)) * kRows + r);
      o[e] = __ldcg(part_o + (sl * kPartChunks + c) * kRows + r);
    }
#pragma unroll
    for (int e = 0; e < kBatch; ++e)
      if (q0 + e >= nparts) lse[e] = -INFINITY;  // padding: weight 0
    float mb = lse[0];
#pragma unroll
    for (int e = 1; e < kBatch; ++e) mb = fmaxf(mb, lse[e]);
    const float Mn = fmaxf(M, mb);
    const float alpha = ex2_approx(M - Mn);  // 0 on the first batch (M = -inf)
    L *= alpha;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] *= alpha;
#pragma unroll
    for (int e = 0; e < kBatch; ++e) {
      const float w = ex2_approx(lse[e] - Mn);
      L += w;
      const float ws = w * isc[e];
      const uint32_t wv[4] = {o[e].x, o[e].y, o[e].z, o[e].w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const float2 f = unpack_f16x2(wv[h]);
        acc[2 * h] = fmaf(ws, f.x, acc[2 * h]);
        acc[2 * h + 1] = fmaf(ws, f.y, acc[2 * h + 1]);
      }
    }
    M = Mn;
  }
  const float invL = 1.0f / L;
  // folded row r of kv head g is row r % 64 of q head 2g + r / 64
  __nv_bfloat16* orow = out_layer + (static_cast<size_t>(u % kHkv) * kRows + r) * kD + 8 * c;
  uint4 v;
  v.x = pack_bf16x2(acc[0] * invL, acc[1] * invL);
  v.y = pack_bf16x2(acc[2] * invL, acc[3] * invL);
  v.z = pack_bf16x2(acc[4] * invL, acc[5] * invL);
  v.w = pack_bf16x2(acc[6] * invL, acc[7] * invL);
  *reinterpret_cast<uint4*>(orow) = v;
}

}  // namespace ea
