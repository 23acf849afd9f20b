// prologue.cu — K1: fused per-head RMSNorm + HF rotate_half RoPE of the 64 expert tokens and
// the own-row write into the cache tail; for an e4m3 cache also the staging of the roped Q (high
// and low codes, per-row scale) in the workspace in the shared-memory layout the attention
// kernel consumes. With a bf16 cache the attention kernel does this work itself; this kernel
// then serves only the stand-alone prologue entry point (cache tail and optional roped q).
//
// alpamayo_tt/expert.py, TTExpert.layer (rms_norm of q and k with the q_norm / k_norm gains,
// rotary_embedding_hf, typecast to the cache dtype, fill_cache at row Smax-64) and
// TTExpert.set_context (positions i + rope_delta + S); alpamayo_tt/EXPERT_NOTES.md, "Layouts".
//
// An octet (8 lanes) owns one token at a time; lane i holds channels [8i, 8i+8) and their RoPE
// partners [64+8i, 64+8i+8), so the rotation is in-thread and the norm needs three shuffles.
// Every global access is a 16-byte vector access.
// Persistent CTAs (one per SM) walk a range of (layer, g) units (q heads 2g, 2g+1, k head g,
// v head g; all 64 tokens: bf16, 256 threads, two tokens per octet; e4m3, 512 threads, one),
// computing the tokens' cos/sin once (positions are the same in every layer and head); the raw
// rows arrive by bulk copy into a shared-memory ring several units ahead. With an e4m3 cache the
// own K and V rows of a head share one scale over all 64 tokens, a CTA-wide maximum.
#include <cuda_fp8.h>

#include "internal.cuh"
#include "ptx.cuh"
#include "rope.cuh"

namespace ea {

namespace {

__device__ __forceinline__ void load_bf16x8(const __nv_bfloat16* src, float (&x)[8]) {
  unpack_bf16x8(*reinterpret_cast<const uint4*>(src), x);
}

// Maximum over the CTA's NW warps (two CTA barriers).
template <int NW>
__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < NW; ++w) r = fmaxf(r, red[w]);
  return r;
}

// Byte offset of the 8 e4m3 values of channels [8k, 8k+8) (k < 16) of row r in an e4m3 tile
// with one 128-byte swizzle atom per row: 16-byte chunk k/2, half k%2, chunk' = chunk ^ (r % 8).
__device__ __forceinline__ uint32_t swz8_off(int r, int k) {
  return static_cast<uint32_t>(r) * 128u + (static_cast<uint32_t>((k >> 1) ^ (r & 7)) << 4) +
         static_cast<uint32_t>(k & 1) * 8u;
}

// 8 fp32 values * inv_scale -> a high and a low set of 8 e4m3 codes with the same scale:
// hi = e4m3(y / s), lo = e4m3(y / s - value(hi)). hi + lo carries about twice the mantissa bits
// of one e4m3 code, and both can feed MMAs that accumulate into the same result.
__device__ __forceinline__ void quant8_hilo(const float (&y)[8], float inv_scale, uint2& hi,
                                            uint2& lo) {
  uint32_t ch[4], cl[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float a = y[2 * e] * inv_scale, b = y[2 * e + 1] * inv_scale;
    const __nv_fp8x2_storage_t h = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    const float2 hv = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(h, __NV_E4M3)));
    ch[e] = h;
    cl[e] = __nv_cvt_float2_to_fp8x2(make_float2(a - hv.x, b - hv.y), __NV_SATFINITE, __NV_E4M3);
  }
  hi = make_uint2(ch[0] | (ch[1] << 16), ch[2] | (ch[3] << 16));
  lo = make_uint2(cl[0] | (cl[1] << 16), cl[2] | (cl[3] << 16));
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

// Persistent CTAs walk a contiguous range of (layer, g) units. The
// raw rows of a unit (q heads 2g and 2g+1: 32 KB, k head g: 16 KB, v head g: 16 KB, each one
// contiguous block) arrive by bulk copy in a three-slot shared-memory ring, so that up to
// 192 KB of loads per SM are in flight while the threads work on an earlier unit.
constexpr int kPRing = 3;
constexpr uint32_t kPUnitBytes = 65536;
constexpr uint32_t kPBarOff = kPRing * kPUnitBytes;
constexpr uint32_t kPSmemBytes = kPBarOff + 8 * kPRing + 16;

// bf16: TPO = 2 (tokens per octet): grid min(number of SMs, units), block 256 = 32 octets, each
// owning tokens oc and oc + 32 of every unit in the CTA's range. TPO = 1 (few units): two CTAs
// per unit, each owning 32 tokens, one per octet; the per-thread work halves.
// F8: the e4m3 cache variant (Q as high and low codes with a per-row scale; the own K and V rows
// quantised with one scale per head over all 64 tokens: CTA-wide maxima). Its CTAs have 512
// threads, 64 octets, one token each, over a range of units (TPO = 2 in the range sense): twice
// the warps of the bf16 block to hide the latencies of its longer per-token chain.
template <bool F8, int CAP, int TPO>
__global__ void __launch_bounds__(F8 ? 512 : 256, 1) prologue_ring_kernel(const __grid_constant__ PrologueParams<CAP> p) {
  static_assert(TPO == 2 || !F8, "the e4m3 own-row scale needs all 64 tokens in one CTA");
  constexpr int kNT = F8 ? 512 : 256;     // threads
  constexpr int kTpt = F8 ? 1 : TPO;      // tokens per octet and unit
  constexpr int kTpc = F8 ? 64 : 32 * TPO;  // tokens per CTA and unit
  __shared__ float red[kNT / 32];
  extern __shared__ __align__(128) uint8_t psm[];
  const uint32_t sbase = smem_u32(psm);
  const uint32_t bar0 = sbase + kPBarOff;
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(psm + kPBarOff + 8 * kPRing);
  const int n_units = p.n_layers * kHkv;
  const int u0 = TPO == 2 ? static_cast<int>(static_cast<long long>(blockIdx.x) * n_units / gridDim.x)
                          : static_cast<int>(blockIdx.x >> 1);
  const int u1 = TPO == 2 ? static_cast<int>(static_cast<long long>(blockIdx.x + 1) * n_units / gridDim.x)
                          : u0 + 1;
  const int t0 = TPO == 2 ? 0 : 32 * static_cast<int>(blockIdx.x & 1);  // first token of the CTA
  const int oc = threadIdx.x >> 3;  // octet: tokens oc (and oc + 32 if kTpt = 2)
  const int i = threadIdx.x & 7;    // channels [8i, 8i+8) and [64+8i, 64+8i+8)
  const int dl = 8 * i, dh = 64 + 8 * i;
  const int Smax = p.Smax;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kPRing; ++s) mbar_init(bar0 + 8 * s, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  __syncthreads();
  // Launched programmatically after the previous kernel in the stream: wait for it (it may have
  // produced q/k/v, or still read the workspace), then let the attention kernel's CTAs start
  // their set-up; they wait for this grid before reading anything written here.
  pdl_wait_primary();
  pdl_launch_dependents();
  if (t0 == 0)
    for (int x = threadIdx.x; x < 2 * (u1 - u0); x += kNT) p.unit_sync[2 * u0 + x] = 0u;

  const uint64_t pol = l2_policy_evict_first();  // raw rows are read once
  // slot layout: q head 2g rows, q head 2g+1 rows, k rows, v rows (kTpc rows of 256 B each)
  constexpr uint32_t kRowsB = kTpc * kD * 2;
  auto issue = [&](int k) {  // one thread: bulk loads of unit u0 + k into slot k % kPRing
    const int u = u0 + k, g = u % kHkv;
    const PrologueLayer& L = p.layer[u / kHkv];
    const uint32_t dst = sbase + (k % kPRing) * kPUnitBytes, bar = bar0 + 8 * (k % kPRing);
    mbar_expect_tx(bar, 4 * kRowsB);
    if (TPO == 2) {  // both q heads are one contiguous block
      bulk_load(dst, L.q_raw + static_cast<size_t>(2 * g) * kTok * kD, 2 * kRowsB, bar, pol);
    } else {
      bulk_load(dst, L.q_raw + (static_cast<size_t>(2 * g) * kTok + t0) * kD, kRowsB, bar, pol);
      bulk_load(dst + kRowsB, L.q_raw + (static_cast<size_t>(2 * g + 1) * kTok + t0) * kD, kRowsB, bar, pol);
    }
    bulk_load(dst + 2 * kRowsB, L.k_raw + (static_cast<size_t>(g) * kTok + t0) * kD, kRowsB, bar, pol);
    bulk_load(dst + 3 * kRowsB, L.v_raw + (static_cast<size_t>(g) * kTok + t0) * kD, kRowsB, bar, pol);
  };
  int issued = 0;
  if (threadIdx.x == 0)
    for (; issued < kPRing && u0 + issued < u1; ++issued) issue(issued);

  // cos/sin of this thread's tokens at its eight frequencies (the same in every unit)
  float cs[kTpt][8], sn[kTpt][8];
  float ih[8], il[8];
  load_inv8(p.inv_hi, p.inv_lo, dl, ih, il);
#pragma unroll
  for (int tt = 0; tt < kTpt; ++tt) {
    const int pos = t0 + oc + 32 * tt + p.rope_delta + p.S;
#pragma unroll
    for (int e = 0; e < 8; ++e) rope_cos_sin(pos, ih[e], il[e], cs[tt][e], sn[tt][e]);
  }

  float gql[8], gqh[8], gkl[8], gkh[8];
  int cur_l = -1;
  bool ok = true;
  int k = 0;
  for (; u0 + k < u1; ++k) {
    const int u = u0 + k, l = u / kHkv, g = u % kHkv;
    ok = __syncthreads_and(bounded_wait(bar0 + 8 * (k % kPRing), (k / kPRing) & 1, abort_flag, p.status,
                                        kErrPrologueWait)) != 0;
    if (!ok) break;
    const PrologueLayer& L = p.layer[l];
    if (l != cur_l) {
      load_bf16x8(L.q_gamma + dl, gql);
      load_bf16x8(L.q_gamma + dh, gqh);
      load_bf16x8(L.k_gamma + dl, gkl);
      load_bf16x8(L.k_gamma + dh, gkh);
      cur_l = l;
    }
    uint8_t* const slot = psm + (k % kPRing) * kPUnitBytes;
    const uint8_t* src = slot;
    if constexpr (F8) {
      // e4m3 cache. The unit's outputs are staged in its own ring slot, over raw rows every
      // thread has already read, and leave by three bulk stores: the Q codes (high then low,
      // 32 KB in the attention kernel's shared-memory layout) over the raw q rows, the own K
      // and V rows' codes (8 KB each, cache-row layout) over the raw k rows.
      const int ncol = Smax / kScaleBlock + 1;
      const int n_main = (p.S + kKeyTile - 1) / kKeyTile;
      // the unit's cache-block V scales, requested now and used after the own rows' maximum
      float vpre = 0.f;
      for (int b = threadIdx.x; b < n_main; b += kNT) vpre = fmaxf(vpre, L.v_scale[g * ncol + b]);
      uint4 rq[kTpt][2][2];  // raw q: token oc + 32 tt, head 2g + hh, channels [8i..), [64+8i..)
#pragma unroll
      for (int tt = 0; tt < kTpt; ++tt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const uint8_t* row = src + (hh * kTok + oc + 32 * tt) * (kD * 2);
          rq[tt][hh][0] = *reinterpret_cast<const uint4*>(row + dl * 2);
          rq[tt][hh][1] = *reinterpret_cast<const uint4*>(row + dh * 2);
        }
      float krl[kTpt][8], krh[kTpt][8];  // roped k, kept for the head's scale
      uint4 rv[kTpt][2];                 // raw v (bf16), likewise
      float kmax = 0.f, vmax = 0.f;
#pragma unroll
      for (int tt = 0; tt < kTpt; ++tt) {
        const int t = oc + 32 * tt;
        const uint8_t* krow = src + 2 * kRowsB + t * (kD * 2);
        const uint8_t* vrow = src + 3 * kRowsB + t * (kD * 2);
        float xl[8], xh[8];
        unpack_bf16x8(*reinterpret_cast<const uint4*>(krow + dl * 2), xl);
        unpack_bf16x8(*reinterpret_cast<const uint4*>(krow + dh * 2), xh);
        norm_rope(xl, xh, gkl, gkh, cs[tt], sn[tt], krl[tt], krh[tt]);
        rv[tt][0] = *reinterpret_cast<const uint4*>(vrow + dl * 2);
        rv[tt][1] = *reinterpret_cast<const uint4*>(vrow + dh * 2);
        float vl[8], vh[8];
        unpack_bf16x8(rv[tt][0], vl);
        unpack_bf16x8(rv[tt][1], vh);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          kmax = fmaxf(kmax, fmaxf(fabsf(krl[tt][e]), fabsf(krh[tt][e])));
          vmax = fmaxf(vmax, fmaxf(fabsf(vl[e]), fabsf(vh[e])));
        }
      }
      // every raw row of the slot is in registers once the CTA-wide maxima are formed (each
      // block_max passes two CTA barriers)
      kmax = block_max<kNT / 32>(kmax, red);
      vmax = block_max<kNT / 32>(vmax, red);
#pragma unroll
      for (int tt = 0; tt < kTpt; ++tt) {
        const int t = oc + 32 * tt;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float xl[8], xh[8], yl[8], yh[8];
          unpack_bf16x8(rq[tt][hh][0], xl);
          unpack_bf16x8(rq[tt][hh][1], xh);
          norm_rope(xl, xh, gql, gqh, cs[tt], sn[tt], yl, yh);
          const int r = hh * kTok + t;
          // the row as two sets of e4m3 codes (high, low) with one scale amax / 448
          float am = 0.f;
#pragma unroll
          for (int e = 0; e < 8; ++e) am = fmaxf(am, fmaxf(fabsf(yl[e]), fabsf(yh[e])));
#pragma unroll
          for (int m = 4; m >= 1; m >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, m));
          const float sq = am > 0.f ? am * (1.0f / 448.0f) : 1.0f;
          const float isq = am > 0.f ? 448.0f / am : 1.0f;
          uint2 hi, lo;  // high codes in the first 16 KB of the staged tile, low codes in the second
          quant8_hilo(yl, isq, hi, lo);
          *reinterpret_cast<uint2*>(slot + swz8_off(r, i)) = hi;
          *reinterpret_cast<uint2*>(slot + kQTileBytesF8 + swz8_off(r, i)) = lo;
          quant8_hilo(yh, isq, hi, lo);
          *reinterpret_cast<uint2*>(slot + swz8_off(r, i + 8)) = hi;
          *reinterpret_cast<uint2*>(slot + kQTileBytesF8 + swz8_off(r, i + 8)) = lo;
          if (i == 0) p.q_scale[static_cast<size_t>(u) * kRows + r] = sq;
          if (L.q_rope != nullptr) {
            __nv_bfloat16* qr = L.q_rope + (static_cast<size_t>(2 * g + hh) * kTok + t) * kD;
            *reinterpret_cast<uint4*>(qr + dl) = pack8(yl, false);
            *reinterpret_cast<uint4*>(qr + dh) = pack8(yh, false);
          }
        }
      }
      // the 64 own rows of this head share one scale slot, column Smax/128; the unit's
      // reference V scale is the largest over the cache blocks it reads and its own rows
      const float ksc = kmax > 0.f ? __fdiv_rn(kmax, 448.0f) : 1.0f;
      const float vsc = vmax > 0.f ? __fdiv_rn(vmax, 448.0f) : 1.0f;
      const float vr = block_max<kNT / 32>(fmaxf(vsc, vpre), red);
      if (threadIdx.x == 0) {
        L.k_scale[g * ncol + ncol - 1] = ksc;
        L.v_scale[g * ncol + ncol - 1] = vsc;
        p.sv_ref[u] = vr;
      }
      uint8_t* kst = slot + 2 * kRowsB;  // own K codes, then own V codes: row t at t * 128
      uint8_t* vst = kst + kTok * kD;
#pragma unroll
      for (int tt = 0; tt < kTpt; ++tt) {
        const int t = oc + 32 * tt;
        uint2 c;
        uint4 w;
        quant8(krl[tt], ksc, c, w);
        *reinterpret_cast<uint2*>(kst + t * kD + dl) = c;
        quant8(krh[tt], ksc, c, w);
        *reinterpret_cast<uint2*>(kst + t * kD + dh) = c;
        float vv[8];
        unpack_bf16x8(rv[tt][0], vv);
        quant8(vv, vsc, c, w);
        *reinterpret_cast<uint2*>(vst + t * kD + dl) = c;
        unpack_bf16x8(rv[tt][1], vv);
        quant8(vv, vsc, c, w);
        *reinterpret_cast<uint2*>(vst + t * kD + dh) = c;
      }
      fence_proxy_async_smem();  // the staged codes are read by the bulk stores (async proxy)
      __syncthreads();
      if (threadIdx.x == 0) {
        const size_t crow = static_cast<size_t>(g) * Smax + (Smax - kTok);
        bulk_store(p.q_ws + static_cast<size_t>(u) * kQTileBytes, smem_u32(slot), kQTileBytes);
        bulk_store(static_cast<uint8_t*>(L.k_cache) + crow * kD, smem_u32(kst), kTok * kD);
        bulk_store(static_cast<uint8_t*>(L.v_cache) + crow * kD, smem_u32(vst), kTok * kD);
        bulk_commit();
        if (u0 + issued < u1) {
          bulk_wait_read0();  // the stores have read the slot before it is refilled
          issue(issued);
          ++issued;
        }
      }
    } else {
      float krl[TPO][8], krh[TPO][8];
#pragma unroll
      for (int tt = 0; tt < TPO; ++tt) {
        const int tl = oc + 32 * tt, t = t0 + tl;  // token within the CTA's block, within the unit
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const uint8_t* row = src + (hh * kTpc + tl) * (kD * 2);
          float xl[8], xh[8], yl[8], yh[8];
          unpack_bf16x8(*reinterpret_cast<const uint4*>(row + dl * 2), xl);
          unpack_bf16x8(*reinterpret_cast<const uint4*>(row + dh * 2), xh);
          norm_rope(xl, xh, gql, gqh, cs[tt], sn[tt], yl, yh);
          const uint4 ql = pack8(yl, false), qh = pack8(yh, false);
          if (L.q_rope != nullptr) {
            __nv_bfloat16* qr = L.q_rope + (static_cast<size_t>(2 * g + hh) * kTok + t) * kD;
            *reinterpret_cast<uint4*>(qr + dl) = ql;
            *reinterpret_cast<uint4*>(qr + dh) = qh;
          }
        }
        const uint8_t* krow = src + 2 * kRowsB + tl * (kD * 2);
        const uint8_t* vrow = src + 3 * kRowsB + tl * (kD * 2);
        float xl[8], xh[8];
        unpack_bf16x8(*reinterpret_cast<const uint4*>(krow + dl * 2), xl);
        unpack_bf16x8(*reinterpret_cast<const uint4*>(krow + dh * 2), xh);
        norm_rope(xl, xh, gkl, gkh, cs[tt], sn[tt], krl[tt], krh[tt]);
        const uint4 vpl = *reinterpret_cast<const uint4*>(vrow + dl * 2);
        const uint4 vph = *reinterpret_cast<const uint4*>(vrow + dh * 2);
        const uint4 kpl = pack8(krl[tt], false), kph = pack8(krh[tt], false);
        const size_t crow = static_cast<size_t>(g) * Smax + (Smax - kTok) + t;
        __nv_bfloat16* kc = static_cast<__nv_bfloat16*>(L.k_cache) + crow * kD;
        __nv_bfloat16* vc = static_cast<__nv_bfloat16*>(L.v_cache) + crow * kD;
        *reinterpret_cast<uint4*>(kc + dl) = kpl;
        *reinterpret_cast<uint4*>(kc + dh) = kph;
        *reinterpret_cast<uint4*>(vc + dl) = vpl;
        *reinterpret_cast<uint4*>(vc + dh) = vph;
      }
      __syncthreads();  // every thread is done with the slot
      if (threadIdx.x == 0 && u0 + issued < u1) {
        fence_proxy_async_smem();  // generic-proxy reads of the slot before the async-proxy refill
        issue(issued);
        ++issued;
      }
    }
  }
  if constexpr (F8)
    if (threadIdx.x == 0) bulk_wait_all0();  // the staged outputs have left shared memory
  if (!ok && threadIdx.x == 0) {
    // let the copies already issued land before the CTA gives its shared memory back
    for (int kk = k; kk < issued; ++kk)
      if (!drain_wait(bar0 + 8 * (kk % kPRing), (kk / kPRing) & 1)) atomicOr(p.status, kErrDrain);
  }
}

template <int CAP>
cudaError_t launch_prologue_kernel(const PrologueParams<CAP>& pp, bool fp8, int sm_count,
                                   cudaLaunchConfig_t cfg) {
  const int n_units = pp.n_layers * kHkv;
  cfg.blockDim = dim3(fp8 ? 512 : 256);
  cfg.dynamicSmemBytes = kPSmemBytes;
  if (fp8) {
    cfg.gridDim = dim3(n_units < sm_count ? n_units : sm_count);
    return cudaLaunchKernelEx(&cfg, prologue_ring_kernel<true, CAP, 2>, pp);
  }
  if (2 * n_units <= sm_count) {  // few units: two CTAs per unit, half the tokens each
    cfg.gridDim = dim3(2 * n_units);
    return cudaLaunchKernelEx(&cfg, prologue_ring_kernel<false, CAP, 1>, pp);
  }
  cfg.gridDim = dim3(n_units < sm_count ? n_units : sm_count);
  return cudaLaunchKernelEx(&cfg, prologue_ring_kernel<false, CAP, 2>, pp);
}

template <bool F8, int CAP, int TPO>
static cudaError_t prologue_smem_attr() {
  return cudaFuncSetAttribute(prologue_ring_kernel<F8, CAP, TPO>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmemBytes);
}

cudaError_t prologue_set_attributes() {
  cudaError_t e = prologue_smem_attr<false, kSmallCap, 2>();
  if (e == cudaSuccess) e = prologue_smem_attr<false, kSmallCap, 1>();
  if (e == cudaSuccess) e = prologue_smem_attr<true, kSmallCap, 2>();
  if (e == cudaSuccess) e = prologue_smem_attr<false, kMaxLayersPerLaunch, 2>();
  if (e == cudaSuccess) e = prologue_smem_attr<false, kMaxLayersPerLaunch, 1>();
  if (e == cudaSuccess) e = prologue_smem_attr<true, kMaxLayersPerLaunch, 2>();
  return e;
}

template cudaError_t launch_prologue_kernel<kSmallCap>(const PrologueParams<kSmallCap>&, bool, int,
                                                       cudaLaunchConfig_t);
template cudaError_t launch_prologue_kernel<kMaxLayersPerLaunch>(
    const PrologueParams<kMaxLayersPerLaunch>&, bool, int, cudaLaunchConfig_t);

}  // namespace ea
