// attention.cu — K2: persistent split-KV expert attention on the sm_103a tensor cores (bf16 cache).
//
// What it computes (alpamayo_tt/expert.py, TTExpert.attention_core; alpamayo_tt/EXPERT_NOTES.md,
// "Attention over the VLM cache: masking approach"): for every (layer, kv head g) unit, the 128
// folded query rows (q heads 2g and 2g+1 x 64 tokens, pre-roped by the prologue) attend to cache
// rows [0, S) and to the 64 own rows, softmax(Q K^T / sqrt(128)) V. Hidden rows [S, Smax-64) are
// never read; the mask is derived from row indices.
//
// Work decomposition: the key tiles of all units (ceil(S/128) tiles of 128 cache rows, then one
// 64-row tile of own rows) are laid out unit-major and cut into one contiguous range per CTA
// (grid = number of SMs, one CTA per SM). A CTA walks its range as "segments" (the part of one
// unit inside the range). A segment that covers a whole unit writes the bf16 output directly;
// a partial one writes a normalised fp32 partial plus its log2-sum-exp for the merge kernel.
//
// Warp roles (192 threads):
//   warps 0-3  softmax: thread r owns folded row r (= TMEM lane r); online softmax in fp32 with
//              lazy rescaling of the TMEM accumulator, P written to shared memory as bf16
//   warp 4     producer: one thread issues bulk copies (roped Q, own rows, both pre-swizzled in
//              the workspace) and 3-D TMA loads of cache K/V tiles into a 4-slot ring
//   warp 5     MMA: one thread issues tcgen05.mma (S = Q K^T into one of two TMEM score buffers,
//              O += P V into the TMEM accumulator) and tcgen05.commit to the barriers
// Shared memory: Q x2 (64 KB), P (32 KB), K/V ring 4 x 32 KB, barriers. TMEM: 512 columns
// (two 128-column score buffers and one 128-column fp32 accumulator).
#include "internal.cuh"
#include "ptx.cuh"

namespace ea {
namespace attn {

constexpr int kThreads = 192;
constexpr int kRing = 4;
constexpr uint32_t kSlotBytes = 32768;  // one K or V tile: 128 rows x 256 bytes, two 16 KB atoms
constexpr uint32_t kAtom = kSlotBytes / 2;
constexpr uint32_t SM_Q = 0;
constexpr uint32_t SM_P = 2 * kQTileBytes;
constexpr uint32_t SM_RING = SM_P + kQTileBytes;
constexpr uint32_t SM_BAR = SM_RING + kRing * kSlotBytes;
enum : int {
  B_QFULL = 0, B_QEMPTY = 2, B_KVFULL = 4, B_KVEMPTY = 4 + kRing, B_SFULL = 4 + 2 * kRing,
  B_PFULL = B_SFULL + 2, B_ODONE = B_PFULL + 1, B_DRAIN = B_ODONE + 1, kNumBars = B_DRAIN + 1
};
constexpr uint32_t SM_TMEM = SM_BAR + kNumBars * 8;
constexpr uint32_t SM_ABORT = SM_TMEM + 4;
constexpr uint32_t kSmemBytes = SM_ABORT + 4 + 1024;  // + slack to align the base to 1024 bytes
static_assert(kSmemBytes <= 232448, "shared memory budget of one sm_103 CTA");

constexpr uint32_t TM_S = 0;    // score buffers at columns 0 and 128
constexpr uint32_t TM_O = 256;  // output accumulator, columns 256..383
constexpr uint32_t kTmemCols = 512;

struct Seg {
  int u, j0, j1;  // unit and its key-tile range [j0, j1)
};

__device__ __forceinline__ bool next_seg(long long& t, long long end, int T, Seg& s) {
  if (t >= end) return false;
  s.u = static_cast<int>(t / T);
  s.j0 = static_cast<int>(t - static_cast<long long>(s.u) * T);
  const long long j1 = s.j0 + (end - t);
  s.j1 = static_cast<int>(j1 < T ? j1 : T);
  t += s.j1 - s.j0;
  return true;
}

struct Ctx {
  uint32_t sbase;
  uint32_t tmem;
  volatile uint32_t* abort_flag;
  uint32_t* status;
  long long start, end;
  __device__ __forceinline__ uint32_t bar(int i) const { return sbase + SM_BAR + 8u * i; }
};

// ------------------------------------------------------------------------------- producer
__device__ __noinline__ void producer(const AttnParams& p, const Ctx& cx) {
  pdl_wait_primary();  // roped Q and own rows are written by the prologue kernel
  const uint64_t pol_stream = l2_policy_evict_first();  // cache tiles are read exactly once
  const uint64_t pol_keep = l2_policy_evict_last();
  uint32_t ring = 0;
  int seg = 0, q_loads = 0;
  bool ok = true;
  long long t = cx.start;
  Seg s;
  while (ok && next_seg(t, cx.end, p.T, s)) {
    const int l = s.u / kHkv, g = s.u % kHkv;
    const int qb = seg & 1;
    if (seg >= 2)
      ok = bounded_wait(cx.bar(B_QEMPTY + qb), ((seg >> 1) - 1) & 1, cx.abort_flag, cx.status,
                        kErrProducerWait);
    if (!ok) break;
    mbar_expect_tx(cx.bar(B_QFULL + qb), kQTileBytes);
    bulk_load(cx.sbase + SM_Q + qb * kQTileBytes, p.q_ws + static_cast<size_t>(s.u) * kQTileBytes,
              kQTileBytes, cx.bar(B_QFULL + qb), pol_keep);
    ++q_loads;
    for (int j = s.j0; j < s.j1 && ok; ++j) {
      for (int h = 0; h < 2; ++h) {  // h = 0: K tile, h = 1: V tile
        const uint32_t slot = ring % kRing, round = ring / kRing;
        if (round > 0) {
          ok = bounded_wait(cx.bar(B_KVEMPTY + slot), (round - 1) & 1, cx.abort_flag, cx.status,
                            kErrProducerWait);
          if (!ok) break;
        }
        const uint32_t dst = cx.sbase + SM_RING + slot * kSlotBytes;
        const uint32_t fb = cx.bar(B_KVFULL + slot);
        if (j < p.n_main) {
          // rows [128 j, 128 j + 128) of head g; rows >= S lie outside the map and arrive as 0
          mbar_expect_tx(fb, kSlotBytes);
          const CUtensorMap* m = h ? &p.vmap[l] : &p.kmap[l];
          tma_load_3d(dst, m, fb, 0, j * kKeyTile, g, pol_stream);
          tma_load_3d(dst + kAtom, m, fb, 64, j * kKeyTile, g, pol_stream);
        } else {
          // the 64 own rows, staged pre-swizzled by the prologue: two 8 KB atoms
          mbar_expect_tx(fb, kTailHalfBytes);
          const uint8_t* src =
              p.tail_ws + static_cast<size_t>(s.u) * kTailUnitBytes + h * kTailHalfBytes;
          bulk_load(dst, src, kTailHalfBytes / 2, fb, pol_keep);
          bulk_load(dst + kAtom, src + kTailHalfBytes / 2, kTailHalfBytes / 2, fb, pol_keep);
        }
        ++ring;
      }
    }
    ++seg;
  }
  pdl_launch_dependents();
  if (!ok) {
    // Let every copy already issued land before the CTA gives its shared memory back.
    for (uint32_t k = 0; k < static_cast<uint32_t>(kRing) && k < ring; ++k) {
      const uint32_t pos = ring - 1 - k;
      if (!drain_wait(cx.bar(B_KVFULL + pos % kRing), (pos / kRing) & 1)) atomicOr(cx.status, kErrDrain);
    }
    for (int b = 0; b < 2; ++b) {
      int last = q_loads - 1;  // last segment whose Q went into buffer b
      if ((last & 1) != b) --last;
      if (last >= 0 && !drain_wait(cx.bar(B_QFULL + b), (last >> 1) & 1))
        atomicOr(cx.status, kErrDrain);
    }
  }
}

// ------------------------------------------------------------------------------------ MMA
// Issue order per segment: QK(0), then for i >= 1: QK(i), PV(i-1); finally PV(nt-1). So QK(i+1)
// is issued only after PV(i-1), whose P came from the softmax of tile i-1: by then the score
// buffer that QK(i+1) overwrites has been read, and every completed S(i) implies PV(i-2) done.
__device__ __noinline__ void mma_issuer(const AttnParams& p, const Ctx& cx) {
  constexpr uint32_t kIdescQK128 = umma_idesc_f16(128, 128, true, false, false);
  constexpr uint32_t kIdescQK64 = umma_idesc_f16(128, 64, true, false, false);
  constexpr uint32_t kIdescPV = umma_idesc_f16(128, 128, true, false, true);  // V is MN-major
  uint32_t ring = 0, n_qk = 0, n_pv = 0;
  int seg = 0;
  bool ok = true;
  long long t = cx.start;
  Seg s;
  while (ok && next_seg(t, cx.end, p.T, s)) {
    const int qb = seg & 1;
    ok = bounded_wait(cx.bar(B_QFULL + qb), (seg >> 1) & 1, cx.abort_flag, cx.status, kErrMmaWait);
    if (!ok) break;
    tc_fence_after();
    const uint32_t qaddr = cx.sbase + SM_Q + qb * kQTileBytes;
    const int nt = s.j1 - s.j0;
    for (int i = 0; i <= nt && ok; ++i) {
      if (i < nt) {
        const int j = s.j0 + i;
        const uint32_t pos = ring + 2 * i, slot = pos % kRing;
        ok = bounded_wait(cx.bar(B_KVFULL + slot), (pos / kRing) & 1, cx.abort_flag, cx.status,
                          kErrMmaWait);
        if (!ok) break;
        tc_fence_after();
        const uint32_t kaddr = cx.sbase + SM_RING + slot * kSlotBytes;
        const uint32_t d = cx.tmem + TM_S + (n_qk & 1) * 128;
        const uint32_t idesc = j < p.n_main ? kIdescQK128 : kIdescQK64;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {  // 8 steps of 16 channels; 4 per 64-channel atom
          const uint32_t off = (kk >> 2) * kAtom + (kk & 3) * 32;
          umma_f16_ss(d, sw128_desc(qaddr + off, 16, 1024), sw128_desc(kaddr + off, 16, 1024),
                      idesc, kk > 0);
        }
        umma_commit(cx.bar(B_SFULL + (n_qk & 1)));
        umma_commit(cx.bar(B_KVEMPTY + slot));
        if (i == nt - 1) umma_commit(cx.bar(B_QEMPTY + qb));
        ++n_qk;
      }
      if (i > 0) {
        const int ii = i - 1, j = s.j0 + ii;
        ok = bounded_wait(cx.bar(B_PFULL), n_pv & 1, cx.abort_flag, cx.status, kErrMmaWait);
        if (!ok) break;
        const uint32_t pos = ring + 2 * ii + 1, slot = pos % kRing;
        ok = bounded_wait(cx.bar(B_KVFULL + slot), (pos / kRing) & 1, cx.abort_flag, cx.status,
                          kErrMmaWait);
        if (!ok) break;
        tc_fence_after();
        const uint32_t vaddr = cx.sbase + SM_RING + slot * kSlotBytes;
        const int nk = j < p.n_main ? 8 : 4;  // 16 keys per step; the own-row tile has 64 keys
        for (int kk = 0; kk < nk; ++kk) {
          const uint32_t aoff = (kk >> 2) * (kQTileBytes / 2) + (kk & 3) * 32;  // P, K-major
          const uint32_t boff = kk * 16 * 128;                                // V, 16 key rows
          umma_f16_ss(cx.tmem + TM_O, sw128_desc(cx.sbase + SM_P + aoff, 16, 1024),
                      sw128_desc(vaddr + boff, kAtom, 1024), kIdescPV, (ii > 0 || kk > 0));
        }
        umma_commit(cx.bar(B_ODONE));
        umma_commit(cx.bar(B_KVEMPTY + slot));
        ++n_pv;
      }
    }
    ring += 2 * nt;
    ++seg;
  }
  // Every MMA issued so far must be complete before TMEM is released.
  umma_commit(cx.bar(B_DRAIN));
  if (!drain_wait(cx.bar(B_DRAIN), 0)) atomicOr(cx.status, kErrDrain);
}

// -------------------------------------------------------------------------------- softmax
// Scores are kept in log2 units: x = s * log2(e) / sqrt(128), p = 2^(x - m). The running max m is
// only raised (and the TMEM accumulator rescaled by 2^(m_old - m_new)) when a tile's max exceeds
// it by more than kLazy, so p <= 2^kLazy and most tiles skip the TMEM round trip.
constexpr float kLazy = 8.0f;

__device__ __forceinline__ void rescale_O(uint32_t taddr, float alpha) {
#pragma unroll
  for (int ch = 0; ch < 4; ++ch) {
    uint32_t o[32];
    tmem_ld32(taddr + ch * 32, o);
    tmem_wait_ld();
    reg_fence32(o);
#pragma unroll
    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
    tmem_st32(taddr + ch * 32, o);
  }
  tmem_wait_st();
}

__device__ __noinline__ void softmax_warps(const AttnParams& p, const Ctx& cx) {
  const int r = threadIdx.x;  // folded row = TMEM lane
  const uint32_t lane_addr = static_cast<uint32_t>(threadIdx.x & ~31) << 16;
  const float c = p.scale_log2;
  const uint32_t prow = cx.sbase + SM_P + static_cast<uint32_t>(r) * 128u;
  const uint32_t rsw = static_cast<uint32_t>(r & 7);
  uint32_t n_s = 0, pv_seen = 0, pv_total = 0;
  int seg = 0;
  bool ok = true;
  long long t = cx.start;
  Seg s;

  // Waits for PV number k of this CTA (all PVs before it are known to be complete).
  auto wait_pv = [&](uint32_t k) -> bool {
    if (pv_seen > k) return true;
    pv_seen = k + 1;
    // warp-uniform outcome: the TMEM loads and shuffles that follow need the full warp
    return __all_sync(0xffffffffu, bounded_wait(cx.bar(B_ODONE), k & 1, cx.abort_flag, cx.status,
                                                kErrSoftmaxWait));
  };

  while (ok && next_seg(t, cx.end, p.T, s)) {
    const int l = s.u / kHkv, g = s.u % kHkv;
    const int nt = s.j1 - s.j0;
    float m_ref = -INFINITY, lsum = 0.f;
    for (int i = 0; i < nt; ++i) {
      const int j = s.j0 + i;
      const uint32_t sb = n_s & 1;
      ok = __all_sync(0xffffffffu, bounded_wait(cx.bar(B_SFULL + sb), (n_s >> 1) & 1,
                                                cx.abort_flag, cx.status, kErrSoftmaxWait));
      if (!ok) break;
      ++n_s;
      tc_fence_after();
      const bool tail = j >= p.n_main;
      const uint32_t sa = cx.tmem + lane_addr + TM_S + sb * 128;
      uint32_t v[4][32];
      tmem_ld32(sa, v[0]);
      tmem_ld32(sa + 32, v[1]);
      if (!tail) {
        tmem_ld32(sa + 64, v[2]);
        tmem_ld32(sa + 96, v[3]);
      }
      tmem_wait_ld();
      reg_fence32(v[0]);
      reg_fence32(v[1]);
      if (!tail) {
        reg_fence32(v[2]);
        reg_fence32(v[3]);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) v[2][e] = v[3][e] = __float_as_uint(-INFINITY);
      }
      // keys >= S of the last cache tile (zero-filled by TMA) are masked out
      const int key0 = j * kKeyTile;
      if (!tail && key0 + kKeyTile > p.S) {
#pragma unroll
        for (int ch = 0; ch < 4; ++ch)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (key0 + ch * 32 + e >= p.S) v[ch][e] = __float_as_uint(-INFINITY);
      }
      float mx = -INFINITY;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch)
#pragma unroll
        for (int e = 0; e < 32; ++e) mx = fmaxf(mx, __uint_as_float(v[ch][e]));
      const float mt = mx * c;
      const bool need = (i == 0) || (mt > m_ref + kLazy);
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = fmaxf(m_ref, mt);
        const float alpha = ex2_approx(m_ref - m_new);
        if (i > 0) {
          ok = wait_pv(pv_total + i - 1);  // the accumulator holds tiles < i
          if (!ok) break;
          tc_fence_after();
          rescale_O(cx.tmem + lane_addr + TM_O, alpha);
        }
        lsum *= alpha;
        m_ref = m_new;
      }
      const float neg = -m_ref;
      float tsum = 0.f;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch)
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float p0 = ex2_approx(fmaf(__uint_as_float(v[ch][2 * e]), c, neg));
          const float p1 = ex2_approx(fmaf(__uint_as_float(v[ch][2 * e + 1]), c, neg));
          tsum += p0 + p1;
          v[ch][e] = pack_bf16x2(p0, p1);  // packed P overwrites the consumed scores
        }
      lsum += tsum;
      if (i > 0) {
        ok = wait_pv(pv_total + i - 1);  // PV(i-1) has finished reading the P buffer
        if (!ok) break;
      }
      const int nq = tail ? 8 : 16;  // 16-byte chunks of 8 keys
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        if (q < nq) {
          const uint32_t addr = prow + (q >> 3) * (kQTileBytes / 2) + (((q & 7) ^ rsw) << 4);
          const int ch = q >> 2, k4 = (q & 3) * 4;
          st_shared_v4(addr, v[ch][k4], v[ch][k4 + 1], v[ch][k4 + 2], v[ch][k4 + 3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(cx.bar(B_PFULL));
    }
    if (!ok) break;

    // ---- epilogue: O / l of this segment
    ok = wait_pv(pv_total + nt - 1);
    if (!ok) break;
    tc_fence_after();
    const float inv = 1.0f / lsum;
    const bool full = (s.j0 == 0 && s.j1 == p.T);
    const int slot = seg == 0 ? 0 : 1;  // a partial segment is the CTA's first or its last
    float* po = p.part_o + ((static_cast<size_t>(blockIdx.x) * 2 + slot) * kRows + r) * kD;
    __nv_bfloat16* orow = p.out[l] + (static_cast<size_t>(g) * kRows + r) * kD;
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
      uint32_t o[32];
      tmem_ld32(cx.tmem + lane_addr + TM_O + ch * 32, o);
      tmem_wait_ld();
      reg_fence32(o);
      if (full) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(o[8 * q + 0]) * inv, __uint_as_float(o[8 * q + 1]) * inv);
          w.y = pack_bf16x2(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv);
          w.z = pack_bf16x2(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv);
          w.w = pack_bf16x2(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv);
          *reinterpret_cast<uint4*>(orow + ch * 32 + 8 * q) = w;
        }
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float4 w = make_float4(__uint_as_float(o[4 * q]) * inv, __uint_as_float(o[4 * q + 1]) * inv,
                                 __uint_as_float(o[4 * q + 2]) * inv, __uint_as_float(o[4 * q + 3]) * inv);
          *reinterpret_cast<float4*>(po + ch * 32 + 4 * q) = w;
        }
      }
    }
    if (!full)
      p.part_lse[(static_cast<size_t>(blockIdx.x) * 2 + slot) * kRows + r] = m_ref + log2f(lsum);
    tc_fence_before();
    pv_total += nt;
    ++seg;
  }
}

}  // namespace attn

// ------------------------------------------------------------------------------------ kernel
__global__ void __launch_bounds__(attn::kThreads, 1)
    attention_kernel(const __grid_constant__ AttnParams p) {
  using namespace attn;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Ctx cx;
  cx.sbase = smem_u32(smem);
  cx.abort_flag = reinterpret_cast<volatile uint32_t*>(smem + SM_ABORT);
  cx.status = p.status;
  cx.start = cta_tile_start(blockIdx.x, p.W, gridDim.x);
  cx.end = cta_tile_start(blockIdx.x + 1, p.W, gridDim.x);

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(cx.bar(B_QFULL + b), 1);
      mbar_init(cx.bar(B_QEMPTY + b), 1);
      mbar_init(cx.bar(B_SFULL + b), 1);
    }
    for (int b = 0; b < kRing; ++b) {
      mbar_init(cx.bar(B_KVFULL + b), 1);
      mbar_init(cx.bar(B_KVEMPTY + b), 1);
    }
    mbar_init(cx.bar(B_PFULL), 128);
    mbar_init(cx.bar(B_ODONE), 1);
    mbar_init(cx.bar(B_DRAIN), 1);
    *cx.abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(cx.sbase + SM_TMEM, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cx.tmem = *reinterpret_cast<volatile uint32_t*>(smem + SM_TMEM);

  if (warp < 4) {
    softmax_warps(p, cx);
  } else if (warp == 4) {
    if (lane == 0) producer(p, cx);
  } else {
    if (lane == 0) mma_issuer(p, cx);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(cx.tmem, kTmemCols);
}

}  // namespace ea

namespace ea {
size_t attention_smem_bytes() { return attn::kSmemBytes; }
int attention_threads() { return attn::kThreads; }
}  // namespace ea
