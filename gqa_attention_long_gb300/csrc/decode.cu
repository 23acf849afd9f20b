// decode.cu — split-KV single-token decode attention of the VLM text model on sm_103a.
//
// What it computes (alpamayo_tt/text.py, TTText._layer_decode and TTText._decode_inputs_host):
// per layer, for the decode token's 64 query heads and 8 KV heads (query head h reads KV head
// h / 8),
//   1. q and k rows RMS-normalised with the q_norm / k_norm gains (eps 1e-6) and rotated with
//      the HF rotate_half RoPE (theta 5e6) at position pos + rope_delta;
//   2. the roped k and the raw v written into row pos of the layer's K and V caches
//      (paged_update_cache);
//   3. softmax(q K[g, 0..pos]^T / sqrt(128)) V[g, 0..pos] for every query head
//      (scaled_dot_product_attention_decode with cur_pos = pos).
//
// Work decomposition: a unit is one (layer, kv head): its 8 query heads against keys [0, pos],
// cut into tiles of 128 keys. The tiles of all units, unit-major, are cut into one contiguous
// range per CTA (one CTA per SM); a CTA walks its range as segments (the part of one unit in
// it). Per tile, on the tensor cores (issued by the MMA warp):
//   S^T  = K Q^T    M = 128 keys (TMEM lanes), N = 16 (the 8 query heads and 8 zero rows),
//                   K = 128 channels; A = the K tile (TMA, 128-byte swizzle, K-major), B = the
//                   unit's roped q rows in shared memory;
//   O^T += V^T P^T  M = 128 channels (TMEM lanes), N = 16, K = 128 keys; A = the same V tile
//                   read MN-major, B = P (bf16) written by the softmax threads.
// Between the two, the 128 compute threads (thread = key = TMEM lane) form the exact online
// softmax per head: the tile's max and sum over keys by warp shuffles and a 4-warp exchange.
// Keys after pos (the end of the last tile) get score -inf and zeroed V rows, so rows the text
// model has not written yet (any content, NaN included) cannot leak. The tensor cores see the
// GQA group's 8 heads as the N dimension; at ~8 flop per cache byte the kernel is bound by HBM,
// and the tensor cores keep the per-key arithmetic (2 x 8 x 128 FMAs) off the issue slots.
//
// The CTA whose segment holds the unit's last tile also writes the new k and v rows into cache
// row pos, and its producer loads that tile only after they are out. A unit cut over several
// CTAs is merged by the part that finishes last (a per-unit arrival count): it combines every
// part's unnormalised output with weights 2^(m_p - M) and writes the bf16 result; no CTA ever
// waits for another. A single-layer call over a short cache (2 to 8 key tiles per unit: the
// decode step of one layer, pos < 1024) runs instead as one thread-block cluster per unit with
// one CTA per tile: the parts leave their partials in shared memory and, after a cluster
// barrier, the CTAs combine the unit's outputs from the cluster's shared memory, so no partial
// travels through global memory. (For longer caches the grid-wide split is faster: clusters of
// 16 CTAs that each hold a whole SM wait for a whole free GPC, which a preceding kernel's tail
// delays.)
// Before waiting for the preceding kernel, the producer asks L2 for the CTA's first tiles (a
// prefetch only: what the preceding kernel writes still wins).
//
// Warp roles (192 threads): warps 0-3 compute (prologue, softmax, epilogue); warp 4 lane 0 issues
// the TMA loads of the K and V tiles into a 3-stage ring; warp 5 lane 0 issues the MMAs. S and P
// are double-buffered, so QK(n) is issued as soon as the softmax of tile n-2 has released its
// score buffer: it runs while the softmax of tile n-1 does, and the compute warps go from one
// tile's softmax to the next without waiting for the tensor core.
#include "internal.cuh"
#include "cluster_exit.cuh"
#include "ptx.cuh"
#include "rope.cuh"

namespace ea {
namespace dec {

constexpr int kThreads = 192;
constexpr int kCompute = 128;
constexpr int kStages = 3;
constexpr uint32_t kAtomBytes = 16384;          // one 64-channel half of a 128-row tile
constexpr uint32_t kTileBytes = 2 * kAtomBytes;  // a K or a V tile
constexpr uint32_t kStageBytes = 2 * kTileBytes;
constexpr uint32_t kOpAtom = 2048;  // one 64-element half of a 16-row operand (Q or P)
// Shared memory (offsets from the 1024-byte-aligned base)
constexpr uint32_t SM_RING = 0;
constexpr uint32_t SM_QT = SM_RING + kStages * kStageBytes;  // 16 rows x 128 channels bf16
constexpr uint32_t SM_PT = SM_QT + 2 * kOpAtom;              // 2 x (16 rows x 128 keys bf16)
constexpr uint32_t kPtBytes = 2 * kOpAtom;
constexpr uint32_t SM_RED = SM_PT + 2 * kPtBytes;            // [2][4 warps][8 heads] fp32
constexpr uint32_t SM_BAR = SM_RED + 2 * 4 * kRepText * 4;
// SDONE, PFULL, ODONE: one barrier per parity of the tile count (tile n uses S and P buffer n % 2);
// QFULL and OFREE complete once per segment
constexpr int B_FULL = 0, B_EMPTY = kStages, B_SDONE = 2 * kStages, B_PFULL = B_SDONE + 2,
              B_ODONE = B_PFULL + 2, B_QFULL = B_ODONE + 2, B_OFREE = B_QFULL + 1,
              B_TAIL = B_OFREE + 1, B_DRAIN = B_TAIL + 1, B_MERGE = B_DRAIN + 1,
              kNumBars = B_MERGE + 1;
constexpr uint32_t SM_TMEM = SM_BAR + kNumBars * 8;
constexpr uint32_t SM_ABORT = SM_TMEM + 4;
constexpr uint32_t SM_MERGE = SM_ABORT + 4;
constexpr int kMaxParts = 160;  // parts of one unit (at most one per CTA; the grid is <= 160)
constexpr int kMergeBatch = 10;  // parts per round of loads in the last arriver's merge
constexpr uint32_t kMaxCluster = 8;  // cluster mode: CTAs per unit (the host launches 2..8)
constexpr uint32_t SM_PARTML = (SM_MERGE + 4 + 15) & ~15u;  // [part][head] (max, sum) of a merge
// cluster mode: this CTA's partial, read by the cluster's other CTAs: O [8 heads][128] fp32, then
// (max, sum) per head
constexpr uint32_t SM_CPART = SM_PARTML + kMaxParts * kRepText * 8;
constexpr uint32_t SM_CPART_ML = SM_CPART + kRepText * kD * 4;
constexpr uint32_t kSmemBytes = SM_CPART_ML + kRepText * 8 + 1024;  // + base alignment
static_assert(kSmemBytes <= 232448, "shared memory budget of one sm_103 CTA");
constexpr uint32_t kTmemCols = 64;  // S^T of even / odd tiles in [0, 16) / [16, 32), O^T in [32, 48)
constexpr uint32_t TM_S = 0, TM_O = 32;

struct Seg {
  int u, j0, j1;  // unit and its key-tile range [j0, j1)
};

// atomicAdd at GPU scope with acquire-release semantics; returns the old value
__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* a, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(a), "r"(v) : "memory");
  return old;
}

// Next segment of a CTA's tile range [t, end): unit u = t / T (tile indices stay below 2^31).
__device__ __forceinline__ bool next_seg(long long& t, long long end, int T, Seg& s) {
  if (t >= end) return false;
  const int ti = static_cast<int>(t);
  s.u = ti / T;
  s.j0 = ti - s.u * T;
  const long long j1 = s.j0 + (end - t);
  s.j1 = static_cast<int>(j1 < T ? j1 : T);
  t += s.j1 - s.j0;
  return true;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, m));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
  return x;
}

// ------------------------------------------------------------------------------ producer
template <int CAP>
__device__ __noinline__ void producer(const DecodeParams<CAP>& p, uint32_t sbase, long long start,
                                      long long end, volatile uint32_t* abort_flag) {
  const uint64_t pol = l2_policy_evict_first();  // every cache tile is read once
  const uint32_t bar0 = sbase + SM_BAR;
  uint32_t n = 0, n_tail = 0;
  bool ok = true;
  long long t = start;
  Seg s;
  while (ok && next_seg(t, end, p.T, s)) {
    const int l = s.u / kHkv, g = s.u % kHkv;
    for (int j = s.j0; j < s.j1 && ok; ++j) {
      if (j == p.T - 1) {
        // the unit's last tile holds row pos, written by this CTA's compute warps
        ok = bounded_wait(bar0 + 8 * B_TAIL, n_tail & 1, abort_flag, p.status, kErrDecodeWait);
        if (!ok) break;
        fence_proxy_async_global();
        ++n_tail;
      }
      const uint32_t slot = n % kStages, round = n / kStages;
      if (round > 0) {
        ok = bounded_wait(bar0 + 8 * (B_EMPTY + slot), (round - 1) & 1, abort_flag, p.status,
                          kErrDecodeWait);
        if (!ok) break;
      }
      const uint32_t fb = bar0 + 8 * (B_FULL + slot);
      const uint32_t dst = sbase + SM_RING + slot * kStageBytes;
      mbar_expect_tx(fb, kStageBytes);
      const int row0 = j * kKeyTile;  // rows past Smax arrive zero-filled
      tma_load_3d(dst, &p.kmap[l], fb, 0, row0, g, pol);
      tma_load_3d(dst + kAtomBytes, &p.kmap[l], fb, 64, row0, g, pol);
      tma_load_3d(dst + kTileBytes, &p.vmap[l], fb, 0, row0, g, pol);
      tma_load_3d(dst + kTileBytes + kAtomBytes, &p.vmap[l], fb, 64, row0, g, pol);
      ++n;
    }
  }
  // every load of this CTA is issued: the next kernel's CTAs may be placed on SMs as they free
  // up (they wait for this grid to complete before they read anything it writes)
  pdl_launch_dependents();
  if (!ok) {  // let every copy already issued land before the CTA gives its shared memory back
    for (uint32_t k = 0; k < static_cast<uint32_t>(kStages) && k < n; ++k) {
      const uint32_t q = n - 1 - k;
      if (!drain_wait(bar0 + 8 * (B_FULL + q % kStages), (q / kStages) & 1)) atomicOr(p.status, kErrDrain);
    }
  }
}

// --------------------------------------------------------------------------- compute warps
// Prologue of a segment: the roped q rows of the unit's 8 heads into QT rows 0-7 (warps 0-1,
// octet o = head o: lane i holds channels [8i, 8i+8) and their RoPE partners [64+8i, 64+8i+8)),
// and, for the segment holding the unit's last tile, the new k row (normed, roped, bf16) and v
// row into cache row pos (warp 2: its four octets compute the same row, octet 0 stores it).
template <int CAP>
__device__ __forceinline__ void segment_prologue(const DecodeParams<CAP>& p, uint32_t sbase, int l,
                                                 int g, bool last, int tid) {
  const int w = tid >> 5;
  if (w > 2 || (w == 2 && !last)) return;
  const int i = tid & 7;
  const int dl = 8 * i, dh = 64 + 8 * i;
  // the row's and the gain's global loads go out first; the rotation angles (kernel parameters
  // only) are computed while they are in flight
  const __nv_bfloat16* row = w < 2 ? p.q_raw[l] + static_cast<size_t>(kRepText * g + (tid >> 3)) * kD
                                   : p.k_raw[l] + static_cast<size_t>(g) * kD;
  const __nv_bfloat16* gam = w < 2 ? p.q_gamma[l] : p.k_gamma[l];
  const uint4 rl = *reinterpret_cast<const uint4*>(row + dl), rh = *reinterpret_cast<const uint4*>(row + dh);
  const uint4 ml = *reinterpret_cast<const uint4*>(gam + dl), mh = *reinterpret_cast<const uint4*>(gam + dh);
  float cs[8], sn[8];
  float ih[8], il[8];
  load_inv8(p.inv_hi, p.inv_lo, dl, ih, il);
#pragma unroll
  for (int e = 0; e < 8; ++e) rope_cos_sin(p.rope_pos, ih[e], il[e], cs[e], sn[e]);
  float xl[8], xh[8], gl[8], gh[8], yl[8], yh[8];
  unpack_bf16x8(rl, xl);
  unpack_bf16x8(rh, xh);
  unpack_bf16x8(ml, gl);
  unpack_bf16x8(mh, gh);
  if (w < 2) {
    const int h = tid >> 3;  // 0..7
    norm_rope(xl, xh, gl, gh, cs, sn, yl, yh);
    const uint4 ql = pack8(yl, false), qh = pack8(yh, false);
    const uint32_t qt = sbase + SM_QT;
    st_shared_v4(qt + swz_off(h, i, kOpAtom), ql.x, ql.y, ql.z, ql.w);
    st_shared_v4(qt + swz_off(h, i + 8, kOpAtom), qh.x, qh.y, qh.z, qh.w);
  } else {
    // the v row's loads go out with the k row's (before any cache store)
    const __nv_bfloat16* vrow = p.v_raw[l] + static_cast<size_t>(g) * kD;
    const uint4 vl = *reinterpret_cast<const uint4*>(vrow + dl), vh = *reinterpret_cast<const uint4*>(vrow + dh);
    norm_rope(xl, xh, gl, gh, cs, sn, yl, yh);
    if (tid < 64 + 8) {
      const size_t ro = (static_cast<size_t>(g) * p.Smax + p.pos) * kD;
      *reinterpret_cast<uint4*>(p.kc[l] + ro + dl) = pack8(yl, false);
      *reinterpret_cast<uint4*>(p.kc[l] + ro + dh) = pack8(yh, false);
      *reinterpret_cast<uint4*>(p.vc[l] + ro + dl) = vl;
      *reinterpret_cast<uint4*>(p.vc[l] + ro + dh) = vh;
      fence_proxy_async_global();  // the rows are read back by TMA (async proxy)
    }
  }
}

// ----------------------------------------------------------------------------- MMA issuer
// Per segment, step i issues QK(i) and PV(i-1), in whichever order their inputs arrive. QK(n) needs
// its tile in the ring and score buffer n % 2 released by the softmax of tile n-2 (its PFULL). PV(n)
// needs P(n) (PFULL of tile n); the segment's first PV, which starts a fresh accumulator, also
// needs the previous segment's epilogue to have read it (OFREE completes once per segment). A PV
// whose P is ready is not held behind a tile still in flight, so its ring stage is released as
// early as the softmax allows.
template <int CAP>
__device__ __noinline__ void mma_issuer(const DecodeParams<CAP>& p, uint32_t sbase, uint32_t tmem,
                                        long long start, long long end, volatile uint32_t* abort_flag) {
  const uint32_t bar0 = sbase + SM_BAR;
  // S^T: A = K tile (K-major), B = QT (K-major); O^T: A = V tile (MN-major), B = PT (K-major)
  constexpr uint32_t kIdescS = umma_idesc_f16(128, 16, true, false, false);
  constexpr uint32_t kIdescO = umma_idesc_f16(128, 16, true, true, false);
  const uint32_t qt = sbase + SM_QT, pt = sbase + SM_PT;
  auto bar = [&](int b) { return bar0 + 8 * b; };
  uint32_t n = 0;  // tiles of this CTA before the current segment
  int sg = 0;
  bool ok = true;
  long long t = start;
  Seg s;
  while (ok && next_seg(t, end, p.T, s)) {
    // this segment's q rows are in QT (the previous segment's QKs were all observed complete by
    // the compute warps before they rewrote it)
    ok = bounded_wait(bar(B_QFULL), sg & 1, abort_flag, p.status, kErrDecodeWait);
    if (!ok) break;
    const int nt = s.j1 - s.j0;
    auto qk_ready = [&](int i) -> bool {
      const uint32_t nn = n + i;
      if (!mbar_test_wait(bar(B_FULL + nn % kStages), (nn / kStages) & 1)) return false;
      return nn < 2 || mbar_test_wait(bar(B_PFULL + (nn & 1)), ((nn - 2) >> 1) & 1);
    };
    auto issue_qk = [&](int i) {
      const uint32_t nn = n + i;
      const uint32_t ka = sbase + SM_RING + (nn % kStages) * kStageBytes;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)  // 16 channels per step; 4 steps per 64-channel half
        umma_f16_ss(tmem + TM_S + (nn & 1) * 16,
                    sw128_desc(ka + (kk >> 2) * kAtomBytes + (kk & 3) * 32, 16, 1024),
                    sw128_desc(qt + (kk >> 2) * kOpAtom + (kk & 3) * 32, 16, 1024), kIdescS, kk > 0);
      umma_commit(bar(B_SDONE + (nn & 1)));
    };
    auto pv_ready = [&](int ii) -> bool {
      const uint32_t nn = n + ii;
      if (ii == 0 && sg > 0 && !mbar_test_wait(bar(B_OFREE), (sg - 1) & 1)) return false;
      return mbar_test_wait(bar(B_PFULL + (nn & 1)), (nn >> 1) & 1);
    };
    auto issue_pv = [&](int ii) {
      const uint32_t nn = n + ii, slot = nn % kStages;
      const uint32_t va = sbase + SM_RING + slot * kStageBytes + kTileBytes;
      const uint32_t ptb = pt + (nn & 1) * kPtBytes;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)  // 16 keys per step
        umma_f16_ss(tmem + TM_O, sw128_desc(va + kk * 16 * 128, kAtomBytes, 1024),
                    sw128_desc(ptb + (kk >> 2) * kOpAtom + (kk & 3) * 32, 16, 1024), kIdescO,
                    (ii > 0 || kk > 0));
      umma_commit(bar(B_EMPTY + slot));  // K and V of this stage are consumed
      umma_commit(bar(B_ODONE + (nn & 1)));
    };
    for (int i = 0; i <= nt && ok; ++i) {
      bool qk_todo = i < nt, pv_todo = i > 0;
      uint64_t t0 = 0;
      for (uint32_t it = 0; qk_todo || pv_todo; ++it) {
        bool moved = false;
        if (qk_todo && qk_ready(i)) {
          issue_qk(i);
          qk_todo = false;
          moved = true;
        }
        if (pv_todo && pv_ready(i - 1)) {
          issue_pv(i - 1);
          pv_todo = false;
          moved = true;
        }
        if (moved) continue;
        // bounded like every other wait: the CTA's abort flag, a time limit and a poll limit
        if ((it & 63u) == 0) {
          if (*abort_flag) {
            ok = false;
            break;
          }
          const uint64_t now = globaltimer_ns();
          if (t0 == 0) t0 = now;
          if (now - t0 > kWaitLimitNs || it >= 0x7fffffc0u) {
            *abort_flag = 1u;
            atomicOr(p.status, kErrDecodeWait);
            ok = false;
            break;
          }
        }
      }
    }
    n += nt;
    ++sg;
  }
  // Every MMA issued must be complete before TMEM is released.
  umma_commit(bar(B_DRAIN));
  if (!drain_wait(bar(B_DRAIN), 0)) atomicOr(p.status, kErrDrain);
}

template <int CAP>
__device__ __noinline__ void compute(const DecodeParams<CAP>& p, uint32_t sbase, uint8_t* smem,
                                     uint32_t tmem, long long start, long long end,
                                     volatile uint32_t* abort_flag) {
  const int tid = threadIdx.x;  // key row (score phase) or channel (output phase) = TMEM lane
  const int warp = tid >> 5;
  const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
  const uint32_t bar0 = sbase + SM_BAR;
  float* red = reinterpret_cast<float*>(smem + SM_RED);  // [2][4][8]
  volatile uint32_t* merge_flag = reinterpret_cast<volatile uint32_t*>(smem + SM_MERGE);
  const uint32_t pt = sbase + SM_PT;
  auto wait = [&](int b, uint32_t parity) -> bool {
    return bounded_wait(bar0 + 8 * b, parity, abort_flag, p.status, kErrDecodeWait);
  };
  if (p.cluster && tid < kRepText)  // an empty partial, for a CTA without tiles (or that gave up)
    reinterpret_cast<float2*>(smem + SM_CPART_ML)[tid] = make_float2(-INFINITY, 0.f);
  uint32_t n = 0;  // tiles of this CTA so far
  bool ok = true, first_seg = true;
  long long t = start;
  Seg s;
  while (ok && next_seg(t, end, p.T, s)) {
    const int l = s.u / kHkv, g = s.u % kHkv;
    const bool last = s.j1 == p.T;
    segment_prologue(p, sbase, l, g, last, tid);
    fence_proxy_async_smem();  // QT is read by the tensor core (async proxy)
    bar_sync(1, kCompute);
    if (tid == 0) {
      if (last) mbar_arrive(bar0 + 8 * B_TAIL);
      mbar_arrive(bar0 + 8 * B_QFULL);
    }
    float m[kRepText], lsum[kRepText];
#pragma unroll
    for (int h = 0; h < kRepText; ++h) {
      m[h] = -INFINITY;
      lsum[h] = 0.f;
    }
    for (int j = s.j0; j < s.j1; ++j, ++n) {
      const uint32_t slot = n % kStages;
      const uint32_t kaddr = sbase + SM_RING + slot * kStageBytes, vaddr = kaddr + kTileBytes;
      // the tile has landed (its V rows of keys after pos are zeroed below), S(n) is complete, and
      // P buffer n % 2 is free: PV(n-2), its last reader, has completed (this warpgroup waits for
      // every PV of a parity in turn, so the phase is unambiguous)
      bool okt = wait(B_FULL + slot, (n / kStages) & 1);
      okt = okt && wait(B_SDONE + (n & 1), (n >> 1) & 1);
      if (n >= 2) okt = okt && wait(B_ODONE + (n & 1), ((n - 2) >> 1) & 1);
      okt = __all_sync(0xffffffffu, okt);
      const uint32_t ptb = pt + (n & 1) * kPtBytes;
      const int key = j * kKeyTile + tid;
      const bool live = key <= p.pos;
      float x[kRepText];
      if (okt) {
        tc_fence_after();
        uint32_t sv[8];
        tmem_ld8(tmem + lane_addr + TM_S + (n & 1) * 16, sv);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < kRepText; ++h) x[h] = live ? __uint_as_float(sv[h]) * p.scale_log2 : -INFINITY;
        if (!live) {  // a row the text model has not written (or past Smax): zero its V row
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            st_shared_v4(vaddr + tid * 128 + 16 * c, 0u, 0u, 0u, 0u);
            st_shared_v4(vaddr + kAtomBytes + tid * 128 + 16 * c, 0u, 0u, 0u, 0u);
          }
        }
#pragma unroll
        for (int h = 0; h < kRepText; ++h) {
          const float mx = warp_max(x[h]);
          if ((tid & 31) == 0) red[warp * kRepText + h] = mx;
        }
      }
      if (!bar_sync_and(1, kCompute, okt)) {
        ok = false;
        break;
      }
      float alpha[kRepText], pr[kRepText];
      bool resc = false;
#pragma unroll
      for (int h = 0; h < kRepText; ++h) {
        const float tm = fmaxf(fmaxf(red[h], red[kRepText + h]), fmaxf(red[2 * kRepText + h], red[3 * kRepText + h]));
        const float mn = fmaxf(m[h], tm);  // every tile has a live key, so mn is finite
        alpha[h] = ex2_approx(m[h] - mn);  // 0 on the segment's first tile
        resc |= alpha[h] != 1.0f;
        m[h] = mn;
        pr[h] = ex2_approx(x[h] - mn);
      }
      // P^T (B operand, K-major): row h = head, column = key; 16-byte chunk c of row h at
      // chunk c ^ (h % 8) of the key's 64-key half
#pragma unroll
      for (int h = 0; h < kRepText; ++h) {
        const uint32_t a = ptb + (tid >> 6) * kOpAtom + h * 128 +
                           ((((tid & 63) >> 3) ^ (h & 7)) << 4) + (tid & 7) * 2;
        st_shared_u16(a, __bfloat16_as_ushort(__float2bfloat16_rn(pr[h])));
      }
#pragma unroll
      for (int h = 0; h < kRepText; ++h) {
        const float sm = warp_sum(pr[h]);
        if ((tid & 31) == 0) red[4 * kRepText + warp * kRepText + h] = sm;
      }
      bar_sync(1, kCompute);
#pragma unroll
      for (int h = 0; h < kRepText; ++h)
        lsum[h] = lsum[h] * alpha[h] + ((red[4 * kRepText + h] + red[5 * kRepText + h]) +
                                        (red[6 * kRepText + h] + red[7 * kRepText + h]));
      bool okr = true;
      if (j > s.j0 && resc) {
        // bring the accumulator (the segment's tiles before this one) to the new max, once PV(n-1)
        // has completed (PV(n-3) was waited for at tile n-1)
        okr = __all_sync(0xffffffffu, wait(B_ODONE + ((n - 1) & 1), ((n - 1) >> 1) & 1));
        if (okr) {
          tc_fence_after();
          uint32_t ov[8];
          tmem_ld8(tmem + lane_addr + TM_O, ov);
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < kRepText; ++h) ov[h] = __float_as_uint(__uint_as_float(ov[h]) * alpha[h]);
          tmem_st8(tmem + lane_addr + TM_O, ov);
          tmem_wait_st();
        }
      }
      fence_proxy_async_smem();  // P^T and zeroed V rows are read by the tensor core
      tc_fence_before();
      if (!bar_sync_and(1, kCompute, okr)) {
        ok = false;
        break;
      }
      if (tid == 0) mbar_arrive(bar0 + 8 * (B_PFULL + (n & 1)));  // P(n) out, S(n) read
    }
    if (!ok) break;
    // ---- segment end: the last PV, PV(n-1), and with it every earlier MMA (PV(n-3), the
    // previous phase of its barrier, was waited for at tile n-1; PV(n+1) is not issued)
    bool oke = wait(B_ODONE + ((n - 1) & 1), ((n - 1) >> 1) & 1);
    oke = __all_sync(0xffffffffu, oke);
    uint32_t ov[8];
    if (oke) {
      tc_fence_after();
      tmem_ld8(tmem + lane_addr + TM_O, ov);  // O^T row = channel tid, column = head
      tmem_wait_ld();
    }
    tc_fence_before();
    if (!bar_sync_and(1, kCompute, oke)) {
      ok = false;
      break;
    }
    if (tid == 0) mbar_arrive(bar0 + 8 * B_OFREE);  // the accumulator is read
    const bool full = s.j0 == 0 && s.j1 == p.T;
    if (p.cluster) {
      // cluster mode: the partial stays in this CTA's shared memory for the cluster's merge
      float* cpo = reinterpret_cast<float*>(smem + SM_CPART) + tid;
#pragma unroll
      for (int h = 0; h < kRepText; ++h) cpo[h * kD] = __uint_as_float(ov[h]);
      float2* cml = reinterpret_cast<float2*>(smem + SM_CPART_ML);
#pragma unroll
      for (int h = 0; h < kRepText; ++h)
        if (tid == h) cml[h] = make_float2(m[h], lsum[h]);
    } else if (full) {
      __nv_bfloat16* o = p.out[l] + static_cast<size_t>(kRepText * g) * kD + tid;
#pragma unroll
      for (int h = 0; h < kRepText; ++h) o[h * kD] = __float2bfloat16_rn(__uint_as_float(ov[h]) / lsum[h]);
    } else {
      // partial: unnormalised output with its (max, sum) per head, then the arrival count; the
      // part that arrives last merges every part of the unit. Part index: 2 c + slot (a partial
      // segment is the CTA's first or its last), or c in the unit-aligned mode (one segment per
      // CTA), where the unit's parts are then contiguous. Layout [part][channel][8 heads]: a
      // thread's 8 values are two 16-byte stores.
      const int slot = first_seg ? 0 : 1;
      const size_t ps = p.per_unit ? static_cast<size_t>(blockIdx.x) : static_cast<size_t>(blockIdx.x) * 2 + slot;
      float4* po = reinterpret_cast<float4*>(p.part_o + ps * kRepText * kD) + 2 * tid;
      po[0] = make_float4(__uint_as_float(ov[0]), __uint_as_float(ov[1]), __uint_as_float(ov[2]), __uint_as_float(ov[3]));
      po[1] = make_float4(__uint_as_float(ov[4]), __uint_as_float(ov[5]), __uint_as_float(ov[6]), __uint_as_float(ov[7]));
      if (tid < kRepText) {  // thread h stores head h's (max, sum): one 8-byte store
        float mh = m[0], lh = lsum[0];
#pragma unroll
        for (int h = 1; h < kRepText; ++h)
          if (tid == h) {
            mh = m[h];
            lh = lsum[h];
          }
        *reinterpret_cast<float2*>(p.part_ml + (ps * kRepText + tid) * 2) = make_float2(mh, lh);
      }
      bar_sync(1, kCompute);
      const long long u0 = static_cast<long long>(s.u) * p.T;
      const int c0 = p.per_unit ? s.u * p.per_unit : cta_of_tile(u0, p.W, gridDim.x);
      const int c1 = p.per_unit ? c0 + p.per_unit - 1 : cta_of_tile(u0 + p.T - 1, p.W, gridDim.x);
      // the count is an acquire-release atomic: the release publishes this part (every thread's
      // stores, ordered before it by the barrier; release is cumulative); for the last part the
      // acquire orders the other parts' partials before its reads (the barrier below extends it
      // to every thread)
      if (tid == 0)
        *merge_flag = atom_add_acq_rel_gpu(p.unit_cnt + s.u, 1u) == static_cast<uint32_t>(c1 - c0) ? 1u : 0u;
      bar_sync(1, kCompute);
      if (*merge_flag) {
        const int np = c1 - c0 + 1;
        // part k's index: see above (the first part's partial may sit in its CTA's second slot)
        const int slot0 = p.per_unit ? 0 : (cta_tile_start(c0, p.W, gridDim.x) >= u0 ? 0 : 1);
        auto part_index = [&](int k) -> size_t {
          return p.per_unit ? static_cast<size_t>(c0 + k)
                            : static_cast<size_t>(c0 + k) * 2 + (k == 0 ? slot0 : 0);
        };
        // Unit-aligned mode: this CTA's only segment is done and its ring is free: thread 0
        // stages the unit's contiguous partials there with one bulk copy (after the acquiring
        // count: a proxy fence orders the copy's reads after it), while the weights are formed.
        const uint32_t mb = bar0 + 8 * B_MERGE;
        if (p.per_unit && tid == 0) {
          fence_proxy_async_global();
          const uint32_t bytes = static_cast<uint32_t>(np) * kRepText * kD * 4;
          mbar_expect_tx(mb, bytes);
          bulk_load(sbase + SM_RING, p.part_o + static_cast<size_t>(c0) * kRepText * kD, bytes, mb,
                    l2_policy_evict_first());
        }
        // Weights w[k][h] = 2^(m_kh - M_h) / L_h (M_h = max_k m_kh, L_h = sum_k l_kh 2^(m_kh - M_h))
        // into shared memory: 16 threads per head, each over parts j, j + 16, ... (up to
        // kMaxParts / 16 = 10), reduced by shuffles within the 16. Every part has a live key, so
        // every m is finite.
        float* sw = reinterpret_cast<float*>(smem + SM_PARTML);  // [part][head]
        {
          constexpr int kPer = kMaxParts / 16;
          const int h = tid >> 4, j = tid & 15;
          float2 ml[kPer];
#pragma unroll
          for (int e = 0; e < kPer; ++e) {
            const int k = j + 16 * e;
            ml[e] = k < np ? __ldcg(reinterpret_cast<const float2*>(p.part_ml + (part_index(k) * kRepText + h) * 2))
                           : make_float2(-INFINITY, 0.f);
          }
          float M = -INFINITY;
#pragma unroll
          for (int e = 0; e < kPer; ++e) M = fmaxf(M, ml[e].x);
#pragma unroll
          for (int m = 8; m >= 1; m >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, m));
          float L = 0.f;
#pragma unroll
          for (int e = 0; e < kPer; ++e) {
            ml[e].x = j + 16 * e < np ? ex2_approx(ml[e].x - M) : 0.f;
            L = fmaf(ml[e].y, ml[e].x, L);
          }
#pragma unroll
          for (int m = 8; m >= 1; m >>= 1) L += __shfl_xor_sync(0xffffffffu, L, m);
          const float inv = 1.0f / L;
#pragma unroll
          for (int e = 0; e < kPer; ++e)
            if (j + 16 * e < np) sw[(j + 16 * e) * kRepText + h] = ml[e].x * inv;
        }
        bar_sync(1, kCompute);
        // thread = channel: the 8 heads as independent sums over the parts
        float acc[kRepText];
#pragma unroll
        for (int h = 0; h < kRepText; ++h) acc[h] = 0.f;
        const float4* sw4 = reinterpret_cast<const float4*>(sw);
        auto add_part = [&](int k, float4 o0, float4 o1) {
          const float4 w0 = sw4[2 * k], w1 = sw4[2 * k + 1];
          acc[0] = fmaf(w0.x, o0.x, acc[0]);
          acc[1] = fmaf(w0.y, o0.y, acc[1]);
          acc[2] = fmaf(w0.z, o0.z, acc[2]);
          acc[3] = fmaf(w0.w, o0.w, acc[3]);
          acc[4] = fmaf(w1.x, o1.x, acc[4]);
          acc[5] = fmaf(w1.y, o1.y, acc[5]);
          acc[6] = fmaf(w1.z, o1.z, acc[6]);
          acc[7] = fmaf(w1.w, o1.w, acc[7]);
        };
        bool okm = true;
        if (p.per_unit) {
          okm = bar_sync_and(1, kCompute, bounded_wait(mb, 0, abort_flag, p.status, kErrDecodeWait));
          if (okm) {
            const float4* so4 = reinterpret_cast<const float4*>(smem + SM_RING) + 2 * tid;
#pragma unroll 4
            for (int k = 0; k < np; ++k) add_part(k, so4[k * 2 * kD], so4[k * 2 * kD + 1]);
          } else if (tid == 0 && !drain_wait(mb, 0)) {  // the copy lands before the CTA exits
            atomicOr(p.status, kErrDrain);
          }
        } else {
          // from L2, kMergeBatch parts per round of independent 16-byte loads
          for (int cb = 0; cb < np; cb += kMergeBatch) {
            float4 v[kMergeBatch][2];
#pragma unroll
            for (int b = 0; b < kMergeBatch; ++b) {
              const int k = cb + b < np ? cb + b : np - 1;  // past the last part: a repeat, unused
              const float4* src = reinterpret_cast<const float4*>(p.part_o + part_index(k) * kRepText * kD) + 2 * tid;
              v[b][0] = __ldcg(src);
              v[b][1] = __ldcg(src + 1);
            }
#pragma unroll
            for (int b = 0; b < kMergeBatch; ++b)
              if (cb + b < np) add_part(cb + b, v[b][0], v[b][1]);
          }
        }
        if (!okm) {
          ok = false;
          break;
        }
#pragma unroll
        for (int h = 0; h < kRepText; ++h)
          p.out[l][static_cast<size_t>(kRepText * g + h) * kD + tid] = __float2bfloat16_rn(acc[h]);
        if (tid == 0) p.unit_cnt[s.u] = 0u;  // every part has arrived: ready for the next call
      }
      bar_sync(1, kCompute);  // the merge flag is read before the next segment overwrites it
    }
    first_seg = false;
  }
}

}  // namespace dec

template <int CAP>
__global__ void __launch_bounds__(dec::kThreads, 1) decode_attention_kernel(const __grid_constant__ DecodeParams<CAP> p) {
  using namespace dec;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + SM_BAR;
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + SM_ABORT);
  long long start, end;
  if (p.cluster) {  // one cluster per unit, rank r: tiles [r T / CS, (r + 1) T / CS) of it
    const long long u = blockIdx.x / p.cluster, r = blockIdx.x % p.cluster;
    start = u * p.T + r * p.T / p.cluster;
    end = u * p.T + (r + 1) * p.T / p.cluster;
  } else if (p.per_unit) {  // unit u = blockIdx.x / per_unit, part r: its share of the unit's tiles
    const long long u = blockIdx.x / p.per_unit, r = blockIdx.x % p.per_unit;
    start = u * p.T + r * p.T / p.per_unit;
    end = u * p.T + (r + 1) * p.T / p.per_unit;
  } else {
    start = cta_tile_start(blockIdx.x, p.W, gridDim.x);
    end = cta_tile_start(blockIdx.x + 1, p.W, gridDim.x);
  }
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int b = 0; b < kStages; ++b) {
      mbar_init(bar0 + 8 * (B_FULL + b), 1);
      mbar_init(bar0 + 8 * (B_EMPTY + b), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar0 + 8 * (B_SDONE + b), 1);
      mbar_init(bar0 + 8 * (B_PFULL + b), 1);
      mbar_init(bar0 + 8 * (B_ODONE + b), 1);
    }
    mbar_init(bar0 + 8 * B_QFULL, 1);
    mbar_init(bar0 + 8 * B_OFREE, 1);
    mbar_init(bar0 + 8 * B_TAIL, 1);
    mbar_init(bar0 + 8 * B_DRAIN, 1);
    mbar_init(bar0 + 8 * B_MERGE, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  // rows 8-15 of the Q operand and of both P operands are the zero padding of N = 16
  for (int i = threadIdx.x; i < 3 * 2 * 64; i += kThreads) {
    const uint32_t op = SM_QT + (i >> 7) * 2 * kOpAtom;  // QT, PT[0], PT[1] are contiguous
    const uint32_t off = op + ((i >> 6) & 1) * kOpAtom + 1024 + (i & 63) * 16;
    st_shared_v4(sbase + off, 0u, 0u, 0u, 0u);
  }
  if (warp == 0) {
    tmem_alloc(sbase + SM_TMEM, kTmemCols);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + SM_TMEM);
  if (warp == 5 && (threadIdx.x & 31) == 0) {
    // While the preceding kernel finishes, the MMA thread (idle until the first Q) asks for the
    // tensor maps and has L2 fetch the first segment's q row block, gains and (for the unit's
    // last tile) new k and v rows, then the CTA's first tiles (hints only: the loads after the
    // wait read whatever that kernel wrote). Not the producer: it would reach its first load
    // only once these requests are accepted.
    if (start < end) {
      const int u = static_cast<int>(start / p.T), l = u / kHkv, g = u % kHkv;
      prefetch_tensormap(&p.kmap[l]);
      prefetch_tensormap(&p.vmap[l]);
      prefetch_l2_bulk(p.q_raw[l] + static_cast<size_t>(kRepText * g) * kD, kRepText * kD * 2u);
      prefetch_l2_bulk(p.q_gamma[l], kD * 2u);
      if (end - static_cast<long long>(u) * p.T >= p.T) {  // the segment holds the unit's last tile
        prefetch_l2_bulk(p.k_raw[l] + static_cast<size_t>(g) * kD, kD * 2u);
        prefetch_l2_bulk(p.v_raw[l] + static_cast<size_t>(g) * kD, kD * 2u);
        prefetch_l2_bulk(p.k_gamma[l], kD * 2u);
      }
    }
    for (long long x = start; x < end && x < start + kStages; ++x) {
      const int u = static_cast<int>(x / p.T), j = static_cast<int>(x - static_cast<long long>(u) * p.T);
      const int l = u / kHkv, g = u % kHkv;
      const int rows = p.Smax - j * kKeyTile < kKeyTile ? p.Smax - j * kKeyTile : kKeyTile;
      const size_t off = (static_cast<size_t>(g) * p.Smax + static_cast<size_t>(j) * kKeyTile) * kD;
      prefetch_l2_bulk(p.kc[l] + off, static_cast<uint32_t>(rows) * kD * 2);
      prefetch_l2_bulk(p.vc[l] + off, static_cast<uint32_t>(rows) * kD * 2);
    }
  }
  // everything below reads what earlier kernels in the stream wrote (inputs, caches)
  pdl_wait_primary();
  if (warp < 4) {
    compute(p, sbase, smem, tmem, start, end, abort_flag);
  } else if (warp == 4 && (threadIdx.x & 31) == 0) {
    producer(p, sbase, start, end, abort_flag);
  } else if (warp == 5 && (threadIdx.x & 31) == 0) {
    mma_issuer(p, sbase, tmem, start, end, abort_flag);
  }
  pdl_launch_dependents();  // (a CTA whose producer gave up early has not triggered yet)
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (p.cluster) {
    // every CTA of the cluster has its partial (or an empty one) in shared memory. The cluster's
    // CS (2..8) CTAs share the unit's 256 output chunks (head h, channels 4 c .. 4 c + 3, chunk
    // 32 h + c): rank r takes chunks [r Q, r Q + Q), Q = ceil(256 / CS), one per thread, each
    // read as one 16-byte load from every part (consecutive threads, consecutive chunks). Every
    // thread of every CTA reaches both cluster barriers exactly once.
    cluster_sync();
    const uint32_t cs = static_cast<uint32_t>(p.cluster), r = cluster_ctarank();
    float2* lml = reinterpret_cast<float2*>(smem + SM_PARTML);  // the parts' (max, sum) [part][head]
    if (threadIdx.x < cs * kRepText)
      lml[threadIdx.x] = ld_shared_cluster_v2(
          mapa_shared(sbase + SM_CPART_ML + (threadIdx.x % kRepText) * 8, threadIdx.x / kRepText));
    __syncthreads();
    const uint32_t q = (256u + cs - 1) / cs, chunk = r * q + threadIdx.x;
    if (threadIdx.x < q && chunk < 256u) {
      const int u = blockIdx.x / p.cluster, l = u / kHkv, g = u % kHkv;
      const uint32_t h = chunk >> 5;
      float4 ov[kMaxCluster];  // the chunk in part k
#pragma unroll
      for (uint32_t k = 0; k < kMaxCluster; ++k)
        if (k < cs) ov[k] = ld_shared_cluster_v4(mapa_shared(sbase + SM_CPART + chunk * 16, k));
      float M = -INFINITY, L = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (uint32_t k = 0; k < kMaxCluster; ++k)
        if (k < cs) M = fmaxf(M, lml[k * kRepText + h].x);
#pragma unroll
      for (uint32_t k = 0; k < kMaxCluster; ++k)
        if (k < cs && lml[k * kRepText + h].x != -INFINITY) {  // parts without tiles add nothing
          const float wgt = ex2_approx(lml[k * kRepText + h].x - M);
          L = fmaf(lml[k * kRepText + h].y, wgt, L);
          acc.x = fmaf(ov[k].x, wgt, acc.x);
          acc.y = fmaf(ov[k].y, wgt, acc.y);
          acc.z = fmaf(ov[k].z, wgt, acc.z);
          acc.w = fmaf(ov[k].w, wgt, acc.w);
        }
      const float inv = 1.0f / L;
      *reinterpret_cast<uint2*>(p.out[l] + static_cast<size_t>(kRepText * g) * kD + 4 * chunk) =
          make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
    }
    cluster_sync_exit();  // no CTA leaves while another still reads its shared memory
  }
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

cudaError_t decode_set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(decode_attention_kernel<kSmallCap>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(dec::kSmemBytes));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(decode_attention_kernel<kDecodeMaxLayers>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(dec::kSmemBytes));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(decode_attention_kernel<kSmallCap>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

template <int CAP>
cudaError_t launch_decode_kernel(const DecodeParams<CAP>& dp, cudaLaunchConfig_t cfg) {
  cfg.blockDim = dim3(dec::kThreads);
  cfg.dynamicSmemBytes = dec::kSmemBytes;
  return cudaLaunchKernelEx(&cfg, decode_attention_kernel<CAP>, dp);
}
template cudaError_t launch_decode_kernel<kSmallCap>(const DecodeParams<kSmallCap>&, cudaLaunchConfig_t);
template cudaError_t launch_decode_kernel<kDecodeMaxLayers>(const DecodeParams<kDecodeMaxLayers>&,
                                                            cudaLaunchConfig_t);

}  // namespace ea
