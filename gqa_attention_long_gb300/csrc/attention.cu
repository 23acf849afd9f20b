// attention.cu — K2: persistent split-KV expert attention on the sm_103a tensor cores.
//
// What it computes (alpamayo_tt/expert.py, TTExpert.attention_core; alpamayo_tt/EXPERT_NOTES.md,
// "Attention over the VLM cache: masking approach"): for every (layer, kv head g) unit, the 128
// folded query rows (q heads 2g and 2g+1 x 64 tokens, RMSNormed and roped) attend to cache rows
// [0, S) and to the 64 own rows, softmax(Q K^T / sqrt(128)) V. Hidden rows [S, Smax-64) are
// masked; the mask is derived from row indices. With a bf16 cache the kernel also does the
// layer's prologue itself (q/k RMSNorm, RoPE, own rows into the cache tail).
//
// Work decomposition: the key tiles of all units (ceil(S/128) tiles of 128 cache rows, then one
// 64-row tile of own rows) are laid out unit-major and cut into one contiguous range per CTA
// (grid = number of SMs, one CTA per SM). A CTA walks its range as "segments" (the part of one
// unit inside the range). A segment that covers a whole unit writes the bf16 output directly;
// a partial one writes a normalised fp32 partial plus its log2-sum-exp per row. When every
// split unit has two parts, the part that finishes second merges the first one's partial into
// its own output here; otherwise the log-sum-exp merge kernel (merge.cu) combines the partials
// once this grid has finished.
//
// Two key streams per CTA: the CTA's tiles alternate between stream 0 (even tile count) and
// stream 1 (odd), each with its own TMEM score buffer, its own TMEM accumulator and its own
// softmax warpgroup with its own running max and sum, so that one warpgroup's exponentials
// overlap the other's TMEM traffic and waits (the softmax, not the tensor core, limits a CTA).
// At the end of a segment the two warpgroups exchange their row statistics through shared
// memory and each writes half of the output columns of the combined rows.
//
// Warp roles (384 threads):
//   warps 0-3, 4-7  softmax of stream 0, 1: thread r of a warpgroup owns folded row r (= TMEM
//              lane r); online softmax in fp32 with lazy rescaling of its TMEM accumulator; P
//              written back to TMEM as bf16 (f16 for an e4m3 cache) over the scores it came
//              from, and read from there by the PV MMA. With a bf16 cache these 256 threads
//              first prepare the CTA's first segment: its unit's own rows (if it holds them) and
//              its Q, with rotation angles computed before the kernel waits for the preceding one.
//   warp 8     K/V producer: one thread issues 3-D TMA loads of the K/V tiles (cache rows, and the
//              unit's own rows from the cache tail) into the ring
//   warp 9     MMA: one thread issues tcgen05.mma (S = Q K^T from shared memory into the score
//              buffer of the tile's stream; O += P V with P from TMEM and V from shared memory
//              into the stream's accumulator) and tcgen05.commit to the barriers
//   warps 10-11  bf16: Q and own-row prep (64 threads): per later segment, RMSNorm + RoPE of the
//              unit's raw q rows straight into one of two Q buffers, one segment ahead, so the
//              K/V stream never waits for it; for a later segment holding the own-row tile, the
//              roped K and the V rows into the cache tail. e4m3: one thread of warp 10 bulk-copies
//              the Q codes that the prologue kernel staged.
// Shared memory: Q x2 (64 KB), K/V ring (bf16: 5 x 32 KB; e4m3: 6 x 16 KB plus two 32 KB f16
// copies of V), barriers, a 1.5 KB row-statistics exchange.
// TMEM: 512 columns (two 128-column score/P buffers, two 128-column fp32 accumulators).
#include "internal.cuh"
#include "merge.cuh"
#include "ptx.cuh"
#include "rope.cuh"

namespace ea {
namespace attn {

constexpr int kThreads = 384;
constexpr int kPrepThreads = 64;  // bf16: warps 10 and 11
constexpr int kSoftmaxThreads = 256;
// named barriers: 0 __syncthreads, 1 prep warps, 2 softmax warps, 3 stream 1's warpgroup (own rows)
constexpr uint32_t kOwnRowsBar = 3;

// Shared-memory layout of one CTA. bf16 cache: a K or V tile is 128 rows x 256 bytes, stored as
// two 16 KB swizzle atoms (channels 0-63, 64-127). e4m3 cache: 128 rows x 128 bytes, one atom;
// each stream also has a 32 KB buffer where its softmax warpgroup widens the V tile to f16 (the
// bf16 tile layout), the B operand of the f16 PV MMA.
template <bool F8>
struct Lay {
  static constexpr uint32_t kQ = kQTileBytes;  // one roped Q tile (e4m3: high then low codes)
  static constexpr uint32_t kSlot = F8 ? 16384u : 32768u;           // one K or V tile
  static constexpr uint32_t kAtom = 16384u;                         // 16-bit tiles: second channel half
  static constexpr int kRing = F8 ? 6 : 5;  // e4m3: even, so ring slot parity = K (even) / V (odd)
  static constexpr uint32_t SM_Q = 0;  // two Q buffers
  static constexpr uint32_t SM_RING = SM_Q + 2 * kQ;
  static constexpr uint32_t SM_V16 = SM_RING + kRing * kSlot;  // e4m3: two widened V tiles
  static constexpr uint32_t SM_BAR = SM_V16 + (F8 ? 2u * 32768u : 0u);
  // per-stream barriers (SFULL, PFULL, ODONE) are indexed by the stream; X1, X2 and OFREE
  // complete once per segment (row-statistics exchange and release of the accumulators)
  static constexpr int B_QFULL = 0, B_QEMPTY = 2, B_KVFULL = 4, B_KVEMPTY = 4 + kRing,
                       B_SFULL = 4 + 2 * kRing, B_PFULL = B_SFULL + 2, B_ODONE = B_PFULL + 2,
                       B_X1 = B_ODONE + 2, B_X2 = B_X1 + 1, B_OFREE = B_X2 + 1,
                       B_STAGED = B_OFREE + 1, B_TAILRDY = B_STAGED + 2, B_DRAIN = B_TAILRDY + 2,
                       B_OWNRAW = B_DRAIN + 1, kNumBars = B_OWNRAW + 1;
  static constexpr uint32_t SM_XCH = SM_BAR + kNumBars * 8;  // three floats per folded row
  static constexpr uint32_t SM_ROLE = SM_XCH + kRows * 12;    // in-kernel merge role
  static constexpr uint32_t SM_SFLAG = SM_ROLE + 4;            // per Q buffer: output staged
  static constexpr uint32_t SM_TMEM = SM_SFLAG + 8;
  static constexpr uint32_t SM_ABORT = SM_TMEM + 4;
  static constexpr uint32_t kSmemBytes = SM_ABORT + 4 + 1024;  // + slack to align the base
  static_assert(kSmemBytes <= 232448, "shared memory budget of one sm_103 CTA");
};

#define EA_LAYOUT_ALIASES                                                                  \
  using LY = Lay<F8>;                                                                      \
  constexpr int kRing = LY::kRing;                                                         \
  constexpr uint32_t kSlotBytes = LY::kSlot, kAtom = LY::kAtom, kQB = LY::kQ;              \
  constexpr uint32_t SM_Q = LY::SM_Q, SM_RING = LY::SM_RING, SM_V16 = LY::SM_V16;          \
  constexpr int B_QFULL = LY::B_QFULL, B_QEMPTY = LY::B_QEMPTY, B_KVFULL = LY::B_KVFULL,   \
                B_KVEMPTY = LY::B_KVEMPTY, B_SFULL = LY::B_SFULL, B_PFULL = LY::B_PFULL,    \
                B_ODONE = LY::B_ODONE, B_X1 = LY::B_X1, B_X2 = LY::B_X2,                   \
                B_OFREE = LY::B_OFREE, B_STAGED = LY::B_STAGED, B_TAILRDY = LY::B_TAILRDY,  \
                B_DRAIN = LY::B_DRAIN;                                                     \
  (void)kRing; (void)kSlotBytes; (void)kAtom; (void)kQB; (void)SM_Q; (void)SM_RING; (void)SM_V16; \
  (void)B_QFULL; (void)B_QEMPTY; (void)B_KVFULL; (void)B_KVEMPTY; (void)B_SFULL;            \
  (void)B_PFULL; (void)B_ODONE; (void)B_X1; (void)B_X2; (void)B_OFREE; (void)B_STAGED;          \
  (void)B_TAILRDY; (void)B_DRAIN

constexpr uint32_t TM_S = 0;    // score buffers of streams 0 and 1 at columns 0 and 128; P(n)
                                // overwrites the first columns of the buffer that held S(n)
constexpr uint32_t TM_O = 256;  // accumulators of streams 0 and 1 at columns 256 and 384
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t kAtomBytes = 16384u;  // one 64-channel half of a 16-bit operand tile

struct Seg {
  int u, j0, j1;  // unit and its key-tile range [j0, j1)
};

// Next segment of a CTA's tile range, in range order: t is the next tile, end the range end.
__device__ __forceinline__ bool next_seg(long long& t, long long end, int T, Seg& s) {
  if (t >= end) return false;
  // tile indices stay below 2^31 (at most 64 layers x 8 heads x (Smax/128 + 1) tiles), so the
  // division is a 32-bit one
  const int ti = static_cast<int>(t);
  s.u = ti / T;
  s.j0 = ti - s.u * T;
  const long long j1 = s.j0 + (end - t);
  s.j1 = static_cast<int>(j1 < T ? j1 : T);
  t += s.j1 - s.j0;
  return true;
}

struct Ctx {
  uint8_t* smem;  // generic address of the aligned shared-memory base
  uint32_t sbase;
  uint32_t tmem;
  volatile uint32_t* abort_flag;
  uint32_t* status;
  long long start, end;
  uint32_t bar_base;  // shared address of barrier 0
  __device__ __forceinline__ uint32_t bar(int i) const { return bar_base + 8u * i; }
};

// bf16: when the CTA's first segment holds its unit's own-row tile and that tile's K and V ring
// positions fall in the ring's first round (the slots are still empty), the softmax threads
// write the roped K rows and the V rows straight into those slots (and to the cache tail, for
// the caller), and the producer skips both loads; otherwise the rows go through the cache tail
// and the producer fetches them back by TMA once TAILRDY says they are written.
template <class PP>
__device__ __forceinline__ bool own_rows_direct(const PP& p, const Seg& first) {
  return first.j1 == p.T && 2 * (first.j1 - 1 - first.j0) + 1 < Lay<false>::kRing;
}

// ------------------------------------------------------------------------------- producer
template <bool F8, class PP>
__device__ __noinline__ void producer(const PP& p, const Ctx cx) {
  EA_LAYOUT_ALIASES;
  pdl_wait_primary();  // e4m3: roped Q and the cache's own rows are written by the prologue kernel
  const uint64_t pol_stream = l2_policy_evict_first();  // cache tiles are read exactly once
  uint32_t ring = 0, n_own = 0;
  bool ok = true;
  long long t = cx.start;
  Seg s;
  bool first = true;
  while (ok && next_seg(t, cx.end, p.T, s)) {
    const int l = s.u / kHkv, g = s.u % kHkv;
    const bool direct = !F8 && first && own_rows_direct(p, s);
    first = false;
    for (int j = s.j0; j < s.j1 && ok; ++j) {
      if (direct && j >= p.n_main) {  // filled by the softmax threads
        ring += 2;
        continue;
      }
      if (!F8 && j >= p.n_main) {
        // bf16 own-row tile: its rows are written into the cache tail by this CTA's prep warps
        ok = bounded_wait(cx.bar(B_TAILRDY + (n_own & 1)), (n_own >> 1) & 1, cx.abort_flag,
                          cx.status, kErrProducerWait);
        if (!ok) break;
        fence_proxy_async_global();
        ++n_own;
      }
      for (int h = 0; h < 2; ++h) {  // h = 0: K tile, h = 1: V tile
        const uint32_t slot = ring % kRing, round = ring / kRing;
        if (round > 0) {
          ok = bounded_wait(cx.bar(B_KVEMPTY + slot), (round - 1) & 1, cx.abort_flag, cx.status,
                            kErrProducerWait);
          if (!ok) break;
        }
        const uint32_t dst = cx.sbase + SM_RING + slot * kSlotBytes;
        const uint32_t fb = cx.bar(B_KVFULL + slot);
        // cache tile j: rows [128 j, 128 j + 128) of head g (keys >= S of the last one are masked,
        // and their V rows zeroed, by the softmax); own-row tile: rows [Smax - 64, Smax), the
        // box's rows past Smax arriving as zeros
        const int row0 = j < p.n_main ? j * kKeyTile : p.Smax - kTok;
        mbar_expect_tx(fb, kSlotBytes);
        const CUtensorMap* m = h ? &p.vmap[l] : &p.kmap[l];
        tma_load_3d(dst, m, fb, 0, row0, g, pol_stream);
        if constexpr (!F8) tma_load_3d(dst + kAtom, m, fb, 64, row0, g, pol_stream);
        ++ring;
      }
    }
  }
  pdl_launch_dependents();
  if (!ok) {
    // Let every copy already issued land before the CTA gives its shared memory back.
    for (uint32_t k = 0; k < static_cast<uint32_t>(kRing) && k < ring; ++k) {
      const uint32_t pos = ring - 1 - k;
      if (!drain_wait(cx.bar(B_KVFULL + pos % kRing), (pos / kRing) & 1)) atomicOr(cx.status, kErrDrain);
    }
  }
}

// ------------------------------------------------------------------- staged-output store
// A segment that produced bf16 output rows staged them in its Q buffer (row-major, the 32 KB
// block of out that its unit u owns): one thread stores them with one bulk copy and waits until
// the copy has read the buffer, which may then be refilled.
template <bool F8, class PP>
__device__ __forceinline__ bool drain_staged(const PP& p, const Ctx& cx, int sg, int u) {
  EA_LAYOUT_ALIASES;
  const int b = sg & 1;
  volatile uint32_t* sflag = reinterpret_cast<volatile uint32_t*>(cx.smem + LY::SM_SFLAG);
  if (!bounded_wait(cx.bar(B_STAGED + b), (sg >> 1) & 1, cx.abort_flag, cx.status, kErrProducerWait))
    return false;
  if (sflag[b] != 0u) {
    bulk_store(p.out[u / kHkv] + static_cast<size_t>(u % kHkv) * kRows * kD, cx.sbase + SM_Q + b * kQB,
               kRows * kD * 2);
    bulk_commit();
  }
  bulk_wait_read0();
  return true;
}

// ------------------------------------------------------------------------ Q loader (e4m3)
// One thread brings each segment's roped e4m3 Q (high and low codes, written by the prologue
// kernel) into one of the two Q buffers, one segment ahead.
template <bool F8, class PP>
__device__ __noinline__ void q_loader(const PP& p, const Ctx cx) {
  EA_LAYOUT_ALIASES;
  const uint64_t pol_keep = l2_policy_evict_last();
  int seg = 0;
  int hist_u[2] = {0, 0};  // units of the last two segments, by Q buffer
  bool ok = true;
  long long t = cx.start;
  Seg s;
  while (ok && next_seg(t, cx.end, p.T, s)) {
    const int qb = seg & 1;
    if (seg >= 2) {  // segment seg-2 has finished with buffer qb (its last QK and its output)
      ok = bounded_wait(cx.bar(B_QEMPTY + qb), ((seg >> 1) - 1) & 1, cx.abort_flag, cx.status,
                        kErrProducerWait);
      if (ok) ok = drain_staged<F8>(p, cx, seg - 2, hist_u[qb]);
    }
    if (!ok) break;
    hist_u[qb] = s.u;
    mbar_expect_tx(cx.bar(B_QFULL + qb), kQB);
    bulk_load(cx.sbase + SM_Q + qb * kQB, p.q_ws + static_cast<size_t>(s.u) * kQTileBytes, kQB,
              cx.bar(B_QFULL + qb), pol_keep);
    ++seg;
  }
  for (int sg = seg >= 2 ? seg - 2 : 0; ok && sg < seg; ++sg) ok = drain_staged<F8>(p, cx, sg, hist_u[sg & 1]);
  bulk_wait_all0();
  if (!ok) {  // let the last load into each buffer land
    for (int b = 0; b < 2; ++b) {
      int last = seg - 1;
      if ((last & 1) != b) --last;
      if (last >= 0 && !drain_wait(cx.bar(B_QFULL + b), (last >> 1) & 1))
        atomicOr(cx.status, kErrDrain);
    }
  }
}

// ---------------------------------------------------------------- Q and own-row prep (bf16)
// alpamayo_tt/expert.py, TTExpert.layer and TTExpert.set_context: per-head RMSNorm of q and k
// (eps 1e-6, q_norm / k_norm gains), HF rotate_half RoPE at positions t + rope_delta + S, and the
// own K/V rows written into the cache at rows [Smax - 64, Smax).
//
// Rows are handled by octets of threads: lane i of an octet holds channels [8i, 8i + 8) and
// their RoPE partners [64 + 8i, 64 + 8i + 8), so that the rotation is in-thread and a row's norm
// takes three shuffles; every global access is a 16-byte vector access. The roped Q goes to a Q
// buffer in the 128-byte-swizzled K-major layout the QK MMA reads.
//
// The first segment's Q is prepared by the 256 softmax threads, which have nothing else to do
// until its first scores; later segments' Q, one segment ahead of the MMA, and the own K/V rows
// of the segment that holds a unit's own-row tile are prepared by warps 10 and 11. The loops
// over rows are straight-line code, so that the rows' load, shuffle and arithmetic latencies
// overlap.

// Roped row (hh, tok) of q heads 2g, 2g + 1 from its raw chunks: stored into the Q buffer at
// folded row hh * 64 + tok; returns the two output chunks.
__device__ __forceinline__ void q_row_to_smem(uint32_t qbuf, int hh, int tok, int i, const uint4 lo,
                                              const uint4 hi, const float (&gl)[8],
                                              const float (&gh)[8], const float (&cs)[8],
                                              const float (&sn)[8], uint4& ql, uint4& qh) {
  float xl[8], xh[8], yl[8], yh[8];
  unpack_bf16x8(lo, xl);
  unpack_bf16x8(hi, xh);
  norm_rope(xl, xh, gl, gh, cs, sn, yl, yh);
  ql = pack8(yl, false);
  qh = pack8(yh, false);
  const int r = hh * kTok + tok;
  st_shared_v4(qbuf + swz_off(r, i, kQTileBytes / 2), ql.x, ql.y, ql.z, ql.w);
  st_shared_v4(qbuf + swz_off(r, i + 8, kQTileBytes / 2), qh.x, qh.y, qh.z, qh.w);
}

// cos/sin of token tok at the eight frequencies whose inverse frequencies are ih + il.
template <class PP>
__device__ __forceinline__ void token_cos_sin(const PP& p, int tok, const float (&ih)[8], const float (&il)[8],
                                              float (&cs)[8], float (&sn)[8]) {
#pragma unroll
  for (int e = 0; e < 8; ++e) rope_cos_sin(p.rope_base + tok, ih[e], il[e], cs[e], sn[e]);
}

// cos/sin of the two tokens (oc, oc + 32) whose rows a softmax thread prepares in the first
// segment, at its eight frequencies [8i, 8i + 8). The positions depend only on the token index, S
// and rope_delta, so this runs before the kernel waits for the preceding one.
// Stream 1's threads also take the angles of tokens oc - 16 and oc + 16 (xcs, xsn), which they
// need for the own K rows when the first segment holds its unit's own-row tile.
template <class PP>
__device__ __forceinline__ void first_angles(const PP& p, float (&cs)[2][8], float (&sn)[2][8],
                                             float (&xcs)[2][8], float (&xsn)[2][8], bool own) {
  const int oc = threadIdx.x >> 3, dl = 8 * (threadIdx.x & 7);
  float ih[8], il[8];
  load_inv8(p.inv_hi, p.inv_lo, dl, ih, il);
  token_cos_sin(p, oc, ih, il, cs[0], sn[0]);
  token_cos_sin(p, oc + 32, ih, il, cs[1], sn[1]);
  if (own && threadIdx.x >= 128) {
    token_cos_sin(p, oc - 16, ih, il, xcs[0], xsn[0]);
    token_cos_sin(p, oc + 16, ih, il, xcs[1], xsn[1]);
  }
}

// The first segment's rows by the 256 softmax threads (32 octets, octet oc: tokens oc and oc + 32,
// whose rotation angles the threads already hold): the Q rows of both heads into Q buffer 0
// (QFULL). When that segment holds its unit's own-row tile, stream 1's warpgroup then writes
// the roped K rows and the V rows of all 64 tokens (its octet oc takes tokens oc - 16, oc,
// oc + 16, oc + 32; it computes the angles of the two it did not hold) into the cache tail and,
// when they fit the ring's first round (own_rows_direct), straight into the two ring slots of
// that tile as well (KVFULL; no fetch back), else TAILRDY for the producer to fetch them.
// Stream 0's warpgroup goes on to its first tile meanwhile: in a two-tile segment that is the
// last cache tile, whose keys >= S it masks, so the CTA no longer waits for both tasks in turn.
template <class PP>
__device__ __forceinline__ void first_q_prep(const PP& p, const Ctx& cx, const float (&cs)[2][8],
                                             const float (&sn)[2][8], const float (&xcs)[2][8],
                                             const float (&xsn)[2][8]) {
  long long t = cx.start;
  Seg s;
  if (!next_seg(t, cx.end, p.T, s)) return;
  const int oc = threadIdx.x >> 3, i = threadIdx.x & 7;
  const int dl = 8 * i, dh = 64 + 8 * i;
  const int l = s.u / kHkv, g = s.u % kHkv;
  const bool own = s.j1 == p.T;
  const bool own_rows = own && threadIdx.x >= 128;  // stream 1's warpgroup
  const bool direct = own && own_rows_direct(p, s);
  const uint32_t n_tile = static_cast<uint32_t>(s.j1 - 1 - s.j0);  // CTA tile index of the own-row tile
  const uint32_t kslot = cx.sbase + Lay<false>::SM_RING + (2 * n_tile) * Lay<false>::kSlot;
  const uint32_t vslot = kslot + Lay<false>::kSlot;
  const size_t unit_rows = static_cast<size_t>(g) * kTok * kD;
  if (direct && threadIdx.x == 128) {
    // The raw own K and V rows (64 x 256 bytes each) by bulk copy into the rows of their ring
    // slots that the 64-key tile never reads (rows 64-127 of each 64-channel atom): raw rows
    // 0-31 into atom 0, rows 32-63 into atom 1, 8 KB each.
    const uint32_t bar = cx.bar(Lay<false>::B_OWNRAW);
    const uint64_t pol = l2_policy_evict_first();
    mbar_expect_tx(bar, 4u * 8192u);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      bulk_load(kslot + h * kAtomBytes + 8192u, p.k_raw[l] + unit_rows + h * 32 * kD, 8192u, bar, pol);
      bulk_load(vslot + h * kAtomBytes + 8192u, p.v_raw[l] + unit_rows + h * 32 * kD, 8192u, bar, pol);
    }
  }
  const __nv_bfloat16* qsrc = p.q_raw[l] + static_cast<size_t>(2 * g) * kTok * kD + oc * kD;
  // every row of both tokens is requested at once
  uint4 raw[2][2][2];  // [token][head][lo, hi]
#pragma unroll
  for (int tt = 0; tt < 2; ++tt)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const __nv_bfloat16* row = qsrc + static_cast<size_t>(hh * kTok + 32 * tt) * kD;
      raw[tt][hh][0] = *reinterpret_cast<const uint4*>(row + dl);
      raw[tt][hh][1] = *reinterpret_cast<const uint4*>(row + dh);
    }
  float gl[8], gh[8];
  unpack_bf16x8(*reinterpret_cast<const uint4*>(p.q_gamma[l] + dl), gl);
  unpack_bf16x8(*reinterpret_cast<const uint4*>(p.q_gamma[l] + dh), gh);
  const uint32_t qbuf = cx.sbase + Lay<false>::SM_Q;
  // the optional roped q output is written by the CTA that holds the unit's own-row tile
  __nv_bfloat16* qr0 = own ? p.q_rope[l] : nullptr;
  if (qr0 != nullptr) qr0 += (static_cast<size_t>(2 * g) * kTok + oc) * kD;
#pragma unroll
  for (int tt = 0; tt < 2; ++tt) {
    const int tok = oc + 32 * tt;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      uint4 ql, qh;
      q_row_to_smem(qbuf, hh, tok, i, raw[tt][hh][0], raw[tt][hh][1], gl, gh, cs[tt], sn[tt], ql, qh);
      if (qr0 != nullptr) {
        __nv_bfloat16* qr = qr0 + static_cast<size_t>(hh * kTok + 32 * tt) * kD;
        *reinterpret_cast<uint4*>(qr + dl) = ql;
        *reinterpret_cast<uint4*>(qr + dh) = qh;
      }
    }
  }
  fence_proxy_async_smem();  // Q is read by the tensor core (async proxy)
  bar_sync(2, kSoftmaxThreads);
  if (threadIdx.x == 0) mbar_arrive(cx.bar(Lay<false>::B_QFULL));
  if (!own_rows) return;
  // K rows: RMSNorm with the k_norm gain and RoPE; V rows as given; into cache rows Smax - 64 + t
  // of head g, and (direct) into the own-row tile's K and V ring slots, row t in the swizzled
  // layout the TMA would have produced (rows 64-127 of the slots are never read). The raw rows
  // (in L2 since before the dependency wait) are requested at once, tokens oc - 16 + 16 m.
  // (the angles of tokens oc - 16 and oc + 16 were computed before the dependency wait, in
  // xcs, xsn; those of oc and oc + 32 are in cs, sn)
  const __nv_bfloat16* ksrc = p.k_raw[l] + unit_rows;
  const __nv_bfloat16* vsrc = p.v_raw[l] + unit_rows;
  const uint4 kg0 = *reinterpret_cast<const uint4*>(p.k_gamma[l] + dl);
  const uint4 kg1 = *reinterpret_cast<const uint4*>(p.k_gamma[l] + dh);
  // raw row tok in shared memory (direct: where the bulk copies put it)
  auto raw_row = [&](uint32_t slot, int tok) -> uint32_t {
    return slot + static_cast<uint32_t>(tok >> 5) * kAtomBytes + 8192u + static_cast<uint32_t>(tok & 31) * 256u;
  };
  uint4 kr[4][2];
  if (direct) {
    if (!bounded_wait(cx.bar(Lay<false>::B_OWNRAW), 0, cx.abort_flag, cx.status, kErrSoftmaxWait)) {
      // the copies land before the CTA can give its shared memory back
      if (!drain_wait(cx.bar(Lay<false>::B_OWNRAW), 0)) atomicOr(cx.status, kErrDrain);
      return;
    }
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const uint32_t a = raw_row(kslot, oc - 16 + 16 * m);
      kr[m][0] = ld_shared_v4(a + 16 * i);
      kr[m][1] = ld_shared_v4(a + 128 + 16 * i);
    }
  } else {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const size_t ro = static_cast<size_t>(oc - 16 + 16 * m) * kD;
      kr[m][0] = *reinterpret_cast<const uint4*>(ksrc + ro + dl);
      kr[m][1] = *reinterpret_cast<const uint4*>(ksrc + ro + dh);
    }
  }
  unpack_bf16x8(kg0, gl);
  unpack_bf16x8(kg1, gh);
  const size_t tail = (static_cast<size_t>(g) * p.Smax + (p.Smax - kTok)) * kD;
  uint4 kst[4][2];  // the roped K rows, kept for the cache tail
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int tok = oc - 16 + 16 * m;
    const size_t ro = tail + static_cast<size_t>(tok) * kD;
    float xl[8], xh[8], yl[8], yh[8], c8[8], s8[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {  // m is a compile-time index: these are register moves
      c8[e] = (m & 1) ? cs[m >> 1][e] : xcs[m >> 1][e];
      s8[e] = (m & 1) ? sn[m >> 1][e] : xsn[m >> 1][e];
    }
    unpack_bf16x8(kr[m][0], xl);
    unpack_bf16x8(kr[m][1], xh);
    norm_rope(xl, xh, gl, gh, c8, s8, yl, yh);
    const uint4 kl = pack8(yl, false), kh = pack8(yh, false);
    kst[m][0] = kl;
    kst[m][1] = kh;
    if (direct) {  // the cache tail is written after the slots are handed to the MMA
      st_shared_v4(kslot + swz_off(tok, i, kAtomBytes), kl.x, kl.y, kl.z, kl.w);
      st_shared_v4(kslot + swz_off(tok, i + 8, kAtomBytes), kh.x, kh.y, kh.z, kh.w);
    } else {
      *reinterpret_cast<uint4*>(p.kc[l] + ro + dl) = kl;
      *reinterpret_cast<uint4*>(p.kc[l] + ro + dh) = kh;
    }
  }
  uint4 vr[4][2];
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    if (direct) {
      const uint32_t a = raw_row(vslot, oc - 16 + 16 * m);
      vr[m][0] = ld_shared_v4(a + 16 * i);
      vr[m][1] = ld_shared_v4(a + 128 + 16 * i);
    } else {
      const size_t ro = static_cast<size_t>(oc - 16 + 16 * m) * kD;
      vr[m][0] = *reinterpret_cast<const uint4*>(vsrc + ro + dl);
      vr[m][1] = *reinterpret_cast<const uint4*>(vsrc + ro + dh);
    }
  }
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int tok = oc - 16 + 16 * m;
    if (direct) {
      const uint4 vl = vr[m][0], vh = vr[m][1];
      st_shared_v4(vslot + swz_off(tok, i, kAtomBytes), vl.x, vl.y, vl.z, vl.w);
      st_shared_v4(vslot + swz_off(tok, i + 8, kAtomBytes), vh.x, vh.y, vh.z, vh.w);
    } else {
      const size_t ro = tail + static_cast<size_t>(tok) * kD;
      *reinterpret_cast<uint4*>(p.vc[l] + ro + dl) = vr[m][0];
      *reinterpret_cast<uint4*>(p.vc[l] + ro + dh) = vr[m][1];
    }
  }
  if (direct) {
    fence_proxy_async_smem();  // the slots are read by the tensor core (async proxy)
    bar_sync(kOwnRowsBar, 128);
    if (threadIdx.x == 128) {
      mbar_arrive(cx.bar(Lay<false>::B_KVFULL + 2 * n_tile));
      mbar_arrive(cx.bar(Lay<false>::B_KVFULL + 2 * n_tile + 1));
    }
    // Then the cache tail, for the caller, from registers (global stores queue behind the
    // cache stream in the memory system, so they stay off the path to the first MMA; the slots
    // themselves may be refilled as soon as the MMA is done with them).
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int tok = oc - 16 + 16 * m;
      const size_t ro = tail + static_cast<size_t>(tok) * kD;
      *reinterpret_cast<uint4*>(p.kc[l] + ro + dl) = kst[m][0];
      *reinterpret_cast<uint4*>(p.kc[l] + ro + dh) = kst[m][1];
      *reinterpret_cast<uint4*>(p.vc[l] + ro + dl) = vr[m][0];
      *reinterpret_cast<uint4*>(p.vc[l] + ro + dh) = vr[m][1];
    }
  } else {
    fence_proxy_async_global();  // the rows are read back by TMA (async proxy)
    bar_sync(kOwnRowsBar, 128);
    if (threadIdx.x == 128) mbar_arrive(cx.bar(Lay<false>::B_TAILRDY));
  }
}

// Before the kernel waits for the preceding one (programmatic dependent launch), one thread
// asks for the tensor maps of its first segment's layer and has L2 fetch that segment's first
// cache tiles (at most kEarlyTiles; not the own-row tile, whose rows this kernel writes). A
// prefetch reads nothing into the CTA, so a preceding kernel that writes those rows later cannot
// make it wrong: the loads after the wait see the current rows. The thread is not the producer,
// which would otherwise reach its first load only once these requests are accepted.
constexpr int kEarlyTiles = 3;

// bf16, before the wait as well: L2 fetch of the layer inputs that the first segment's
// preparation reads right after it, requested ahead of the cache tiles so that those loads do
// not queue behind the tiles: the unit's q rows (both heads, 32 KB contiguous), the q gain and,
// when the segment holds the unit's own-row tile, its raw k and v rows (16 KB each) and the k
// gain. The preceding kernel may still be writing them; its writes land in L2 as well.
template <class PP>
__device__ __noinline__ void early_inputs(const PP& p, const Ctx cx) {
  long long t = cx.start;
  Seg s;
  if (!next_seg(t, cx.end, p.T, s)) return;
  const int l = s.u / kHkv, g = s.u % kHkv;
  prefetch_l2_bulk(p.q_raw[l] + static_cast<size_t>(2 * g) * kTok * kD, 2u * kTok * kD * 2u);
  prefetch_l2_bulk(p.q_gamma[l], kD * 2u);
  if (s.j1 == p.T) {
    prefetch_l2_bulk(p.k_raw[l] + static_cast<size_t>(g) * kTok * kD, kTok * kD * 2u);
    prefetch_l2_bulk(p.v_raw[l] + static_cast<size_t>(g) * kTok * kD, kTok * kD * 2u);
    prefetch_l2_bulk(p.k_gamma[l], kD * 2u);
  }
}
template <bool F8, class PP>
__device__ __noinline__ void early_prefetch(const PP& p, const Ctx cx) {
  long long t = cx.start;
  Seg s;
  if (!next_seg(t, cx.end, p.T, s)) return;
  const int l = s.u / kHkv, g = s.u % kHkv;
  prefetch_tensormap(&p.kmap[l]);
  prefetch_tensormap(&p.vmap[l]);
  for (int j = s.j0, k = 0; j < s.j1 && j < p.n_main && k < kEarlyTiles; ++j, ++k) {
    tma_prefetch_3d(&p.kmap[l], 0, j * kKeyTile, g);
    tma_prefetch_3d(&p.vmap[l], 0, j * kKeyTile, g);
    if constexpr (!F8) {
      tma_prefetch_3d(&p.kmap[l], 64, j * kKeyTile, g);
      tma_prefetch_3d(&p.vmap[l], 64, j * kKeyTile, g);
    }
  }
}

// Warps 10 and 11 (64 threads, 8 octets; octet oc: tokens oc + 8 it, it < 8). A pass handles
// one token, with the raw rows of the next kAhead tokens already requested.
constexpr int kAhead = 1;
template <class PP>
__device__ __noinline__ void prep_warps(const PP& p, const Ctx cx) {
  constexpr bool F8 = false;
  EA_LAYOUT_ALIASES;
  const int px = static_cast<int>(threadIdx.x) - (kThreads - kPrepThreads);
  const int oc = px >> 3, i = px & 7;
  const int dl = 8 * i, dh = 64 + 8 * i;
  int hist_u[2] = {0, 0};  // units of the last two segments, by Q buffer
  int seg = 0, n_own = 0, cur_l = -1;
  float gql[8], gqh[8];
  float ih[8], il[8];  // this thread's eight RoPE inverse frequencies, read once
  load_inv8(p.inv_hi, p.inv_lo, dl, ih, il);
  bool ok = true;
  long long t = cx.start;
  Seg s;
  // raw rows of a segment's unit into L2 ahead of their use: q (both heads, 32 KB) unless it is
  // the first segment (read at once by the softmax threads), and k and v (16 KB each) if the
  // segment holds the own-row tile
  auto prefetch = [&](const Seg& x, bool q) {
    const int l = x.u / kHkv, g = x.u % kHkv;
    if (q) prefetch_l2_bulk(p.q_raw[l] + static_cast<size_t>(2 * g) * kTok * kD, 2 * kTok * kD * 2);
    if (x.j1 == p.T) {
      prefetch_l2_bulk(p.k_raw[l] + static_cast<size_t>(g) * kTok * kD, kTok * kD * 2);
      prefetch_l2_bulk(p.v_raw[l] + static_cast<size_t>(g) * kTok * kD, kTok * kD * 2);
    }
  };
  while (next_seg(t, cx.end, p.T, s)) {
    const int qb = seg & 1;
    bool good = true;
    if (px == 0) {
      long long t2 = t;
      Seg s2;
      if (next_seg(t2, cx.end, p.T, s2)) prefetch(s2, true);
      if (seg >= 2) {
        // segment seg-2 has finished with buffer qb: its last QK is done and its output stored
        good = bounded_wait(cx.bar(B_QEMPTY + qb), ((seg >> 1) - 1) & 1, cx.abort_flag, cx.status,
                            kErrProducerWait);
        if (good) good = drain_staged<F8>(p, cx, seg - 2, hist_u[qb]);
      }
    }
    ok = bar_sync_and(1, kPrepThreads, good);
    if (!ok) break;
    hist_u[qb] = s.u;
    const int l = s.u / kHkv, g = s.u % kHkv;
    const bool own = s.j1 == p.T;  // this segment holds the unit's own-row tile
    if (seg > 0) {
      if (l != cur_l) {
        unpack_bf16x8(*reinterpret_cast<const uint4*>(p.q_gamma[l] + dl), gql);
        unpack_bf16x8(*reinterpret_cast<const uint4*>(p.q_gamma[l] + dh), gqh);
        cur_l = l;
      }
      const __nv_bfloat16* qsrc = p.q_raw[l] + static_cast<size_t>(2 * g) * kTok * kD;
      __nv_bfloat16* qr0 = own ? p.q_rope[l] : nullptr;  // optional; one CTA per unit writes it
      if (qr0 != nullptr) qr0 += static_cast<size_t>(2 * g) * kTok * kD;
      const uint32_t qbuf = cx.sbase + SM_Q + qb * kQB;
      // one token (both heads' rows) per pass, with the rows of the next kAhead tokens in flight
      // (rotated through registers): a short loop body, which stays in the instruction cache
      uint4 nx[kAhead][2][2];
#pragma unroll
      for (int a = 0; a < kAhead; ++a)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const __nv_bfloat16* row = qsrc + static_cast<size_t>(hh * kTok + oc + 8 * a) * kD;
          nx[a][hh][0] = *reinterpret_cast<const uint4*>(row + dl);
          nx[a][hh][1] = *reinterpret_cast<const uint4*>(row + dh);
        }
#pragma unroll 1
      for (int it = 0; it < 8; ++it) {
        const int tok = oc + 8 * it;
        uint4 cur[2][2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          cur[hh][0] = nx[0][hh][0];
          cur[hh][1] = nx[0][hh][1];
#pragma unroll
          for (int a = 0; a + 1 < kAhead; ++a) {
            nx[a][hh][0] = nx[a + 1][hh][0];
            nx[a][hh][1] = nx[a + 1][hh][1];
          }
        }
        const int nt = oc + 8 * (it + kAhead < 8 ? it + kAhead : 7);  // past the end: token 7 again
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const __nv_bfloat16* row = qsrc + static_cast<size_t>(hh * kTok + nt) * kD;
          nx[kAhead - 1][hh][0] = *reinterpret_cast<const uint4*>(row + dl);
          nx[kAhead - 1][hh][1] = *reinterpret_cast<const uint4*>(row + dh);
        }
        float cs[8], sn[8];
        token_cos_sin(p, tok, ih, il, cs, sn);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint4 ql, qh;
          q_row_to_smem(qbuf, hh, tok, i, cur[hh][0], cur[hh][1], gql, gqh, cs, sn, ql, qh);
          if (qr0 != nullptr) {
            __nv_bfloat16* qr = qr0 + static_cast<size_t>(hh * kTok + tok) * kD;
            *reinterpret_cast<uint4*>(qr + dl) = ql;
            *reinterpret_cast<uint4*>(qr + dh) = qh;
          }
        }
      }
      fence_proxy_async_smem();  // Q is read by the tensor core (async proxy)
      bar_sync(1, kPrepThreads);
      if (px == 0) mbar_arrive(cx.bar(B_QFULL + qb));
    }
    if (own && seg == 0 && !own_rows_direct(p, s)) ++n_own;  // written by the softmax threads
    if (own && seg > 0) {
      // K rows: RMSNorm with the k_norm gain and RoPE; V rows: as given; both into cache rows
      // Smax - 64 + t of head g, which the producer then loads as the own-row tile
      float gkl[8], gkh[8];
      unpack_bf16x8(*reinterpret_cast<const uint4*>(p.k_gamma[l] + dl), gkl);
      unpack_bf16x8(*reinterpret_cast<const uint4*>(p.k_gamma[l] + dh), gkh);
      const size_t tail = (static_cast<size_t>(g) * p.Smax + (p.Smax - kTok)) * kD;
      const __nv_bfloat16* ksrc = p.k_raw[l] + static_cast<size_t>(g) * kTok * kD;
      const __nv_bfloat16* vsrc = p.v_raw[l] + static_cast<size_t>(g) * kTok * kD;
      __nv_bfloat16* kdst = p.kc[l] + tail;
      __nv_bfloat16* vdst = p.vc[l] + tail;
      uint4 nk[kAhead][2], nv[kAhead][2];  // rows of the next kAhead tokens, in flight
#pragma unroll
      for (int a = 0; a < kAhead; ++a) {
        const size_t ro = static_cast<size_t>(oc + 8 * a) * kD;
        nk[a][0] = *reinterpret_cast<const uint4*>(ksrc + ro + dl);
        nk[a][1] = *reinterpret_cast<const uint4*>(ksrc + ro + dh);
        nv[a][0] = *reinterpret_cast<const uint4*>(vsrc + ro + dl);
        nv[a][1] = *reinterpret_cast<const uint4*>(vsrc + ro + dh);
      }
#pragma unroll 1
      for (int it = 0; it < 8; ++it) {
        const int tok = oc + 8 * it;
        const uint4 k0 = nk[0][0], k1 = nk[0][1], v0 = nv[0][0], v1 = nv[0][1];
#pragma unroll
        for (int a = 0; a + 1 < kAhead; ++a) {
          nk[a][0] = nk[a + 1][0];
          nk[a][1] = nk[a + 1][1];
          nv[a][0] = nv[a + 1][0];
          nv[a][1] = nv[a + 1][1];
        }
        const size_t rn = static_cast<size_t>(oc + 8 * (it + kAhead < 8 ? it + kAhead : 7)) * kD;
        nk[kAhead - 1][0] = *reinterpret_cast<const uint4*>(ksrc + rn + dl);
        nk[kAhead - 1][1] = *reinterpret_cast<const uint4*>(ksrc + rn + dh);
        nv[kAhead - 1][0] = *reinterpret_cast<const uint4*>(vsrc + rn + dl);
        nv[kAhead - 1][1] = *reinterpret_cast<const uint4*>(vsrc + rn + dh);
        const size_t ro = static_cast<size_t>(tok) * kD;
        float cs[8], sn[8], xl[8], xh[8], yl[8], yh[8];
        token_cos_sin(p, tok, ih, il, cs, sn);
        unpack_bf16x8(k0, xl);
        unpack_bf16x8(k1, xh);
        norm_rope(xl, xh, gkl, gkh, cs, sn, yl, yh);
        *reinterpret_cast<uint4*>(kdst + ro + dl) = pack8(yl, false);
        *reinterpret_cast<uint4*>(kdst + ro + dh) = pack8(yh, false);
        *reinterpret_cast<uint4*>(vdst + ro + dl) = v0;
        *reinterpret_cast<uint4*>(vdst + ro + dh) = v1;
      }
      fence_proxy_async_global();  // the rows are read back by TMA (async proxy)
      bar_sync(1, kPrepThreads);
      if (px == 0) mbar_arrive(cx.bar(B_TAILRDY + (n_own & 1)));
      ++n_own;
    }
    ++seg;
  }
  if (px == 0) {
    for (int sg = seg >= 2 ? seg - 2 : 0; ok && sg < seg; ++sg)
      ok = drain_staged<F8>(p, cx, sg, hist_u[sg & 1]);
    bulk_wait_all0();
  }
}

// ------------------------------------------------------------------------------------ MMA
// Per segment, step i (0 <= i <= nt) has up to two MMAs to issue: QK(i) (if i < nt) and PV(i-1)
// (if i > 0). Tile n of the CTA (counted over all its segments) belongs to stream n & 1: QK(n)
// writes that stream's score buffer, PV(n) accumulates into that stream's accumulator. QK(n) is
// issued only after PV(n-2), the previous MMA that read the same buffer, has completed; so a
// completed S(n) also tells the softmax that every earlier PV of its stream is done. The two MMAs
// of a step belong to different streams (different TMEM buffers, ring slots and barriers), so
// whichever has its inputs first is issued first: PV(i-1) does not wait behind QK(i), whose
// inputs (K(i), and the completion of PV(i-2)) may arrive later than P(i-1).
template <bool F8, class PP>
__device__ __noinline__ void mma_issuer(const PP& p, const Ctx cx) {
  EA_LAYOUT_ALIASES;
  // bf16: format code 1 (kind::f16); e4m3: format code 0 (kind::f8f6f4). V is MN-major.
  constexpr uint32_t kIdescQK128 = umma_idesc_f16(128, 128, !F8, false, false);
  constexpr uint32_t kIdescQK64 = umma_idesc_f16(128, 64, !F8, false, false);
  // PV: bf16 P and V, or (e4m3 cache) f16 P and the f16-widened V; V is MN-major
  constexpr uint32_t kIdescPV = umma_idesc_f16(128, 128, !F8, false, true);
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
    const uint32_t qaddr = cx.sbase + SM_Q + qb * kQB;
    const int nt = s.j1 - s.j0;
    // Inputs of QK(i): K(i) in its ring slot; PV(n_qk - 2) complete, since QK(n) overwrites the
    // score buffer whose first columns hold P(n-2), the A operand of PV(n-2) (even and odd PVs
    // complete on separate barriers; this thread observes every PV completion in order).
    auto qk_ready = [&](int i) -> bool {
      const uint32_t pos = ring + 2 * i;
      if (!mbar_test_wait(cx.bar(B_KVFULL + pos % kRing), (pos / kRing) & 1)) return false;
      return n_qk < 2 || mbar_test_wait(cx.bar(B_ODONE + ((n_qk - 2) & 1)), ((n_qk - 2) >> 1) & 1);
    };
    auto issue_qk = [&](int i) {
      const int j = s.j0 + i;
      const uint32_t slot = (ring + 2 * i) % kRing;
      tc_fence_after();
      const uint32_t kaddr = cx.sbase + SM_RING + slot * kSlotBytes;
      const uint32_t d = cx.tmem + TM_S + (n_qk & 1) * 128;
      const uint32_t idesc = j < p.n_main ? kIdescQK128 : kIdescQK64;
      if constexpr (F8) {
        // 4 steps of 32 channels within the 128-byte atom, for the high Q codes and then the
        // low ones (same scale), both accumulating into S
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_f8_ss(d, sw128_desc(qaddr + (kk >> 2) * kQTileBytesF8 + (kk & 3) * 32, 16, 1024),
                     sw128_desc(kaddr + (kk & 3) * 32, 16, 1024), idesc, kk > 0);
      } else {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {  // 8 steps of 16 channels; 4 per 64-channel atom
          const uint32_t off = (kk >> 2) * kAtom + (kk & 3) * 32;
          umma_f16_ss(d, sw128_desc(qaddr + off, 16, 1024), sw128_desc(kaddr + off, 16, 1024),
                      idesc, kk > 0);
        }
      }
      umma_commit(cx.bar(B_SFULL + (n_qk & 1)));
      umma_commit(cx.bar(B_KVEMPTY + slot));
      if (i == nt - 1) umma_commit(cx.bar(B_QEMPTY + qb));
      ++n_qk;
    };
    // Inputs of PV(ii): the softmax warpgroup's P(ii) (P of even and odd tiles arrive on separate
    // barriers); bf16: V(ii) in its ring slot (e4m3: the stream's widened copy, written before the
    // warpgroup arrived on PFULL); for the first PV of a segment, which overwrites both
    // accumulators' previous contents, the softmax warpgroups' release of the previous segment's
    // accumulators (OFREE completes once per segment).
    auto pv_ready = [&](int ii) -> bool {
      if (ii == 0 && seg > 0 && !mbar_test_wait(cx.bar(B_OFREE), (seg - 1) & 1)) return false;
      if (!mbar_test_wait(cx.bar(B_PFULL + (n_pv & 1)), (n_pv >> 1) & 1)) return false;
      if constexpr (!F8) {
        const uint32_t pos = ring + 2 * ii + 1;
        if (!mbar_test_wait(cx.bar(B_KVFULL + pos % kRing), (pos / kRing) & 1)) return false;
      }
      return true;
    };
    auto issue_pv = [&](int ii) {
      const int j = s.j0 + ii;
      const uint32_t slot = (ring + 2 * ii + 1) % kRing;
      tc_fence_after();
      const uint32_t vaddr = F8 ? cx.sbase + SM_V16 + (n_pv & 1) * 32768u
                                : cx.sbase + SM_RING + slot * kSlotBytes;
      // P(ii) sits in TMEM, in the score buffer of QK(ii) (PV and QK counts advance together),
      // as 16-bit pairs: a K step of 16 keys spans 8 TMEM columns
      const uint32_t pcol = cx.tmem + TM_S + (n_pv & 1) * 128;
      // the first PV of each stream in a segment (segment tiles 0 and 1) starts a fresh sum
      const uint32_t ocol = cx.tmem + TM_O + (n_pv & 1) * 128;
      const int nk = j < p.n_main ? 8 : 4;  // 16 keys per step; the own-row tile has 64 keys
      for (int kk = 0; kk < nk; ++kk)        // V: 16 key rows of 128 bytes per step and atom
        umma_f16_ts(ocol, pcol + kk * 8, sw128_desc(vaddr + kk * 16 * 128, kAtom, 1024), kIdescPV,
                    (ii > 1 || kk > 0));
      // even and odd PVs complete on separate barriers: a waiter that knows PV k-2 is done
      // can then always tell PV k's completion from an older phase
      umma_commit(cx.bar(B_ODONE + (n_pv & 1)));
      if constexpr (!F8) umma_commit(cx.bar(B_KVEMPTY + slot));
      ++n_pv;
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
        // Nothing to issue: suspend on the barrier the next MMA most likely waits for, for at
        // most ~0.3 us, then look at both again (a spinning thread takes issue slots from the
        // softmax warps that share its SM sub-partition).
        if (pv_todo)
          mbar_try_wait_hint(cx.bar(B_PFULL + (n_pv & 1)), (n_pv >> 1) & 1, 300);
        else if (n_qk >= 2)
          mbar_try_wait_hint(cx.bar(B_ODONE + ((n_qk - 2) & 1)), ((n_qk - 2) >> 1) & 1, 300);
        // bounded like every other wait: the CTA's abort flag, a time limit and a poll limit
        if ((it & 63u) == 0) {
          if (*cx.abort_flag) {
            ok = false;
            break;
          }
          const uint64_t now = globaltimer_ns();
          if (t0 == 0) t0 = now;
          if (now - t0 > kWaitLimitNs || it >= 0x7fffffc0u) {
            *cx.abort_flag = 1u;
            atomicOr(cx.status, kErrMmaWait);
            ok = false;
            break;
          }
        }
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

// The rare rescale of a running max move while a chunk's scores are live in registers: the
// stream's accumulator O (128 columns) if it holds earlier tiles, and the current tile's P of
// the earlier chunk (32 columns of 16-bit pairs) if there is one. Kept out of line, so that only
// this path pays for the registers it needs.
template <bool F8>
__device__ __noinline__ void rescale_rare(uint32_t o_addr, uint32_t p_addr, float alpha, bool do_o, bool do_p) {
  if (do_o) rescale_O(o_addr, alpha);
  if (do_p) {
    uint32_t q[32];
    tmem_ld32(p_addr, q);
    tmem_wait_ld();
    reg_fence32(q);
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      float2 f;
      if constexpr (F8) {
        f = __half22float2(*reinterpret_cast<const __half2*>(&q[e]));
      } else {
        f = make_float2(__uint_as_float(q[e] << 16), __uint_as_float(q[e] & 0xFFFF0000u));
      }
      q[e] = F8 ? pack_f16x2(f.x * alpha, f.y * alpha) : pack_bf16x2(f.x * alpha, f.y * alpha);
    }
    tmem_st32(p_addr, q);
    tmem_wait_st();
  }
}

template <bool F8, class PP>
__device__ __noinline__ void softmax_warps(const PP& p, const Ctx cx) {
  EA_LAYOUT_ALIASES;
  const int k = threadIdx.x >> 7;   // stream of this warpgroup
  const int r = threadIdx.x & 127;  // folded row = TMEM lane
  const uint32_t lane_addr = static_cast<uint32_t>(r & ~31) << 16;
  const uint32_t s_col = TM_S + k * 128, o_col = TM_O + k * 128;
  const uint32_t pa_base = cx.tmem + lane_addr + s_col;  // P(n) of this stream
  const float c = p.scale_log2;
  float* xw = reinterpret_cast<float*>(cx.smem + LY::SM_XCH) + 3 * r;  // this row's exchange slot
  volatile uint32_t* role = reinterpret_cast<volatile uint32_t*>(cx.smem + LY::SM_ROLE);
  volatile uint32_t* sflag = reinterpret_cast<volatile uint32_t*>(cx.smem + LY::SM_SFLAG);
  uint32_t base = 0, seg = 0;  // tiles of this CTA before the current segment; segment count
  bool ok = true, first_seg = true;
  long long t = cx.start;
  Seg s;

  // warp-uniform outcome: the TMEM loads and shuffles that follow need the full warp
  auto wait_bar = [&](int b, uint32_t parity) -> bool {
    return __all_sync(0xffffffffu, bounded_wait(cx.bar(b), parity, cx.abort_flag, cx.status,
                                                kErrSoftmaxWait));
  };

  while (ok && next_seg(t, cx.end, p.T, s)) {
    const int l = s.u / kHkv, g = s.u % kHkv;
    const int nt = s.j1 - s.j0;
    float m_ref = -INFINITY, lsum = 0.f;
    // FP8: e4m3 Q row scale, and the unit's reference V scale (P is stored relative to it)
    float sq = 1.f, svr = 1.f;
    if constexpr (F8) {
      sq = p.q_scale[static_cast<size_t>(s.u) * kRows + r];
      svr = p.sv_ref[s.u];
    }
    int last_n = -1;  // last tile of this stream in the segment (-1: none yet)
    // In-kernel merge of a two-part unit (see the epilogue): the leader counts this part's
    // arrival now and polls the other part's ready flag once per tile, each load consumed one
    // tile later, so that neither round trip lands on the epilogue.
    const bool full = (s.j0 == 0 && s.j1 == p.T);
    const bool fused = !full && p.fused_merge != 0;
    const bool leader = threadIdx.x == 0;
    uint32_t* usync = p.unit_sync + 2 * static_cast<size_t>(s.u);  // [arrivals, ready]
    uint32_t arr_old = 0u, flag_pend = 0u, flag_seen = 0u;
    if (fused && leader) arr_old = atomicAdd(usync, 1u);
    // segment tile i is CTA tile base + i and belongs to stream (base + i) & 1
    for (int i = (k - static_cast<int>(base)) & 1; i < nt; i += 2) {
      const int n = static_cast<int>(base) + i;
      const int j = s.j0 + i;
      if (fused && leader) {
        flag_seen |= flag_pend;
        flag_pend = ld_relaxed_gpu(usync + 1);
      }
      if constexpr (F8) {
        // e4m3 cache: widen V(n) to f16 in the stream's buffer while QK(n) runs. The buffer
        // held V(n-2): wait until PV(n-2) has read it (PV(n-4) is known complete, since S(n-2)
        // was). V(n) is ring position 2n + 1; the slot is released once it has been read.
        if (n >= 2) ok = wait_bar(B_ODONE + k, ((n - 2) >> 1) & 1);
        const uint32_t vpos = 2 * static_cast<uint32_t>(n) + 1, vslot = vpos % kRing;
        if (ok) ok = wait_bar(B_KVFULL + vslot, (vpos / kRing) & 1);
        if (!ok) break;
        if (j < p.n_main || r < kTok) {  // the own-row tile has 64 keys
          const uint32_t src = cx.sbase + SM_RING + vslot * kSlotBytes + r * 128;
          const uint32_t dst = cx.sbase + SM_V16 + k * 32768u + r * 128;
          const int sw = r & 7;
          // rows of keys >= S in the last cache tile (hidden rows, any content) become zeros
          const bool live = j >= p.n_main || j * kKeyTile + r < p.S;
#pragma unroll
          for (int c = 0; c < 8; ++c) {  // 16-byte chunk c: channels 16c .. 16c + 15
            uint4 v = ld_shared_v4(src + 16 * (c ^ sw));
            if (!live) v = make_uint4(0u, 0u, 0u, 0u);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t h[8];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              h[2 * q] = cvt_f16x2_e4m3x2(static_cast<uint16_t>(w[q] & 0xFFFFu));
              h[2 * q + 1] = cvt_f16x2_e4m3x2(static_cast<uint16_t>(w[q] >> 16));
            }
            // f16 channels 16c .. 16c + 15: atom c / 4, 8-channel chunks 2 (c % 4) and + 1
            const uint32_t atom = dst + (c >> 2) * kAtom;
            const int d0 = 2 * (c & 3);
            st_shared_v4(atom + 16 * (d0 ^ sw), h[0], h[1], h[2], h[3]);
            st_shared_v4(atom + 16 * ((d0 + 1) ^ sw), h[4], h[5], h[6], h[7]);
          }
        }
        fence_proxy_async_smem();  // the f16 tile is read by the tensor core (async proxy)
        mbar_arrive(cx.bar(B_KVEMPTY + vslot));
      }
      ok = wait_bar(B_SFULL + k, (n >> 1) & 1);
      if (!ok) break;
      tc_fence_after();
      const bool tail = j >= p.n_main;
      const uint32_t sa = cx.tmem + lane_addr + s_col;
      // The score row is read in chunks of 64 columns (a cache tile has two, the 64-key own-row
      // tile one), each in one pass: its max, then its exponentials against the running max, so
      // that no more than 64 scores are live per thread (two softmax warpgroups share the
      // register file). The running max moves (lazily, see kLazy) when a chunk's max exceeds it.
      const int npair = tail ? 1 : 2;
      const int key0 = j * kKeyTile;
      const bool ragged = !tail && key0 + kKeyTile > p.S;  // keys >= S (hidden rows) are masked
      auto load_pair = [&](int pr, uint32_t (&v)[2][32]) {
        tmem_ld32(sa + 64 * pr, v[0]);
        tmem_ld32(sa + 64 * pr + 32, v[1]);
        tmem_wait_ld();
        reg_fence32(v[0]);
        reg_fence32(v[1]);
        if (ragged) {
#pragma unroll
          for (int ch = 0; ch < 2; ++ch)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (key0 + 64 * pr + 32 * ch + e >= p.S) v[ch][e] = __float_as_uint(-INFINITY);
        }
      };
      // per-tile factors: scores in log2 units are s * ct; FP8 adds the block scales, and P is
      // stored as 2^(x - m) * (sv / svr) (exponent offset lgv) so that it carries the tile's V
      // scale relative to the unit's largest one (V itself stays as its e4m3 code values); the
      // row sum counts 2^(x - m).
      float ct = c, lgv = 0.f, lmul = 1.f;
      if constexpr (F8) {
        const int col = tail ? p.ncol - 1 : j;
        const float sk = p.ks[l][g * p.ncol + col], sv = p.vs[l][g * p.ncol + col];
        ct = c * sq * sk;
        lgv = __log2f(sv / svr);
        lmul = svr / sv;
      }
      float2 ts4[4];  // row sum of this tile with 4 independent pairs of accumulators
#pragma unroll
      for (int q = 0; q < 4; ++q) ts4[q] = make_float2(0.f, 0.f);
      const float2 ct2 = make_float2(ct, ct);
      // P(n) goes to TMEM over the columns of S(n). Chunk pr's P lands in columns [32 pr,
      // 32 pr + 32), which hold scores of chunks <= pr, already read. The buffer's previous P,
      // P(n-2), was consumed by PV(n-2), which completed before QK(n).
#pragma unroll 1
      for (int pr = 0; pr < npair; ++pr) {
        uint32_t v[2][32];
        load_pair(pr, v);
        // the chunk's max with 8 independent accumulators
        float mx8[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) mx8[q] = -INFINITY;
#pragma unroll
        for (int ch = 0; ch < 2; ++ch)
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            mx8[(e >> 1) & 7] = fmax3(mx8[(e >> 1) & 7], __uint_as_float(v[ch][e]), __uint_as_float(v[ch][e + 1]));
        const float mc = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                               fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) * ct;
        // a chunk 0 always holds a live key (key0 < S), so m_ref is finite after it
        const bool need = (m_ref == -INFINITY) || (mc > m_ref + kLazy);
        if (__any_sync(0xffffffffu, need)) {
          const float m_new = fmaxf(m_ref, mc);
          const float alpha = ex2_approx(m_ref - m_new);  // 0 for the segment's first chunk
          // S(n) is complete, so PV(n-2) and every earlier PV of this stream are done: the
          // accumulator is stable and holds this stream's tiles before n; this tile's P of the
          // earlier chunk, already in TMEM columns [0, 32), moves too. The chunk's scores are
          // not kept in registers across that (rare) step: they are read again from TMEM,
          // where they stay until this chunk's P is written.
          if (last_n >= 0 || pr > 0) {
            rescale_rare<F8>(cx.tmem + lane_addr + o_col, pa_base, alpha, last_n >= 0, pr > 0);
            load_pair(pr, v);
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) ts4[q] = make_float2(ts4[q].x * alpha, ts4[q].y * alpha);
          lsum *= alpha;
          m_ref = m_new;
        }
        const float neg = lgv - m_ref;
        const float2 neg2 = make_float2(neg, neg);
        // 16-bit pairs (bf16; f16 for an e4m3 cache, whose V is widened to f16): column c of
        // the chunk's P block holds keys 2c and 2c + 1
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {  // 32 keys -> 16 TMEM columns at a time
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            // two keys per packed fma (x * ct + neg, one rounding each, as fmaf)
            const float2 x = __ffma2_rn(
                make_float2(__uint_as_float(v[ch][2 * e]), __uint_as_float(v[ch][2 * e + 1])), ct2, neg2);
            const float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
            ts4[e & 3] = __fadd2_rn(ts4[e & 3], make_float2(p0, p1));
            pk[e] = F8 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
          }
          tmem_st16(pa_base + 32 * pr + 16 * ch, pk);
        }
      }
      lsum += (((ts4[0].x + ts4[0].y) + (ts4[1].x + ts4[1].y)) + ((ts4[2].x + ts4[2].y) + (ts4[3].x + ts4[3].y))) * lmul;
      if constexpr (!F8) {
        if (ragged) {
          // the last cache tile: V rows of keys >= S (hidden rows, any content, NaN included)
          // become zeros before PV reads them, as P is 0 there
          const uint32_t vpos = 2 * static_cast<uint32_t>(n) + 1, vslot = vpos % kRing;
          ok = wait_bar(B_KVFULL + vslot, (vpos / kRing) & 1);
          if (!ok) break;
          if (key0 + r >= p.S) {
            const uint32_t row = cx.sbase + SM_RING + vslot * kSlotBytes + r * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              st_shared_v4(row + 16 * c, 0u, 0u, 0u, 0u);
              st_shared_v4(row + kAtom + 16 * c, 0u, 0u, 0u, 0u);
            }
          }
          fence_proxy_async_smem();
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(cx.bar(B_PFULL + k));
      last_n = n;
    }
    if (!ok) break;

    // ---- epilogue. Each stream waits for its last PV (the one before it is done: S(last)
    // completed after it). Stream 1 hands its (max, sum) to stream 0, which forms the row's
    // weights w_k = 2^(m_k - M) * svr / L and hands them back; each warpgroup then writes the
    // combined rows' output columns [64 k, 64 k + 64). A stream without tiles in the segment
    // has m = -inf and weight 0 and its accumulator is not read.
    //
    // A partial segment of a two-part unit (fused_merge) is merged here: the part whose CTA
    // arrives second (a per-unit atomic count) waits for the first part's ready flag, then
    // weights its own rows by 2^(lse - M2) and the first part's normalised partial by
    // 2^(lse_1 - M2) (M2 the larger lse, both over their sum) and writes the bf16 output. The
    // first part writes its partial and raises the flag; it never waits for the other.
    if (last_n >= 0) {
      ok = wait_bar(B_ODONE + k, (last_n >> 1) & 1);
      if (!ok) break;
    }
    const uint32_t sp = seg & 1;
    const bool has0 = nt >= 2 || (base & 1) == 0, has1 = nt >= 2 || (base & 1) == 1;
    const int slot = first_seg ? 0 : 1;  // a partial segment is the CTA's first or its last
    first_seg = false;
    // the other part of a two-part unit: its CTA and partial slot
    const long long ufirst = static_cast<long long>(s.u) * p.T;
    int other = 0, other_slot = 0;
    if (fused) {
      const int c0 = cta_of_tile(ufirst, p.W, gridDim.x);
      other = static_cast<int>(blockIdx.x) == c0 ? c0 + 1 : c0;
      other_slot = cta_tile_start(other, p.W, gridDim.x) >= ufirst ? 0 : 1;
    }
    float w0, w1, w2 = 0.f, lse_row = 0.f;
    bool second = false;
    if (k == 1) {
      xw[0] = m_ref;
      xw[1] = lsum;
      mbar_arrive(cx.bar(B_X1));
      ok = wait_bar(B_X2, sp);
      if (!ok) break;
      w0 = xw[0];
      w1 = xw[1];
      w2 = xw[2];
      // only a second part gives the other part's partial a weight (2^(lse_1 - M2) / sum > 0);
      // the role word itself may already belong to the next segment
      second = w2 != 0.f;
    } else {
      if (leader) {  // the leader also arrives on X1 (its count is 128 + 1), with the role
        uint32_t rl = 0u;
        if (fused && arr_old == 1u) {  // second part: wait until the first part's partial is out
          if ((flag_seen | flag_pend) != 0u) {
            fence_acq_rel_gpu();  // with the relaxed read that saw the flag: an acquire
            rl = 1u;
          } else {
            rl = bounded_flag_wait(usync + 1, cx.abort_flag, cx.status, kErrMergeWait) ? 1u : 2u;
          }
          if (rl == 1u) {
            // both parts are done with the unit's words: leave them zero for the next grid
            reinterpret_cast<volatile uint32_t*>(usync)[0] = 0u;
            reinterpret_cast<volatile uint32_t*>(usync)[1] = 0u;
          }
        }
        *role = rl;
        mbar_arrive(cx.bar(B_X1));
      }
      ok = wait_bar(B_X1, sp);
      if (!ok) break;
      const uint32_t rl = *role;
      if (rl == 2u) {
        ok = false;
        break;
      }
      second = rl == 1u;
      const float mo = xw[0], lo = xw[1];  // stream 1's (max, sum)
      const float M = fmaxf(m_ref, mo);
      const float a0 = has0 ? ex2_approx(m_ref - M) : 0.f;
      const float a1 = has1 ? ex2_approx(mo - M) : 0.f;
      const float L = lsum * a0 + lo * a1;
      const float inv = svr / L;  // FP8: P was stored relative to the reference V scale
      w0 = a0 * inv;
      w1 = a1 * inv;
      lse_row = M + log2f(L);
      if (second) {
        const float lse_o =
            __ldcg(p.part_lse + (static_cast<size_t>(other) * 2 + other_slot) * 3 * kRows + r);
        const float M2 = fmaxf(lse_row, lse_o);
        const float ea = ex2_approx(lse_row - M2), eb = ex2_approx(lse_o - M2);
        const float rs = 1.0f / (ea + eb);
        w0 *= ea * rs;
        w1 *= ea * rs;
        w2 = eb * rs;
      }
      xw[0] = w0;
      xw[1] = w1;
      xw[2] = w2;
      mbar_arrive(cx.bar(B_X2));
    }
    tc_fence_after();
    // ---- this warpgroup's 64 columns of both accumulators, combined (a second part starts from
    // the first part's weighted partial)
    // partials are f16, stored chunk-major (16-byte chunk c of row r at index c * 128 + r), so
    // that a warp's 32 rows of one chunk are 512 contiguous bytes; half row k of a partial is
    // scaled by a power of two whose inverse sits beside the lse
    const size_t oslot = static_cast<size_t>(other) * 2 + other_slot;
    const uint4* pother = p.part_o + oslot * kPartChunks * kRows + static_cast<size_t>(8 * k) * kRows + r;
    const float w2s = second ? w2 * __ldcg(p.part_lse + (oslot * 3 + 1 + k) * kRows + r) : 0.f;
    float o[2][32];
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
      const uint32_t col = cx.tmem + lane_addr + TM_O + 64 * k + 32 * ch;
      if (second) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 v = __ldcg(pother + static_cast<size_t>(4 * ch + q) * kRows);
          const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const float2 f = unpack_f16x2(wv[h]);
            o[ch][8 * q + 2 * h] = f.x * w2s;
            o[ch][8 * q + 2 * h + 1] = f.y * w2s;
          }
        }
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) o[ch][e] = 0.f;
      }
#pragma unroll
      for (int st = 0; st < 2; ++st) {  // the two streams' accumulators, one after the other
        if (st == 0 ? !has0 : !has1) continue;
        uint32_t x[32];
        tmem_ld32(col + 128 * st, x);
        tmem_wait_ld();
        reg_fence32(x);
        const float w = st == 0 ? w0 : w1;
#pragma unroll
        for (int e = 0; e < 32; ++e) o[ch][e] = fmaf(__uint_as_float(x[e]), w, o[ch][e]);
      }
    }
    // The accumulators are read: release them to the next segment's PVs (the MMA issuer waits
    // for all 256 arrivals before the first one).
    tc_fence_before();
    mbar_arrive(cx.bar(B_OFREE));
    const bool staged = full || second;
    if (staged) {
      // bf16 rows into this segment's Q buffer (its last QK is done), row-major like the unit's
      // block of out: row r, columns [64 k, 64 k + 64) at byte r * 256 + 128 k. Store q of a
      // thread writes chunk q ^ (r % 8) (columns 8 c .. 8 c + 7, c = q ^ (r % 8)), so that the
      // eight rows of a warp quarter hit eight different bank groups; the chunks are permuted
      // into that order in registers by three conditional swap stages. The Q loader stores the
      // block with one bulk copy.
      uint32_t w[8][4];
#pragma unroll
      for (int c = 0; c < 8; ++c)
#pragma unroll
        for (int h = 0; h < 4; ++h)
          w[c][h] = pack_bf16x2(o[c >> 2][8 * (c & 3) + 2 * h], o[c >> 2][8 * (c & 3) + 2 * h + 1]);
      const int m = r & 7;
#pragma unroll
      for (int bit = 1; bit < 8; bit <<= 1) {
        const bool sw = (m & bit) != 0;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          if (c & bit) continue;
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const uint32_t a0 = w[c][h], a1 = w[c | bit][h];
            w[c][h] = sw ? a1 : a0;
            w[c | bit][h] = sw ? a0 : a1;
          }
        }
      }
      const uint32_t srow = cx.sbase + SM_Q + (seg & 1) * kQB + r * (kD * 2) + k * 128;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        st_shared_v4(srow + 16 * (q ^ m), w[q][0], w[q][1], w[q][2], w[q][3]);
      fence_proxy_async_smem();  // visible to the bulk copy (async proxy)
    } else {
      // f16, chunk-major (see above): each store instruction of a warp writes 512 contiguous
      // bytes. The half row is scaled by 2^(e - 127), e chosen from the exponent of its largest
      // magnitude so that it lands in [2^14, 2^15) (f16 keeps 11 significant bits there and
      // cannot overflow); a zero or tiny half row takes the largest scale, 2^126. The inverse,
      // also a power of two, is stored beside the lse.
      float mx = 0.f;
#pragma unroll
      for (int ch = 0; ch < 2; ++ch)
#pragma unroll
        for (int e = 0; e < 32; ++e) mx = fmaxf(mx, fabsf(o[ch][e]));
      const int ex = static_cast<int>(__float_as_uint(mx) >> 23) & 0xff;  // mx < 2^(ex - 126)
      const int es = min(max(268 - ex, 1), 253);
      const float sc = __uint_as_float(static_cast<uint32_t>(es) << 23);
      const float isc = __uint_as_float(static_cast<uint32_t>(254 - es) << 23);
      const size_t mslot = static_cast<size_t>(blockIdx.x) * 2 + slot;
      // The chunks go into this segment's Q buffer (its last QK is done) in the global layout,
      // and the leader stores the whole 32 KB partial with one bulk copy: a handful of global
      // store instructions per thread cost more, on this path, than the copy's round trip.
      const uint32_t qst = cx.sbase + SM_Q + (seg & 1) * kQB + static_cast<uint32_t>(8 * k * kRows + r) * 16u;
#pragma unroll
      for (int ch = 0; ch < 2; ++ch)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float* x = &o[ch][8 * q];
          st_shared_v4(qst + static_cast<uint32_t>((4 * ch + q) * kRows) * 16u,
                       pack_f16x2(x[0] * sc, x[1] * sc), pack_f16x2(x[2] * sc, x[3] * sc),
                       pack_f16x2(x[4] * sc, x[5] * sc), pack_f16x2(x[6] * sc, x[7] * sc));
        }
      p.part_lse[(mslot * 3 + 1 + k) * kRows + r] = isc;
      if (k == 0) p.part_lse[mslot * 3 * kRows + r] = lse_row;
      fence_proxy_async_smem();  // the chunks are read by the bulk copy (async proxy)
      bar_sync(2, kSoftmaxThreads);
      if (leader) {
        bulk_store(p.part_o + mslot * kPartChunks * kRows, cx.sbase + SM_Q + (seg & 1) * kQB, kQTileBytes);
        bulk_commit();
        bulk_wait_all0();           // written (and its source read: the buffer may be refilled)
        fence_proxy_async_global();  // ordered before this thread's release of the partial
      }
      // The other threads' lse and scale stores reach the leader's release through the CTA
      // barrier that follows (the flag's STAGED wait, or the grid merge's __syncthreads):
      // release is cumulative.
    }
    if (leader) sflag[seg & 1] = staged ? 1u : 0u;
    mbar_arrive(cx.bar(B_STAGED + (seg & 1)));
    // The leader of a first part waits until every half row of the partial is out, then raises
    // the unit's ready flag.
    if (!staged && fused && leader) {
      ok = bounded_wait(cx.bar(B_STAGED + (seg & 1)), (seg >> 1) & 1, cx.abort_flag, cx.status,
                        kErrSoftmaxWait);
      if (ok) st_release_gpu(usync + 1, 1u);
    }
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    base += nt;
    ++seg;
  }
}

// ------------------------------------------------------------------------- grid-wide merge
// Units cut into more than two parts (a single layer spread over every SM) are merged by the
// grid itself once every CTA has written its partials: each CTA counts its arrival (after a
// GPU-scope fence on its partial stores), one thread waits, bounded, until all CTAs have arrived,
// and then the CTA merges its share of the split units' (unit, 8-column chunk) pairs, three
// pairs at a time (128 threads, one per folded row, per pair). The grid has one CTA per SM at
// most, so every CTA is resident or becomes so as soon as an earlier kernel frees its SM (a
// kernel launched after this one cannot start before every CTA of this grid has started). The
// last CTA to leave resets both counters.
template <bool F8, class PP>
__device__ __noinline__ void grid_merge(const PP& p, const Ctx cx) {
  EA_LAYOUT_ALIASES;
  volatile uint32_t* go = reinterpret_cast<volatile uint32_t*>(cx.smem + LY::SM_ROLE);
  __syncthreads();
  if (threadIdx.x == 0) {
    // the CTA's partial stores (ordered before this thread by the barrier) are visible at GPU
    // scope before the count: a fence cumulative over them, then the arrival
    __threadfence();
    atomicAdd(p.grid_sync, 1u);
    const uint64_t t0 = globaltimer_ns();
    bool ok = false;
    for (uint32_t it = 0; it < 0x80000000u; ++it) {
      uint32_t v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p.grid_sync) : "memory");
      if (v >= gridDim.x) {
        ok = true;
        break;
      }
      if ((it & 15u) == 15u && globaltimer_ns() - t0 > kWaitLimitNs) break;
      __nanosleep(64);
    }
    if (!ok) atomicOr(p.status, kErrMergeWait);
    // the acquire load that saw the full count orders the partial reads after it (the other
    // threads are ordered after this one by the barrier below)
    *go = ok ? 1u : 0u;
  }
  __syncthreads();
  if (*go != 0u) {
    const int P = p.n_split * kPartChunks;
    const int c0 = static_cast<int>(static_cast<long long>(blockIdx.x) * P / gridDim.x);
    const int c1 = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * P / gridDim.x);
    for (int pi = c0 + static_cast<int>(threadIdx.x) / kRows; pi < c1; pi += kThreads / kRows) {
      const SplitUnit su = p.split[pi / kPartChunks];
      merge_row_chunk<20>(p.part_o, p.part_lse, su, pi % kPartChunks, threadIdx.x % kRows,
                          p.out[su.u / kHkv]);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && atomicAdd(p.grid_sync + 1, 1u) == gridDim.x - 1) {
    p.grid_sync[0] = 0u;  // every CTA has passed the wait
    p.grid_sync[1] = 0u;
  }
}

}  // namespace attn

// ------------------------------------------------------------------------------------ kernel
template <bool F8, int CAP>
__global__ void __launch_bounds__(attn::kThreads, 1)
    attention_kernel(const __grid_constant__ AttnParams<CAP> p) {
  using namespace attn;
  EA_LAYOUT_ALIASES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Ctx cx;
  cx.smem = smem;
  cx.sbase = smem_u32(smem);
  cx.bar_base = cx.sbase + LY::SM_BAR;
  cx.abort_flag = reinterpret_cast<volatile uint32_t*>(smem + LY::SM_ABORT);
  cx.status = p.status;
  cx.start = cta_tile_start(blockIdx.x, p.W, gridDim.x);
  cx.end = cta_tile_start(blockIdx.x + 1, p.W, gridDim.x);

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(cx.bar(B_QFULL + b), 1);  // e4m3: the bulk copy; bf16: one thread per preparing group
      mbar_init(cx.bar(B_TAILRDY + b), 1);
      mbar_init(cx.bar(B_QEMPTY + b), 1);
      mbar_init(cx.bar(B_SFULL + b), 1);
      mbar_init(cx.bar(B_PFULL + b), 128);
      mbar_init(cx.bar(B_ODONE + b), 1);
    }
    mbar_init(cx.bar(B_X1), 128 + 1);  // stream 1's threads and stream 0's leader
    mbar_init(cx.bar(B_X2), 128);
    mbar_init(cx.bar(B_OFREE), kSoftmaxThreads);
    mbar_init(cx.bar(B_STAGED), kSoftmaxThreads);
    mbar_init(cx.bar(B_STAGED + 1), kSoftmaxThreads);
    for (int b = 0; b < kRing; ++b) {
      mbar_init(cx.bar(B_KVFULL + b), 1);
      // e4m3: a V slot (odd) is released by the 128 threads of the warpgroup that widened it
      mbar_init(cx.bar(B_KVEMPTY + b), F8 && (b & 1) ? 128 : 1);
    }
    mbar_init(cx.bar(B_DRAIN), 1);
    mbar_init(cx.bar(LY::B_OWNRAW), 1);
    *cx.abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(cx.sbase + LY::SM_TMEM, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cx.tmem = *reinterpret_cast<volatile uint32_t*>(smem + LY::SM_TMEM);
  // Work that reads nothing a preceding kernel writes, done while it may still run.
  float fcs[2][8], fsn[2][8], xcs[2][8], xsn[2][8];
  if (warp == 11 && lane == 0) {
    if constexpr (!F8) early_inputs(p, cx);
    early_prefetch<F8>(p, cx);
  }
  if constexpr (!F8) {
    if (warp < 8) {
      long long t0 = cx.start;
      Seg s0;
      const bool own0 = next_seg(t0, cx.end, p.T, s0) && s0.j1 == p.T;
      first_angles(p, fcs, fsn, xcs, xsn, own0);
    }
  }
  // Everything below reads what earlier kernels in the stream wrote (layer inputs, caches; e4m3:
  // the prologue's staged Q and own rows).
  pdl_wait_primary();

  if (warp < 8) {
    if constexpr (!F8) first_q_prep(p, cx, fcs, fsn, xcs, xsn);
    softmax_warps<F8>(p, cx);
  } else if (warp == 8) {
    if (lane == 0) producer<F8>(p, cx);
  } else if (warp == 9) {
    if (lane == 0) mma_issuer<F8>(p, cx);
  } else if constexpr (F8) {
    if (warp == 10 && lane == 0) q_loader<F8>(p, cx);
  } else {
    prep_warps(p, cx);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(cx.tmem, kTmemCols);
  if (p.grid_merge) grid_merge<F8>(p, cx);
}

// Host side: attributes and launch of the four instances (kept in this file, where the kernel
// template is instantiated).
template <bool F8, int CAP>
static cudaError_t set_smem_attr() {
  return cudaFuncSetAttribute(attention_kernel<F8, CAP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(attn::Lay<F8>::kSmemBytes));
}

cudaError_t attention_set_attributes() {
  cudaError_t e = set_smem_attr<false, kSmallCap>();
  if (e == cudaSuccess) e = set_smem_attr<true, kSmallCap>();
  if (e == cudaSuccess) e = set_smem_attr<false, kMaxLayersPerLaunch>();
  if (e == cudaSuccess) e = set_smem_attr<true, kMaxLayersPerLaunch>();
  return e;
}

template <int CAP>
cudaError_t launch_attention_kernel(const AttnParams<CAP>& ap, bool f8, cudaLaunchConfig_t cfg) {
  cfg.blockDim = dim3(attn::kThreads);
  cfg.dynamicSmemBytes = f8 ? attn::Lay<true>::kSmemBytes : attn::Lay<false>::kSmemBytes;
  return f8 ? cudaLaunchKernelEx(&cfg, attention_kernel<true, CAP>, ap)
            : cudaLaunchKernelEx(&cfg, attention_kernel<false, CAP>, ap);
}
template cudaError_t launch_attention_kernel<kSmallCap>(const AttnParams<kSmallCap>&, bool,
                                                        cudaLaunchConfig_t);
template cudaError_t launch_attention_kernel<kMaxLayersPerLaunch>(
    const AttnParams<kMaxLayersPerLaunch>&, bool, cudaLaunchConfig_t);

}  // namespace ea
