// internal.cuh — constants, kernel parameter blocks and the workspace layout shared by the
// kernels and the host side of libexpert_attn.so.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stddef.h>
#include <stdint.h>

namespace ea {

// Problem dimensions (alpamayo_tt/EXPERT_NOTES.md, section "Layouts"): 16 query heads, 8 KV
// heads, head width 128, 64 expert tokens. Folding the two query heads of a GQA group over the
// token axis gives 128 query rows per KV head (section "Attention over the VLM cache").
constexpr int kHq = 16;
constexpr int kHkv = 8;
constexpr int kD = 128;
constexpr int kTok = 64;
constexpr int kRows = 128;        // folded query rows per KV head: row r = (h % 2) * 64 + t
constexpr int kKeyTile = 128;     // cache rows per key tile
constexpr int kMaxLayersPerLaunch = 64;
// Kernel parameter blocks come in two capacities: calls with few layers use the small one, so
// that their launches carry ~2 KB of parameters instead of ~19 KB.
constexpr int kSmallCap = 8;
constexpr int kScaleBlock = 128;  // FP8 scale granularity (rows)
constexpr int kPartChunks = kD / 8;  // 16-byte chunks (8 f16 columns) per row of a partial output

// Bytes of one staged operand tile in the 128-byte-swizzled K-major layout: two 64-column
// halves ("atoms"), each [rows][128 bytes]; inside every 8-row group of 1024 bytes the 16-byte
// chunks of row r are permuted as chunk' = chunk ^ (r % 8).
constexpr uint32_t kQTileBytes = kRows * kD * 2;          // 32 KB: roped Q of one (layer, kv head)
// FP8 (e4m3) variant: one 128-byte swizzle atom per row, so a Q tile is 16 KB (high codes, then
// low codes in the next 16 KB of the same workspace slot).
constexpr uint32_t kQTileBytesF8 = kRows * kD;

// Status bits recorded in the workspace when a bounded wait gives up.
enum : uint32_t {
  kErrProducerWait = 1u << 0,
  kErrMmaWait = 1u << 1,
  kErrSoftmaxWait = 1u << 2,
  kErrDrain = 1u << 3,
  kErrPrologueWait = 1u << 4,
  kErrMergeWait = 1u << 5,
  kErrSelftestWait = 1u << 6,
  kErrLinearWait = 1u << 7,
  kErrDecodeWait = 1u << 8,
};

// ------------------------------------------------------------------------- workspace layout
//   [0, 1024)                    status word (bytes 0-3); grid-merge arrival and departure
//                                 counts (bytes 4-11, zero between calls); rest reserved
//   sync    n_layers * 8 * 2 uint32  per unit: arrival count and partial-ready flag of the
//                                   in-kernel merge of two-part units (zero between calls)
//   qscale  n_layers * 8 * 128 fp32    FP8 only: per-row scale of the e4m3 roped Q
//   svref   n_layers * 8 fp32          FP8 only: per-unit reference V scale (max over its tiles)
//   q       n_layers * 8 * 32 KB  e4m3 only: roped Q per (layer, kv head) as high and low e4m3
//                                 codes, swizzled K-major (a bf16 call prepares Q in the
//                                 attention kernel's shared memory and has no such region)
//   part_o  n_ctas * 2 * 128*128 f16   split partial outputs (normalised), per slot chunk-major:
//                                     16-byte chunk c (columns 8c .. 8c+7) of row r at c * 128 + r;
//                                     each half row (64 columns) is stored times a power of two
//                                     that puts its largest magnitude in [2^14, 2^15)
//   part_lse n_ctas * 2 * 3*128 fp32   per slot: the rows' log2-sum-exp (in units of log2-scaled
//                                     scores), then per half row the inverse of that power of two
struct WsLayout {
  size_t sync_off, qscale_off, svref_off, q_off, part_o_off, part_lse_off, total;
};

constexpr WsLayout ws_layout(int n_layers_per_launch, int max_ctas, bool fp8) {
  WsLayout w{};
  size_t off = 1024;
  w.sync_off = off;
  off += ((static_cast<size_t>(n_layers_per_launch) * kHkv * 2 * sizeof(uint32_t)) + 1023) &
         ~static_cast<size_t>(1023);
  w.qscale_off = off;
  off += static_cast<size_t>(n_layers_per_launch) * kHkv * kRows * sizeof(float);
  w.svref_off = off;
  off += ((static_cast<size_t>(n_layers_per_launch) * kHkv * sizeof(float)) + 1023) & ~static_cast<size_t>(1023);
  w.q_off = off;
  if (fp8) off += static_cast<size_t>(n_layers_per_launch) * kHkv * kQTileBytes;
  w.part_o_off = off;
  off += static_cast<size_t>(max_ctas) * 2 * kRows * kD * 2;
  w.part_lse_off = off;
  off += static_cast<size_t>(max_ctas) * 2 * 3 * kRows * sizeof(float);
  w.total = (off + 1023) & ~static_cast<size_t>(1023);
  return w;
}

// ------------------------------------------------------------------------ parameter blocks
struct PrologueLayer {
  const __nv_bfloat16* q_raw;
  const __nv_bfloat16* k_raw;
  const __nv_bfloat16* v_raw;
  const __nv_bfloat16* q_gamma;
  const __nv_bfloat16* k_gamma;
  void* k_cache;
  void* v_cache;
  float* k_scale;
  float* v_scale;
  __nv_bfloat16* q_rope;
};

template <int CAP>
struct PrologueParams {
  PrologueLayer layer[CAP];
  // RoPE inverse frequencies theta^(-j/64) as an fp32 pair hi + lo (16-byte aligned: a thread
  // reads its eight as two 16-byte vectors)
  alignas(16) float inv_hi[kD / 2];
  alignas(16) float inv_lo[kD / 2];
  uint8_t* q_ws;   // FP8: staged roped Q codes (bf16: null, nothing staged)
  float* q_scale;  // FP8: [unit][128] scale of each e4m3 Q row
  float* sv_ref;   // FP8: [unit] reference V scale
  uint32_t* unit_sync;  // [unit][2]: zeroed here for the attention kernel's in-kernel merge
  uint32_t* status;  // workspace status word (bounded-wait failures)
  int n_layers, S, Smax, rope_delta, fp8;
};

// Units split across CTAs (at most one per CTA boundary), merged after the attention grid.
constexpr int kMaxSplitUnits = 256;

// One split unit: its parts are CTAs c0 .. c0 + nparts - 1; the partial of CTA c sits in slot
// 2 c + 0, except the first CTA's, which sits in slot 2 c0 + slot0 (1 when the unit is that
// CTA's last segment, its range having started in an earlier unit).
struct SplitUnit {
  int u;
  short c0, nparts;
  int slot0;
};

template <int CAP>
struct AttnParams {
  CUtensorMap kmap[CAP];  // all Smax rows of K: dims {128, Smax, 8}, box {64 (e4m3: 128), 128, 1}
  CUtensorMap vmap[CAP];
  // bf16: the layer's inputs, normed and roped inside the attention kernel
  const __nv_bfloat16* q_raw[CAP];
  const __nv_bfloat16* k_raw[CAP];
  const __nv_bfloat16* v_raw[CAP];
  const __nv_bfloat16* q_gamma[CAP];
  const __nv_bfloat16* k_gamma[CAP];
  __nv_bfloat16* q_rope[CAP];  // optional
  __nv_bfloat16* kc[CAP];      // the caches, whose rows [Smax-64, Smax) the kernel writes
  __nv_bfloat16* vc[CAP];
  // RoPE inverse frequencies theta^(-j/64) as an fp32 pair hi + lo (16-byte aligned: a thread
  // reads its eight as two 16-byte vectors)
  alignas(16) float inv_hi[kD / 2];
  alignas(16) float inv_lo[kD / 2];
  int rope_base;         // S + rope_delta: token t sits at position rope_base + t
  __nv_bfloat16* out[CAP];
  const float* ks[CAP];      // FP8: block scales [8][Smax/128 + 1] (else null)
  const float* vs[CAP];
  const uint8_t* q_ws;  // FP8: the prologue's staged Q codes (bf16: null)
  uint4* part_o;     // f16 partials, 16-byte chunks (see the workspace layout)
  float* part_lse;   // per slot: lse[128], then the inverse scales of both half rows
  const float* q_scale;  // FP8: [unit][128]
  const float* sv_ref;   // FP8: [unit]
  uint32_t* unit_sync;   // [unit][2]: arrival count, partial-ready flag (in-kernel merge)
  uint32_t* status;
  long long W;         // total key tiles = n_layers * 8 * T
  int T;               // key tiles per (layer, kv head): n_main cache tiles + 1 own-row tile
  int n_main;          // ceil(S / 128)
  int S, Smax;
  int ncol;            // FP8: scale columns per kv head, Smax/128 + 1 (the last one: own rows)
  int fused_merge;     // every split unit has two parts: the second one merges in-kernel
  float scale_log2;    // log2(e) / sqrt(128)
  // Units of more than two parts (one layer spread over every SM) are merged by the whole grid
  // after a grid-wide arrival count: grid_sync[0] counts arrivals, grid_sync[1] departures (both
  // zero between calls: the last CTA to leave resets them).
  uint32_t* grid_sync;
  int grid_merge;      // 1 when some unit has more than two parts
  int n_split;         // the split units, in order
  SplitUnit split[kMaxSplitUnits];
};

// ------------------------------------------------------------ text-model decode attention
// One decode step of the VLM text model (alpamayo_tt/text.py, TTText._layer_decode): 64 query
// heads, 8 KV heads; query head h reads KV head h / 8. A unit is one (layer, kv head): its 8
// query heads against cache rows [0, pos], cut into key tiles of 128 rows.
constexpr int kHqText = 64;
constexpr int kRepText = kHqText / kHkv;  // query heads per KV head
constexpr int kDecodeMaxLayers = 64;
constexpr int kDecodeMaxPerUnit = 32;  // CTAs per unit in the decode kernel's unit-aligned mode

template <int CAP>
struct DecodeParams {
  CUtensorMap kmap[CAP];  // all Smax rows of K: dims {128, Smax, 8}, box {64, 128, 1}, 128B swizzle
  CUtensorMap vmap[CAP];
  const __nv_bfloat16* q_raw[CAP];  // [64][128]
  const __nv_bfloat16* k_raw[CAP];  // [8][128]
  const __nv_bfloat16* v_raw[CAP];  // [8][128]
  const __nv_bfloat16* q_gamma[CAP];
  const __nv_bfloat16* k_gamma[CAP];
  __nv_bfloat16* kc[CAP];  // caches [8][Smax][128]; the kernel writes row pos
  __nv_bfloat16* vc[CAP];
  __nv_bfloat16* out[CAP];  // [64][128]
  // RoPE inverse frequencies theta^(-j/64) as an fp32 pair hi + lo (16-byte aligned: a thread
  // reads its eight as two 16-byte vectors)
  alignas(16) float inv_hi[kD / 2];
  alignas(16) float inv_lo[kD / 2];
  float* part_o;         // [n_ctas][2 slots][8 heads][128] unnormalised partial outputs
  float* part_ml;        // [n_ctas][2 slots][8 heads][2]: running max (log2 units) and sum
  uint32_t* unit_cnt;    // [unit]: parts that have written their partial (zero between calls)
  uint32_t* status;
  long long W;           // total key tiles = n_layers * 8 * T
  int T;                 // key tiles per unit: ceil((pos + 1) / 128)
  int pos, rope_pos;     // the token's cache row, and its RoPE position pos + rope_delta
  int Smax;              // cache rows per head
  int cluster;           // 0: tiles of all units over all CTAs, split units merged through global
                         // memory; else the cluster size: one cluster per unit, merged through
                         // distributed shared memory
  int per_unit;          // > 0 (no cluster): that many CTAs per unit, each with one segment of
                         // its unit (ranges aligned to units); the unit's last part to arrive
                         // stages every part in its drained ring by bulk copy and merges there
  float scale_log2;      // log2(e) / sqrt(128)
};

// Decode workspace: [0, 1024) status word; unit counters n_layers * 8 uint32 (1 KB aligned);
// partial outputs and statistics for at most max_ctas CTAs.
struct DecodeWs {
  size_t cnt_off, part_o_off, part_ml_off, total;
};
constexpr DecodeWs decode_ws_layout(int n_layers, int max_ctas) {
  DecodeWs w{};
  size_t off = 1024;
  w.cnt_off = off;
  off += ((static_cast<size_t>(n_layers) * kHkv * sizeof(uint32_t)) + 1023) & ~static_cast<size_t>(1023);
  w.part_o_off = off;
  off += static_cast<size_t>(max_ctas) * 2 * kRepText * kD * sizeof(float);
  w.part_ml_off = off;
  off += static_cast<size_t>(max_ctas) * 2 * kRepText * 2 * sizeof(float);
  w.total = (off + 1023) & ~static_cast<size_t>(1023);
  return w;
}

// ------------------------------------------------------------ decoder-layer projections
constexpr int kMaxHidden = 8192;   // widest residual stream of the decoder layer
constexpr int kMaxInter = 32768;

// One projection Y[t][n] = sum_k X[t][k] W[n][k] for the 64 tokens (linear.cu), with the
// epilogue `mode`. Each weight map is 2-D {K, rows} with a {64, 128} box ({64, 64} for the
// gate/up pair of kLinSwiglu, whose tile i takes rows [64 i, 64 i + 64) of wmap[0] and of
// wmap[1]); the activation map is 4-D {64, c1, 64, c3} with a {64, 1, 64, 1} box, k-step kk at
// coordinates (0, kk % c1, 0, kk / c1) (row-major X: c1 = K / 64, c3 = 1; the attention output
// [16][64][128]: c1 = 2 halves of a head, c3 = 16 heads).
enum : int { kLinPlain = 0, kLinResidual = 1, kLinQkvHeads = 2, kLinSwiglu = 3 };
// A projection with a fused RMSNorm stages the gains of its CTA's channels in shared memory: at
// most this many 64-channel k-steps per CTA (the split planner takes enough splits).
constexpr int kNormMaxSteps = 64;

struct LinearParams {
  CUtensorMap wmap[2];
  CUtensorMap xmap;
  uint32_t* status;          // workspace status word
  const __nv_bfloat16* res;  // kLinResidual: residual input [64][N]
  __nv_bfloat16* y;          // kLinPlain, kLinResidual, kLinSwiglu: output [64][N]
  __nv_bfloat16* q;          // kLinQkvHeads: [16][64][128], k and v [8][64][128]
  __nv_bfloat16* k;
  __nv_bfloat16* v;
  int N;                     // output features (kLinSwiglu: of the gate projection alone)
  int ksteps;                // K / 64
  int kps;                   // k-steps per split (the splits of a tile form one cluster)
  int c1;
  int mode;
  const __nv_bfloat16* norm_gamma;  // non-null: X is replaced by rms_norm(X) * norm_gamma (over K)
};


// The key tiles of all (layer, kv head) units, in unit-major order, are cut into n_ctas
// contiguous ranges; CTA c owns tiles [c*W/n, (c+1)*W/n). A launch has at most kMaxGridCtas CTAs
// and W <= 64 layers x 8 units x (2^22 / 128 + 1) tiles, so c * W and x * n stay below 2^32 and
// both are taken in 32-bit unsigned arithmetic (a 64-bit division is a long software routine on
// the GPU, on the path of every partial segment).
constexpr int kMaxGridCtas = 160;
static_assert(64ull * kHkv * ((1ull << 22) / kKeyTile + 1) * kMaxGridCtas < (1ull << 32),
              "tile-range products must fit 32 bits");
__host__ __device__ inline long long cta_tile_start(int c, long long W, int n_ctas) {
  return static_cast<long long>(static_cast<uint32_t>(c) * static_cast<uint32_t>(W) /
                                static_cast<uint32_t>(n_ctas));
}

// The CTA whose range holds tile x.
__host__ __device__ inline int cta_of_tile(long long x, long long W, int n_ctas) {
  int c = static_cast<int>(static_cast<uint32_t>(x) * static_cast<uint32_t>(n_ctas) /
                           static_cast<uint32_t>(W));
  while (c + 1 < n_ctas && cta_tile_start(c + 1, W, n_ctas) <= x) ++c;
  while (c > 0 && cta_tile_start(c, W, n_ctas) > x) --c;
  return c;
}

}  // namespace ea
