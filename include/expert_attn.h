/*
 * expert_attn.h — C ABI of the GB300 (sm_103a) expert-attention library, libexpert_attn.so.
 *
 * The operation (alpamayo_tt/expert.py, TTExpert.layer and TTExpert.attention_core;
 * alpamayo_tt/EXPERT_NOTES.md, sections "Layouts" and "Attention over the VLM cache: masking
 * approach"): per layer, 64 expert tokens with 16 query heads and 8 KV heads of width 128
 *   1. RMS-normalise every q and k head row over its 128 channels with a multiplicative gain
 *      (eps 1e-6) and rotate it with the HF rotate_half RoPE, theta 5e6, at position
 *      t + rope_delta + S for token t;
 *   2. write the 64 roped k rows and the 64 raw v rows into rows [Smax-64, Smax) of the
 *      layer's K and V caches;
 *   3. let every token attend, non-causally, to cache rows [0, S) and to those 64 own rows
 *      (rows [S, Smax-64) are hidden: they are never read nor written); query head h uses
 *      KV head h/2, the score scale is 1/sqrt(128), softmax statistics are kept in fp32.
 *
 * Layouts (all row-major, little-endian, no padding):
 *   q_raw    bf16 [16][64][128]   head-major (q_raw[h][t][d])
 *   k_raw    bf16 [8][64][128]
 *   v_raw    bf16 [8][64][128]
 *   q_gamma  bf16 [128]           q_norm gain;   k_gamma bf16 [128] k_norm gain
 *   k_cache  [8][Smax][128]       bf16, or e4m3 bytes for EA_KV_FP8_E4M3; v_cache likewise
 *   k_scale  fp32 [8][Smax/128 + 1] (FP8 only): column b scales rows [128b, 128b+128);
 *            column Smax/128 scales the 64 own rows [Smax-64, Smax). v_scale likewise.
 *   out      bf16 [16][64][128]   attention output, head-major
 *   q_rope   optional bf16 [16][64][128]: the normalised, roped q (NULL to skip)
 *
 * Ownership: the caller owns every buffer. The library allocates no device memory. It
 * writes only out, q_rope, the workspace, cache rows [Smax-64, Smax) and (FP8) the last
 * scale column. Calls are asynchronous on the given stream (a cudaStream_t, NULL = legacy
 * default stream). Calls that share one workspace must not overlap on the GPU.
 *
 * Errors: argument errors return before anything is launched. EA_ERR_CUDA reports a failed
 * launch. A kernel that gives up a bounded wait records EA_ERR_TIMEOUT in the workspace's
 * status word, which expert_attn_read_status returns; the outputs of that call are then
 * undefined, and the workspace must be cleared again with expert_attn_workspace_init before
 * its next use.
 */
#ifndef EXPERT_ATTN_H
#define EXPERT_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  EA_OK = 0,
  EA_ERR_INVALID_ARG = 1,  /* null pointer, bad size, S out of [0, Smax-64], ... */
  EA_ERR_MISALIGNED = 2,   /* a pointer is not aligned as documented below */
  EA_ERR_UNSUPPORTED = 3,  /* no sm_103 GPU, or a dtype / size this build does not cover */
  EA_ERR_WORKSPACE = 4,    /* workspace smaller than expert_attn_workspace_size() */
  EA_ERR_CUDA = 5,         /* a CUDA runtime call or a launch failed */
  EA_ERR_TIMEOUT = 6       /* a kernel gave up a bounded wait (see expert_attn_read_status) */
} ea_status;

typedef enum { EA_KV_BF16 = 0, EA_KV_FP8_E4M3 = 1 } ea_kv_dtype;

/* A cudaStream_t, passed as an opaque pointer so that this header needs no CUDA header. */
typedef void* ea_stream_t;

/* One layer's buffers (device pointers). Alignment: every pointer 16 bytes; Smax a multiple
 * of 64 (bf16) or 128 (FP8). */
typedef struct {
  const void* q_raw;
  const void* k_raw;
  const void* v_raw;
  const void* q_gamma;
  const void* k_gamma;
  void* k_cache;
  void* v_cache;
  float* k_scale; /* FP8 only, else NULL */
  float* v_scale; /* FP8 only, else NULL */
  void* out;
  void* q_rope;   /* optional, may be NULL */
} ea_layer_args;

/* Utility (no counterpart on the pages). Bytes of device workspace needed by a call over
 * n_layers layers of the given cache dtype on
 * the current device (0 if no suitable device is present; an e4m3 workspace also serves bf16
 * calls). The workspace must be 256-byte aligned and, before
 * its first use, cleared with expert_attn_workspace_init. */
size_t expert_attn_workspace_size(int n_layers, int Smax, int kv_dtype);

/* Clears the workspace's status word and the per-unit words of the attention kernel's
 * in-kernel merge (asynchronous on stream). Every call leaves those words zero again unless it
 * reports EA_ERR_TIMEOUT. */
int expert_attn_workspace_init(void* workspace, size_t ws_bytes, ea_stream_t stream);

/* Steps 1 + 2 only (alpamayo_tt/expert.py, TTExpert.layer: q/k rms_norm, rotary_embedding_hf,
 * fill_cache): norm and rope q and k of one layer, write the own k/v rows into the cache tail
 * (FP8: quantised with their own scale slot, and the roped q staged in the workspace as e4m3
 * codes), and write the roped q to a->q_rope when it is not NULL. Requires 0 <= S <= Smax-64
 * and |S + rope_delta| + 64 < 2^24. */
int expert_attn_prologue(const ea_layer_args* a, int S, int Smax, int rope_delta, int kv_dtype,
                         void* workspace, size_t ws_bytes, ea_stream_t stream);

/* Steps 1-3 for one layer (the unit TTExpert.layer_fn can hand to a fused kernel): split-KV
 * attention on the tensor cores, whose kernel also does steps 1 and 2 for a bf16 cache (an e4m3
 * cache runs the prologue kernel first) and the log-sum-exp merge of the key ranges that it
 * split across SMs; writes a->out and, if not NULL, a->q_rope. */
int expert_attn_layer(const ea_layer_args* a, int S, int Smax, int rope_delta, int kv_dtype,
                      void* workspace, size_t ws_bytes, ea_stream_t stream);

/* Steps 1-3 for n_layers independent layers in one call (the 64 layers of one Euler step,
 * alpamayo_tt/expert.py, TTExpert._forward_dev), all with the same S, Smax and rope_delta.
 * layers is a HOST array of n_layers entries. Per 64 layers it launches the attention kernel,
 * after the prologue kernel for an e4m3 cache; the attention kernel merges the units it splits
 * across CTAs itself (two-part units in the epilogue of the part that finishes second, units of
 * more parts across the whole grid once every CTA has written its partials). */
int expert_attn_layers(const ea_layer_args* layers, int n_layers, int S, int Smax, int rope_delta,
                       int kv_dtype, void* workspace, size_t ws_bytes, ea_stream_t stream);

/* As expert_attn_layers, and records four cudaEvent_t (passed as void*, each may be NULL) on
 * the stream, around the first 64 layers: before the prologue kernel, before the attention
 * kernel (right after the first event for a bf16 cache, which has no prologue kernel), after
 * it, and a fourth right after the third (no kernel follows the attention kernel). Recording
 * events between the kernels removes their launch overlap; use it to time the kernels. */
int expert_attn_layers_profiled(const ea_layer_args* layers, int n_layers, int S, int Smax,
                                int rope_delta, int kv_dtype, void* workspace, size_t ws_bytes,
                                ea_stream_t stream, void* const events[4]);

/* FP8 cache producer: quantises rows [0, n_rows) of one bf16 cache [8][Smax][128] into e4m3
 * codes (round to nearest even, saturating) with one fp32 scale amax/448 per (kv head, 128-row
 * block) over the block's rows below n_rows (1 when amax is 0). Rows >= n_rows and their
 * scale columns are not written. Requires Smax % 128 == 0, 0 <= n_rows <= Smax-64. */
int expert_attn_quantize_cache(const void* src_bf16, int n_rows, int Smax, void* dst_codes,
                               float* scales, ea_stream_t stream);

/* 4-bit cache producer (OCP MX v1.0 MXFP4; the pages' lowest-precision cache is Tenstorrent
 * block-float, which has no GPU counterpart): quantises rows [0, n_rows) of every kv head of a
 * bf16 cache [8][Smax][128] into E2M1 codes with one power-of-two scale 2^e per 32 consecutive
 * channels of a row, e = floor(log2(amax)) - 2 clamped to [-127, 127] (0 for an all-zero
 * block); codes round to nearest, ties to the even code, saturating at +-6.
 * dst_codes: uint8 [8][Smax][64], two codes per byte, the lower channel in the low nibble (bit 3
 * of a code is the sign). dst_scales: uint8 [8][Smax][4], the biased exponent e + 127 of each
 * block. Rows >= n_rows are not written. Requires 0 <= n_rows <= Smax <= 2^22; src_bf16 and
 * dst_codes 16-byte aligned. Returns EA_ERR_INVALID_ARG / EA_ERR_MISALIGNED before any launch. */
int expert_attn_quantize_cache_mxfp4(const void* src_bf16, int n_rows, int Smax, void* dst_codes,
                                     void* dst_scales, ea_stream_t stream);

/* Utility (no counterpart on the pages). Tuning knob: number of persistent attention CTAs
 * (0 = one per SM, the default). Values above the SM count are clamped. The setting is
 * process-wide, not per stream or per thread: a call made on one thread changes the plan of
 * calls launched afterwards from every thread. Returns the previous setting. */
int expert_attn_set_splits(int n_ctas_or_0_for_auto);

/* Synchronises the stream and returns the status recorded in the workspace by the kernels
 * (EA_OK or EA_ERR_TIMEOUT) in *status_out; the raw status bits go to *bits_out if not NULL. */
int expert_attn_read_status(const void* workspace, ea_stream_t stream, int* status_out,
                            uint32_t* bits_out);

/* Utility (no counterpart on the pages). A static string naming a status code. */
const char* expert_attn_status_string(int status);

/* Failure-detection self-test (the pages have no counterpart): launches one CTA on the stream
 * whose thread waits on a shared-memory barrier that nothing ever arrives on, giving up after
 * limit_us microseconds (1 .. 2000000) exactly as the library's kernels give up a bounded wait:
 * it records a timeout bit in the workspace's status word and returns (no trap, no hang), so
 * that expert_attn_read_status then reports EA_ERR_TIMEOUT and the context stays usable.
 * Returns EA_ERR_INVALID_ARG for a null workspace or an out-of-range limit. */
int expert_attn_selftest_wait_timeout(int limit_us, void* workspace, size_t ws_bytes,
                                      ea_stream_t stream);

/* ---- Variant without a caller-provided workspace (the pages have no counterpart to this).
 *
 * Some callers cannot allocate device memory at all: a plugin hosted by an engine that owns the
 * whole device-memory budget and hands plugins no allocator, or a latency-critical loop where
 * cudaMalloc / cudaFree are banned because they can synchronise the device. This entry point
 * serves them: it does exactly what expert_attn_layers does, but its scratch (staged roped q,
 * own rows, split partials, status word) lives in one static device array compiled into the
 * library, EA_NOALLOC_SCRATCH_BYTES large, which every GPU that loads the library holds until the
 * process exits. It calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * Limits: at most EA_NOALLOC_MAX_LAYERS layers per call (more return EA_ERR_WORKSPACE before
 * anything is launched) and at most EA_NOALLOC_MAX_CTAS attention CTAs (fewer than one per SM on
 * a GB300, so it is slower than expert_attn_layers for large steps).
 * Set-up: the first call on a device looks up the array's device address on that device (which
 * must be current); make that first call before any stream capture.
 * Sharing: all calls in the process share the array and find the previous call's contents in
 * it; each call clears the words that must start at zero itself. Calls that overlap on the GPU
 * (for example on two streams) race on the array and must be avoided.
 * Errors: argument errors and failed launches are returned as by expert_attn_layers. A kernel
 * that gives up a bounded wait records it in the array's status word, which stays set across
 * later calls until expert_attn_noalloc_read_status reads it; the outputs of the call that
 * timed out are undefined. */
#define EA_NOALLOC_MAX_LAYERS 4
#define EA_NOALLOC_MAX_CTAS 64
#define EA_NOALLOC_SCRATCH_BYTES 5458944u /* 2 KB + 4 layers x 260 KB + 1 KB + 64 CTAs x 67 KB */
int expert_attn_layers_noalloc(const ea_layer_args* layers, int n_layers, int S, int Smax,
                               int rope_delta, int kv_dtype, ea_stream_t stream);

/* Status of the calls above (no counterpart on the pages either): synchronises the stream and
 * returns in *status_out EA_OK, or EA_ERR_TIMEOUT if a kernel of some expert_attn_layers_noalloc
 * call on the current device gave up a bounded wait since the status was last read; the raw
 * status bits go to *bits_out if not NULL. A set status is cleared by this read. Allocates
 * nothing. Returns EA_ERR_INVALID_ARG for a null status_out, EA_ERR_UNSUPPORTED without an
 * sm_103 device, EA_ERR_CUDA if the copy fails. */
int expert_attn_noalloc_read_status(ea_stream_t stream, int* status_out, uint32_t* bits_out);

/* ------------------------------------------------------------------ whole decoder layer
 * One decoder layer of the expert around the attention above (alpamayo_tt/expert.py,
 * TTExpert.layer):
 *   h  = rms_norm(x, ln1)                       (per token over the hidden channels, eps 1e-6)
 *   q, k, v = heads of h wqkv^T                  (wqkv rows: q features 128 h + d of the 16 heads,
 *                                                then k, then v of the 8 KV heads)
 *   a  = the attention above (q/k norms, RoPE, own rows into the cache tail, masked GQA)
 *   x1 = x + concat_heads(a) wo^T                (token row = the 16 heads side by side)
 *   x_out = x1 + (silu(h2 w1^T) * (h2 w3^T)) w2^T,  h2 = rms_norm(x1, ln2)
 * Every weight is bf16 row-major [out_features][in_features] (y = x W^T); activations between
 * the steps are kept in bf16 (h and h2 as bf16(gain * x), their 1 / rms applied in fp32) and
 * products accumulate in fp32. Widths: hidden and inter are
 * multiples of 128 with hidden <= 8192 and inter <= 32768 (the expert: 1536 and 6144). The
 * cache is bf16 [8][Smax][128] with the same rules as expert_attn_layer (rows [Smax-64, Smax)
 * are written). All pointers are device pointers, 16-byte aligned. The projections start
 * streaming their weights before the preceding kernel on the stream has finished when that
 * kernel allows programmatic dependent launch (the library's own kernels do, ordinary
 * launches do not), so weights must not be produced by such a kernel. */
typedef struct {
  const void* x;      /* bf16 [64][hidden] layer input (residual stream) */
  void* x_out;        /* bf16 [64][hidden] layer output; must not be x */
  int hidden, inter;
  const void* ln1;    /* bf16 [hidden] */
  const void* wqkv;   /* bf16 [4096][hidden] */
  const void* q_norm; /* bf16 [128] */
  const void* k_norm; /* bf16 [128] */
  const void* wo;     /* bf16 [hidden][2048] */
  const void* ln2;    /* bf16 [hidden] */
  const void* w1;     /* bf16 [inter][hidden] (gate) */
  const void* w3;     /* bf16 [inter][hidden] (up) */
  const void* w2;     /* bf16 [hidden][inter] (down) */
  void* k_cache;      /* bf16 [8][Smax][128] */
  void* v_cache;
  void* q_rope;       /* optional bf16 [16][64][128]: the normalised, roped q (NULL to skip) */
} ea_decoder_layer_args;

/* Bytes of workspace for expert_decoder_layer on the current device (0 for invalid widths or
 * no suitable device). The workspace must be 256-byte aligned and cleared once with
 * expert_attn_workspace_init; expert_attn_read_status reads its status word. */
size_t expert_decoder_layer_workspace_size(int hidden, int inter);

/* One decoder layer (see above): four projections on the tensor cores and the attention kernel,
 * five launches. Each projection applies its epilogue (head split, residual add or SwiGLU); the
 * two RMSNorms are fused into the projections that consume them (wqkv and w1|w3): the input
 * rows, scaled by the gains, are rounded to bf16 for the tensor cores, and 1 / rms, from the
 * rows' sums of squares over all channels, scales the fp32 sums before the epilogue. */
int expert_decoder_layer(const ea_decoder_layer_args* a, int S, int Smax, int rope_delta,
                         void* workspace, size_t ws_bytes, ea_stream_t stream);

/* One projection of the 64 tokens on the tensor cores: y[64][N] = x[64][K] W^T in bf16 with fp32
 * accumulation (W bf16 [N][K]); K a multiple of 64, N a multiple of 128, device pointers
 * 16-byte aligned; the workspace (size from expert_linear64_workspace_size, 256-byte aligned,
 * cleared once with expert_attn_workspace_init) holds the status word. */
size_t expert_linear64_workspace_size(int K, int N);
int expert_linear64(const void* x, const void* w, void* y, int K, int N, void* workspace,
                    size_t ws_bytes, ea_stream_t stream);

/* ------------------------------------------------------------ text-model decode attention
 * One decode step of the VLM text model over the same per-layer caches (alpamayo_tt/text.py,
 * TTText._layer_decode, with the cos/sin of TTText._decode_inputs_host): for the new token at
 * cache row pos, with 64 query heads and 8 KV heads of width 128 (query head h reads KV head
 * h / 8),
 *   1. RMS-normalise every q and k head row with the q_norm / k_norm gains (eps 1e-6) and rotate
 *      it with the HF rotate_half RoPE, theta 5e6, at position pos + rope_delta (the text
 *      model's multimodal RoPE with its three position ids equal);
 *   2. write the roped k (rounded to bf16) and the raw v into row pos of the layer's K and V
 *      caches (paged_update_cache);
 *   3. out[h] = softmax(q_h K[h/8, 0..pos]^T / sqrt(128)) V[h/8, 0..pos]
 *      (scaled_dot_product_attention_decode with cur_pos = pos: the new row is included).
 * Rows after pos are never read (their content, NaN included, does not matter) and only row pos
 * is written. Layouts: q_raw bf16 [64][128], k_raw and v_raw bf16 [8][128], gains bf16 [128],
 * caches bf16 [8][Smax][128] row-major per head (the layout of ea_layer_args), out bf16
 * [64][128]. All pointers are device pointers, 16-byte aligned; 0 <= pos < Smax, Smax a
 * multiple of 64 and >= 128. Ownership, asynchrony and errors as for expert_attn_layers. */
typedef struct {
  const void* q_raw;
  const void* k_raw;
  const void* v_raw;
  const void* q_gamma;
  const void* k_gamma;
  void* k_cache;
  void* v_cache;
  void* out;
} ea_decode_args;

/* Bytes of workspace for text_decode_attention over n_layers layers per call on the current
 * device (0 if no suitable device is present). */
size_t text_decode_workspace_size(int n_layers);

/* Zeroes the status word and the per-unit arrival counts (cudaMemsetAsync on `stream`). Call
 * once before the first use of a workspace; the kernel leaves the counts zero after every
 * call that completes, and after a call that reported EA_ERR_TIMEOUT the workspace must be
 * cleared again. The status word is read with expert_attn_read_status. */
int text_decode_workspace_init(void* workspace, size_t ws_bytes, ea_stream_t stream);

/* The decode step of n_layers independent layers (an array of n_layers ea_decode_args in host
 * memory) at the same pos and rope_delta, one kernel launch per 64 layers: every layer's keys
 * are cut into 128-row tiles that are spread over all SMs; a layer's KV head split over several
 * CTAs is merged by the part that finishes last. The workspace (256-byte aligned, size from
 * text_decode_workspace_size, cleared once) must not be shared by calls that overlap. */
int text_decode_attention(const ea_decode_args* layers, int n_layers, int pos, int Smax,
                          int rope_delta, void* workspace, size_t ws_bytes, ea_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* EXPERT_ATTN_H */
