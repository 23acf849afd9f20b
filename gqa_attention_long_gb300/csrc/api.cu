// api.cu — host side of libexpert_attn.so: argument validation, launch planning, TMA tensor-map
// encoding (cached), workspace layout and the launches per chunk of layers (e4m3 cache: the
// prologue kernel; the attention kernel, which does the bf16 prologue itself and merges the split
// units), chained with programmatic dependent launch.
// See include/expert_attn.h for the contract.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "expert_attn.h"
#include "internal.cuh"
#include "ptx.cuh"

namespace ea {
template <int CAP>
cudaError_t launch_prologue_kernel(const PrologueParams<CAP>& pp, bool fp8, int sm_count,
                                   cudaLaunchConfig_t cfg);
cudaError_t prologue_set_attributes();
cudaError_t attention_set_attributes();
template <int CAP>
cudaError_t launch_attention_kernel(const AttnParams<CAP>& ap, bool f8, cudaLaunchConfig_t cfg);
cudaError_t launch_quantize_mxfp4(const __nv_bfloat16* src, uint8_t* codes, uint8_t* scales, int n_rows,
                                  int Smax, cudaStream_t stream);
__global__ void quantize_cache_kernel(const __nv_bfloat16* src, uint8_t* dst, float* scales,
                                      int n_rows, int Smax);
}  // namespace ea

namespace {

using namespace ea;

constexpr int kMaxDevices = 64;

// One thread waits, with a time limit, on an mbarrier that nothing arrives on: the bounded-wait
// failure path of the library's kernels, made to run out on purpose (see the header).
__global__ void selftest_wait_kernel(uint32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint64_t t0 = globaltimer_ns();
    bool done = false;
    for (uint32_t it = 0; it < 0x80000000u; ++it) {
      if (mbar_try_wait(b, 0)) {
        done = true;
        break;
      }
      if ((it & 63u) == 0 && globaltimer_ns() - t0 > limit_ns) break;
    }
    if (!done) atomicOr(status, kErrSelftestWait);
  }
}

struct DeviceInfo {
  bool init = false;
  bool ok = false;
  int sm_count = 0;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;
int g_splits = 0;

// Queries (once per device) the SM count and that the device is an sm_103 part, and raises
// the attention kernel's dynamic shared-memory limit.
bool device_info(int* dev_out, DeviceInfo* info) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return false;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.init) {
    d.init = true;
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
        major == 10 && minor == 3 && sms > 0) {
      d.sm_count = sms;
      d.ok = attention_set_attributes() == cudaSuccess && prologue_set_attributes() == cudaSuccess;
    }
    cudaGetLastError();
  }
  *dev_out = dev;
  *info = d;
  return d.ok;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    cudaGetLastError();
  });
  return fn;
}

// Map of all Smax rows of one cache [8][Smax][128]: dims {128 channels, Smax, 8}, strides
// {row bytes, Smax * row bytes}, 128-byte swizzle; it serves the cache tiles and, at row
// Smax - 64, the own-row tile (its box rows past Smax arrive zero-filled). Keys >= S of the last
// cache tile are masked by the softmax, and their V rows zeroed in shared memory.
struct MapKey {
  const void* ptr;
  int S, Smax;
  bool f8;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && S == o.S && Smax == o.Smax && f8 == o.f8;
  }
};
struct MapKeyHash {
  size_t operator()(const MapKey& k) const {
    return std::hash<const void*>()(k.ptr) ^ (static_cast<size_t>(k.S) * 0x9E3779B97F4A7C15ull) ^
           (static_cast<size_t>(k.Smax) << 1) ^ (k.f8 ? 0x5bd1e995ull : 0);
  }
};
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_maps;

// bf16 cache: box {64 channels, 128 rows, 1}; e4m3 cache: box {128 channels (bytes), 128, 1}.
bool cache_map(const void* base, int S, int Smax, bool f8, CUtensorMap* out) {
  const MapKey key{base, S, Smax, f8};
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_maps.find(key);
    if (it != g_maps.end()) {
      *out = it->second;
      return true;
    }
  }
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  CUtensorMap m;
  std::memset(&m, 0, sizeof(m));
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(Smax),
                              static_cast<cuuint64_t>(kHkv)};
  const cuuint64_t esz = f8 ? 1 : 2;
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD) * esz,
                                 static_cast<cuuint64_t>(Smax) * kD * esz};
  const cuuint32_t box[3] = {f8 ? 128u : 64u, static_cast<cuuint32_t>(kKeyTile), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (fn(&m, f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
         const_cast<void*>(base), dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_maps.size() > 16384) g_maps.clear();
  g_maps[key] = m;
  *out = m;
  return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Pure argument checks (no CUDA call), so that they also run on machines without a GPU.
int validate(const ea_layer_args* a, int n_layers, int S, int Smax, int rope_delta, int kv_dtype,
             const void* ws, bool need_ws) {
  if (a == nullptr || n_layers < 1) return EA_ERR_INVALID_ARG;
  if (kv_dtype != EA_KV_BF16 && kv_dtype != EA_KV_FP8_E4M3) return EA_ERR_INVALID_ARG;
  const int row_align = kv_dtype == EA_KV_BF16 ? kTok : kScaleBlock;
  if (Smax < 2 * kTok || Smax % row_align != 0 || Smax > (1 << 22)) return EA_ERR_INVALID_ARG;
  if (S < 0 || S > Smax - kTok) return EA_ERR_INVALID_ARG;
  const long long p0 = static_cast<long long>(S) + rope_delta;
  if (p0 <= -(1LL << 24) + kTok || p0 + kTok >= (1LL << 24)) return EA_ERR_INVALID_ARG;
  if (need_ws && ws == nullptr) return EA_ERR_INVALID_ARG;
  if (need_ws && (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return EA_ERR_MISALIGNED;
  for (int l = 0; l < n_layers; ++l) {
    const ea_layer_args& x = a[l];
    const void* req[] = {x.q_raw, x.k_raw, x.v_raw, x.q_gamma, x.k_gamma, x.k_cache, x.v_cache, x.out};
    for (const void* p : req) {
      if (p == nullptr) return EA_ERR_INVALID_ARG;
      if (!aligned16(p)) return EA_ERR_MISALIGNED;
    }
    if (x.q_rope != nullptr && !aligned16(x.q_rope)) return EA_ERR_MISALIGNED;
    if (kv_dtype == EA_KV_FP8_E4M3) {
      if (x.k_scale == nullptr || x.v_scale == nullptr) return EA_ERR_INVALID_ARG;
      if ((reinterpret_cast<uintptr_t>(x.k_scale) & 3u) || (reinterpret_cast<uintptr_t>(x.v_scale) & 3u))
        return EA_ERR_MISALIGNED;
    }
  }
  return EA_OK;
}

}  // namespace

namespace {

// Bytes that expert_attn_workspace_init zeroes: everything before the first region that the
// kernels fully rewrite on every call.
constexpr size_t kInitBytes = ws_layout(kMaxLayersPerLaunch, 1, true).qscale_off;

// RoPE inverse frequencies theta^(-2j/128) = 5e6^(-j/64), j < 64, as fp32 (hi, lo) pairs
// (computed once per process).
void rope_inv_freq(float* hi, float* lo) {
  static float t_hi[kD / 2], t_lo[kD / 2];
  static std::once_flag once;
  std::call_once(once, [] {
    for (int j = 0; j < kD / 2; ++j) {
      const double inv = std::pow(5.0e6, -static_cast<double>(j) / (kD / 2));
      t_hi[j] = static_cast<float>(inv);
      t_lo[j] = static_cast<float>(inv - static_cast<double>(t_hi[j]));
    }
  });
  std::memcpy(hi, t_hi, sizeof(t_hi));
  std::memcpy(lo, t_lo, sizeof(t_lo));
}

int n_ctas_for(long long W, int sm_count) {
  int n = g_splits > 0 && g_splits < sm_count ? g_splits : sm_count;
  if (n > kMaxSplitUnits + 1) n = kMaxSplitUnits + 1;  // at most one split unit per boundary
  if (n > kMaxGridCtas) n = kMaxGridCtas;
  if (static_cast<long long>(n) > W) n = static_cast<int>(W);
  return n < 1 ? 1 : n;
}

cudaLaunchConfig_t launch_config(cudaStream_t st, cudaLaunchAttribute* attr, bool pdl) {
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cfg;
}

// The prologue is launched with programmatic stream serialization: its CTAs may become resident
// while the preceding kernel drains, and wait (griddepcontrol.wait) for it before touching memory.
template <int CAP>
int launch_prologue_t(const ea_layer_args* a, int n, int S, int Smax, int rope_delta, bool fp8,
                      uint8_t* ws, const WsLayout& wl, int sm_count, cudaStream_t st, bool pdl) {
  PrologueParams<CAP> pp;
  std::memset(&pp, 0, sizeof(pp));
  for (int l = 0; l < n; ++l) {
    PrologueLayer& d = pp.layer[l];
    d.q_raw = static_cast<const __nv_bfloat16*>(a[l].q_raw);
    d.k_raw = static_cast<const __nv_bfloat16*>(a[l].k_raw);
    d.v_raw = static_cast<const __nv_bfloat16*>(a[l].v_raw);
    d.q_gamma = static_cast<const __nv_bfloat16*>(a[l].q_gamma);
    d.k_gamma = static_cast<const __nv_bfloat16*>(a[l].k_gamma);
    d.k_cache = a[l].k_cache;
    d.v_cache = a[l].v_cache;
    d.k_scale = a[l].k_scale;
    d.v_scale = a[l].v_scale;
    d.q_rope = static_cast<__nv_bfloat16*>(a[l].q_rope);
  }
  rope_inv_freq(pp.inv_hi, pp.inv_lo);
  pp.q_ws = fp8 ? ws + wl.q_off : nullptr;  // bf16: Q is prepared inside the attention kernel
  pp.q_scale = reinterpret_cast<float*>(ws + wl.qscale_off);
  pp.sv_ref = reinterpret_cast<float*>(ws + wl.svref_off);
  pp.unit_sync = reinterpret_cast<uint32_t*>(ws + wl.sync_off);
  pp.status = reinterpret_cast<uint32_t*>(ws);
  pp.n_layers = n;
  pp.S = S;
  pp.Smax = Smax;
  pp.rope_delta = rope_delta;
  pp.fp8 = fp8 ? 1 : 0;
  cudaLaunchAttribute attr[1];
  if (launch_prologue_kernel<CAP>(pp, fp8, sm_count, launch_config(st, attr, pdl)) != cudaSuccess) {
    cudaGetLastError();
    return EA_ERR_CUDA;
  }
  return EA_OK;
}

int launch_prologue(const ea_layer_args* a, int n, int S, int Smax, int rope_delta, bool fp8,
                    uint8_t* ws, const WsLayout& wl, int sm_count, cudaStream_t st, bool pdl) {
  return n <= kSmallCap
             ? launch_prologue_t<kSmallCap>(a, n, S, Smax, rope_delta, fp8, ws, wl, sm_count, st, pdl)
             : launch_prologue_t<kMaxLayersPerLaunch>(a, n, S, Smax, rope_delta, fp8, ws, wl, sm_count,
                                                      st, pdl);
}

// Attention parameter blocks are large (~25 KB at full capacity): kept off the stack, one per
// capacity, guarded by their own mutex.
template <int CAP>
struct LaunchBlocks {
  AttnParams<CAP> ap;
  std::mutex mu;
};
template <int CAP>
LaunchBlocks<CAP>& launch_blocks() {
  static LaunchBlocks<CAP> b;
  return b;
}

template <int CAP>
int launch_chunk_t(const ea_layer_args* a, int n, int S, int Smax, int rope_delta, bool fp8,
                   uint8_t* ws, const WsLayout& wl, const DeviceInfo& di, cudaStream_t st,
                   cudaEvent_t const* ev) {
  const bool pdl = ev == nullptr;
  if (ev && ev[0] && cudaEventRecord(ev[0], st) != cudaSuccess) return EA_ERR_CUDA;
  if (fp8) {  // bf16: the attention kernel norms and ropes q and k and writes the own rows itself
    const int rc = launch_prologue_t<CAP>(a, n, S, Smax, rope_delta, fp8, ws, wl, di.sm_count, st, pdl);
    if (rc != EA_OK) return rc;
  }
  if (ev && ev[1] && cudaEventRecord(ev[1], st) != cudaSuccess) return EA_ERR_CUDA;

  LaunchBlocks<CAP>& lb = launch_blocks<CAP>();
  std::lock_guard<std::mutex> lk(lb.mu);
  AttnParams<CAP>& ap = lb.ap;
  std::memset(&ap, 0, sizeof(ap));
  for (int l = 0; l < n; ++l) {
    if (!cache_map(a[l].k_cache, S, Smax, fp8, &ap.kmap[l]) ||
        !cache_map(a[l].v_cache, S, Smax, fp8, &ap.vmap[l]))
      return EA_ERR_CUDA;
    ap.out[l] = static_cast<__nv_bfloat16*>(a[l].out);
    ap.ks[l] = a[l].k_scale;
    ap.vs[l] = a[l].v_scale;
    ap.q_raw[l] = static_cast<const __nv_bfloat16*>(a[l].q_raw);
    ap.k_raw[l] = static_cast<const __nv_bfloat16*>(a[l].k_raw);
    ap.v_raw[l] = static_cast<const __nv_bfloat16*>(a[l].v_raw);
    ap.q_gamma[l] = static_cast<const __nv_bfloat16*>(a[l].q_gamma);
    ap.k_gamma[l] = static_cast<const __nv_bfloat16*>(a[l].k_gamma);
    ap.q_rope[l] = static_cast<__nv_bfloat16*>(a[l].q_rope);
    ap.kc[l] = static_cast<__nv_bfloat16*>(a[l].k_cache);
    ap.vc[l] = static_cast<__nv_bfloat16*>(a[l].v_cache);
  }
  rope_inv_freq(ap.inv_hi, ap.inv_lo);
  ap.rope_base = S + rope_delta;
  const int n_main = (S + kKeyTile - 1) / kKeyTile;
  ap.T = n_main + 1;
  ap.n_main = n_main;
  ap.S = S;
  ap.Smax = Smax;
  ap.W = static_cast<long long>(n) * kHkv * ap.T;
  ap.q_ws = fp8 ? ws + wl.q_off : nullptr;
  ap.part_o = reinterpret_cast<uint4*>(ws + wl.part_o_off);
  ap.part_lse = reinterpret_cast<float*>(ws + wl.part_lse_off);
  ap.q_scale = reinterpret_cast<const float*>(ws + wl.qscale_off);
  ap.sv_ref = reinterpret_cast<const float*>(ws + wl.svref_off);
  ap.ncol = Smax / kScaleBlock + 1;
  ap.unit_sync = reinterpret_cast<uint32_t*>(ws + wl.sync_off);
  ap.status = reinterpret_cast<uint32_t*>(ws);
  ap.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(kD)));
  const int n_ctas = n_ctas_for(ap.W, di.sm_count);

  // Units cut by a CTA boundary (each listed once, in order). When every one of them has two
  // parts, the part that finishes second merges them inside the attention kernel; otherwise the
  // whole grid merges them after a grid-wide arrival count (see the kernel).
  ap.n_split = 0;
  bool all_two = true;
  for (int b = 1; b < n_ctas; ++b) {
    const long long tb = cta_tile_start(b, ap.W, n_ctas);
    if (tb % ap.T == 0) continue;
    const int u = static_cast<int>(tb / ap.T);
    if (ap.n_split > 0 && ap.split[ap.n_split - 1].u == u) continue;
    const long long first = static_cast<long long>(u) * ap.T;
    SplitUnit& su = ap.split[ap.n_split++];
    su.u = u;
    su.c0 = static_cast<short>(cta_of_tile(first, ap.W, n_ctas));
    su.nparts = static_cast<short>(cta_of_tile(first + ap.T - 1, ap.W, n_ctas) - su.c0 + 1);
    su.slot0 = cta_tile_start(su.c0, ap.W, n_ctas) >= first ? 0 : 1;
    all_two = all_two && su.nparts == 2;
  }
  ap.fused_merge = all_two ? 1 : 0;
  ap.grid_merge = ap.n_split > 0 && !all_two ? 1 : 0;
  ap.grid_sync = reinterpret_cast<uint32_t*>(ws) + 1;  // words 1 and 2 of the status block

  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = launch_config(st, attr, pdl);
  cfg.gridDim = dim3(n_ctas);
  if (launch_attention_kernel<CAP>(ap, fp8, cfg) != cudaSuccess) {
    cudaGetLastError();
    return EA_ERR_CUDA;
  }
  if (ev && ev[2] && cudaEventRecord(ev[2], st) != cudaSuccess) return EA_ERR_CUDA;
  if (ev && ev[3] && cudaEventRecord(ev[3], st) != cudaSuccess) return EA_ERR_CUDA;
  return EA_OK;
}

int launch_chunk(const ea_layer_args* a, int n, int S, int Smax, int rope_delta, bool fp8,
                 uint8_t* ws, const WsLayout& wl, const DeviceInfo& di, cudaStream_t st,
                 cudaEvent_t const* ev) {
  return n <= kSmallCap
             ? launch_chunk_t<kSmallCap>(a, n, S, Smax, rope_delta, fp8, ws, wl, di, st, ev)
             : launch_chunk_t<kMaxLayersPerLaunch>(a, n, S, Smax, rope_delta, fp8, ws, wl, di, st, ev);
}

int run_layers(const ea_layer_args* a, int n_layers, int S, int Smax, int rope_delta, int kv_dtype,
               void* workspace, size_t ws_bytes, ea_stream_t stream, cudaEvent_t const* ev) {
  int rc = validate(a, n_layers, S, Smax, rope_delta, kv_dtype, workspace, true);
  if (rc != EA_OK) return rc;
  int dev;
  DeviceInfo di;
  if (!device_info(&dev, &di)) return EA_ERR_UNSUPPORTED;
  const int per = n_layers < kMaxLayersPerLaunch ? n_layers : kMaxLayersPerLaunch;
  const WsLayout wl = ws_layout(per, di.sm_count, kv_dtype == EA_KV_FP8_E4M3);
  if (ws_bytes < wl.total) return EA_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  for (int l0 = 0; l0 < n_layers; l0 += per) {
    const int n = n_layers - l0 < per ? n_layers - l0 : per;
    rc = launch_chunk(a + l0, n, S, Smax, rope_delta, kv_dtype == EA_KV_FP8_E4M3, ws, wl, di, st,
                      l0 == 0 ? ev : nullptr);
    if (rc != EA_OK) return rc;
  }
  return EA_OK;
}

}  // namespace

extern "C" {

size_t expert_attn_workspace_size(int n_layers, int Smax, int kv_dtype) {
  if (n_layers < 1 || Smax < 2 * kTok) return 0;
  if (kv_dtype != EA_KV_BF16 && kv_dtype != EA_KV_FP8_E4M3) return 0;
  int dev;
  DeviceInfo di;
  if (!device_info(&dev, &di)) return 0;
  const int per = n_layers < kMaxLayersPerLaunch ? n_layers : kMaxLayersPerLaunch;
  return ws_layout(per, di.sm_count, kv_dtype == EA_KV_FP8_E4M3).total;
}

int expert_attn_workspace_init(void* workspace, size_t ws_bytes, ea_stream_t stream) {
  if (workspace == nullptr || ws_bytes < 1024) return EA_ERR_INVALID_ARG;
  // the status word and the in-kernel merge words of up to 64 layers per launch
  const size_t n = ws_bytes < kInitBytes ? ws_bytes : kInitBytes;
  if (cudaMemsetAsync(workspace, 0, n, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return EA_ERR_CUDA;
  }
  return EA_OK;
}

int expert_attn_prologue(const ea_layer_args* a, int S, int Smax, int rope_delta, int kv_dtype,
                         void* workspace, size_t ws_bytes, ea_stream_t stream) {
  int rc = validate(a, 1, S, Smax, rope_delta, kv_dtype, workspace, true);
  if (rc != EA_OK) return rc;
  int dev;
  DeviceInfo di;
  if (!device_info(&dev, &di)) return EA_ERR_UNSUPPORTED;
  const WsLayout wl = ws_layout(1, di.sm_count, kv_dtype == EA_KV_FP8_E4M3);
  if (ws_bytes < wl.total) return EA_ERR_WORKSPACE;
  return launch_prologue(a, 1, S, Smax, rope_delta, kv_dtype == EA_KV_FP8_E4M3,
                         static_cast<uint8_t*>(workspace), wl, di.sm_count,
                         static_cast<cudaStream_t>(stream), true);
}

int expert_attn_layer(const ea_layer_args* a, int S, int Smax, int rope_delta, int kv_dtype,
                      void* workspace, size_t ws_bytes, ea_stream_t stream) {
  return run_layers(a, 1, S, Smax, rope_delta, kv_dtype, workspace, ws_bytes, stream, nullptr);
}

int expert_attn_layers(const ea_layer_args* layers, int n_layers, int S, int Smax, int rope_delta,
                       int kv_dtype, void* workspace, size_t ws_bytes, ea_stream_t stream) {
  return run_layers(layers, n_layers, S, Smax, rope_delta, kv_dtype, workspace, ws_bytes, stream,
                    nullptr);
}

int expert_attn_layers_profiled(const ea_layer_args* layers, int n_layers, int S, int Smax,
                                int rope_delta, int kv_dtype, void* workspace, size_t ws_bytes,
                                ea_stream_t stream, void* const events[4]) {
  if (events == nullptr) return EA_ERR_INVALID_ARG;
  cudaEvent_t ev[4];
  for (int i = 0; i < 4; ++i) ev[i] = static_cast<cudaEvent_t>(events[i]);
  return run_layers(layers, n_layers, S, Smax, rope_delta, kv_dtype, workspace, ws_bytes, stream, ev);
}

int expert_attn_quantize_cache(const void* src_bf16, int n_rows, int Smax, void* dst_codes,
                               float* scales, ea_stream_t stream) {
  if (src_bf16 == nullptr || dst_codes == nullptr || scales == nullptr) return EA_ERR_INVALID_ARG;
  if (Smax < 2 * kTok || Smax % kScaleBlock != 0 || Smax > (1 << 22)) return EA_ERR_INVALID_ARG;
  if (n_rows < 0 || n_rows > Smax - kTok) return EA_ERR_INVALID_ARG;
  if (!aligned16(src_bf16) || !aligned16(dst_codes) || (reinterpret_cast<uintptr_t>(scales) & 3u))
    return EA_ERR_MISALIGNED;
  int dev;
  DeviceInfo di;
  if (!device_info(&dev, &di)) return EA_ERR_UNSUPPORTED;
  if (n_rows == 0) return EA_OK;
  quantize_cache_kernel<<<kHkv * (Smax / kScaleBlock), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const __nv_bfloat16*>(src_bf16), static_cast<uint8_t*>(dst_codes), scales, n_rows,
      Smax);
  return cudaGetLastError() == cudaSuccess ? EA_OK : EA_ERR_CUDA;
}

int expert_attn_quantize_cache_mxfp4(const void* src_bf16, int n_rows, int Smax, void* dst_codes,
                                     void* dst_scales, ea_stream_t stream) {
  if (src_bf16 == nullptr || dst_codes == nullptr || dst_scales == nullptr) return EA_ERR_INVALID_ARG;
  if (Smax < 1 || Smax > (1 << 22) || n_rows < 0 || n_rows > Smax) return EA_ERR_INVALID_ARG;
  if (!aligned16(src_bf16) || !aligned16(dst_codes)) return EA_ERR_MISALIGNED;
  int dev;
  DeviceInfo di;
  if (!device_info(&dev, &di)) return EA_ERR_UNSUPPORTED;
  if (n_rows == 0) return EA_OK;
  return launch_quantize_mxfp4(static_cast<const __nv_bfloat16*>(src_bf16), static_cast<uint8_t*>(dst_codes),
                               static_cast<uint8_t*>(dst_scales), n_rows, Smax,
                               static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? EA_OK
             : EA_ERR_CUDA;
}

int expert_attn_set_splits(int n_ctas_or_0_for_auto) {
  std::lock_guard<std::mutex> lk(g_mu);
  const int prev = g_splits;
  g_splits = n_ctas_or_0_for_auto > 0 ? n_ctas_or_0_for_auto : 0;
  return prev;
}

int expert_attn_read_status(const void* workspace, ea_stream_t stream, int* status_out,
                            uint32_t* bits_out) {
  if (workspace == nullptr || status_out == nullptr) return EA_ERR_INVALID_ARG;
  uint32_t bits = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&bits, workspace, sizeof(bits), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess) {
    cudaGetLastError();
    return EA_ERR_CUDA;
  }
  *status_out = bits == 0 ? EA_OK : EA_ERR_TIMEOUT;
  if (bits_out) *bits_out = bits;
  return EA_OK;
}

int expert_attn_selftest_wait_timeout(int limit_us, void* workspace, size_t ws_bytes,
                                      ea_stream_t stream) {
  if (workspace == nullptr || ws_bytes < 1024 || limit_us < 1 || limit_us > 2000000)
    return EA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return EA_ERR_MISALIGNED;
  int dev;
  DeviceInfo di;
  if (!device_info(&dev, &di)) return EA_ERR_UNSUPPORTED;
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint32_t*>(workspace), static_cast<uint64_t>(limit_us) * 1000ull);
  return cudaGetLastError() == cudaSuccess ? EA_OK : EA_ERR_CUDA;
}

const char* expert_attn_status_string(int status) {
  switch (status) {
    case EA_OK: return "EA_OK";
    case EA_ERR_INVALID_ARG: return "EA_ERR_INVALID_ARG: invalid argument";
    case EA_ERR_MISALIGNED: return "EA_ERR_MISALIGNED: pointer not aligned as required";
    case EA_ERR_UNSUPPORTED: return "EA_ERR_UNSUPPORTED: no sm_103 device or unsupported variant";
    case EA_ERR_WORKSPACE: return "EA_ERR_WORKSPACE: workspace too small";
    case EA_ERR_CUDA: return "EA_ERR_CUDA: CUDA call or kernel launch failed";
    case EA_ERR_TIMEOUT: return "EA_ERR_TIMEOUT: a kernel gave up a bounded wait";
    default: return "unknown status";
  }
}

}  // extern "C"

// -------------------------------------------------------------- no-allocation variant
// expert_attn_layers_noalloc runs the same launches as expert_attn_layers, with the
// workspace replaced by a static device array. Host code must not use the array's name as a
// pointer (that is a host-side stand-in); its device address is looked up once per device.
namespace {

constexpr size_t noalloc_bytes() {
  return ws_layout(EA_NOALLOC_MAX_LAYERS, EA_NOALLOC_MAX_CTAS, true).total;
}
static_assert(noalloc_bytes() == EA_NOALLOC_SCRATCH_BYTES, "scratch size in the header is stale");

static __device__ __align__(256) unsigned char g_noalloc_scratch[EA_NOALLOC_SCRATCH_BYTES];

void* g_noalloc_ptr[kMaxDevices];

// Device address of the scratch on the current device (looked up on first use per device).
void* noalloc_scratch(int dev) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return nullptr;
    }
    g_noalloc_ptr[dev] = p;
  }
  return g_noalloc_ptr[dev];
}

}  // namespace

extern "C" int expert_attn_layers_noalloc(const ea_layer_args* layers, int n_layers, int S,
                                          int Smax, int rope_delta, int kv_dtype,
                                          ea_stream_t stream) {
  int rc = validate(layers, n_layers, S, Smax, rope_delta, kv_dtype, nullptr, false);
  if (rc != EA_OK) return rc;
  if (n_layers > EA_NOALLOC_MAX_LAYERS) return EA_ERR_WORKSPACE;
  int dev;
  DeviceInfo di;
  if (!device_info(&dev, &di)) return EA_ERR_UNSUPPORTED;
  DeviceInfo capped = di;
  if (capped.sm_count > EA_NOALLOC_MAX_CTAS) capped.sm_count = EA_NOALLOC_MAX_CTAS;
  const WsLayout wl = ws_layout(n_layers, capped.sm_count, kv_dtype == EA_KV_FP8_E4M3);
  if (wl.total > EA_NOALLOC_SCRATCH_BYTES) return EA_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(noalloc_scratch(dev));
  if (ws == nullptr) return EA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the in-kernel merge words and the grid-merge counts start at 0; the status word (the first 4
  // bytes) is left alone, so that a timeout stays visible until expert_attn_noalloc_read_status
  // reads and clears it
  if (cudaMemsetAsync(ws + sizeof(uint32_t), 0, wl.qscale_off - sizeof(uint32_t), st) != cudaSuccess) {
    cudaGetLastError();
    return EA_ERR_CUDA;
  }
  return launch_chunk(layers, n_layers, S, Smax, rope_delta, kv_dtype == EA_KV_FP8_E4M3, ws, wl,
                      capped, st, nullptr);
}

extern "C" int expert_attn_noalloc_read_status(ea_stream_t stream, int* status_out,
                                               uint32_t* bits_out) {
  if (status_out == nullptr) return EA_ERR_INVALID_ARG;
  int dev;
  DeviceInfo di;
  if (!device_info(&dev, &di)) return EA_ERR_UNSUPPORTED;
  uint8_t* ws = static_cast<uint8_t*>(noalloc_scratch(dev));
  if (ws == nullptr) return EA_ERR_CUDA;
  uint32_t bits = 0;
  const int rc = expert_attn_read_status(ws, stream, status_out, &bits);
  if (rc != EA_OK) return rc;
  if (bits_out) *bits_out = bits;
  if (bits != 0) {  // reported once: clear it for the calls that follow
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, sizeof(uint32_t), st) != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess) {
      cudaGetLastError();
      return EA_ERR_CUDA;
    }
  }
  return EA_OK;
}

// ------------------------------------------------------------------ whole decoder layer
// Host side of expert_decoder_layer and expert_linear64: tensor maps of the projections'
// operands (cached), split-K planning, the layer workspace, and the launches (all chained with
// programmatic dependent launch).
namespace ea {
cudaError_t linear_set_attributes();
cudaError_t launch_linear(const LinearParams& lp, int tiles, int splits, cudaLaunchConfig_t cfg);
}  // namespace ea

namespace {

struct TmapKey {
  const void* ptr;
  int rank;
  cuuint64_t dims[4];
  cuuint64_t strides[3];
  cuuint32_t box[4];
  bool operator==(const TmapKey& o) const { return std::memcmp(this, &o, sizeof(TmapKey)) == 0; }
};
struct TmapKeyHash {
  size_t operator()(const TmapKey& k) const {
    const unsigned char* p = reinterpret_cast<const unsigned char*>(&k);
    size_t h = 1469598103934665603ull;
    for (size_t i = 0; i < sizeof(TmapKey); ++i) h = (h ^ p[i]) * 1099511628211ull;
    return h;
  }
};
std::unordered_map<TmapKey, CUtensorMap, TmapKeyHash> g_tmaps;

// bf16 tiled map with 128-byte swizzle (boxes are 64 channels = 128 bytes wide).
bool bf16_map(const void* ptr, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
              const cuuint32_t* box, CUtensorMap* out) {
  TmapKey key;
  std::memset(&key, 0, sizeof(key));
  key.ptr = ptr;
  key.rank = rank;
  for (int i = 0; i < rank; ++i) {
    key.dims[i] = dims[i];
    key.box[i] = box[i];
    if (i + 1 < rank) key.strides[i] = strides[i];
  }
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_tmaps.find(key);
    if (it != g_tmaps.end()) {
      *out = it->second;
      return true;
    }
  }
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  CUtensorMap m;
  std::memset(&m, 0, sizeof(m));
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  if (fn(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank), const_cast<void*>(ptr),
         dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_tmaps.size() > 16384) g_tmaps.clear();
  g_tmaps[key] = m;
  *out = m;
  return true;
}

// Weights [rows][K] (row-major): 2-D {K, rows}, box {64, box_rows}.
bool weight_map(const void* w, int K, int rows, int box_rows, CUtensorMap* out) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  return bf16_map(w, 2, dims, strides, box, out);
}

// Row-major activations [64][K]: 4-D {64, K/64, 64, 1}, box {64, 1, 64, 1}; k-step kk at
// (0, kk, 0, 0).
bool rows_map(const void* x, int K, CUtensorMap* out) {
  const cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(K / 64), kTok, 1};
  const cuuint64_t strides[3] = {128, static_cast<cuuint64_t>(K) * 2, static_cast<cuuint64_t>(K) * 2 * kTok};
  const cuuint32_t box[4] = {64, 1, kTok, 1};
  return bf16_map(x, 4, dims, strides, box, out);
}

// The attention output [16][64][128] read as the [64][2048] input of wo (feature 128 h + d):
// 4-D {64 channels, 2 halves, 64 tokens, 16 heads}, box {64, 1, 64, 1}; k-step kk at
// (0, kk % 2, 0, kk / 2).
bool heads_map(const void* a, CUtensorMap* out) {
  const cuuint64_t dims[4] = {64, 2, kTok, kHq};
  const cuuint64_t strides[3] = {128, kD * 2, static_cast<cuuint64_t>(kTok) * kD * 2};
  const cuuint32_t box[4] = {64, 1, kTok, 1};
  return bf16_map(a, 4, dims, strides, box, out);
}

// Split count of a projection (the cluster size of a tile): about two CTAs per SM (two fit), at
// least two k-steps per CTA where the k-steps allow it, at most 16 (the largest cluster), and no
// empty split.
constexpr int kMaxLinearCluster = 16;
void plan_splits(int tiles, int ksteps, int sm_count, bool norm, int* splits, int* kps) {
  int s = (2 * sm_count) / tiles;
  if (s > ksteps / 2) s = ksteps / 2;
  if (s > kMaxLinearCluster) s = kMaxLinearCluster;
  if (s < 1) s = 1;
  // a fused RMSNorm stages at most kNormMaxSteps k-steps of gains per CTA
  if (norm && s < (ksteps + kNormMaxSteps - 1) / kNormMaxSteps) s = (ksteps + kNormMaxSteps - 1) / kNormMaxSteps;
  *kps = (ksteps + s - 1) / s;
  *splits = (ksteps + *kps - 1) / *kps;
}

size_t align_kb(size_t x) { return (x + 1023) & ~static_cast<size_t>(1023); }

struct LayerWs {
  size_t attn_ws, q, k, v, attn, x1, gu, total;
};

// Layer workspace: the attention's own workspace first (its status word, at offset 0, is
// the one every kernel of the layer reports to), then the layer's bf16 activations.
LayerWs layer_ws_layout(int hidden, int inter, int sm_count) {
  LayerWs w{};
  size_t off = 0;
  w.attn_ws = off;
  off += align_kb(ws_layout(1, sm_count, false).total);
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align_kb(bytes);
    return o;
  };
  w.q = take(static_cast<size_t>(kHq) * kTok * kD * 2);
  w.k = take(static_cast<size_t>(kHkv) * kTok * kD * 2);
  w.v = take(static_cast<size_t>(kHkv) * kTok * kD * 2);
  w.attn = take(static_cast<size_t>(kHq) * kTok * kD * 2);
  w.x1 = take(static_cast<size_t>(kTok) * hidden * 2);
  w.gu = take(static_cast<size_t>(kTok) * inter * 2);
  w.total = off;
  return w;
}

bool layer_dims_ok(int hidden, int inter) {
  return hidden >= 128 && hidden <= kMaxHidden && hidden % 128 == 0 && inter >= 128 &&
         inter <= kMaxInter && inter % 128 == 0;
}

// One projection with its epilogue (LinearParams). w1 != nullptr: the gate/up pair of SwiGLU
// (tiles of 64 features of both), else tiles of 128 output features. norm_gamma != nullptr: the
// input rows are RMS-normalised over their K channels and scaled by norm_gamma first.
int run_linear(const CUtensorMap& xmap, int c1, const void* w0, const void* w1, int N, int K, int mode,
               const __nv_bfloat16* res, __nv_bfloat16* y, __nv_bfloat16* q, __nv_bfloat16* k,
               __nv_bfloat16* v, uint32_t* status, int sm_count, cudaStream_t st,
               const void* norm_gamma = nullptr) {
  static_assert(sizeof(LinearParams) < 4096, "linear parameter block");
  LinearParams lp;
  std::memset(&lp, 0, sizeof(lp));
  const bool pair = w1 != nullptr;
  if (!weight_map(w0, K, N, pair ? 64 : 128, &lp.wmap[0])) return EA_ERR_CUDA;
  if (pair && !weight_map(w1, K, N, 64, &lp.wmap[1])) return EA_ERR_CUDA;
  lp.xmap = xmap;
  lp.status = status;
  lp.res = res;
  lp.y = y;
  lp.q = q;
  lp.k = k;
  lp.v = v;
  lp.N = N;
  lp.ksteps = K / 64;
  lp.c1 = c1;
  lp.mode = mode;
  lp.norm_gamma = static_cast<const __nv_bfloat16*>(norm_gamma);
  const int tiles = pair ? N / 64 : N / 128;
  int splits, kps;
  plan_splits(tiles, lp.ksteps, sm_count, norm_gamma != nullptr, &splits, &kps);
  lp.kps = kps;
  cudaLaunchAttribute attr[2];  // PDL, and the cluster shape added by the launcher
  if (launch_linear(lp, tiles, splits, launch_config(st, attr, true)) != cudaSuccess) {
    cudaGetLastError();
    return EA_ERR_CUDA;
  }
  return EA_OK;
}

bool linear_attrs_ready() {
  static std::once_flag once;
  static bool ok = false;
  std::call_once(once, [] {
    ok = linear_set_attributes() == cudaSuccess;
    cudaGetLastError();
  });
  return ok;
}

}  // namespace

extern "C" {

size_t expert_decoder_layer_workspace_size(int hidden, int inter) {
  if (!layer_dims_ok(hidden, inter)) return 0;
  int dev;
  DeviceInfo di;
  if (!device_info(&dev, &di)) return 0;
  return layer_ws_layout(hidden, inter, di.sm_count).total;
}

int expert_decoder_layer(const ea_decoder_layer_args* a, int S, int Smax, int rope_delta,
                         void* workspace, size_t ws_bytes, ea_stream_t stream) {
  if (a == nullptr || workspace == nullptr) return EA_ERR_INVALID_ARG;
  if (!layer_dims_ok(a->hidden, a->inter)) return EA_ERR_INVALID_ARG;
  const void* req[] = {a->x, a->x_out, a->ln1, a->wqkv, a->q_norm, a->k_norm, a->wo, a->ln2,
                       a->w1, a->w3, a->w2, a->k_cache, a->v_cache};
  for (const void* p : req) {
    if (p == nullptr) return EA_ERR_INVALID_ARG;
    if (!aligned16(p)) return EA_ERR_MISALIGNED;
  }
  if (a->x == a->x_out) return EA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return EA_ERR_MISALIGNED;
  int dev;
  DeviceInfo di;
  if (!device_info(&dev, &di) || !linear_attrs_ready()) return EA_ERR_UNSUPPORTED;
  const int H = a->hidden, I = a->inter;
  const LayerWs wl = layer_ws_layout(H, I, di.sm_count);
  if (ws_bytes < wl.total) return EA_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto bf = [&](size_t off) { return reinterpret_cast<__nv_bfloat16*>(ws + off); };
  uint32_t* status = reinterpret_cast<uint32_t*>(ws + wl.attn_ws);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(a->x);

  // the attention step's arguments (validated like any expert_attn_layer call)
  ea_layer_args la;
  std::memset(&la, 0, sizeof(la));
  la.q_raw = bf(wl.q);
  la.k_raw = bf(wl.k);
  la.v_raw = bf(wl.v);
  la.q_gamma = a->q_norm;
  la.k_gamma = a->k_norm;
  la.k_cache = a->k_cache;
  la.v_cache = a->v_cache;
  la.out = bf(wl.attn);
  la.q_rope = a->q_rope;
  int rc = validate(&la, 1, S, Smax, rope_delta, EA_KV_BF16, ws + wl.attn_ws, true);
  if (rc != EA_OK) return rc;

  CUtensorMap xm_x, xm_attn, xm_x1, xm_gu;
  if (!rows_map(x, H, &xm_x) || !heads_map(bf(wl.attn), &xm_attn) || !rows_map(bf(wl.x1), H, &xm_x1) ||
      !rows_map(bf(wl.gu), I, &xm_gu))
    return EA_ERR_CUDA;
  // q, k, v = heads of h wqkv^T, h = rms_norm(x, ln1) (the norm fused into the projection)
  rc = run_linear(xm_x, H / 64, a->wqkv, nullptr, (kHq + 2 * kHkv) * kD, H, kLinQkvHeads, nullptr,
                  nullptr, bf(wl.q), bf(wl.k), bf(wl.v), status, di.sm_count, st, a->ln1);
  if (rc != EA_OK) return rc;
  // attention (q/k norm, RoPE, own rows into the cache tail, split-KV attention, merge)
  rc = launch_chunk(&la, 1, S, Smax, rope_delta, false, ws + wl.attn_ws, ws_layout(1, di.sm_count, false),
                    di, st, nullptr);
  if (rc != EA_OK) return rc;
  // x1 = x + concat_heads(attn) wo^T
  rc = run_linear(xm_attn, 2, a->wo, nullptr, H, kHq * kD, kLinResidual, x, bf(wl.x1), nullptr, nullptr,
                  nullptr, status, di.sm_count, st);
  if (rc != EA_OK) return rc;
  // gu = silu(h2 w1^T) * (h2 w3^T), h2 = rms_norm(x1, ln2) (fused)
  rc = run_linear(xm_x1, H / 64, a->w1, a->w3, I, H, kLinSwiglu, nullptr, bf(wl.gu), nullptr, nullptr,
                  nullptr, status, di.sm_count, st, a->ln2);
  if (rc != EA_OK) return rc;
  // x_out = x1 + gu w2^T
  return run_linear(xm_gu, I / 64, a->w2, nullptr, H, I, kLinResidual, bf(wl.x1),
                    static_cast<__nv_bfloat16*>(a->x_out), nullptr, nullptr, nullptr, status, di.sm_count, st);
}

size_t expert_linear64_workspace_size(int K, int N) {
  if (K < 64 || K % 64 != 0 || N < 128 || N % 128 != 0) return 0;
  return 1024;  // the status word (partial sums stay in the clusters' shared memory)
}

int expert_linear64(const void* x, const void* w, void* y, int K, int N, void* workspace,
                    size_t ws_bytes, ea_stream_t stream) {
  if (x == nullptr || w == nullptr || y == nullptr || workspace == nullptr) return EA_ERR_INVALID_ARG;
  if (K < 64 || K % 64 != 0 || N < 128 || N % 128 != 0 || K > (1 << 20) || N > (1 << 20))
    return EA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w) || !aligned16(y)) return EA_ERR_MISALIGNED;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return EA_ERR_MISALIGNED;
  if (ws_bytes < 1024) return EA_ERR_WORKSPACE;
  int dev;
  DeviceInfo di;
  if (!device_info(&dev, &di) || !linear_attrs_ready()) return EA_ERR_UNSUPPORTED;
  CUtensorMap xm;
  if (!rows_map(x, K, &xm)) return EA_ERR_CUDA;
  return run_linear(xm, K / 64, w, nullptr, N, K, kLinPlain, nullptr, static_cast<__nv_bfloat16*>(y),
                    nullptr, nullptr, nullptr, static_cast<uint32_t*>(workspace), di.sm_count,
                    static_cast<cudaStream_t>(stream));
}

}  // extern "C"

// ------------------------------------------------------------ text-model decode attention
// Host side of text_decode_attention: validation, the cache tensor maps (shared with the expert
// path's cache), the tile partition and one launch of the decode kernel per chunk of <= 64
// layers (programmatic dependent launch).
namespace ea {
cudaError_t decode_set_attributes();
template <int CAP>
cudaError_t launch_decode_kernel(const DecodeParams<CAP>& dp, cudaLaunchConfig_t cfg);
}  // namespace ea

namespace {

bool decode_attrs_ready() {
  static std::once_flag once;
  static bool ok = false;
  std::call_once(once, [] {
    ok = decode_set_attributes() == cudaSuccess;
    cudaGetLastError();
  });
  return ok;
}

int validate_decode(const ea_decode_args* a, int n_layers, int pos, int Smax, int rope_delta,
                    const void* ws) {
  if (a == nullptr || n_layers < 1 || ws == nullptr) return EA_ERR_INVALID_ARG;
  if (Smax < kKeyTile || Smax % kTok != 0 || Smax > (1 << 22)) return EA_ERR_INVALID_ARG;
  if (pos < 0 || pos >= Smax) return EA_ERR_INVALID_ARG;
  const long long p0 = static_cast<long long>(pos) + rope_delta;
  if (p0 <= -(1LL << 24) || p0 >= (1LL << 24)) return EA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return EA_ERR_MISALIGNED;
  for (int l = 0; l < n_layers; ++l) {
    const ea_decode_args& x = a[l];
    const void* req[] = {x.q_raw, x.k_raw, x.v_raw, x.q_gamma, x.k_gamma, x.k_cache, x.v_cache, x.out};
    for (const void* p : req) {
      if (p == nullptr) return EA_ERR_INVALID_ARG;
      if (!aligned16(p)) return EA_ERR_MISALIGNED;
    }
  }
  return EA_OK;
}

template <int CAP>
struct DecodeBlock {
  DecodeParams<CAP> dp;
  std::mutex mu;
};
template <int CAP>
DecodeBlock<CAP>& decode_block() {
  static DecodeBlock<CAP> b;
  return b;
}

template <int CAP>
int launch_decode_t(const ea_decode_args* a, int n, int pos, int Smax, int rope_delta, uint8_t* ws,
                    const DecodeWs& wl, int sm_count, cudaStream_t st) {
  DecodeBlock<CAP>& b = decode_block<CAP>();
  std::lock_guard<std::mutex> lk(b.mu);
  DecodeParams<CAP>& dp = b.dp;
  std::memset(&dp, 0, sizeof(dp));
  for (int l = 0; l < n; ++l) {
    if (!cache_map(a[l].k_cache, 0, Smax, false, &dp.kmap[l]) ||
        !cache_map(a[l].v_cache, 0, Smax, false, &dp.vmap[l]))
      return EA_ERR_CUDA;
    dp.q_raw[l] = static_cast<const __nv_bfloat16*>(a[l].q_raw);
    dp.k_raw[l] = static_cast<const __nv_bfloat16*>(a[l].k_raw);
    dp.v_raw[l] = static_cast<const __nv_bfloat16*>(a[l].v_raw);
    dp.q_gamma[l] = static_cast<const __nv_bfloat16*>(a[l].q_gamma);
    dp.k_gamma[l] = static_cast<const __nv_bfloat16*>(a[l].k_gamma);
    dp.kc[l] = static_cast<__nv_bfloat16*>(a[l].k_cache);
    dp.vc[l] = static_cast<__nv_bfloat16*>(a[l].v_cache);
    dp.out[l] = static_cast<__nv_bfloat16*>(a[l].out);
  }
  rope_inv_freq(dp.inv_hi, dp.inv_lo);
  dp.T = (pos + 1 + kKeyTile - 1) / kKeyTile;
  dp.W = static_cast<long long>(n) * kHkv * dp.T;
  dp.pos = pos;
  dp.rope_pos = pos + rope_delta;
  dp.Smax = Smax;
  dp.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(kD)));
  dp.part_o = reinterpret_cast<float*>(ws + wl.part_o_off);
  dp.part_ml = reinterpret_cast<float*>(ws + wl.part_ml_off);
  dp.unit_cnt = reinterpret_cast<uint32_t*>(ws + wl.cnt_off);
  dp.status = reinterpret_cast<uint32_t*>(ws);
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = launch_config(st, attr, true);
  if (n == 1 && dp.T >= 2 && dp.T <= 8) {
    // one layer over a short cache: a cluster of T CTAs (one per key tile) per kv head,
    // merged through distributed shared memory
    dp.cluster = dp.T;
    cfg.gridDim = dim3(kHkv * dp.cluster);
    attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
    attr[cfg.numAttrs].val.clusterDim.x = static_cast<unsigned>(dp.cluster);
    attr[cfg.numAttrs].val.clusterDim.y = 1;
    attr[cfg.numAttrs].val.clusterDim.z = 1;
    ++cfg.numAttrs;
  } else if (n == 1 && dp.T > 8) {
    // one layer over a longer cache: the same number of CTAs for every kv head (at most one per
    // key tile, at most kDecodeMaxPerUnit, whose partials fit the drained ring), so that every
    // CTA holds one segment and the last part of a unit can merge from its own shared memory
    int per = (sm_count < kMaxGridCtas ? sm_count : kMaxGridCtas) / kHkv;
    if (per > dp.T) per = dp.T;
    if (per > kDecodeMaxPerUnit) per = kDecodeMaxPerUnit;
    dp.per_unit = per;
    cfg.gridDim = dim3(kHkv * per);
  } else {
    // one CTA per SM (at most 160: the merge stages at most that many parts in shared memory)
    int n_ctas = sm_count < kMaxGridCtas ? sm_count : kMaxGridCtas;
    if (static_cast<long long>(n_ctas) > dp.W) n_ctas = static_cast<int>(dp.W);
    cfg.gridDim = dim3(n_ctas);
  }
  if (launch_decode_kernel<CAP>(dp, cfg) != cudaSuccess) {
    cudaGetLastError();
    return EA_ERR_CUDA;
  }
  return EA_OK;
}

}  // namespace

extern "C" {

size_t text_decode_workspace_size(int n_layers) {
  if (n_layers < 1) return 0;
  int dev;
  DeviceInfo di;
  if (!device_info(&dev, &di)) return 0;
  const int per = n_layers < kDecodeMaxLayers ? n_layers : kDecodeMaxLayers;
  return decode_ws_layout(per, di.sm_count).total;
}

int text_decode_workspace_init(void* workspace, size_t ws_bytes, ea_stream_t stream) {
  if (workspace == nullptr || ws_bytes < 1024) return EA_ERR_INVALID_ARG;
  // the status word and the per-unit arrival counts of up to 64 layers per launch
  const size_t init = decode_ws_layout(kDecodeMaxLayers, 1).part_o_off;
  const size_t n = ws_bytes < init ? ws_bytes : init;
  if (cudaMemsetAsync(workspace, 0, n, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return EA_ERR_CUDA;
  }
  return EA_OK;
}

int text_decode_attention(const ea_decode_args* layers, int n_layers, int pos, int Smax,
                          int rope_delta, void* workspace, size_t ws_bytes, ea_stream_t stream) {
  int rc = validate_decode(layers, n_layers, pos, Smax, rope_delta, workspace);
  if (rc != EA_OK) return rc;
  int dev;
  DeviceInfo di;
  if (!device_info(&dev, &di) || !decode_attrs_ready()) return EA_ERR_UNSUPPORTED;
  const int per = n_layers < kDecodeMaxLayers ? n_layers : kDecodeMaxLayers;
  const DecodeWs wl = decode_ws_layout(per, di.sm_count);
  if (ws_bytes < wl.total) return EA_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  for (int l0 = 0; l0 < n_layers; l0 += per) {
    const int n = n_layers - l0 < per ? n_layers - l0 : per;
    rc = n <= kSmallCap ? launch_decode_t<kSmallCap>(layers + l0, n, pos, Smax, rope_delta, ws, wl, di.sm_count, st)
                        : launch_decode_t<kDecodeMaxLayers>(layers + l0, n, pos, Smax, rope_delta, ws, wl,
                                                            di.sm_count, st);
    if (rc != EA_OK) return rc;
  }
  return EA_OK;
}

}  // extern "C"
