// pkv_api.cu -- the extern "C" entry points of libpkv (declared in pkv.h):
// host-side validation, per-device state (error word, decode workspace,
// tensor-map cache), the split-K plan, and the kernel-timing profiler.
//
// The device error word is a file-scope __device__ variable: every device
// that loads the library has its own copy, and no call has to allocate
// memory to report a device-side check.  Host code reaches it through the
// address cudaGetSymbolAddress gives for the current device (the variable's
// name on the host is only a stand-in).
#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "pkv.h"
#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "pkv_pair_gap.h"

namespace {

using pkv::CacheMaps;
using pkv::DeviceError;

constexpr int kMaxDevices = 64;
constexpr int kMapCacheSize = 8;

// One error word per device (first recorded error code and its site).
__device__ DeviceError g_device_error;

struct MapEntry {
  const void* k = nullptr;
  const void* v = nullptr;
  int64_t num_blocks = 0;
  int hkv = 0, d = 0;
  uint64_t stamp = 0;
  CacheMaps maps;
};

struct DeviceState {
  bool ready = false;
  bool usable = false;
  int num_sms = 0;
  DeviceError* err = nullptr;
  float* ws = nullptr;  // decode partials
  size_t ws_bytes = 0;
  unsigned long long* cnt = nullptr;  // decode arrival counters (zeroed once)
  size_t cnt_bytes = 0;
  float* sh = nullptr;  // cascade decode: shared-prefix partial states
  size_t sh_bytes = 0;
  MapEntry maps[kMapCacheSize];
  uint64_t clock = 0;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
pkv::EncodeTiledFn g_encode = nullptr;
std::atomic<int> g_max_splits{0};
std::atomic<int> g_shared_units{0};
std::atomic<int64_t> g_wait_limit_ns{1000000000};

// ------------------------------------------------------------------ profiler
struct ProfRecord {
  const char* name;
  cudaEvent_t start, stop;
};
std::mutex g_prof_mu;
std::atomic<int> g_prof_on{0};
std::vector<ProfRecord> g_prof;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t take_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

template <typename F>
cudaError_t timed_launch(const char* name, cudaStream_t stream, F&& launch) {
  if (!g_prof_on.load()) return launch();
  std::lock_guard<std::mutex> lk(g_prof_mu);
  cudaEvent_t a = take_event(), b = take_event();
  if (!a || !b) return cudaErrorMemoryAllocation;
  cudaEventRecord(a, stream);
  cudaError_t e = launch();
  cudaEventRecord(b, stream);
  g_prof.push_back({name, a, b});
  return e;
}

// ------------------------------------------------------------------ helpers
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

pkv_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return PKV_OK;
  if (e == cudaErrorMemoryAllocation) return PKV_ERR_NO_MEMORY;
  return PKV_ERR_CUDA;
}

bool load_encoder() {
  if (g_encode) return true;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return false;
  g_encode = reinterpret_cast<pkv::EncodeTiledFn>(fn);
  return true;
}

// Must be called with g_mu held.  Set-up allocates nothing: it checks the
// architecture, finds the tensor-map encoder and looks up the device address
// of the error word.  A device that is not sm_103a is marked unusable for
// good; any other failure (a lookup refused while a stream is being
// captured, say) is retried by the next call.
DeviceState* device_state(pkv_status* st) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    *st = PKV_ERR_CUDA;
    return nullptr;
  }
  DeviceState& d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0;
    const bool attrs =
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess;
    void* err = nullptr;
    if (attrs && !(major == 10 && minor == 3)) {
      d.ready = true;  // not an sm_103a device: never usable
      d.usable = false;
    } else if (attrs && load_encoder() &&
               cudaGetSymbolAddress(&err, g_device_error) == cudaSuccess && err != nullptr) {
      d.err = static_cast<DeviceError*>(err);
      d.num_sms = sms;
      d.ready = true;
      d.usable = true;
    }
    cudaGetLastError();
  }
  if (!d.ready || !d.usable) {
    *st = PKV_ERR_CUDA;
    return nullptr;
  }
  *st = PKV_OK;
  return &d;
}

bool encode_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
               uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1,
               uint32_t b2, CUtensorMapSwizzle swz,
               CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  const cuuint32_t box[3] = {b0, b1, b2};
  const cuuint32_t elem[3] = {1, 1, 1};
  return g_encode(map, dtype, 3, const_cast<void*>(base), dims, strides, box, elem,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor maps over INT8 codes [num_blocks][Hkv][256][D] bytes viewed as 3-D
// {D, 256, num_blocks * Hkv}; a box of `rows` consecutive tokens of one
// (block, KV head) is one contiguous tile.  The decode takes 64 rows (one
// INT8 chunk) with the 128-byte swizzle for D = 128 and 64-byte for D = 64
// (the swizzle span is the row); the prefill takes 64 rows unswizzled (its
// producers dequantise them with plain loads).
bool encode_int8_maps(CUtensorMap* kmap, CUtensorMap* vmap, const void* k, const void* v,
                      int64_t num_blocks, int hkv, int d, bool prefill = false) {
  const uint64_t tiles = static_cast<uint64_t>(num_blocks) * hkv;
  const uint64_t blk = pkv::kBlockSize;
  const uint32_t rows = prefill ? pkv::kPrefillKeyTile : 2 * pkv::kDecodeChunk;
  const CUtensorMapSwizzle swz = prefill    ? CU_TENSOR_MAP_SWIZZLE_NONE
                                 : d == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                            : CU_TENSOR_MAP_SWIZZLE_64B;
  return encode_3d(kmap, k, d, blk, tiles, d, blk * d, d, rows, 1, swz,
                   CU_TENSOR_MAP_DATA_TYPE_UINT8) &&
         encode_3d(vmap, v, d, blk, tiles, d, blk * d, d, rows, 1, swz,
                   CU_TENSOR_MAP_DATA_TYPE_UINT8);
}

// Tensor maps over the cache viewed as [slots][Hkv][D] (3-D: D, Hkv, slots).
const CacheMaps* cache_maps(DeviceState* ds, const void* k, const void* v, int64_t num_blocks,
                            int hkv, int d) {
  ++ds->clock;
  for (auto& e : ds->maps) {
    if (e.k == k && e.v == v && e.num_blocks == num_blocks && e.hkv == hkv && e.d == d) {
      e.stamp = ds->clock;
      return &e.maps;
    }
  }
  MapEntry* victim = &ds->maps[0];
  for (auto& e : ds->maps)
    if (e.stamp < victim->stamp) victim = &e;
  MapEntry e;
  if (!pkv::encode_cache_maps(&e.maps, k, v, num_blocks, hkv, d)) return nullptr;
  e.k = k;
  e.v = v;
  e.num_blocks = num_blocks;
  e.hkv = hkv;
  e.d = d;
  e.stamp = ds->clock;
  *victim = e;
  return &victim->maps;
}

bool supported_group(int g) { return g == 1 || g == 2 || g == 4 || g == 8 || g == 16; }

// Grows the decode partials to `part_bytes` and the counter region to
// `cnt_bytes`.  The counters are zeroed when allocated and never reset
// afterwards (the kernel tags them with a generation it keeps on the
// device, so captured graphs replay correctly).
pkv_status ensure_workspace(DeviceState* ds, size_t part_bytes, size_t cnt_bytes) {
  if (part_bytes > ds->ws_bytes) {
    if (ds->ws) cudaFree(ds->ws);
    ds->ws = nullptr;
    ds->ws_bytes = 0;
    if (cudaMalloc(&ds->ws, part_bytes) != cudaSuccess) {
      cudaGetLastError();
      return PKV_ERR_NO_MEMORY;
    }
    ds->ws_bytes = part_bytes;
  }
  if (cnt_bytes > ds->cnt_bytes) {
    if (ds->cnt) cudaFree(ds->cnt);
    ds->cnt = nullptr;
    ds->cnt_bytes = 0;
    if (cudaMalloc(&ds->cnt, cnt_bytes) != cudaSuccess) {
      cudaGetLastError();
      return PKV_ERR_NO_MEMORY;
    }
    if (cudaMemset(ds->cnt, 0, cnt_bytes) != cudaSuccess) {
      cudaFree(ds->cnt);
      ds->cnt = nullptr;
      cudaGetLastError();
      return PKV_ERR_CUDA;
    }
    ds->cnt_bytes = cnt_bytes;
  }
  return PKV_OK;
}

// Grows the cascade decode's shared-prefix partial buffer.
pkv_status ensure_shared_workspace(DeviceState* ds, size_t bytes) {
  if (bytes <= ds->sh_bytes) return PKV_OK;
  if (ds->sh) cudaFree(ds->sh);
  ds->sh = nullptr;
  ds->sh_bytes = 0;
  if (cudaMalloc(&ds->sh, bytes) != cudaSuccess) {
    cudaGetLastError();
    return PKV_ERR_NO_MEMORY;
  }
  ds->sh_bytes = bytes;
  return PKV_OK;
}

// Cascade decode plan: row tiles of 128 / G sequences, and the units (one
// cluster of CTAs per row tile and KV head, a power of two up to 16) the
// shared prefix's key tiles are cut into: a set value, or the most that
// keep the grid within one CTA per SM (at most 8, the portable cluster
// size).  The cluster merges its units, so one partial state per row
// remains: KV heads x padded rows x (head_dim + 2) fp32, and the decode's
// private states of the same rows after them.
struct SharedPlan {
  int tiles;     // row tiles
  int units;
  int rows_pad;  // tiles * 128
  int key_tiles;
  size_t bytes;
};

SharedPlan shared_plan(int num_seqs, int hkv, int group, int head_dim, int shared_blocks,
                       int num_sms) {
  SharedPlan p;
  const int qt = 128 / group;
  p.tiles = (num_seqs + qt - 1) / qt;
  p.rows_pad = p.tiles * 128;
  p.key_tiles = shared_blocks * (pkv::kBlockSize / pkv::kPrefillKeyTile);
  const int set = g_shared_units.load();
  const int want = set > 0 ? set : std::min(8, num_sms / std::max(1, hkv * p.tiles));
  int u = 1;
  while (u * 2 <= want && u * 2 <= p.key_tiles && u * 2 <= 16) u *= 2;
  p.units = u;
  // The shared partial states, then as many rows of private states.
  const size_t rows = static_cast<size_t>(hkv) * p.rows_pad;
  p.bytes = 2 * (rows * head_dim * sizeof(float) + rows * 2 * sizeof(float));
  return p;
}

}  // namespace

namespace pkv {

int max_splits_setting() { return g_max_splits.load(); }

// Tensor maps over the cache viewed as [slots][Hkv][D] (3-D: D, Hkv, slots).
bool encode_cache_maps(CacheMaps* maps, const void* k, const void* v, int64_t num_blocks, int hkv,
                       int d) {
  const uint64_t slots = static_cast<uint64_t>(num_blocks) * kBlockSize;
  const uint64_t s1 = static_cast<uint64_t>(d) * 2;
  const uint64_t s2 = static_cast<uint64_t>(hkv) * d * 2;
  return encode_3d(&maps->k_rows, k, d, hkv, slots, s1, s2, 64, 1, kDecodeChunk,
                   CU_TENSOR_MAP_SWIZZLE_128B) &&
         encode_3d(&maps->v_rows, v, d, hkv, slots, s1, s2, 64, 1, kDecodeChunk,
                   CU_TENSOR_MAP_SWIZZLE_128B) &&
         encode_3d(&maps->k_sw128, k, d, hkv, slots, s1, s2, 64, 1, kPrefillKeyTile,
                   CU_TENSOR_MAP_SWIZZLE_128B) &&
         encode_3d(&maps->v_sw128, v, d, hkv, slots, s1, s2, 64, 1, kPrefillKeyTile,
                   CU_TENSOR_MAP_SWIZZLE_128B);
}

bool load_tensor_map_encoder() { return load_encoder(); }

DeviceError* device_error_word() {
  std::lock_guard<std::mutex> lk(g_mu);
  pkv_status st;
  DeviceState* ds = device_state(&st);
  return ds ? ds->err : nullptr;
}

uint64_t wait_limit_ns() { return static_cast<uint64_t>(g_wait_limit_ns.load()); }

pkv_status validate_attention_args(const void* q, int64_t q_row_stride, const void* k_cache,
                                   const void* v_cache, int64_t num_blocks,
                                   const int32_t* block_tables, int32_t max_blocks,
                                   const int32_t* lens, int32_t num_seqs, int32_t hq, int32_t hkv,
                                   int32_t d, const void* out) {
  if (num_seqs < 0 || num_blocks <= 0 || max_blocks <= 0 || hq <= 0 || hkv <= 0)
    return PKV_ERR_INVALID_ARG;
  if (!k_cache || !v_cache || !q || !block_tables || !lens || !out) return PKV_ERR_INVALID_ARG;
  if (hq % hkv != 0) return PKV_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return PKV_ERR_UNSUPPORTED;
  if (!supported_group(hq / hkv)) return PKV_ERR_UNSUPPORTED;
  if (q_row_stride < static_cast<int64_t>(hq) * d) return PKV_ERR_INVALID_ARG;
  if ((q_row_stride * 2) % 16) return PKV_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return PKV_ERR_UNSUPPORTED;
  if (num_blocks > (int64_t{1} << 31) / pkv::kBlockSize ||
      max_blocks > (int64_t{1} << 31) / pkv::kBlockSize)
    return PKV_ERR_UNSUPPORTED;
  return PKV_OK;
}

}  // namespace pkv

extern "C" {

const char* pkv_status_string(pkv_status s) {
  switch (s) {
    case PKV_OK: return "PKV_OK";
    case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG";
    case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
    case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
    case PKV_ERR_DEVICE_CHECK: return "PKV_ERR_DEVICE_CHECK";
    case PKV_ERR_TIMEOUT: return "PKV_ERR_TIMEOUT";
    case PKV_ERR_NO_MEMORY: return "PKV_ERR_NO_MEMORY";
  }
  return "PKV_ERR_UNKNOWN";
}

const char* pkv_version(void) { return "pkv 0.1.0 sm_103a"; }

pkv_status pkv_store_kvcache(const void* k, const void* v, int64_t k_row_stride,
                             int64_t v_row_stride, const int32_t* slot_mapping,
                             int64_t num_tokens, void* k_cache, void* v_cache,
                             int64_t num_blocks, int32_t num_kv_heads, int32_t head_dim,
                             pkv_stream_t stream) {
  if (num_tokens < 0 || num_blocks <= 0 || num_kv_heads <= 0 || head_dim <= 0)
    return PKV_ERR_INVALID_ARG;
  if (!k_cache || !v_cache) return PKV_ERR_INVALID_ARG;
  if (num_tokens > 0 && (!k || !v || !slot_mapping)) return PKV_ERR_INVALID_ARG;
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (k_row_stride < row || v_row_stride < row) return PKV_ERR_INVALID_ARG;
  if ((row * 2) % 16 || (k_row_stride * 2) % 16 || (v_row_stride * 2) % 16)
    return PKV_ERR_UNSUPPORTED;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_UNSUPPORTED;
  if (num_blocks > (int64_t{1} << 31) / pkv::kBlockSize) return PKV_ERR_UNSUPPORTED;
  pkv_status st;
  DeviceState* ds;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    ds = device_state(&st);
  }
  if (!ds) return st;
  if (num_tokens == 0) return PKV_OK;
  pkv::StoreArgs a{k, v, k_row_stride, v_row_stride, slot_mapping, num_tokens, k_cache, v_cache,
                   num_blocks, num_kv_heads, head_dim, ds->err};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return cuda_status(
      timed_launch("store_kvcache", s, [&] { return pkv::launch_store_kvcache(a, s); }));
}

pkv_status pkv_store_kvcache_int8(const void* k, const void* v, int64_t k_row_stride,
                                  int64_t v_row_stride, const int32_t* slot_mapping,
                                  int64_t num_tokens, int8_t* k_codes, int8_t* v_codes,
                                  float* k_scales, float* v_scales, int64_t num_blocks,
                                  int32_t num_kv_heads, int32_t head_dim, pkv_stream_t stream) {
  if (num_tokens < 0 || num_blocks <= 0 || num_kv_heads <= 0 || head_dim <= 0)
    return PKV_ERR_INVALID_ARG;
  if (!k_codes || !v_codes || !k_scales || !v_scales) return PKV_ERR_INVALID_ARG;
  if (num_tokens > 0 && (!k || !v || !slot_mapping)) return PKV_ERR_INVALID_ARG;
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (k_row_stride < row || v_row_stride < row) return PKV_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if ((k_row_stride * 2) % 16 || (v_row_stride * 2) % 16) return PKV_ERR_UNSUPPORTED;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_codes) || !aligned16(v_codes) ||
      !aligned16(k_scales) || !aligned16(v_scales))
    return PKV_ERR_UNSUPPORTED;
  if (num_blocks > (int64_t{1} << 31) / pkv::kBlockSize) return PKV_ERR_UNSUPPORTED;
  pkv_status st;
  DeviceState* ds;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    ds = device_state(&st);
  }
  if (!ds) return st;
  if (num_tokens == 0) return PKV_OK;
  pkv::StoreI8Args a{k, v, k_row_stride, v_row_stride, slot_mapping, num_tokens, k_codes,
                     v_codes, k_scales, v_scales, num_blocks, num_kv_heads, head_dim, ds->err};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return cuda_status(timed_launch("store_kvcache_int8", s,
                                  [&] { return pkv::launch_store_kvcache_int8(a, s); }));
}

pkv_status pkv_decode_attention_int8(const void* q, int64_t q_row_stride, const int8_t* k_codes,
                                     const int8_t* v_codes, const float* k_scales,
                                     const float* v_scales, int64_t num_blocks,
                                     const int32_t* block_tables, int32_t max_blocks_per_seq,
                                     const int32_t* context_lens, int32_t num_seqs,
                                     int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                     float scale, void* out, pkv_stream_t stream) {
  pkv_status st = pkv::validate_attention_args(q, q_row_stride, k_codes, v_codes, num_blocks,
                                               block_tables, max_blocks_per_seq, context_lens,
                                               num_seqs, num_q_heads, num_kv_heads, head_dim, out);
  if (st != PKV_OK) return st;
  if (!k_scales || !v_scales) return PKV_ERR_INVALID_ARG;
  if (!aligned16(k_scales) || !aligned16(v_scales)) return PKV_ERR_UNSUPPORTED;
  // The split-K decode kernel over the codes (TMA ring, tensor cores, the
  // same stream-K plan and in-kernel merge as the bf16 decode).
  pkv::DecodeArgs a{};
  CUtensorMap kmap, vmap;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState* ds = device_state(&st);
    if (!ds) return st;
    if (num_seqs == 0) return PKV_OK;
    if (!encode_int8_maps(&kmap, &vmap, k_codes, v_codes, num_blocks, num_kv_heads, head_dim))
      return PKV_ERR_CUDA;
    a.q = q;
    a.q_row_stride = q_row_stride;
    a.block_tables = block_tables;
    a.max_blocks = max_blocks_per_seq;
    a.context_lens = context_lens;
    a.num_seqs = num_seqs;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.num_blocks = num_blocks;
    a.scale = scale;
    a.out = out;
    a.wait_limit_ns = static_cast<uint64_t>(g_wait_limit_ns.load());
    a.err = ds->err;
    a.k_scales = k_scales;
    a.v_scales = v_scales;
    const int g = num_q_heads / num_kv_heads;
    const int64_t pairs = static_cast<int64_t>(num_seqs) * num_kv_heads;
    a.num_ctas =
        pkv::decode_num_ctas(head_dim, g, ds->num_sms, pairs, g_max_splits.load(), true);
    a.pair_gap = pkv::kPairGapInt8;
    st = ensure_workspace(ds, pkv::decode_partial_bytes(a.num_ctas, g, head_dim),
                          pkv::decode_counter_bytes(pairs));
    if (st != PKV_OK) return st;
    a.counters = ds->cnt;
    a.part_o = ds->ws;
    a.part_ml = a.part_o + static_cast<size_t>(a.num_ctas) * 2 * g * head_dim;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return cuda_status(
      timed_launch("decode_int8", s, [&] { return pkv::launch_decode_i8(a, kmap, vmap, s); }));
}

pkv_status pkv_decode_attention(const void* q, int64_t q_row_stride, const void* k_cache,
                                const void* v_cache, int64_t num_blocks,
                                const int32_t* block_tables, int32_t max_blocks_per_seq,
                                const int32_t* context_lens, int32_t num_seqs,
                                int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                float scale, void* out, pkv_stream_t stream) {
  pkv_status st = pkv::validate_attention_args(q, q_row_stride, k_cache, v_cache, num_blocks,
                                               block_tables, max_blocks_per_seq, context_lens,
                                               num_seqs, num_q_heads, num_kv_heads, head_dim, out);
  if (st != PKV_OK) return st;
  pkv::DecodeArgs a{};
  const CacheMaps* maps = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState* ds = device_state(&st);
    if (!ds) return st;
    if (num_seqs == 0) return PKV_OK;
    maps = cache_maps(ds, k_cache, v_cache, num_blocks, num_kv_heads, head_dim);
    if (!maps) return PKV_ERR_CUDA;
    a.q = q;
    a.q_row_stride = q_row_stride;
    a.block_tables = block_tables;
    a.max_blocks = max_blocks_per_seq;
    a.context_lens = context_lens;
    a.num_seqs = num_seqs;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.num_blocks = num_blocks;
    a.scale = scale;
    a.out = out;
    a.wait_limit_ns = static_cast<uint64_t>(g_wait_limit_ns.load());
    a.err = ds->err;
    // Stream-K plan: one slice of the pairs' chunks per block; the workspace
    // holds two partial slots per block, the counters one word per pair.
    const int g = num_q_heads / num_kv_heads;
    const int64_t pairs = static_cast<int64_t>(num_seqs) * num_kv_heads;
    a.num_ctas = pkv::decode_num_ctas(head_dim, g, ds->num_sms, pairs, g_max_splits.load());
    a.pair_gap = pkv::kPairGapDecode;
    st = ensure_workspace(ds, pkv::decode_partial_bytes(a.num_ctas, g, head_dim),
                          pkv::decode_counter_bytes(pairs));
    if (st != PKV_OK) return st;
    a.counters = ds->cnt;
    a.part_o = ds->ws;
    a.part_ml = a.part_o + static_cast<size_t>(a.num_ctas) * 2 * g * head_dim;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const CacheMaps m = *maps;
  return cuda_status(
      timed_launch("decode", s, [&] { return pkv::launch_decode(a, m, s); }));
}

pkv_status pkv_decode_attention_append(const void* q, int64_t q_row_stride, const void* k_new,
                                       const void* v_new, int64_t k_row_stride,
                                       int64_t v_row_stride, const int32_t* slot_mapping,
                                       void* k_cache, void* v_cache, int64_t num_blocks,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* context_lens, int32_t num_seqs,
                                       int32_t num_q_heads, int32_t num_kv_heads,
                                       int32_t head_dim, float scale, void* out,
                                       pkv_stream_t stream) {
  pkv_status st = pkv::validate_attention_args(q, q_row_stride, k_cache, v_cache, num_blocks,
                                               block_tables, max_blocks_per_seq, context_lens,
                                               num_seqs, num_q_heads, num_kv_heads, head_dim, out);
  if (st != PKV_OK) return st;
  if (num_seqs > 0 && (!k_new || !v_new || !slot_mapping)) return PKV_ERR_INVALID_ARG;
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (k_row_stride < row || v_row_stride < row) return PKV_ERR_INVALID_ARG;
  if ((k_row_stride * 2) % 16 || (v_row_stride * 2) % 16) return PKV_ERR_UNSUPPORTED;
  if (!aligned16(k_new) || !aligned16(v_new)) return PKV_ERR_UNSUPPORTED;
  pkv::DecodeArgs a{};
  const CacheMaps* maps = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState* ds = device_state(&st);
    if (!ds) return st;
    if (num_seqs == 0) return PKV_OK;
    maps = cache_maps(ds, k_cache, v_cache, num_blocks, num_kv_heads, head_dim);
    if (!maps) return PKV_ERR_CUDA;
    a.q = q;
    a.q_row_stride = q_row_stride;
    a.block_tables = block_tables;
    a.max_blocks = max_blocks_per_seq;
    a.context_lens = context_lens;
    a.num_seqs = num_seqs;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.num_blocks = num_blocks;
    a.scale = scale;
    a.out = out;
    a.wait_limit_ns = static_cast<uint64_t>(g_wait_limit_ns.load());
    a.err = ds->err;
    const int g = num_q_heads / num_kv_heads;
    const int64_t pairs = static_cast<int64_t>(num_seqs) * num_kv_heads;
    a.num_ctas = pkv::decode_num_ctas(head_dim, g, ds->num_sms, pairs, g_max_splits.load());
    a.pair_gap = pkv::kPairGapDecode;
    st = ensure_workspace(ds, pkv::decode_partial_bytes(a.num_ctas, g, head_dim),
                          pkv::decode_counter_bytes(pairs));
    if (st != PKV_OK) return st;
    a.counters = ds->cnt;
    a.part_o = ds->ws;
    a.part_ml = a.part_o + static_cast<size_t>(a.num_ctas) * 2 * g * head_dim;
    a.k_new = k_new;
    a.v_new = v_new;
    a.k_new_stride = k_row_stride;
    a.v_new_stride = v_row_stride;
    a.slot_mapping = slot_mapping;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const CacheMaps m = *maps;
  return cuda_status(
      timed_launch("decode_append", s, [&] { return pkv::launch_decode(a, m, s); }));
}

pkv_status pkv_decode_attention_shared_prefix(
    const void* q, int64_t q_row_stride, const void* k_cache, const void* v_cache,
    int64_t num_blocks, const int32_t* block_tables, int32_t max_blocks_per_seq,
    const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_dim, float scale, int32_t shared_blocks, void* out, pkv_stream_t stream) {
  pkv_status st = pkv::validate_attention_args(q, q_row_stride, k_cache, v_cache, num_blocks,
                                               block_tables, max_blocks_per_seq, context_lens,
                                               num_seqs, num_q_heads, num_kv_heads, head_dim, out);
  if (st != PKV_OK) return st;
  if (shared_blocks < 0 || shared_blocks > max_blocks_per_seq) return PKV_ERR_INVALID_ARG;
  if (shared_blocks == 0)
    return pkv_decode_attention(q, q_row_stride, k_cache, v_cache, num_blocks, block_tables,
                                max_blocks_per_seq, context_lens, num_seqs, num_q_heads,
                                num_kv_heads, head_dim, scale, out, stream);
  pkv::DecodeArgs a{};
  pkv::PrefillArgs sp{};
  CacheMaps m;
  CUtensorMap qmap;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState* ds = device_state(&st);
    if (!ds) return st;
    if (num_seqs == 0) return PKV_OK;
    const CacheMaps* maps = cache_maps(ds, k_cache, v_cache, num_blocks, num_kv_heads, head_dim);
    if (!maps) return PKV_ERR_CUDA;
    m = *maps;
    const int g = num_q_heads / num_kv_heads;
    // The decode queries viewed as {D, Hq, num_seqs}: a box holds the G
    // heads of one KV head for 128 / G sequences (128 MMA rows).
    if (!encode_3d(&qmap, q, head_dim, num_q_heads, num_seqs,
                   static_cast<uint64_t>(head_dim) * 2, static_cast<uint64_t>(q_row_stride) * 2,
                   64, g, 128 / g, CU_TENSOR_MAP_SWIZZLE_128B))
      return PKV_ERR_CUDA;
    const SharedPlan plan =
        shared_plan(num_seqs, num_kv_heads, g, head_dim, shared_blocks, ds->num_sms);
    st = ensure_shared_workspace(ds, plan.bytes);
    if (st != PKV_OK) return st;
    const int64_t pairs = static_cast<int64_t>(num_seqs) * num_kv_heads;
    int num_ctas = pkv::decode_num_ctas(head_dim, g, ds->num_sms, pairs, g_max_splits.load());
    // The decode starts while the shared-prefix kernel still runs, and each
    // of that kernel's CTAs holds one decode slot of its SM.  A grid of the
    // slots left starts whole and streams the private parts meanwhile; a
    // full grid would leave its last blocks to start, each with a full
    // slice, only once the shared kernel is done.
    const int64_t shared_ctas = static_cast<int64_t>(plan.tiles) * plan.units * num_kv_heads;
    const int64_t free_slots =
        pkv::decode_num_ctas(head_dim, g, ds->num_sms, pairs, 0) - shared_ctas;
    if (free_slots >= ds->num_sms && num_ctas > free_slots) num_ctas = static_cast<int>(free_slots);
    st = ensure_workspace(ds, pkv::decode_partial_bytes(num_ctas, g, head_dim),
                          pkv::decode_counter_bytes(pairs));
    if (st != PKV_OK) return st;
    const size_t sh_rows = static_cast<size_t>(num_kv_heads) * plan.rows_pad;
    float* sh_o = ds->sh;
    float* sh_ml = sh_o + sh_rows * head_dim;
    float* pv_o = sh_ml + sh_rows * 2;
    float* pv_ml = pv_o + sh_rows * head_dim;
    const uint64_t wait = static_cast<uint64_t>(g_wait_limit_ns.load());

    sp.q = q;
    sp.q_row_stride = q_row_stride;
    sp.block_tables = block_tables;
    sp.max_blocks = max_blocks_per_seq;
    sp.num_seqs = num_seqs;
    sp.total_q = num_seqs;
    sp.num_q_heads = num_q_heads;
    sp.num_kv_heads = num_kv_heads;
    sp.head_dim = head_dim;
    sp.num_blocks = num_blocks;
    sp.scale = scale;
    sp.wait_limit_ns = wait;
    sp.err = ds->err;
    sp.shared_tiles = plan.key_tiles;
    sp.shared_units = plan.units;
    sp.shared_rows_pad = plan.rows_pad;
    sp.shared_o = sh_o;
    sp.shared_ml = sh_ml;

    a.q = q;
    a.q_row_stride = q_row_stride;
    a.block_tables = block_tables;
    a.max_blocks = max_blocks_per_seq;
    a.context_lens = context_lens;
    a.num_seqs = num_seqs;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.num_blocks = num_blocks;
    a.scale = scale;
    a.out = out;
    a.wait_limit_ns = wait;
    a.err = ds->err;
    a.num_ctas = num_ctas;
    a.pair_gap = pkv::kPairGapCascade;
    a.counters = ds->cnt;
    a.part_o = ds->ws;
    a.part_ml = a.part_o + static_cast<size_t>(num_ctas) * 2 * g * head_dim;
    a.shared_len = shared_blocks * pkv::kBlockSize;
    a.shared_units = 1;  // the cluster merged the units: one state per row
    a.shared_rows_pad = plan.rows_pad;
    a.shared_o = sh_o;
    a.shared_ml = sh_ml;
    a.private_o = pv_o;
    a.private_ml = pv_ml;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = timed_launch("shared_prefix", s,
                               [&] { return pkv::launch_shared_prefix(sp, m, qmap, s); });
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(timed_launch("decode", s, [&] { return pkv::launch_decode(a, m, s); }));
}

pkv_status pkv_set_shared_prefix_units(int32_t units) {
  if (units < 0 || units > 16 || (units & (units - 1))) return PKV_ERR_INVALID_ARG;
  g_shared_units.store(units);
  return PKV_OK;
}

pkv_status pkv_prefill_attention(const void* q, int64_t q_row_stride, const void* k_cache,
                                 const void* v_cache, int64_t num_blocks,
                                 const int32_t* block_tables, int32_t max_blocks_per_seq,
                                 const int32_t* cu_seqlens_q, const int32_t* context_lens,
                                 int32_t num_seqs, int64_t total_q, int32_t num_q_heads,
                                 int32_t num_kv_heads, int32_t head_dim, float scale, void* out,
                                 pkv_stream_t stream) {
  pkv_status st = pkv::validate_attention_args(q, q_row_stride, k_cache, v_cache, num_blocks,
                                               block_tables, max_blocks_per_seq, context_lens,
                                               num_seqs, num_q_heads, num_kv_heads, head_dim, out);
  if (st != PKV_OK) return st;
  if (!cu_seqlens_q || total_q < 0 || total_q > 0x7FFFFFFF) return PKV_ERR_INVALID_ARG;
  pkv::PrefillArgs a{};
  CacheMaps m;
  CUtensorMap qmap;
  int num_sms = 0;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState* ds = device_state(&st);
    if (!ds) return st;
    if (num_seqs == 0 || total_q == 0) return PKV_OK;
    const CacheMaps* maps = cache_maps(ds, k_cache, v_cache, num_blocks, num_kv_heads, head_dim);
    if (!maps) return PKV_ERR_CUDA;
    m = *maps;
    const int g = num_q_heads / num_kv_heads;
    if (!encode_3d(&qmap, q, head_dim, num_q_heads, total_q, static_cast<uint64_t>(head_dim) * 2,
                   static_cast<uint64_t>(q_row_stride) * 2, 64, g, 128 / g,
                   CU_TENSOR_MAP_SWIZZLE_128B))
      return PKV_ERR_CUDA;
    num_sms = ds->num_sms;
    a.q = q;
    a.q_row_stride = q_row_stride;
    a.block_tables = block_tables;
    a.max_blocks = max_blocks_per_seq;
    a.cu_seqlens_q = cu_seqlens_q;
    a.context_lens = context_lens;
    a.num_seqs = num_seqs;
    a.total_q = total_q;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.num_blocks = num_blocks;
    a.scale = scale;
    a.out = out;
    a.wait_limit_ns = static_cast<uint64_t>(g_wait_limit_ns.load());
    a.err = ds->err;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return cuda_status(
      timed_launch("prefill", s, [&] { return pkv::launch_prefill(a, m, qmap, num_sms, s); }));
}

pkv_status pkv_prefill_attention_int8(const void* q, int64_t q_row_stride, const int8_t* k_codes,
                                      const int8_t* v_codes, const float* k_scales,
                                      const float* v_scales, int64_t num_blocks,
                                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                                      const int32_t* cu_seqlens_q, const int32_t* context_lens,
                                      int32_t num_seqs, int64_t total_q, int32_t num_q_heads,
                                      int32_t num_kv_heads, int32_t head_dim, float scale,
                                      void* out, pkv_stream_t stream) {
  pkv_status st = pkv::validate_attention_args(q, q_row_stride, k_codes, v_codes, num_blocks,
                                               block_tables, max_blocks_per_seq, context_lens,
                                               num_seqs, num_q_heads, num_kv_heads, head_dim, out);
  if (st != PKV_OK) return st;
  if (!cu_seqlens_q || total_q < 0 || total_q > 0x7FFFFFFF) return PKV_ERR_INVALID_ARG;
  if (!k_scales || !v_scales) return PKV_ERR_INVALID_ARG;
  if (!aligned16(k_scales) || !aligned16(v_scales)) return PKV_ERR_UNSUPPORTED;
  pkv::PrefillArgs a{};
  CUtensorMap kmap, vmap, qmap;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState* ds = device_state(&st);
    if (!ds) return st;
    if (num_seqs == 0 || total_q == 0) return PKV_OK;
    if (!encode_int8_maps(&kmap, &vmap, k_codes, v_codes, num_blocks, num_kv_heads, head_dim,
                          true))
      return PKV_ERR_CUDA;
    const int g = num_q_heads / num_kv_heads;
    if (!encode_3d(&qmap, q, head_dim, num_q_heads, total_q, static_cast<uint64_t>(head_dim) * 2,
                   static_cast<uint64_t>(q_row_stride) * 2, 64, g, 128 / g,
                   CU_TENSOR_MAP_SWIZZLE_128B))
      return PKV_ERR_CUDA;
    a.q = q;
    a.q_row_stride = q_row_stride;
    a.block_tables = block_tables;
    a.max_blocks = max_blocks_per_seq;
    a.cu_seqlens_q = cu_seqlens_q;
    a.context_lens = context_lens;
    a.num_seqs = num_seqs;
    a.total_q = total_q;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.num_blocks = num_blocks;
    a.scale = scale;
    a.out = out;
    a.wait_limit_ns = static_cast<uint64_t>(g_wait_limit_ns.load());
    a.err = ds->err;
    a.k_scales = k_scales;
    a.v_scales = v_scales;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return cuda_status(timed_launch("prefill_int8", s, [&] {
    return pkv::launch_prefill_i8(a, kmap, vmap, qmap, s);
  }));
}

pkv_status pkv_get_device_error(pkv_stream_t stream, int32_t* code, int32_t* info) {
  if (!code) return PKV_ERR_INVALID_ARG;
  pkv_status st;
  DeviceState* ds;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    ds = device_state(&st);
  }
  if (!ds) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return PKV_ERR_CUDA;
  DeviceError h{0, 0};
  if (cudaMemcpy(&h, ds->err, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess) return PKV_ERR_CUDA;
  if (cudaMemset(ds->err, 0, sizeof h) != cudaSuccess) return PKV_ERR_CUDA;
  *code = h.code;
  if (info) *info = h.info;
  return PKV_OK;
}

pkv_status pkv_set_max_splits(int32_t max_splits) {
  if (max_splits < 0) return PKV_ERR_INVALID_ARG;
  g_max_splits.store(max_splits);
  return PKV_OK;
}

pkv_status pkv_reserve_workspace(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                                 int32_t max_blocks_per_seq) {
  if (num_seqs < 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0 ||
      (head_dim != 64 && head_dim != 128))
    return PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  pkv_status st;
  DeviceState* ds = device_state(&st);
  if (!ds) return st;
  // Worst case over the group sizes num_q_heads allows (the call does not
  // name num_kv_heads).
  size_t part = 0, cnt = 0, shared = 0;
  for (int g = 1; g <= 16; g *= 2) {
    if (num_q_heads % g) continue;
    const int64_t pairs = static_cast<int64_t>(num_seqs) * (num_q_heads / g);
    // The cascade decode's shared-prefix partials and private states, for a
    // prefix of up to the whole table width.
    shared = std::max(shared, shared_plan(std::max(num_seqs, 1), num_q_heads / g, g, head_dim,
                                          max_blocks_per_seq, ds->num_sms).bytes);
    // The bf16 and INT8 decodes (their grids may differ) share the workspace.
    for (const bool int8 : {false, true}) {
      const int ctas =
          pkv::decode_num_ctas(head_dim, g, ds->num_sms, pairs, g_max_splits.load(), int8);
      part = std::max(part, pkv::decode_partial_bytes(ctas, g, head_dim));
    }
    cnt = std::max(cnt, pkv::decode_counter_bytes(pairs));
  }
  const pkv_status st2 = ensure_workspace(ds, part, cnt);
  if (st2 != PKV_OK) return st2;
  return ensure_shared_workspace(ds, shared);
}

pkv_status pkv_set_wait_limit_ns(int64_t limit_ns) {
  if (limit_ns < 0) return PKV_ERR_INVALID_ARG;
  g_wait_limit_ns.store(limit_ns);
  return PKV_OK;
}

pkv_status pkv_profiler_enable(int32_t enable) {
  g_prof_on.store(enable ? 1 : 0);
  return PKV_OK;
}

pkv_status pkv_profiler_reset(void) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (auto& r : g_prof) {
    g_event_pool.push_back(r.start);
    g_event_pool.push_back(r.stop);
  }
  g_prof.clear();
  return PKV_OK;
}

pkv_status pkv_profiler_read(const char* name, double* total_ms, int64_t* launches) {
  if (!name || !total_ms || !launches) return PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  double sum = 0.0;
  int64_t n = 0;
  for (auto& r : g_prof) {
    if (std::strcmp(r.name, name) != 0) continue;
    if (cudaEventSynchronize(r.stop) != cudaSuccess) return PKV_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess) return PKV_ERR_CUDA;
    sum += ms;
    ++n;
  }
  *total_ms = sum;
  *launches = n;
  return PKV_OK;
}

}  // extern "C"
