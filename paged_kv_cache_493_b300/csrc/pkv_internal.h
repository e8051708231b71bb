// pkv_internal.h -- host-side launch interface between the C ABI layer
// (pkv_api.cu) and the kernel files.  Arguments here are already validated.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

struct DeviceError;

struct StoreArgs {
  const void* k;
  const void* v;
  int64_t k_row_stride;  // elements
  int64_t v_row_stride;  // elements
  const int32_t* slot_mapping;
  int64_t num_tokens;
  void* k_cache;
  void* v_cache;
  int64_t num_blocks;
  int num_kv_heads;
  int head_dim;
  DeviceError* err;
};

struct DecodeArgs {
  const void* q;
  int64_t q_row_stride;  // elements
  const int32_t* block_tables;
  int max_blocks;
  const int32_t* context_lens;
  int num_seqs;
  int num_q_heads;
  int num_kv_heads;
  int head_dim;
  int64_t num_blocks;
  float scale;
  void* out;
  // split-K plan
  int split_tokens;  // tokens per split (multiple of the chunk size)
  int max_splits;    // splits of the longest possible sequence
  float* part_o;     // [num_seqs][num_q_heads][max_splits][head_dim]
  float* part_ml;    // [num_seqs][num_q_heads][max_splits][2]
  uint64_t wait_limit_ns;
  DeviceError* err;
};

struct PrefillArgs {
  const void* q;
  int64_t q_row_stride;  // elements
  const int32_t* block_tables;
  int max_blocks;
  const int32_t* cu_seqlens_q;
  const int32_t* context_lens;
  int num_seqs;
  int64_t total_q;
  int num_q_heads;
  int num_kv_heads;
  int head_dim;
  int64_t num_blocks;
  float scale;
  void* out;
  uint64_t wait_limit_ns;
  DeviceError* err;
};

// Tensor maps built by the API layer (cached per cache pointer).
struct CacheMaps {
  CUtensorMap k_rows;   // decode: box {head_dim, 1, 32} over [slots][Hkv][D]
  CUtensorMap v_rows;
  CUtensorMap k_sw128;  // prefill: box {64, 1, 128}, 128-byte swizzle
  CUtensorMap v_sw128;
};

// Decode chunk geometry (tokens per TMA transfer).
constexpr int kDecodeChunk = 32;

cudaError_t launch_store_kvcache(const StoreArgs& a, cudaStream_t stream);

// Launches the split kernel and the combine kernel (profiled separately
// through the callbacks in the API layer).
cudaError_t launch_decode_split(const DecodeArgs& a, const CacheMaps& maps, cudaStream_t stream);
cudaError_t launch_decode_combine(const DecodeArgs& a, cudaStream_t stream);

cudaError_t launch_prefill(const PrefillArgs& a, const CacheMaps& maps, const CUtensorMap& qmap,
                           int num_sms, cudaStream_t stream);

// Helpers shared by the C entry points (defined in pkv_api.cu).
// Split-K plan of a decode batch: tokens per context range and the number of
// ranges of the longest possible sequence (max_blocks * 256 tokens).
void plan_decode_splits(int num_seqs, int num_kv_heads, int max_blocks, int num_sms,
                        int* split_tokens, int* max_splits);
// Host-side shape, pointer and alignment checks of the attention calls.
pkv_status validate_attention_args(const void* q, int64_t q_row_stride, const void* k_cache,
                                   const void* v_cache, int64_t num_blocks,
                                   const int32_t* block_tables, int32_t max_blocks,
                                   const int32_t* lens, int32_t num_seqs, int32_t hq, int32_t hkv,
                                   int32_t d, const void* out);
// Resolves cuTensorMapEncodeTiled from the driver (once); false if unavailable.
bool load_tensor_map_encoder();
// Encodes the decode and prefill tensor maps of a cache (host only, no allocation).
bool encode_cache_maps(CacheMaps* maps, const void* k, const void* v, int64_t num_blocks,
                       int num_kv_heads, int head_dim);
// Current bound on every in-kernel wait (pkv_set_wait_limit_ns).
uint64_t wait_limit_ns();

// Tensor-map encoder obtained from the driver at first use.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

}  // namespace pkv
