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
  // Stream-K plan: the (sequence, KV head) pairs' 32-token chunks, laid end
  // to end, are cut into num_ctas equal slices, one per block.  A pair cut
  // by a slice boundary leaves one partial state per piece; the block that
  // writes the pair's last piece merges them.
  int num_ctas;      // blocks of the decode kernel
  // The stream is cut into num_ctas equal slices of cost: a pair of nch
  // chunks costs pair_gap + nch units, the pair_gap units before its first
  // chunk holding nothing.  pair_gap > 0 charges each piece boundary as
  // pair_gap chunks, so a block that crosses many short pairs gets fewer
  // chunks; 0 cuts the chunks evenly.
  int pair_gap;
  // Counter region (zero when first used, never reset): a 256-byte header
  // (word 0: launch epoch; word 1: blocks finished in this launch) and then
  // one arrival counter per (sequence, KV head) pair, [num_seqs *
  // num_kv_heads].  Every counter is tagged with the launch generation
  // (epoch + 1, read by each block at its start; the last block to finish
  // advances the epoch), so values left by earlier launches, even aborted
  // ones or replays of the same captured graph, count as zero.
  unsigned long long* counters;
  float* part_o;     // [num_ctas][2][G][head_dim]
  float* part_ml;    // [num_ctas][2][G][2] (running max, sum)
  uint64_t wait_limit_ns;
  DeviceError* err;
  // Cascade decode: the first shared_len tokens of every sequence (whole
  // blocks, the same physical blocks as in table row 0) were attended by the
  // shared-prefix kernel, which left shared_units partial states per row
  // (layout of PrefillArgs::shared_o / shared_ml).  This kernel streams
  // tokens [shared_len, context_lens[s]) only, checks that the sequence's
  // leading table entries are row 0's, and folds the partials into each
  // output.  shared_len = 0: plain decode.
  int shared_len;
  int shared_units;
  int shared_rows_pad;
  const float* shared_o;
  const float* shared_ml;
  // Cascade decode: private states (unnormalised output; running max, sum)
  // of pairs streamed whole, set aside while the shared-prefix kernel may
  // still run and folded once the block's stream is done.  Rows as in
  // shared_o / shared_ml with one unit: kvh * shared_rows_pad + seq * G + h.
  float* private_o;
  float* private_ml;
  // Fused store (pkv_decode_attention_append; slot_mapping == nullptr: off):
  // row s of k_new / v_new is sequence s's new token, the one at position
  // context_lens[s] - 1.  The block that streams that position's chunk of
  // pair (s, h) writes head h of the row into the cache at slot_mapping[s]
  // and uses it in place of the pool row it loaded.  A slot of -1 stores
  // nothing; any other slot than the position's is rejected (reported, not
  // stored).
  const void* k_new;
  const void* v_new;
  int64_t k_new_stride;  // elements
  int64_t v_new_stride;
  const int32_t* slot_mapping;
  void* k_cache;
  void* v_cache;
  // INT8 cache (launch_decode_i8): the fp32 scales [slots][Hkv] of the codes
  // the tensor maps cover.
  const float* k_scales;
  const float* v_scales;
};

// Most partial states per row the decode's fold of a shared prefix accepts
// (DecodeArgs::shared_units; the cascade's shared-prefix kernel merges its
// units in the cluster and leaves one).
constexpr int kMaxSharedUnits = 32;

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
  // Shared-prefix role of the cascade decode (launch_shared_prefix only):
  // the decode queries of all num_seqs sequences attend the first
  // shared_tiles * 64 tokens reached through table row 0, cut into
  // shared_units key ranges, one CTA each; the units of a (row tile, KV head)
  // form a cluster and merge their states, and row (s * G + g) of KV head h
  // leaves the merged state at index h * shared_rows_pad + row of shared_o
  // ([..][head_dim] fp32, unnormalised) and shared_ml ([..][2]: the
  // reference max in the log2 domain and the sum; sum -1 marks a failed row).
  int shared_tiles;
  int shared_units;
  int shared_rows_pad;  // row tiles * 128
  float* shared_o;
  float* shared_ml;
  // INT8 cache (launch_prefill_i8 only): scales [num_blocks][Hkv][256].
  const float* k_scales;
  const float* v_scales;
};

// INT8 KV cache: codes int8 [num_blocks][Hkv][256][D], scales float32
// [num_blocks][Hkv][256] (each block holds its KV heads one after another);
// a code stands for code * scale.
struct StoreI8Args {
  const void* k;
  const void* v;
  int64_t k_row_stride;  // elements
  int64_t v_row_stride;  // elements
  const int32_t* slot_mapping;
  int64_t num_tokens;
  int8_t* k_codes;
  int8_t* v_codes;
  float* k_scales;
  float* v_scales;
  int64_t num_blocks;
  int num_kv_heads;
  int head_dim;
  DeviceError* err;
};

// Tensor maps built by the API layer (cached per cache pointer).
struct CacheMaps {
  CUtensorMap k_rows;   // decode: box {64, 1, 32} over [slots][Hkv][D], 128-byte swizzle
  CUtensorMap v_rows;
  CUtensorMap k_sw128;  // prefill: box {64, 1, kPrefillKeyTile}, 128-byte swizzle
  CUtensorMap v_sw128;
};

// Decode chunk geometry (tokens per TMA transfer).
constexpr int kDecodeChunk = 32;
// Prefill key tile (keys per TMA transfer and per S tile).
constexpr int kPrefillKeyTile = 64;

cudaError_t launch_store_kvcache(const StoreArgs& a, cudaStream_t stream);
cudaError_t launch_store_kvcache_int8(const StoreI8Args& a, cudaStream_t stream);

// Blocks of the decode kernel for a batch: as many as fit on the GPU at
// once, at most num_pairs * max_splits when max_splits > 0.
int decode_num_ctas(int head_dim, int group, int num_sms, int64_t num_pairs, int max_splits,
                    bool int8 = false);
// Bytes of the decode kernel's arrival counters (zero when first used) and of
// its partial slots.
size_t decode_counter_bytes(int64_t num_pairs);
size_t decode_partial_bytes(int num_ctas, int group, int head_dim);
cudaError_t launch_decode(const DecodeArgs& a, const CacheMaps& maps, cudaStream_t stream);
// The same split-K decode over an INT8 cache, in chunks of 64 tokens: kmap /
// vmap view the codes as uint8 {D, 256, num_blocks * Hkv} with box {D, 64, 1}
// (128-byte swizzle for D = 128, 64-byte for D = 64); a.k_scales /
// a.v_scales are set.
cudaError_t launch_decode_i8(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                             cudaStream_t stream);

cudaError_t launch_prefill(const PrefillArgs& a, const CacheMaps& maps, const CUtensorMap& qmap,
                           int num_sms, cudaStream_t stream);
// The same prefill over an INT8 cache: kmap / vmap view the codes as uint8
// {D, 256, num_blocks * Hkv} with box {D, 64, 1}, no swizzle; a.k_scales /
// a.v_scales are set.
cudaError_t launch_prefill_i8(const PrefillArgs& a, const CUtensorMap& kmap,
                              const CUtensorMap& vmap, const CUtensorMap& qmap,
                              cudaStream_t stream);
// The shared-prefix kernel of the cascade decode (qmap: the decode queries
// viewed as {D, Hq, num_seqs} with the prefill's box).
cudaError_t launch_shared_prefix(const PrefillArgs& a, const CacheMaps& maps,
                                 const CUtensorMap& qmap, cudaStream_t stream);

// Helpers shared by the C entry points (defined in pkv_api.cu).
// Process-wide cap on the number of pieces a pair is cut into
// (pkv_set_max_splits; 0 = no cap).
int max_splits_setting();
// Host-side shape, pointer and alignment checks of the attention calls.
pkv_status validate_attention_args(const void* q, int64_t q_row_stride, const void* k_cache,
                                   const void* v_cache, int64_t num_blocks,
                                   const int32_t* block_tables, int32_t max_blocks,
                                   const int32_t* lens, int32_t num_seqs, int32_t hq, int32_t hkv,
                                   int32_t d, const void* out);
// Resolves cuTensorMapEncodeTiled from the driver (once); false if unavailable.
bool load_tensor_map_encoder();
// Device address of the current device's error word (a file-scope __device__
// variable, looked up once per device; no allocation), or nullptr when the
// device is unusable.  pkv_get_device_error reads and clears it.
DeviceError* device_error_word();
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
