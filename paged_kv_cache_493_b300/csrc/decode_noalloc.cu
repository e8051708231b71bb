// decode_noalloc.cu -- pkv_decode_attention_noalloc: the paged decode call
// with its split-K scratch in a fixed device array that the library defines
// at file scope, so that the call itself allocates nothing.
//
// Who needs it: callers that cannot let a library call cudaMalloc.
//  - Serving engines that give (nearly) all free device memory to the KV
//    block pool at start-up: a workspace allocated later by the library can
//    fail for lack of memory, or sit outside the engine's own accounting.
//  - Processes whose device memory must all go through one caching
//    allocator, so that a library's private cudaMalloc would break its
//    bookkeeping (or the allocator has already reserved the memory).
// pkv_decode_attention grows a cudaMalloc'ed workspace on first need; this
// entry point uses the static array below instead, and the caller still
// passes every input and output.
//
// The array is part of the library image: every device that loads libpkv
// holds its kScratchBytes until the process exits.  Host code cannot use the
// array's name as a device address (on the host it names a stand-in), so
// the first call on each device, with that device current, asks the runtime
// for the device address with cudaGetSymbolAddress and keeps it.  That
// first call should therefore come before any stream capture.
#include <mutex>

#include "pkv.h"
#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "pkv_pair_gap.h"

namespace {

// Layout of the per-device scratch: the decode kernel's counters in a fixed
// region of their own (zero at load, never reset, never overlapped by other
// data whatever the batch shape): a 256-byte header with the launch epoch,
// then 8 bytes per (sequence, KV head) pair; then two partial slots per
// decode block of G * (head_dim + 2) fp32 values.  Device-side check
// failures and wait timeouts go to the library's error word (also a static
// device variable), which pkv_get_device_error reads and clears.
constexpr size_t kScratchBytes = size_t{16} << 20;
constexpr size_t kCounterBytes = (size_t{2} << 20) + 256;  // 262144 (sequence, KV head) pairs
constexpr size_t kPartialBytes = kScratchBytes - kCounterBytes;

static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;

struct NoAllocDevice {
  bool ready = false;
  bool usable = false;
  int num_sms = 0;
  unsigned char* scratch = nullptr;  // device address of g_decode_scratch
  pkv::DeviceError* err = nullptr;   // device address of the library's error word
};

std::mutex g_mu;
NoAllocDevice g_dev[kMaxDevices];

// Once per device, with that device current: check the architecture, find
// the tensor-map encoder and look up the device addresses of the scratch and
// of the error word.  A device that is not sm_103a is marked unusable for
// good; a failed lookup is retried by the next call, so one refused first
// call does not disable the entry point.  Must be called with g_mu held.
NoAllocDevice* device_setup(pkv_status* st) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    *st = PKV_ERR_CUDA;
    return nullptr;
  }
  NoAllocDevice& d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0;
    const bool attrs =
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess;
    void* ptr = nullptr;
    if (attrs && !(major == 10 && minor == 3)) {
      d.ready = true;  // not an sm_103a device: never usable
      d.usable = false;
    } else if (attrs && pkv::load_tensor_map_encoder() &&
               cudaGetSymbolAddress(&ptr, g_decode_scratch) == cudaSuccess && ptr != nullptr) {
      pkv::DeviceError* err = pkv::device_error_word();
      if (err != nullptr) {
        d.scratch = static_cast<unsigned char*>(ptr);
        d.err = err;
        d.num_sms = sms;
        d.ready = true;
        d.usable = true;
      }
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

}  // namespace

extern "C" pkv_status pkv_decode_attention_noalloc(
    const void* q, int64_t q_row_stride, const void* k_cache, const void* v_cache,
    int64_t num_blocks, const int32_t* block_tables, int32_t max_blocks_per_seq,
    const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_dim, float scale, void* out, pkv_stream_t stream) {
  pkv_status st = pkv::validate_attention_args(q, q_row_stride, k_cache, v_cache, num_blocks,
                                               block_tables, max_blocks_per_seq, context_lens,
                                               num_seqs, num_q_heads, num_kv_heads, head_dim, out);
  if (st != PKV_OK) return st;
  int num_sms = 0;
  unsigned char* scratch = nullptr;
  pkv::DeviceError* err = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    NoAllocDevice* d = device_setup(&st);
    if (!d) return st;
    num_sms = d->num_sms;
    scratch = d->scratch;
    err = d->err;
  }
  if (num_seqs == 0) return PKV_OK;

  pkv::DecodeArgs a{};
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
  a.wait_limit_ns = pkv::wait_limit_ns();
  a.err = err;
  const int g = num_q_heads / num_kv_heads;
  const int64_t pairs = static_cast<int64_t>(num_seqs) * num_kv_heads;
  a.num_ctas = pkv::decode_num_ctas(head_dim, g, num_sms, pairs, pkv::max_splits_setting());
  a.pair_gap = pkv::kPairGapDecode;
  if (pkv::decode_counter_bytes(pairs) > kCounterBytes ||
      pkv::decode_partial_bytes(a.num_ctas, g, head_dim) > kPartialBytes)
    return PKV_ERR_UNSUPPORTED;
  a.counters = reinterpret_cast<unsigned long long*>(scratch);
  a.part_o = reinterpret_cast<float*>(scratch + kCounterBytes);
  a.part_ml = a.part_o + static_cast<size_t>(a.num_ctas) * 2 * g * head_dim;

  pkv::CacheMaps maps;
  if (!pkv::encode_cache_maps(&maps, k_cache, v_cache, num_blocks, num_kv_heads, head_dim))
    return PKV_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return pkv::launch_decode(a, maps, s) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
