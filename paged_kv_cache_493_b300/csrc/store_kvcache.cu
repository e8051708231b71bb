// store_kvcache.cu -- scatter of new K/V rows into paged cache slots.
//
// Row i of k and v (num_kv_heads * head_dim bf16) is copied, bit for bit,
// into cache slot slot_mapping[i]; slot -1 skips the row (tuning guide
// "Nano-vLLM性能调优实战", §2.2: the store_kvcache kernel writes the cache).
//
// Pure data movement: each thread moves 16-byte vectors, several in flight
// (all loads issued before any store), rows of K and V handled by the same
// thread so that one slot lookup serves both.  The source loads do not wait
// for the slot lookup (a source row is always in bounds), so the two
// latencies overlap.  Source rows are streamed (no L1 allocation);
// destination writes go to L2 normally because the attention kernel that
// follows reads them.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

constexpr int kStoreVecPerThread = 2;  // 16-byte vectors per tensor per thread
constexpr int kStoreThreads = 256;

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__global__ void __launch_bounds__(kStoreThreads)
store_kvcache_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                     int64_t k_row_vecs, int64_t v_row_vecs,  // row strides in 16-byte units
                     const int32_t* __restrict__ slot_mapping, int64_t num_tokens,
                     uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                     int64_t num_slots, int row_vecs, DeviceError* err) {
  grid_dependency_wait();
  const int64_t total = num_tokens * row_vecs;
  const int64_t base = (static_cast<int64_t>(blockIdx.x) * kStoreThreads * kStoreVecPerThread) +
                       threadIdx.x;
  uint4 kv[kStoreVecPerThread], vv[kStoreVecPerThread];
  int64_t dst[kStoreVecPerThread];
#pragma unroll
  for (int j = 0; j < kStoreVecPerThread; ++j) {
    const int64_t idx = base + static_cast<int64_t>(j) * kStoreThreads;
    dst[j] = -1;
    if (idx < total) {
      const int64_t row = idx / row_vecs;
      const int col = static_cast<int>(idx - row * row_vecs);
      const int64_t slot = slot_mapping[row];
      kv[j] = ld_stream(k + row * k_row_vecs + col);
      vv[j] = ld_stream(v + row * v_row_vecs + col);
      if (slot >= 0 && slot < num_slots) {
        dst[j] = slot * row_vecs + col;
      } else if (slot != -1 && col == 0) {
        report_error(err, kErrDeviceCheck, kSiteStoreSlot);
      }
    }
  }
  grid_dependents_launch();
#pragma unroll
  for (int j = 0; j < kStoreVecPerThread; ++j) {
    if (dst[j] >= 0) {
      k_cache[dst[j]] = kv[j];
      v_cache[dst[j]] = vv[j];
    }
  }
}

cudaError_t launch_store_kvcache(const StoreArgs& a, cudaStream_t stream) {
  const int row_vecs = a.num_kv_heads * a.head_dim * 2 / 16;
  const int64_t total = a.num_tokens * row_vecs;
  if (total == 0) return cudaSuccess;
  const int64_t per_block = static_cast<int64_t>(kStoreThreads) * kStoreVecPerThread;
  const int64_t blocks = (total + per_block - 1) / per_block;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kStoreThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, store_kvcache_kernel, static_cast<const uint4*>(a.k),
                            static_cast<const uint4*>(a.v), a.k_row_stride * 2 / 16,
                            a.v_row_stride * 2 / 16, a.slot_mapping, a.num_tokens,
                            static_cast<uint4*>(a.k_cache), static_cast<uint4*>(a.v_cache),
                            a.num_blocks * kBlockSize, row_vecs, a.err);
}

}  // namespace pkv
