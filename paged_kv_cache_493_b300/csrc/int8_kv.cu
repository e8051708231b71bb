// int8_kv.cu -- the quantising store of the INT8 variant of the KV cache
// (half the bytes of bf16); the INT8 decode is the split-K decode kernel of
// decode_attention.cu reading codes.
//
// Format (intelliparadigm.com Nano-vLLM article §2.2, "kv_cache_dtype: int8";
// ocdem.com nano-vllm article §4.1 KV Cache 量化; the pages give no formula):
// every (token, KV head) row of head_dim values is held as int8 codes plus
// one binary32 scale, symmetric absmax:
//   scale = max_d |x_d| / 127,  code_d = nearest(x_d / scale), ties to even,
// both computed with IEEE binary32 division, codes in [-127, 127]; an
// all-zero row has scale 0.  A code stands for code * scale.
//   codes  int8    [num_blocks][num_kv_heads][256][head_dim]
//   scales float32 [num_blocks][num_kv_heads][256]
// (each block holds its KV heads one after another, so a run of one head's
// tokens is contiguous: the decode reads 32 of them as one 4 KB tile).
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int kStoreWarps = 8;

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

// Quantises one row held by a warp (DPL values per lane, lane-major) and
// stores its codes and scale.
template <int DPL>
__device__ __forceinline__ void quantise_row(const float (&x)[DPL], int lane, int8_t* codes,
                                             float* scale) {
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < DPL; ++e) amax = fmaxf(amax, fabsf(x[e]));
  amax = warp_max(amax);
  const float s = __fdiv_rn(amax, 127.f);
  uint32_t packed = 0;
#pragma unroll
  for (int e = 0; e < DPL; ++e) {
    int c = s > 0.f ? __float2int_rn(__fdiv_rn(x[e], s)) : 0;
    c = min(max(c, -127), 127);
    packed |= (static_cast<uint32_t>(c) & 0xFFu) << (8 * e);
  }
  if constexpr (DPL == 4)
    *reinterpret_cast<uint32_t*>(codes + lane * 4) = packed;
  else
    *reinterpret_cast<uint16_t*>(codes + lane * 2) = static_cast<uint16_t>(packed);
  if (lane == 0) *scale = s;
}

template <int D>
__global__ void __launch_bounds__(kStoreWarps * 32) store_kvcache_int8_kernel(StoreI8Args a) {
  constexpr int DPL = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kStoreWarps + (threadIdx.x >> 5);
  if (row >= a.num_tokens * a.num_kv_heads) return;
  const int64_t i = row / a.num_kv_heads;
  const int h = static_cast<int>(row % a.num_kv_heads);
  const int64_t slot = a.slot_mapping[i];
  if (slot == -1) return;
  if (slot < 0 || slot >= a.num_blocks * kBlockSize) {
    if (lane == 0) report_error(a.err, kErrDeviceCheck, kSiteStoreI8Slot);
    return;
  }
  // Head-major blocks: row (block * Hkv + h) * 256 + offset.
  const int64_t dst =
      ((slot / kBlockSize) * a.num_kv_heads + h) * kBlockSize + (slot % kBlockSize);
#pragma unroll
  for (int which = 0; which < 2; ++which) {
    const __nv_bfloat16* src =
        static_cast<const __nv_bfloat16*>(which == 0 ? a.k : a.v) +
        i * (which == 0 ? a.k_row_stride : a.v_row_stride) + static_cast<int64_t>(h) * D +
        lane * DPL;
    float x[DPL];
    if constexpr (DPL == 4) {
      const uint2 raw = *reinterpret_cast<const uint2*>(src);
      x[0] = bf16_lo(raw.x);
      x[1] = bf16_hi(raw.x);
      x[2] = bf16_lo(raw.y);
      x[3] = bf16_hi(raw.y);
    } else {
      const uint32_t raw = *reinterpret_cast<const uint32_t*>(src);
      x[0] = bf16_lo(raw);
      x[DPL - 1] = bf16_hi(raw);
    }
    quantise_row<DPL>(x, lane, (which == 0 ? a.k_codes : a.v_codes) + dst * D,
                      (which == 0 ? a.k_scales : a.v_scales) + dst);
  }
}

}  // namespace

cudaError_t launch_store_kvcache_int8(const StoreI8Args& a, cudaStream_t stream) {
  const int64_t rows = a.num_tokens * a.num_kv_heads;
  if (rows <= 0) return cudaSuccess;
  const int64_t blocks = (rows + kStoreWarps - 1) / kStoreWarps;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  if (a.head_dim == 128)
    store_kvcache_int8_kernel<128><<<static_cast<unsigned>(blocks), kStoreWarps * 32, 0, stream>>>(a);
  else if (a.head_dim == 64)
    store_kvcache_int8_kernel<64><<<static_cast<unsigned>(blocks), kStoreWarps * 32, 0, stream>>>(a);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace pkv
