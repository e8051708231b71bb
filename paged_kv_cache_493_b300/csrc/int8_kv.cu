// int8_kv.cu -- the INT8 variant of the KV cache: a store that quantises new
// K/V rows, and a decode that reads int8 codes (half the bytes of bf16).
//
// Format (intelliparadigm.com Nano-vLLM article §2.2, "kv_cache_dtype: int8";
// ocdem.com nano-vllm article §4.1 KV Cache 量化; the pages give no formula):
// every (token, KV head) row of head_dim values is held as int8 codes plus
// one binary32 scale, symmetric absmax:
//   scale = max_d |x_d| / 127,  code_d = nearest(x_d / scale), ties to even,
// both computed with IEEE binary32 division, codes in [-127, 127]; an
// all-zero row has scale 0.  A code stands for code * scale.
//   codes  int8    [num_blocks][256][num_kv_heads][head_dim]
//   scales float32 [num_blocks][256][num_kv_heads]
//
// Decode is a split-K kernel followed by a log-sum-exp combine kernel.  A
// block of 4 warps takes one (sequence, KV head, split of 512 tokens) and all
// G query heads of the KV head, so each code row is read once for the group.
// In a chunk of 32 tokens lane i scores token i (its 16-byte code loads
// against the pre-scaled query in shared memory), the warp updates its
// running max and sum per head, and for P V the lanes own head_dim / 32
// dimensions each while the tokens' probabilities are broadcast by shuffle.
// The 4 warps merge in shared memory and the block writes one partial state
// per query head; the combine kernel merges a pair's splits and writes bf16.
// No block waits for another.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int kI8Warps = 4;
constexpr int kI8Threads = kI8Warps * 32;
constexpr int kStoreWarps = 8;

// Sign-extended byte e of a 32-bit word of codes, as float.
__device__ __forceinline__ float code_at(int w, int e) {
  return static_cast<float>(static_cast<int8_t>(static_cast<uint32_t>(w) >> (8 * e)));
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
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
  const int64_t dst = slot * a.num_kv_heads + h;
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

template <int D, int G>
__global__ void __launch_bounds__(kI8Threads, G >= 8 ? 2 : 4) decode_int8_split_kernel(DecodeI8Args a) {
  constexpr int DPL = D / 32;  // dimensions per lane in P V
  __shared__ float qs[G][D];   // query, times scale * log2(e)
  __shared__ float wm[kI8Warps][G], wl[kI8Warps][G];
  __shared__ float wo[kI8Warps][G][D];
  __shared__ int wbad[kI8Warps];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t item = blockIdx.x;
  const int sp = static_cast<int>(item % a.splits);
  const int64_t pair = item / a.splits;
  const int s = static_cast<int>(pair / a.num_kv_heads);
  const int kvh = static_cast<int>(pair % a.num_kv_heads);
  const int64_t hkv = a.num_kv_heads;
  float* part = a.part + item * (G * (D + 2));  // o [G][D], then (m, l) [G][2]

  const int ctx = a.context_lens[s];
  const bool bad_ctx = ctx < 0 || ctx > a.max_blocks * kBlockSize;
  if (bad_ctx && sp == 0 && threadIdx.x == 0)
    report_error(a.err, kErrDeviceCheck, kSiteDecodeI8Context);
  const int t0 = sp * kInt8SplitTokens;
  const int t1 = bad_ctx ? t0 : min(ctx, t0 + kInt8SplitTokens);

  const float sl2 = a.scale * 1.4426950408889634f;
  const __nv_bfloat16* qp = static_cast<const __nv_bfloat16*>(a.q) +
                            static_cast<int64_t>(s) * a.q_row_stride +
                            static_cast<int64_t>(kvh) * G * D;
  for (int i = threadIdx.x; i < G * D; i += kI8Threads)
    qs[i / D][i % D] = __bfloat162float(qp[i]) * sl2;
  __syncthreads();

  float m[G], l[G], acc[G][DPL];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int e = 0; e < DPL; ++e) acc[g][e] = 0.f;
  }
  bool bad = false;
  const int32_t* table = a.block_tables + static_cast<int64_t>(s) * a.max_blocks;

  for (int c0 = t0 + warp * 32; c0 < t1; c0 += kI8Warps * 32) {
    const int t = c0 + lane;
    int slot = -1;
    if (t < t1) {
      const int blk = table[t >> 8];
      if (blk >= 0 && blk < a.num_blocks)
        slot = blk * kBlockSize + (t & (kBlockSize - 1));
      else
        bad = true;
    }
    // Scores of this lane's token (log2 domain); its V scale, for P V.
    float sc[G];
    float vs_mine = 0.f;
    if (slot >= 0) {
      const int8_t* krow = a.k_codes + (static_cast<int64_t>(slot) * hkv + kvh) * D;
      const float ks = a.k_scales[static_cast<int64_t>(slot) * hkv + kvh];
      vs_mine = a.v_scales[static_cast<int64_t>(slot) * hkv + kvh];
      float dot[G];
#pragma unroll
      for (int g = 0; g < G; ++g) dot[g] = 0.f;
      constexpr int kKUnroll = (G <= 4 && D == 128) ? 4 : 2;  // 16-byte loads in flight per lane
#pragma unroll kKUnroll
      for (int d0 = 0; d0 < D; d0 += 16) {
        const int4 raw = *reinterpret_cast<const int4*>(krow + d0);
        const int w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float kf = code_at(w[e >> 2], e & 3);
#pragma unroll
          for (int g = 0; g < G; ++g) dot[g] = fmaf(qs[g][d0 + e], kf, dot[g]);
        }
      }
#pragma unroll
      for (int g = 0; g < G; ++g) sc[g] = dot[g] * ks;
    } else {
#pragma unroll
      for (int g = 0; g < G; ++g) sc[g] = -INFINITY;
    }
    // Running max and sum per head.
    float p[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float m_new = fmaxf(m[g], warp_max(sc[g]));
      const float alpha = m_new == -INFINITY ? 1.f : fast_exp2(m[g] - m_new);
      p[g] = sc[g] == -INFINITY ? 0.f : fast_exp2(sc[g] - m_new);
      l[g] = l[g] * alpha + warp_sum(p[g]);
#pragma unroll
      for (int e = 0; e < DPL; ++e) acc[g][e] *= alpha;
      m[g] = m_new;
    }
    // O += P V: lane owns dimensions lane * DPL .. lane * DPL + DPL - 1.
    // Unrolled without branches so that several rows' loads are in flight;
    // a token outside the context has weight 0 and reads the row of slot 0.
#pragma unroll 8
    for (int j = 0; j < 32; ++j) {
      const int sj = __shfl_sync(0xffffffffu, slot, j);
      const float vs = __shfl_sync(0xffffffffu, vs_mine, j);
      const int64_t r = static_cast<int64_t>(sj < 0 ? 0 : sj) * hkv + kvh;
      const int8_t* vrow = a.v_codes + r * D + lane * DPL;
      float vf[DPL];
      if constexpr (DPL == 4) {
        const int w = *reinterpret_cast<const int*>(vrow);
#pragma unroll
        for (int e = 0; e < DPL; ++e) vf[e] = code_at(w, e);
      } else {
        const int w = *reinterpret_cast<const uint16_t*>(vrow);
        vf[0] = code_at(w, 0);
        vf[DPL - 1] = code_at(w, 1);
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float pj = __shfl_sync(0xffffffffu, p[g], j) * vs;
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[g][e] = fmaf(pj, vf[e], acc[g][e]);
      }
    }
  }

  // Merge the warps (log-sum-exp) and write this split's state.
  bad = __any_sync(0xffffffffu, bad);
  if (bad && lane == 0) report_error(a.err, kErrDeviceCheck, kSiteDecodeI8Block);
#pragma unroll
  for (int g = 0; g < G; ++g) {
    if (lane == 0) {
      wm[warp][g] = m[g];
      wl[warp][g] = l[g];
    }
#pragma unroll
    for (int e = 0; e < DPL; ++e) wo[warp][g][lane * DPL + e] = acc[g][e];
  }
  if (lane == 0) wbad[warp] = bad ? 1 : 0;
  __syncthreads();
  for (int i = threadIdx.x; i < G * D; i += kI8Threads) {
    const int g = i / D, d = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kI8Warps; ++w) M = fmaxf(M, wm[w][g]);
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < kI8Warps; ++w)
      if (wm[w][g] != -INFINITY) o += wo[w][g][d] * fast_exp2(wm[w][g] - M);
    part[g * D + d] = o;
  }
  if (threadIdx.x < G) {
    const int g = threadIdx.x;
    float M = -INFINITY;
    for (int w = 0; w < kI8Warps; ++w) M = fmaxf(M, wm[w][g]);
    float L = 0.f;
    for (int w = 0; w < kI8Warps; ++w)
      if (wm[w][g] != -INFINITY) L += wl[w][g] * fast_exp2(wm[w][g] - M);
    const bool any_bad = bad_ctx || wbad[0] || wbad[1] || wbad[2] || wbad[3];
    part[G * D + 2 * g] = M;
    part[G * D + 2 * g + 1] = any_bad ? -1.f : L;  // -1 marks a discarded split
  }
}

template <int D, int G>
__global__ void __launch_bounds__(kI8Threads) decode_int8_combine_kernel(DecodeI8Args a) {
  constexpr int DPL = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t w = static_cast<int64_t>(blockIdx.x) * kI8Warps + (threadIdx.x >> 5);
  if (w >= static_cast<int64_t>(a.num_seqs) * a.num_q_heads) return;
  const int s = static_cast<int>(w / a.num_q_heads);
  const int h = static_cast<int>(w % a.num_q_heads);
  const int kvh = h / G, g = h % G;
  const int64_t stride = G * (D + 2);
  const float* base = a.part + (static_cast<int64_t>(s) * a.num_kv_heads + kvh) * a.splits * stride;
  float M = -INFINITY;
  bool bad = false;
  for (int sp = lane; sp < a.splits; sp += 32) {
    const float* pp = base + sp * stride + G * D + 2 * g;
    M = fmaxf(M, pp[0]);
    bad |= pp[1] < 0.f;
  }
  M = warp_max(M);
  bad = __any_sync(0xffffffffu, bad);
  float L = 0.f, o[DPL];
#pragma unroll
  for (int e = 0; e < DPL; ++e) o[e] = 0.f;
  if (!bad && M != -INFINITY) {
    for (int sp = 0; sp < a.splits; ++sp) {
      const float* pp = base + sp * stride;
      const float mm = pp[G * D + 2 * g];
      if (mm == -INFINITY) continue;
      const float wgt = fast_exp2(mm - M);
      L += wgt * pp[G * D + 2 * g + 1];
#pragma unroll
      for (int e = 0; e < DPL; ++e) o[e] = fmaf(wgt, pp[g * D + lane * DPL + e], o[e]);
    }
  }
  const float inv = (!bad && L > 0.f) ? 1.f / L : 0.f;
  __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) +
                       (static_cast<int64_t>(s) * a.num_q_heads + h) * D + lane * DPL;
  if constexpr (DPL == 4) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(o[0] * inv, o[1] * inv),
                                                pack_bf16x2(o[2] * inv, o[3] * inv));
  } else {
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(o[0] * inv, o[DPL - 1] * inv);
  }
}

template <int D, int G>
cudaError_t launch_decode_t(const DecodeI8Args& a, cudaStream_t stream) {
  const int64_t items = static_cast<int64_t>(a.num_seqs) * a.num_kv_heads * a.splits;
  if (items <= 0) return cudaSuccess;
  if (items > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  decode_int8_split_kernel<D, G><<<static_cast<unsigned>(items), kI8Threads, 0, stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t warps = static_cast<int64_t>(a.num_seqs) * a.num_q_heads;
  decode_int8_combine_kernel<D, G>
      <<<static_cast<unsigned>((warps + kI8Warps - 1) / kI8Warps), kI8Threads, 0, stream>>>(a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_decode_d(const DecodeI8Args& a, cudaStream_t stream) {
  switch (a.num_q_heads / a.num_kv_heads) {
    case 1: return launch_decode_t<D, 1>(a, stream);
    case 2: return launch_decode_t<D, 2>(a, stream);
    case 4: return launch_decode_t<D, 4>(a, stream);
    case 8: return launch_decode_t<D, 8>(a, stream);
    case 16: return launch_decode_t<D, 16>(a, stream);
    default: return cudaErrorInvalidValue;
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

int decode_int8_splits(int max_blocks) {
  const int64_t tokens = static_cast<int64_t>(max_blocks) * kBlockSize;
  return static_cast<int>((tokens + kInt8SplitTokens - 1) / kInt8SplitTokens);
}

size_t decode_int8_partial_bytes(int64_t num_seqs, int num_kv_heads, int splits, int group,
                                 int head_dim) {
  return sizeof(float) * static_cast<size_t>(num_seqs) * num_kv_heads * splits * group *
         (head_dim + 2);
}

cudaError_t launch_decode_int8(const DecodeI8Args& a, cudaStream_t stream) {
  if (a.head_dim == 128) return launch_decode_d<128>(a, stream);
  if (a.head_dim == 64) return launch_decode_d<64>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
