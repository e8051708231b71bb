// decode_attention.cu -- paged GQA decode attention, split-K over the
// context (flash decoding) plus a log-sum-exp combine.
//
// What is computed (intelliparadigm.com Nano-vLLM article §7.1 增量解码;
// tuning guide "Nano-vLLM性能调优实战" §2.2 flash_attn_with_kvcache over the
// paged cache; ocdem.com nano-vllm article §2.1 block tables): for sequence
// s and query head h with KV head g = h / G,
//   out[s][h] = sum_t softmax_t(scale * q[s][h] . K[s][t][g]) V[s][t][g],
// t over the context_lens[s] cached tokens, reached through the block table.
// The context is cut into ranges ("splits"; the pages' max_splits knob,
// intelliparadigm.com article §8) that run as separate blocks; each split
// keeps an fp32 online softmax (running max m, running sum l, unnormalised
// output o) and the combine kernel merges the splits:
//   M = max_j m_j,  L = sum_j l_j 2^(m_j - M),  out = sum_j o_j 2^(m_j - M) / L.
// Scores are kept in the log2 domain (q is pre-scaled by scale * log2 e).
//
// Block structure (one CTA = one sequence x one KV head x one split):
//   warp 4        producer: one lane walks the split in 32-token chunks,
//                 looks up the physical block, and issues two TMA tile loads
//                 (K and V rows of this KV head, 32 x head_dim bf16 each) into
//                 a 4-stage shared-memory ring, completing on mbarriers;
//   warps 0..3    consumers: each takes a group of tokens of every chunk.
//                 A lane owns head_dim/32 dimensions of the G query heads of
//                 the group, so each K/V row loaded once from shared memory
//                 serves all G query heads.  The G x T partial dot products of
//                 a group (T = 16/G tokens) are reduced across the warp with a
//                 butterfly in which every shuffle halves the values a lane
//                 still holds (16 shuffles for 16 dot products instead of 80);
//                 the slot order of the partials is permuted per lane so that
//                 no selects are needed.  After the reduction lane l holds the
//                 score of pair g(l) (twice: lanes l and l^1).
// The pipeline is HBM-bound: per token and KV head the kernel reads
// 2 * head_dim * 2 bytes of K/V and does 4 * G * head_dim flops.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int kStages = 4;
constexpr int kConsumerWarps = 4;
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;
constexpr int kPairs = 16;  // (token, head) dot products per warp step

template <int D, int G>
struct DecodeSmem {
  alignas(128) __nv_bfloat16 k[kStages][kDecodeChunk][D];
  alignas(128) __nv_bfloat16 v[kStages][kDecodeChunk][D];
  float merge_o[kConsumerWarps][G][D];
  float merge_m[kConsumerWarps][G];
  float merge_l[kConsumerWarps][G];
  alignas(8) uint64_t full[kStages];
  alignas(8) uint64_t empty[kStages];
  int abort_flag;
  int bad_split;
};

// After the butterfly, lanes 2j and 2j+1 hold the score of pair j: at the
// level that exchanges across lane bit b+1 the slots split on bit b.
__device__ __forceinline__ int lane_of_pair(int j) { return j << 1; }

template <int DPL>
__device__ __forceinline__ void load_row(const __nv_bfloat16* row, int lane, float (&x)[DPL]) {
  if constexpr (DPL == 4) {
    const uint2 u = *reinterpret_cast<const uint2*>(row + lane * 4);
    x[0] = bf16_lo(u.x);
    x[1] = bf16_hi(u.x);
    x[2] = bf16_lo(u.y);
    x[3] = bf16_hi(u.y);
  } else {
    const uint32_t u = *reinterpret_cast<const uint32_t*>(row + lane * 2);
    x[0] = bf16_lo(u);
    x[1] = bf16_hi(u);
  }
}

template <int D, int G>
__global__ void __launch_bounds__(kDecodeThreads)
decode_split_kernel(const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap, DecodeArgs a) {
  constexpr int DPL = D / 32;          // dimensions per lane
  constexpr int TW = kPairs / G;       // tokens per warp step
  constexpr int LG = (G == 1) ? 0 : (G == 2) ? 1 : (G == 4) ? 2 : (G == 8) ? 3 : 4;
  constexpr int GROUPS = kDecodeChunk / TW;  // warp steps per chunk
  constexpr uint32_t kChunkBytes = kDecodeChunk * D * 2;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  DecodeSmem<D, G>& sm = *reinterpret_cast<DecodeSmem<D, G>*>(smem_raw);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // blockIdx.x = (split * num_seqs + seq) * num_kv_heads + kv_head
  const int kvh = blockIdx.x % a.num_kv_heads;
  const int rest = blockIdx.x / a.num_kv_heads;
  const int seq = rest % a.num_seqs;
  const int split = rest / a.num_seqs;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), kConsumerWarps);
    }
    sm.abort_flag = 0;
    sm.bad_split = 0;
    fence_barrier_init();
  }
  if (warp == kConsumerWarps && lane == 0) {
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
  }
  grid_dependency_wait();
  grid_dependents_launch();

  const int ctx = a.context_lens[seq];
  const int s0 = split * a.split_tokens;
  const int max_ctx = a.max_blocks * kBlockSize;
  if (ctx < 0 || ctx > max_ctx) {
    if (threadIdx.x == 0 && split == 0) report_error(a.err, kErrDeviceCheck, kSiteDecodeContext);
  }
  const int ctx_ok = (ctx >= 0 && ctx <= max_ctx) ? ctx : 0;
  const int n_splits = (ctx_ok + a.split_tokens - 1) / a.split_tokens;
  if (split >= n_splits && !(split == 0 && n_splits == 0)) return;  // nothing for this block
  const int s1 = min(s0 + a.split_tokens, ctx_ok);
  const int n_tok = max(s1 - s0, 0);
  const int n_chunks = (n_tok + kDecodeChunk - 1) / kDecodeChunk;
  const int32_t* table = a.block_tables + static_cast<int64_t>(seq) * a.max_blocks;

  // Validate the physical blocks of this split before touching memory.
  if (threadIdx.x < 32) {
    const int b0 = s0 / kBlockSize;
    const int b1 = (s1 + kBlockSize - 1) / kBlockSize;
    bool bad = false;
    for (int b = b0 + lane; b < b1; b += 32) {
      const int id = table[b];
      bad |= (id < 0 || id >= a.num_blocks);
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) {
      sm.bad_split = 1;
      report_error(a.err, kErrDeviceCheck, kSiteDecodeBlock);
    }
  }
  __syncthreads();
  const bool bad_split = sm.bad_split != 0 || (ctx != ctx_ok);

  const int h0 = kvh * G;  // first query head of the group
  const int64_t row_base = (static_cast<int64_t>(seq) * a.num_q_heads + h0);

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && !bad_split) {
      int last_issued[kStages];
#pragma unroll
      for (int s = 0; s < kStages; ++s) last_issued[s] = -1;
      for (int c = 0; c < n_chunks; ++c) {
        const int st = c % kStages;
        if (c >= kStages) {
          if (!mbar_wait(smem_u32(&sm.empty[st]), ((c / kStages) - 1) & 1, a.wait_limit_ns)) {
            report_error(a.err, kErrTimeout, kSiteDecodeWaitEmpty);
            atomicExch(&sm.abort_flag, 1);
            break;
          }
        }
        if (*reinterpret_cast<volatile int*>(&sm.abort_flag)) break;
        const int tok = s0 + c * kDecodeChunk;
        const int slot = table[tok >> 8] * kBlockSize + (tok & (kBlockSize - 1));
        const uint32_t fb = smem_u32(&sm.full[st]);
        mbar_arrive_expect_tx(fb, 2 * kChunkBytes);
        tma_load_3d(smem_u32(&sm.k[st][0][0]), &kmap, fb, 0, kvh, slot);
        tma_load_3d(smem_u32(&sm.v[st][0][0]), &vmap, fb, 0, kvh, slot);
        last_issued[st] = c;
      }
      // Every copy issued must land before the block may exit, whether or
      // not the consumers gave up on it (after a normal run these waits
      // return at once: the consumers have already seen each phase).
      for (int s = 0; s < kStages; ++s)
        if (last_issued[s] >= 0)
          mbar_wait(smem_u32(&sm.full[s]), (last_issued[s] / kStages) & 1, kDrainLimitNs);
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int gl = lane >> 1;  // pair held by this lane after the butterfly
    const int hl = gl & (G - 1);      // its head within the group
    const int tl = gl >> LG;          // its token within the step
    const float qscale = a.scale * 1.4426950408889634f;

    // q of the G heads for this lane's dimensions, permuted by hl so that
    // slot x*G + hh multiplies head hh ^ hl.
    float qp[G][DPL];
    {
      const __nv_bfloat16* qbase =
          static_cast<const __nv_bfloat16*>(a.q) + static_cast<int64_t>(seq) * a.q_row_stride +
          static_cast<int64_t>(h0) * D;
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        float x[DPL];
        load_row<DPL>(qbase + static_cast<int64_t>(hh ^ hl) * D, lane, x);
#pragma unroll
        for (int d = 0; d < DPL; ++d) qp[hh][d] = x[d] * qscale;
      }
    }
    int rowoff[TW];
#pragma unroll
    for (int x = 0; x < TW; ++x) rowoff[x] = (x ^ tl) * D;

    float o[G][DPL];
#pragma unroll
    for (int hh = 0; hh < G; ++hh)
#pragma unroll
      for (int d = 0; d < DPL; ++d) o[hh][d] = 0.f;
    float m_own = -INFINITY;  // running max of head hl (log2 domain)
    float l_own = 0.f;        // running sum of this lane's pairs

    if (!bad_split) {
      for (int c = 0; c < n_chunks; ++c) {
        const int st = c % kStages;
        // Every exit decision is taken warp-uniformly (the shuffles below use
        // the full mask).
        const bool got = mbar_wait(smem_u32(&sm.full[st]), (c / kStages) & 1, a.wait_limit_ns);
        if (!__all_sync(0xffffffffu, got)) {
          if (lane == 0) {
            report_error(a.err, kErrTimeout, kSiteDecodeWaitFull);
            atomicExch(&sm.abort_flag, 1);
          }
          break;
        }
        if (__shfl_sync(0xffffffffu, *reinterpret_cast<volatile int*>(&sm.abort_flag), 0)) break;
        const int valid = min(kDecodeChunk, n_tok - c * kDecodeChunk);
        const __nv_bfloat16* kb = &sm.k[st][0][0];
        const __nv_bfloat16* vb = &sm.v[st][0][0];
#pragma unroll 1
        for (int grp = warp; grp < GROUPS; grp += kConsumerWarps) {
          const int t0 = grp * TW;
          const int nv = valid - t0;
          if (nv <= 0) break;
          // ---- partial dot products, slot x*G + hh = pair ((x^tl)*G + (hh^hl))
          float acc[kPairs];
#pragma unroll
          for (int x = 0; x < TW; ++x) {
            float kx[DPL];
            load_row<DPL>(kb + t0 * D + rowoff[x], lane, kx);
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
              float s = qp[hh][0] * kx[0];
#pragma unroll
              for (int d = 1; d < DPL; ++d) s = fmaf(qp[hh][d], kx[d], s);
              acc[x * G + hh] = s;
            }
          }
          // ---- butterfly: each level keeps the lower half of the slots
#pragma unroll
          for (int half = 8, mask = 16; half >= 1; half >>= 1, mask >>= 1) {
#pragma unroll
            for (int i = 0; i < half; ++i)
              acc[i] += __shfl_xor_sync(0xffffffffu, acc[i + half], mask);
          }
          float s = acc[0] + __shfl_xor_sync(0xffffffffu, acc[0], 1);
          if (tl >= nv) s = -INFINITY;
          // ---- online softmax per head (max over the token bits of the lane id)
          float tm = s;
#pragma unroll
          for (int b = LG + 1; b <= 4; ++b)
            tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 1 << b));
          const float m_new = fmaxf(m_own, tm);
          const float alpha_own = fast_exp2(m_own - m_new);
          const float p = fast_exp2(s - m_new);
          l_own = l_own * alpha_own + p;
          m_own = m_new;
#pragma unroll
          for (int hh = 0; hh < G; ++hh) {
            const float al = __shfl_sync(0xffffffffu, alpha_own, lane_of_pair(hh));
#pragma unroll
            for (int d = 0; d < DPL; ++d) o[hh][d] *= al;
          }
          // ---- o += p V over the step's tokens
#pragma unroll
          for (int x = 0; x < TW; ++x) {
            float pv[G];
#pragma unroll
            for (int hh = 0; hh < G; ++hh)
              pv[hh] = __shfl_sync(0xffffffffu, p, lane_of_pair(x * G + hh));
            if (x < nv) {
              float vx[DPL];
              load_row<DPL>(vb + (t0 + x) * D, lane, vx);
#pragma unroll
              for (int hh = 0; hh < G; ++hh)
#pragma unroll
                for (int d = 0; d < DPL; ++d) o[hh][d] = fmaf(pv[hh], vx[d], o[hh][d]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.empty[st]));
      }
    }
    // ---- per-warp state -> shared memory
    // l_own summed over the lanes of the same head (token bits only; lanes
    // l and l^1 hold duplicates).
    float l_sum = l_own;
#pragma unroll
    for (int b = LG + 1; b <= 4; ++b) l_sum += __shfl_xor_sync(0xffffffffu, l_sum, 1 << b);
    if ((lane & 1) == 0 && tl == 0) {
      sm.merge_m[warp][hl] = m_own;
      sm.merge_l[warp][hl] = l_sum;
    }
#pragma unroll
    for (int hh = 0; hh < G; ++hh)
#pragma unroll
      for (int d = 0; d < DPL; ++d) sm.merge_o[warp][hh][lane * DPL + d] = o[hh][d];
  }
  __syncthreads();
  if (sm.abort_flag) return;

  // ---- merge the consumer warps and write the split result
  const bool single = (n_splits <= 1);
  for (int idx = threadIdx.x; idx < G * D; idx += kDecodeThreads) {
    const int hh = idx / D;
    const int d = idx - hh * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, sm.merge_m[w][hh]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float f = fast_exp2(sm.merge_m[w][hh] - M);
        L += sm.merge_l[w][hh] * f;
        O += sm.merge_o[w][hh][d] * f;
      }
    }
    if (single) {
      const float r = (L > 0.f && !bad_split) ? O / L : 0.f;
      static_cast<__nv_bfloat16*>(a.out)[(row_base + hh) * D + d] = __float2bfloat16_rn(r);
    } else {
      const int64_t prow = (row_base + hh) * a.max_splits + split;
      a.part_o[prow * D + d] = O;
      if (d == 0) {
        a.part_ml[prow * 2 + 0] = M;
        a.part_ml[prow * 2 + 1] = bad_split ? -1.f : L;
      }
    }
  }
}

// One CTA per (sequence, query head); one thread per dimension.
template <int D>
__global__ void __launch_bounds__(D)
decode_combine_kernel(DecodeArgs a) {
  grid_dependency_wait();
  const int row = blockIdx.x;  // seq * num_q_heads + head
  const int seq = row / a.num_q_heads;
  const int ctx = a.context_lens[seq];
  const int max_ctx = a.max_blocks * kBlockSize;
  const int ctx_ok = (ctx >= 0 && ctx <= max_ctx) ? ctx : 0;
  const int n_splits = (ctx_ok + a.split_tokens - 1) / a.split_tokens;
  if (n_splits <= 1) return;  // written directly by the split kernel
  const int d = threadIdx.x;
  const float* ml = a.part_ml + static_cast<int64_t>(row) * a.max_splits * 2;
  const float* po = a.part_o + static_cast<int64_t>(row) * a.max_splits * D;
  float M = -INFINITY;
  bool bad = false;
  for (int j = 0; j < n_splits; ++j) {
    M = fmaxf(M, ml[2 * j]);
    bad |= ml[2 * j + 1] < 0.f;
  }
  float L = 0.f, O = 0.f;
  if (M != -INFINITY) {
    for (int j = 0; j < n_splits; ++j) {
      const float f = fast_exp2(ml[2 * j] - M);
      L += ml[2 * j + 1] * f;
      O += po[static_cast<int64_t>(j) * D + d] * f;
    }
  }
  const float r = (L > 0.f && !bad) ? O / L : 0.f;
  static_cast<__nv_bfloat16*>(a.out)[static_cast<int64_t>(row) * D + d] = __float2bfloat16_rn(r);
}

template <int D, int G>
cudaError_t launch_split_t(const DecodeArgs& a, const CacheMaps& maps, cudaStream_t stream) {
  const size_t smem = sizeof(DecodeSmem<D, G>);
  auto kern = decode_split_kernel<D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int64_t blocks =
      static_cast<int64_t>(a.max_splits) * a.num_seqs * a.num_kv_heads;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kDecodeThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, maps.k_rows, maps.v_rows, a);
}

template <int D>
cudaError_t launch_split_d(const DecodeArgs& a, const CacheMaps& maps, cudaStream_t stream) {
  switch (a.num_q_heads / a.num_kv_heads) {
    case 1: return launch_split_t<D, 1>(a, maps, stream);
    case 2: return launch_split_t<D, 2>(a, maps, stream);
    case 4: return launch_split_t<D, 4>(a, maps, stream);
    case 8: return launch_split_t<D, 8>(a, maps, stream);
    case 16: return launch_split_t<D, 16>(a, maps, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_decode_split(const DecodeArgs& a, const CacheMaps& maps, cudaStream_t stream) {
  if (a.head_dim == 128) return launch_split_d<128>(a, maps, stream);
  if (a.head_dim == 64) return launch_split_d<64>(a, maps, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode_combine(const DecodeArgs& a, cudaStream_t stream) {
  if (a.max_splits <= 1) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  const int64_t rows = static_cast<int64_t>(a.num_seqs) * a.num_q_heads;
  if (rows <= 0) return cudaSuccess;
  cfg.gridDim = dim3(static_cast<unsigned>(rows));
  cfg.blockDim = dim3(a.head_dim);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (a.head_dim == 128) return cudaLaunchKernelEx(&cfg, decode_combine_kernel<128>, a);
  if (a.head_dim == 64) return cudaLaunchKernelEx(&cfg, decode_combine_kernel<64>, a);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
