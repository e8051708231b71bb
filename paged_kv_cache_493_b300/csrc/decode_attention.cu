// decode_attention.cu -- paged GQA decode attention, split-K over the
// context (flash decoding) with a log-sum-exp merge of the pieces.
//
// What is computed (intelliparadigm.com Nano-vLLM article §7.1 增量解码;
// tuning guide "Nano-vLLM性能调优实战" §2.2 flash_attn_with_kvcache over the
// paged cache; ocdem.com nano-vllm article §2.1 block tables): for sequence
// s and query head h with KV head g = h / G,
//   out[s][h] = sum_t softmax_t(scale * q[s][h] . K[s][t][g]) V[s][t][g],
// t over the context_lens[s] cached tokens, reached through the block table.
// A context may be cut into pieces ("splits"; the pages' max_splits knob,
// intelliparadigm.com article §8) that run in separate blocks; each piece
// keeps an fp32 online softmax (running max m, running sum l, unnormalised
// output o) and the pieces are merged:
//   M = max_j m_j,  L = sum_j l_j 2^(m_j - M),  out = sum_j o_j 2^(m_j - M) / L.
// Scores are kept in the log2 domain (q is pre-scaled by scale * log2 e).
//
// Work structure (stream-K).  Every (sequence, KV head) pair's context is
// a run of 32-token chunks (an empty or rejected context counts as one
// chunk, where its zero output is written).  The runs of all pairs, laid end
// to end, are cut into equal contiguous slices, one per block of a grid that
// fills the GPU once: every block has the same number of chunks to stream,
// so all blocks finish together.  Each block computes the prefix sums of the
// chunk counts over the sequences itself (the lengths live on the device).
// The piece of a pair inside one slice is either the whole pair (its output
// is written directly) or a cut piece: its partial state goes to one of the
// block's two partial slots and the block counts it on the pair's arrival
// counter; the block that writes the pair's last piece merges all of them
// once its own slice is done, with all its threads (there is no second
// kernel).  Counters carry a generation kept on the device (the last block of
// a launch advances it), so nothing is ever reset between launches.
// In one block:
//   warp 4        producer: one lane walks the block's slice, looks up each
//                 chunk's physical block, and issues TMA tile loads (K and V
//                 rows of the KV head, 32 x head_dim bf16 each; with a
//                 piece's first chunk also the G query rows) into a 4-stage
//                 ring completing on mbarriers.  Each stage carries a
//                 descriptor (sequence, KV head, slot, valid tokens, first /
//                 last chunk of the piece); a final stage marks the end.
//   warps 0..3    consumers: each takes a group of tokens of every chunk.
//                 A lane owns head_dim/32 dimensions of the G query heads of
//                 the group, so each K/V row loaded once from shared memory
//                 serves all G query heads.  The G x T partial dot products of
//                 a group (T = 16/G tokens) are reduced across the warp with a
//                 butterfly in which every shuffle halves the values a lane
//                 still holds (16 shuffles for 16 dot products instead of 80);
//                 the slot order of the partials is permuted per lane so that
//                 no selects are needed.  After the reduction lane l holds the
//                 score of pair g(l) (twice: lanes l and l^1).  At the last
//                 chunk of a piece the four warps merge their states and write
//                 the output (a whole pair) or the piece's partials.
// The pipeline is HBM-bound: per token and KV head the kernel reads
// 2 * head_dim * 2 bytes of K/V and does 4 * G * head_dim flops.
#include <algorithm>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int kStages = 4;
constexpr int kConsumerWarps = 4;
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;
constexpr int kPairs = 16;  // (token, head) dot products per warp step

// Descriptor of one ring stage, written by the producer before it arrives
// on the stage's full barrier.
struct StageInfo {
  int seq, kvh, slot, n_valid, flags;
  int c_first, c_last;  // blocks holding the pair's first and last chunk
  int first_slot;       // partial slot of the pair's piece in block c_first
};
constexpr int kFirst = 1;   // first chunk of a piece: reset the state, load q
constexpr int kLast = 2;    // last chunk of a piece: merge and write
constexpr int kBad = 4;     // the chunk's length or block id is out of range
constexpr int kSingle = 8;  // the piece is the whole pair: write the output itself
constexpr int kEnd = 16;    // the slice is done: leave the loop

// The block whose slice holds chunk x when T chunks are cut into nb equal
// slices (slice c = [c T / nb, (c + 1) T / nb)).
__device__ __forceinline__ int block_of_chunk(long long x, long long T, long long nb) {
  return static_cast<int>(((x + 1) * nb - 1) / T);
}
__device__ __forceinline__ long long slice_begin(long long c, long long T, long long nb) {
  return c * T / nb;
}

// Tagged counters: high bits the launch generation, low kCountBits bits a
// count.  A counter whose tag is not this launch's counts as zero.
constexpr int kCountBits = 24;
constexpr unsigned long long kCountMask = (1ull << kCountBits) - 1;
constexpr unsigned long long kGenMask = (1ull << (64 - kCountBits)) - 1;
constexpr int kPairCounterOffset = 256 / sizeof(unsigned long long);  // after the header

// Adds one to a tagged counter; returns the count after the addition.  Two
// plain atomics and no compare-and-swap loop, so many blocks arriving at
// once do not retry: the max lifts a counter of an older generation to
// (gen, 0) and leaves one of this generation alone; the add then counts.
__device__ __forceinline__ unsigned long long tagged_increment(unsigned long long* cnt,
                                                               unsigned long long gen) {
  atomicMax(cnt, gen << kCountBits);
  return (atomicAdd(cnt, 1ull) & kCountMask) + 1;
}

template <int D, int G>
struct DecodeSmem {
  alignas(128) __nv_bfloat16 k[kStages][kDecodeChunk][D];
  alignas(128) __nv_bfloat16 v[kStages][kDecodeChunk][D];
  alignas(128) __nv_bfloat16 q[kStages][G * D];
  float merge_o[kConsumerWarps][G][D];
  float merge_m[kConsumerWarps][G];
  float merge_l[kConsumerWarps][G];
  StageInfo info[kStages];
  long long scan[kDecodeThreads / 32];
  long long start_base;  // chunk offset (per KV head) of the slice's first sequence
  unsigned long long gen;  // this launch's generation (counter tag)
  StageInfo merge_todo[2];  // cut pairs whose last piece this block wrote
  int n_merge;
  int start_seq;
  alignas(8) uint64_t full[kStages];
  alignas(8) uint64_t empty[kStages];
  alignas(8) uint64_t merge_full;  // the four warps' piece states are in merge_*
  alignas(8) uint64_t merge_free;  // ... and have been read
  int abort_flag;
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

// Chunks of each of sequence s's pairs: ceil(C / 32), and 1 for an empty
// or out-of-range context (that chunk carries no tokens).
__device__ __forceinline__ int seq_chunks(const DecodeArgs& a, int s, int max_ctx) {
  const int ctx = a.context_lens[s];
  return (ctx <= 0 || ctx > max_ctx) ? 1 : (ctx + kDecodeChunk - 1) / kDecodeChunk;
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
  constexpr uint32_t kQBytes = G * D * 2;
  constexpr int kConsumerThreads = kConsumerWarps * 32;
  constexpr int kWarps = kDecodeThreads / 32;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  DecodeSmem<D, G>& sm = *reinterpret_cast<DecodeSmem<D, G>*>(smem_raw);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), kConsumerWarps);
    }
    mbar_init(smem_u32(&sm.merge_full), kConsumerWarps);
    mbar_init(smem_u32(&sm.merge_free), kConsumerWarps);
    sm.abort_flag = 0;
    sm.n_merge = 0;
    sm.start_seq = -1;
    sm.start_base = 0;
    fence_barrier_init();
  }
  if (warp == kConsumerWarps && lane == 0) {
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
  }
  // Inputs may be written by the previous kernel in the stream: nothing
  // global is read before this point.
  grid_dependency_wait();
  grid_dependents_launch();

  const int max_ctx = a.max_blocks * kBlockSize;
  const int hkv = a.num_kv_heads;
  // The epoch changes only after every block of this launch has passed this
  // point (the last block to finish advances it), so all blocks agree.
  if (threadIdx.x == 0) sm.gen = ((__ldcg(a.counters) + 1) & kGenMask);

  // ---- prefix sums of the chunk counts over the sequences (whole block):
  // thread t owns sequences [seg0, seg1).
  const int per = (a.num_seqs + kDecodeThreads - 1) / kDecodeThreads;
  const int seg0 = min(static_cast<int>(threadIdx.x) * per, a.num_seqs);
  const int seg1 = min(seg0 + per, a.num_seqs);
  long long mine = 0;
  for (int s = seg0; s < seg1; ++s) mine += seq_chunks(a, s, max_ctx);
  long long incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sm.scan[warp] = incl;
  __syncthreads();
  long long before = 0, total = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    if (w < warp) before += sm.scan[w];
    total += sm.scan[w];
  }
  const long long excl = before + incl - mine;  // chunks per KV head before seg0
  const long long T = total * hkv;              // chunks of all pairs
  const long long nb = gridDim.x;
  const long long ca = static_cast<long long>(blockIdx.x) * T / nb;        // slice begin
  const long long cb = (static_cast<long long>(blockIdx.x) + 1) * T / nb;  // slice end
  if (ca < cb && ca >= excl * hkv && ca < (excl + mine) * hkv) {
    long long p = excl;
    for (int s = seg0; s < seg1; ++s) {
      const int n = seq_chunks(a, s, max_ctx);
      if (ca < (p + n) * hkv) {
        sm.start_seq = s;
        sm.start_base = p;
        break;
      }
      p += n;
    }
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // Last post of each stage (copies or descriptor only): phases of one
      // barrier complete in order, so once that one is complete every copy
      // ever issued into the stage has landed.
      int last_posted[kStages];
#pragma unroll
      for (int s = 0; s < kStages; ++s) last_posted[s] = -1;
      int c = 0;  // stages posted so far (stage c % kStages, phase c / kStages)
      bool aborted = false;
      // Claims the next ring stage; false when the wait for it expired.
      auto claim = [&](int st) -> bool {
        if (c >= kStages &&
            !mbar_wait(smem_u32(&sm.empty[st]), ((c / kStages) - 1) & 1, a.wait_limit_ns)) {
          report_error(a.err, kErrTimeout, kSiteDecodeWaitEmpty);
          atomicExch(&sm.abort_flag, 1);
          return false;
        }
        return *reinterpret_cast<volatile int*>(&sm.abort_flag) == 0;
      };

      int seq = sm.start_seq;
      if (ca < cb && seq >= 0) {
        long long base = sm.start_base * hkv;  // first chunk of seq's pairs
        int ctx = a.context_lens[seq];
        bool ctx_bad = ctx < 0 || ctx > max_ctx;
        int nch = seq_chunks(a, seq, max_ctx);
        if (ctx_bad && base >= ca) report_error(a.err, kErrDeviceCheck, kSiteDecodeContext);
        long long pos = ca;
        int piece = 0;
        while (pos < cb && !aborted) {
          const int kvh = static_cast<int>((pos - base) / nch);
          const int k0 = static_cast<int>((pos - base) % nch);
          const long long pair_end = base + static_cast<long long>(kvh + 1) * nch;
          const long long piece_end = pair_end < cb ? pair_end : cb;
          const int n = static_cast<int>(piece_end - pos);
          const bool whole = k0 == 0 && piece_end == pair_end;
          const int slot = piece == 0 ? 0 : 1;
          const long long pair_begin = pair_end - nch;
          const int c_first = block_of_chunk(pair_begin, T, nb);
          const int c_last = block_of_chunk(pair_end - 1, T, nb);
          const int first_slot = slice_begin(c_first, T, nb) == pair_begin ? 0 : 1;
          const int32_t* table = a.block_tables + static_cast<int64_t>(seq) * a.max_blocks;
          for (int k = k0; k < k0 + n; ++k, ++c) {
            const int st = c % kStages;
            if (!claim(st)) {
              aborted = true;
              break;
            }
            const int tok = k * kDecodeChunk;
            const int n_valid = (ctx_bad || ctx <= 0) ? 0 : min(kDecodeChunk, ctx - tok);
            int id = 0;
            bool bad = ctx_bad;
            if (n_valid > 0) {
              id = table[tok >> 8];
              if (id < 0 || id >= a.num_blocks) {
                bad = true;
                report_error(a.err, kErrDeviceCheck, kSiteDecodeBlock);
              }
            }
            StageInfo& inf = sm.info[st];
            inf.seq = seq;
            inf.kvh = kvh;
            inf.slot = slot;
            inf.n_valid = bad ? 0 : n_valid;
            inf.flags = (bad ? kBad : 0) | (whole ? kSingle : 0) | (k == k0 ? kFirst : 0) |
                        (k == k0 + n - 1 ? kLast : 0);
            inf.c_first = c_first;
            inf.c_last = c_last;
            inf.first_slot = first_slot;
            const uint32_t fb = smem_u32(&sm.full[st]);
            last_posted[st] = c;
            if (inf.n_valid <= 0) {
              mbar_arrive(fb);  // descriptor only
            } else {
              const int slot_row = id * kBlockSize + (tok & (kBlockSize - 1));
              mbar_arrive_expect_tx(fb, 2 * kChunkBytes + (k == k0 ? kQBytes : 0u));
              tma_load_3d(smem_u32(&sm.k[st][0][0]), &kmap, fb, 0, kvh, slot_row);
              tma_load_3d(smem_u32(&sm.v[st][0][0]), &vmap, fb, 0, kvh, slot_row);
              if (k == k0)
                bulk_load(smem_u32(&sm.q[st][0]),
                          static_cast<const __nv_bfloat16*>(a.q) +
                              static_cast<int64_t>(seq) * a.q_row_stride +
                              static_cast<int64_t>(kvh) * G * D,
                          kQBytes, fb);
            }
          }
          pos = piece_end;
          ++piece;
          if (pos == pair_end && kvh + 1 == hkv && pos < cb) {  // next sequence
            ++seq;
            base = pair_end;
            ctx = a.context_lens[seq];
            ctx_bad = ctx < 0 || ctx > max_ctx;
            nch = seq_chunks(a, seq, max_ctx);
            if (ctx_bad) report_error(a.err, kErrDeviceCheck, kSiteDecodeContext);
          }
        }
      }
      if (!aborted) {  // end marker
        const int st = c % kStages;
        if (claim(st)) {
          sm.info[st].flags = kEnd;
          last_posted[st] = c;
          mbar_arrive(smem_u32(&sm.full[st]));
        }
      }
      // Every copy issued must land before the block may exit, whether or
      // not the consumers gave up on it (after a normal run these waits
      // return at once: the consumers have already seen each phase).
      for (int s = 0; s < kStages; ++s)
        if (last_posted[s] >= 0)
          mbar_wait(smem_u32(&sm.full[s]), (last_posted[s] / kStages) & 1, kDrainLimitNs);
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int gl = lane >> 1;  // pair held by this lane after the butterfly
    const int hl = gl & (G - 1);      // its head within the group
    const int tl = gl >> LG;          // its token within the step
    const float qscale = a.scale * 1.4426950408889634f;
    int rowoff[TW];
#pragma unroll
    for (int x = 0; x < TW; ++x) rowoff[x] = (x ^ tl) * D;

    float qp[G][DPL];
    float o[G][DPL];
    float m_own = -INFINITY;  // running max of head hl (log2 domain)
    float l_own = 0.f;        // running sum of this lane's pairs
    bool piece_bad = false;
#pragma unroll
    for (int hh = 0; hh < G; ++hh)
#pragma unroll
      for (int d = 0; d < DPL; ++d) qp[hh][d] = o[hh][d] = 0.f;

    int pieces_done = 0;  // pieces this block's consumers have merged
    for (int c = 0;; ++c) {
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
      const StageInfo inf = sm.info[st];
      if (inf.flags & kEnd) break;
      if (inf.flags & kFirst) {
        m_own = -INFINITY;
        l_own = 0.f;
        piece_bad = false;
#pragma unroll
        for (int hh = 0; hh < G; ++hh)
#pragma unroll
          for (int d = 0; d < DPL; ++d) o[hh][d] = 0.f;
        if (inf.n_valid > 0) {
          // q of the G heads for this lane's dimensions, permuted by hl so
          // that slot x*G + hh multiplies head hh ^ hl.
#pragma unroll
          for (int hh = 0; hh < G; ++hh) {
            float x[DPL];
            load_row<DPL>(&sm.q[st][(hh ^ hl) * D], lane, x);
#pragma unroll
            for (int d = 0; d < DPL; ++d) qp[hh][d] = x[d] * qscale;
          }
        }
      }
      piece_bad |= (inf.flags & kBad) != 0;
      const int valid = inf.n_valid;
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

      if (inf.flags & kLast) {
        // ---- merge the four warps' states and write the piece's result.
        // The hand-over between the warps uses mbarriers with bounded waits
        // (not bar.sync), so a warp that gave up cannot strand the others.
        // l_own summed over the lanes of the same head (token bits only;
        // lanes l and l^1 hold duplicates).
        float l_sum = l_own;
#pragma unroll
        for (int b = LG + 1; b <= 4; ++b) l_sum += __shfl_xor_sync(0xffffffffu, l_sum, 1 << b);
        const int k = pieces_done++;
        const bool freed = k == 0 || mbar_wait(smem_u32(&sm.merge_free), (k - 1) & 1,
                                               a.wait_limit_ns);
        if (!__all_sync(0xffffffffu, freed)) {
          if (lane == 0) {
            report_error(a.err, kErrTimeout, kSiteDecodeWaitMerge);
            atomicExch(&sm.abort_flag, 1);
          }
          break;
        }
        if ((lane & 1) == 0 && tl == 0) {
          sm.merge_m[warp][hl] = m_own;
          sm.merge_l[warp][hl] = l_sum;
        }
#pragma unroll
        for (int hh = 0; hh < G; ++hh)
#pragma unroll
          for (int d = 0; d < DPL; ++d) sm.merge_o[warp][hh][lane * DPL + d] = o[hh][d];
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.merge_full));
        const bool merged = mbar_wait(smem_u32(&sm.merge_full), k & 1, a.wait_limit_ns);
        if (!__all_sync(0xffffffffu, merged)) {
          if (lane == 0) {
            report_error(a.err, kErrTimeout, kSiteDecodeWaitMerge);
            atomicExch(&sm.abort_flag, 1);
          }
          break;
        }
        const int64_t row_base = static_cast<int64_t>(inf.seq) * a.num_q_heads + inf.kvh * G;
        const int64_t prow = (static_cast<int64_t>(blockIdx.x) * 2 + inf.slot) * G;
        for (int idx = threadIdx.x; idx < G * D; idx += kConsumerThreads) {
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
          if (inf.flags & kSingle) {
            const float r = (L > 0.f && !piece_bad) ? O / L : 0.f;
            static_cast<__nv_bfloat16*>(a.out)[(row_base + hh) * D + d] = __float2bfloat16_rn(r);
          } else {
            a.part_o[(prow + hh) * D + d] = O;
            if (d == 0) {
              a.part_ml[(prow + hh) * 2 + 0] = M;
              a.part_ml[(prow + hh) * 2 + 1] = piece_bad ? -1.f : L;
            }
          }
        }
        if (!(inf.flags & kSingle)) __threadfence();  // partials visible before the arrival
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.merge_free));
        if (!(inf.flags & kSingle) && warp == 0) {
          // ---- a cut pair: once all four warps have written the piece,
          // count it on the pair's arrival counter; the block that brings
          // the count to the pair's number of pieces merges them.
          const bool all_written =
              mbar_wait(smem_u32(&sm.merge_free), k & 1, a.wait_limit_ns);
          if (!__all_sync(0xffffffffu, all_written)) {
            if (lane == 0) {
              report_error(a.err, kErrTimeout, kSiteDecodeWaitMerge);
              atomicExch(&sm.abort_flag, 1);
            }
            break;
          }
          // A block holds at most two cut pieces (the first and the last of
          // its slice), so at most two merges land here; they run after
          // the slice, with every thread of the block.
          if (lane == 0) {
            int pieces = 0;  // blocks with a non-empty slice in [c_first, c_last]
            for (int cb2 = inf.c_first; cb2 <= inf.c_last; ++cb2)
              pieces += slice_begin(cb2 + 1, T, nb) > slice_begin(cb2, T, nb);
            unsigned long long* cnt = a.counters + kPairCounterOffset +
                                      static_cast<int64_t>(inf.seq) * hkv + inf.kvh;
            if (static_cast<int>(tagged_increment(cnt, sm.gen)) == pieces && sm.n_merge < 2)
              sm.merge_todo[sm.n_merge++] = inf;
            __threadfence();
          }
          __syncwarp();
        }
      }
    }
  }
  __syncthreads();
  // ---- merge the cut pairs whose last piece arrived here (log-sum-exp):
  //   M = max_j m_j, L = sum_j l_j 2^(m_j - M), out = sum_j o_j 2^(m_j - M) / L.
  if (!*reinterpret_cast<volatile int*>(&sm.abort_flag)) {
    for (int j = 0; j < sm.n_merge; ++j) {
      const StageInfo inf = sm.merge_todo[j];
      const int64_t row_base = static_cast<int64_t>(inf.seq) * a.num_q_heads + inf.kvh * G;
      for (int idx = threadIdx.x; idx < G * D; idx += kDecodeThreads) {
        const int hh = idx / D;
        const int d = idx - hh * D;
        float M = -INFINITY;
        bool bad = false;
        for (int cb2 = inf.c_first; cb2 <= inf.c_last; ++cb2) {
          if (slice_begin(cb2 + 1, T, nb) <= slice_begin(cb2, T, nb)) continue;
          const int sl = cb2 == inf.c_first ? inf.first_slot : 0;
          const int64_t r2 = (static_cast<int64_t>(cb2) * 2 + sl) * G + hh;
          M = fmaxf(M, __ldcg(a.part_ml + r2 * 2));
          bad |= __ldcg(a.part_ml + r2 * 2 + 1) < 0.f;
        }
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
          for (int cb2 = inf.c_first; cb2 <= inf.c_last; ++cb2) {
            if (slice_begin(cb2 + 1, T, nb) <= slice_begin(cb2, T, nb)) continue;
            const int sl = cb2 == inf.c_first ? inf.first_slot : 0;
            const int64_t r2 = (static_cast<int64_t>(cb2) * 2 + sl) * G + hh;
            const float f = fast_exp2(__ldcg(a.part_ml + r2 * 2) - M);
            L += __ldcg(a.part_ml + r2 * 2 + 1) * f;
            O += __ldcg(a.part_o + r2 * D + d) * f;
          }
        }
        const float r = (L > 0.f && !bad) ? O / L : 0.f;
        static_cast<__nv_bfloat16*>(a.out)[(row_base + hh) * D + d] = __float2bfloat16_rn(r);
      }
    }
  }
  __syncthreads();
  // Count this block as finished; the last one advances the epoch, which
  // gives the next launch a new generation.
  if (threadIdx.x == 0) {
    __threadfence();
    if (tagged_increment(a.counters + 1, sm.gen) == gridDim.x)
      atomicExch(a.counters, sm.gen);  // epoch := generation (epoch + 1)
  }
}

template <int D, int G>
int ctas_per_sm() {
  static int per_sm = 0;
  if (per_sm == 0) {
    const size_t smem = sizeof(DecodeSmem<D, G>);
    auto kern = decode_split_kernel<D, G>;
    int n = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kDecodeThreads, smem) !=
            cudaSuccess) {
      cudaGetLastError();
      return 1;
    }
    per_sm = n > 0 ? n : 1;
  }
  return per_sm;
}

template <int D>
int ctas_per_sm_d(int group) {
  switch (group) {
    case 1: return ctas_per_sm<D, 1>();
    case 2: return ctas_per_sm<D, 2>();
    case 4: return ctas_per_sm<D, 4>();
    case 8: return ctas_per_sm<D, 8>();
    default: return ctas_per_sm<D, 16>();
  }
}

template <int D, int G>
cudaError_t launch_split_t(const DecodeArgs& a, const CacheMaps& maps, cudaStream_t stream) {
  const size_t smem = sizeof(DecodeSmem<D, G>);
  auto kern = decode_split_kernel<D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (a.num_ctas <= 0) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(a.num_ctas));
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

int decode_num_ctas(int head_dim, int group, int num_sms, int64_t num_pairs, int max_splits) {
  const int per_sm = head_dim == 64 ? ctas_per_sm_d<64>(group) : ctas_per_sm_d<128>(group);
  int64_t n = static_cast<int64_t>(per_sm) * (num_sms > 0 ? num_sms : 1);
  if (max_splits > 0 && num_pairs * max_splits < n) n = num_pairs * max_splits;
  if (n < 1) n = 1;
  return static_cast<int>(n);
}

size_t decode_counter_bytes(int64_t num_pairs) {
  return 256 + ((static_cast<size_t>(num_pairs) * sizeof(unsigned long long) + 255) / 256) * 256;
}

size_t decode_partial_bytes(int num_ctas, int group, int head_dim) {
  const size_t rows = static_cast<size_t>(num_ctas) * 2 * group;
  return rows * head_dim * sizeof(float) + rows * 2 * sizeof(float);
}

cudaError_t launch_decode(const DecodeArgs& a, const CacheMaps& maps, cudaStream_t stream) {
  if (a.head_dim == 128) return launch_split_d<128>(a, maps, stream);
  if (a.head_dim == 64) return launch_split_d<64>(a, maps, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
