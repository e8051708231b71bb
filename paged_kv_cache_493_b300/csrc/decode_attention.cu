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
// Scores are kept in the log2 domain (scaled by scale * log2 e after the
// product; q itself is used unscaled).
//
// Work structure (stream-K).  Every (sequence, KV head) pair's context is
// a run of 32-token chunks (an empty or rejected context counts as one
// chunk, where its zero output is written), preceded by pair_gap cost units
// that hold nothing (what a piece boundary costs, in chunks).  The runs of
// all pairs, laid end to end, are cut into equal contiguous slices of cost,
// one per block of a grid that fills the GPU once, so that all blocks
// finish together.  Each block computes the prefix sums of the costs over
// the sequences itself (the lengths live on the device).
// The piece of a pair inside one slice is either the whole pair (its output
// is written directly) or a cut piece: its partial state goes to one of the
// block's two partial slots and is counted on the pair's arrival counter;
// the block that brings the count to the pair's number of pieces merges all
// of them (there is no second kernel).  A slice's trailing cut piece is
// streamed first, so that cross-block merges happen while the streams go on
// and every block ends on a piece that needs none.  Counters carry a launch
// generation kept on the device (the last block of a launch to start
// advances it), so nothing is ever reset between launches, and replays of
// a captured graph stay correct.
// In one block (seven warps):
//   warp 4        producer: one lane walks the block's slice, looks up each
//                 chunk's physical block, and issues TMA tile loads (K and V
//                 rows of the KV head, 32 tokens x 64 dimensions per panel,
//                 128-byte swizzle; with a piece's first chunk also the G
//                 query rows) into a 4-stage ring completing on mbarriers.
//                 Each stage carries a descriptor (sequence, KV head, slot,
//                 valid tokens, first / last chunk of the piece); a final
//                 stage marks the end.
//   warps 0..3    consumers: bf16: warp w computes the chunks c with
//                 c % 4 == w; INT8 (64-token chunks): every warp computes
//                 its 16 tokens of every chunk.  Each reads every stage's
//                 descriptor.  A chunk is two
//                 small contractions on the tensor cores (mma.sync m16n8k16,
//                 bf16 in, fp32 accumulate): S^T = K q^T with the 32 tokens
//                 as rows and the G query heads as columns (padded to 8), so
//                 one K row fetched from shared memory serves the whole GQA
//                 group; then O^T += V^T P^T with the head dimensions as rows.
//                 The accumulator layout of S^T becomes the operand layout of
//                 P^T by one 8x8 transpose in registers (movmatrix) per 16
//                 tokens; the per-head running max is reduced over the eight
//                 lanes that hold a head's tokens.  At the last chunk of a
//                 piece each warp posts its state to a shared-memory mailbox
//                 and goes on.
//   warp 5        merger: combines the four warps' states of each posted
//                 piece, frees the mailbox, then writes a whole pair's output
//                 or a cut piece's partials and counts it.  Cascade decode:
//                 a whole pair's private state is set aside and folded with
//                 the shared-prefix partials after the stream (fold_deferred).
//   warp 6        merge warp: merges the pieces of the cut pairs whose count
//                 this block completed (reads of partials written by other
//                 blocks: L2 round trips, kept off the consumers' path).
// P is rounded to bf16 for the PV product (its sum l stays fp32).  V rows
// past the context in a final, partial chunk are zeroed in shared memory
// before the product (their pool contents may be anything).
// The pipeline is HBM-bound: per token and KV head the kernel reads
// 2 * head_dim * 2 bytes of K/V and does 4 * G * head_dim flops.
#include <algorithm>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

// Tokens per chunk (the unit of the stream-K plan and of a ring stage): 32
// for bf16, 64 for INT8, so that an INT8 stage carries as many bytes (16 KB
// of K + V at D = 128) and the per-chunk costs (descriptor, copies, barrier
// hand-overs) are paid per 16 KB either way.  Ring stages: 4.
template <bool kI8>
constexpr int kChunkOf = kI8 ? 2 * kDecodeChunk : kDecodeChunk;
template <bool kI8>
constexpr int kStagesOf = 4;
constexpr int kConsumerWarps = 4;  // warps 0..3 (which tokens each computes: see the header)
constexpr int kProducerWarp = 4;   // TMA issue
constexpr int kMergerWarp = 5;     // combines the consumers' states, writes results, counts pieces
constexpr int kMergeWarp = 6;      // merges the pieces of cut contexts (log-sum-exp over L2)
constexpr int kDecodeThreads = 7 * 32;
constexpr int kSliceTable = 1024;  // table entries of a slice's sequences kept in shared memory
constexpr int kSliceSlots = 256;   // fused store: slots of a slice's sequences kept likewise
constexpr int kDeferRows = 64;     // cascade decode: rows of whole pairs folded after the stream
constexpr int kPrefetchLines = 256;  // L2 prefetch of the tables per block, in 128-byte lines

// Descriptor of one ring stage, written by the producer before it arrives
// on the stage's full barrier.
struct alignas(16) StageInfo {  // 48 bytes: copied with three 16-byte accesses
  int seq, kvh, slot, n_valid, flags;
  int c_first, c_last;  // blocks holding the pair's first and last chunk
  int first_slot;       // partial slot of the pair's piece in block c_first
  // Fused store: the cache slot of the sequence's new token when this chunk
  // holds it and its row is to be stored (else -1), and its row in the chunk.
  int store_slot, store_row;
  int pad[2];
};
constexpr int kFirst = 1;   // first chunk of a piece: reset the state, load q
constexpr int kLast = 2;    // last chunk of a piece: merge and write
constexpr int kBad = 4;     // the chunk's length or block id is out of range
constexpr int kSingle = 8;  // the piece is the whole pair: write the output itself
constexpr int kEnd = 16;    // the slice is done: leave the loop

// The block whose slice holds position x when T cost units are cut into nb
// equal slices (slice c = [c T / nb, (c + 1) T / nb)); a chunk is one unit,
// and belongs to the block whose slice holds it.
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
// The add has acquire-release semantics at GPU scope: the caller's earlier
// writes (and those of its warp, ordered by a preceding __syncwarp) are
// visible to whoever observes the count, and the caller sees what the
// earlier arrivals wrote.
__device__ __forceinline__ unsigned long long tagged_increment(unsigned long long* cnt,
                                                               unsigned long long gen) {
  atomicMax(cnt, gen << kCountBits);
  unsigned long long old;
  asm volatile("atom.add.acq_rel.gpu.global.u64 %0, [%1], %2;"
               : "=l"(old)
               : "l"(cnt), "l"(1ull)
               : "memory");
  return (old & kCountMask) + 1;
}

// Acquire-release fence at GPU scope (lighter than the sequentially
// consistent __threadfence).
__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

constexpr int kPanelBytes = kDecodeChunk * 128;  // 32 rows x 64 dimensions (bf16)

// Scratch of one warp folding the shared-prefix partials of a pair into the
// state of its private part (cascade decode).
template <int G>
struct FoldScratch {
  float fp[G];     // factor of the private state, 2^(M_private - M)
  float L[G];      // merged sum
  int bad[G];      // a unit's row failed
  float w[G][kMaxSharedUnits];  // factor of unit u, 2^(m_u - M)
};

// Cascade decode, one head h of pair (seq, kvh), by one warp: given the
// private part's reference max Mp and sum Lp, reads the shared_units partial
// states (m_u, l_u) of the row and computes the merged reference
// M = max(Mp, max_u m_u), the factors fp = 2^(Mp - M) and w_u = 2^(m_u - M),
// and L = Lp fp + sum_u l_u w_u (log-sum-exp merge, as for split pieces).
// Lane u handles unit u (shared_units <= 32).  Results go to f (lane 0
// writes fp, L, bad; lane u writes w[h][u]); the caller syncs the warp.
template <int G>
__device__ __forceinline__ void fold_head(const DecodeArgs& a, int seq, int kvh, int h, float Mp,
                                          float Lp, FoldScratch<G>& f, int lane) {
  const int U = a.shared_units;
  const int64_t row = (static_cast<int64_t>(kvh) * U + lane) * a.shared_rows_pad +
                      static_cast<int64_t>(seq) * G + h;
  float2 ml = make_float2(-INFINITY, 0.f);
  if (lane < U) ml = __ldcg(reinterpret_cast<const float2*>(a.shared_ml) + row);
  const bool bad = __any_sync(0xffffffffu, lane < U && ml.y < 0.f);
  float M = ml.x;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  M = fmaxf(M, Mp);
  const bool none = M == -INFINITY;
  const float w = (lane < U && !none && ml.x != -INFINITY) ? fast_exp2(ml.x - M) : 0.f;
  float Ls = ml.y * w;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
  if (lane < U) f.w[h][lane] = w;
  if (lane == 0) {
    const float fp = (none || Mp == -INFINITY) ? 0.f : fast_exp2(Mp - M);
    f.fp[h] = fp;
    f.L[h] = Lp * fp + Ls;
    f.bad[h] = bad ? 1 : 0;
  }
}

// Address of dimension d of head h's unnormalised output in unit u's partial
// state of pair (seq, kvh).
template <int D, int G>
__device__ __forceinline__ const float* shared_o_at(const DecodeArgs& a, int seq, int kvh, int h,
                                                    int u, int d) {
  return a.shared_o +
         ((static_cast<int64_t>(kvh) * a.shared_units + u) * a.shared_rows_pad +
          static_cast<int64_t>(seq) * G + h) * D + d;
}

// Cascade decode, one warp, after the block's stream: folds the shared-prefix
// partial states (one per row: the cluster merged the units) into the private
// states the merger set aside for the n pairs of list, and writes their
// outputs.  Per row, with (Mp, Lp, Op) private and (m, l, Os) shared:
//   M = max(Mp, m), L = Lp 2^(Mp - M) + l 2^(m - M),
//   out = (Op 2^(Mp - M) + Os 2^(m - M)) / L.
// A sequence whose leading table entries are not row 0's, or a row the
// shared kernel failed on (l < 0), gets zeros (the former is reported).  Both
// outputs of every pair come in by bulk copies into `stage` (the K/V ring,
// idle once the stream is done; 2 x kDeferRows x D fp32) at once, while the
// lanes take the pairs' table entries and then their rows' (max, sum).
template <int D, int G>
__device__ __noinline__ void fold_deferred(const DecodeArgs& a, const int2* list, int* unshared,
                                           float2* f, int n, float* stage, uint32_t bar,
                                           int lane) {
  // The private rows were written by this warp's lanes: order them before
  // the bulk copies (async proxy) that read them.
  asm volatile("fence.proxy.async.global;" ::: "memory");
  const int nsb = a.shared_len / kBlockSize;
  for (int j = lane; j < n; j += 32) unshared[j] = 0;
  __syncwarp();
  for (int i = lane; i < n * nsb; i += 32) {
    const int j = i / nsb;
    const int b = i - j * nsb;
    const int32_t* t = a.block_tables + static_cast<int64_t>(list[j].x) * a.max_blocks;
    if (__ldg(t + b) != __ldg(a.block_tables + b)) unshared[j] = 1;
  }
  __syncwarp();
  grid_dependency_wait();  // the shared-prefix kernel's partials (see the kernel's start)
  constexpr uint32_t kPairBytes = G * D * sizeof(float);
  float* so = stage;                     // [n][G][D]: the shared partial outputs
  float* po = stage + kDeferRows * D;    // [n][G][D]: the private outputs
  if (lane == 0) {
    mbar_arrive_expect_tx(bar, 2u * static_cast<uint32_t>(n) * kPairBytes);
    for (int j = 0; j < n; ++j) {
      const int64_t row0 = static_cast<int64_t>(list[j].y) * a.shared_rows_pad +
                           static_cast<int64_t>(list[j].x) * G;
      bulk_load(smem_u32(so + j * G * D), a.shared_o + row0 * D, kPairBytes, bar);
      bulk_load(smem_u32(po + j * G * D), a.private_o + row0 * D, kPairBytes, bar);
    }
  }
  bool any_unshared = false;
  for (int r = lane; r < n * G; r += 32) {
    const int j = r / G;
    const int h = r - j * G;
    const int64_t row = static_cast<int64_t>(list[j].y) * a.shared_rows_pad +
                        static_cast<int64_t>(list[j].x) * G + h;
    const float2 pv = __ldcg(reinterpret_cast<const float2*>(a.private_ml) + row);
    const float2 sh = __ldcg(reinterpret_cast<const float2*>(a.shared_ml) + row);
    const float M = fmaxf(pv.x, sh.x);
    const bool none = M == -INFINITY;
    const float fp = (none || pv.x == -INFINITY) ? 0.f : fast_exp2(pv.x - M);
    const float fsh = (none || sh.x == -INFINITY) ? 0.f : fast_exp2(sh.x - M);
    const float L = pv.y * fp + sh.y * fsh;
    any_unshared |= unshared[j] != 0;
    const float inv = (L > 0.f && !unshared[j] && !(sh.y < 0.f)) ? 1.f / L : 0.f;
    f[r] = make_float2(fp * inv, fsh * inv);
  }
  if (__any_sync(0xffffffffu, any_unshared) && lane == 0)
    report_error(a.err, kErrDeviceCheck, kSiteDecodeShared);
  if (!__all_sync(0xffffffffu, mbar_wait(bar, 0, a.wait_limit_ns))) {
    if (lane == 0) {
      report_error(a.err, kErrTimeout, kSiteDecodeWaitMerge);
      mbar_wait(bar, 0, kDrainLimitNs);  // the copies land before the block exits
    }
    __syncwarp();
    return;
  }
  constexpr int kGroups = D / 4;
  const int total = n * G * kGroups;
#pragma unroll 4
  for (int i = lane; i < total; i += 32) {
    const int r = i / kGroups;
    const int d = (i - r * kGroups) * 4;
    const int j = r / G;
    const int h = r - j * G;
    const int seq = list[j].x;
    const int kvh = list[j].y;
    const float4 x = *reinterpret_cast<const float4*>(po + r * D + d);
    const float4 y = *reinterpret_cast<const float4*>(so + r * D + d);
    const float2 w = f[r];
    uint2 packed;
    packed.x = pack_bf16x2(x.x * w.x + y.x * w.y, x.y * w.x + y.y * w.y);
    packed.y = pack_bf16x2(x.z * w.x + y.z * w.y, x.w * w.x + y.w * w.y);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) +
                              (static_cast<int64_t>(seq) * a.num_q_heads + kvh * G + h) * D + d) =
        packed;
  }
}

// The ring's K/V tiles.  bf16: per stage, D / 64 panels of 32 rows x 128
// bytes (128-byte swizzle).  INT8: per stage, 64 rows x D bytes of codes
// (128-byte swizzle for D = 128, 64-byte for D = 64) and the 64 tokens'
// scales of the stage's KV head.
template <int D, bool kI8>
struct KvTiles {
  uint8_t k[kStagesOf<false>][D / 64][kPanelBytes];
  uint8_t v[kStagesOf<false>][D / 64][kPanelBytes];
};
template <int D>
struct KvTiles<D, true> {
  uint8_t k[kStagesOf<true>][kChunkOf<true> * D];
  uint8_t v[kStagesOf<true>][kChunkOf<true> * D];
  alignas(16) float ks[kStagesOf<true>][kChunkOf<true>];
  alignas(16) float vs[kStagesOf<true>][kChunkOf<true>];
};

// Byte offset of 16-byte piece `chunk` of row `row` in a TMA tile of D-byte
// int8 rows: 128-byte swizzle for D = 128 (the piece index XOR row % 8),
// 64-byte swizzle for D = 64 (XOR (row / 2) % 4).
template <int D>
__device__ __forceinline__ uint32_t i8_offset(int row, int chunk) {
  if constexpr (D == 128) return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
  else return static_cast<uint32_t>(row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4));
}

// INT8 codes as exact f16 values.  With x = codes XOR 0x80808080 (each byte
// biased to u = code + 128), the f16 with bits 0x64uu is 1024 + u, and
// subtracting 1152 (0x6480) leaves the code; both steps are exact.  One byte
// permute and one packed subtraction per pair.
constexpr uint32_t kF16Magic = 0x64646464u;
constexpr uint32_t kF16Bias = 0x64806480u;
// Bytes 0, 1 of x as an f16 pair (lo = byte 0).
__device__ __forceinline__ uint32_t i8_b01_f16x2(uint32_t x) {
  return sub_f16x2(__byte_perm(x, kF16Magic, 0x4140), kF16Bias);
}
// Bytes 2, 3 of x as an f16 pair (lo = byte 2).
__device__ __forceinline__ uint32_t i8_b23_f16x2(uint32_t x) {
  return sub_f16x2(__byte_perm(x, kF16Magic, 0x4342), kF16Bias);
}
// The f16 pairs (byte e of xa, byte e of xb) for e = 0, 1 (lo01) and
// e = 2, 3 (hi23): one interleaving permute per two pairs.
__device__ __forceinline__ void i8_cross_f16x2(uint32_t xa, uint32_t xb, uint32_t (&e01)[2],
                                               uint32_t (&e23)[2]) {
  const uint32_t t01 = __byte_perm(xa, xb, 0x5140);  // a0 b0 a1 b1
  const uint32_t t23 = __byte_perm(xa, xb, 0x7362);  // a2 b2 a3 b3
  e01[0] = i8_b01_f16x2(t01);
  e01[1] = i8_b23_f16x2(t01);
  e23[0] = i8_b01_f16x2(t23);
  e23[1] = i8_b23_f16x2(t23);
}

// Placed at a 1024-byte-aligned address (the 128-byte swizzle repeats every
// 1024 bytes and the panels must start on that boundary).
template <int D, int G, bool kI8 = false>
struct DecodeSmem : KvTiles<D, kI8> {
  static constexpr int kPanels = D / 64;
  static constexpr int kStages = kStagesOf<kI8>;
  alignas(16) __nv_bfloat16 q[kStages][G * D];
  // Mailbox from the consumer warps to the merger: each warp's state of a
  // finished piece.
  alignas(16) float mail_o[kConsumerWarps][G][D];
  float mail_m[kConsumerWarps][G];
  float mail_l[kConsumerWarps][G];
  StageInfo mail_info;
  StageInfo info[kStages];
  long long scan[kDecodeThreads / 32];
  long long start_base;  // chunk offset (per KV head) of the slice's first sequence
  long long end_base;    // ... and of the sequence of its last chunk
  unsigned long long gen;  // this launch's generation (counter tag)
  int start_seq;
  int end_seq;
  alignas(8) uint64_t full[kStages];
  alignas(8) uint64_t empty[kStages];
  alignas(8) uint64_t mail_full;  // the consumer warps' states are posted
  alignas(8) uint64_t mail_free;  // ... and have been taken by the merger
  // Merge jobs for the merge warp: a block holds at most two cut pieces, so
  // at most two merges and then an end marker; each slot is used once.
  StageInfo job[3];
  alignas(8) uint64_t job_full[3];
  int abort_flag;
  // The launch generation is published by the merge warp (off the critical
  // path) and read by the merger before its first count.
  alignas(8) uint64_t gen_full;
  // Table rows of the slice's sequences (when they fit).
  int slice_tab[kSliceTable];
  int slice_slot[kSliceSlots];  // fused store: their slots
  // Fused store: the new token's K and V rows of the stage's KV head, copied
  // in with the chunk that holds the token.
  alignas(16) __nv_bfloat16 knew[kStages][D];
  alignas(16) __nv_bfloat16 vnew[kStages][D];
  // Cascade decode: fold scratch of the merger and of the merge warp.
  FoldScratch<G> fold_merger;
  FoldScratch<G> fold_merge;
  // Cascade decode: pairs streamed whole whose private states wait for the
  // fold after the stream, (seq, kvh); whether each shares the prefix; and
  // the fold's two factors per row.
  int2 defer_pair[kDeferRows / G];
  int defer_unshared[kDeferRows / G];
  float2 defer_f[kDeferRows];
  alignas(8) uint64_t fold_bar;  // their outputs' bulk copies into the ring
};

template <int D, int G, bool kI8 = false>
constexpr size_t decode_smem_bytes() {
  return sizeof(DecodeSmem<D, G, kI8>) + 1024;  // slack for the 1024-byte alignment
}
// Two blocks per SM (228 KB of shared memory, 1 KB reserved per block) for
// the group sizes up to 8 (bf16) and 4 (INT8, whose ring is twice as deep).
static_assert(decode_smem_bytes<128, 8, false>() <= 113 * 1024, "bf16 decode: 2 blocks per SM");
static_assert(decode_smem_bytes<128, 4, true>() <= 113 * 1024, "INT8 decode: 2 blocks per SM");

// A context this kernel rejects: out of range, or (cascade decode) shorter
// than the shared prefix.
__device__ __forceinline__ bool bad_context(const DecodeArgs& a, int ctx, int max_ctx) {
  return ctx < 0 || ctx > max_ctx || ctx < a.shared_len;
}

// Chunks of each of sequence s's pairs: ceil((C - shared_len) / kChunk) (the
// tokens this kernel streams), and 1 for an empty private part or a rejected
// context (that chunk carries no tokens).
template <int kChunk>
__device__ __forceinline__ int ctx_chunks(const DecodeArgs& a, int ctx, int max_ctx) {
  const int priv = ctx - a.shared_len;
  return (bad_context(a, ctx, max_ctx) || priv <= 0) ? 1 : (priv + kChunk - 1) / kChunk;
}
template <int kChunk>
__device__ __forceinline__ int seq_chunks(const DecodeArgs& a, int s, int max_ctx) {
  return ctx_chunks<kChunk>(a, a.context_lens[s], max_ctx);
}

// The partial slot of the piece of a cut pair held by block cb2 (the pair
// spans blocks c_first .. c_last; only blocks with a non-empty slice hold a
// piece).
__device__ __forceinline__ int64_t piece_row(const StageInfo& inf, int cb2, int G) {
  const int sl = cb2 == inf.c_first ? inf.first_slot : 0;
  return (static_cast<int64_t>(cb2) * 2 + sl) * G;
}

// Cascade decode: whether sequence seq's leading table entries are row 0's
// (the shared blocks whose partial states are folded into its output).
// One warp, lanes compare entries in parallel; a sequence that does not
// share them is reported and gets a zero output.
__device__ __forceinline__ bool shares_prefix(const DecodeArgs& a, int seq, int lane) {
  const int nsb = a.shared_len / kBlockSize;
  const int32_t* t = a.block_tables + static_cast<int64_t>(seq) * a.max_blocks;
  bool same = true;
  for (int i = lane; i < nsb; i += 32) same &= __ldg(t + i) == __ldg(a.block_tables + i);
  const bool all = __all_sync(0xffffffffu, same);
  if (!all && lane == 0) report_error(a.err, kErrDeviceCheck, kSiteDecodeShared);
  return all;
}

// Cascade decode, lane = dimension: scales a head's private accumulator
// by fp and adds sum_u w_u o_u over the shared-prefix partial states (the
// factors fold_head left in f).
template <int D, int G>
__device__ __forceinline__ void fold_acc(const DecodeArgs& a, int seq, int kvh, int h,
                                         const FoldScratch<G>& f, float (&acc)[D / 32], int lane) {
  const float fp = f.fp[h];
#pragma unroll
  for (int i = 0; i < D / 32; ++i) acc[i] *= fp;
#pragma unroll 2
  for (int u = 0; u < a.shared_units; ++u) {
    const float w = f.w[h][u];
    if (w == 0.f) continue;  // the same for every lane
    const float* src = shared_o_at<D, G>(a, seq, kvh, h, u, lane);
#pragma unroll
    for (int i = 0; i < D / 32; ++i) acc[i] += w * __ldcg(src + i * 32);
  }
}

// Merge of all pieces of a cut pair by one warp (log-sum-exp):
//   M = max_j m_j, L = sum_j l_j 2^(m_j - M), out = sum_j o_j 2^(m_j - M) / L.
// Pieces go to lanes in batches of 32, so every load of a pass is
// independent of the others: lane j reads piece j's (m, l), the warp
// reduces M and L, and the weights w_j = 2^(m_j - M) / L are broadcast by
// shuffle while each lane accumulates its own dimensions.  In a cascade
// decode the shared-prefix partial states are folded in the same way before
// the division (f: this warp's fold scratch).
template <int D, int G>
__device__ void merge_pair(const DecodeArgs& a, const StageInfo& inf, long long T, long long nb,
                           int64_t row_base, int lane, FoldScratch<G>& f) {
  const int n = inf.c_last - inf.c_first + 1;  // blocks spanned (empty ones hold no piece)
  const bool unshared = a.shared_len > 0 && !shares_prefix(a, inf.seq, lane);
  const bool cascade = a.shared_len > 0 && !unshared;
  if (n <= 32) {
    // Lane j holds piece j's (m, l) for every head: one round of loads.
    const int cb2 = inf.c_first + lane;
    const bool has = lane < n && slice_begin(cb2 + 1, T, nb) > slice_begin(cb2, T, nb);
    const int64_t r = has ? piece_row(inf, cb2, G) : 0;
    float w[G], Mh[G], Lh[G];
    bool badh[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float m = has ? __ldcg(a.part_ml + (r + h) * 2) : -INFINITY;
      const float l = has ? __ldcg(a.part_ml + (r + h) * 2 + 1) : 0.f;
      float M = m;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      const float fw = (has && M != -INFINITY) ? fast_exp2(m - M) : 0.f;
      float L = l * fw;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
      badh[h] = __any_sync(0xffffffffu, l < 0.f) || unshared;
      Mh[h] = M;
      Lh[h] = L;
      w[h] = fw;
    }
    // Lane = dimension: every piece's rows of every head, loads independent
    // of each other (an empty block's weight is 0 and its slot is selected
    // away, never multiplied).
    float acc[G][D / 32];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int i = 0; i < D / 32; ++i) acc[h][i] = 0.f;
#pragma unroll 2
    for (int j = 0; j < n; ++j) {
      const int64_t rj = piece_row(inf, inf.c_first + j, G);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float wj = __shfl_sync(0xffffffffu, w[h], j);
#pragma unroll
        for (int i = 0; i < D / 32; ++i) {
          const float x = __ldcg(a.part_o + (rj + h) * D + i * 32 + lane);
          acc[h][i] += wj != 0.f ? wj * x : 0.f;
        }
      }
    }
    if (cascade) {
      grid_dependency_wait();  // the shared-prefix kernel's partials (see the kernel's start)
#pragma unroll
      for (int h = 0; h < G; ++h) fold_head<G>(a, inf.seq, inf.kvh, h, Mh[h], Lh[h], f, lane);
      __syncwarp();
#pragma unroll
      for (int h = 0; h < G; ++h) {
        fold_acc<D, G>(a, inf.seq, inf.kvh, h, f, acc[h], lane);
        Lh[h] = f.L[h];
        badh[h] |= f.bad[h] != 0;
      }
      __syncwarp();
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float inv = (Lh[h] > 0.f && !badh[h]) ? 1.f / Lh[h] : 0.f;
#pragma unroll
      for (int i = 0; i < D / 32; ++i)
        static_cast<__nv_bfloat16*>(a.out)[(row_base + h) * D + i * 32 + lane] =
            __float2bfloat16_rn(acc[h][i] * inv);
    }
    return;
  }
  for (int h = 0; h < G; ++h) {
    // pass 1: M and the bad flag, then L (lane j: piece j of a batch of 32)
    float M = -INFINITY;
    bool bad = false;
    for (int j0 = 0; j0 < n; j0 += 32) {
      const int cb2 = inf.c_first + j0 + lane;
      const bool has = j0 + lane < n && slice_begin(cb2 + 1, T, nb) > slice_begin(cb2, T, nb);
      const int64_t r = has ? piece_row(inf, cb2, G) + h : 0;
      M = fmaxf(M, has ? __ldcg(a.part_ml + r * 2) : -INFINITY);
      bad |= has && __ldcg(a.part_ml + r * 2 + 1) < 0.f;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    bad = __any_sync(0xffffffffu, bad) || unshared;
    float L = 0.f;
    for (int j0 = 0; j0 < n; j0 += 32) {
      const int cb2 = inf.c_first + j0 + lane;
      const bool has = j0 + lane < n && slice_begin(cb2 + 1, T, nb) > slice_begin(cb2, T, nb);
      const int64_t r = has ? piece_row(inf, cb2, G) + h : 0;
      if (has && M != -INFINITY)
        L += __ldcg(a.part_ml + r * 2 + 1) * fast_exp2(__ldcg(a.part_ml + r * 2) - M);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    // pass 2: out[d] = sum_j w_j o_j[d], weights broadcast by shuffle
    float acc[D / 32];
#pragma unroll
    for (int i = 0; i < D / 32; ++i) acc[i] = 0.f;
    for (int j0 = 0; j0 < n; j0 += 32) {
      const int cb2 = inf.c_first + j0 + lane;
      const bool has = j0 + lane < n && slice_begin(cb2 + 1, T, nb) > slice_begin(cb2, T, nb);
      const float w = (has && M != -INFINITY)
                          ? fast_exp2(__ldcg(a.part_ml + (piece_row(inf, cb2, G) + h) * 2) - M)
                          : 0.f;
      const int cnt = min(32, n - j0);
#pragma unroll 4
      for (int j = 0; j < cnt; ++j) {
        const float wj = __shfl_sync(0xffffffffu, w, j);
        const int64_t r = piece_row(inf, inf.c_first + j0 + j, G) + h;
#pragma unroll
        for (int i = 0; i < D / 32; ++i) {
          const float x = __ldcg(a.part_o + r * D + i * 32 + lane);
          acc[i] += wj != 0.f ? wj * x : 0.f;
        }
      }
    }
    if (cascade) {
      grid_dependency_wait();  // the shared-prefix kernel's partials (see the kernel's start)
      fold_head<G>(a, inf.seq, inf.kvh, h, M, L, f, lane);
      __syncwarp();
      fold_acc<D, G>(a, inf.seq, inf.kvh, h, f, acc, lane);
      L = f.L[h];
      bad |= f.bad[h] != 0;
      __syncwarp();
    }
    const float inv = (L > 0.f && !bad) ? 1.f / L : 0.f;
#pragma unroll
    for (int i = 0; i < D / 32; ++i)
      static_cast<__nv_bfloat16*>(a.out)[(row_base + h) * D + i * 32 + lane] =
          __float2bfloat16_rn(acc[i] * inv);
  }
}

// Two blocks per SM (measured best for the HBM-bound decode: more, shorter
// slices cost more cut contexts than the extra streams gain) need at most
// 65536 / (2 * 224) registers per thread.
template <int G>
constexpr int decode_max_regs() {
  return G <= 8 ? 128 : 255;
}

// kI8 = false: bf16 cache (kmap / vmap over the bf16 pools), 32-token chunks.
// kI8 = true: INT8 cache, 64-token chunks (kmap / vmap over the head-major
// int8 codes, box {D bytes, 64, 1}; the scales a.k_scales / a.v_scales come
// in by plain bulk copies).
template <int D, int G, bool kI8>
__global__ void __launch_bounds__(kDecodeThreads) __maxnreg__(decode_max_regs<G>())
decode_split_kernel(const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap, DecodeArgs a) {
  constexpr int kPanels = D / 64;
  constexpr int kStages = kStagesOf<kI8>;
  constexpr int kChunk = kChunkOf<kI8>;  // tokens per chunk
  constexpr uint32_t kChunkBytes = kChunk * D * (kI8 ? 1 : 2);
  constexpr uint32_t kQBytes = G * D * 2;
  constexpr int kWarps = kDecodeThreads / 32;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t sraw = smem_u32(smem_raw);
  DecodeSmem<D, G, kI8>& sm =
      *reinterpret_cast<DecodeSmem<D, G, kI8>*>(smem_raw + (((sraw + 1023u) & ~1023u) - sraw));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), kConsumerWarps);
    }
    mbar_init(smem_u32(&sm.mail_full), kConsumerWarps);
    mbar_init(smem_u32(&sm.mail_free), 1);
    mbar_init(smem_u32(&sm.gen_full), 1);
    for (int j = 0; j < 3; ++j) mbar_init(smem_u32(&sm.job_full[j]), 1);
    mbar_init(smem_u32(&sm.fold_bar), 1);
    sm.abort_flag = 0;
    sm.start_seq = -1;
    sm.start_base = 0;
    sm.end_seq = -1;
    sm.end_base = 0;
    fence_barrier_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
  }
  // Inputs may be written by the previous kernel in the stream: nothing
  // global is read before this point.  Cascade decode (shared_len > 0): the
  // previous kernel is the shared-prefix kernel, launched just before by the
  // same call, and only its partial states are this kernel's inputs from it
  // (everything else was written before it ran, and it waited for that
  // itself before letting this grid start).  So the private parts stream
  // while it runs, and the wait is taken just before those partials are
  // read (the folds below).
  if (a.shared_len == 0) grid_dependency_wait();
  grid_dependents_launch();

  // The producer stages its slice's table rows (and slots) once the plan
  // below is known: bring the tables to L2 while the plan reads the lengths
  // (one line per thread and step, the last element included; at most
  // kPrefetchLines lines per block).
  {
    auto prefetch_range = [&](const void* base, int64_t bytes) {
      const char* p = static_cast<const char*>(base);
      for (int64_t off = static_cast<int64_t>(threadIdx.x) * 128;
           off < bytes && off < kPrefetchLines * 128ll; off += kDecodeThreads * 128ll)
        prefetch_l2(p + off);
      if (threadIdx.x == 0 && bytes > 0) prefetch_l2(p + bytes - 4);
    };
    prefetch_range(a.block_tables, static_cast<int64_t>(a.num_seqs) * a.max_blocks * 4);
    if (a.slot_mapping != nullptr) prefetch_range(a.slot_mapping, static_cast<int64_t>(a.num_seqs) * 4);
  }

  const int max_ctx = a.max_blocks * kBlockSize;
  const int hkv = a.num_kv_heads;

  // ---- prefix sums of the pairs' costs (pair_gap + chunks) over the
  // sequences (whole block): thread t owns sequences [seg0, seg1).
  const int per = (a.num_seqs + kDecodeThreads - 1) / kDecodeThreads;
  const int seg0 = min(static_cast<int>(threadIdx.x) * per, a.num_seqs);
  const int seg1 = min(seg0 + per, a.num_seqs);
  const int gap = a.pair_gap;
  long long mine = 0;
  for (int s = seg0; s < seg1; ++s) mine += seq_chunks<kChunk>(a, s, max_ctx) + gap;
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
  const long long excl = before + incl - mine;  // cost per KV head before seg0
  const long long T = total * hkv;              // cost of all pairs
  const long long nb = gridDim.x;
  const long long ca = static_cast<long long>(blockIdx.x) * T / nb;        // slice begin
  const long long cb = (static_cast<long long>(blockIdx.x) + 1) * T / nb;  // slice end
  // The sequences holding the slice's first and last cost units.
  if (ca < cb && ca >= excl * hkv && ca < (excl + mine) * hkv) {
    long long p = excl;
    for (int s = seg0; s < seg1; ++s) {
      const int n = seq_chunks<kChunk>(a, s, max_ctx) + gap;
      if (ca < (p + n) * hkv) {
        sm.start_seq = s;
        sm.start_base = p;
        break;
      }
      p += n;
    }
  }
  if (ca < cb && cb - 1 >= excl * hkv && cb - 1 < (excl + mine) * hkv) {
    long long p = excl;
    for (int s = seg0; s < seg1; ++s) {
      const int n = seq_chunks<kChunk>(a, s, max_ctx) + gap;
      if (cb - 1 < (p + n) * hkv) {
        sm.end_seq = s;
        sm.end_base = p;
        break;
      }
      p += n;
    }
  }
  __syncthreads();

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    // The table rows of the slice's sequences, copied to shared memory by
    // the whole warp at once when they fit, so the stream never waits on a
    // table load.
    const int tab_seq0 = sm.start_seq;
    const bool tab_smem = tab_seq0 >= 0 && sm.end_seq >= tab_seq0 &&
                          static_cast<int64_t>(sm.end_seq - tab_seq0 + 1) * a.max_blocks <=
                              kSliceTable;
    if (tab_smem) {
      const int n = (sm.end_seq - tab_seq0 + 1) * a.max_blocks;
      const int32_t* src = a.block_tables + static_cast<int64_t>(tab_seq0) * a.max_blocks;
      for (int i = lane; i < n; i += 32) sm.slice_tab[i] = __ldg(src + i);
    }
    // Fused store: the slice's sequences' slots, likewise.
    const bool fused = a.slot_mapping != nullptr;
    const bool slot_smem = fused && tab_seq0 >= 0 && sm.end_seq >= tab_seq0 &&
                           sm.end_seq - tab_seq0 + 1 <= kSliceSlots;
    if (slot_smem)
      for (int i = lane; i <= sm.end_seq - tab_seq0; i += 32)
        sm.slice_slot[i] = __ldg(a.slot_mapping + tab_seq0 + i);
    __syncwarp();
    if (lane == 0) {
      // Posts go to the stages in turn (post c to stage c % kStages, phase
      // c / kStages); a claimed stage is always posted.
      int c = 0;  // stages posted so far
      bool aborted = false;
      // Claims the next ring stage; false when the wait for it expired, or
      // when the consumers gave up (checked every 8th post: a consumer that
      // stopped also stops freeing stages, so a later wait expires anyway).
      auto claim = [&](int st) -> bool {
        if (c >= kStages &&
            !mbar_wait(smem_u32(&sm.empty[st]), ((c / kStages) - 1) & 1, a.wait_limit_ns)) {
          report_error(a.err, kErrTimeout, kSiteDecodeWaitEmpty);
          atomicExch(&sm.abort_flag, 1);
          return false;
        }
        return (c & 7) != 0 || *reinterpret_cast<volatile int*>(&sm.abort_flag) == 0;
      };

      // Emits one piece of sequence pseq: the chunks [k0, k0 + n) of its pair
      // kvh (pnch chunks; the pair's cost units start at pstart, its chunk 0
      // sits at pfirst = pstart + pair_gap); false on abort.
      auto emit_piece = [&](int pseq, int pctx, bool pbad_ctx, int pnch, int kvh, int k0, int n,
                            long long pfirst, long long pstart, int slot) -> bool {
        const bool whole = k0 == 0 && n == pnch;
        // A cut pair's merge bookkeeping (below): computed once the piece's
        // first copies are on their way, since its divisions are slow and the
        // consumers read it only at the piece's end.
        int c_first = static_cast<int>(blockIdx.x), c_last = c_first, first_slot = 0;
        const int32_t* table = a.block_tables + static_cast<int64_t>(pseq) * a.max_blocks;
        const int32_t* stab = tab_smem ? sm.slice_tab + (pseq - tab_seq0) * a.max_blocks : table;
        for (int k = k0; k < k0 + n; ++k, ++c) {
          const int st = c % kStages;
          if (!claim(st)) return false;
          const int tok = a.shared_len + k * kChunk;
          const int n_valid = (pbad_ctx || pctx - tok <= 0) ? 0 : min(kChunk, pctx - tok);
          int id = 0;
          bool bad = pbad_ctx;
          if (n_valid > 0 && !bad) {
            id = stab[tok >> 8];
            if (id < 0 || id >= a.num_blocks) {
              bad = true;
              report_error(a.err, kErrDeviceCheck, kSiteDecodeBlock);
            }
          }
          const int valid = bad ? 0 : n_valid;
          const int slot_row = id * kBlockSize + (tok & (kBlockSize - 1));
          int store_slot = -1, store_row = 0;
          if (fused && k == pnch - 1) {
            // The pair's last chunk holds the new token (position ctx - 1).
            const int want = slot_smem ? sm.slice_slot[pseq - tab_seq0] : a.slot_mapping[pseq];
            if (valid > 0 && want == slot_row + valid - 1) {
              store_slot = want;
              store_row = valid - 1;
            } else if (want != -1) {
              report_error(a.err, kErrDeviceCheck, kSiteDecodeStoreSlot);
            }
          }
          // The copies go first: the barrier is told their bytes, and its
          // phase cannot complete before the arrive below, which publishes
          // the descriptor written after them.
          const uint32_t fb = smem_u32(&sm.full[st]);
          if (valid > 0) {
            constexpr uint32_t kRowBytes = D * 2;
            constexpr uint32_t kScaleBytes = kI8 ? kChunk * 4 : 0u;
            mbar_expect_tx(fb, 2 * kChunkBytes + 2 * kScaleBytes + (k == k0 ? kQBytes : 0u) +
                                   (store_slot >= 0 ? 2 * kRowBytes : 0u));
            if constexpr (kI8) {
              // Head-major INT8 blocks: the chunk's codes of this KV head are
              // one contiguous 64 x D tile (rows of (block, head) = id * Hkv
              // + kvh), and its 64 scales 256 contiguous bytes.
              const int bh = id * a.num_kv_heads + kvh;
              tma_load_3d(smem_u32(&sm.k[st][0]), &kmap, fb, 0, tok & (kBlockSize - 1), bh);
              tma_load_3d(smem_u32(&sm.v[st][0]), &vmap, fb, 0, tok & (kBlockSize - 1), bh);
              const int64_t srow =
                  static_cast<int64_t>(bh) * kBlockSize + (tok & (kBlockSize - 1));
              bulk_load(smem_u32(&sm.ks[st][0]), a.k_scales + srow, kScaleBytes, fb);
              bulk_load(smem_u32(&sm.vs[st][0]), a.v_scales + srow, kScaleBytes, fb);
            } else {
#pragma unroll
              for (int pn = 0; pn < kPanels; ++pn) {
                tma_load_3d(smem_u32(&sm.k[st][pn][0]), &kmap, fb, pn * 64, kvh, slot_row);
                tma_load_3d(smem_u32(&sm.v[st][pn][0]), &vmap, fb, pn * 64, kvh, slot_row);
              }
            }
            if (k == k0)
              bulk_load(smem_u32(&sm.q[st][0]),
                        static_cast<const __nv_bfloat16*>(a.q) +
                            static_cast<int64_t>(pseq) * a.q_row_stride +
                            static_cast<int64_t>(kvh) * G * D,
                        kQBytes, fb);
            if (store_slot >= 0) {
              bulk_load(smem_u32(&sm.knew[st][0]),
                        static_cast<const __nv_bfloat16*>(a.k_new) +
                            static_cast<int64_t>(pseq) * a.k_new_stride +
                            static_cast<int64_t>(kvh) * D,
                        kRowBytes, fb);
              bulk_load(smem_u32(&sm.vnew[st][0]),
                        static_cast<const __nv_bfloat16*>(a.v_new) +
                            static_cast<int64_t>(pseq) * a.v_new_stride +
                            static_cast<int64_t>(kvh) * D,
                        kRowBytes, fb);
            }
          }
          if (k == k0 && !whole) {
            // The blocks holding the pair's first and last chunk, and the
            // partial slot of its piece in the first: the cross-block merge's
            // bookkeeping, needed only for a cut pair (a whole pair's output
            // is written by the merger directly).  The piece is that block's
            // first (slot 0) when its slice holds no chunk of an earlier pair:
            // it starts at or after the pair's first cost unit (every unit
            // before that, back to the previous pair's gap, is a chunk of the
            // previous pair).
            c_first = block_of_chunk(pfirst, T, nb);
            c_last = block_of_chunk(pfirst + pnch - 1, T, nb);
            first_slot = slice_begin(c_first, T, nb) >= pstart ? 0 : 1;
          }
          // The descriptor is built in registers and stored once.
          StageInfo inf;
          inf.seq = pseq;
          inf.kvh = kvh;
          inf.slot = slot;
          inf.n_valid = valid;
          inf.flags = (bad ? kBad : 0) | (whole ? kSingle : 0) | (k == k0 ? kFirst : 0) |
                      (k == k0 + n - 1 ? kLast : 0);
          inf.c_first = c_first;
          inf.c_last = c_last;
          inf.first_slot = first_slot;
          inf.store_slot = store_slot;
          inf.store_row = store_row;
          inf.pad[0] = inf.pad[1] = 0;
          sm.info[st] = inf;
          mbar_arrive(fb);
        }
        return true;
      };

      int seq = sm.start_seq;
      if (ca < cb && seq >= 0) {
        // A piece cut at the slice's end is processed first: its pair's
        // cross-block merge then happens while the stream goes on, and the
        // block ends on a piece that needs none.
        long long stop = cb;
        if (sm.end_seq >= 0) {
          const int eseq = sm.end_seq;
          const long long ebase = sm.end_base * hkv;
          const int ectx = a.context_lens[eseq];
          const int enc = ctx_chunks<kChunk>(a, ectx, max_ctx);
          const int epl = enc + gap;  // the pair's cost
          const long long epair_begin = ebase + ((cb - 1 - ebase) / epl) * epl;
          const long long efirst = epair_begin + gap;
          if (epair_begin + epl > cb && epair_begin > ca) {
            // (none when the slice ends in the pair's gap)
            if (efirst < cb &&
                !emit_piece(eseq, ectx, bad_context(a, ectx, max_ctx), enc,
                            static_cast<int>((epair_begin - ebase) / epl), 0,
                            static_cast<int>(cb - efirst), efirst, epair_begin, 1))
              aborted = true;
            stop = epair_begin;
          }
        }
        long long base = sm.start_base * hkv;  // first cost unit of seq's pairs
        int ctx = a.context_lens[seq];
        bool ctx_bad = bad_context(a, ctx, max_ctx);
        int nch = ctx_chunks<kChunk>(a, ctx, max_ctx);
        int pl = nch + gap;  // a pair's cost
        if (ctx_bad && base >= ca) report_error(a.err, kErrDeviceCheck, kSiteDecodeContext);
        long long pos = ca;
        // The pair of unit pos, and the first of its chunks at or after pos:
        // divided out once, then carried along (every piece after the first
        // starts a pair).
        int kvh = static_cast<int>((pos - base) / pl);
        int k0 = max(0, static_cast<int>(pos - base) - kvh * pl - gap);
        int piece = 0;
        while (pos < stop && !aborted) {
          const long long pair_start = base + static_cast<long long>(kvh) * pl;
          const long long pair_end = pair_start + pl;
          const long long piece_end = pair_end < stop ? pair_end : stop;
          // Its chunks in [pos, piece_end): none when the slice stops in the
          // pair's gap.
          const int n = static_cast<int>(piece_end - (pair_start + gap)) - k0;
          if (n > 0) {
            if (!emit_piece(seq, ctx, ctx_bad, nch, kvh, k0, n, pair_start + gap, pair_start,
                            piece == 0 ? 0 : 1)) {
              aborted = true;
              break;
            }
            ++piece;
          }
          pos = piece_end;
          k0 = 0;
          if (pos == pair_end) {
            if (kvh + 1 < hkv) {
              ++kvh;
            } else if (pos < stop) {  // next sequence
              ++seq;
              base = pair_end;
              kvh = 0;
              ctx = a.context_lens[seq];
              ctx_bad = bad_context(a, ctx, max_ctx);
              nch = ctx_chunks<kChunk>(a, ctx, max_ctx);
              pl = nch + gap;
              if (ctx_bad) report_error(a.err, kErrDeviceCheck, kSiteDecodeContext);
            }
          }
        }
      }
      if (!aborted) {  // end marker
        const int st = c % kStages;
        if (claim(st)) {
          sm.info[st].flags = kEnd;
          mbar_arrive(smem_u32(&sm.full[st]));
          ++c;
        }
      }
      // Every copy issued must land before the block may exit, whether or
      // not the consumers gave up on it (after a normal run these waits
      // return at once: the consumers have already seen each phase).  The
      // last post of stage s is its newest phase: once that one is complete,
      // every copy ever issued into the stage has landed.
      for (int s = 0; s < kStages && s < c; ++s) {
        const int last = s + ((c - 1 - s) / kStages) * kStages;
        mbar_wait(smem_u32(&sm.full[s]), (last / kStages) & 1, kDrainLimitNs);
      }
    }
  } else if (warp < kConsumerWarps) {
    // ------------------------------------------------------------ consumers
    constexpr int NT = (G + 7) / 8;  // n-tiles of 8 query heads
    constexpr int KS = D / 16;       // k-steps of S^T = K q^T; m-tiles of O^T
    const int g = lane >> 2;         // fragment row group
    const int cq = lane & 3;         // fragment column pair
    const int li = lane >> 3, lr = lane & 7;  // ldmatrix: matrix and row this lane addresses
    const float qscale = a.scale * 1.4426950408889634f;

    uint32_t qb[KS][NT][2];  // q^T operand fragments: dims ks*16 + 2cq (+8), head nt*8 + g
    float o[KS][NT][4];      // O^T: dims md*16 + g (+8), heads nt*8 + 2cq (+1)
    float m_run[NT][2];      // running max of heads nt*8 + 2cq + j (log2 domain)
    float l_run[NT][2];      // this lane's share of their running sums
    bool piece_bad = false;
    // INT8 (f16 operands): q of head h is scaled by a power of two so that
    // max |q| lies in [1/2, 1) (exact, then rounded to f16); qmul undoes it for
    // the scores of heads nt*8 + 2cq + j.  P is multiplied by vscale_t /
    // vs_ref, vs_ref the running maximum of the piece's V scales (so P <= 1
    // in f16), and the accumulator is scaled by vs_ref when posted.
    float qmul[NT][2];
    float vs_ref = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) qmul[nt][0] = qmul[nt][1] = 0.f;
#pragma unroll
    for (int md = 0; md < KS; ++md)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) qb[md][nt][0] = qb[md][nt][1] = 0u;

    int posts = 0;  // pieces (and the final end marker) posted to the merger
    // Claims the mailbox (bounded wait for the merger to take the last post).
    auto claim_mail = [&](int k) -> bool {
      const bool ok = k < 1 || mbar_wait(smem_u32(&sm.mail_free), (k - 1) & 1, a.wait_limit_ns);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) {
          report_error(a.err, kErrTimeout, kSiteDecodeWaitMerge);
          atomicExch(&sm.abort_flag, 1);
        }
        return false;
      }
      return true;
    };
    bool mail_ok = true;
    for (int c = 0;; ++c) {
      const int st = c % kStages;
      // Every exit decision is taken warp-uniformly (the shuffles and the
      // warp-wide matrix instructions below need the full warp).
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
        piece_bad = false;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            m_run[nt][j] = -INFINITY;
            l_run[nt][j] = 0.f;
          }
#pragma unroll
        for (int md = 0; md < KS; ++md)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[md][nt][e] = 0.f;
        if (inf.n_valid > 0) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const int h = nt * 8 + g;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
              // The k index of the MMA runs over head dimensions: bf16 keys
              // use them in order; INT8 keys are read four bytes (four
              // dimensions) per lane, so logical k 2cq, 2cq+1 | 2cq+8, 2cq+9
              // of step ks stand for dimensions 16 ks + 4 cq + 0, 1 | 2, 3.
              const __nv_bfloat16* qr = kI8 ? &sm.q[st][h * D + ks * 16 + 4 * cq]
                                            : &sm.q[st][h * D + ks * 16 + 2 * cq];
              qb[ks][nt][0] = h < G ? *reinterpret_cast<const uint32_t*>(qr) : 0u;
              qb[ks][nt][1] = h < G ? *reinterpret_cast<const uint32_t*>(qr + (kI8 ? 2 : 8)) : 0u;
            }
            if constexpr (kI8) {
              // max |q| of head h over the four lanes of row group g
              float amax = 0.f;
#pragma unroll
              for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                for (int k2 = 0; k2 < 2; ++k2)
                  amax = fmax3(amax, fabsf(bf16_lo(qb[ks][nt][k2])), fabsf(bf16_hi(qb[ks][nt][k2])));
              amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
              amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
              // 2^-(E+1) and 2^(E+1) for amax = m 2^E, 1 <= m < 2
              const uint32_t eb = min((__float_as_uint(amax) >> 23) & 0xFFu, 252u);
              const float down = amax > 0.f ? __uint_as_float((253u - eb) << 23) : 1.f;
              const float up = amax > 0.f ? __uint_as_float((eb + 1u) << 23) : 0.f;
#pragma unroll
              for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                for (int k2 = 0; k2 < 2; ++k2)
                  qb[ks][nt][k2] = pack_f16x2(bf16_lo(qb[ks][nt][k2]) * down,
                                              bf16_hi(qb[ks][nt][k2]) * down);
#pragma unroll
              for (int j = 0; j < 2; ++j)
                qmul[nt][j] = __shfl_sync(0xffffffffu, up, (2 * cq + j) * 4);
            }
          }
        }
        vs_ref = 0.f;
      }
      piece_bad |= (inf.flags & kBad) != 0;
      const int valid = inf.n_valid;
      bool zeroed = false;
      // Who computes what.  bf16: warp c % 4 takes the whole 32-token chunk
      // c in one step of two m-tiles.  INT8: every warp takes its 16 of the
      // chunk's 64 tokens in one step of one m-tile, so that a stage is done
      // (and freed for the next copy) four times sooner; the four states
      // meet in the merger as for bf16.  Per-token work is the same.
      constexpr int MT = kI8 ? 1 : 2;  // m-tiles (16 tokens) per step
      constexpr int kStep = 16 * MT;
      const int hoff = kI8 ? warp * kStep : 0;
      if ((kI8 || (c % kConsumerWarps) == warp) && valid > hoff) {
        {
          const int hvalid = min(valid - hoff, kStep);  // tokens of this step
          // INT8: the K and V scales of this lane's four tokens (mt * 16 +
          // hf * 8 + g); read for tokens past the context too, but always
          // selected away there (pool contents may be anything).
          float ksc[MT][2], vsc[MT][2];
          if constexpr (kI8) {
  #pragma unroll
            for (int mt = 0; mt < MT; ++mt)
  #pragma unroll
              for (int hf = 0; hf < 2; ++hf) {
                const int tok = mt * 16 + hf * 8 + g;
                ksc[mt][hf] = sm.ks[st][hoff + tok];
                vsc[mt][hf] = sm.vs[st][hoff + tok];
              }
          } else {
            if (hvalid < kDecodeChunk) {
              // V rows past the context: zero them (pool contents may be
              // anything, and 0 x NaN would poison the product).
              for (int i = lane; i < (kStep - hvalid) * 8 * kPanels; i += 32) {
                const int pn = i % kPanels;
                const int rest = i / kPanels;
                *reinterpret_cast<uint4*>(&sm.v[st][pn][(hvalid + rest / 8) * 128 + (rest % 8) * 16]) =
                    make_uint4(0u, 0u, 0u, 0u);
              }
              __syncwarp();
              zeroed = true;
            }
            if (inf.store_slot >= 0) {
              // Fused store: the new token's K and V rows of this KV head replace
              // the pool rows loaded for its position, and are written to the
              // cache slot (each pair stores its own head; one 16-byte piece per
              // lane).
              constexpr int kPieces = D / 8;
              if (lane < 2 * kPieces) {
                const bool is_v = lane >= kPieces;
                const int ci = is_v ? lane - kPieces : lane;
                const uint4 x =
                    *reinterpret_cast<const uint4*>((is_v ? sm.vnew[st] : sm.knew[st]) + ci * 8);
                uint8_t* tile = is_v ? &sm.v[st][ci / 8][0] : &sm.k[st][ci / 8][0];
                *reinterpret_cast<uint4*>(tile + sw128_offset(inf.store_row, ci % 8)) = x;
                __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(is_v ? a.v_cache : a.k_cache) +
                                     static_cast<int64_t>(inf.store_slot) * a.num_kv_heads * D +
                                     static_cast<int64_t>(inf.kvh) * D + ci * 8;
                *reinterpret_cast<uint4*>(dst) = x;
              }
              __syncwarp();
              zeroed = true;
            }
          }
          // ---- S^T = K q^T: MT m-tiles of 16 tokens x NT n-tiles of 8 heads
          float sc[MT][NT][4];
  #pragma unroll
          for (int mt = 0; mt < MT; ++mt)
  #pragma unroll
            for (int nt = 0; nt < NT; ++nt)
  #pragma unroll
              for (int e = 0; e < 4; ++e) sc[mt][nt][e] = 0.f;
          if constexpr (kI8) {
            // Codes converted to bf16 exactly in registers: lane (g, cq) reads
            // four bytes (dimensions 16 ks + 4 cq .. + 3) of token rows g and
            // g + 8 of each m-tile (conflict-free under the swizzle).
            const uint8_t* k8 = sm.k[st] + hoff * D;
  #pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
  #pragma unroll
              for (int mt = 0; mt < MT; ++mt) {
                const int r0 = mt * 16 + g;
                const uint32_t w0 =
                    *reinterpret_cast<const uint32_t*>(k8 + i8_offset<D>(r0, ks) + 4 * cq) ^
                    0x80808080u;
                const uint32_t w1 =
                    *reinterpret_cast<const uint32_t*>(k8 + i8_offset<D>(r0 + 8, ks) + 4 * cq) ^
                    0x80808080u;
                uint32_t af[4];
                af[0] = i8_b01_f16x2(w0);
                af[2] = i8_b23_f16x2(w0);
                af[1] = i8_b01_f16x2(w1);
                af[3] = i8_b23_f16x2(w1);
  #pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                  mma_16816_f16(sc[mt][nt], af, qb[ks][nt][0], qb[ks][nt][1]);
              }
            }
          } else {
            const uint32_t kb = smem_u32(&sm.k[st][0][0]);
  #pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
  #pragma unroll
              for (int mt = 0; mt < MT; ++mt) {
                uint32_t af[4];
                ldsm_x4(kb + (ks >> 2) * kPanelBytes +
                            sw128_offset(mt * 16 + (li & 1) * 8 + lr, (ks & 3) * 2 + (li >> 1)),
                        af);
  #pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                  mma_16816(sc[mt][nt], af, qb[ks][nt][0], qb[ks][nt][1]);
              }
            }
          }
          // INT8: the running maximum of the piece's V scales (valid tokens;
          // the eight row groups hold the chunk's tokens).  When it grows the
          // accumulator, kept in units of it, is rescaled with the softmax's
          // alpha below.
          float vfix = 1.f, inv_vs = 0.f;
          if constexpr (kI8) {
            float cm = 0.f;
  #pragma unroll
            for (int mt = 0; mt < MT; ++mt)
  #pragma unroll
              for (int hf = 0; hf < 2; ++hf)
                if (mt * 16 + hf * 8 + g < hvalid) cm = fmaxf(cm, vsc[mt][hf]);
            cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 4));
            cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 8));
            cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 16));
            if (cm > vs_ref) {
              vfix = vs_ref / cm;
              vs_ref = cm;
            }
            inv_vs = vs_ref > 0.f ? 1.f / vs_ref : 0.f;
          }
          // ---- online softmax per head (a head's 16 MT scores sit in the lanes
          // with the same cq: two per m-tile in each of the 8 row groups)
          float alpha[NT][2];
  #pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
  #pragma unroll
            for (int j = 0; j < 2; ++j) {
              float mx = -INFINITY;
  #pragma unroll
              for (int mt = 0; mt < MT; ++mt)
  #pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                  const int tok = mt * 16 + hf * 8 + g;
                  const float sx = kI8 ? qscale * ksc[mt][hf] * qmul[nt][j] : qscale;
                  const float x = tok < hvalid ? sc[mt][nt][hf * 2 + j] * sx : -INFINITY;
                  sc[mt][nt][hf * 2 + j] = x;
                  mx = fmaxf(mx, x);
                }
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
              const float m_new = fmaxf(m_run[nt][j], mx);  // finite: hvalid > 0
              alpha[nt][j] = fast_exp2(m_run[nt][j] - m_new);
              m_run[nt][j] = m_new;
              float ls = 0.f;
  #pragma unroll
              for (int mt = 0; mt < MT; ++mt)
  #pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                  const float pv = fast_exp2(sc[mt][nt][hf * 2 + j] - m_new);
                  ls += pv;
                  // INT8: P V = vs_ref sum_t (p_t vscale_t / vs_ref) code_t,
                  // with p_t vscale_t / vs_ref <= 1 in f16; the sum keeps p_t.
                  const int tok = mt * 16 + hf * 8 + g;
                  sc[mt][nt][hf * 2 + j] =
                      kI8 ? (tok < hvalid ? pv * (vsc[mt][hf] * inv_vs) : 0.f) : pv;
                }
              l_run[nt][j] = l_run[nt][j] * alpha[nt][j] + ls;
              if constexpr (kI8) alpha[nt][j] *= vfix;
            }
          }
  #pragma unroll
          for (int md = 0; md < KS; ++md)
  #pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              o[md][nt][0] *= alpha[nt][0];
              o[md][nt][1] *= alpha[nt][1];
              o[md][nt][2] *= alpha[nt][0];
              o[md][nt][3] *= alpha[nt][1];
            }
          // ---- P^T operand fragments: the S^T accumulator of tokens
          // mt*16 + (0..7 | 8..15) is an 8x8 16-bit matrix per lane pair of
          // columns; its transpose is the operand layout (bf16, or f16 for
          // INT8).
          uint32_t pb[MT][NT][2];
  #pragma unroll
          for (int mt = 0; mt < MT; ++mt)
  #pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              pb[mt][nt][0] = movmatrix_trans(kI8 ? pack_f16x2(sc[mt][nt][0], sc[mt][nt][1])
                                                  : pack_bf16x2(sc[mt][nt][0], sc[mt][nt][1]));
              pb[mt][nt][1] = movmatrix_trans(kI8 ? pack_f16x2(sc[mt][nt][2], sc[mt][nt][3])
                                                  : pack_bf16x2(sc[mt][nt][2], sc[mt][nt][3]));
            }
          // ---- O^T += V^T P^T: D/16 m-tiles of dimensions, MT k-steps of 16 tokens
          if constexpr (kI8) {
            // Lane (g, cq) reads four bytes (dimensions 4 (g + 8 p) .. + 3) of
            // token rows 2 cq, 2 cq + 1, 2 cq + 8, 2 cq + 9 of the k-step and
            // pairs the tokens per dimension; dimension 4 (g + 8 p) + e is row
            // g + 8 (e & 1) of m-tile 2 p + (e >> 1) (the output rows are put
            // back in order when the state is posted).
            const uint8_t* v8 = sm.v[st] + hoff * D;
  #pragma unroll
            for (int kt = 0; kt < MT; ++kt) {
              const int t0 = kt * 16 + 2 * cq;
  #pragma unroll
              for (int p = 0; p < D / 32; ++p) {
                const int ch = (g >> 2) + 2 * p;
                const int wo = 4 * (g & 3);
                const uint32_t x0 =
                    *reinterpret_cast<const uint32_t*>(v8 + i8_offset<D>(t0, ch) + wo) ^ 0x80808080u;
                const uint32_t x1 =
                    *reinterpret_cast<const uint32_t*>(v8 + i8_offset<D>(t0 + 1, ch) + wo) ^
                    0x80808080u;
                const uint32_t x2 =
                    *reinterpret_cast<const uint32_t*>(v8 + i8_offset<D>(t0 + 8, ch) + wo) ^
                    0x80808080u;
                const uint32_t x3 =
                    *reinterpret_cast<const uint32_t*>(v8 + i8_offset<D>(t0 + 9, ch) + wo) ^
                    0x80808080u;
                // Token pairs (t0, t0 + 1) and (t0 + 8, t0 + 9) per byte e.
                uint32_t lo01[2], lo23[2], hi01[2], hi23[2];
                i8_cross_f16x2(x0, x1, lo01, lo23);
                i8_cross_f16x2(x2, x3, hi01, hi23);
                const uint32_t af0[4] = {lo01[0], lo01[1], hi01[0], hi01[1]};  // e = 0, 1
                const uint32_t af1[4] = {lo23[0], lo23[1], hi23[0], hi23[1]};  // e = 2, 3
  #pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                  mma_16816_f16(o[2 * p][nt], af0, pb[kt][nt][0], pb[kt][nt][1]);
                  mma_16816_f16(o[2 * p + 1][nt], af1, pb[kt][nt][0], pb[kt][nt][1]);
                }
              }
            }
          } else {
            const uint32_t vb = smem_u32(&sm.v[st][0][0]);
  #pragma unroll
            for (int kt = 0; kt < MT; ++kt) {
  #pragma unroll
              for (int md = 0; md < KS; ++md) {
                uint32_t af[4];
                ldsm_x4_trans(vb + (md >> 2) * kPanelBytes +
                                  sw128_offset(kt * 16 + (li >> 1) * 8 + lr, (md & 3) * 2 + (li & 1)),
                              af);
  #pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                  mma_16816(o[md][nt], af, pb[kt][nt][0], pb[kt][nt][1]);
              }
            }
          }
        }
      }
      if (zeroed) fence_proxy_async_smem();  // generic writes before the next TMA into the stage
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.empty[st]));

      if (inf.flags & kLast) {
        // ---- post this warp's state of the piece (max, sum, unnormalised
        // output) to the merger and go on with the next chunk at once.
        const int k = posts++;
        if (!claim_mail(k)) {
          mail_ok = false;
          break;
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            float x = l_run[nt][j];  // a head's sum: this lane's share over the 8 row groups
            x += __shfl_xor_sync(0xffffffffu, x, 4);
            x += __shfl_xor_sync(0xffffffffu, x, 8);
            x += __shfl_xor_sync(0xffffffffu, x, 16);
            const int h = nt * 8 + 2 * cq + j;
            if (g == 0 && h < G) {
              sm.mail_m[warp][h] = m_run[nt][j];
              sm.mail_l[warp][h] = x;
            }
          }
#pragma unroll
        for (int md = 0; md < KS; ++md)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int h = nt * 8 + 2 * cq + (e & 1);
              // Dimension of accumulator row g + 8 (e >> 1) of m-tile md.
              const int dim = kI8 ? 4 * (g + 8 * (md >> 1)) + (md & 1) * 2 + (e >> 1)
                                  : md * 16 + g + (e >> 1) * 8;
              if (h < G) sm.mail_o[warp][h][dim] = kI8 ? o[md][nt][e] * vs_ref : o[md][nt][e];
            }
        if (warp == 0 && lane == 0) {  // every warp saw the same descriptors
          StageInfo post = inf;
          post.flags = (inf.flags & ~kBad) | (piece_bad ? kBad : 0);
          sm.mail_info = post;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.mail_full));
      }
    }
    // End marker for the merger.
    if (mail_ok) {
      const int k = posts++;
      if (claim_mail(k)) {
        if (warp == 0 && lane == 0) sm.mail_info.flags = kEnd;
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.mail_full));
      }
    }
  } else if (warp == kMergerWarp) {
    // ------------------------------------------------------------ merger
    // Takes the consumer warps' posts in order and combines their four
    // states of the piece (log-sum-exp, as below).  A whole pair's output is
    // written here; a cut piece's state goes to one of the block's two
    // partial slots, is counted on the pair's arrival counter, and the post
    // that brings the count to the pair's number of pieces merges all of
    // them:
    //   M = max_j m_j, L = sum_j l_j 2^(m_j - M), out = sum_j o_j 2^(m_j - M) / L.
    int n_jobs = 0;  // merges handed to the merge warp
    int n_defer = 0;  // cascade decode: whole pairs set aside for the fold after the stream
    bool ended = false;  // the consumers' end marker came (the ring is idle)
    bool gen_seen = false;  // lane 0: the launch generation has been published
    for (int k = 0;; ++k) {
      const bool got = mbar_wait_sleepy(smem_u32(&sm.mail_full), k & 1, a.wait_limit_ns, 200);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) {
          report_error(a.err, kErrTimeout, kSiteDecodeWaitMerge);
          atomicExch(&sm.abort_flag, 1);
        }
        break;
      }
      const StageInfo inf = sm.mail_info;
      if (inf.flags & kEnd) {
        ended = true;
        break;
      }
      const bool bad = (inf.flags & kBad) != 0;
      const bool single = (inf.flags & kSingle) != 0;
      const int64_t row_base = static_cast<int64_t>(inf.seq) * a.num_q_heads + inf.kvh * G;
      const int64_t prow = (static_cast<int64_t>(blockIdx.x) * 2 + inf.slot) * G;
      // Per head: M = max over the four warps, weights 2^(m_w - M), L.
      // Lane h (< G) computes head h's and the others read them by shuffle.
      float hw[kConsumerWarps], hM = -INFINITY, hL = 0.f;
      {
        const int h = lane < G ? lane : 0;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) hM = fmaxf(hM, sm.mail_m[w][h]);
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          hw[w] = hM == -INFINITY ? 0.f : fast_exp2(sm.mail_m[w][h] - hM);
          hL += sm.mail_l[w][h] * hw[w];
        }
      }
      // Each lane combines 4 consecutive dimensions per step (float4).
      constexpr int kVec = G * D / 4;                   // float4 groups of the piece
      constexpr int kPer = (kVec + 31) / 32;            // per lane
      float4 res[kPer];
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int v = lane + 32 * i;
        const int hh = (v * 4) / D;
        float wv[kConsumerWarps];
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) wv[w] = __shfl_sync(0xffffffffu, hw[w], hh & 31);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (v < kVec) {
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) {
            const float4 x = reinterpret_cast<const float4*>(&sm.mail_o[w][0][0])[v];
            acc.x += wv[w] * x.x;
            acc.y += wv[w] * x.y;
            acc.z += wv[w] * x.z;
            acc.w += wv[w] * x.w;
          }
        }
        res[i] = acc;
      }
      // The mailbox has been read: let the consumers post again.
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.mail_free));
      // Cascade decode: a whole pair's private state is set aside while the
      // list has room (the shared-prefix kernel may still be running; the
      // fold comes after the stream, fold_deferred) ...
      if (!kI8 && single && a.shared_len > 0 && !bad && a.shared_units == 1 &&
          n_defer < kDeferRows / G) {
        const int64_t prow0 = static_cast<int64_t>(inf.kvh) * a.shared_rows_pad +
                              static_cast<int64_t>(inf.seq) * G;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          const int v = lane + 32 * i;
          if (v >= kVec) continue;
          const int hh = (v * 4) / D;
          const int d = v * 4 - hh * D;
          *reinterpret_cast<float4*>(a.private_o + (prow0 + hh) * D + d) = res[i];
        }
        if (lane < G)
          *reinterpret_cast<float2*>(a.private_ml + (prow0 + lane) * 2) = make_float2(hM, hL);
        if (lane == 0) sm.defer_pair[n_defer] = make_int2(inf.seq, inf.kvh);
        ++n_defer;
        continue;
      }
      // ... else it is merged here with the shared-prefix partial states
      // (log-sum-exp), before the division.
      const bool unshared = single && a.shared_len > 0 && !shares_prefix(a, inf.seq, lane);
      const bool fold = single && a.shared_len > 0 && !bad && !unshared;
      FoldScratch<G>& fs = sm.fold_merger;
      if (fold) {
        grid_dependency_wait();  // the shared-prefix kernel's partials (see the kernel's start)
#pragma unroll 1
        for (int h = 0; h < G; ++h)
          fold_head<G>(a, inf.seq, inf.kvh, h, __shfl_sync(0xffffffffu, hM, h),
                       __shfl_sync(0xffffffffu, hL, h), fs, lane);
        __syncwarp();
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          const int v = lane + 32 * i;
          if (v >= kVec) continue;
          const int hh = (v * 4) / D;
          const int d = v * 4 - hh * D;
          const float fp = fs.fp[hh];
          float4 acc = make_float4(res[i].x * fp, res[i].y * fp, res[i].z * fp, res[i].w * fp);
#pragma unroll 4
          for (int u = 0; u < a.shared_units; ++u) {
            const float w = fs.w[hh][u];
            if (w == 0.f) continue;
            const float4 x =
                __ldcg(reinterpret_cast<const float4*>(shared_o_at<D, G>(a, inf.seq, inf.kvh, hh, u, d)));
            acc.x += w * x.x;
            acc.y += w * x.y;
            acc.z += w * x.z;
            acc.w += w * x.w;
          }
          res[i] = acc;
        }
      }
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int v = lane + 32 * i;
        const int hh = (v * 4) / D;
        float L = __shfl_sync(0xffffffffu, hL, hh & 31);
        const float M = __shfl_sync(0xffffffffu, hM, hh & 31);
        if (v >= kVec) continue;
        const int d = v * 4 - hh * D;
        bool bad_row = bad || unshared;
        if (fold) {
          L = fs.L[hh];
          bad_row = fs.bad[hh] != 0;
        }
        if (single) {
          const float inv = (L > 0.f && !bad_row) ? 1.f / L : 0.f;
          uint2 packed;
          packed.x = pack_bf16x2(res[i].x * inv, res[i].y * inv);
          packed.y = pack_bf16x2(res[i].z * inv, res[i].w * inv);
          *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + (row_base + hh) * D + d) =
              packed;
        } else {
          *reinterpret_cast<float4*>(a.part_o + (prow + hh) * D + d) = res[i];
          if (d == 0) {
            a.part_ml[(prow + hh) * 2 + 0] = M;
            a.part_ml[(prow + hh) * 2 + 1] = bad ? -1.f : L;
          }
        }
      }
      if (single) continue;
      __syncwarp();  // the partials of every lane precede lane 0's releasing add
      int last = 0;
      if (lane == 0) {
        int pieces = 0;  // blocks with a non-empty slice in [c_first, c_last]
        for (int cb2 = inf.c_first; cb2 <= inf.c_last; ++cb2)
          pieces += slice_begin(cb2 + 1, T, nb) > slice_begin(cb2, T, nb);
        unsigned long long* cnt =
            a.counters + kPairCounterOffset + static_cast<int64_t>(inf.seq) * hkv + inf.kvh;
        if (!gen_seen) {
          // The merge warp publishes the launch generation at its start.
          gen_seen = mbar_wait(smem_u32(&sm.gen_full), 0, kDrainLimitNs);
          if (!gen_seen) report_error(a.err, kErrTimeout, kSiteDecodeWaitMerge);
        }
        last = gen_seen && static_cast<int>(tagged_increment(cnt, sm.gen)) == pieces;
      }
      if (__shfl_sync(0xffffffffu, last, 0) && n_jobs < 2) {
        if (lane == 0) {
          sm.job[n_jobs] = inf;
          mbar_arrive(smem_u32(&sm.job_full[n_jobs]));
        }
        ++n_jobs;
      }
    }
    if (lane == 0) {  // end marker for the merge warp
      sm.job[n_jobs].flags = kEnd;
      mbar_arrive(smem_u32(&sm.job_full[n_jobs]));
    }
    if constexpr (!kI8) {
      static_assert(sizeof(KvTiles<D, false>) >= 2 * kDeferRows * D * sizeof(float),
                    "the ring holds both outputs of kDeferRows rows");
      if (n_defer > 0 && ended &&
          !__shfl_sync(0xffffffffu, *reinterpret_cast<volatile int*>(&sm.abort_flag), 0)) {
        __syncwarp();  // lane 0's list entries
        fold_deferred<D, G>(a, sm.defer_pair, sm.defer_unshared, sm.defer_f, n_defer,
                            reinterpret_cast<float*>(&sm.k[0][0][0]), smem_u32(&sm.fold_bar),
                            lane);
      }
    }
  } else if (warp == kMergeWarp) {
    // ------------------------------------------------------------ merge warp
    // Cut contexts whose last piece this block counted: merge all their
    // pieces from the partial slots.  Off the consumers' path: the partial
    // reads are L2 round trips, slow while the streams load the memory system.
    if (lane == 0) {
      // Launch generation: epoch + 1.  Each block reads the epoch, then
      // counts itself on the start counter; the block that completes the
      // count (so every block has read the epoch) advances the epoch for the
      // next launch, which cannot start before this one ends.  Done here,
      // off the stream's path; the merger waits for it before its first
      // count.
      const unsigned long long gen = (__ldcg(a.counters) + 1) & kGenMask;
      sm.gen = gen;
      mbar_arrive(smem_u32(&sm.gen_full));
      if (tagged_increment(a.counters + 1, gen) == gridDim.x)
        atomicExch(a.counters, gen);  // epoch := generation
    }
    for (int j = 0; j < 3; ++j) {
      const bool got = mbar_wait_sleepy(smem_u32(&sm.job_full[j]), 0, a.wait_limit_ns, 500);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) report_error(a.err, kErrTimeout, kSiteDecodeWaitMerge);
        break;
      }
      const StageInfo inf = sm.job[j];
      if (inf.flags & kEnd) break;
      fence_acq_rel_gpu();  // every lane: the other pieces' partials are visible
      const int64_t row_base = static_cast<int64_t>(inf.seq) * a.num_q_heads + inf.kvh * G;
      merge_pair<D, G>(a, inf, T, nb, row_base, lane, sm.fold_merge);
    }
  }
}

template <int D, int G, bool kI8>
int ctas_per_sm() {
  static int per_sm = 0;
  if (per_sm == 0) {
    const size_t smem = decode_smem_bytes<D, G, kI8>();
    auto kern = decode_split_kernel<D, G, kI8>;
    int n = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kDecodeThreads, smem) !=
            cudaSuccess) {
      cudaGetLastError();
      return 1;
    }
    per_sm = n > 0 ? n : 1;
  }
  return per_sm;
}

template <int D, bool kI8>
int ctas_per_sm_d(int group) {
  switch (group) {
    case 1: return ctas_per_sm<D, 1, kI8>();
    case 2: return ctas_per_sm<D, 2, kI8>();
    case 4: return ctas_per_sm<D, 4, kI8>();
    case 8: return ctas_per_sm<D, 8, kI8>();
    default: return ctas_per_sm<D, 16, kI8>();
  }
}

template <int D, int G, bool kI8>
cudaError_t launch_split_t(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                           cudaStream_t stream) {
  const size_t smem = decode_smem_bytes<D, G, kI8>();
  auto kern = decode_split_kernel<D, G, kI8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
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
  return cudaLaunchKernelEx(&cfg, kern, kmap, vmap, a);
}

template <int D, bool kI8>
cudaError_t launch_split_d(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                           cudaStream_t stream) {
  switch (a.num_q_heads / a.num_kv_heads) {
    case 1: return launch_split_t<D, 1, kI8>(a, kmap, vmap, stream);
    case 2: return launch_split_t<D, 2, kI8>(a, kmap, vmap, stream);
    case 4: return launch_split_t<D, 4, kI8>(a, kmap, vmap, stream);
    case 8: return launch_split_t<D, 8, kI8>(a, kmap, vmap, stream);
    case 16: return launch_split_t<D, 16, kI8>(a, kmap, vmap, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int decode_num_ctas(int head_dim, int group, int num_sms, int64_t num_pairs, int max_splits,
                    bool int8) {
  const int per_sm = int8 ? (head_dim == 64 ? ctas_per_sm_d<64, true>(group)
                                            : ctas_per_sm_d<128, true>(group))
                          : (head_dim == 64 ? ctas_per_sm_d<64, false>(group)
                                            : ctas_per_sm_d<128, false>(group));
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
  if (a.head_dim == 128) return launch_split_d<128, false>(a, maps.k_rows, maps.v_rows, stream);
  if (a.head_dim == 64) return launch_split_d<64, false>(a, maps.k_rows, maps.v_rows, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode_i8(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                             cudaStream_t stream) {
  if (!a.k_scales || !a.v_scales) return cudaErrorInvalidValue;
  if (a.head_dim == 128) return launch_split_d<128, true>(a, kmap, vmap, stream);
  if (a.head_dim == 64) return launch_split_d<64, true>(a, kmap, vmap, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
