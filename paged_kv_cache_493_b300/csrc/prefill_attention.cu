// prefill_attention.cu -- chunked causal prefill over a paged KV cache on
// the tcgen05 tensor cores.
//
// What is computed (tuning guide "Nano-vLLM性能调优实战" §3.2: prompts are
// processed in chunks bounded by max_num_batched_tokens; §2.2 variable-length
// batches over the cache; intelliparadigm.com Nano-vLLM article §7.1 预填充阶段;
// ocdem.com nano-vllm article §2.1 block tables): sequence s has a chunk of
// Lq query rows and C cached tokens (chunk included).  Query i sits at
// position C - Lq + i and attends to keys 0 .. C - Lq + i:
//   out = softmax(scale * Q K^T + causal mask) V.
//
// One CTA computes a 128-row tile: 128/G consecutive queries x the G query
// heads of one KV head, so every K/V tile is loaded once for the whole GQA
// group.  Keys are visited in tiles of 64, looked up through the block table
// and loaded by TMA with 128-byte swizzle.  Two CTAs share an SM (96 KB of
// shared memory and 256 tensor-memory columns each): the softmax of one is
// latency-bound, so a second independent pipeline fills its gaps.
//   warp 4     TMA producer: Q once, then K tiles (2 stages);
//   warp 6     TMA producer: V tiles (2 stages; K loads never queue behind a
//              V stage that a PV still reads);
//   warp 5     allocates 256 tensor-memory columns and issues the MMAs from
//              one thread, as two streams each issued as soon as it is ready:
//              S_j = Q K_j^T into one of two 64-column S buffers (needs K_j,
//              and PV_{j-2} issued: P_{j-2} sits in that buffer and the tensor
//              pipe executes in order), and O += P_j V_j with P_j read from
//              tensor memory (needs P_j and V_j), fp32 accumulators;
//   warps 0-3  softmax: thread r owns row r (tensor-memory lane r).  It loads
//              S_j, applies scale and mask, keeps the running max m and sum
//              l, writes P_j = exp2(S - m) as bf16 pairs over the first half
//              of S_j's own columns (so P is double-buffered with S, and no
//              shared memory is used for it), and rescales its O row in
//              tensor memory when the max grew by more than 2^8 (the final
//              division by l makes any reference value exact, so the rescale
//              is deferred); finally O / l is written out as bf16.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int kRows = 128;        // MMA M: query rows per tile
constexpr int kKeyTile = kPrefillKeyTile;  // keys per tile (MMA N of QK^T, K of PV)
constexpr int kKvStages = 2;
constexpr int kSoftmaxWarps = 4;
constexpr int kProducerWarp = 4;  // Q and K tiles
constexpr int kMmaWarp = 5;
constexpr int kVProducerWarp = 6;
constexpr int kPrefillThreads = 7 * 32;
constexpr int kCtasPerSm = 2;
constexpr int kTmemCols = 256;
constexpr int kSCol0 = 0;         // S buffers at columns 0 and kKeyTile
constexpr int kOCol = 2 * kKeyTile;  // O at columns kOCol .. kOCol + D
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct PrefillLayout {
  static constexpr int kPanels = D / 64;                 // 64-element (128-byte) column panels
  static constexpr int kQPanel = kRows * 128;            // 128 query rows x 128 bytes
  static constexpr int kKvPanel = kKeyTile * 128;        // 64 key rows x 128 bytes
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kPanels * kQPanel;      // stages of K
  static constexpr int kV = kK + kKvStages * kPanels * kKvPanel;
  static constexpr int kBar = kV + kKvStages * kPanels * kKvPanel;
  // barriers: q_full, k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[2],
  //           p_full[2], pv_done[2], drain   (17 x 8 bytes) + misc words
  static constexpr int kMisc = kBar + 24 * 8;
  // Shared-prefix role only: each row's (m, l) for the cluster merge, then
  // the per-row merge factors of the rows this CTA merges.
  static constexpr int kRowMl = kMisc + 64;              // float2 [128]
  static constexpr int kMergeW = kRowMl + kRows * 8;     // float [128] (rows x units)
  static constexpr int kMergeRow = kMergeW + kRows * 4;  // float M, L; int bad [<= 128]
  static constexpr int kBytes = kMergeRow + kRows * 12;
  // INT8 cache only (the shared-prefix region is unused there): the scales
  // of the K and V tiles in flight, float [2 stages][64] each.
  static constexpr int kKScales = kRowMl;
  static constexpr int kVScales = kKScales + kKvStages * kKeyTile * 4;
  static_assert(kVScales + kKvStages * kKeyTile * 4 <= kBytes, "scale stages fit");
  // After the last PV the Q/K/V buffers are free: each row's O (fp32) is
  // staged there for the cluster merge, rows padded by 4 floats.
  static constexpr int kOStride = D + 4;
  static_assert(kRows * kOStride * 4 <= kBar, "O staging fits in the Q/K/V buffers");
};

// Barrier addresses from the first barrier's: computed, not stored, so a
// stage picked at run time costs no local-memory load on the hot loops.
// Byte offsets of stage 0's barriers (stage 1: + 8).
constexpr uint32_t kBarKFull = 8, kBarKEmpty = 24, kBarVFull = 40, kBarVEmpty = 56;
constexpr uint32_t kBarSFull = 72, kBarPFull = 88, kBarPvDone = 104, kBarDrain = 120;
// INT8 cache only: the codes and scales of a K (V) stage have landed.
constexpr uint32_t kBarKRaw = 128, kBarVRaw = 144;

struct PrefillBars {
  uint32_t base;
  __device__ __forceinline__ uint32_t q_full() const { return base; }
  __device__ __forceinline__ uint32_t k_full(int s) const { return base + kBarKFull + 8 * s; }
  __device__ __forceinline__ uint32_t k_empty(int s) const { return base + kBarKEmpty + 8 * s; }
  __device__ __forceinline__ uint32_t v_full(int s) const { return base + kBarVFull + 8 * s; }
  __device__ __forceinline__ uint32_t v_empty(int s) const { return base + kBarVEmpty + 8 * s; }
  __device__ __forceinline__ uint32_t s_full(int s) const { return base + kBarSFull + 8 * s; }
  __device__ __forceinline__ uint32_t p_full(int s) const { return base + kBarPFull + 8 * s; }
  __device__ __forceinline__ uint32_t pv_done(int s) const { return base + kBarPvDone + 8 * s; }
  __device__ __forceinline__ uint32_t drain() const { return base + kBarDrain; }
};

__device__ __forceinline__ PrefillBars make_bars(uint32_t base) { return PrefillBars{base}; }

struct TileInfo {
  int seq, qt_start, lq, ctx, q_row0;
  bool valid;
};

// Tile t of the CTA list -> (sequence, first query of the tile).  Sequences
// are taken in order; inside a sequence the last (longest) tiles come first.
__device__ __forceinline__ TileInfo find_tile(const PrefillArgs& a, int t, int qt_rows) {
  TileInfo ti;
  ti.valid = false;
  ti.seq = -1;
  int base = 0;
  for (int s = 0; s < a.num_seqs; ++s) {
    const int c0 = a.cu_seqlens_q[s], c1 = a.cu_seqlens_q[s + 1];
    const int lq = max(c1 - c0, 0);
    const int nt = (lq + qt_rows - 1) / qt_rows;
    if (t < base + nt) {
      const int k = t - base;
      ti.seq = s;
      ti.qt_start = (nt - 1 - k) * qt_rows;
      ti.lq = lq;
      ti.ctx = a.context_lens[s];
      ti.q_row0 = c0;
      ti.valid = true;
      return ti;
    }
    base += nt;
  }
  return ti;
}

// Four int8 codes (one word) times their row's scale, as two bf16 pairs
// (round to nearest even).  A code c becomes exact in fp32 as the float with
// bit pattern 0x4B0000xx, xx = c + 128 (that is 2^23 + c + 128), minus
// 2^23 + 128; the product with the scale is rounded to fp32, then to bf16.
__device__ __forceinline__ void dequant4(uint32_t w, uint64_t s2, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  const uint64_t bias = f2_pack(-8388736.0f, -8388736.0f);
  const uint64_t c01 = f2_add(f2_pack(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7440)),
                                      __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7441))),
                              bias);
  const uint64_t c23 = f2_add(f2_pack(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7442)),
                                      __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7443))),
                              bias);
  float x0, x1, x2, x3;
  f2_unpack(f2_mul(c01, s2), x0, x1);
  f2_unpack(f2_mul(c23, s2), x2, x3);
  lo = pack_bf16x2(x0, x1);
  hi = pack_bf16x2(x2, x3);
}

// One warp turns a stage holding an INT8 tile -- 64 keys x D codes, key k at
// byte k * D (no swizzle), and the keys' scales -- into the bf16 tile the
// tensor cores read, in place: 64-column panels of 128-byte rows with the
// 128-byte swizzle.  D / 16 lanes share a key, 16 codes each.  A key's bf16
// row overlaps only the codes of keys >= its own (for D = 128 exactly its
// own; for D = 64 those of keys 2k and 2k + 1), so batches are taken from
// the last key down, and a batch reads all its codes before any lane
// writes.
template <int D>
__device__ __forceinline__ void dequant_stage(uint8_t* stage, const float* scales, int lane) {
  constexpr int kLanesPerKey = D / 16;
  constexpr int kKeysPerPass = 32 / kLanesPerKey;
  constexpr int kPasses = 4;
  constexpr int kKeysPerBatch = kKeysPerPass * kPasses;
  constexpr int kPanelBytes = kKeyTile * 128;
  const int piece = lane % kLanesPerKey;  // codes 16 piece .. 16 piece + 15
  const int kk = lane / kLanesPerKey;
  const int panel = piece >> 2;
  const int ch0 = (2 * piece) & 7;
  // Panel-1 lanes store their odd chunk first: the eight lanes of a store
  // phase then hit eight different 16-byte bank groups.
  const int first = ch0 + (panel & 1), second = ch0 + 1 - (panel & 1);
#pragma unroll 1
  for (int b = kKeyTile / kKeysPerBatch - 1; b >= 0; --b) {
    uint4 c[kPasses];
    float sc[kPasses];
#pragma unroll
    for (int p = 0; p < kPasses; ++p) {
      const int k = b * kKeysPerBatch + p * kKeysPerPass + kk;
      c[p] = *reinterpret_cast<const uint4*>(stage + k * D + piece * 16);
      sc[p] = scales[k];
    }
    __syncwarp();
#pragma unroll
    for (int p = 0; p < kPasses; ++p) {
      const int k = b * kKeysPerBatch + p * kKeysPerPass + kk;
      const uint64_t s2 = f2_pack(sc[p], sc[p]);
      uint4 lo, hi;  // codes 0-7 and 8-15 of the piece
      dequant4(c[p].x, s2, lo.x, lo.y);
      dequant4(c[p].y, s2, lo.z, lo.w);
      dequant4(c[p].z, s2, hi.x, hi.y);
      dequant4(c[p].w, s2, hi.z, hi.w);
      uint8_t* row = stage + panel * kPanelBytes;
      *reinterpret_cast<uint4*>(row + sw128_offset(k, first)) = first == ch0 ? lo : hi;
      *reinterpret_cast<uint4*>(row + sw128_offset(k, second)) = second == ch0 ? lo : hi;
    }
  }
}

// kShared = false: chunked causal prefill (grid: tiles x KV heads).
// kShared = true: the shared-prefix role of the cascade decode (grid: row
// tiles x units x KV heads).  The "queries" of a tile are then 128/G
// sequences' decode queries (q viewed as [num_seqs][Hq][D]), the keys are
// the unit's share of the shared prefix (the leading blocks of table row 0,
// the same in every sharing sequence's table), nothing is masked, and the
// epilogue writes each row's partial state -- the reference max m (log2
// domain), the sum l and the unnormalised O, fp32 -- for the decode kernel
// to merge with the sequence's private part.
// kI8 = true (with kShared = false): the cache holds INT8 codes and scales
// (head-major blocks); kmap / vmap view the codes as {D, 256, blocks x Hkv}
// with box {D, 64, 1}.  The two producer warps load a stage's codes and
// scales and, all 32 lanes, dequantise it in place to the bf16 layout of the
// bf16 cache; the MMA and softmax warps are unchanged.
template <int D, int G, bool kShared, bool kI8>
__global__ void __launch_bounds__(kPrefillThreads, kCtasPerSm)
prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
               const __grid_constant__ CUtensorMap vmap, PrefillArgs a) {
  static_assert(!(kShared && kI8), "no INT8 shared-prefix role");
  using L = PrefillLayout<D>;
  constexpr int QT = kRows / G;  // queries per tile
  constexpr uint32_t kKTileBytes = kKeyTile * D * 2;
  constexpr uint32_t kQBytes = kRows * D * 2;

  // The 128-byte swizzle repeats every 1024 bytes: the panels need a
  // 1024-byte-aligned base.  Dynamic shared memory starts there (no static
  // shared memory in this kernel); a misaligned base is reported, not used.
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t sbase = smem_u32(smem_raw);
  if (sbase & 1023u) {
    if (threadIdx.x == 0) report_error(a.err, kErrDeviceCheck, kSitePrefillAlign);
    return;
  }
  uint8_t* sgen = smem_raw;
  const PrefillBars bar = make_bars(sbase + L::kBar);
  volatile int* misc = reinterpret_cast<volatile int*>(sgen + L::kMisc);
  // misc[0] tmem base, misc[1] abort flag, misc[2] bad tile

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Shared-prefix role: the shared_units CTAs of one (row tile, KV head) are
  // consecutive, one cluster; unit = rank in the cluster.
  const int kvh = kShared ? (blockIdx.x / a.shared_units) % a.num_kv_heads
                          : blockIdx.x % a.num_kv_heads;
  const int tile = kShared ? (blockIdx.x / a.shared_units) / a.num_kv_heads
                           : blockIdx.x / a.num_kv_heads;
  const int unit = kShared ? blockIdx.x % a.shared_units : 0;

  if (threadIdx.x == 0) {
    mbar_init(bar.q_full(), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar.k_full(s), 1);
      mbar_init(bar.k_empty(s), 1);
      mbar_init(bar.v_full(s), 1);
      mbar_init(bar.v_empty(s), 1);
      mbar_init(bar.s_full(s), 1);
      mbar_init(bar.p_full(s), kSoftmaxWarps * 32);
      mbar_init(bar.pv_done(s), 1);
    }
    mbar_init(bar.drain(), 1);
    if constexpr (kI8) {
      for (int s = 0; s < 2; ++s) {
        mbar_init(sbase + L::kBar + kBarKRaw + 8 * s, 1);
        mbar_init(sbase + L::kBar + kBarVRaw + 8 * s, 1);
      }
    }
    misc[1] = 0;
    misc[2] = 0;
    fence_barrier_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&qmap);
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(sbase + L::kMisc, kTmemCols);
    tmem_relinquish();
  }
  grid_dependency_wait();
  grid_dependents_launch();

  TileInfo ti;
  const int max_ctx = a.max_blocks * kBlockSize;
  bool bad = false;
  int nkt = 0;
  int kbase = 0;  // first key of the CTA's range
  if constexpr (kShared) {
    // Tile `tile` holds sequences [tile * QT, tile * QT + QT); unit `unit`
    // takes key tiles [t0, t1) of the shared prefix.
    ti.seq = 0;
    ti.qt_start = tile * QT;
    ti.lq = a.num_seqs;
    ti.ctx = a.shared_tiles * kKeyTile;
    ti.q_row0 = 0;
    ti.valid = ti.qt_start < a.num_seqs;
    const int t0 = static_cast<int>(static_cast<int64_t>(unit) * a.shared_tiles / a.shared_units);
    const int t1 =
        static_cast<int>(static_cast<int64_t>(unit + 1) * a.shared_tiles / a.shared_units);
    nkt = ti.valid ? t1 - t0 : 0;
    kbase = t0 * kKeyTile;
  } else {
    ti = find_tile(a, tile, QT);
    if (ti.valid) {
      bad = ti.ctx < 0 || ti.ctx > max_ctx || ti.lq > ti.ctx || ti.q_row0 < 0 ||
            static_cast<int64_t>(ti.q_row0) + ti.lq > a.total_q;
      if (!bad) {
        const int q_end = min(ti.qt_start + QT, ti.lq);      // one past the last real query
        const int kmax = ti.ctx - ti.lq + q_end;              // keys the tile needs
        nkt = (kmax + kKeyTile - 1) / kKeyTile;
      }
    }
  }
  const int32_t* table = a.block_tables + static_cast<int64_t>(max(ti.seq, 0)) * a.max_blocks;
  if (warp == kProducerWarp && ti.valid && !bad) {
    const int nblk = (kbase + nkt * kKeyTile + kBlockSize - 1) / kBlockSize;
    bool b = false;
    for (int i = kbase / kBlockSize + lane; i < nblk; i += 32) {
      const int id = table[i];
      b |= (id < 0 || id >= a.num_blocks);
    }
    if (__any_sync(0xffffffffu, b) && lane == 0) misc[2] = 1;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(misc[0]);
  if (ti.valid && (bad || misc[2]) && threadIdx.x == 0)
    report_error(a.err, kErrDeviceCheck, bad ? kSitePrefillChunk : kSitePrefillBlock);
  const bool run = ti.valid && !bad && misc[2] == 0 && nkt > 0;

  if (kI8 && (warp == kProducerWarp || warp == kVProducerWarp)) {
    // ------------------------------------------------- INT8 producers (Q, K) and (V)
    // Event loop of the whole warp (lane 0 decides, the warp follows):
    // issue the next tile's codes and scales into a free stage, or
    // dequantise the oldest stage that has landed and hand it to the MMA.
    if (run) {
      const bool is_k = warp == kProducerWarp;
      const CUtensorMap* map = is_k ? &kmap : &vmap;
      const float* gscales = is_k ? a.k_scales : a.v_scales;
      // Stage st's barriers: raw + 8 st (copies landed), full + 8 st (bf16
      // tile ready for the MMA), empty + 8 st (the MMA is done with it).
      const uint32_t bars = sbase + L::kBar;
      const uint32_t raw = bars + (is_k ? kBarKRaw : kBarVRaw);
      const uint32_t full = bars + (is_k ? kBarKFull : kBarVFull);
      const uint32_t empty = bars + (is_k ? kBarKEmpty : kBarVEmpty);
      const int stage0 = is_k ? L::kK : L::kV;
      const int scale0 = is_k ? L::kKScales : L::kVScales;
      const int site = kSitePrefillWait + (is_k ? 8 : 9);
      constexpr uint32_t kCodeBytes = kKeyTile * D;
      constexpr uint32_t kScaleBytes = kKeyTile * 4;
      constexpr int kStageBytes = L::kPanels * L::kKvPanel;
      if (is_k && lane == 0) {
        mbar_arrive_expect_tx(bar.q_full(), kQBytes);
#pragma unroll
        for (int p = 0; p < L::kPanels; ++p)
          tma_load_3d(sbase + L::kQ + p * L::kQPanel, &qmap, bar.q_full(), p * 64, kvh * G,
                      ti.q_row0 + ti.qt_start);
      }
      int ji = 0, jc = 0;  // next tile to issue, to convert
      bool idle = false;
      uint64_t idle_since = 0;
      while (jc < nkt) {
        int act = 0;  // 1 issue, 2 convert, -1 stop
        if (lane == 0) {
          if (misc[1]) {
            act = -1;
          } else if (ji < nkt &&
                     (ji < kKvStages || mbar_test(empty + 8 * (ji & 1), ((ji >> 1) - 1) & 1))) {
            act = 1;
          } else if (jc < ji && mbar_test(raw + 8 * (jc & 1), (jc >> 1) & 1)) {
            act = 2;
          } else {
            const uint64_t now = global_timer_ns();
            if (!idle) {
              idle = true;
              idle_since = now;
            } else if (now - idle_since > a.wait_limit_ns) {
              report_error(a.err, kErrTimeout, site);
              misc[1] = 1;
              act = -1;
            }
          }
          if (act != 0) idle = false;
        }
        act = __shfl_sync(0xffffffffu, act, 0);
        if (act < 0) break;
        if (act == 1) {
          if (lane == 0) {
            const int st = ji & 1;
            const int k0 = kbase + ji * kKeyTile;
            const int row = k0 % kBlockSize;
            const int tile_id = table[k0 / kBlockSize] * a.num_kv_heads + kvh;
            const uint32_t rb = raw + 8 * st;
            mbar_arrive_expect_tx(rb, kCodeBytes + kScaleBytes);
            tma_load_3d(sbase + stage0 + st * kStageBytes, map, rb, 0, row, tile_id);
            bulk_load(sbase + scale0 + st * static_cast<int>(kScaleBytes),
                      gscales + static_cast<int64_t>(tile_id) * kBlockSize + row, kScaleBytes, rb);
          }
          ++ji;
        } else if (act == 2) {
          const int st = jc & 1;
          // Completed phase: returns at once, and makes the copied bytes
          // visible to every lane.
          mbar_wait(raw + 8 * st, (jc >> 1) & 1, kDrainLimitNs);
          dequant_stage<D>(sgen + stage0 + st * kStageBytes,
                           reinterpret_cast<const float*>(sgen + scale0) + st * kKeyTile, lane);
          fence_proxy_async_smem();  // the tensor cores read what the lanes wrote
          __syncwarp();
          if (lane == 0) mbar_arrive(full + 8 * st);
          ++jc;
        } else {
          __nanosleep(64);
        }
      }
      if (lane == 0) {
        // Every copy issued must land before the block may exit.
        if (is_k) mbar_wait(bar.q_full(), 0, kDrainLimitNs);
        for (int t = jc; t < ji; ++t) mbar_wait(raw + 8 * (t & 1), (t >> 1) & 1, kDrainLimitNs);
      }
    }
  } else if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer (Q, K)
    if (lane == 0 && run) {
      int issued = 0;  // tiles issued (tile j into stage j & 1)
      mbar_arrive_expect_tx(bar.q_full(), kQBytes);
#pragma unroll
      for (int p = 0; p < L::kPanels; ++p)
        tma_load_3d(sbase + L::kQ + p * L::kQPanel, &qmap, bar.q_full(), p * 64, kvh * G,
                    ti.q_row0 + ti.qt_start);
      for (int j = 0; j < nkt; ++j) {
        const int st = j & 1;
        const int k0 = kbase + j * kKeyTile;
        const int slot = table[k0 / kBlockSize] * kBlockSize + (k0 % kBlockSize);
        if (j >= kKvStages &&
            !mbar_wait(bar.k_empty(st), ((j >> 1) - 1) & 1, a.wait_limit_ns)) {
          report_error(a.err, kErrTimeout, kSitePrefillWait + 0);
          misc[1] = 1;
          break;
        }
        if (misc[1]) break;
        mbar_arrive_expect_tx(bar.k_full(st), kKTileBytes);
#pragma unroll
        for (int p = 0; p < L::kPanels; ++p)
          tma_load_3d(sbase + L::kK + (st * L::kPanels + p) * L::kKvPanel, &kmap, bar.k_full(st),
                      p * 64, kvh, slot);
        issued = j + 1;
      }
      // Every copy issued must land before the block may exit, whether or
      // not its consumer gave up on it (after a normal run these waits
      // return at once): the last tile issued into each stage holds its
      // newest phase.
      mbar_wait(bar.q_full(), 0, kDrainLimitNs);
      for (int t = max(issued - kKvStages, 0); t < issued; ++t)
        mbar_wait(bar.k_full(t & 1), (t >> 1) & 1, kDrainLimitNs);
    }
  } else if (warp == kVProducerWarp) {
    // ------------------------------------------------------------ producer (V)
    if (lane == 0 && run) {
      int issued = 0;  // tiles issued (tile j into stage j & 1)
      for (int j = 0; j < nkt; ++j) {
        const int st = j & 1;
        const int k0 = kbase + j * kKeyTile;
        const int slot = table[k0 / kBlockSize] * kBlockSize + (k0 % kBlockSize);
        if (j >= kKvStages &&
            !mbar_wait(bar.v_empty(st), ((j >> 1) - 1) & 1, a.wait_limit_ns)) {
          report_error(a.err, kErrTimeout, kSitePrefillWait + 1);
          misc[1] = 1;
          break;
        }
        if (misc[1]) break;
        mbar_arrive_expect_tx(bar.v_full(st), kKTileBytes);
#pragma unroll
        for (int p = 0; p < L::kPanels; ++p)
          tma_load_3d(sbase + L::kV + (st * L::kPanels + p) * L::kKvPanel, &vmap, bar.v_full(st),
                      p * 64, kvh, slot);
        issued = j + 1;
      }
      for (int t = max(issued - kKvStages, 0); t < issued; ++t)
        mbar_wait(bar.v_full(t & 1), (t >> 1) & 1, kDrainLimitNs);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && run) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kRows, kKeyTile, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(kRows, D, true);
      bool ok = mbar_wait(bar.q_full(), 0, a.wait_limit_ns);
      if (!ok) report_error(a.err, kErrTimeout, kSitePrefillWait + 2);
      int js = 0, jp = 0;
      bool idle = false;
      uint64_t idle_since = 0;
      while (ok && jp < nkt) {
        bool did = false;
        // S_js overwrites the columns where P_{js-2} sits: only after PV_{js-2}
        // has been issued (the tensor pipe executes in order).
        if (js < nkt && js - 2 < jp && mbar_test(bar.k_full(js & 1), (js >> 1) & 1)) {  // S_js = Q K_js^T
          const int st = js & 1;
          tc_fence_after();
          const uint32_t d_tmem = tmem + kSCol0 + st * kKeyTile;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t qoff = (kk >> 2) * L::kQPanel + (kk & 3) * 32;
            const uint32_t koff = (kk >> 2) * L::kKvPanel + (kk & 3) * 32;
            const uint64_t ad = smem_desc_sw128(sbase + L::kQ + qoff, 16, 1024);
            const uint64_t bd =
                smem_desc_sw128(sbase + L::kK + st * L::kPanels * L::kKvPanel + koff, 16, 1024);
            tc_mma_ss(d_tmem, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
          }
          tc_commit(bar.s_full(st));
          tc_commit(bar.k_empty(st));
          ++js;
          did = true;
        }
        if (jp < js && mbar_test(bar.p_full(jp & 1), (jp >> 1) & 1) &&
            mbar_test(bar.v_full(jp & 1), (jp >> 1) & 1)) {  // O += P_jp V_jp
          const int st = jp & 1;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kKeyTile / 16; ++kk) {
            // P_jp: bf16 pairs in the first kKeyTile / 2 columns of S buffer st.
            const uint32_t a_tmem = tmem + kSCol0 + st * kKeyTile + kk * 8;
            // V stage: [64 keys][64 d] panels; 16 keys = 2 x 8-row groups.
            const uint64_t bd = smem_desc_sw128(
                sbase + L::kV + st * L::kPanels * L::kKvPanel + kk * 16 * 128, L::kKvPanel, 1024);
            tc_mma_ts(tmem + kOCol, a_tmem, bd, idesc_o, (jp > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(bar.pv_done(st));
          tc_commit(bar.v_empty(st));
          ++jp;
          did = true;
        }
        if (did) {
          idle = false;
          continue;
        }
        if (misc[1]) {
          ok = false;
          break;
        }
        const uint64_t now = global_timer_ns();
        if (!idle) {
          idle = true;
          idle_since = now;
        } else if (now - idle_since > a.wait_limit_ns) {
          report_error(a.err, kErrTimeout, kSitePrefillWait + 3);
          ok = false;
          break;
        }
        __nanosleep(32);  // leave the scheduler's issue slots to the softmax warps
      }
      if (!ok) misc[1] = 1;
      // Every MMA issued must finish before tensor memory is released.
      tc_commit(bar.drain());
      mbar_wait(bar.drain(), 0, kDrainLimitNs);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int r = threadIdx.x;  // tile row == tensor-memory lane
    const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const float sl2 = a.scale * 1.4426950408889634f;
    const int qi = (ti.valid ? ti.qt_start : 0) + r / G;  // query index inside the chunk
    const int head = kvh * G + (r % G);
    const bool row_real = run && qi < ti.lq;
    const int lim = run ? min(ti.ctx - ti.lq + qi, ti.ctx - 1) : 0;  // last visible key
    const int pos_min = run ? ti.ctx - ti.lq + ti.qt_start : 0;       // smallest row position
    float m = -INFINITY, l = 0.f;  // reference max (log2 domain, may lag by < 2^8) and sum
    bool ok = run;
    // A masked raw score: it must vanish in the max (or min, for a negative
    // scale) and give exp2(-inf) = 0.
    const float masked = sl2 >= 0.f ? -INFINITY : INFINITY;
    for (int j = 0; ok && j < nkt; ++j) {
      // Exit decisions are warp-uniform: tcgen05.ld/st are warp-collective.
      const bool got = mbar_wait(bar.s_full(j & 1), (j >> 1) & 1, a.wait_limit_ns);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) report_error(a.err, kErrTimeout, kSitePrefillWait + 5);
        ok = false;
        break;
      }
      tc_fence_after();
      float x[kKeyTile];
#pragma unroll
      for (int c = 0; c < kKeyTile / 32; ++c)
        tmem_ld_32x32b_x32(trow + kSCol0 + (j & 1) * kKeyTile + c * 32,
                           *reinterpret_cast<uint32_t(*)[32]>(&x[c * 32]));
      // The abort flag is read while the loads are in flight.
      const int abort = __shfl_sync(0xffffffffu, misc[1], 0);
      tmem_wait_ld();
      if (abort) {
        ok = false;
        break;
      }
      const int k0 = j * kKeyTile;  // key of x[0]
      if (!kShared && ((k0 + kKeyTile - 1 > pos_min) || (k0 + kKeyTile > ti.ctx))) {
#pragma unroll
        for (int c = 0; c < kKeyTile; ++c)
          if (k0 + c > lim) x[c] = masked;
      }
      // Row max of the scaled scores, from 8 independent partial maxima of
      // the raw ones (three-input max; the scale's sign decides max or min).
      float mp[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mp[i] = x[i];
      if (sl2 >= 0.f) {
#pragma unroll
        for (int c = 8; c < kKeyTile; c += 2) mp[(c >> 1) & 7] = fmax3(mp[(c >> 1) & 7], x[c], x[c + 1]);
        mp[0] = fmax3(mp[0], mp[1], mp[2]);
        mp[3] = fmax3(mp[3], mp[4], mp[5]);
        mp[0] = fmax3(mp[0], mp[3], fmaxf(mp[6], mp[7]));
      } else {
#pragma unroll
        for (int c = 8; c < kKeyTile; c += 2) mp[(c >> 1) & 7] = fmin3(mp[(c >> 1) & 7], x[c], x[c + 1]);
        mp[0] = fmin3(mp[0], mp[1], mp[2]);
        mp[3] = fmin3(mp[3], mp[4], mp[5]);
        mp[0] = fmin3(mp[0], mp[3], fminf(mp[6], mp[7]));
      }
      const float m_new = fmaxf(m, mp[0] * sl2);
      const bool need = m_new > m + kRescaleThreshold;  // true on the first tile
      if (__any_sync(0xffffffffu, need)) {
        const float alpha = need ? fast_exp2(m - m_new) : 1.f;
        if (j >= 1) {
          // O holds PV up to tile j - 1: wait for it before rescaling.
          const bool got_o =
              mbar_wait(bar.pv_done((j - 1) & 1), ((j - 1) >> 1) & 1, a.wait_limit_ns);
          if (!__all_sync(0xffffffffu, got_o)) {
            if (lane == 0) report_error(a.err, kErrTimeout, kSitePrefillWait + 6);
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            tmem_ld_32x32b_x32(trow + kOCol + c * 32, ov);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            tmem_st_32x32b_x32(trow + kOCol + c * 32, ov);
          }
          tmem_wait_st();
        }
        if (need) {
          l *= alpha;
          m = m_new;
        }
      }
      // P = exp2(scale * x - m) -> bf16 pairs over the first half of S_j's
      // columns, where the PV MMA reads them (every key of the row masked so
      // far: m = -inf, P = 0)
      const float neg_m = m == -INFINITY ? 0.f : -m;
      // Pairs of keys in packed two-wide fp32 (scale-and-shift, row sum).
      const uint64_t sc2 = f2_pack(sl2, sl2), nm2 = f2_pack(neg_m, neg_m);
      uint64_t rs2[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) rs2[i] = 0ull;
      uint32_t pw[kKeyTile / 2];
#pragma unroll
      for (int c = 0; c < kKeyTile / 2; ++c) {
        float y0, y1;
        f2_unpack(f2_fma(f2_pack(x[2 * c], x[2 * c + 1]), sc2, nm2), y0, y1);
        const float p0 = fast_exp2(y0);
        const float p1 = fast_exp2(y1);
        rs2[c & 3] = f2_add(rs2[c & 3], f2_pack(p0, p1));
        pw[c] = pack_bf16x2_nonneg(p0, p1);
      }
      static_assert(kKeyTile / 2 == 32, "one 32-column store per row");
      tmem_st_32x32b_x32(trow + kSCol0 + (j & 1) * kKeyTile, pw);
      tmem_wait_st();
      float rs[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) f2_unpack(rs2[i], rs[i], rs[i + 4]);
      l += ((rs[0] + rs[1]) + (rs[2] + rs[3])) + ((rs[4] + rs[5]) + (rs[6] + rs[7]));
      tc_fence_before();
      mbar_arrive(bar.p_full(j & 1));
    }
    // ---- epilogue: O / l -> bf16
    if (ok && nkt > 0) {  // ok is warp-uniform here
      const bool got =
          mbar_wait(bar.pv_done((nkt - 1) & 1), ((nkt - 1) >> 1) & 1, a.wait_limit_ns);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) report_error(a.err, kErrTimeout, kSitePrefillWait + 7);
        ok = false;
      }
    }
    const bool epilogue = __shfl_sync(0xffffffffu, (ok && nkt > 0 && !misc[1]) ? 1 : 0, 0) != 0;
    if constexpr (kShared) {
      // This unit's partial state of row r (sequence qi, head r % G) --
      // unnormalised O, reference max m, sum l -- is staged in shared
      // memory for the cluster merge below.  A row whose unit failed
      // (rejected block id, expired wait) is marked l = -1.
      float2* row_ml = reinterpret_cast<float2*>(sgen + L::kRowMl);
      if (epilogue) {
        tc_fence_after();
        float* orow = reinterpret_cast<float*>(sgen) + r * L::kOStride;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld_32x32b_x32(trow + kOCol + c * 32, ov);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 8; ++e)
            *reinterpret_cast<uint4*>(orow + c * 32 + 4 * e) =
                make_uint4(ov[4 * e], ov[4 * e + 1], ov[4 * e + 2], ov[4 * e + 3]);
        }
        row_ml[r] = make_float2(m, l);
      } else {
        row_ml[r] = make_float2(0.f, -1.f);
      }
    } else if (epilogue) {
      tc_fence_after();
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.out) +
                            (static_cast<int64_t>(ti.q_row0 + qi) * a.num_q_heads + head) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tmem_ld_32x32b_x32(trow + kOCol + c * 32, ov);
        tmem_wait_ld();
        if (row_real) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(ov[8 * e + 0]) * inv, __uint_as_float(ov[8 * e + 1]) * inv);
            v.y = pack_bf16x2(__uint_as_float(ov[8 * e + 2]) * inv, __uint_as_float(ov[8 * e + 3]) * inv);
            v.z = pack_bf16x2(__uint_as_float(ov[8 * e + 4]) * inv, __uint_as_float(ov[8 * e + 5]) * inv);
            v.w = pack_bf16x2(__uint_as_float(ov[8 * e + 6]) * inv, __uint_as_float(ov[8 * e + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + c * 32 + 8 * e) = v;
          }
        }
      }
    } else if (ti.valid && !run && qi < ti.lq && ti.q_row0 >= 0) {
      // Rejected tile (bad lengths or block ids): zero output for its rows.
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.out) +
                            (static_cast<int64_t>(ti.q_row0 + qi) * a.num_q_heads + head) * D;
      if (ti.q_row0 + qi < a.total_q)
        for (int d = 0; d < D; d += 8) *reinterpret_cast<uint4*>(orow + d) = make_uint4(0, 0, 0, 0);
    }
    if (!ok && run) misc[1] = 1;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }

  if constexpr (kShared) {
    // ---- cluster merge of the units' partial states (log-sum-exp):
    //   M = max_u m_u, L = sum_u l_u 2^(m_u - M), O = sum_u O_u 2^(m_u - M)
    // CTA of rank c merges rows [c R, c R + R), R = 128 / units, reading the
    // other units' staged rows from their shared memory, and writes the
    // merged state of each real row to global memory (a row any unit failed
    // on is marked l = -1).  Every thread of every CTA of the cluster passes
    // both cluster barriers (no early exit above in this role).
    const int U = a.shared_units;
    const int R = kRows / U;
    const uint32_t rank = cluster_ctarank();
    const int row0 = static_cast<int>(rank) * R;
    const uint32_t s_ml = sbase + L::kRowMl;
    float* mw = reinterpret_cast<float*>(sgen + L::kMergeW);         // [R][U]
    float* mrow = reinterpret_cast<float*>(sgen + L::kMergeRow);     // M [R], L [R]
    int* mbad = reinterpret_cast<int*>(sgen + L::kMergeRow + 8 * R);  // [R]
    cluster_sync_all();  // every unit's rows are staged
    constexpr int kMaxUnits = 16;
    if (static_cast<int>(threadIdx.x) < R) {
      // All units' (m, l) of the row in one round of remote loads.
      const int row = row0 + threadIdx.x;
      float2 ml[kMaxUnits];
#pragma unroll
      for (int u = 0; u < kMaxUnits; ++u)
        ml[u] = u < U ? dsmem_ld_f2(dsmem_map(s_ml + row * 8, u)) : make_float2(-INFINITY, 0.f);
      float M = -INFINITY;
      bool bad = false;
#pragma unroll
      for (int u = 0; u < kMaxUnits; ++u) {
        M = fmaxf(M, ml[u].x);
        bad |= ml[u].y < 0.f;
      }
      float Ls = 0.f;
#pragma unroll
      for (int u = 0; u < kMaxUnits; ++u) {
        const float w = (M == -INFINITY || ml[u].x == -INFINITY) ? 0.f : fast_exp2(ml[u].x - M);
        if (u < U) mw[threadIdx.x * U + u] = w;
        Ls += ml[u].y * w;
      }
      mrow[threadIdx.x] = M;
      mrow[R + threadIdx.x] = Ls;
      mbad[threadIdx.x] = bad ? 1 : 0;
    }
    __syncthreads();
    const int64_t prow0 = static_cast<int64_t>(kvh) * a.shared_rows_pad +
                          static_cast<int64_t>(tile) * kRows + row0;
    const int real_rows = min(R, max(0, a.num_seqs * G - (tile * kRows + row0)));
    constexpr int kGroups = D / 4;
    for (int i = threadIdx.x; i < real_rows * kGroups; i += kPrefillThreads) {
      const int rr = i / kGroups, g4 = (i % kGroups) * 4;
      const uint32_t src = sbase + static_cast<uint32_t>(((row0 + rr) * L::kOStride + g4) * 4);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      if (!mbad[rr]) {
        // Every unit's four values in one round of remote loads.
        float4 x[kMaxUnits];
#pragma unroll
        for (int u = 0; u < kMaxUnits; ++u)
          x[u] = u < U ? dsmem_ld_f4(dsmem_map(src, u)) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int u = 0; u < kMaxUnits; ++u) {
          const float w = u < U ? mw[rr * U + u] : 0.f;
          acc.x += w * x[u].x;
          acc.y += w * x[u].y;
          acc.z += w * x[u].z;
          acc.w += w * x[u].w;
        }
      }
      *reinterpret_cast<float4*>(a.shared_o + (prow0 + rr) * D + g4) = acc;
      if (g4 == 0)
        *reinterpret_cast<float2*>(a.shared_ml + (prow0 + rr) * 2) =
            make_float2(mrow[rr], mbad[rr] ? -1.f : mrow[R + rr]);
    }
    cluster_sync_all();  // no CTA leaves while others read its shared memory
  }
}

template <int D, int G, bool kShared, bool kI8>
cudaError_t launch_t(const PrefillArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                     const CUtensorMap& qmap, cudaStream_t stream) {
  using L = PrefillLayout<D>;
  auto kern = prefill_kernel<D, G, kShared, kI8>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
  if (e != cudaSuccess) return e;
  // Two CTAs per SM need the largest shared-memory carve-out.
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  constexpr int QT = kRows / G;
  int64_t blocks;
  if (kShared) {
    // Row tiles of QT sequences x units x KV heads.
    const int64_t tiles = (static_cast<int64_t>(a.num_seqs) + QT - 1) / QT;
    blocks = tiles * a.shared_units * a.num_kv_heads;
  } else {
    // Upper bound on the number of tiles: sum_s ceil(Lq_s / QT) <= total/QT + num_seqs.
    const int64_t tiles = a.total_q / QT + a.num_seqs;
    blocks = tiles * a.num_kv_heads;
  }
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = 1;
  if (kShared) {
    // The units of one (row tile, KV head) form a cluster (merged through
    // distributed shared memory); more than 8 needs the non-portable size.
    if (a.shared_units > 8) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
    }
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(a.shared_units);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kPrefillThreads);
  cfg.dynamicSmemBytes = L::kBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  return cudaLaunchKernelEx(&cfg, kern, qmap, kmap, vmap, a);
}

template <int D, bool kShared, bool kI8>
cudaError_t launch_d(const PrefillArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                     const CUtensorMap& qmap, cudaStream_t stream) {
  switch (a.num_q_heads / a.num_kv_heads) {
    case 1: return launch_t<D, 1, kShared, kI8>(a, kmap, vmap, qmap, stream);
    case 2: return launch_t<D, 2, kShared, kI8>(a, kmap, vmap, qmap, stream);
    case 4: return launch_t<D, 4, kShared, kI8>(a, kmap, vmap, qmap, stream);
    case 8: return launch_t<D, 8, kShared, kI8>(a, kmap, vmap, qmap, stream);
    case 16: return launch_t<D, 16, kShared, kI8>(a, kmap, vmap, qmap, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, const CacheMaps& maps, const CUtensorMap& qmap,
                           int num_sms, cudaStream_t stream) {
  (void)num_sms;
  if (a.head_dim == 128) return launch_d<128, false, false>(a, maps.k_sw128, maps.v_sw128, qmap, stream);
  if (a.head_dim == 64) return launch_d<64, false, false>(a, maps.k_sw128, maps.v_sw128, qmap, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_prefill_i8(const PrefillArgs& a, const CUtensorMap& kmap,
                              const CUtensorMap& vmap, const CUtensorMap& qmap,
                              cudaStream_t stream) {
  if (!a.k_scales || !a.v_scales) return cudaErrorInvalidValue;
  if (a.head_dim == 128) return launch_d<128, false, true>(a, kmap, vmap, qmap, stream);
  if (a.head_dim == 64) return launch_d<64, false, true>(a, kmap, vmap, qmap, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_shared_prefix(const PrefillArgs& a, const CacheMaps& maps,
                                 const CUtensorMap& qmap, cudaStream_t stream) {
  if (a.shared_units <= 0 || a.shared_units > 16 || (a.shared_units & (a.shared_units - 1)) ||
      a.shared_tiles < a.shared_units)
    return cudaErrorInvalidValue;
  if (a.head_dim == 128) return launch_d<128, true, false>(a, maps.k_sw128, maps.v_sw128, qmap, stream);
  if (a.head_dim == 64) return launch_d<64, true, false>(a, maps.k_sw128, maps.v_sw128, qmap, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
