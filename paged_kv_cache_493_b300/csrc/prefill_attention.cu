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
// group.  Keys are visited in tiles of 128 (half a cache block), looked up
// through the block table and loaded by TMA with 128-byte swizzle.
//   warp 4     TMA producer (Q once, then K and V tiles, 2 stages each);
//   warp 5     allocates 512 tensor-memory columns and issues the MMAs from
//              one thread: S_j = Q K_j^T into one of two 128-column S buffers,
//              then O += P_j V_j into the O columns (fp32 accumulators);
//   warps 0-3  softmax: thread r owns row r (tensor-memory lane r).  It reads
//              S_j, applies scale and mask, keeps the running max m and sum
//              l, writes P_j = exp2(S - m) as bf16 into shared memory in the
//              layout the MMA reads, and rescales its O row in tensor memory
//              when the max grew by more than 2^8 (the final division by l
//              makes any reference value exact, so the rescale is deferred);
//              finally O / l is written out as bf16.
// MMA order S_0, S_1, PV_0, S_2, PV_1, ... lets S_{j+1} run while the softmax
// works on S_j.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int kRows = 128;      // MMA M: query rows per tile
constexpr int kKeyTile = 128;   // keys per tile (MMA N of QK^T, K of PV)
constexpr int kKvStages = 2;
constexpr int kPrefillThreads = 192;
constexpr int kTmemCols = 512;
constexpr int kSCol0 = 0;       // S buffers at columns 0 and 128
constexpr int kOCol = 256;      // O at columns 256 .. 256 + D
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct PrefillLayout {
  static constexpr int kPanels = D / 64;                 // 64-element (128-byte) column panels
  static constexpr int kPanelBytes = kRows * 128;        // 128 rows x 128 bytes
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kPanels * kPanelBytes;  // stages of K
  static constexpr int kV = kK + kKvStages * kPanels * kPanelBytes;
  static constexpr int kP = kV + kKvStages * kPanels * kPanelBytes;
  static constexpr int kBar = kP + 2 * kPanelBytes;      // P: 128 keys = 2 panels
  // barriers: q_full, k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[2],
  //           p_full, o_done, drain   (15 x 8 bytes) + misc words
  static constexpr int kMisc = kBar + 16 * 8;
  static constexpr int kBytes = kMisc + 64;
  static constexpr int kAlloc = kBytes + 1024;           // slack for 1024-byte alignment
};

struct PrefillBars {
  uint32_t q_full, k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[2], p_full, o_done, drain;
};

__device__ __forceinline__ PrefillBars make_bars(uint32_t base) {
  PrefillBars b;
  b.q_full = base;
  b.k_full[0] = base + 8;
  b.k_full[1] = base + 16;
  b.k_empty[0] = base + 24;
  b.k_empty[1] = base + 32;
  b.v_full[0] = base + 40;
  b.v_full[1] = base + 48;
  b.v_empty[0] = base + 56;
  b.v_empty[1] = base + 64;
  b.s_full[0] = base + 72;
  b.s_full[1] = base + 80;
  b.p_full = base + 88;
  b.o_done = base + 96;
  b.drain = base + 104;
  return b;
}

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

template <int D, int G>
__global__ void __launch_bounds__(kPrefillThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
               const __grid_constant__ CUtensorMap vmap, PrefillArgs a) {
  using L = PrefillLayout<D>;
  constexpr int QT = kRows / G;  // queries per tile
  constexpr uint32_t kKTileBytes = kKeyTile * D * 2;
  constexpr uint32_t kQBytes = kRows * D * 2;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - smem_u32(smem_raw));
  const PrefillBars bar = make_bars(sbase + L::kBar);
  volatile int* misc = reinterpret_cast<volatile int*>(sgen + L::kMisc);
  // misc[0] tmem base, misc[1] abort flag, misc[2] bad tile

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int kvh = blockIdx.x % a.num_kv_heads;
  const int tile = blockIdx.x / a.num_kv_heads;

  if (threadIdx.x == 0) {
    mbar_init(bar.q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar.k_full[s], 1);
      mbar_init(bar.k_empty[s], 1);
      mbar_init(bar.v_full[s], 1);
      mbar_init(bar.v_empty[s], 1);
      mbar_init(bar.s_full[s], 1);
    }
    mbar_init(bar.p_full, kRows);
    mbar_init(bar.o_done, 1);
    mbar_init(bar.drain, 1);
    misc[1] = 0;
    misc[2] = 0;
    fence_barrier_init();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&qmap);
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
  }
  if (warp == 5) {
    tmem_alloc(sbase + L::kMisc, kTmemCols);
    tmem_relinquish();
  }
  grid_dependency_wait();
  grid_dependents_launch();

  const TileInfo ti = find_tile(a, tile, QT);
  const int max_ctx = a.max_blocks * kBlockSize;
  bool bad = false;
  int nkt = 0;
  if (ti.valid) {
    bad = ti.ctx < 0 || ti.ctx > max_ctx || ti.lq > ti.ctx || ti.q_row0 < 0 ||
          static_cast<int64_t>(ti.q_row0) + ti.lq > a.total_q;
    if (!bad) {
      const int q_end = min(ti.qt_start + QT, ti.lq);      // one past the last real query
      const int kmax = ti.ctx - ti.lq + q_end;              // keys the tile needs
      nkt = (kmax + kKeyTile - 1) / kKeyTile;
    }
  }
  const int32_t* table = a.block_tables + static_cast<int64_t>(max(ti.seq, 0)) * a.max_blocks;
  if (warp == 4 && ti.valid && !bad) {
    const int nblk = (nkt * kKeyTile + kBlockSize - 1) / kBlockSize;
    bool b = false;
    for (int i = lane; i < nblk; i += 32) {
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

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && run) {
      int k_last[2] = {-1, -1}, v_last[2] = {-1, -1};
      mbar_arrive_expect_tx(bar.q_full, kQBytes);
#pragma unroll
      for (int p = 0; p < L::kPanels; ++p)
        tma_load_3d(sbase + L::kQ + p * L::kPanelBytes, &qmap, bar.q_full, p * 64, kvh * G,
                    ti.q_row0 + ti.qt_start);
      for (int j = 0; j < nkt; ++j) {
        const int st = j & 1;
        const int k0 = j * kKeyTile;
        const int slot = table[k0 / kBlockSize] * kBlockSize + (k0 % kBlockSize);
        if (j >= kKvStages &&
            !mbar_wait(bar.k_empty[st], ((j >> 1) - 1) & 1, a.wait_limit_ns)) {
          report_error(a.err, kErrTimeout, kSitePrefillWait + 0);
          misc[1] = 1;
          break;
        }
        if (misc[1]) break;
        mbar_arrive_expect_tx(bar.k_full[st], kKTileBytes);
#pragma unroll
        for (int p = 0; p < L::kPanels; ++p)
          tma_load_3d(sbase + L::kK + (st * L::kPanels + p) * L::kPanelBytes, &kmap,
                      bar.k_full[st], p * 64, kvh, slot);
        k_last[st] = j;
        if (j >= kKvStages &&
            !mbar_wait(bar.v_empty[st], ((j >> 1) - 1) & 1, a.wait_limit_ns)) {
          report_error(a.err, kErrTimeout, kSitePrefillWait + 1);
          misc[1] = 1;
          break;
        }
        if (misc[1]) break;
        mbar_arrive_expect_tx(bar.v_full[st], kKTileBytes);
#pragma unroll
        for (int p = 0; p < L::kPanels; ++p)
          tma_load_3d(sbase + L::kV + (st * L::kPanels + p) * L::kPanelBytes, &vmap,
                      bar.v_full[st], p * 64, kvh, slot);
        v_last[st] = j;
      }
      // Every copy issued must land before the block may exit, whether or
      // not its consumer gave up on it (after a normal run these waits
      // return at once).
      mbar_wait(bar.q_full, 0, kDrainLimitNs);
      for (int s = 0; s < 2; ++s) {
        if (k_last[s] >= 0) mbar_wait(bar.k_full[s], (k_last[s] >> 1) & 1, kDrainLimitNs);
        if (v_last[s] >= 0) mbar_wait(bar.v_full[s], (v_last[s] >> 1) & 1, kDrainLimitNs);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && run) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kRows, kKeyTile, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(kRows, D, true);
      bool ok = mbar_wait(bar.q_full, 0, a.wait_limit_ns);
      if (!ok) report_error(a.err, kErrTimeout, kSitePrefillWait + 2);
      for (int j = 0; ok && j <= nkt; ++j) {
        if (j < nkt) {  // S_j = Q K_j^T
          const int st = j & 1;
          if (!mbar_wait(bar.k_full[st], (j >> 1) & 1, a.wait_limit_ns)) {
            report_error(a.err, kErrTimeout, kSitePrefillWait + 3);
            ok = false;
            break;
          }
          if (misc[1]) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem + kSCol0 + st * kKeyTile;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * L::kPanelBytes + (kk & 3) * 32;
            const uint64_t ad = smem_desc_sw128(sbase + L::kQ + off, 16, 1024);
            const uint64_t bd =
                smem_desc_sw128(sbase + L::kK + st * L::kPanels * L::kPanelBytes + off, 16, 1024);
            tc_mma_ss(d_tmem, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
          }
          tc_commit(bar.s_full[st]);
          tc_commit(bar.k_empty[st]);
        }
        if (j >= 1) {  // O += P_{j-1} V_{j-1}
          const int jj = j - 1;
          const int st = jj & 1;
          if (!mbar_wait(bar.p_full, jj & 1, a.wait_limit_ns) ||
              !mbar_wait(bar.v_full[st], (jj >> 1) & 1, a.wait_limit_ns)) {
            report_error(a.err, kErrTimeout, kSitePrefillWait + 4);
            ok = false;
            break;
          }
          if (misc[1]) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kKeyTile / 16; ++kk) {
            const uint32_t a_off = (kk >> 2) * L::kPanelBytes + (kk & 3) * 32;
            const uint64_t ad = smem_desc_sw128(sbase + L::kP + a_off, 16, 1024);
            // V stage: [128 keys][64 d] panels; 16 keys = 2 x 8-row groups.
            const uint64_t bd = smem_desc_sw128(
                sbase + L::kV + st * L::kPanels * L::kPanelBytes + kk * 16 * 128,
                L::kPanelBytes, 1024);
            tc_mma_ss(tmem + kOCol, ad, bd, idesc_o, (jj > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(bar.o_done);
          tc_commit(bar.v_empty[st]);
        }
      }
      if (!ok) misc[1] = 1;
      // Every MMA issued must finish before tensor memory is released.
      tc_commit(bar.drain);
      mbar_wait(bar.drain, 0, kDrainLimitNs);
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
    float m = -INFINITY, l = 0.f;
    bool ok = run;
    uint8_t* prow = sgen + L::kP + r * 128;
    for (int j = 0; ok && j < nkt; ++j) {
      // Exit decisions are warp-uniform: tcgen05.ld/st are warp-collective.
      const bool got = mbar_wait(bar.s_full[j & 1], (j >> 1) & 1, a.wait_limit_ns);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) report_error(a.err, kErrTimeout, kSitePrefillWait + 5);
        ok = false;
        break;
      }
      if (__shfl_sync(0xffffffffu, misc[1], 0)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float x[kKeyTile];
#pragma unroll
      for (int c = 0; c < kKeyTile / 32; ++c)
        tmem_ld_32x32b_x32(trow + kSCol0 + (j & 1) * kKeyTile + c * 32,
                           *reinterpret_cast<uint32_t(*)[32]>(&x[c * 32]));
      tmem_wait_ld();
      const int k0 = j * kKeyTile;
      const bool need_mask = (k0 + kKeyTile - 1 > pos_min) || (k0 + kKeyTile > ti.ctx);
      float mt = -INFINITY;
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < kKeyTile; ++c) {
          x[c] = (k0 + c <= lim) ? x[c] * sl2 : -INFINITY;
          mt = fmaxf(mt, x[c]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < kKeyTile; ++c) {
          x[c] *= sl2;
          mt = fmaxf(mt, x[c]);
        }
      }
      const float m_new = fmaxf(m, mt);
      const bool got_o = (j == 0) || mbar_wait(bar.o_done, (j - 1) & 1, a.wait_limit_ns);
      if (!__all_sync(0xffffffffu, got_o)) {
        if (lane == 0) report_error(a.err, kErrTimeout, kSitePrefillWait + 6);
        ok = false;
        break;
      }
      const bool need = m_new > m + kRescaleThreshold;  // true on the first tile
      if (__any_sync(0xffffffffu, need)) {
        const float alpha = need ? fast_exp2(m - m_new) : 1.f;
        if (j > 0) {
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
      // P = exp2(x - m) -> bf16, row r of two 128-byte-swizzled panels
      float rs = 0.f;
#pragma unroll
      for (int pnl = 0; pnl < 2; ++pnl) {
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float p0 = fast_exp2(x[pnl * 64 + ch * 8 + 2 * e] - m);
            const float p1 = fast_exp2(x[pnl * 64 + ch * 8 + 2 * e + 1] - m);
            rs += p0 + p1;
            w[e] = pack_bf16x2(p0, p1);
          }
          const uint32_t addr = smem_u32(prow) + pnl * L::kPanelBytes + ((ch ^ (r & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]),
                       "r"(w[1]), "r"(w[2]), "r"(w[3])
                       : "memory");
        }
      }
      l += rs;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar.p_full);
    }
    // ---- epilogue: O / l -> bf16
    if (ok && nkt > 0) {  // ok is warp-uniform here
      const bool got = mbar_wait(bar.o_done, (nkt - 1) & 1, a.wait_limit_ns);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) report_error(a.err, kErrTimeout, kSitePrefillWait + 7);
        ok = false;
      }
    }
    const bool epilogue = __shfl_sync(0xffffffffu, (ok && nkt > 0 && !misc[1]) ? 1 : 0, 0) != 0;
    if (epilogue) {
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
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, int G>
cudaError_t launch_t(const PrefillArgs& a, const CacheMaps& maps, const CUtensorMap& qmap,
                     cudaStream_t stream) {
  using L = PrefillLayout<D>;
  auto kern = prefill_kernel<D, G>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  constexpr int QT = kRows / G;
  // Upper bound on the number of tiles: sum_s ceil(Lq_s / QT) <= total/QT + num_seqs.
  const int64_t tiles = a.total_q / QT + a.num_seqs;
  const int64_t blocks = tiles * a.num_kv_heads;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kPrefillThreads);
  cfg.dynamicSmemBytes = L::kAlloc;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, qmap, maps.k_sw128, maps.v_sw128, a);
}

template <int D>
cudaError_t launch_d(const PrefillArgs& a, const CacheMaps& maps, const CUtensorMap& qmap,
                     cudaStream_t stream) {
  switch (a.num_q_heads / a.num_kv_heads) {
    case 1: return launch_t<D, 1>(a, maps, qmap, stream);
    case 2: return launch_t<D, 2>(a, maps, qmap, stream);
    case 4: return launch_t<D, 4>(a, maps, qmap, stream);
    case 8: return launch_t<D, 8>(a, maps, qmap, stream);
    case 16: return launch_t<D, 16>(a, maps, qmap, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, const CacheMaps& maps, const CUtensorMap& qmap,
                           int num_sms, cudaStream_t stream) {
  (void)num_sms;
  if (a.head_dim == 128) return launch_d<128>(a, maps, qmap, stream);
  if (a.head_dim == 64) return launch_d<64>(a, maps, qmap, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
