/*
 * pkv.h -- C ABI of libpkv: attention over a paged KV cache on one B300
 * (sm_103a) GPU.
 *
 * The cache is cut into fixed blocks of 256 token slots (tuning guide
 * "Nano-vLLM性能调优实战", §1.1 KV缓存块配置: kvcache_block_size 256).  Each
 * sequence reaches its physically scattered blocks through a block table,
 * and sequences that share a prefix point at the same physical blocks
 * (ocdem.com nano-vllm article, §2.1 "基石PagedAttention 与 vLLM 的精髓").
 * Three calls make up the hot path of one attention layer (tuning guide
 * §2.2 缓存复用策略: a store_kvcache kernel writes new rows, attention then
 * reads the cache, variable-length batches allowed):
 *
 *   pkv_store_kvcache      scatter of new K/V rows into cache slots;
 *   pkv_decode_attention   one query token per sequence over its cache
 *                          (contexts split across blocks, pieces merged
 *                          by log-sum-exp inside the same kernel);
 *   pkv_prefill_attention  a chunk of query tokens per sequence over its
 *                          cached prefix plus the chunk itself, causal.
 *
 * Conventions shared by every call
 * --------------------------------
 * - All tensor arguments are DEVICE pointers on the current CUDA device,
 *   owned by the caller.  The library never frees them and keeps no
 *   reference after the call returns.  Base pointers must be 16-byte
 *   aligned and row strides (given in elements) must keep every row 16-byte
 *   aligned.
 * - bf16 is IEEE bfloat16 (the upper half of a binary32).  Index arrays are
 *   int32.
 * - Cache layout: k_cache and v_cache are bf16
 *   [num_blocks][256][num_kv_heads][head_dim], contiguous.  Token slot
 *   s = block_id * 256 + offset is the row k_cache + s * num_kv_heads * head_dim.
 * - block_tables is int32 [num_seqs][max_blocks_per_seq], contiguous; entry
 *   (s, i) is the physical block of logical block i of sequence s.  Entries
 *   past ceil(context_lens[s] / 256) are never read (pad them with -1).
 * - context_lens[s] counts every cached token of sequence s, including the
 *   ones stored by this step's pkv_store_kvcache.
 * - GQA: query head h reads KV head h / (num_q_heads / num_kv_heads).
 * - Supported: head_dim 64 or 128; num_q_heads a multiple of num_kv_heads
 *   with group size 1, 2, 4, 8 or 16.
 * - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 *   legacy default stream) and returns a pkv_status.  Shape, alignment and
 *   pointer checks run on the host before any launch; a failed check
 *   launches nothing.  Values that live on the device (block ids, slots,
 *   lengths) are checked by the kernels: an out-of-range value is skipped
 *   (its output row is written as zeros), never dereferenced, and recorded
 *   in a per-device error word that pkv_get_device_error reads.
 * - There is no CPU fallback: without a usable sm_103a device every call
 *   that launches a kernel returns PKV_ERR_CUDA.  (The host block manager at
 *   the end of this file is host code and needs no device.)
 */
#ifndef PKV_H_
#define PKV_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef void* pkv_stream_t; /* a cudaStream_t */

typedef enum pkv_status {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1,  /* null pointer, negative size, inconsistent shapes */
  PKV_ERR_UNSUPPORTED = 2,  /* head_dim, group size or alignment not supported */
  PKV_ERR_CUDA = 3,         /* a CUDA runtime call failed (no device, launch error) */
  PKV_ERR_DEVICE_CHECK = 4, /* a kernel found an out-of-range block id, slot or length */
  PKV_ERR_TIMEOUT = 5,      /* a bounded wait inside a kernel expired */
  PKV_ERR_NO_MEMORY = 6     /* the library could not allocate its workspace */
} pkv_status;

#define PKV_BLOCK_SIZE 256

/*
 * pkv_store_kvcache -- write new K/V rows into their cache slots.
 * (tuning guide §2.2: store_kvcache; ocdem.com article §2.1: slots live in
 * fixed-size blocks)
 *
 *   k, v          bf16 [num_tokens][*]: row i starts at k + i * k_row_stride
 *                 (v + i * v_row_stride) and holds num_kv_heads * head_dim
 *                 contiguous values (heads outer, head_dim inner).
 *   slot_mapping  int32 [num_tokens]: destination slot of row i, or -1 to
 *                 skip the row.  Any other value outside
 *                 [0, num_blocks * 256) is skipped and reported as
 *                 PKV_ERR_DEVICE_CHECK.  Two rows with the same slot: which
 *                 one lands is unspecified.
 *   k_cache, v_cache  bf16 [num_blocks][256][num_kv_heads][head_dim],
 *                 updated in place.  Slots that no row maps to are untouched.
 *
 * The copy is bit-exact.  num_tokens == 0 is a no-op.
 */
pkv_status pkv_store_kvcache(const void* k, const void* v, int64_t k_row_stride,
                             int64_t v_row_stride, const int32_t* slot_mapping,
                             int64_t num_tokens, void* k_cache, void* v_cache,
                             int64_t num_blocks, int32_t num_kv_heads, int32_t head_dim,
                             pkv_stream_t stream);

/*
 * pkv_decode_attention -- one query token per sequence attends to all
 * context_lens[s] cached tokens of its sequence (intelliparadigm.com
 * Nano-vLLM article, §7.1 增量解码; tuning guide §2.2 flash_attn_with_kvcache).
 *
 *   q             bf16 [num_seqs][*]: the query of sequence s starts at
 *                 q + s * q_row_stride and holds num_q_heads * head_dim values.
 *   k_cache, v_cache, num_blocks   the cache, as above.
 *   block_tables  int32 [num_seqs][max_blocks_per_seq].
 *   context_lens  int32 [num_seqs], 0 <= context_lens[s] <= 256 * max_blocks_per_seq.
 *   scale         softmax scale applied to q.k (typically 1/sqrt(head_dim)).
 *   out           bf16 [num_seqs][num_q_heads][head_dim], contiguous; written.
 *
 *   out[s][h] = sum_t softmax_t(scale * q[s][h] . K[s][t][g(h)]) * V[s][t][g(h)]
 *
 * with fp32 accumulation and bf16 (round to nearest even) output.  A
 * sequence with context 0 gets a zero output.  Contexts are split and
 * processed in parallel (flash decoding): the (sequence, KV head) contexts
 * of the batch, laid end to end, are cut into equal slices, one per block
 * of a grid that fills the GPU once (stream-K), so long and short contexts
 * balance; a context cut by a slice boundary has its pieces merged by
 * log-sum-exp by the block that finishes its last piece (one kernel launch
 * in all).  pkv_set_max_splits caps the grid.  The per-context arrival
 * counters and the partials live in a library-owned workspace on the
 * current device, allocated (and grown) with cudaMalloc on first need; call
 * pkv_reserve_workspace before capturing this call in a CUDA graph (replays
 * of the captured call are then correct: the counters carry a launch
 * generation kept on the device).  Calls on different streams that overlap
 * share that workspace and must be serialised by the caller.
 */
pkv_status pkv_decode_attention(const void* q, int64_t q_row_stride, const void* k_cache,
                                const void* v_cache, int64_t num_blocks,
                                const int32_t* block_tables, int32_t max_blocks_per_seq,
                                const int32_t* context_lens, int32_t num_seqs,
                                int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                float scale, void* out, pkv_stream_t stream);

/*
 * pkv_decode_attention_append -- one decode step's store and attention in one
 * kernel: the same result as pkv_store_kvcache(k_new, v_new, k_row_stride,
 * v_row_stride, slot_mapping, num_seqs, ...) followed by pkv_decode_attention
 * (tuning guide §2.2: store_kvcache writes the new rows, attention then reads
 * the cache; intelliparadigm.com article §7.1: each decode step appends one
 * token's K/V to the cache).
 *
 *   k_new, v_new  bf16 [num_seqs][*]: row s (at k_new + s * k_row_stride) is
 *                 sequence s's new token, the one at position
 *                 context_lens[s] - 1, num_kv_heads * head_dim values.
 *   slot_mapping  int32 [num_seqs]: the cache slot of that position, or -1
 *                 to store nothing for the sequence.  Any other value is
 *                 not stored and is reported as PKV_ERR_DEVICE_CHECK (the
 *                 attention then reads the pool row as it stands, as for -1).
 *   k_cache, v_cache  updated in place at those slots (bit-exact copies).
 *   other arguments as for pkv_decode_attention.
 *
 * The block that streams the chunk holding position context_lens[s] - 1 of
 * (sequence s, KV head h) copies head h of the new row in with the chunk,
 * writes it to the cache and uses it in place of the pool row it loaded, so
 * the step is one launch and the new rows cross HBM once.  The new token's
 * slot must not lie in another sequence's context (it is a private block's
 * next slot in a decode step).
 */
pkv_status pkv_decode_attention_append(const void* q, int64_t q_row_stride, const void* k_new,
                                       const void* v_new, int64_t k_row_stride,
                                       int64_t v_row_stride, const int32_t* slot_mapping,
                                       void* k_cache, void* v_cache, int64_t num_blocks,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* context_lens, int32_t num_seqs,
                                       int32_t num_q_heads, int32_t num_kv_heads,
                                       int32_t head_dim, float scale, void* out,
                                       pkv_stream_t stream);

/*
 * pkv_decode_attention_shared_prefix -- pkv_decode_attention for a batch whose
 * sequences share a prefix of whole blocks ("cascade" decode; ocdem.com
 * nano-vllm article §2.1: sequences with a common prefix point at the same
 * physical blocks, "高效的内存共享"; blog.hotdry.top "1200行代码挑战vLLM",
 * §性能优化 1 前缀缓存).  Same arguments and result as pkv_decode_attention,
 * plus
 *
 *   shared_blocks  the number of leading blocks every sequence shares: for
 *                  every s, block_tables[s][i] == block_tables[0][i] for
 *                  i < shared_blocks, and context_lens[s] >= 256 * shared_blocks
 *                  (0 <= shared_blocks <= max_blocks_per_seq; 0 is exactly
 *                  pkv_decode_attention).
 *
 * The shared blocks are read from HBM once for the whole batch instead of
 * once per sequence: a tcgen05 kernel attends the queries of all sequences
 * of a KV head (128 query rows per tile) to the shared keys, cut into key
 * ranges ("units") that run in parallel on the CTAs of one thread-block
 * cluster and are merged through distributed shared memory into one fp32
 * partial state per query row (max, sum, unnormalised output); the split-K
 * decode kernel, launched to overlap it, streams each sequence's private
 * tokens [256 * shared_blocks, context_lens[s]) only and merges the shared
 * partial state into the output by log-sum-exp once the first kernel is
 * done.  The result equals
 * pkv_decode_attention's up to fp32 rounding (softmax is invariant to how
 * the keys are grouped).  A sequence whose leading table entries differ from
 * row 0's, or whose context is shorter than the shared prefix, gets a zero
 * output and PKV_ERR_DEVICE_CHECK.  Workspace as for pkv_decode_attention
 * (plus the shared partial states and as many private ones, sized by
 * pkv_reserve_workspace too).
 * Two kernel launches on `stream`.
 */
pkv_status pkv_decode_attention_shared_prefix(const void* q, int64_t q_row_stride,
                                              const void* k_cache, const void* v_cache,
                                              int64_t num_blocks, const int32_t* block_tables,
                                              int32_t max_blocks_per_seq,
                                              const int32_t* context_lens, int32_t num_seqs,
                                              int32_t num_q_heads, int32_t num_kv_heads,
                                              int32_t head_dim, float scale,
                                              int32_t shared_blocks, void* out,
                                              pkv_stream_t stream);

/* Key ranges (the CTAs of one cluster) the shared prefix of
 * pkv_decode_attention_shared_prefix is cut into: 1, 2, 4, 8 or 16 (capped
 * at the prefix's 64-key tiles), or 0 for automatic (the default: up to 8,
 * about one CTA per SM).  Other values are PKV_ERR_INVALID_ARG.
 * Process-wide. */
pkv_status pkv_set_shared_prefix_units(int32_t units);

/*
 * pkv_prefill_attention -- chunked causal prefill over cached blocks
 * (tuning guide §3.2: chunks bounded by max_num_batched_tokens; §2.2:
 * variable-length batches; intelliparadigm.com article §7.1 预填充阶段).
 *
 *   q             bf16 [total_q][*]: query row r starts at q + r * q_row_stride
 *                 and holds num_q_heads * head_dim values.  Sequence s owns rows
 *                 cu_seqlens_q[s] .. cu_seqlens_q[s+1]-1 (its chunk, Lq rows).
 *                 q_row_stride * 2 bytes must be a multiple of 16.
 *   cu_seqlens_q  int32 [num_seqs + 1], non-decreasing, cu_seqlens_q[0] = 0,
 *                 cu_seqlens_q[num_seqs] = total_q.
 *   context_lens  int32 [num_seqs]: C = cached tokens including the chunk
 *                 (the chunk's K/V must already be stored); Lq <= C.
 *   out           bf16 [total_q][num_q_heads][head_dim], contiguous; written.
 *
 * Query i of the chunk sits at position C - Lq + i and attends to keys
 * 0 .. C - Lq + i (causal, aligned to the end of the context).  QK^T and PV
 * run on the tcgen05 tensor cores with fp32 accumulation in tensor memory;
 * P is rounded to bf16 before PV.  Output is bf16.
 */
pkv_status pkv_prefill_attention(const void* q, int64_t q_row_stride, const void* k_cache,
                                 const void* v_cache, int64_t num_blocks,
                                 const int32_t* block_tables, int32_t max_blocks_per_seq,
                                 const int32_t* cu_seqlens_q, const int32_t* context_lens,
                                 int32_t num_seqs, int64_t total_q, int32_t num_q_heads,
                                 int32_t num_kv_heads, int32_t head_dim, float scale, void* out,
                                 pkv_stream_t stream);

/*
 * pkv_decode_attention_noalloc -- pkv_decode_attention for callers that
 * cannot let the library allocate device memory: serving engines that hand
 * nearly all free memory to the KV block pool at start-up (a workspace the
 * library allocated later could fail, or escape the engine's accounting),
 * and processes whose device memory must all come from one caching
 * allocator.  The pages describe no such variant; it is an addition of this
 * library.
 *
 * Arguments, layouts, results and the split plan are those of
 * pkv_decode_attention.  The difference is where the split-K partials go:
 * into a 16 MiB array that the library defines statically on every device
 * that loads it (held until the process exits), not into a cudaMalloc'ed
 * workspace.  The call itself calls no cudaMalloc, cudaFree or allocating
 * library routine.
 *
 * - Size limit: the array holds a 2 MiB region of arrival counters (8 bytes
 *   per (sequence, KV head) pair after a 256-byte header, so at most 262144
 *   pairs: num_seqs * num_kv_heads <= 262144) and the partials,
 *   2 * B * G * (head_dim + 2) * 4 bytes, where G = num_q_heads /
 *   num_kv_heads and B is the decode kernel's grid (the blocks that fit on
 *   the GPU at once, a few per SM; at most num_seqs * num_kv_heads * cap
 *   under pkv_set_max_splits(cap)), which must fit in the remaining
 *   14 MiB - 256 bytes (a few MB on a 148-SM B300).  A batch beyond either
 *   limit returns PKV_ERR_UNSUPPORTED and launches nothing.
 * - Set-up: the first call on each device, with that device current, looks
 *   up the array's device address (cudaGetSymbolAddress); make that first
 *   call before any stream capture.  A failed lookup is retried by the next
 *   call.
 * - Sharing: every call on a device uses the same array, which keeps the
 *   last call's contents.  Nothing needs clearing: the kernel writes every
 *   partial it reads, and its arrival counters (zero at load) carry the
 *   number of the call that wrote them, so older values count as zero.
 *   Calls whose kernels overlap on the GPU (on different streams without
 *   ordering) race on it: serialise them.
 * - Device-side checks zero the output rows of out-of-range block ids or
 *   lengths and record PKV_ERR_DEVICE_CHECK (or PKV_ERR_TIMEOUT) in the
 *   library's error word, a static device variable too: pkv_get_device_error
 *   reports it as for every other call.
 */
pkv_status pkv_decode_attention_noalloc(const void* q, int64_t q_row_stride, const void* k_cache,
                                        const void* v_cache, int64_t num_blocks,
                                        const int32_t* block_tables, int32_t max_blocks_per_seq,
                                        const int32_t* context_lens, int32_t num_seqs,
                                        int32_t num_q_heads, int32_t num_kv_heads,
                                        int32_t head_dim, float scale, void* out,
                                        pkv_stream_t stream);

/* ------------------------------------------------------------------------
 * Helpers
 * --------------------------------------------------------------------- */

/* Human-readable name of a status code.  Never NULL. */
const char* pkv_status_string(pkv_status status);

/* Library version string, e.g. "pkv 0.1.0 sm_103a". */
const char* pkv_version(void);

/*
 * INT8 KV cache (intelliparadigm.com Nano-vLLM article §2.2,
 * "kv_cache_dtype: int8"; ocdem.com nano-vllm article §4.1 KV Cache 量化):
 * half the bytes of the bf16 cache for the same tokens.  Every (token, KV
 * head) row of head_dim values is held as int8 codes and one binary32 scale:
 *   scale = max_d |x_d| / 127,  code_d = nearest(x_d / scale), ties to even,
 * with IEEE binary32 division (codes in [-127, 127]; an all-zero row has
 * scale 0); a code stands for code * scale.  (The pages give no formula:
 * this is symmetric absmax quantisation per row.)
 *   k_codes, v_codes    int8 [num_blocks][num_kv_heads][256][head_dim]
 *   k_scales, v_scales  float32 [num_blocks][num_kv_heads][256]
 * all device pointers, 16-byte aligned, owned by the caller.  Each block
 * holds its KV heads one after another (the row of token slot
 * s = block * 256 + offset and head h is (block * num_kv_heads + h) * 256 +
 * offset), so a run of one head's tokens is contiguous.
 *
 * pkv_store_kvcache_int8 -- as pkv_store_kvcache (same k, v, strides and
 * slot_mapping rules, slot -1 skipped, out-of-range slots skipped and
 * reported as PKV_ERR_DEVICE_CHECK), writing each row's codes and scale.
 * The codes and scales are exactly those the definition above gives.
 * head_dim 64 or 128.
 */
pkv_status pkv_store_kvcache_int8(const void* k, const void* v, int64_t k_row_stride,
                                  int64_t v_row_stride, const int32_t* slot_mapping,
                                  int64_t num_tokens, int8_t* k_codes, int8_t* v_codes,
                                  float* k_scales, float* v_scales, int64_t num_blocks,
                                  int32_t num_kv_heads, int32_t head_dim, pkv_stream_t stream);

/*
 * pkv_decode_attention_int8 -- pkv_decode_attention over an INT8 cache: the
 * same arguments, with the bf16 cache replaced by codes and scales, and the
 * same result on the values the codes stand for (fp32 accumulation, bf16
 * output).  The split-K decode kernel of pkv_decode_attention (same
 * stream-K plan, in-kernel log-sum-exp merge, same workspace and the same
 * rules for CUDA graphs and overlapping calls) reading 64-token tiles of
 * codes and their scales; the codes become exact f16 values in registers,
 * the K scale multiplies each score and the V scale each probability.  Out-
 * of-range block ids or context lengths give a zero output for the sequence
 * and PKV_ERR_DEVICE_CHECK.
 */
pkv_status pkv_decode_attention_int8(const void* q, int64_t q_row_stride, const int8_t* k_codes,
                                     const int8_t* v_codes, const float* k_scales,
                                     const float* v_scales, int64_t num_blocks,
                                     const int32_t* block_tables, int32_t max_blocks_per_seq,
                                     const int32_t* context_lens, int32_t num_seqs,
                                     int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                     float scale, void* out, pkv_stream_t stream);

/*
 * pkv_prefill_attention_int8 -- pkv_prefill_attention over an INT8 cache:
 * the same arguments and chunk rules, with the bf16 cache replaced by codes
 * and scales, and the same causal attention on the values the codes stand
 * for (fp32 accumulation, bf16 output).  The tensor-core prefill kernel of
 * pkv_prefill_attention; each 64-key tile of codes and its scales is
 * loaded into shared memory and turned there into the bf16 values
 * code * scale (rounded to nearest even) before the matrix products, so the
 * result differs from the exact values only by that rounding, of the order
 * of the bf16 cache's own.  Allocates nothing.  Bad chunk lengths or block
 * ids give a zero output for the rows of the tile and PKV_ERR_DEVICE_CHECK.
 */
pkv_status pkv_prefill_attention_int8(const void* q, int64_t q_row_stride, const int8_t* k_codes,
                                      const int8_t* v_codes, const float* k_scales,
                                      const float* v_scales, int64_t num_blocks,
                                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                                      const int32_t* cu_seqlens_q, const int32_t* context_lens,
                                      int32_t num_seqs, int64_t total_q, int32_t num_q_heads,
                                      int32_t num_kv_heads, int32_t head_dim, float scale,
                                      void* out, pkv_stream_t stream);

/*
 * Synchronise `stream`, then read and clear the current device's error
 * word (a static device variable of the library, shared by every call on
 * that device; reading it allocates nothing).  *code receives PKV_OK or the first PKV_ERR_DEVICE_CHECK /
 * PKV_ERR_TIMEOUT recorded since the last read; *info (may be NULL) an
 * internal site code for diagnostics.  Returns PKV_ERR_CUDA if the
 * synchronisation failed.
 */
pkv_status pkv_get_device_error(pkv_stream_t stream, int32_t* code, int32_t* info);

/*
 * Cap the parallelism of pkv_decode_attention: with a cap n > 0 the decode
 * grid has at most num_seqs * num_kv_heads * n blocks, so a context of
 * average length is cut into at most about n + 1 pieces (0 = no cap, the
 * default: the grid fills the GPU).  A larger cap raises parallelism for few
 * long sequences; the merge costs a little extra memory traffic.
 * Process-wide.
 */
pkv_status pkv_set_max_splits(int32_t max_splits);

/*
 * Allocate, on the current device, the decode workspace for batches up to
 * the given shape (pkv_decode_attention and pkv_decode_attention_int8), so
 * that later calls of that size or smaller never allocate (required before
 * stream capture).  Grows, never shrinks.
 */
pkv_status pkv_reserve_workspace(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                                 int32_t max_blocks_per_seq);

/*
 * Bound, in nanoseconds, on every wait inside the kernels (default
 * 1000000000).  When a wait expires the kernel records PKV_ERR_TIMEOUT,
 * lets its own copies in flight land, releases its tensor memory and
 * returns; the context stays usable.  0 makes the first wait of every block
 * expire at once, which tests that path.  Process-wide.
 */
pkv_status pkv_set_wait_limit_ns(int64_t limit_ns);

/*
 * Kernel timing: while enabled, every kernel launch of the library is
 * bracketed by CUDA events on its own stream.  pkv_profiler_read
 * synchronises the recorded events and returns, for kernel `name`
 * ("store_kvcache", "decode", "decode_append", "shared_prefix", "prefill",
 * "store_kvcache_int8", "decode_int8", "prefill_int8"), the summed
 * duration in milliseconds and the launch count since the last reset.
 */
pkv_status pkv_profiler_enable(int32_t enable);
pkv_status pkv_profiler_reset(void);
pkv_status pkv_profiler_read(const char* name, double* total_ms, int64_t* launches);

/*
 * Host block manager
 * ------------------
 * Produces the block_tables, context_lens and slot_mapping arguments of the
 * calls above.  It runs on the host only: every pointer below is a HOST
 * pointer owned by the caller, no call touches a device, and the calls work
 * without a GPU.  It manages a pool of num_blocks cache blocks of 256 slots:
 *
 * - Blocks are handed out from the front of a free deque, ceil(tokens / 256)
 *   per sequence (intelliparadigm.com Nano-vLLM article, §2.1 动态分块内存管理).
 * - Each block carries a reference count; a block is free when its count is
 *   zero (blog.hotdry.top "1200行代码挑战vLLM", §2 内存管理策略: direct
 *   reference counting).
 * - Prefix cache (same article, §性能优化 1 前缀缓存): every FULL block is
 *   registered under a 64-bit key chained over the token ids of the whole
 *   prefix up to its end.  A new sequence whose prompt starts with cached full
 *   blocks shares them (their counts go up) instead of getting fresh ones;
 *   those tokens' K/V is already in the cache (ocdem.com nano-vllm article,
 *   §2.1: sequences with a common prefix point at the same physical blocks).
 *   A hit also compares the block's 256 stored token ids and its
 *   predecessor's key.  Only the leading run of cached blocks is reused.
 * - Delayed release (intelliparadigm.com article, §7.2 延迟释放策略): a block
 *   whose count reaches zero goes to the BACK of the free deque and keeps its
 *   cached content until it is handed out again, so a later prompt with the
 *   same prefix still finds it.  A freed sequence releases its blocks from
 *   last to first.
 *
 * Sequences are named by caller-chosen int64 ids.  Calls return
 * PKV_ERR_INVALID_ARG for a null manager or pointer, a negative size or an
 * unknown (or, for allocate, already present) sequence id, and
 * PKV_ERR_NO_MEMORY when the free blocks do not suffice; a failed call
 * changes nothing.  A manager is not thread-safe: serialise calls on it.
 */
typedef struct pkv_block_manager pkv_block_manager;

/* Create a manager of blocks 0 .. num_blocks - 1, all free (in that order).
 * num_blocks * 256 must fit in int32 (the slots are int32).  *out receives the
 * manager, to be released with pkv_bm_destroy. */
pkv_status pkv_bm_create(int32_t num_blocks, pkv_block_manager** out);
void pkv_bm_destroy(pkv_block_manager* bm);

/* Number of blocks with count zero (cached or not); 0 for a null manager. */
int32_t pkv_bm_num_free_blocks(const pkv_block_manager* bm);

/* Reference count of `block` (number of live sequences whose table holds it),
 * or -1 for an index out of range. */
int32_t pkv_bm_ref_count(const pkv_block_manager* bm, int32_t block);

/* Add sequence seq_id with its prompt tokens[0 .. num_tokens).  Leading full
 * blocks found in the prefix cache are shared; the rest come fresh from the
 * free deque.  *num_cached_tokens (may be NULL) receives how many leading
 * tokens already have their K/V in the cache (a multiple of 256): the caller
 * stores and computes only tokens [*num_cached_tokens, num_tokens), whose
 * slots pkv_bm_slots gives. */
pkv_status pkv_bm_allocate(pkv_block_manager* bm, int64_t seq_id, const int32_t* tokens,
                           int32_t num_tokens, int32_t* num_cached_tokens);

/* Append n tokens to sequence seq_id (a prefill chunk, or one decoded token),
 * opening new blocks as needed; a block that becomes full enters the prefix
 * cache.  slots (may be NULL) receives the n cache slots, the slot_mapping
 * of pkv_store_kvcache. */
pkv_status pkv_bm_append(pkv_block_manager* bm, int64_t seq_id, const int32_t* tokens, int32_t n,
                         int32_t* slots);

/* One decode step: append tokens[s] to sequence seq_ids[s] for every s
 * (distinct, known ids) and write its slot to slot_mapping[s], the
 * slot_mapping of that step's pkv_store_kvcache.  Fails as a whole
 * (PKV_ERR_NO_MEMORY) when fewer blocks are free than the sequences whose
 * last block is full.  Same as num_seqs calls of pkv_bm_append with one
 * token each, in one call. */
pkv_status pkv_bm_append_decode(pkv_block_manager* bm, const int64_t* seq_ids, int32_t num_seqs,
                                const int32_t* tokens, int32_t* slot_mapping);

/* One decode step in one call: pkv_bm_append_decode, then the step's
 * block_tables [num_seqs][max_blocks] and context_lens [num_seqs] as
 * pkv_bm_block_tables gives them.  Fails as a whole, changing nothing:
 * PKV_ERR_INVALID_ARG for an unknown or repeated id or a table that would
 * outgrow max_blocks, PKV_ERR_NO_MEMORY when too few blocks are free. */
pkv_status pkv_bm_decode_step(pkv_block_manager* bm, const int64_t* seq_ids, int32_t num_seqs,
                              const int32_t* tokens, int32_t max_blocks, int32_t* slot_mapping,
                              int32_t* block_tables, int32_t* context_lens);

/* Drop sequence seq_id: every block of its table loses one count. */
pkv_status pkv_bm_free(pkv_block_manager* bm, int64_t seq_id);

/* Fill block_tables [num_seqs][max_blocks] (row s: the physical blocks of
 * sequence seq_ids[s] in logical order, then -1) and context_lens[num_seqs]
 * (its token count): the arguments of pkv_decode_attention and
 * pkv_prefill_attention.  A sequence with more than max_blocks blocks is
 * PKV_ERR_INVALID_ARG. */
pkv_status pkv_bm_block_tables(const pkv_block_manager* bm, const int64_t* seq_ids,
                               int32_t num_seqs, int32_t max_blocks, int32_t* block_tables,
                               int32_t* context_lens);

/* slots[0 .. end - begin) = cache slots of tokens [begin, end) of sequence
 * seq_id (slot = block * 256 + position in block); end must not exceed its
 * token count. */
pkv_status pkv_bm_slots(const pkv_block_manager* bm, int64_t seq_id, int32_t begin, int32_t end,
                        int32_t* slots);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
