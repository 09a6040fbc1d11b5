/*
 * pkv.h -- C ABI of libpkv.so: attention over a paged KV cache on GB300
 * (sm_103a).
 *
 * The operations are the attention-layer steps of the vLLM / Aphrodite
 * attention backends described on the pages
 *   "aphrodite-engine/aphrodite/attention/backends/xformers.py"   (xformers.py)
 *   "vllm.v1.attention.backends.cpu_attn"                         (cpu_attn)
 *   "vllm.v1.attention.backends.utils"                            (backends.utils)
 * Each entry point cites the class or function there that defines it.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Memory: every pointer is a DEVICE pointer (or pinned host memory mapped
 *   into the device's address space where stated) unless marked "host".  The
 *   caller owns and allocates all buffers; the library allocates nothing per
 *   call and keeps no pointer after a call returns.
 * - Device: the kernels run on the device that owns `stream`; a call makes
 *   it current while it launches and restores the calling thread's previous
 *   current device before it returns.  The legacy and per-thread default
 *   streams belong to the current device.  While `stream` is being captured
 *   into a CUDA graph the library cannot ask it for its device (the query
 *   would end the capture), so it uses the current device: capture with the
 *   stream's device current.
 * - Ordering: work is enqueued on `stream` (a cudaStream_t; NULL = the legacy
 *   default stream) and the call returns without synchronising.  No call
 *   reads device memory on the host.  The decode calls launch their kernels
 *   as programmatic dependents of the kernel before them in the stream: they
 *   may be scheduled while it finishes, but read nothing before it has
 *   completed, so stream order holds as for ordinary launches.
 * - CUDA graphs: a call only launches kernels on `stream`, its arguments
 *   passed by value or living in device memory, so it can be captured in a
 *   CUDA graph and replayed on new contents of the same buffers (the
 *   backends.utils AttentionCGSupport levels).  Make one call per
 *   configuration on the device before capturing (the first call sets
 *   kernel attributes and resolves a driver entry point), and capture with
 *   the stream's device current.  kv_swap_blocks
 *   takes its pair list by value: a captured swap replays the pairs of the
 *   capture.
 * - Element type: fp16 or bf16 (pkv_attn_params.dtype) for queries, keys,
 *   values and outputs; the cache holds the same type, or 8-bit E4M3 codes
 *   (pkv_attn_params.kv_cache_dtype); arithmetic is fp32; outputs are
 *   rounded to nearest even.
 * - KV cache: kv_cache is [2][num_blocks][block_size * num_kv_heads *
 *   head_size] elements, contiguous (the shape of xformers.py
 *   XFormersImpl.forward and cpu_attn TorchSDPABackendImpl.forward).  Half 0
 *   holds keys, half 1 values.  Inside a block the layout is token-major,
 *   [block_size][num_kv_heads][head_size], so one slot holds one token's
 *   key (or value) row exactly as it appears in the `key` input.
 *   Slot s is token s % block_size of block s / block_size (cpu_attn,
 *   TorchSDPAMetadata.slot_mapping).
 * - Errors: argument errors are found on the host before anything is
 *   enqueued and return PKV_ERR_INVALID / PKV_ERR_UNSUPPORTED with nothing
 *   done.  A failed launch returns PKV_ERR_CUDA.  Indices that live in
 *   device memory (slots, block-table entries, lengths, copy pairs) are
 *   range-checked inside the kernels: a bad one is never dereferenced, the
 *   affected output is unspecified, and a sticky per-device error word
 *   records the first such event; read it with pkv_device_error().
 * - Empty work (num_tokens, num_seqs or num_pairs == 0) returns PKV_OK and
 *   enqueues nothing (the profiling run with an empty cache in xformers.py
 *   XFormersImpl.forward and cpu_attn TorchSDPABackendImpl.forward).
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKV_ABI_VERSION 3

typedef struct CUstream_st *pkv_stream_t; /* == cudaStream_t */

typedef enum pkv_status {
  PKV_OK = 0,
  PKV_ERR_INVALID = 1,     /* bad argument (null pointer, bad size, ...)   */
  PKV_ERR_UNSUPPORTED = 2, /* valid but not built (head size, dtype, ...)  */
  PKV_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed          */
  PKV_ERR_BOUNDS = 4,      /* pkv_device_error: an index was out of range   */
  PKV_ERR_TIMEOUT = 5      /* pkv_device_error: a bounded wait gave up      */
} pkv_status;

typedef enum pkv_dtype { PKV_FP16 = 0, PKV_BF16 = 1 } pkv_dtype;

/* Element type of the KV cache: the model dtype, or 8-bit E4M3 codes with a
 * per-layer scale for keys and one for values (the kv_cache_dtype, k_scale
 * and v_scale of xformers.py write_to_paged_cache / forward_decode and
 * cpu_attn forward_decode).  E4M3 is the "fn" form: sign, 4 exponent bits
 * (bias 7), 3 mantissa bits, no infinities, largest finite 448.  A key x is
 * stored as the code nearest to x / k_scale (quotient in fp32, ties to the
 * even code, saturating at +-448) and read back as code * k_scale; values
 * likewise with v_scale. */
typedef enum pkv_cache_dtype { PKV_CACHE_AUTO = 0, PKV_CACHE_FP8_E4M3 = 1 } pkv_cache_dtype;

/*
 * Per-layer attention constants: the constructor arguments of
 * xformers.py XFormersImpl / cpu_attn TorchSDPABackendImpl (num_heads,
 * head_size, scale, num_kv_heads, alibi_slopes, sliding_window) plus the
 * cache block size and the element type.
 *   num_heads % num_kv_heads == 0 (xformers.py XFormersImpl.__init__);
 *     query head h reads KV head h / (num_heads / num_kv_heads).
 *   head_size: 64 or 128.  block_size: 16 or 32 (others: PKV_ERR_UNSUPPORTED).
 *   scale: > 0, multiplies q.k before the softmax.
 *   alibi_slopes: device fp32[num_heads] or NULL; adds slope_h * (j - i) to
 *     the score of key position j for query position i
 *     (xformers.py _make_alibi_bias).
 *   sliding_window: W > 0 keeps keys i - W < j <= i; W <= 0 means none.
 *     It applies together with ALiBi when both are given.
 *   non_causal: 0 for decoder self-attention (causal); 1 for encoder /
 *     encoder-only attention, where every query row of a sequence sees all
 *     of its keys 0 .. L-1 (cpu_attn _run_sdpa_forward runs SDPA causally
 *     only for decoder attention).  Affects the prefill call; a decode query
 *     is the last position, so it sees the same keys either way.  A window
 *     together with non_causal is PKV_ERR_UNSUPPORTED.
 *   kv_cache_dtype: pkv_cache_dtype.  With PKV_CACHE_FP8_E4M3 the cache holds
 *     one byte per element ([2][num_blocks][block_size * num_kv_heads *
 *     head_size] codes) and k_scale, v_scale (finite, > 0) apply; every call
 *     supports it.  Decode computes in fp32 from the exact code values;
 *     prefill multiplies on fp16 operands (exact for the codes) with each
 *     128-row tile of bf16 queries rewritten as fp16 times a power of two
 *     chosen from the tile's largest magnitude, so no query overflows fp16.
 */
typedef struct pkv_attn_params {
  int32_t num_heads;
  int32_t num_kv_heads;
  int32_t head_size;
  int32_t block_size;
  int32_t dtype; /* pkv_dtype */
  float scale;
  const float *alibi_slopes;
  int32_t sliding_window;
  int32_t non_causal;
  int32_t kv_cache_dtype; /* pkv_cache_dtype */
  float k_scale;
  float v_scale;
} pkv_attn_params;

/*
 * kv_cache_write -- store each new token's key and value in its cache slot
 * (reshape_and_cache).  xformers.py XFormersImpl.forward and cpu_attn
 * TorchSDPABackendImpl.forward call PagedAttention.write_to_paged_cache with
 * key, value, the split cache and slot_mapping before any attention.
 *
 *   key, value    [num_tokens][num_kv_heads * head_size] elements, contiguous
 *   num_tokens    >= 0
 *   kv_cache      the cache (layout above), written in place
 *   num_blocks    blocks per cache half
 *   slot_mapping  int64[num_tokens]; slot < 0 is a padding token and is
 *                 skipped; slot >= num_blocks * block_size is recorded as a
 *                 bounds error and skipped.
 * Result is a bit-exact row copy.  Two tokens with the same slot race.
 */
pkv_status kv_cache_write(const void *key, const void *value,
                          int64_t num_tokens, void *kv_cache,
                          int64_t num_blocks, const int64_t *slot_mapping,
                          const pkv_attn_params *params, pkv_stream_t stream);

/*
 * paged_attn_decode -- one query token per sequence attending to its cached
 * K/V, gathered through block_tables (xformers.py XFormersImpl.forward ->
 * PagedAttention.forward_decode; cpu_attn TorchSDPABackendImpl.forward ->
 * forward_decode).  The new token was already written, so seq_lens counts it
 * and the query sits at position seq_len - 1 (xformers.py XFormersMetadata
 * note on context_len).  Split-KV: when the batch alone would leave SMs idle,
 * or a sequence is longer than 4096 keys, a sequence's keys are cut into
 * pieces processed in parallel whose partial softmax states are merged by a
 * second kernel (needs `workspace`; paged_attn_decode_workspace_size returns
 * 0 when no sequence is split).
 *
 *   out            [num_seqs][num_heads * head_size] elements
 *   query          [num_seqs][num_heads * head_size] elements
 *   block_tables   int32[num_seqs][max_blocks_per_seq]: physical block of
 *                  each logical block (cpu_attn TorchSDPAMetadata
 *                  .block_tables); entries past a sequence's length unused
 *   seq_lens       int32[num_seqs]; 0 gives an all-zero output row;
 *                  must be <= max_seq_len and <= max_blocks_per_seq *
 *                  block_size (else a bounds error is recorded)
 *   max_seq_len    host upper bound on seq_lens (sizes the grid)
 *   workspace      device scratch of at least
 *                  paged_attn_decode_workspace_size(...) bytes, 256-byte
 *                  aligned; may be NULL when that size is 0.  Contents on
 *                  entry do not matter; calls sharing a workspace must not
 *                  overlap on the GPU.
 */
pkv_status paged_attn_decode(void *out, const void *query, int32_t num_seqs,
                             const void *kv_cache, int64_t num_blocks,
                             const int32_t *block_tables,
                             int32_t max_blocks_per_seq,
                             const int32_t *seq_lens, int32_t max_seq_len,
                             const pkv_attn_params *params, void *workspace,
                             size_t workspace_bytes, pkv_stream_t stream);

/*
 * paged_attn_decode_noalloc -- paged_attn_decode for callers that cannot
 * allocate device memory.  The attention-backend pages have no counterpart of
 * this call; it exists for code that is handed its device buffers by a host
 * framework and may not call cudaMalloc itself (an inference-server plugin
 * working inside the framework's memory budget, or a serving loop where an
 * allocation would synchronise the device and stall the other streams).
 *
 * Arguments and results are those of paged_attn_decode without the
 * workspace: the split partials go to a static device array of
 * PKV_DECODE_STATIC_SCRATCH_BYTES bytes that is part of the library, so every
 * GPU that loads the library holds it until the process exits.  The call
 * allocates nothing and calls no allocating routine.
 *   - Sizes whose workspace (paged_attn_decode_workspace_size) exceeds
 *     PKV_DECODE_STATIC_SCRATCH_BYTES return PKV_ERR_UNSUPPORTED, nothing
 *     enqueued.
 *   - The array used is the one of the device the kernels run on (the
 *     stream's device; while `stream` is being captured, the current device,
 *     which must then be the stream's device, as for every call).
 *   - The first call on a device looks up the array's device address (a
 *     one-time set-up per device, with that device current); make that
 *     first call before any stream capture.
 *   - All calls share the one array, which keeps the last call's contents.
 *     Nothing in it needs to start at zero, but calls that overlap on the GPU
 *     (on different streams, or otherwise unordered) race on it.
 */
#define PKV_DECODE_STATIC_SCRATCH_BYTES (64u << 20)
pkv_status paged_attn_decode_noalloc(void *out, const void *query, int32_t num_seqs,
                                     const void *kv_cache, int64_t num_blocks,
                                     const int32_t *block_tables,
                                     int32_t max_blocks_per_seq,
                                     const int32_t *seq_lens, int32_t max_seq_len,
                                     const pkv_attn_params *params,
                                     pkv_stream_t stream);

/* Bytes of workspace paged_attn_decode needs for these sizes (host only,
 * never fails; 0 when no split is used).  Returns 0 for invalid params. */
size_t paged_attn_decode_workspace_size(int32_t num_seqs, int32_t max_seq_len,
                                        const pkv_attn_params *params);

/*
 * paged_attn_decode_multi -- a uniform batch of decodes of query_len tokens
 * each: speculative decoding's "decodes" of 1 + num_speculative_tokens
 * tokens (backends.utils AttentionCGSupport.UNIFORM_BATCH; the
 * reorder_batch_threshold of AttentionMetadataBuilder
 * ._init_reorder_batch_threshold pulls them to the front of the batch for
 * spec-as-decode kernels).  Token t of sequence b is the query at position
 * seq_lens[b] - query_len + t and attends to the keys up to and including
 * its own position (and within sliding_window), all read through the block
 * table; the cache write of the query_len new tokens comes first.  With
 * query_len = 1 this is paged_attn_decode.
 *
 *   out, query   [num_seqs * query_len][num_heads * head_size] elements,
 *                row b * query_len + t = token t of sequence b
 *   query_len    1 .. 64
 *   seq_lens     int32[num_seqs]: length including the query_len new
 *                tokens; 0 gives all-zero rows; 0 < seq_len < query_len,
 *                or above max_seq_len or max_blocks_per_seq * block_size,
 *                records PKV_ERR_BOUNDS and gives zero rows
 *   workspace    >= paged_attn_decode_multi_workspace_size(...) bytes of
 *                device scratch, 256-byte aligned (NULL when that is 0)
 *   Other arguments as paged_attn_decode (the fp8 cache included: products
 *   on fp16 operands, queries scaled by a power of two as in the prefill
 *   call); non_causal returns PKV_ERR_UNSUPPORTED.
 */
pkv_status paged_attn_decode_multi(void *out, const void *query, int32_t num_seqs,
                                   int32_t query_len, const void *kv_cache,
                                   int64_t num_blocks, const int32_t *block_tables,
                                   int32_t max_blocks_per_seq,
                                   const int32_t *seq_lens, int32_t max_seq_len,
                                   const pkv_attn_params *params, void *workspace,
                                   size_t workspace_bytes, pkv_stream_t stream);

/* Bytes of workspace paged_attn_decode_multi needs (host only; 0 when no
 * split is used or the arguments are not supported). */
size_t paged_attn_decode_multi_workspace_size(int32_t num_seqs, int32_t query_len,
                                              int32_t max_seq_len,
                                              const pkv_attn_params *params);

/*
 * Decode context parallelism (backends.utils CommonAttentionMetadata
 * dcp_local_seq_lens: the sequence lengths of the local rank in the decode
 * context parallel world; AttentionMetadataBuilder._init_reorder_batch_threshold
 * and use_cascade_attention take the group's size).  A group of
 * dcp_world_size ranks shares each sequence's cached tokens: token j lives on
 * rank j % dcp_world_size at local position j / dcp_world_size (the pages give
 * only the local lengths; this placement keeps them within one of each other).
 * Each rank computes its share with paged_attn_decode_dcp_partial, the ranks
 * all-gather the shares (rank-major), and paged_attn_dcp_combine merges them
 * into the output.
 *
 * paged_attn_decode_dcp_partial -- this rank's share of a (single- or
 * multi-token) decode: for every query row (as paged_attn_decode_multi:
 * rows b * query_len + t at positions seq_lens[b] - query_len + t) and head,
 * attention over the keys this rank holds, as
 *   part_o   fp32 [num_seqs * query_len * num_heads][head_size]: the
 *            softmax-normalised output over those keys (0 if none visible)
 *   part_ml  fp32 [num_seqs * query_len * num_heads][2]: the score maximum m
 *            (base-2 logits: scale * log2(e) * q.k + log2(e) * ALiBi) and the
 *            sum l of 2^(score - m); (-inf, 0) if no key is visible here.
 *   kv_cache, num_blocks, block_tables, max_blocks_per_seq: the rank's own
 *            pool and tables over its local positions
 *   seq_lens      int32[num_seqs]: GLOBAL lengths (the rank derives its local
 *                 lengths from them), max_seq_len their host bound
 *   dcp_world_size 1 .. 1024, dcp_rank 0 .. dcp_world_size - 1
 *   workspace     >= paged_attn_decode_dcp_workspace_size(...) bytes
 * Other arguments and errors as paged_attn_decode_multi.
 */
pkv_status paged_attn_decode_dcp_partial(float *part_o, float *part_ml, const void *query,
                                         int32_t num_seqs, int32_t query_len,
                                         const void *kv_cache, int64_t num_blocks,
                                         const int32_t *block_tables,
                                         int32_t max_blocks_per_seq, const int32_t *seq_lens,
                                         int32_t max_seq_len, int32_t dcp_world_size,
                                         int32_t dcp_rank, const pkv_attn_params *params,
                                         void *workspace, size_t workspace_bytes,
                                         pkv_stream_t stream);

size_t paged_attn_decode_dcp_workspace_size(int32_t num_seqs, int32_t query_len,
                                            int32_t max_seq_len, int32_t dcp_world_size,
                                            const pkv_attn_params *params);

/*
 * paged_attn_dcp_combine -- merge num_parts shares (the split combine, a3,
 * across ranks): out [num_rows][num_heads * head_size] elements from
 * part_o fp32 [num_parts][num_rows * num_heads][head_size] and part_ml fp32
 * [num_parts][num_rows * num_heads][2], rank-major as an all-gather of the
 * ranks' paged_attn_decode_dcp_partial outputs lays them out.  Shares with
 * l = 0 drop out; a row no share sees is zero.
 */
pkv_status paged_attn_dcp_combine(void *out, const float *part_o, const float *part_ml,
                                  int32_t num_parts, int64_t num_rows,
                                  const pkv_attn_params *params, pkv_stream_t stream);

/*
 * paged_attn_prefill_varlen -- packed prompts or prompt chunks attending
 * causally to their cached context plus themselves, all K/V read from the
 * paged cache (the chunk's own K/V are stored by kv_cache_write first).
 * xformers.py XFormersImpl.forward -> PagedAttention.forward_prefix (and,
 * with no cached context, _run_memory_efficient_xformers_forward); cpu_attn
 * flash_attn_varlen_func(out, query, key_cache, value_cache,
 * query_start_loc, seq_start_loc, max_query_len, max_seq_len, scale,
 * causal, block_tables, alibi_slopes).
 *
 *   out, query     [num_query_tokens][num_heads * head_size] elements
 *   num_query_tokens  rows of query / out; every cu_seqlens_q entry must lie
 *                  in [0, num_query_tokens] (else a bounds error is recorded
 *                  and the sequence skipped)
 *   cu_seqlens_q   int32[num_seqs + 1] (subquery_start_loc / query_start_loc)
 *   cu_seqlens_k   int32[num_seqs + 1] (seq_start_loc): sequence b has
 *                  L_b = cu_k[b+1] - cu_k[b] tokens, of which the last
 *                  q_b = cu_q[b+1] - cu_q[b] are its query rows, at positions
 *                  L_b - q_b + t (backends.utils CommonAttentionMetadata:
 *                  computed tokens = seq_lens - query lens).  q_b > L_b is
 *                  recorded as a bounds error and sequence b is skipped.
 *   max_query_len  host upper bound on q_b;  max_seq_len: on L_b
 *   block_tables   int32[num_seqs][max_blocks_per_seq]
 */
pkv_status paged_attn_prefill_varlen(
    void *out, const void *query, int64_t num_query_tokens, int32_t num_seqs,
    const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
    int32_t max_query_len, int32_t max_seq_len, const void *kv_cache,
    int64_t num_blocks, const int32_t *block_tables,
    int32_t max_blocks_per_seq, const pkv_attn_params *params,
    pkv_stream_t stream);

/*
 * kv_copy_blocks -- for every layer's cache and every pair (s, d), copy block
 * s to block d in both halves (xformers.py XFormersBackend.copy_blocks,
 * kv_caches: List[Tensor], src_to_dists: Dict[int, List[int]] flattened to
 * pairs).
 *
 *   kv_caches   host array of num_layers device pointers, each a cache of
 *               num_blocks blocks (same params); num_layers <= 256
 *   pairs       device int64[num_pairs][2] (src, dst).  Destinations must be
 *               unique and never also a source (undefined result otherwise);
 *               an index outside [0, num_blocks) is a bounds error.
 */
pkv_status kv_copy_blocks(void *const *kv_caches, int32_t num_layers,
                          int64_t num_blocks, const int64_t *pairs,
                          int64_t num_pairs, const pkv_attn_params *params,
                          pkv_stream_t stream);

/*
 * kv_swap_blocks -- dst[:, d] = src[:, s] for every pair, between two caches
 * (xformers.py XFormersBackend.swap_blocks(src_kv_cache, dst_kv_cache,
 * src_to_dst)).  A one-way move: swap out, later swap in.
 *
 *   src_cache, dst_cache  caches of src_num_blocks / dst_num_blocks blocks;
 *                         each is device memory or pinned host memory that
 *                         the device can address (cudaHostAlloc /
 *                         cudaHostRegister); anything else is
 *                         PKV_ERR_INVALID
 *   pairs                 HOST int64[num_pairs][2] (src, dst), checked on
 *                         the host against both block counts; destinations
 *                         must be unique.  Read during the call only.
 * The copy runs as a kernel on `stream` (reading or writing host memory over
 * the chip-to-host link), so it is stream-ordered like the other calls.
 */
pkv_status kv_swap_blocks(const void *src_cache, int64_t src_num_blocks,
                          void *dst_cache, int64_t dst_num_blocks,
                          const int64_t *pairs, int64_t num_pairs,
                          const pkv_attn_params *params, pkv_stream_t stream);

/* Static, never-NULL description of a status code. */
const char *pkv_status_string(pkv_status status);

/*
 * pkv_device_error -- synchronise the current device, then read and clear
 * its sticky device-side error word.  Returns PKV_OK when no kernel recorded
 * an error since the last read; otherwise PKV_ERR_BOUNDS or PKV_ERR_TIMEOUT,
 * with *detail (if non-NULL) set to the first offending index.  Diagnostic
 * call: it blocks the host, so keep it off hot paths.
 */
pkv_status pkv_device_error(int64_t *detail);

/*
 * pkv_check_wait_timeout -- a diagnostic of the library's failure handling.
 * Every wait in the kernels (on a TMA copy, an MMA, another warp) gives up
 * after a bound of one second, records PKV_ERR_TIMEOUT in the device error
 * word, releases what it holds and lets its CTA end, so a lost arrival
 * surfaces as a status instead of a hang.  This call launches one CTA whose
 * wait is on a barrier nothing will complete: about one second later the
 * error word holds PKV_ERR_TIMEOUT with detail `tag` (read it with
 * pkv_device_error), and the device stays usable.  No fault is involved.
 */
pkv_status pkv_check_wait_timeout(int64_t tag, pkv_stream_t stream);

/* PKV_ABI_VERSION of the built library. */
int32_t pkv_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
