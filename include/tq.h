/*
 * tq.h -- C ABI of the TurboQuant KV-cache store and fused decode attention
 * for NVIDIA GB300 (sm_103a).
 *
 * Sources (cited by page title and section):
 *   [TQC] vLLM API docs, "vllm.model_executor.layers.quantization.turboquant",
 *         class TurboQuantConfig: docstring (presets, seed rule, norm
 *         correction), key_fp8, mse_bits, key_packed_size, value_packed_size,
 *         slot_size, slot_size_aligned, from_cache_dtype.
 *   [PR]  prhub digest of vLLM PR #39931, "TurboQuant supports hybrid models
 *         + fixes page-size alignment", key source snippet
 *         (vllm/platforms/interface.py, _align_hybrid_block_size).
 *   [ART] hnwysp.cn TurboQuant article, "Direction 1: fused Triton kernels"
 *         (rotate the query instead of the keys; online softmax block by
 *         block; no materialised fp16 K/V).
 *
 * Conventions for every call:
 *   - Pointers named *_dev are device pointers (cudaMalloc'd or torch CUDA
 *     memory); everything else is host memory.  The caller owns all buffers;
 *     the library allocates nothing and keeps no state between calls.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Device work is asynchronous on that stream; a TQ_OK return
 *     means the work was validated and enqueued.
 *   - Calls never abort and never fall back to the CPU.  A non-OK status is
 *     returned for invalid arguments before anything is enqueued, or
 *     TQ_ERR_CUDA when a launch fails; tq_last_error() then describes it.
 *   - Element layouts are dense row-major (innermost index last):
 *       keys / values   bf16  [num_tokens, num_kv_heads, head_dim]
 *       queries         bf16  [num_seqs, num_q_heads, head_dim]
 *       decode output   fp32  [num_seqs, num_q_heads, head_dim]
 *       slot_mapping    int64 [num_tokens]   slot = block * block_size + offset
 *       block_table     int32 [num_seqs, max_blocks_per_seq]
 *       seq_lens        int32 [num_seqs]
 *       cu_seqlens      int32 [num_seqs + 1] (prefix sums of seq_lens)
 *   - Grouped-query attention: query head hq reads KV head hq / (Hq / H).
 */
#ifndef TQ_H
#define TQ_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TQ_API __attribute__((visibility("default")))
#else
#define TQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum tq_status {
    TQ_OK = 0,
    TQ_ERR_INVALID_ARG = 1,     /* null pointer, bad size, inconsistent geometry */
    TQ_ERR_UNKNOWN_PRESET = 2,  /* preset name not one of the four [TQC] presets  */
    TQ_ERR_UNSUPPORTED = 3,     /* valid for the pages but not built here (e.g. d=96) */
    TQ_ERR_WORKSPACE = 4,       /* decode workspace missing or too small */
    TQ_ERR_OUT_OF_RANGE = 5,    /* reported through tq_cache.error_flags, see below */
    TQ_ERR_CUDA = 6             /* a CUDA launch or query failed */
} tq_status;

#define TQ_MAX_HEAD_DIM 256
#define TQ_MAX_CENTROIDS 16
/* most sequences of one decode or dequant call: their kernels take one grid
 * row per sequence (TQ_ERR_UNSUPPORTED above) */
#define TQ_MAX_SEQS 65535

/* Bits a kernel ORs into *tq_cache.error_flags when it meets bad input.  The
 * offending access is skipped; nothing outside the given buffers is touched. */
#define TQ_FLAG_SLOT_OUT_OF_RANGE  1u  /* slot_mapping[t] >= num_blocks * block_size */
#define TQ_FLAG_BLOCK_OUT_OF_RANGE 2u  /* block_table entry < 0 or >= num_blocks */
#define TQ_FLAG_SEQ_TOO_LONG       4u  /* seq_len > max_blocks_per_seq * block_size or > max_seq_len */
#define TQ_FLAG_WAIT_TIMEOUT       8u  /* a decode kernel gave up waiting (about 1 s) for a staged
                                          chunk; that call's outputs are not valid */

/*
 * Quantiser configuration: [TQC] TurboQuantConfig fields plus every derived
 * size and the Lloyd-Max codebook.  Plain data, filled by tq_config_init or
 * tq_config_from_preset; the caller owns it and may copy it freely.
 *
 *   key_fp8            key_quant_bits == 8: FP8 e4m3 keys, no rotation or norm
 *   mse_bits           codebook width: key bits, or value bits in FP8 mode
 *   key_packed_size    d (FP8) or ceil(d * key_bits / 8) + 2   (indices | fp16 norm)
 *   value_packed_size  ceil(d * value_bits / 8) + 4            (codes | fp16 scale | fp16 zero)
 *   slot_size          key_packed_size + value_packed_size; slot_size_aligned rounds it up to even
 *   centroids          2^mse_bits Lloyd-Max levels of N(0, 1/d), ascending, fp32
 *   boundaries         the 2^mse_bits - 1 midpoints between them, fp32
 */
typedef struct tq_config {
    int32_t head_dim;
    int32_t key_quant_bits;
    int32_t value_quant_bits;
    int32_t norm_correction;
    uint64_t seed;
    int32_t key_fp8;
    int32_t mse_bits;
    int32_t key_mse_bits;
    int32_t n_centroids;
    int32_t key_packed_size;
    int32_t value_packed_size;
    int32_t slot_size;
    int32_t slot_size_aligned;
    float centroids[TQ_MAX_CENTROIDS];
    float boundaries[TQ_MAX_CENTROIDS - 1];
    int32_t lloyd_max_iterations;
} tq_config;

/*
 * One layer's paged cache: uint8 [num_blocks, block_size, num_kv_heads,
 * slot_size_aligned] with consecutive blocks block_stride_bytes apart.
 * Slot (token at `slot`, head h) starts at
 *     data_dev + (slot / block_size) * block_stride_bytes
 *              + ((slot % block_size) * num_kv_heads + h) * slot_size_aligned.
 * block_stride_bytes = 0 means dense blocks; a larger stride (a multiple of
 * 16) lets TQ pages share the lcm-unified page size of hybrid models ([PR]).
 * layer_idx selects the random signs: seed + layer_idx * 1337 ([TQC]).
 * error_flags_dev, if not NULL, is a device uint32 that kernels OR the
 * TQ_FLAG_* bits into; it is never cleared by the library.
 */
typedef struct tq_cache {
    uint8_t* data_dev;
    int64_t num_blocks;
    int32_t block_size;
    int32_t num_kv_heads;
    int32_t layer_idx;
    int32_t reserved0;
    int64_t block_stride_bytes;
    uint32_t* error_flags_dev;
} tq_cache;

/*
 * tq_config_init -- [TQC] TurboQuantConfig(head_dim, key_quant_bits,
 * value_quant_bits, seed, norm_correction) with its derived sizes.  Solves
 * the Lloyd-Max quantiser of N(0,1) by fixed-point iteration in fp64 (cells'
 * conditional means and midpoint boundaries, symmetric about 0, until no level
 * moves by 1e-13), scales it by 1/sqrt(d) and rounds to fp32.  Host only.
 *   head_dim: power of two in [16, 256] (else TQ_ERR_UNSUPPORTED; the pages'
 *             d=96 example has no Walsh-Hadamard transform of that order)
 *   key_quant_bits: 3, 4 (Lloyd-Max keys) or 8 (FP8 keys); value bits: 3 or 4
 *   out: written on TQ_OK only.
 */
TQ_API tq_status tq_config_init(int32_t head_dim, int32_t key_quant_bits, int32_t value_quant_bits,
                         int32_t norm_correction, uint64_t seed, tq_config* out);

/*
 * tq_config_from_preset -- [TQC] from_cache_dtype(cache_dtype, head_dim) with
 * the default seed 42.  Presets: turboquant_k8v4 (8/4, no NC),
 * turboquant_4bit_nc (4/4, NC), turboquant_k3v4_nc (3/4, NC),
 * turboquant_3bit_nc (3/3, NC).  Unknown names return TQ_ERR_UNKNOWN_PRESET
 * and tq_last_error() lists the valid ones.  Host only.
 */
TQ_API tq_status tq_config_from_preset(int32_t head_dim, const char* preset, tq_config* out);

/*
 * tq_layer_signs -- the random-sign diagonal of one layer's rotation
 * Pi = H_d diag(s) / sqrt(d): s_i = -1 where draw i of a SplitMix64 stream
 * seeded with seed + layer_idx * 1337 has its top bit set, else +1.
 * signs_out: host int8 [head_dim].  Host only.
 */
TQ_API tq_status tq_layer_signs(const tq_config* cfg, int32_t layer_idx, int8_t* signs_out);

/*
 * tq_store_kv -- quantise and write num_tokens tokens into the paged cache.
 * Per (token, KV head): keys are rotated by Pi, scaled to unit norm and
 * bucketed against the boundaries (indices packed LSB-first, then the fp16
 * norm), or stored as FP8 e4m3 (round to nearest even, saturating); values
 * get uniform codes with fp16 scale = (max - min) / (2^bits - 1) and fp16
 * zero = min, packed LSB-first, then scale, then zero ([TQC] slot layout
 * [key_packed | value_packed]; pad byte 0).
 *   k_dev, v_dev: bf16 [num_tokens, cache->num_kv_heads, head_dim]
 *   slot_mapping_dev: int64 [num_tokens]; negative slots are skipped
 *   cache: descriptor (host struct, device data)
 * num_tokens == 0 enqueues nothing and returns TQ_OK.
 */
TQ_API tq_status tq_store_kv(const tq_config* cfg, const void* k_dev, const void* v_dev, int64_t num_tokens,
                      const int64_t* slot_mapping_dev, const tq_cache* cache, void* stream);

/*
 * tq_decode_workspace_size -- bytes of device workspace tq_decode_attention
 * needs for these sizes and split count (num_splits = 0: the count the call
 * would choose for the current device).  The workspace must be zero-filled
 * once before its first use; every decode call leaves it ready for the next.
 */
TQ_API size_t tq_decode_workspace_size(const tq_config* cfg, int32_t num_seqs, int32_t num_q_heads,
                                int32_t num_kv_heads, int32_t block_size, int32_t max_seq_len,
                                int32_t num_splits);

/*
 * tq_decode_attention -- one decode step of attention read straight from the
 * packed cache ([ART] Direction 1): for each sequence s and query head hq,
 *     out[s, hq] = sum_t softmax_t(sm_scale * q[s,hq] . k_hat_t) * v_hat_t
 * over the seq_lens[s] cached tokens found through block_table, where k_hat
 * = vec_norm * Pi^T c~ (c~ divided by ||c~|| under norm correction, [TQC]) or
 * the FP8 key, and v_hat = scale * code + zero.  Keys are never expanded: the
 * query is rotated once (Pi q) and scored against centroids.  The history is
 * cut into num_splits ranges (0 = chosen from the SM count) whose partial
 * softmax states are merged by log-sum-exp; the result depends on the split
 * count only through rounding (the tensor-core path rounds the softmax
 * weights to fp16 relative to each split's running maximum).
 *   q_dev: bf16 [num_seqs, num_q_heads, head_dim]; num_q_heads % num_kv_heads == 0
 *   block_table_dev: int32 [num_seqs, max_blocks_per_seq]
 *   seq_lens_dev: int32 [num_seqs]; each <= max_seq_len; 0 gives a zero row
 *   sm_scale: softmax scale; <= 0 selects 1/sqrt(head_dim)
 *   out_dev: fp32 [num_seqs, num_q_heads, head_dim]
 *   workspace_dev: >= tq_decode_workspace_size(...) bytes, 16-byte aligned,
 *                  zero-filled before first use (see above)
 * Requires block_size % 16 == 0, a 16-byte aligned cache and num_seqs <=
 * TQ_MAX_SEQS.  Concurrent calls sharing one workspace race.
 */
TQ_API tq_status tq_decode_attention(const tq_config* cfg, const void* q_dev, int32_t num_seqs,
                              int32_t num_q_heads, const tq_cache* cache,
                              const int32_t* block_table_dev, int32_t max_blocks_per_seq,
                              const int32_t* seq_lens_dev, int32_t max_seq_len, float sm_scale,
                              int32_t num_splits, float* out_dev, void* workspace_dev,
                              size_t workspace_bytes, void* stream);

/*
 * tq_dequant -- expand cached tokens back to bf16 K and V for continuation
 * prefill ([TQC] mse_bits docstring: centroids serve the continuation-prefill
 * dequant).  Token j of sequence s is written to row cu_seqlens[s] + j of
 *   k_out_dev, v_out_dev: bf16 [cu_seqlens[num_seqs], num_kv_heads, head_dim]
 * with k_hat = vec_norm * Pi^T c~ (NC: c~ / ||c~||) or the FP8 key, and
 * v_hat = scale * code + zero, each computed in fp32 and rounded to bf16.
 *   cu_seqlens_dev: int32 [num_seqs + 1], host-visible bound max_seq_len on
 *   every sequence length.
 * num_seqs <= TQ_MAX_SEQS.
 */
TQ_API tq_status tq_dequant(const tq_config* cfg, const tq_cache* cache, const int32_t* block_table_dev,
                     int32_t max_blocks_per_seq, const int32_t* cu_seqlens_dev, int32_t num_seqs,
                     int32_t max_seq_len, void* k_out_dev, void* v_out_dev, void* stream);

/*
 * Ring-buffered store ([ART] hnwysp.cn article, "full_tq zero-allocation
 * mode", item 3 "the write path": new decode tokens first enter an exact
 * bf16 ring of 128 tokens and only a full ring is compressed, a whole block
 * at a time).  With a ring of R tokens, a sequence of L tokens keeps the
 * positions [0, R floor(L/R)) packed in the paged cache and the rest exact,
 * position p in ring row p mod R of
 *   ring_k_dev, ring_v_dev: bf16 [num_seqs, R, num_kv_heads, head_dim]
 * (reading: ring blocks are aligned to multiples of R from position 0; the
 * caller owns the rings, which need no initialisation).
 */
#define TQ_RING_TOKENS 128     /* the ring length the article names */
#define TQ_RING_MAX_TOKENS 128 /* largest ring the decode accepts */

/* Device workspace bytes of tq_ring_append for num_seqs sequences. */
TQ_API size_t tq_ring_workspace_size(int32_t num_seqs);

/*
 * tq_ring_append -- append new tokens to ring-buffered sequences.  Sequence
 * s holds seq_lens_dev[s] tokens before the call (negative: it takes none)
 * and its new tokens are rows cu_new_dev[s] .. cu_new_dev[s+1]-1 of
 *   k_dev, v_dev: bf16 [num_tokens, num_kv_heads, head_dim] (16-byte aligned)
 * at positions seq_lens[s], seq_lens[s] + 1, ...  Every ring block the new
 * tokens complete is quantised exactly as tq_store_kv would quantise its
 * tokens and written to its positions through block_table_dev (int32
 * [num_seqs, max_blocks_per_seq]); the tokens after the last whole block
 * are copied into the ring.  A decode step is one token per sequence
 * (cu_new = 0, 1, ..., num_seqs); a prefill is the prompt with seq_lens 0.
 *   ring_tokens: R in [1, TQ_RING_MAX_TOKENS]; the same R for every call
 *   workspace_dev: >= tq_ring_workspace_size(num_seqs) bytes, 16-byte
 *                  aligned, no initialisation
 * A sequence whose new length exceeds max_blocks_per_seq * block_size, or
 * whose cu_new range leaves [0, num_tokens], takes no tokens and sets
 * TQ_FLAG_SEQ_TOO_LONG; a block_table entry outside the cache sets
 * TQ_FLAG_BLOCK_OUT_OF_RANGE and that token is not written.  Concurrent
 * calls sharing one workspace race.
 */
TQ_API tq_status tq_ring_append(const tq_config* cfg, const void* k_dev, const void* v_dev, int64_t num_tokens,
                                const int32_t* cu_new_dev, int32_t num_seqs, const int32_t* seq_lens_dev,
                                void* ring_k_dev, void* ring_v_dev, int32_t ring_tokens, const tq_cache* cache,
                                const int32_t* block_table_dev, int32_t max_blocks_per_seq, void* workspace_dev,
                                size_t workspace_bytes, void* stream);

/*
 * tq_ring_step -- one decode step of ring-buffered sequences in a single
 * kernel and without workspace: the same result as tq_ring_append with one
 * new token per sequence (cu_new = 0, 1, ..., num_seqs).
 *   k_dev, v_dev: bf16 [num_seqs, num_kv_heads, head_dim], row s the new
 *                 token of sequence s (16-byte aligned)
 *   seq_lens_dev: int32 [num_seqs], tokens of s before the step (negative:
 *                 no token for s)
 * The token completes a ring block when (seq_lens[s] + 1) mod R = 0: then
 * ring rows 0 .. R-2 and the token are quantised into positions
 * seq_lens[s] + 1 - R .. seq_lens[s]; otherwise the token is copied into
 * ring row seq_lens[s] mod R.  Flags and ring arguments as tq_ring_append.
 */
TQ_API tq_status tq_ring_step(const tq_config* cfg, const void* k_dev, const void* v_dev, int32_t num_seqs,
                              const int32_t* seq_lens_dev, void* ring_k_dev, void* ring_v_dev, int32_t ring_tokens,
                              const tq_cache* cache, const int32_t* block_table_dev, int32_t max_blocks_per_seq,
                              void* stream);

/*
 * tq_decode_ring_workspace_size -- as tq_decode_workspace_size, for
 * tq_decode_attention_ring (one more partial state per query head).
 */
TQ_API size_t tq_decode_ring_workspace_size(const tq_config* cfg, int32_t num_seqs, int32_t num_q_heads,
                                            int32_t num_kv_heads, int32_t block_size, int32_t max_seq_len,
                                            int32_t num_splits);

/*
 * tq_decode_attention_ring -- tq_decode_attention for ring-buffered
 * sequences (the article's hybrid mode: history from the compressed store,
 * the newest tokens from the exact ring).  seq_lens_dev[s] = L counts all
 * of a sequence's tokens: the packed positions [0, R floor(L/R)) are read
 * from the cache as tq_decode_attention reads them, and ring rows 0 .. (L
 * mod R) - 1 exactly (fp32 scores and sums); one softmax covers both.
 * Arguments as tq_decode_attention, plus the rings of tq_ring_append
 * (16-byte aligned) and R; workspace >= tq_decode_ring_workspace_size(...).
 * Up to 8 query heads per KV head.
 */
TQ_API tq_status tq_decode_attention_ring(const tq_config* cfg, const void* q_dev, int32_t num_seqs,
                                          int32_t num_q_heads, const tq_cache* cache,
                                          const int32_t* block_table_dev, int32_t max_blocks_per_seq,
                                          const int32_t* seq_lens_dev, int32_t max_seq_len, float sm_scale,
                                          int32_t num_splits, const void* ring_k_dev, const void* ring_v_dev,
                                          int32_t ring_tokens, float* out_dev, void* workspace_dev,
                                          size_t workspace_bytes, void* stream);

/*
 * tq_hybrid_page -- per-token page geometry of a TQ layer in a hybrid model
 * ([PR] _align_hybrid_block_size snippet).  The TQ page of one token is
 * num_kv_heads * slot_size_aligned bytes (reading of TQFullAttentionSpec with
 * block_size=1); an unquantised skip layer's page is 2 (K and V) *
 * num_kv_heads * head_dim * skip_dtype_bytes; with skip layers present the
 * unified page is lcm(tq_page, skip_page), else tq_page.
 *   skip_dtype_bytes: element size of the skip layers' cache (2 for bf16),
 *                     0 = no skip layers
 *   page_bytes_out: the unified page size in bytes
 *   tokens_per_page_out: TQ tokens that fill one unified page
 *                        (page / tq_page: the TQ block size whose blocks are
 *                        exactly one page, dense stride)
 * Host only.
 */
TQ_API tq_status tq_hybrid_page(const tq_config* cfg, int32_t num_kv_heads, int32_t skip_dtype_bytes,
                                int64_t* page_bytes_out, int32_t* tokens_per_page_out);

/*
 * tq_dense_decode_workspace_size / tq_dense_decode_attention -- the
 * comparison path of [ART] "Obstacle 1": attention over K and V that were
 * first expanded to full precision (here bf16, by tq_dequant), instead of the
 * fused decode over the packed cache.  For each sequence s and query head hq,
 *     out[s, hq] = sum_t softmax_t(sm_scale * q[s,hq] . k_t) * v_t
 * over rows t = cu_seqlens[s] .. cu_seqlens[s+1] - 1 of k and v, with query
 * head hq reading KV head hq / (num_q_heads / num_kv_heads); products and
 * sums in fp32, softmax by split-KV online softmax and a log-sum-exp merge.
 *   q_dev: bf16 [num_seqs, num_q_heads, head_dim], 16-byte aligned
 *   k_dev, v_dev: bf16 [cu_seqlens[num_seqs], num_kv_heads, head_dim] (the
 *                 layout tq_dequant writes), 16-byte aligned
 *   cu_seqlens_dev: int32 [num_seqs + 1]; every length <= max_seq_len
 *   sm_scale: <= 0 selects 1/sqrt(head_dim)
 *   out_dev: fp32 [num_seqs, num_q_heads, head_dim]
 *   workspace_dev: >= tq_dense_decode_workspace_size(...) bytes, 16-byte
 *                  aligned; every call writes all of it that it reads
 * head_dim a power of two in [16, 256]; 1 to 8 query heads per KV head;
 * num_seqs <= TQ_MAX_SEQS.  The workspace size depends on the device's SM
 * count (the split count is chosen from it); query it on the device used.
 * Asynchronous on `stream`; invalid arguments return before anything is
 * enqueued.
 */
TQ_API size_t tq_dense_decode_workspace_size(int32_t head_dim, int32_t num_seqs, int32_t num_q_heads,
                                             int32_t num_kv_heads, int32_t max_seq_len);
TQ_API tq_status tq_dense_decode_attention(int32_t head_dim, const void* q_dev, int32_t num_seqs,
                                           int32_t num_q_heads, int32_t num_kv_heads, const void* k_dev,
                                           const void* v_dev, const int32_t* cu_seqlens_dev,
                                           int32_t max_seq_len, float sm_scale, float* out_dev,
                                           void* workspace_dev, size_t workspace_bytes, void* stream);

/*
 * tq_decode_attention_noalloc -- the same decode as tq_decode_attention, for
 * callers that cannot allocate device memory for its workspace.  The pages
 * have no counterpart: they do not discuss how decode scratch is allocated.
 *
 * Who needs it: a serving engine that gave nearly all free device memory to
 * its KV-cache pool at start-up (a later cudaMalloc fails); a plugin inside a
 * host application that owns every device allocation; real-time code that
 * cannot accept the device-wide synchronisation of cudaMalloc / cudaFree.
 *
 * Instead of a caller workspace it uses a fixed scratch array of
 * TQ_NOALLOC_SCRATCH_BYTES in the library's static device memory, which every
 * GPU that loads the library holds until the process exits.  It allocates
 * nothing and calls no cudaMalloc or cudaFree.
 *   - Arguments, layouts and results are those of tq_decode_attention.
 *   - With num_splits = 0, when the automatic split count's workspace
 *     (tq_decode_workspace_size) exceeds the limit, the decode runs with the
 *     largest split count that fits.  A decode that does not fit even with
 *     one split, or with the caller's num_splits > 0, is rejected with
 *     TQ_ERR_WORKSPACE before anything is enqueued.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) and caches it; make that first call before any
 *     stream capture.
 *   - All calls on a device share the one array and it keeps the last call's
 *     contents: calls that overlap on the GPU (other streams, other host
 *     threads) race and give wrong results.  Serialise them.
 */
#define TQ_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
TQ_API tq_status tq_decode_attention_noalloc(const tq_config* cfg, const void* q_dev, int32_t num_seqs,
                                             int32_t num_q_heads, const tq_cache* cache,
                                             const int32_t* block_table_dev, int32_t max_blocks_per_seq,
                                             const int32_t* seq_lens_dev, int32_t max_seq_len, float sm_scale,
                                             int32_t num_splits, float* out_dev, void* stream);

/* Static text naming a status. */
TQ_API const char* tq_status_str(tq_status status);

/* Description of the last non-OK status returned on this host thread. */
TQ_API const char* tq_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* TQ_H */
