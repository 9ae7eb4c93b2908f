// Internal interface between the host core (tq_host.cpp) and the CUDA
// kernels.  Nothing here is part of the public ABI (include/tq.h).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace tq {

// Everything a kernel needs to know about one layer's quantiser; passed by
// value as a kernel parameter (under 300 bytes).
struct LayerParams {
    int32_t d;
    int32_t kbits;
    int32_t vbits;
    int32_t nc;
    int32_t key_fp8;
    int32_t mse_bits;
    int32_t n_centroids;
    int32_t key_packed;
    int32_t value_packed;
    int32_t slot_al;
    uint32_t sign_mask[8];  // bit i set: s_i = -1 (d <= 256)
    float centroids[16];
    float boundaries[15];
};

struct CacheGeom {
    uint8_t* data;
    int64_t num_blocks;
    int32_t block_size;
    int32_t num_kv_heads;
    int64_t block_stride;  // bytes, > 0
    uint32_t* flags;       // may be null
};

constexpr uint32_t kFlagSlot = 1u;
constexpr uint32_t kFlagBlock = 2u;
constexpr uint32_t kFlagSeq = 4u;
constexpr uint32_t kFlagWait = 8u;

struct DecodePlan {
    int32_t num_splits;
    int32_t chunks_per_split;  // 16-token chunks handled by one split
    int32_t slot_stride;       // partial slots per (sequence, query head): the splits, + 1 for a ring
    size_t partial_bytes;      // fp32 partial states
    size_t workspace_bytes;    // total, including alignment padding
};

// Chooses the split count for a decode call (num_splits_req = 0: automatic);
// ring: one more partial slot, for the exact ring rows.
DecodePlan plan_decode(const LayerParams& p, int num_seqs, int num_q_heads, int num_kv_heads,
                       int max_seq_len, int num_splits_req, int sm_count, bool ring = false);

// The exact ring of the ring-buffered store: bf16 [num_seqs, tokens, H, d].
struct RingBuf {
    const uint16_t* k;
    const uint16_t* v;
    int tokens;  // 0: no ring
};

cudaError_t launch_store(const LayerParams& p, const CacheGeom& c, const uint16_t* k,
                         const uint16_t* v, int64_t num_tokens, const int64_t* slot_mapping,
                         int sm_count, cudaStream_t stream);

// Decode over the packed cache and, with a ring, over the exact ring rows
// (seq_lens counting both; the packed part is the whole ring blocks).
cudaError_t launch_decode(const LayerParams& p, const CacheGeom& c, const uint16_t* q, int num_seqs,
                          int num_q_heads, const int32_t* block_table, int max_blocks_per_seq,
                          const int32_t* seq_lens, int max_seq_len, float sm_scale,
                          const DecodePlan& plan, const RingBuf& ring, float* out, void* workspace,
                          cudaStream_t stream);

// Ring-buffered store: packs every ring block the new tokens complete and
// copies the rest into the ring (tq_store.cu).  workspace: ring_workspace_bytes.
size_t ring_workspace_bytes(int num_seqs);
// One new token per sequence (row s of k / v), one kernel: packs the ring
// blocks the tokens complete and copies the other tokens into the ring.
cudaError_t launch_ring_step(const LayerParams& p, const CacheGeom& c, const uint16_t* k, const uint16_t* v,
                             int num_seqs, const int32_t* seq_lens, uint16_t* ring_k, uint16_t* ring_v,
                             int ring_tokens, const int32_t* block_table, int max_blocks_per_seq, int sm_count,
                             cudaStream_t stream);
cudaError_t launch_ring_append(const LayerParams& p, const CacheGeom& c, const uint16_t* k, const uint16_t* v,
                               int64_t num_tokens, const int32_t* cu_new, int num_seqs, const int32_t* seq_lens,
                               uint16_t* ring_k, uint16_t* ring_v, int ring_tokens, const int32_t* block_table,
                               int max_blocks_per_seq, void* workspace, int sm_count, cudaStream_t stream);

// Tensor-core decode (tq_decode_mma.cu): H in {1,2,4,8}, G <= 8, d in {64,128,256}.
bool decode_mma_supported(const LayerParams& p, int num_kv_heads, int num_q_heads);
// Resident CTAs per SM of the tensor-core decode for these shapes (0 on error).
int decode_mma_ctas_per_sm(const LayerParams& p, int num_kv_heads, int num_q_heads);
// Writes the split partials of the packed positions (ring_tokens > 0: the
// whole ring blocks only); the caller merges them.
cudaError_t launch_decode_mma(const LayerParams& p, const CacheGeom& c, const uint16_t* q, int num_seqs,
                              int num_q_heads, const int32_t* block_table, int max_blocks_per_seq,
                              const int32_t* seq_lens, int max_seq_len, float sm_scale, const DecodePlan& plan,
                              int ring_tokens, void* workspace, cudaStream_t stream);
// Log-sum-exp merge of the partials [S, Hq, slots, d + 2] into out [S, Hq, d].
// after_decode_kernel: the previous launch on the stream is the decode
// kernel (programmatic dependent launch applies).
cudaError_t launch_combine(const float* partials, float* out, int num_seqs, int num_q_heads, int d,
                           int slots, cudaStream_t stream, bool after_decode_kernel);

cudaError_t launch_dequant(const LayerParams& p, const CacheGeom& c, const int32_t* block_table,
                           int max_blocks_per_seq, const int32_t* cu_seqlens, int num_seqs,
                           int max_seq_len, uint16_t* k_out, uint16_t* v_out, int sm_count, cudaStream_t stream);

// Dense decode over bf16 K/V rows (the dequant-then-attend comparison path).
struct DensePlan {
    int32_t num_splits;
    int32_t tokens_per_split;
    size_t workspace_bytes;
};
DensePlan plan_dense(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int max_seq_len, int sm_count);
cudaError_t launch_dense_decode(int head_dim, const uint16_t* q, int num_seqs, int num_q_heads, int num_kv_heads,
                                const uint16_t* k, const uint16_t* v, const int32_t* cu_seqlens, int max_seq_len,
                                float sm_scale, const DensePlan& plan, float* out, void* workspace,
                                cudaStream_t stream);

// Records the text tq_last_error() returns on this host thread.
void set_last_error(const char* msg);

// Supported compile-time shapes.
inline bool supported_head_dim(int d) {
    return d == 16 || d == 32 || d == 64 || d == 128 || d == 256;
}

}  // namespace tq
