// Host side of the tensor-core decode: shape support, the centroid table
// scale, occupancy queries and the launch of the split kernel (tq_decode.cu
// merges the partials).  The kernel itself is in tq_decode_mma.cuh.
#include <cmath>
#include <mutex>

#include "tq_decode_mma.cuh"

namespace tq {

namespace {

// Round to the nearest fp16 value (ties to even), on the host.
float round_half(float x) { return __half2float(__float2half_rn(x)); }

// A factor gamma in [1, 2) for which the centroids, in units of 1/sqrt(d)
// and multiplied by gamma, have the smallest worst-case fp16 rounding error
// (searched on a 2^16 grid once per codebook).  Any gamma gives the same
// attention; this one makes the fp16 table values nearly exact.
float table_gamma(const LayerParams& p) {
    static float cache[9][9] = {};  // [mse_bits][log2 d]
    static std::mutex mu;
    if (p.key_fp8) return 1.0f;
    int lg = 0;
    while ((1 << lg) < p.d) ++lg;
    std::lock_guard<std::mutex> lock(mu);
    float& g = cache[p.mse_bits][lg];
    if (g != 0.f) return g;
    const int half = p.n_centroids / 2;
    const float unit = sqrtf(static_cast<float>(p.d));
    float best = 1.f, best_err = 1e30f;
    for (int k = 0; k < (1 << 16); ++k) {
        const float cand = 1.0f + static_cast<float>(k) / 65536.0f;
        float worst = 0.f;
        for (int j = half; j < p.n_centroids; ++j) {
            const float v = p.centroids[j] * unit * cand;
            worst = fmaxf(worst, fabsf(round_half(v) - v) / v);
        }
        if (worst < best_err) {
            best_err = worst;
            best = cand;
        }
    }
    g = best;
    return g;
}

cudaError_t run(const LayerParams& p, const CacheGeom& c, const mma::Args& a, int num_seqs, int num_kv_heads,
                cudaStream_t stream, int* ctas) {
    switch (p.d) {
        case 64: return decode_mma_run_d64(p, c, a, num_seqs, num_kv_heads, stream, ctas);
        case 128: return decode_mma_run_d128(p, c, a, num_seqs, num_kv_heads, stream, ctas);
        case 256: return decode_mma_run_d256(p, c, a, num_seqs, num_kv_heads, stream, ctas);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool decode_mma_supported(const LayerParams& p, int num_kv_heads, int num_q_heads) {
    const int h = num_kv_heads;
    if (!(h == 1 || h == 2 || h == 4 || h == 8)) return false;
    if (num_q_heads % h != 0 || num_q_heads / h > 8) return false;
    return p.d == 64 || p.d == 128 || p.d == 256;
}

int decode_mma_ctas_per_sm(const LayerParams& p, int num_kv_heads, int num_q_heads) {
    mma::Args a{};
    a.num_q_heads = num_q_heads;
    CacheGeom c{};
    int ctas = 0;
    if (run(p, c, a, 0, num_kv_heads, nullptr, &ctas) != cudaSuccess) return 0;
    return ctas;
}

cudaError_t launch_decode_mma(const LayerParams& p, const CacheGeom& c, const uint16_t* q, int num_seqs,
                              int num_q_heads, const int32_t* block_table, int max_blocks_per_seq,
                              const int32_t* seq_lens, int max_seq_len, float sm_scale, const DecodePlan& plan,
                              int ring_tokens, void* workspace, cudaStream_t stream) {
    mma::Args a{};
    a.q = q;
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.partials = static_cast<float*>(workspace);
    a.num_q_heads = num_q_heads;
    a.max_blocks = max_blocks_per_seq;
    a.max_seq_len = max_seq_len;
    a.chunks_per_split = plan.chunks_per_split;
    a.num_splits = plan.num_splits;
    a.slot_stride = plan.slot_stride;
    a.ring_tokens = ring_tokens;
    a.qscale = sm_scale * mma::kLog2e;
    a.lut_scale = table_gamma(p) * sqrtf(static_cast<float>(p.d));
    return run(p, c, a, num_seqs, c.num_kv_heads, stream, nullptr);
}

}  // namespace tq
