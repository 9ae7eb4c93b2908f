// Host core of libtq: configuration, Lloyd-Max codebook, per-layer signs,
// argument validation and the C entry points declared in include/tq.h.
//
// [TQC] vLLM API docs, "vllm.model_executor.layers.quantization.turboquant",
// class TurboQuantConfig: fields, derived sizes, presets, seed rule.
#include "tq.h"

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include <cuda_runtime.h>

#include "tq_internal.h"

namespace {

thread_local char g_last_error[512] = "";

tq_status fail(tq_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return st;
}

tq_status cuda_fail(cudaError_t e, const char* what) {
    return fail(TQ_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// ---------------------------------------------------------------------------
// Lloyd-Max quantiser of N(0,1), positive half.
//
// The optimal quantiser of a symmetric density is symmetric, with a decision
// boundary at 0, so only the levels above 0 are iterated: each level moves to
// the conditional mean of N(0,1) over its cell [a, b], (phi(a) - phi(b)) /
// (P(Z > a) - P(Z > b)), where the cell edges are 0, the midpoints between
// neighbouring levels, and +inf.  Start: the positive half of the uniform
// grid on [-3, 3]; stop when no level moves by 1e-13.
// ---------------------------------------------------------------------------
int lloyd_max_positive(int levels, std::vector<double>& pos) {
    const int half = levels / 2;
    pos.assign(half, 0.0);
    for (int k = 0; k < half; ++k) pos[k] = -3.0 + 6.0 * static_cast<double>(half + k) / (levels - 1);
    const double inv_sqrt2 = 1.0 / std::sqrt(2.0);
    const double inv_sqrt2pi = 1.0 / std::sqrt(2.0 * M_PI);
    auto tail = [&](double x) { return std::isinf(x) ? 0.0 : 0.5 * std::erfc(x * inv_sqrt2); };
    auto dens = [&](double x) { return std::isinf(x) ? 0.0 : inv_sqrt2pi * std::exp(-0.5 * x * x); };
    std::vector<double> next(half);
    for (int it = 1; it <= 100000; ++it) {
        double moved = 0.0;
        for (int k = 0; k < half; ++k) {
            const double a = k == 0 ? 0.0 : 0.5 * (pos[k - 1] + pos[k]);
            const double b = k == half - 1 ? INFINITY : 0.5 * (pos[k] + pos[k + 1]);
            next[k] = (dens(a) - dens(b)) / (tail(a) - tail(b));
            moved = std::fmax(moved, std::fabs(next[k] - pos[k]));
        }
        pos.swap(next);
        if (moved < 1e-13) return it;
    }
    return -1;
}

uint64_t splitmix64_next(uint64_t& state) {
    state += 0x9E3779B97F4A7C15ull;
    uint64_t z = state;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// Bit i of the mask: draw i of the layer's SplitMix64 stream has its top bit
// set, i.e. s_i = -1.
void sign_mask(uint64_t seed_l, int d, uint32_t mask[8]) {
    std::memset(mask, 0, 8 * sizeof(uint32_t));
    uint64_t st = seed_l;
    for (int i = 0; i < d; ++i)
        if (splitmix64_next(st) >> 63) mask[i >> 5] |= 1u << (i & 31);
}

int ceil_div(int a, int b) { return (a + b - 1) / b; }

struct Preset {
    const char* name;
    int kbits, vbits, nc;
};
// [TQC] docstring "Named presets" (TQ_PRESETS itself is not printed).
constexpr Preset kPresets[] = {
    {"turboquant_k8v4", 8, 4, 0},
    {"turboquant_4bit_nc", 4, 4, 1},
    {"turboquant_k3v4_nc", 3, 4, 1},
    {"turboquant_3bit_nc", 3, 3, 1},
};

// Recomputes every derived field of a caller-supplied config and builds the
// kernel parameters; rejects configs that were edited inconsistently.
// The argument checks and slot sizes of a configuration ([TQC]
// key_packed_size / value_packed_size / slot_size_aligned); no codebook.
tq_status config_sizes(int32_t head_dim, int32_t key_quant_bits, int32_t value_quant_bits, int32_t norm_correction,
                       uint64_t seed, tq_config* out) {
    if (head_dim <= 0) return fail(TQ_ERR_INVALID_ARG, "head_dim must be positive (got %d)", head_dim);
    if (!tq::supported_head_dim(head_dim))
        return fail(TQ_ERR_UNSUPPORTED, "head_dim %d: the Walsh-Hadamard rotation needs a power of two in [16, 256]",
                    head_dim);
    if (key_quant_bits != 3 && key_quant_bits != 4 && key_quant_bits != 8)
        return fail(TQ_ERR_INVALID_ARG, "key_quant_bits must be 3, 4 (Lloyd-Max) or 8 (FP8), got %d",
                    key_quant_bits);
    if (value_quant_bits != 3 && value_quant_bits != 4)
        return fail(TQ_ERR_INVALID_ARG, "value_quant_bits must be 3 or 4, got %d", value_quant_bits);
    tq_config& c = *out;
    std::memset(&c, 0, sizeof c);
    c.head_dim = head_dim;
    c.key_quant_bits = key_quant_bits;
    c.value_quant_bits = value_quant_bits;
    c.norm_correction = norm_correction ? 1 : 0;
    c.seed = seed;
    c.key_fp8 = key_quant_bits == 8;
    c.mse_bits = c.key_fp8 ? value_quant_bits : key_quant_bits;
    c.key_mse_bits = c.key_fp8 ? 0 : key_quant_bits;
    c.n_centroids = 1 << c.mse_bits;
    c.key_packed_size = c.key_fp8 ? head_dim : ceil_div(head_dim * c.key_mse_bits, 8) + 2;
    c.value_packed_size = ceil_div(head_dim * value_quant_bits, 8) + 4;
    c.slot_size = c.key_packed_size + c.value_packed_size;
    c.slot_size_aligned = c.slot_size + (c.slot_size & 1);

    return TQ_OK;
}

tq_status layer_params(const tq_config* cfg, int layer_idx, tq::LayerParams* lp) {
    if (cfg == nullptr) return fail(TQ_ERR_INVALID_ARG, "config is NULL");
    tq_config ref;  // sizes only: the codebook is the config's own
    const tq_status st = config_sizes(cfg->head_dim, cfg->key_quant_bits, cfg->value_quant_bits,
                                      cfg->norm_correction, cfg->seed, &ref);
    if (st != TQ_OK) return st;
    if (ref.slot_size_aligned != cfg->slot_size_aligned || ref.key_packed_size != cfg->key_packed_size ||
        ref.value_packed_size != cfg->value_packed_size || ref.n_centroids != cfg->n_centroids)
        return fail(TQ_ERR_INVALID_ARG, "config sizes do not match its bit widths");
    if (layer_idx < 0) return fail(TQ_ERR_INVALID_ARG, "layer_idx < 0");
    std::memset(lp, 0, sizeof *lp);
    lp->d = cfg->head_dim;
    lp->kbits = cfg->key_quant_bits;
    lp->vbits = cfg->value_quant_bits;
    lp->nc = cfg->norm_correction ? 1 : 0;
    lp->key_fp8 = cfg->key_fp8;
    lp->mse_bits = cfg->mse_bits;
    lp->n_centroids = cfg->n_centroids;
    lp->key_packed = cfg->key_packed_size;
    lp->value_packed = cfg->value_packed_size;
    lp->slot_al = cfg->slot_size_aligned;
    sign_mask(cfg->seed + static_cast<uint64_t>(layer_idx) * 1337ull, cfg->head_dim, lp->sign_mask);
    for (int i = 0; i < TQ_MAX_CENTROIDS; ++i) lp->centroids[i] = cfg->centroids[i];
    for (int i = 0; i < TQ_MAX_CENTROIDS - 1; ++i) lp->boundaries[i] = cfg->boundaries[i];
    return TQ_OK;
}

tq_status cache_geom(const tq_cache* cache, const tq_config* cfg, bool need_16b, tq::CacheGeom* g) {
    if (cache == nullptr) return fail(TQ_ERR_INVALID_ARG, "cache is NULL");
    if (cache->data_dev == nullptr) return fail(TQ_ERR_INVALID_ARG, "cache data is NULL");
    if (cache->num_blocks <= 0 || cache->block_size <= 0 || cache->num_kv_heads <= 0)
        return fail(TQ_ERR_INVALID_ARG, "cache geometry must be positive");
    const int64_t dense = static_cast<int64_t>(cache->block_size) * cache->num_kv_heads * cfg->slot_size_aligned;
    const int64_t stride = cache->block_stride_bytes == 0 ? dense : cache->block_stride_bytes;
    if (stride < dense) return fail(TQ_ERR_INVALID_ARG, "block_stride_bytes %lld < block bytes %lld",
                                    static_cast<long long>(stride), static_cast<long long>(dense));
    const uintptr_t base = reinterpret_cast<uintptr_t>(cache->data_dev);
    if (need_16b) {
        if ((base & 15u) != 0 || (stride & 15) != 0)
            return fail(TQ_ERR_INVALID_ARG, "decode needs a 16-byte aligned cache and block stride");
        if (cache->block_size % 16 != 0)
            return fail(TQ_ERR_UNSUPPORTED, "decode needs block_size %% 16 == 0 (got %d)", cache->block_size);
    } else if ((base & 1u) != 0 || (stride & 1) != 0) {
        return fail(TQ_ERR_INVALID_ARG, "cache and block stride must be 2-byte aligned");
    }
    g->data = cache->data_dev;
    g->num_blocks = cache->num_blocks;
    g->block_size = cache->block_size;
    g->num_kv_heads = cache->num_kv_heads;
    g->block_stride = stride;
    g->flags = cache->error_flags_dev;
    return TQ_OK;
}

tq_status sm_count(int* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    e = cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    return TQ_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

void tq::set_last_error(const char* msg) { std::snprintf(g_last_error, sizeof g_last_error, "%s", msg); }

extern "C" {

const char* tq_status_str(tq_status s) {
    switch (s) {
        case TQ_OK: return "TQ_OK";
        case TQ_ERR_INVALID_ARG: return "TQ_ERR_INVALID_ARG";
        case TQ_ERR_UNKNOWN_PRESET: return "TQ_ERR_UNKNOWN_PRESET";
        case TQ_ERR_UNSUPPORTED: return "TQ_ERR_UNSUPPORTED";
        case TQ_ERR_WORKSPACE: return "TQ_ERR_WORKSPACE";
        case TQ_ERR_OUT_OF_RANGE: return "TQ_ERR_OUT_OF_RANGE";
        case TQ_ERR_CUDA: return "TQ_ERR_CUDA";
    }
    return "TQ_ERR_UNKNOWN_STATUS";
}

const char* tq_last_error(void) { return g_last_error; }

tq_status tq_config_init(int32_t head_dim, int32_t key_quant_bits, int32_t value_quant_bits,
                         int32_t norm_correction, uint64_t seed, tq_config* out) {
    if (out == nullptr) return fail(TQ_ERR_INVALID_ARG, "output config is NULL");
    tq_config c;
    const tq_status sz = config_sizes(head_dim, key_quant_bits, value_quant_bits, norm_correction, seed, &c);
    if (sz != TQ_OK) return sz;

    std::vector<double> pos;
    const int iters = lloyd_max_positive(c.n_centroids, pos);
    if (iters < 0) return fail(TQ_ERR_INVALID_ARG, "Lloyd-Max iteration did not converge");
    c.lloyd_max_iterations = iters;
    const int half = c.n_centroids / 2;
    const double sigma = 1.0 / std::sqrt(static_cast<double>(head_dim));
    for (int k = 0; k < half; ++k) {
        const double v = pos[k] * sigma;
        c.centroids[half + k] = static_cast<float>(v);
        c.centroids[half - 1 - k] = static_cast<float>(-v);
    }
    c.boundaries[half - 1] = 0.0f;
    for (int k = 0; k + 1 < half; ++k) {
        const float b = static_cast<float>(0.5 * (pos[k] * sigma + pos[k + 1] * sigma));
        c.boundaries[half + k] = b;
        c.boundaries[half - 2 - k] = -b;
    }
    *out = c;
    return TQ_OK;
}

tq_status tq_config_from_preset(int32_t head_dim, const char* preset, tq_config* out) {
    if (preset == nullptr) return fail(TQ_ERR_INVALID_ARG, "preset is NULL");
    for (const Preset& p : kPresets)
        if (std::strcmp(p.name, preset) == 0) return tq_config_init(head_dim, p.kbits, p.vbits, p.nc, 42, out);
    std::string valid;
    for (const Preset& p : kPresets) {
        if (!valid.empty()) valid += ", ";
        valid += p.name;
    }
    return fail(TQ_ERR_UNKNOWN_PRESET, "unknown TurboQuant preset '%s'; valid presets: %s", preset, valid.c_str());
}

tq_status tq_layer_signs(const tq_config* cfg, int32_t layer_idx, int8_t* signs_out) {
    if (signs_out == nullptr) return fail(TQ_ERR_INVALID_ARG, "signs_out is NULL");
    tq::LayerParams lp;
    const tq_status st = layer_params(cfg, layer_idx, &lp);
    if (st != TQ_OK) return st;
    for (int i = 0; i < lp.d; ++i) signs_out[i] = ((lp.sign_mask[i >> 5] >> (i & 31)) & 1u) ? -1 : 1;
    return TQ_OK;
}

tq_status tq_store_kv(const tq_config* cfg, const void* k_dev, const void* v_dev, int64_t num_tokens,
                      const int64_t* slot_mapping_dev, const tq_cache* cache, void* stream) {
    if (cache == nullptr) return fail(TQ_ERR_INVALID_ARG, "cache is NULL");
    tq::LayerParams lp;
    tq_status st = layer_params(cfg, cache->layer_idx, &lp);
    if (st != TQ_OK) return st;
    tq::CacheGeom g;
    st = cache_geom(cache, cfg, false, &g);
    if (st != TQ_OK) return st;
    if (num_tokens < 0) return fail(TQ_ERR_INVALID_ARG, "num_tokens < 0");
    if (num_tokens == 0) return TQ_OK;
    if (k_dev == nullptr || v_dev == nullptr || slot_mapping_dev == nullptr)
        return fail(TQ_ERR_INVALID_ARG, "k, v and slot_mapping must not be NULL");
    if (!aligned(k_dev, 16) || !aligned(v_dev, 16) || !aligned(slot_mapping_dev, 8))
        return fail(TQ_ERR_INVALID_ARG, "k and v must be 16-byte aligned, slot_mapping 8-byte aligned");
    int sms = 0;
    st = sm_count(&sms);
    if (st != TQ_OK) return st;
    const cudaError_t e = tq::launch_store(lp, g, static_cast<const uint16_t*>(k_dev),
                                           static_cast<const uint16_t*>(v_dev), num_tokens, slot_mapping_dev, sms,
                                           static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tq_store_kv launch");
    return TQ_OK;
}

size_t tq_decode_workspace_size(const tq_config* cfg, int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                int32_t block_size, int32_t max_seq_len, int32_t num_splits) {
    (void)block_size;
    tq::LayerParams lp;
    if (layer_params(cfg, 0, &lp) != TQ_OK) return 0;
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_seq_len < 0) return 0;
    int sms = 1;
    if (num_splits <= 0 && sm_count(&sms) != TQ_OK) return 0;
    return tq::plan_decode(lp, num_seqs, num_q_heads, num_kv_heads, max_seq_len, num_splits, sms).workspace_bytes;
}

namespace {
tq_status decode_common(const tq_config* cfg, const void* q_dev, int32_t num_seqs, int32_t num_q_heads,
                        const tq_cache* cache, const int32_t* block_table_dev, int32_t max_blocks_per_seq,
                        const int32_t* seq_lens_dev, int32_t max_seq_len, float sm_scale, int32_t num_splits,
                        const tq::RingBuf& ring, float* out_dev, void* workspace_dev, size_t workspace_bytes,
                        void* stream) {
    if (cache == nullptr) return fail(TQ_ERR_INVALID_ARG, "cache is NULL");
    tq::LayerParams lp;
    tq_status st = layer_params(cfg, cache->layer_idx, &lp);
    if (st != TQ_OK) return st;
    tq::CacheGeom g;
    st = cache_geom(cache, cfg, true, &g);
    if (st != TQ_OK) return st;
    if (num_seqs < 0 || max_seq_len < 0 || max_blocks_per_seq <= 0 || num_splits < 0)
        return fail(TQ_ERR_INVALID_ARG, "negative size argument");
    if (num_seqs > TQ_MAX_SEQS)
        return fail(TQ_ERR_UNSUPPORTED, "num_seqs (%d) above %d (one grid row per sequence)", num_seqs, TQ_MAX_SEQS);
    if (num_q_heads <= 0 || num_q_heads % cache->num_kv_heads != 0)
        return fail(TQ_ERR_INVALID_ARG, "num_q_heads (%d) must be a positive multiple of num_kv_heads (%d)",
                    num_q_heads, cache->num_kv_heads);
    const int group = num_q_heads / cache->num_kv_heads;
    if (cache->num_kv_heads > 8 || group > 8)
        return fail(TQ_ERR_UNSUPPORTED, "decode supports up to 8 KV heads and 8 query heads per KV head");
    if (num_seqs == 0) return TQ_OK;
    if (q_dev == nullptr || block_table_dev == nullptr || seq_lens_dev == nullptr || out_dev == nullptr)
        return fail(TQ_ERR_INVALID_ARG, "q, block_table, seq_lens and out must not be NULL");
    if (!aligned(q_dev, 4) || !aligned(out_dev, 4) || !aligned(block_table_dev, 4) || !aligned(seq_lens_dev, 4))
        return fail(TQ_ERR_INVALID_ARG, "q, out, block_table and seq_lens must be 4-byte aligned");
    int sms = 1;
    st = sm_count(&sms);
    if (st != TQ_OK) return st;
    const tq::DecodePlan plan =
        tq::plan_decode(lp, num_seqs, num_q_heads, cache->num_kv_heads, max_seq_len, num_splits, sms,
                        ring.tokens > 0);
    if (workspace_dev == nullptr || workspace_bytes < plan.workspace_bytes)
        return fail(TQ_ERR_WORKSPACE, "decode workspace needs %zu bytes (got %zu)", plan.workspace_bytes,
                    workspace_bytes);
    if (!aligned(workspace_dev, 16)) return fail(TQ_ERR_WORKSPACE, "workspace must be 16-byte aligned");
    const float scale = sm_scale > 0.f ? sm_scale : 1.0f / std::sqrt(static_cast<float>(cfg->head_dim));
    const cudaError_t e = tq::launch_decode(lp, g, static_cast<const uint16_t*>(q_dev), num_seqs, num_q_heads,
                                            block_table_dev, max_blocks_per_seq, seq_lens_dev, max_seq_len, scale,
                                            plan, ring, out_dev, workspace_dev, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tq_decode_attention launch");
    return TQ_OK;
}
}  // namespace

tq_status tq_decode_attention(const tq_config* cfg, const void* q_dev, int32_t num_seqs, int32_t num_q_heads,
                              const tq_cache* cache, const int32_t* block_table_dev, int32_t max_blocks_per_seq,
                              const int32_t* seq_lens_dev, int32_t max_seq_len, float sm_scale, int32_t num_splits,
                              float* out_dev, void* workspace_dev, size_t workspace_bytes, void* stream) {
    return decode_common(cfg, q_dev, num_seqs, num_q_heads, cache, block_table_dev, max_blocks_per_seq, seq_lens_dev,
                         max_seq_len, sm_scale, num_splits, tq::RingBuf{nullptr, nullptr, 0}, out_dev, workspace_dev,
                         workspace_bytes, stream);
}

size_t tq_decode_ring_workspace_size(const tq_config* cfg, int32_t num_seqs, int32_t num_q_heads,
                                     int32_t num_kv_heads, int32_t block_size, int32_t max_seq_len,
                                     int32_t num_splits) {
    (void)block_size;
    tq::LayerParams lp;
    if (layer_params(cfg, 0, &lp) != TQ_OK) return 0;
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_seq_len < 0) return 0;
    int sms = 1;
    if (num_splits <= 0 && sm_count(&sms) != TQ_OK) return 0;
    return tq::plan_decode(lp, num_seqs, num_q_heads, num_kv_heads, max_seq_len, num_splits, sms, true)
        .workspace_bytes;
}

tq_status tq_decode_attention_ring(const tq_config* cfg, const void* q_dev, int32_t num_seqs, int32_t num_q_heads,
                                   const tq_cache* cache, const int32_t* block_table_dev,
                                   int32_t max_blocks_per_seq, const int32_t* seq_lens_dev, int32_t max_seq_len,
                                   float sm_scale, int32_t num_splits, const void* ring_k_dev,
                                   const void* ring_v_dev, int32_t ring_tokens, float* out_dev, void* workspace_dev,
                                   size_t workspace_bytes, void* stream) {
    if (ring_tokens < 1 || ring_tokens > TQ_RING_MAX_TOKENS)
        return fail(TQ_ERR_UNSUPPORTED, "ring_tokens must be in [1, %d] (got %d)", TQ_RING_MAX_TOKENS, ring_tokens);
    if (num_seqs > 0 && (ring_k_dev == nullptr || ring_v_dev == nullptr))
        return fail(TQ_ERR_INVALID_ARG, "ring_k and ring_v must not be NULL");
    if (!aligned(ring_k_dev, 16) || !aligned(ring_v_dev, 16))
        return fail(TQ_ERR_INVALID_ARG, "ring_k and ring_v must be 16-byte aligned");
    if (cache != nullptr && (num_q_heads <= 0 || num_q_heads % cache->num_kv_heads != 0 ||
                             num_q_heads / cache->num_kv_heads > 8))
        return fail(TQ_ERR_UNSUPPORTED, "the ring decode supports up to 8 query heads per KV head");
    const tq::RingBuf ring{static_cast<const uint16_t*>(ring_k_dev), static_cast<const uint16_t*>(ring_v_dev),
                           ring_tokens};
    return decode_common(cfg, q_dev, num_seqs, num_q_heads, cache, block_table_dev, max_blocks_per_seq, seq_lens_dev,
                         max_seq_len, sm_scale, num_splits, ring, out_dev, workspace_dev, workspace_bytes, stream);
}

size_t tq_ring_workspace_size(int32_t num_seqs) { return num_seqs < 0 ? 0 : tq::ring_workspace_bytes(num_seqs); }

tq_status tq_ring_step(const tq_config* cfg, const void* k_dev, const void* v_dev, int32_t num_seqs,
                       const int32_t* seq_lens_dev, void* ring_k_dev, void* ring_v_dev, int32_t ring_tokens,
                       const tq_cache* cache, const int32_t* block_table_dev, int32_t max_blocks_per_seq,
                       void* stream) {
    if (cache == nullptr) return fail(TQ_ERR_INVALID_ARG, "cache is NULL");
    tq::LayerParams lp;
    tq_status st = layer_params(cfg, cache->layer_idx, &lp);
    if (st != TQ_OK) return st;
    tq::CacheGeom g;
    st = cache_geom(cache, cfg, false, &g);
    if (st != TQ_OK) return st;
    if (num_seqs < 0 || max_blocks_per_seq <= 0) return fail(TQ_ERR_INVALID_ARG, "negative size argument");
    if (ring_tokens < 1 || ring_tokens > TQ_RING_MAX_TOKENS)
        return fail(TQ_ERR_UNSUPPORTED, "ring_tokens must be in [1, %d] (got %d)", TQ_RING_MAX_TOKENS, ring_tokens);
    if (num_seqs == 0) return TQ_OK;
    if (k_dev == nullptr || v_dev == nullptr || seq_lens_dev == nullptr || ring_k_dev == nullptr ||
        ring_v_dev == nullptr || block_table_dev == nullptr)
        return fail(TQ_ERR_INVALID_ARG, "k, v, seq_lens, rings and block_table must not be NULL");
    if (!aligned(k_dev, 16) || !aligned(v_dev, 16) || !aligned(ring_k_dev, 16) || !aligned(ring_v_dev, 16))
        return fail(TQ_ERR_INVALID_ARG, "k, v, ring_k and ring_v must be 16-byte aligned");
    if (!aligned(seq_lens_dev, 4) || !aligned(block_table_dev, 4))
        return fail(TQ_ERR_INVALID_ARG, "seq_lens and block_table must be 4-byte aligned");
    int sms = 0;
    st = sm_count(&sms);
    if (st != TQ_OK) return st;
    const cudaError_t e = tq::launch_ring_step(
        lp, g, static_cast<const uint16_t*>(k_dev), static_cast<const uint16_t*>(v_dev), num_seqs, seq_lens_dev,
        static_cast<uint16_t*>(ring_k_dev), static_cast<uint16_t*>(ring_v_dev), ring_tokens, block_table_dev,
        max_blocks_per_seq, sms, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tq_ring_step launch");
    return TQ_OK;
}

tq_status tq_ring_append(const tq_config* cfg, const void* k_dev, const void* v_dev, int64_t num_tokens,
                         const int32_t* cu_new_dev, int32_t num_seqs, const int32_t* seq_lens_dev, void* ring_k_dev,
                         void* ring_v_dev, int32_t ring_tokens, const tq_cache* cache,
                         const int32_t* block_table_dev, int32_t max_blocks_per_seq, void* workspace_dev,
                         size_t workspace_bytes, void* stream) {
    if (cache == nullptr) return fail(TQ_ERR_INVALID_ARG, "cache is NULL");
    tq::LayerParams lp;
    tq_status st = layer_params(cfg, cache->layer_idx, &lp);
    if (st != TQ_OK) return st;
    tq::CacheGeom g;
    st = cache_geom(cache, cfg, false, &g);
    if (st != TQ_OK) return st;
    if (num_seqs < 0 || num_tokens < 0 || max_blocks_per_seq <= 0)
        return fail(TQ_ERR_INVALID_ARG, "negative size argument");
    if (ring_tokens < 1 || ring_tokens > TQ_RING_MAX_TOKENS)
        return fail(TQ_ERR_UNSUPPORTED, "ring_tokens must be in [1, %d] (got %d)", TQ_RING_MAX_TOKENS, ring_tokens);
    if (num_seqs == 0) return TQ_OK;
    if (cu_new_dev == nullptr || seq_lens_dev == nullptr || ring_k_dev == nullptr || ring_v_dev == nullptr ||
        block_table_dev == nullptr || (num_tokens > 0 && (k_dev == nullptr || v_dev == nullptr)))
        return fail(TQ_ERR_INVALID_ARG, "k, v, cu_new, seq_lens, rings and block_table must not be NULL");
    if (!aligned(k_dev, 16) || !aligned(v_dev, 16) || !aligned(ring_k_dev, 16) || !aligned(ring_v_dev, 16))
        return fail(TQ_ERR_INVALID_ARG, "k, v, ring_k and ring_v must be 16-byte aligned");
    if (!aligned(cu_new_dev, 4) || !aligned(seq_lens_dev, 4) || !aligned(block_table_dev, 4))
        return fail(TQ_ERR_INVALID_ARG, "cu_new, seq_lens and block_table must be 4-byte aligned");
    if (workspace_dev == nullptr || workspace_bytes < tq::ring_workspace_bytes(num_seqs))
        return fail(TQ_ERR_WORKSPACE, "ring append workspace needs %zu bytes (got %zu)",
                    tq::ring_workspace_bytes(num_seqs), workspace_bytes);
    if (!aligned(workspace_dev, 16)) return fail(TQ_ERR_WORKSPACE, "workspace must be 16-byte aligned");
    int sms = 0;
    st = sm_count(&sms);
    if (st != TQ_OK) return st;
    const cudaError_t e = tq::launch_ring_append(
        lp, g, static_cast<const uint16_t*>(k_dev), static_cast<const uint16_t*>(v_dev), num_tokens, cu_new_dev,
        num_seqs, seq_lens_dev, static_cast<uint16_t*>(ring_k_dev), static_cast<uint16_t*>(ring_v_dev), ring_tokens,
        block_table_dev, max_blocks_per_seq, workspace_dev, sms, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tq_ring_append launch");
    return TQ_OK;
}

tq_status tq_dequant(const tq_config* cfg, const tq_cache* cache, const int32_t* block_table_dev,
                     int32_t max_blocks_per_seq, const int32_t* cu_seqlens_dev, int32_t num_seqs,
                     int32_t max_seq_len, void* k_out_dev, void* v_out_dev, void* stream) {
    if (cache == nullptr) return fail(TQ_ERR_INVALID_ARG, "cache is NULL");
    tq::LayerParams lp;
    tq_status st = layer_params(cfg, cache->layer_idx, &lp);
    if (st != TQ_OK) return st;
    tq::CacheGeom g;
    st = cache_geom(cache, cfg, false, &g);
    if (st != TQ_OK) return st;
    if (num_seqs < 0 || max_seq_len < 0 || max_blocks_per_seq <= 0)
        return fail(TQ_ERR_INVALID_ARG, "negative size argument");
    if (num_seqs > TQ_MAX_SEQS)
        return fail(TQ_ERR_UNSUPPORTED, "num_seqs (%d) above %d (one grid row per sequence)", num_seqs, TQ_MAX_SEQS);
    if (num_seqs == 0 || max_seq_len == 0) return TQ_OK;
    if (block_table_dev == nullptr || cu_seqlens_dev == nullptr || k_out_dev == nullptr || v_out_dev == nullptr)
        return fail(TQ_ERR_INVALID_ARG, "block_table, cu_seqlens, k_out and v_out must not be NULL");
    if (!aligned(k_out_dev, 16) || !aligned(v_out_dev, 16))
        return fail(TQ_ERR_INVALID_ARG, "k_out and v_out must be 16-byte aligned");
    int sms = 0;
    st = sm_count(&sms);
    if (st != TQ_OK) return st;
    const cudaError_t e = tq::launch_dequant(lp, g, block_table_dev, max_blocks_per_seq, cu_seqlens_dev, num_seqs,
                                             max_seq_len, static_cast<uint16_t*>(k_out_dev),
                                             static_cast<uint16_t*>(v_out_dev), sms, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tq_dequant launch");
    return TQ_OK;
}

size_t tq_dense_decode_workspace_size(int32_t head_dim, int32_t num_seqs, int32_t num_q_heads,
                                      int32_t num_kv_heads, int32_t max_seq_len) {
    if (!tq::supported_head_dim(head_dim) || num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        max_seq_len < 0)
        return 0;
    int sms = 1;
    if (sm_count(&sms) != TQ_OK) return 0;
    return tq::plan_dense(num_seqs, num_q_heads, num_kv_heads, head_dim, max_seq_len, sms).workspace_bytes;
}

tq_status tq_dense_decode_attention(int32_t head_dim, const void* q_dev, int32_t num_seqs, int32_t num_q_heads,
                                    int32_t num_kv_heads, const void* k_dev, const void* v_dev,
                                    const int32_t* cu_seqlens_dev, int32_t max_seq_len, float sm_scale,
                                    float* out_dev, void* workspace_dev, size_t workspace_bytes, void* stream) {
    if (!tq::supported_head_dim(head_dim))
        return fail(TQ_ERR_UNSUPPORTED, "head_dim %d is not a power of two in [16, 256]", head_dim);
    if (num_seqs < 0 || max_seq_len < 0 || num_q_heads <= 0 || num_kv_heads <= 0)
        return fail(TQ_ERR_INVALID_ARG, "negative size argument");
    if (num_q_heads % num_kv_heads != 0 || num_q_heads / num_kv_heads > 8)
        return fail(TQ_ERR_UNSUPPORTED, "num_q_heads (%d) must be 1 to 8 times num_kv_heads (%d)", num_q_heads,
                    num_kv_heads);
    if (num_seqs > TQ_MAX_SEQS)
        return fail(TQ_ERR_UNSUPPORTED, "num_seqs (%d) above %d (one grid row per sequence)", num_seqs, TQ_MAX_SEQS);
    if (num_kv_heads > 65535) return fail(TQ_ERR_UNSUPPORTED, "num_kv_heads above 65535");
    if (num_seqs == 0) return TQ_OK;
    if (q_dev == nullptr || k_dev == nullptr || v_dev == nullptr || cu_seqlens_dev == nullptr || out_dev == nullptr)
        return fail(TQ_ERR_INVALID_ARG, "q, k, v, cu_seqlens and out must not be NULL");
    if (!aligned(q_dev, 16) || !aligned(k_dev, 16) || !aligned(v_dev, 16) || !aligned(out_dev, 4) ||
        !aligned(cu_seqlens_dev, 4))
        return fail(TQ_ERR_INVALID_ARG, "q, k and v must be 16-byte aligned, out and cu_seqlens 4-byte aligned");
    int sms = 1;
    tq_status st = sm_count(&sms);
    if (st != TQ_OK) return st;
    const tq::DensePlan plan = tq::plan_dense(num_seqs, num_q_heads, num_kv_heads, head_dim, max_seq_len, sms);
    if (workspace_dev == nullptr || workspace_bytes < plan.workspace_bytes)
        return fail(TQ_ERR_WORKSPACE, "dense decode workspace needs %zu bytes (got %zu)", plan.workspace_bytes,
                    workspace_bytes);
    if (!aligned(workspace_dev, 16)) return fail(TQ_ERR_WORKSPACE, "workspace must be 16-byte aligned");
    const float scale = sm_scale > 0.f ? sm_scale : 1.0f / std::sqrt(static_cast<float>(head_dim));
    const cudaError_t e = tq::launch_dense_decode(
        head_dim, static_cast<const uint16_t*>(q_dev), num_seqs, num_q_heads, num_kv_heads,
        static_cast<const uint16_t*>(k_dev), static_cast<const uint16_t*>(v_dev), cu_seqlens_dev, max_seq_len, scale,
        plan, out_dev, workspace_dev, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tq_dense_decode_attention launch");
    return TQ_OK;
}

tq_status tq_hybrid_page(const tq_config* cfg, int32_t num_kv_heads, int32_t skip_dtype_bytes,
                         int64_t* page_bytes_out, int32_t* tokens_per_page_out) {
    tq::LayerParams lp;
    const tq_status st = layer_params(cfg, 0, &lp);
    if (st != TQ_OK) return st;
    if (num_kv_heads <= 0 || skip_dtype_bytes < 0 || page_bytes_out == nullptr || tokens_per_page_out == nullptr)
        return fail(TQ_ERR_INVALID_ARG, "invalid hybrid page query");
    const int64_t tq_page = static_cast<int64_t>(num_kv_heads) * cfg->slot_size_aligned;
    int64_t page = tq_page;
    if (skip_dtype_bytes > 0) {
        const int64_t skip_page = 2ll * num_kv_heads * cfg->head_dim * skip_dtype_bytes;
        int64_t a = tq_page, b = skip_page;
        while (b != 0) {
            const int64_t r = a % b;
            a = b;
            b = r;
        }
        page = tq_page / a * skip_page;
    }
    if (page / tq_page > INT32_MAX) return fail(TQ_ERR_UNSUPPORTED, "unified page holds too many tokens");
    *page_bytes_out = page;
    *tokens_per_page_out = static_cast<int32_t>(page / tq_page);
    return TQ_OK;
}

}  // extern "C"
