// Decode attention for callers that cannot allocate device memory.
//
// tq_decode_attention needs a caller-provided workspace for its split-KV
// partial results.  Some callers cannot provide one.  A serving engine may
// have handed nearly all free device memory to its KV-cache pool at start-up,
// so a later cudaMalloc fails.  A plugin may run inside a host application
// that owns every device allocation.  Real-time code cannot accept the
// device-wide synchronisation a cudaMalloc or cudaFree can cause.  For these
// callers this file keeps a fixed scratch area in the library's own static
// device memory and runs the regular decode on it.
//
// The area is one file-scope __device__ array of TQ_NOALLOC_SCRATCH_BYTES.
// Every GPU that loads the library holds it until the process exits.  In
// host code the array's name is not a device address, so its address is
// looked up once per device with cudaGetSymbolAddress and cached.
#include <cstdio>
#include <mutex>

#include <cuda_runtime.h>

#include "tq.h"
#include "tq_internal.h"

namespace {

constexpr size_t kScratchBytes = static_cast<size_t>(TQ_NOALLOC_SCRATCH_BYTES);
constexpr int kMaxDevices = 64;

// Zero when the module loads.  The decode kernels need no zeroed scratch
// between calls: every call writes each partial it later reads.
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device `dev`.  The
// first call on a device looks it up; later calls reuse the cached address.
cudaError_t scratch_on(int dev, void** ptr) {
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *ptr = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" {

tq_status tq_decode_attention_noalloc(const tq_config* cfg, const void* q_dev, int32_t num_seqs,
                                      int32_t num_q_heads, const tq_cache* cache, const int32_t* block_table_dev,
                                      int32_t max_blocks_per_seq, const int32_t* seq_lens_dev, int32_t max_seq_len,
                                      float sm_scale, int32_t num_splits, float* out_dev, void* stream) {
    if (cache != nullptr && cfg != nullptr && num_seqs > 0 && num_q_heads > 0) {
        size_t need = tq_decode_workspace_size(cfg, num_seqs, num_q_heads, cache->num_kv_heads,
                                               cache->block_size, max_seq_len, num_splits);
        if (need > kScratchBytes && num_splits == 0 && cfg->head_dim > 0) {
            // The automatic split count does not fit: take the most splits
            // whose partial states do fit (fewer splits only lengthen each
            // CTA's share of the sequence; the result is the same decode).
            const size_t per_split = static_cast<size_t>(num_seqs) * static_cast<size_t>(num_q_heads) *
                                     (static_cast<size_t>(cfg->head_dim) + 2) * sizeof(float);
            int32_t splits = static_cast<int32_t>(kScratchBytes / per_split);
            while (splits >= 1) {
                need = tq_decode_workspace_size(cfg, num_seqs, num_q_heads, cache->num_kv_heads, cache->block_size,
                                                max_seq_len, splits);
                if (need <= kScratchBytes) break;
                --splits;
            }
            if (splits >= 1) num_splits = splits;
        }
        if (need > kScratchBytes) {
            char msg[256];
            std::snprintf(msg, sizeof msg,
                          "this decode needs %zu bytes of scratch but the no-allocation entry point has %zu; "
                          "use fewer sequences or splits, or tq_decode_attention with a workspace",
                          need, kScratchBytes);
            tq::set_last_error(msg);
            return TQ_ERR_WORKSPACE;
        }
    }
    int dev = 0;
    void* scratch = nullptr;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = scratch_on(dev, &scratch);
    if (e != cudaSuccess) {
        char msg[256];
        std::snprintf(msg, sizeof msg, "no-allocation scratch lookup: %s (%s)", cudaGetErrorName(e),
                      cudaGetErrorString(e));
        tq::set_last_error(msg);
        return TQ_ERR_CUDA;
    }
    return tq_decode_attention(cfg, q_dev, num_seqs, num_q_heads, cache, block_table_dev, max_blocks_per_seq,
                               seq_lens_dev, max_seq_len, sm_scale, num_splits, out_dev, scratch, kScratchBytes,
                               stream);
}

}  // extern "C"
