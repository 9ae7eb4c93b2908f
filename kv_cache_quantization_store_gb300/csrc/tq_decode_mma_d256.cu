// Tensor-core decode kernels for head size 256 (all key/value widths and
// KV-head counts the dispatcher supports).
#include "tq_decode_mma.cuh"

namespace tq {

cudaError_t decode_mma_run_d256(const LayerParams& p, const CacheGeom& c, const mma::Args& a, int num_seqs,
                               int num_kv_heads, cudaStream_t stream, int* ctas) {
    return mma::run<256>(p, c, a, num_seqs, num_kv_heads, stream, ctas);
}

}  // namespace tq
