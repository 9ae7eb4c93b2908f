// Dense decode attention over bf16 K and V: the comparison path.
//
// [ART] hnwysp.cn TurboQuant article, "Obstacle 1": the hybrid-model path
// stores the compressed cache but, at every decode step, expands the whole
// history back to full precision and runs ordinary attention over it
// ("storage yes, compute no").  This file is the second half of that path on
// the GPU: after tq_dequant has written every cached token of the batch as
// bf16 K and V rows, one warp per (split, sequence, KV head) runs an online
// softmax over its share of the rows, and the split merge of the fused
// decode (combine_kernel) finishes the job.  It exists to measure what the
// fused decode saves; the fused decode never materialises K or V.
//
// Lane layout.  A token's head vector (D bf16) is read by LPT = D / 8 lanes,
// 16 bytes each (8 consecutive dims); a warp covers TPW = 32 / LPT tokens per
// step and unrolls U steps so that 2U 16-byte loads per lane are in flight.
// A lane group's score is its lanes' partial dot products summed by xor
// shuffles; each lane group keeps its own running (m, l, o) for the G query
// heads of the KV head, merged across the groups at the end.
#include <cuda_runtime.h>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kDenseUnroll = 4;

__device__ __forceinline__ float exp2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4 w, float (&x)[8]) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(u[i] << 16);
        x[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
    }
}

template <int D, int G>
__global__ void __launch_bounds__(32)
dense_decode_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                    const uint16_t* __restrict__ v, const int32_t* __restrict__ cu_seqlens, int num_kv_heads,
                    int max_seq_len, int tokens_per_split, float qscale, float* __restrict__ partials,
                    int num_splits) {
    constexpr int LPT = D / 8;
    constexpr int TPW = 32 / LPT;
    const int lane = threadIdx.x;
    const int part = lane % LPT;  // dims [8 part, 8 part + 8)
    const int grp = lane / LPT;   // token slot within a step
    const int split = blockIdx.x;
    const int s = blockIdx.y;
    const int h = blockIdx.z;
    const int H = num_kv_heads;
    const int Hq = H * G;
    const int64_t row0 = cu_seqlens[s];
    int n = cu_seqlens[s + 1] - cu_seqlens[s];
    n = n < 0 ? 0 : (n > max_seq_len ? max_seq_len : n);
    const int t0 = split * tokens_per_split;
    const int t1 = min(n, t0 + tokens_per_split);

    // the G query rows of this KV head, this lane's 8 dims, in log2 units
    float qv[G][8];
#pragma unroll
    for (int j = 0; j < G; ++j) {
        const uint4 w = *reinterpret_cast<const uint4*>(q + (static_cast<int64_t>(s) * Hq + h * G + j) * D + 8 * part);
        bf16x8_to_f32(w, qv[j]);
#pragma unroll
        for (int e = 0; e < 8; ++e) qv[j][e] *= qscale;
    }
    float m[G], l[G], o[G][8];
#pragma unroll
    for (int j = 0; j < G; ++j) {
        m[j] = -INFINITY;
        l[j] = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) o[j][e] = 0.f;
    }
    const int64_t row_stride = static_cast<int64_t>(H) * D;  // elements between consecutive tokens
    const uint16_t* kb = k + (row0 * H + h) * D + 8 * part;
    const uint16_t* vb = v + (row0 * H + h) * D + 8 * part;

    for (int base = t0; base < t1; base += TPW * kDenseUnroll) {
        uint4 kw[kDenseUnroll], vw[kDenseUnroll];
        bool ok[kDenseUnroll];
#pragma unroll
        for (int u = 0; u < kDenseUnroll; ++u) {
            const int t = base + u * TPW + grp;
            ok[u] = t < t1;
            const int tc = ok[u] ? t : t0;  // in range: re-read a valid row
            kw[u] = __ldg(reinterpret_cast<const uint4*>(kb + tc * row_stride));
            vw[u] = __ldg(reinterpret_cast<const uint4*>(vb + tc * row_stride));
        }
        float sc[kDenseUnroll][G];
#pragma unroll
        for (int u = 0; u < kDenseUnroll; ++u) {
            float kx[8];
            bf16x8_to_f32(kw[u], kx);
#pragma unroll
            for (int j = 0; j < G; ++j) {
                float acc = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc = fmaf(qv[j][e], kx[e], acc);
                sc[u][j] = acc;
            }
        }
#pragma unroll
        for (int off = LPT / 2; off > 0; off >>= 1) {
#pragma unroll
            for (int u = 0; u < kDenseUnroll; ++u)
#pragma unroll
                for (int j = 0; j < G; ++j) sc[u][j] += __shfl_xor_sync(kFull, sc[u][j], off);
        }
#pragma unroll
        for (int j = 0; j < G; ++j) {
            float mx = m[j];
#pragma unroll
            for (int u = 0; u < kDenseUnroll; ++u) mx = ok[u] ? fmaxf(mx, sc[u][j]) : mx;
            if (mx == -INFINITY) continue;  // no token of this lane group yet
            const float alpha = exp2_approx(m[j] - mx);
            l[j] *= alpha;
#pragma unroll
            for (int e = 0; e < 8; ++e) o[j][e] *= alpha;
            m[j] = mx;
        }
#pragma unroll
        for (int u = 0; u < kDenseUnroll; ++u) {
            float vx[8];
            bf16x8_to_f32(vw[u], vx);
#pragma unroll
            for (int j = 0; j < G; ++j) {
                const float p = ok[u] ? exp2_approx(sc[u][j] - m[j]) : 0.f;
                l[j] += p;
#pragma unroll
                for (int e = 0; e < 8; ++e) o[j][e] = fmaf(p, vx[e], o[j][e]);
            }
        }
    }

    // merge the lane groups (lanes part, part + LPT, ...)
#pragma unroll
    for (int off = LPT; off < 32; off <<= 1) {
#pragma unroll
        for (int j = 0; j < G; ++j) {
            const float om = __shfl_xor_sync(kFull, m[j], off);
            const float ol = __shfl_xor_sync(kFull, l[j], off);
            const float nm = fmaxf(m[j], om);
            const float a = nm == -INFINITY ? 0.f : exp2_approx(m[j] - nm);
            const float b = nm == -INFINITY ? 0.f : exp2_approx(om - nm);
            l[j] = l[j] * a + ol * b;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float oo = __shfl_xor_sync(kFull, o[j][e], off);
                o[j][e] = o[j][e] * a + oo * b;
            }
            m[j] = nm;
        }
    }
    if (grp != 0) return;
#pragma unroll
    for (int j = 0; j < G; ++j) {
        float* dst = partials + ((static_cast<int64_t>(s) * Hq + h * G + j) * num_splits + split) * (D + 2);
        if (part == 0) {
            dst[0] = m[j];
            dst[1] = l[j];
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) dst[2 + 8 * part + e] = o[j][e];
    }
}

template <int D>
cudaError_t launch_d(int group, const uint16_t* q, const uint16_t* k, const uint16_t* v, const int32_t* cu,
                     int num_seqs, int num_kv_heads, int max_seq_len, int tps, float qscale, float* partials,
                     int splits, cudaStream_t stream) {
    const dim3 grid(static_cast<unsigned>(splits), static_cast<unsigned>(num_seqs),
                    static_cast<unsigned>(num_kv_heads));
    switch (group) {
#define TQ_DENSE_CASE(GG)                                                                               \
    case GG:                                                                                            \
        dense_decode_kernel<D, GG><<<grid, 32, 0, stream>>>(q, k, v, cu, num_kv_heads, max_seq_len, tps, \
                                                            qscale, partials, splits);                  \
        break;
        TQ_DENSE_CASE(1)
        TQ_DENSE_CASE(2)
        TQ_DENSE_CASE(3)
        TQ_DENSE_CASE(4)
        TQ_DENSE_CASE(5)
        TQ_DENSE_CASE(6)
        TQ_DENSE_CASE(7)
        TQ_DENSE_CASE(8)
#undef TQ_DENSE_CASE
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

DensePlan plan_dense(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int max_seq_len, int sm_count) {
    // About 24 warps per SM in all: enough splits of at least 64 tokens.
    DensePlan plan{};
    const long long base = static_cast<long long>(num_seqs) * num_kv_heads;
    const long long target = static_cast<long long>(sm_count > 0 ? sm_count : 1) * 24;
    long long splits = base > 0 ? (target + base - 1) / base : 1;
    const long long max_splits = (static_cast<long long>(max_seq_len) + 63) / 64;
    if (splits > max_splits) splits = max_splits;
    if (splits < 1) splits = 1;
    const long long tps = max_seq_len > 0 ? (max_seq_len + splits - 1) / splits : 1;
    splits = max_seq_len > 0 ? (max_seq_len + tps - 1) / tps : 1;
    plan.num_splits = static_cast<int32_t>(splits);
    plan.tokens_per_split = static_cast<int32_t>(tps);
    size_t bytes = static_cast<size_t>(num_seqs) * num_q_heads * splits * (head_dim + 2) * sizeof(float);
    plan.workspace_bytes = bytes == 0 ? 256 : ((bytes + 255) & ~static_cast<size_t>(255));
    return plan;
}

cudaError_t launch_dense_decode(int head_dim, const uint16_t* q, int num_seqs, int num_q_heads, int num_kv_heads,
                                const uint16_t* k, const uint16_t* v, const int32_t* cu_seqlens, int max_seq_len,
                                float sm_scale, const DensePlan& plan, float* out, void* workspace,
                                cudaStream_t stream) {
    const int group = num_q_heads / num_kv_heads;
    float* partials = static_cast<float*>(workspace);
    const float qscale = sm_scale * 1.4426950408889634f;
    cudaError_t e = cudaErrorInvalidValue;
    switch (head_dim) {
        case 16: e = launch_d<16>(group, q, k, v, cu_seqlens, num_seqs, num_kv_heads, max_seq_len, plan.tokens_per_split, qscale, partials, plan.num_splits, stream); break;
        case 32: e = launch_d<32>(group, q, k, v, cu_seqlens, num_seqs, num_kv_heads, max_seq_len, plan.tokens_per_split, qscale, partials, plan.num_splits, stream); break;
        case 64: e = launch_d<64>(group, q, k, v, cu_seqlens, num_seqs, num_kv_heads, max_seq_len, plan.tokens_per_split, qscale, partials, plan.num_splits, stream); break;
        case 128: e = launch_d<128>(group, q, k, v, cu_seqlens, num_seqs, num_kv_heads, max_seq_len, plan.tokens_per_split, qscale, partials, plan.num_splits, stream); break;
        case 256: e = launch_d<256>(group, q, k, v, cu_seqlens, num_seqs, num_kv_heads, max_seq_len, plan.tokens_per_split, qscale, partials, plan.num_splits, stream); break;
        default: break;
    }
    if (e != cudaSuccess) return e;
    return launch_combine(partials, out, num_seqs, num_q_heads, head_dim, plan.num_splits, stream, false);
}

}  // namespace tq
