// Decode host entry (launch_decode) and the kernels around the
// tensor-core decode of tq_decode_mma.cuh:
//   - the CUDA-core decode for the shapes the tensor-core path does not
//     take (d < 64, other KV-head counts, G > 8);
//   - the split planner;
//   - the log-sum-exp merge of the split partials;
//   - the ring rows' partial state and the side stream it runs on.
//
// [ART] hnwysp.cn TurboQuant article, "Direction 1": score the rotated query
// against the compressed keys (q . k_hat = vec_norm * (Pi q) . c~), run an
// online softmax block by block, never expand K or V.  [TQC] norm_correction
// divides by ||c~|| (the centroid vector's norm).
//
// CUDA-core decode.  Grid: (split, sequence).  A CTA walks its range of
// 16-token chunks; each chunk is the contiguous span of 16 token rows (all
// KV heads) inside one paged block, staged into shared memory with 16-byte
// cp.async copies (double-buffered).  Per chunk:
//   1. scores: (token, head) items, a few threads each, dot the rotated,
//      pre-scaled queries with the looked-up centroids (or FP8 keys);
//   2. online-softmax update per query head (max, rescale, probabilities);
//   3. P.V: warp h owns KV head h, each lane d/32 dims of all its queries.
// Each CTA writes a partial (m, l, o) per query head; the merge kernel
// combines the splits by log-sum-exp.
#include <cmath>

#include <mutex>

#include "tq_device.cuh"

namespace tq {
namespace {

constexpr int kThreads = 256;
constexpr int kTokPerChunk = 16;
constexpr int kMaxG = 8;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

struct DecodeArgs {
    const uint16_t* q;
    const int32_t* block_table;
    const int32_t* seq_lens;
    float* partials;  // [S, Hq, slot_stride, D + 2]
    int num_q_heads;
    int max_blocks;
    int max_seq_len;
    int chunks_per_split;
    int num_splits;
    int slot_stride;  // partial slots per (sequence, query head)
    int ring_tokens;  // > 0: the last L mod ring_tokens tokens are in an exact ring, not in the cache
    float qscale;     // sm_scale * log2(e)
};

__host__ __device__ constexpr int align16(int x) { return (x + 15) & ~15; }

// Shared-memory layout (bytes), all offsets 16-byte aligned.
struct SmemLayout {
    int q_off, sc_off, st_off, buf_off, buf_bytes, total;
    __host__ __device__ SmemLayout(int hq, int d, int h, int slot_al) {
        q_off = 0;
        sc_off = align16(q_off + hq * d * 4);
        st_off = align16(sc_off + hq * kTokPerChunk * 4);
        buf_off = align16(st_off + (3 * hq + 16) * 4);
        buf_bytes = kTokPerChunk * h * slot_al;
        total = buf_off + 2 * buf_bytes;
    }
};

template <int D, int KB, int VB>
__global__ void __launch_bounds__(kThreads)
decode_kernel(const LayerParams p, const CacheGeom c, const DecodeArgs a) {
    using S = Slot<D, KB, VB>;
    constexpr int SA = S::kAligned;
    constexpr int DPT = D >= 32 ? D / 32 : 1;  // P.V dims per lane
    extern __shared__ __align__(16) uint8_t smem[];

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int split = blockIdx.x;
    const int s = blockIdx.y;
    const int H = c.num_kv_heads;
    const int Hq = a.num_q_heads;
    const int G = Hq / H;
    const SmemLayout lay(Hq, D, H, SA);
    float* qs = reinterpret_cast<float*>(smem + lay.q_off);   // [Hq][D] rotated, scaled queries
    float* sc = reinterpret_cast<float*>(smem + lay.sc_off);  // [Hq][16] scores -> probabilities
    float* m_s = reinterpret_cast<float*>(smem + lay.st_off); // [Hq]
    float* l_s = m_s + Hq;
    float* al_s = l_s + Hq;
    float* ctab = al_s + Hq;                                  // [16] centroids
    uint8_t* bufs = smem + lay.buf_off;

    // ---- sequence range ----------------------------------------------------
    int L = a.seq_lens[s];
    if (a.ring_tokens > 0 && L > 0) L -= L % a.ring_tokens;  // packed positions: the whole ring blocks
    const int cap = min(a.max_seq_len, a.max_blocks * c.block_size);
    if (L > cap || L < 0) {
        if (tid == 0 && split == 0) set_flag(c.flags, kFlagSeq);
        L = L < 0 ? 0 : cap;
    }
    const int n_chunks = (L + kTokPerChunk - 1) / kTokPerChunk;
    const int c0 = split * a.chunks_per_split;
    const int c1 = min(c0 + a.chunks_per_split, n_chunks);

    // ---- prologue: queries -> Pi q (MSE keys) scaled for exp2 ---------------
    const uint16_t* qg = a.q + static_cast<int64_t>(s) * Hq * D;
    for (int i = tid; i < Hq * D; i += kThreads) {
        float x = __uint_as_float(static_cast<uint32_t>(qg[i]) << 16);
        if constexpr (KB != 8) {
            const int dim = i % D;
            if ((p.sign_mask[dim >> 5] >> (dim & 31)) & 1u) x = -x;
        }
        qs[i] = x;
    }
    if constexpr (KB != 8) {
#pragma unroll 1
        for (int st = 1; st < D; st <<= 1) {
            __syncthreads();
            for (int b = tid; b < Hq * D / 2; b += kThreads) {
                const int row = b / (D / 2);
                const int j = b % (D / 2);
                const int i = (j / st) * 2 * st + (j % st);
                float* r = qs + row * D;
                const float x0 = r[i], x1 = r[i + st];
                r[i] = x0 + x1;
                r[i + st] = x0 - x1;
            }
        }
    }
    __syncthreads();
    {
        const float f = (KB != 8) ? a.qscale * rsqrtf(static_cast<float>(D)) : a.qscale;
        for (int i = tid; i < Hq * D; i += kThreads) qs[i] *= f;
    }
    if (tid < Hq) {
        m_s[tid] = -INFINITY;
        l_s[tid] = 0.f;
        al_s[tid] = 1.f;
    }
    if (tid < 16) ctab[tid] = tid < p.n_centroids ? p.centroids[tid] : 0.f;

    // ---- chunk staging ------------------------------------------------------
    auto chunk_block = [&](int ci) -> int {
        const int b = a.block_table[static_cast<int64_t>(s) * a.max_blocks + (ci * kTokPerChunk) / c.block_size];
        return (b >= 0 && b < c.num_blocks) ? b : -1;
    };
    auto stage = [&](int ci, uint8_t* dst) {
        const int b = chunk_block(ci);
        if (b < 0) return;
        const uint8_t* src = c.data + static_cast<int64_t>(b) * c.block_stride +
                             static_cast<int64_t>((ci * kTokPerChunk) % c.block_size) * H * SA;
        const int pieces = lay.buf_bytes / 16;
        for (int i = tid; i < pieces; i += kThreads) cp_async16(dst + 16 * i, src + 16 * i);
    };

    // P.V accumulators: warp h = KV head h, lane owns dims [lane*DPT, +DPT).
    float o[kMaxG][DPT];
#pragma unroll
    for (int g = 0; g < kMaxG; ++g)
#pragma unroll
        for (int k = 0; k < DPT; ++k) o[g][k] = 0.f;

    // Score work split: 16*H (token, head) items, tpi threads each.  When
    // tpi > 1, items * tpi is a multiple of 32, so the shuffles below run in
    // whole warps.
    const int items = kTokPerChunk * H;
    int tpi = 1;
    while (tpi * 2 * items <= kThreads && tpi * 2 <= 32 && tpi * 2 <= D) tpi *= 2;
    const int item = tid / tpi;
    const int sub = tid % tpi;
    const int dpt = D / tpi;

    if (c0 < c1) stage(c0, bufs);
    cp_async_commit();
#pragma unroll 1
    for (int ci = c0; ci < c1; ++ci) {
        uint8_t* cur = bufs + ((ci - c0) & 1) * lay.buf_bytes;
        if (ci + 1 < c1) stage(ci + 1, bufs + ((ci + 1 - c0) & 1) * lay.buf_bytes);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        const bool chunk_ok = chunk_block(ci) >= 0;
        if (!chunk_ok && tid == 0) set_flag(c.flags, kFlagBlock);
        const int tok0 = ci * kTokPerChunk;

        // 1. scores
        if (item < items) {
            const int t = item % kTokPerChunk;
            const int h = item / kTokPerChunk;
            const uint8_t* slot = cur + (t * H + h) * SA;
            float acc[kMaxG];
#pragma unroll
            for (int g = 0; g < kMaxG; ++g) acc[g] = 0.f;
            float nsq = 0.f;
            const float* qrow = qs + h * G * D;
#pragma unroll 4
            for (int i = sub * dpt; i < (sub + 1) * dpt; ++i) {
                float cv;
                if constexpr (KB == 8) {
                    cv = e4m3_to_float(slot[i]);
                } else {
                    const int bit = i * KB;
                    const uint32_t win = static_cast<uint32_t>(slot[bit >> 3]) |
                                         (static_cast<uint32_t>(slot[(bit >> 3) + 1]) << 8);
                    cv = ctab[(win >> (bit & 7)) & ((1u << KB) - 1u)];
                    nsq = fmaf(cv, cv, nsq);
                }
#pragma unroll
                for (int g = 0; g < kMaxG; ++g)
                    if (g < G) acc[g] = fmaf(qrow[g * D + i], cv, acc[g]);
            }
            for (int m = 1; m < tpi; m <<= 1) {
#pragma unroll
                for (int g = 0; g < kMaxG; ++g) acc[g] += __shfl_xor_sync(kFull, acc[g], m);
                nsq += __shfl_xor_sync(kFull, nsq, m);
            }
            if (sub == 0) {
                const bool ok = chunk_ok && (tok0 + t < L);
                float f = 1.f;
                if constexpr (KB != 8) {
                    f = half_from_bits(*reinterpret_cast<const uint16_t*>(slot + S::kKeyIdxBytes));
                    if (p.nc) f = f / sqrtf(nsq);
                }
#pragma unroll
                for (int g = 0; g < kMaxG; ++g)
                    if (g < G) sc[(h * G + g) * kTokPerChunk + t] = ok ? acc[g] * f : -INFINITY;
            }
        }
        __syncthreads();

        // 2. online softmax state per query head
        if (tid < Hq) {
            float* row = sc + tid * kTokPerChunk;
            const float m_old = m_s[tid];
            float mx = m_old;
#pragma unroll
            for (int t = 0; t < kTokPerChunk; ++t) mx = fmaxf(mx, row[t]);
            const float alpha = (mx == -INFINITY) ? 1.f : exp2f(m_old - mx);
            float sum = 0.f;
#pragma unroll
            for (int t = 0; t < kTokPerChunk; ++t) {
                const float pr = (row[t] == -INFINITY) ? 0.f : exp2f(row[t] - mx);
                row[t] = pr;
                sum += pr;
            }
            l_s[tid] = l_s[tid] * alpha + sum;
            m_s[tid] = mx;
            al_s[tid] = alpha;
        }
        __syncthreads();

        // 3. P.V
        if (warp < H && (D >= 32 || lane < D)) {
            const int h = warp;
#pragma unroll
            for (int g = 0; g < kMaxG; ++g) {
                if (g < G) {
                    const float al = al_s[h * G + g];
#pragma unroll
                    for (int k = 0; k < DPT; ++k) o[g][k] *= al;
                }
            }
            const int ntok = chunk_ok ? min(kTokPerChunk, L - tok0) : 0;
            for (int t = 0; t < ntok; ++t) {
                const uint8_t* slot = cur + (t * H + h) * SA;
                const uint16_t* sz = reinterpret_cast<const uint16_t*>(slot + S::kKeyBytes + S::kValCodeBytes);
                const float vs = half_from_bits(sz[0]);
                const float vz = half_from_bits(sz[1]);
                const uint8_t* codes = slot + S::kKeyBytes;
                float val[DPT];
#pragma unroll
                for (int k = 0; k < DPT; ++k) {
                    const int i = lane * DPT + k;
                    const int bit = i * VB;
                    const uint32_t win = static_cast<uint32_t>(codes[bit >> 3]) |
                                         (static_cast<uint32_t>(codes[(bit >> 3) + 1]) << 8);
                    val[k] = fmaf(vs, static_cast<float>((win >> (bit & 7)) & ((1u << VB) - 1u)), vz);
                }
#pragma unroll
                for (int g = 0; g < kMaxG; ++g) {
                    if (g < G) {
                        const float pr = sc[(h * G + g) * kTokPerChunk + t];
#pragma unroll
                        for (int k = 0; k < DPT; ++k) o[g][k] = fmaf(pr, val[k], o[g][k]);
                    }
                }
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();

    // ---- partial state -------------------------------------------------------
    if (warp < H && (D >= 32 || lane < D)) {
        const int h = warp;
#pragma unroll
        for (int g = 0; g < kMaxG; ++g) {
            if (g < G) {
                const int hq = h * G + g;
                float* part = a.partials + ((static_cast<int64_t>(s) * Hq + hq) * a.slot_stride + split) * (D + 2);
                if (lane == 0) {
                    part[0] = m_s[hq];
                    part[1] = l_s[hq];
                }
#pragma unroll
                for (int k = 0; k < DPT; ++k) part[2 + lane * DPT + k] = o[g][k];
            }
        }
    }
}

// Log-sum-exp merge of the split partials: one CTA per (query head,
// sequence) with nw warps (nw grows with the split count), or, for up to
// 8 splits, one warp per (sequence, query head) and 8 of them per CTA.
// Warp w merges splits w, w + nw, ... on its own: its lanes first fold the
// splits' (m, l) with a running maximum, then sum the weighted o over those
// splits (two dims per lane and load, the splits' loads independent of one
// another).  With several warps their (m, l, o) meet in shared memory.
constexpr int kCombineMaxWarps = 8;

// 2^(m - M), 0 for a split without tokens (m = -inf)
__device__ __forceinline__ float lse_weight(float m, float M) { return m == -INFINITY ? 0.f : exp2f(m - M); }

__global__ void __launch_bounds__(32 * kCombineMaxWarps)
combine_kernel(const float* __restrict__ partials, float* __restrict__ out, int num_seqs, int Hq, int D,
               int num_splits, int one_warp) {
    __shared__ float wm[kCombineMaxWarps], wl[kCombineMaxWarps];
    __shared__ float wacc[kCombineMaxWarps][256];
    const int lane = threadIdx.x & 31;
    int warp = threadIdx.x >> 5, nw = blockDim.x >> 5, hq, s;
    if (one_warp) {
        // few splits: each warp merges one (sequence, query head) on its own
        const int pair = blockIdx.x * nw + warp;
        if (pair >= num_seqs * Hq) return;
        s = pair / Hq;
        hq = pair - s * Hq;
        warp = 0;
        nw = 1;
    } else {
        hq = blockIdx.x;
        s = blockIdx.y;
    }
    grid_dependency_wait();  // the decode grid has finished writing the partials
    const int row = D + 2;
    const float* base = partials + (static_cast<int64_t>(s) * Hq + hq) * num_splits * row;
    // (m, l) of this warp's splits, folded per lane, then across the lanes
    float M = -INFINITY, L = 0.f;
    for (int sp = warp + nw * lane; sp < num_splits; sp += 32 * nw) {
        const float m = base[static_cast<int64_t>(sp) * row], l = base[static_cast<int64_t>(sp) * row + 1];
        const float nm = fmaxf(M, m);
        L = L * lse_weight(M, nm) + l * lse_weight(m, nm);
        M = nm;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, M, o), ol = __shfl_xor_sync(0xffffffffu, L, o);
        const float nm = fmaxf(M, om);
        L = L * lse_weight(M, nm) + ol * lse_weight(om, nm);
        M = nm;
    }
    // weighted o of this warp's splits: lane covers float2 columns lane + 32 j
    float2 acc[4] = {};
    const int ncol = D / 2;
    if (M != -INFINITY) {
#pragma unroll 4
        for (int sp = warp; sp < num_splits; sp += nw) {
            const float* ps = base + static_cast<int64_t>(sp) * row;
            const float w = lse_weight(ps[0], M);
            const float2* o2 = reinterpret_cast<const float2*>(ps + 2);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int col = lane + 32 * j;
                if (col < ncol) {
                    const float2 o = o2[col];
                    acc[j].x = fmaf(o.x, w, acc[j].x);
                    acc[j].y = fmaf(o.y, w, acc[j].y);
                }
            }
        }
    }
    float* dst = out + (static_cast<int64_t>(s) * Hq + hq) * D;
    if (nw == 1) {
        const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int col = lane + 32 * j;
            if (col < ncol) {  // out is only 4-byte aligned
                dst[2 * col] = acc[j].x * inv;
                dst[2 * col + 1] = acc[j].y * inv;
            }
        }
        return;
    }
    if (lane == 0) {
        wm[warp] = M;
        wl[warp] = L;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int col = lane + 32 * j;
        if (col < ncol) {
            wacc[warp][2 * col] = acc[j].x;
            wacc[warp][2 * col + 1] = acc[j].y;
        }
    }
    __syncthreads();
    float Mt = -INFINITY;
    for (int w = 0; w < nw; ++w) Mt = fmaxf(Mt, wm[w]);
    float Lt = 0.f;
    for (int w = 0; w < nw; ++w) Lt = fmaf(wl[w], lse_weight(wm[w], Mt), Lt);
    const float inv = Lt > 0.f ? 1.f / Lt : 0.f;
    for (int i = threadIdx.x; i < D; i += blockDim.x) {
        float a = 0.f;
        for (int w = 0; w < nw; ++w) a = fmaf(wacc[w][i], lse_weight(wm[w], Mt), a);
        dst[i] = a * inv;
    }
}

template <int D, int KB, int VB>
cudaError_t launch(const LayerParams& p, const CacheGeom& c, const DecodeArgs& a, int num_seqs,
                   cudaStream_t stream) {
    const SmemLayout lay(a.num_q_heads, D, c.num_kv_heads, Slot<D, KB, VB>::kAligned);
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, KB, VB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         lay.total);
    if (e != cudaSuccess) return e;
    dim3 grid(static_cast<unsigned>(a.num_splits), static_cast<unsigned>(num_seqs));
    decode_kernel<D, KB, VB><<<grid, kThreads, lay.total, stream>>>(p, c, a);
    return cudaGetLastError();
}

template <int D>
cudaError_t dispatch_bits(const LayerParams& p, const CacheGeom& c, const DecodeArgs& a, int ns, cudaStream_t st) {
    const int kb = p.kbits, vb = p.vbits;
    if (kb == 3 && vb == 3) return launch<D, 3, 3>(p, c, a, ns, st);
    if (kb == 3 && vb == 4) return launch<D, 3, 4>(p, c, a, ns, st);
    if (kb == 4 && vb == 3) return launch<D, 4, 3>(p, c, a, ns, st);
    if (kb == 4 && vb == 4) return launch<D, 4, 4>(p, c, a, ns, st);
    if (kb == 8 && vb == 3) return launch<D, 8, 3>(p, c, a, ns, st);
    if (kb == 8 && vb == 4) return launch<D, 8, 4>(p, c, a, ns, st);
    return cudaErrorInvalidValue;
}

// Partial state of the exact ring rows ([ART] hnwysp.cn article: in the
// hybrid mode the newest tokens come from the exact ring): for sequence s
// of L tokens and KV head h, the n = L mod R rows 0 .. n - 1 of the ring
// (positions R floor(L / R) onward) against the G query heads of h, in the
// split partials' form (log2-domain running maximum m, l = sum 2^(s - m),
// o = sum 2^(s - m) v) in partial slot `slot`.  One CTA of kRingThreads per
// (KV head, sequence).  Scores: a row is read by D / 8 lanes, 16 bytes
// each, so a warp instruction covers 256 / D rows; each lane keeps its 8
// dims of every query in registers, and the lanes' partial dot products
// meet by shuffles.  Softmax per query over the rows in shared memory.
// P.V: each warp owns a quarter of the dims and accumulates all G outputs
// over every row.
constexpr int kRingThreads = 128;
constexpr int kRingMaxTokens = 128;

__device__ __forceinline__ void bf16x8(const uint4 u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

template <int D>
__global__ void __launch_bounds__(kRingThreads)
ring_partial_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ ring_k,
                    const uint16_t* __restrict__ ring_v, const int32_t* __restrict__ seq_lens, int R, int H, int Hq,
                    float qscale, float* __restrict__ partials, int slot_stride, int slot) {
    constexpr int kWarps = kRingThreads / 32;
    constexpr int LPT = D / 8;    // lanes per row
    constexpr int TPW = 32 / LPT; // rows per warp instruction
    constexpr int kStep = kWarps * TPW;
    __shared__ float pr[8][kRingMaxTokens];
    __shared__ float ms[8], ls[8];
    const int h = blockIdx.x, s = blockIdx.y;
    const int G = Hq / H;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane / LPT;  // row of the warp instruction
    const int u = lane % LPT;    // 16-byte unit: dims 8u .. 8u + 7
    const int L = seq_lens[s];
    const int n = L > 0 ? L % R : 0;
    const int64_t row_stride = static_cast<int64_t>(H) * D;  // one ring row: all heads
    const int64_t base = (static_cast<int64_t>(s) * R * H + h) * D + 8 * u;
    // this lane's 8 dims of every query, scaled to log2 units (2-byte loads:
    // q is only 4-byte aligned)
    float qv[8][8];
    const uint16_t* qs = q + (static_cast<int64_t>(s) * Hq + static_cast<int64_t>(h) * G) * D + 8 * u;
#pragma unroll
    for (int g = 0; g < 8; ++g)
#pragma unroll
        for (int e = 0; e < 8; ++e)
            qv[g][e] = g < G ? __uint_as_float(static_cast<uint32_t>(qs[g * D + e]) << 16) * qscale : 0.f;
    // scores: kBatch rows per lane are loaded before any is used
    constexpr int kBatch = 8;
    for (int t0 = warp * TPW + sub; t0 - sub < n; t0 += kStep * kBatch) {
        uint4 raw[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const int t = t0 + k * kStep;
            raw[k] = t < n ? *reinterpret_cast<const uint4*>(ring_k + base + t * row_stride) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const int t = t0 + k * kStep;
            float kf[8];
            bf16x8(raw[k], kf);
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                if (g >= G) break;
                float acc = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc = fmaf(qv[g][e], kf[e], acc);
#pragma unroll
                for (int o = LPT / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
                if (u == 0 && t < n) pr[g][t] = acc;
            }
        }
    }
    __syncthreads();
    // softmax per query: warp w takes queries w, w + kWarps, ...
    for (int g = warp; g < G; g += kWarps) {
        float m = -INFINITY;
        for (int t = lane; t < n; t += 32) m = fmaxf(m, pr[g][t]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float l = 0.f;
        for (int t = lane; t < n; t += 32) {
            const float e = exp2f(pr[g][t] - m);
            pr[g][t] = e;
            l += e;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) {
            ms[g] = m;
            ls[g] = l;
        }
    }
    __syncthreads();
    // P.V.  Warp w owns dims [w D/4, (w + 1) D/4) of the output and reads
    // every row's slice of them: PL lanes per row (8 dims each), PT rows per
    // warp instruction; the PT row groups meet by shuffles.  (d = 16: the
    // warps split the rows instead and meet in shared memory.)
    constexpr bool kDimSplit = D / kWarps >= 8;
    constexpr int PL = kDimSplit ? D / kWarps / 8 : LPT;
    constexpr int PT = 32 / PL;
    const int psub = lane / PL, pu = lane % PL;
    const int dim0 = kDimSplit ? warp * (D / kWarps) + 8 * pu : 8 * u;
    const int64_t vbase = (static_cast<int64_t>(s) * R * H + h) * D + dim0;
#pragma unroll
    for (int g = 0; g < 8; ++g)
#pragma unroll
        for (int e = 0; e < 8; ++e) qv[g][e] = 0.f;
    const int t_first = kDimSplit ? psub : warp * TPW + sub;
    const int t_step = kDimSplit ? PT : kStep;
    for (int t0 = t_first; t0 < n; t0 += t_step * kBatch) {
        uint4 raw[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const int t = t0 + k * t_step;
            raw[k] = t < n ? *reinterpret_cast<const uint4*>(ring_v + vbase + t * row_stride) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const int t = t0 + k * t_step;
            if (t >= n) break;
            float vf[8];
            bf16x8(raw[k], vf);
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                if (g >= G) break;
                const float pg = pr[g][t];
#pragma unroll
                for (int e = 0; e < 8; ++e) qv[g][e] = fmaf(pg, vf[e], qv[g][e]);
            }
        }
    }
    // add the row groups of the warp (lanes pu, pu + PL, ...)
#pragma unroll
    for (int o = PL; o < 32; o <<= 1)
#pragma unroll
        for (int g = 0; g < 8; ++g)
#pragma unroll
            for (int e = 0; e < 8; ++e) qv[g][e] += __shfl_xor_sync(0xffffffffu, qv[g][e], o);
    auto part_of = [&](int g) -> float* {
        return partials + ((static_cast<int64_t>(s) * Hq + h * G + g) * slot_stride + slot) * (D + 2);
    };
    if constexpr (kDimSplit) {
        if (psub == 0) {
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                if (g >= G) break;
                float* part = part_of(g);
#pragma unroll
                for (int e = 0; e < 8; ++e) part[2 + dim0 + e] = qv[g][e];
            }
        }
        if (threadIdx.x < G) {
            float* part = part_of(threadIdx.x);
            part[0] = n > 0 ? ms[threadIdx.x] : -INFINITY;
            part[1] = n > 0 ? ls[threadIdx.x] : 0.f;
        }
    } else {
        __shared__ float red[kWarps][8][D];
        if (sub == 0) {
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                if (g >= G) break;
#pragma unroll
                for (int e = 0; e < 8; ++e) red[warp][g][8 * u + e] = qv[g][e];
            }
        }
        __syncthreads();
        for (int i = threadIdx.x; i < G * D; i += kRingThreads) {
            const int g = i / D, dim = i % D;
            float o = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) o += red[w][g][dim];
            float* part = part_of(g);
            if (dim == 0) {
                part[0] = n > 0 ? ms[g] : -INFINITY;
                part[1] = n > 0 ? ls[g] : 0.f;
            }
            part[2 + dim] = o;
        }
    }
}

cudaError_t launch_ring_partial(const LayerParams& p, const uint16_t* q, const RingBuf& ring,
                                const int32_t* seq_lens, int num_seqs, int H, int Hq, float qscale, float* partials,
                                int slot_stride, int slot, cudaStream_t stream) {
    if (ring.tokens <= 0 || ring.tokens > kRingMaxTokens || Hq % H != 0 || Hq / H > 8) return cudaErrorInvalidValue;
    dim3 grid(static_cast<unsigned>(H), static_cast<unsigned>(num_seqs));
    switch (p.d) {
#define TQ_RING_CASE(DD)                                                                                  \
    case DD:                                                                                              \
        ring_partial_kernel<DD><<<grid, kRingThreads, 0, stream>>>(q, ring.k, ring.v, seq_lens, ring.tokens, \
                                                                   H, Hq, qscale, partials, slot_stride, slot); \
        break;
        TQ_RING_CASE(16)
        TQ_RING_CASE(32)
        TQ_RING_CASE(64)
        TQ_RING_CASE(128)
        TQ_RING_CASE(256)
#undef TQ_RING_CASE
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_combine(const float* partials, float* out, int num_seqs, int num_q_heads, int d,
                           int num_splits, cudaStream_t stream, bool after_decode_kernel) {
    dim3 cgrid(static_cast<unsigned>(num_q_heads), static_cast<unsigned>(num_seqs));
    if (d > 256 || d % 2 != 0) return cudaErrorInvalidValue;
    // about 8 splits per warp, at most kCombineMaxWarps warps; with one warp
    // per (sequence, head), kCombineMaxWarps of them share a CTA
    int nw = (num_splits + 7) / 8;
    nw = nw < 1 ? 1 : (nw > kCombineMaxWarps ? kCombineMaxWarps : nw);
    // Right after the decode kernel it is launched with programmatic stream
    // serialisation: its CTAs may become resident while the decode grid
    // finishes, and wait for it on the device.  After an event wait (the
    // ring's join) it is launched plainly.
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = after_decode_kernel ? 1 : 0;
    cfg.stream = stream;
    cfg.dynamicSmemBytes = 0;
    int one_warp = 0;
    if (nw == 1) {
        const long long pairs = static_cast<long long>(num_seqs) * num_q_heads;
        cfg.gridDim = dim3(static_cast<unsigned>((pairs + kCombineMaxWarps - 1) / kCombineMaxWarps));
        cfg.blockDim = dim3(32 * kCombineMaxWarps);
        one_warp = 1;
    } else {
        cfg.gridDim = cgrid;
        cfg.blockDim = dim3(32 * nw);
    }
    return cudaLaunchKernelEx(&cfg, combine_kernel, partials, out, num_seqs, num_q_heads, d, num_splits, one_warp);
}

// Resident CTAs per SM of the CUDA-core decode for these shapes.
int v1_ctas_per_sm(const LayerParams& p, int num_kv_heads, int num_q_heads) {
    int ctas = 0;
    auto query = [&](auto kern) {
        const SmemLayout lay(num_q_heads, p.d, num_kv_heads, p.slot_al);
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, lay.total) != cudaSuccess) return;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&ctas, kern, kThreads, lay.total) != cudaSuccess) ctas = 0;
    };
    // every instantiation of a head size has the same shared memory and near the same registers
    switch (p.d) {
        case 16: query(decode_kernel<16, 4, 4>); break;
        case 32: query(decode_kernel<32, 4, 4>); break;
        case 64: query(decode_kernel<64, 4, 4>); break;
        case 128: query(decode_kernel<128, 4, 4>); break;
        case 256: query(decode_kernel<256, 4, 4>); break;
        default: break;
    }
    return ctas;
}

DecodePlan plan_decode(const LayerParams& p, int num_seqs, int num_q_heads, int num_kv_heads, int max_seq_len,
                       int num_splits_req, int sm_count, bool ring) {
    DecodePlan plan{};
    const int max_chunks = (max_seq_len + kTokPerChunk - 1) / kTokPerChunk;
    int splits = 1;
    if (num_splits_req > 0) {
        splits = num_splits_req;
    } else if (num_seqs > 0 && max_chunks > 0) {
        // Pick the split count that finishes soonest.  CTAs run in waves of
        // sm_count * (resident CTAs per SM); each costs its chunks plus a
        // fixed prologue (tables, query rotation) worth about kPrologue
        // chunks.  A last, partial wave with at most one CTA per SM runs
        // faster (its CTAs share no SM: measured about 1.6x), so it counts
        // 10/16 of a wave.  Costs are in 1/16 chunk.
        constexpr int kPrologue = 4;
        const int sms = sm_count > 0 ? sm_count : 1;
        int per_sm = decode_mma_supported(p, num_kv_heads, num_q_heads)
                         ? decode_mma_ctas_per_sm(p, num_kv_heads, num_q_heads)
                         : v1_ctas_per_sm(p, num_kv_heads, num_q_heads);
        if (per_sm < 1) per_sm = 1;
        const long long capacity = static_cast<long long>(sms) * per_sm;
        long long best_cost = -1;
        const int limit = max_chunks < 512 ? max_chunks : 512;
        for (int cand = 1; cand <= limit; ++cand) {
            const long long ctas = static_cast<long long>(num_seqs) * cand;
            const long long full = ctas / capacity, rem = ctas % capacity;
            const long long len = kPrologue + (max_chunks + cand - 1) / cand;
            const long long last = rem == 0 ? 0 : (per_sm > 1 && rem <= sms ? 10 : 16);
            const long long cost = (full * 16 + last) * len;
            if (best_cost < 0 || cost < best_cost) {
                best_cost = cost;
                splits = cand;
            }
        }
    }
    if (splits > max_chunks) splits = max_chunks;
    if (splits < 1) splits = 1;
    int cps = max_chunks > 0 ? (max_chunks + splits - 1) / splits : 0;
    if (cps > 0) splits = (max_chunks + cps - 1) / cps;
    plan.num_splits = splits;
    plan.chunks_per_split = cps;
    plan.slot_stride = splits + (ring ? 1 : 0);
    plan.partial_bytes =
        static_cast<size_t>(num_seqs) * num_q_heads * plan.slot_stride * (p.d + 2) * sizeof(float);
    plan.workspace_bytes = (plan.partial_bytes + 255) & ~static_cast<size_t>(255);
    if (plan.workspace_bytes == 0) plan.workspace_bytes = 256;
    return plan;
}

namespace {
// A non-blocking stream and two events per device for the ring partial's
// fork and join, created on first use and kept for the process (the lock
// keeps concurrent calls from interleaving their record / wait pairs).
struct Side {
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    std::mutex mu;
};

cudaError_t side_stream(Side** out) {
    constexpr int kDevs = 16;
    static Side sides[kDevs];
    static std::mutex init_mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kDevs) return cudaErrorInvalidDevice;
    Side& sd = sides[dev];
    std::lock_guard<std::mutex> lock(init_mu);
    if (sd.stream == nullptr) {
        e = cudaStreamCreateWithFlags(&sd.stream, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&sd.fork, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&sd.join, cudaEventDisableTiming);
        if (e != cudaSuccess) {
            sd.stream = nullptr;
            return e;
        }
    }
    *out = &sd;
    return cudaSuccess;
}
}  // namespace

cudaError_t launch_decode(const LayerParams& p, const CacheGeom& c, const uint16_t* q, int num_seqs,
                          int num_q_heads, const int32_t* block_table, int max_blocks_per_seq,
                          const int32_t* seq_lens, int max_seq_len, float sm_scale, const DecodePlan& plan,
                          const RingBuf& ring, float* out, void* workspace, cudaStream_t stream) {
    float* partials = static_cast<float*>(workspace);
    // With a ring, the ring rows' partial runs on a side stream next to the
    // packed decode (it needs only q, the rings and seq_lens): forked before
    // the decode is enqueued, launched after it, so that its CTAs take the
    // SM slots the decode leaves free; the combine waits for both.
    Side* side = nullptr;
    std::unique_lock<std::mutex> lock;
    cudaError_t e = cudaSuccess;
    if (ring.tokens > 0) {
        if (plan.slot_stride != plan.num_splits + 1) return cudaErrorInvalidValue;
        e = side_stream(&side);
        if (e != cudaSuccess) return e;
        lock = std::unique_lock<std::mutex>(side->mu);
        e = cudaEventRecord(side->fork, stream);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(side->stream, side->fork, 0);
        if (e != cudaSuccess) return e;
    }
    if (decode_mma_supported(p, c.num_kv_heads, num_q_heads)) {
        e = launch_decode_mma(p, c, q, num_seqs, num_q_heads, block_table, max_blocks_per_seq, seq_lens, max_seq_len,
                              sm_scale, plan, ring.tokens, workspace, stream);
    } else {
        DecodeArgs a{};
        a.q = q;
        a.block_table = block_table;
        a.seq_lens = seq_lens;
        a.partials = partials;
        a.num_q_heads = num_q_heads;
        a.max_blocks = max_blocks_per_seq;
        a.max_seq_len = max_seq_len;
        a.chunks_per_split = plan.chunks_per_split;
        a.num_splits = plan.num_splits;
        a.slot_stride = plan.slot_stride;
        a.ring_tokens = ring.tokens;
        a.qscale = sm_scale * kLog2e;
        switch (p.d) {
            case 16: e = dispatch_bits<16>(p, c, a, num_seqs, stream); break;
            case 32: e = dispatch_bits<32>(p, c, a, num_seqs, stream); break;
            case 64: e = dispatch_bits<64>(p, c, a, num_seqs, stream); break;
            case 128: e = dispatch_bits<128>(p, c, a, num_seqs, stream); break;
            case 256: e = dispatch_bits<256>(p, c, a, num_seqs, stream); break;
            default: e = cudaErrorInvalidValue; break;
        }
    }
    if (side != nullptr) {
        // join the side stream even after a failed decode launch
        cudaError_t er = launch_ring_partial(p, q, ring, seq_lens, num_seqs, c.num_kv_heads, num_q_heads,
                                             sm_scale * kLog2e, partials, plan.slot_stride, plan.num_splits,
                                             side->stream);
        const cudaError_t ej = cudaEventRecord(side->join, side->stream);
        const cudaError_t ew = ej == cudaSuccess ? cudaStreamWaitEvent(stream, side->join, 0) : ej;
        if (er == cudaSuccess) er = ew;
        if (e == cudaSuccess) e = er;
    }
    if (e != cudaSuccess) return e;
    return launch_combine(partials, out, num_seqs, num_q_heads, p.d, plan.slot_stride, stream, side == nullptr);
}

}  // namespace tq
