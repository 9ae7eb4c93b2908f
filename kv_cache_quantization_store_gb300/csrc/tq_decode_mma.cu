// Fused decode attention on the packed cache with tensor-core QK and P.V
// (mma.sync m16n8k16, f16 operands, f32 accumulation).
//
// [ART] hnwysp.cn TurboQuant article, "Direction 1": rotate the query once
// (q' = Pi q) and score it against the compressed keys; run an online
// softmax block by block; never materialise fp16 K or V.  [TQC]
// TurboQuantConfig docstring, norm_correction: divide each score by the
// norm of its centroid vector.
//
// Work decomposition.  A CTA owns one sequence's split (a range of 16-token
// chunks) and has one warp per KV head.  Each chunk -- 16 consecutive tokens
// of every head, contiguous and 16-byte aligned in a paged block -- is staged
// into shared memory with 16-byte cp.async copies through an NS-deep ring.
// A warp then turns its head's 16 slots into one m16 tile:
//
//   QK   S[16 tok x 8 q] = Khat[16 x d] * Q'^T[d x 8]   (d/16 k-steps)
//        Thread (r = lane/4, c = lane%4) feeds key dims [c d/4, (c+1) d/4)
//        of tokens r and r+8: each A register is one pair of consecutive
//        dims, looked up from a per-lane-replicated pair table in shared
//        memory (3-bit: 64 entries of {half2 c, float c0^2+c1^2}; 4-bit: 256
//        entries of half2 c), or converted from two FP8 bytes.  Q' is
//        permuted to the same dim order and split into fp16 hi + lo parts
//        (two MMAs), and the table holds the centroids times a scale chosen
//        so that their fp16 rounding error is small; together they keep the
//        scores near fp32 accuracy.
//   norm 3-bit: the table's squared sums; 4-bit: Khat*Khat (HMUL2) against
//        a ones column, one extra MMA per k-step.
//   softmax  per query column, lazily rescaled (only when the running max
//        grows by more than 2^8).
//   PV   O^T[d x 8 q] += V^T[d x 16 tok] * P'[16 tok x 8 q], P' = p * scale_t.
//        Thread r feeds value dims [r d/8, (r+1) d/8) of tokens 2c, 2c+1,
//        2c+8, 2c+9 as fp16 1 + code / 2^VB (bit placement, no conversion);
//        an extra M-tile whose row 0 is all ones accumulates sum P', which
//        removes the +1 exactly and re-centres the codes on the middle of
//        their range (halving the effect of P' rounding).  P is moved into
//        the B layout with movmatrix.  The zero points enter as
//        sum p * (zero_t + centre * scale_t) in fp32.
//
// Each warp writes a partial (m, l, o) per query head; the combine kernel of
// tq_decode.cu merges the splits by log-sum-exp.
#include <cmath>
#include <mutex>

#include "tq_device.cuh"

namespace tq {

cudaError_t launch_combine(const float* partials, float* out, int num_seqs, int num_q_heads, int d,
                           int num_splits, cudaStream_t stream);

namespace {

constexpr int kTok = 16;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

__device__ __forceinline__ void cp_async16(uint32_t smem_addr, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_addr), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
    return y;
}

// Two fp32 values -> f16x2 (lo = first element, hi = second).
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;\n" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];\n" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];\n" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint16_t lds16(uint32_t addr) {
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];\n" : "=h"(v) : "r"(addr));
    return v;
}

// NW consecutive little-endian words starting at any byte address of shared
// memory (reads one aligned word beyond the range; buffers carry padding).
template <int NW>
__device__ __forceinline__ void lds_words(uint32_t addr, uint32_t (&w)[NW]) {
    const uint32_t base = addr & ~3u;
    const uint32_t sh = (addr & 3u) * 8u;
    uint32_t raw[NW + 1];
#pragma unroll
    for (int i = 0; i <= NW; ++i) raw[i] = lds32(base + 4u * i);
#pragma unroll
    for (int i = 0; i < NW; ++i) w[i] = __funnelshift_r(raw[i], raw[i + 1], sh);
}

template <int D, int KB, int VB>
struct Geo {
    using S = Slot<D, KB, VB>;
    static constexpr int SA = S::kAligned;
    static constexpr int KSTEPS = D / 16;
    static constexpr int MTILES = D / 16;
    static constexpr int KBYTES = (D / 4) * KB / 8;  // key code bytes of one thread, one token
    static constexpr int KWORDS = (KBYTES + 3) / 4;
    static constexpr int VBITS = (D / 8) * VB;       // value code bits of one thread, one token
    static constexpr int VWORDS = (VBITS + 31) / 32;
    static constexpr int LUT_ENTRY = KB == 3 ? 8 : 4;
    static constexpr int LUT_ENTRIES = KB == 3 ? 64 : (KB == 4 ? 256 : 0);
    static constexpr int LUT_BYTES = LUT_ENTRIES * 32 * LUT_ENTRY;
    static constexpr int QFRAG_BYTES_PER_WARP = KSTEPS * 32 * 16;  // hi and lo B fragments
    static constexpr int CHUNK_BYTES_PER_HEAD = kTok * SA;
};

struct MmaArgs {
    const uint16_t* q;
    const int32_t* block_table;
    const int32_t* seq_lens;
    float* partials;
    int num_q_heads;
    int max_blocks;
    int max_seq_len;
    int chunks_per_split;
    int num_splits;
    float qscale;     // sm_scale * log2(e)
    float lut_scale;  // table value = centroid * lut_scale (= gamma * sqrt(d))
};

// Dynamic shared memory: [LUT][Q' fragments][stage ring (+16 B pad)],
// the stage ring doubles as fp32 scratch for the query rotation.
template <int D, int KB, int VB, int NS>
struct MmaSmem {
    using G = Geo<D, KB, VB>;
    int lut_off, q_off, ring_off, stage_bytes, total;
    __host__ __device__ MmaSmem(int h, int hq) {
        lut_off = 0;
        q_off = G::LUT_BYTES;
        ring_off = q_off + h * G::QFRAG_BYTES_PER_WARP;
        stage_bytes = (h * G::CHUNK_BYTES_PER_HEAD + 15) & ~15;
        int ring = NS * stage_bytes + 16;
        const int qrot = hq * D * 4;
        if (ring < qrot) ring = qrot;
        total = ring_off + ring;
    }
};

// Value codes of local dim n for two tokens as f16x2: 1 + code / 2^VB,
// tokens a in the low half and b in the high half.
template <int VB, int NW>
__device__ __forceinline__ uint32_t value_pair(const uint32_t (&wa)[NW], const uint32_t (&wb)[NW], int n) {
    constexpr int kPlace = 10 - VB;  // code lands in mantissa bits [kPlace, 10)
    constexpr uint32_t kMask = ((1u << VB) - 1u) << kPlace;
    const int bit = n * VB;
    int b0;  // first byte of a 16-bit window that holds the field
    if ((bit % 16) + VB <= 16) b0 = 2 * (bit / 16);
    else b0 = bit / 8;
    uint32_t win;
    if (b0 % 4 <= 2) {
        const int o = b0 % 4;
        const uint32_t sel = o | ((o + 1) << 4) | ((o + 4) << 8) | ((o + 5) << 12);
        win = prmt(wa[b0 / 4], wb[b0 / 4], sel);
    } else {
        const uint32_t fa = __funnelshift_r(wa[b0 / 4], wa[b0 / 4 + 1], 24);
        const uint32_t fb = __funnelshift_r(wb[b0 / 4], wb[b0 / 4 + 1], 24);
        win = prmt(fa, fb, 0x5410);
    }
    const int pos = bit - 8 * b0;  // field position inside each 16-bit half
    const int sh = kPlace - pos;
    const uint32_t x = sh >= 0 ? (win << sh) : (win >> (-sh));
    return (x & (kMask | (kMask << 16))) | 0x3C003C00u;
}

template <int D, int KB, int VB, bool NC, int NS>
__global__ void __launch_bounds__(256)
decode_mma_kernel(const LayerParams p, const CacheGeom c, const MmaArgs a) {
    using G = Geo<D, KB, VB>;
    using S = typename G::S;
    constexpr int SA = G::SA;
    constexpr float kValW = static_cast<float>(1 << VB);  // 1 / weight of a code in the fp16 operand
    constexpr float kCentre = 0.5f * static_cast<float>((1 << VB) - 1);
    extern __shared__ __align__(16) uint8_t smem[];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int r = lane >> 2;
    const int cc = lane & 3;
    const int H = c.num_kv_heads;
    const int Hq = a.num_q_heads;
    const int Gq = Hq / H;
    const int h = warp;
    const int split = blockIdx.x;
    const int s = blockIdx.y;
    const int nthreads = blockDim.x;
    const MmaSmem<D, KB, VB, NS> lay(H, Hq);
    const uint32_t smem_base = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    const uint32_t lut_base = smem_base + lay.lut_off;
    const uint32_t q_base = smem_base + lay.q_off + warp * G::QFRAG_BYTES_PER_WARP;
    const uint32_t ring_base = smem_base + lay.ring_off;

    // ---- sequence range ------------------------------------------------------
    int L = a.seq_lens[s];
    const int cap = min(a.max_seq_len, a.max_blocks * c.block_size);
    if (L > cap || L < 0) {
        if (threadIdx.x == 0 && split == 0) set_flag(c.flags, kFlagSeq);
        L = L < 0 ? 0 : cap;
    }
    const int n_chunks = (L + kTok - 1) / kTok;
    const int c0 = split * a.chunks_per_split;
    const int c1 = min(c0 + a.chunks_per_split, n_chunks);

    // ---- pair lookup table: centroids * lut_scale as fp16 ------------------------
    const float ls = a.lut_scale;
    if constexpr (KB == 3) {
        for (int i = threadIdx.x; i < 64 * 32; i += nthreads) {
            const int e = i >> 5;
            const float ca = p.centroids[e & 7] * ls;
            const float cb = p.centroids[e >> 3] * ls;
            const uint32_t hv = pack_half2(ca, cb);
            // squared norm of the fp16-rounded pair, as the MMA sees it
            const float ra = __low2float(*reinterpret_cast<const __half2*>(&hv));
            const float rb = __high2float(*reinterpret_cast<const __half2*>(&hv));
            uint2* t = reinterpret_cast<uint2*>(smem + lay.lut_off);
            t[i] = make_uint2(hv, __float_as_uint(ra * ra + rb * rb));
        }
    } else if constexpr (KB == 4) {
        for (int i = threadIdx.x; i < 256 * 32; i += nthreads) {
            const int e = i >> 5;
            const float ca = p.centroids[e & 15] * ls;
            const float cb = p.centroids[e >> 4] * ls;
            reinterpret_cast<uint32_t*>(smem + lay.lut_off)[i] = pack_half2(ca, cb);
        }
    }

    // ---- queries: q' = Pi q (MSE keys), scaled, into B fragments ---------------
    {
        float* qs = reinterpret_cast<float*>(smem + lay.ring_off);
        const uint16_t* qg = a.q + static_cast<int64_t>(s) * Hq * D;
        for (int i = threadIdx.x; i < Hq * D; i += nthreads) {
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
                for (int b = threadIdx.x; b < Hq * D / 2; b += nthreads) {
                    const int row = b / (D / 2);
                    const int j = b % (D / 2);
                    const int i = (j / st) * 2 * st + (j % st);
                    float* rw = qs + row * D;
                    const float x0 = rw[i], x1 = rw[i + st];
                    rw[i] = x0 + x1;
                    rw[i + st] = x0 - x1;
                }
            }
        }
        __syncthreads();
        // Scores come out in log2 units.  MSE keys: the table holds
        // c * lut_scale and Pi carries 1/sqrt(d); without NC the table scale
        // is divided out here (with NC it cancels in c / ||c||).
        float f = a.qscale;
        if constexpr (KB != 8) f *= rsqrtf(static_cast<float>(D)) * (NC ? 1.0f : 1.0f / ls);
        const float* qrow = qs + (h * Gq + r) * D;
        for (int j = 0; j < G::KSTEPS; ++j) {
            const int u = cc * (D / 8) + 2 * j;  // pair index of b0; b1 is u + 1
            uint32_t hi0 = 0, hi1 = 0, lo0 = 0, lo1 = 0;
            if (r < Gq) {
                const float x0 = qrow[2 * u] * f, x1 = qrow[2 * u + 1] * f;
                const float x2 = qrow[2 * u + 2] * f, x3 = qrow[2 * u + 3] * f;
                hi0 = pack_half2(x0, x1);
                hi1 = pack_half2(x2, x3);
                const __half2 h0 = *reinterpret_cast<const __half2*>(&hi0);
                const __half2 h1 = *reinterpret_cast<const __half2*>(&hi1);
                lo0 = pack_half2(x0 - __low2float(h0), x1 - __high2float(h0));
                lo1 = pack_half2(x2 - __low2float(h1), x3 - __high2float(h1));
            }
            uint4* dst = reinterpret_cast<uint4*>(smem + lay.q_off + warp * G::QFRAG_BYTES_PER_WARP);
            dst[j * 32 + lane] = make_uint4(hi0, hi1, lo0, lo1);
        }
        __syncthreads();
    }

    // ---- chunk staging -----------------------------------------------------------
    auto chunk_block = [&](int ci) -> int {
        const int b = a.block_table[static_cast<int64_t>(s) * a.max_blocks + (ci * kTok) / c.block_size];
        return (b >= 0 && b < c.num_blocks) ? b : -1;
    };
    const int stage_bytes = lay.stage_bytes;
    const int chunk_bytes = H * G::CHUNK_BYTES_PER_HEAD;
    auto issue = [&](int ci, int slot) {
        const int b = chunk_block(ci);
        if (b < 0) return;
        const uint8_t* src = c.data + static_cast<int64_t>(b) * c.block_stride +
                             static_cast<int64_t>((ci * kTok) % c.block_size) * H * SA;
        const uint32_t dst = ring_base + slot * stage_bytes;
        for (int i = threadIdx.x; i < chunk_bytes / 16; i += nthreads) cp_async16(dst + 16 * i, src + 16 * i);
    };

    // ---- running state ---------------------------------------------------------------
    float o[G::MTILES][4];
#pragma unroll
    for (int mt = 0; mt < G::MTILES; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[mt][e] = 0.f;
    float ob[4] = {0.f, 0.f, 0.f, 0.f};  // row 0: sum of P' per query column
    float m_ref[2] = {-INFINITY, -INFINITY};
    float l_acc[2] = {0.f, 0.f};
    float z_acc[2] = {0.f, 0.f};
    const uint32_t bias_a = (r == 0) ? 0x3C003C00u : 0u;
    const uint32_t a_bias[4] = {bias_a, 0u, bias_a, 0u};

    const int nch = c1 - c0;
#pragma unroll
    for (int st = 0; st < NS - 1; ++st) {
        if (st < nch) issue(c0 + st, st);
        cp_async_commit();
    }

#pragma unroll 1
    for (int it = 0; it < nch; ++it) {
        cp_async_wait<NS - 2>();
        __syncthreads();
        if (it + NS - 1 < nch) issue(c0 + it + NS - 1, (it + NS - 1) % NS);
        cp_async_commit();

        const int ci = c0 + it;
        const bool chunk_ok = chunk_block(ci) >= 0;
        if (!chunk_ok) {
            if (lane == 0 && warp == 0) set_flag(c.flags, kFlagBlock);
            continue;
        }
        const int tok0 = ci * kTok;
        const uint32_t stage = ring_base + (it % NS) * stage_bytes;
        // slot of token t, head h
        auto slot_addr = [&](int t) -> uint32_t { return stage + static_cast<uint32_t>((t * H + h) * SA); };
        const bool v_r = tok0 + r < L;
        const bool v_r8 = tok0 + r + 8 < L;

        // ---- QK ----------------------------------------------------------------
        float sacc[4] = {0.f, 0.f, 0.f, 0.f};
        float nsq[2] = {0.f, 0.f};
        float nacc[4] = {0.f, 0.f, 0.f, 0.f};
        {
            uint32_t kw0[G::KWORDS], kw1[G::KWORDS];
            lds_words(slot_addr(r) + cc * G::KBYTES, kw0);
            lds_words(slot_addr(r + 8) + cc * G::KBYTES, kw1);
#pragma unroll
            for (int j = 0; j < G::KSTEPS; ++j) {
                uint32_t af[4];
                if constexpr (KB == 3) {
                    // pair u = 2j (a0/a1) and 2j+1 (a2/a3): 6-bit fields at bit 6u
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int bit = 6 * (2 * j + e);
                        const int wi = bit / 32, off = bit % 32;
                        uint32_t x0, x1;
                        if (off + 6 <= 32) {
                            x0 = off <= 8 ? (kw0[wi] << (8 - off)) : (kw0[wi] >> (off - 8));
                            x1 = off <= 8 ? (kw1[wi] << (8 - off)) : (kw1[wi] >> (off - 8));
                        } else {
                            x0 = __funnelshift_r(kw0[wi], kw0[wi + 1], off - 8);
                            x1 = __funnelshift_r(kw1[wi], kw1[wi + 1], off - 8);
                        }
                        const uint2 t0 = lds64(lut_base + ((x0 & 0x3F00u) | (lane << 3)));
                        const uint2 t1 = lds64(lut_base + ((x1 & 0x3F00u) | (lane << 3)));
                        af[2 * e] = t0.x;
                        af[2 * e + 1] = t1.x;
                        if constexpr (NC) {
                            nsq[0] += __uint_as_float(t0.y);
                            nsq[1] += __uint_as_float(t1.y);
                        }
                    }
                } else if constexpr (KB == 4) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int bit = 8 * (2 * j + e);
                        const int wi = bit / 32, off = bit % 32;
                        const uint32_t x0 = off <= 7 ? (kw0[wi] << (7 - off)) : (kw0[wi] >> (off - 7));
                        const uint32_t x1 = off <= 7 ? (kw1[wi] << (7 - off)) : (kw1[wi] >> (off - 7));
                        af[2 * e] = lds32(lut_base + ((x0 & 0x7F80u) | (lane << 2)));
                        af[2 * e + 1] = lds32(lut_base + ((x1 & 0x7F80u) | (lane << 2)));
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int bit = 16 * (2 * j + e);
                        const int wi = bit / 32, off = bit % 32;
                        const __half2_raw h0 = __nv_cvt_fp8x2_to_halfraw2(
                            static_cast<__nv_fp8x2_storage_t>((kw0[wi] >> off) & 0xffffu), __NV_E4M3);
                        const __half2_raw h1 = __nv_cvt_fp8x2_to_halfraw2(
                            static_cast<__nv_fp8x2_storage_t>((kw1[wi] >> off) & 0xffffu), __NV_E4M3);
                        af[2 * e] = static_cast<uint32_t>(h0.x) | (static_cast<uint32_t>(h0.y) << 16);
                        af[2 * e + 1] = static_cast<uint32_t>(h1.x) | (static_cast<uint32_t>(h1.y) << 16);
                    }
                }
                // af = {tok r pair 2j, tok r+8 pair 2j, tok r pair 2j+1, tok r+8 pair 2j+1}
                const uint32_t afrag[4] = {af[0], af[1], af[2], af[3]};
                const uint4 qb = lds128(q_base + (j * 32 + lane) * 16);
                mma16816(sacc, afrag, qb.x, qb.y);
                mma16816(sacc, afrag, qb.z, qb.w);
                if constexpr (NC && KB == 4) {
                    uint32_t sq[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const __half2 x = *reinterpret_cast<const __half2*>(&afrag[e]);
                        const __half2 y = __hmul2(x, x);
                        sq[e] = *reinterpret_cast<const uint32_t*>(&y);
                    }
                    mma16816(nacc, sq, 0x3C003C00u, 0x3C003C00u);  // every column: sum of squares
                }
            }
        }

        // ---- per-token factors: vec_norm, norm correction, masking -------------
        float f_r = 1.f, f_r8 = 1.f;
        if constexpr (KB != 8) {
            f_r = half_from_bits(lds16(slot_addr(r) + S::kKeyIdxBytes));
            f_r8 = half_from_bits(lds16(slot_addr(r + 8) + S::kKeyIdxBytes));
            if constexpr (NC) {
                float n0, n1;
                if constexpr (KB == 3) {
                    n0 = nsq[0] + __shfl_xor_sync(kFull, nsq[0], 1);
                    n0 += __shfl_xor_sync(kFull, n0, 2);
                    n1 = nsq[1] + __shfl_xor_sync(kFull, nsq[1], 1);
                    n1 += __shfl_xor_sync(kFull, n1, 2);
                } else {
                    n0 = nacc[0];  // token r
                    n1 = nacc[2];  // token r + 8
                }
                f_r *= rsqrtf(n0);
                f_r8 *= rsqrtf(n1);
            }
        }
        float sc[4];
        sc[0] = v_r ? sacc[0] * f_r : -INFINITY;
        sc[1] = v_r ? sacc[1] * f_r : -INFINITY;
        sc[2] = v_r8 ? sacc[2] * f_r8 : -INFINITY;
        sc[3] = v_r8 ? sacc[3] * f_r8 : -INFINITY;

        // ---- online softmax (log2 domain), lazy rescale ---------------------------
        float mx0 = fmaxf(sc[0], sc[2]);
        float mx1 = fmaxf(sc[1], sc[3]);
#pragma unroll
        for (int m = 4; m < 32; m <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, m));
            mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, m));
        }
        const bool grow = (mx0 > m_ref[0] + kRescaleThreshold) || (mx1 > m_ref[1] + kRescaleThreshold);
        if (__any_sync(kFull, grow)) {
            const float n0 = fmaxf(m_ref[0], mx0);
            const float n1 = fmaxf(m_ref[1], mx1);
            const float al0 = (n0 == -INFINITY) ? 1.f : fast_exp2(m_ref[0] - n0);
            const float al1 = (n1 == -INFINITY) ? 1.f : fast_exp2(m_ref[1] - n1);
#pragma unroll
            for (int mt = 0; mt < G::MTILES; ++mt) {
                o[mt][0] *= al0;
                o[mt][1] *= al1;
                o[mt][2] *= al0;
                o[mt][3] *= al1;
            }
            ob[0] *= al0;
            ob[1] *= al1;
            ob[2] *= al0;
            ob[3] *= al1;
            l_acc[0] *= al0;
            l_acc[1] *= al1;
            z_acc[0] *= al0;
            z_acc[1] *= al1;
            m_ref[0] = n0;
            m_ref[1] = n1;
        }
        float pr[4];
        pr[0] = (sc[0] == -INFINITY) ? 0.f : fast_exp2(sc[0] - m_ref[0]);
        pr[1] = (sc[1] == -INFINITY) ? 0.f : fast_exp2(sc[1] - m_ref[1]);
        pr[2] = (sc[2] == -INFINITY) ? 0.f : fast_exp2(sc[2] - m_ref[0]);
        pr[3] = (sc[3] == -INFINITY) ? 0.f : fast_exp2(sc[3] - m_ref[1]);
        l_acc[0] += pr[0] + pr[2];
        l_acc[1] += pr[1] + pr[3];

        // value scale / zero of tokens r and r + 8
        const uint32_t vsz_off = S::kKeyBytes + S::kValCodeBytes;
        float vs_r = 0.f, vz_r = 0.f, vs_r8 = 0.f, vz_r8 = 0.f;
        if (v_r) {
            vs_r = half_from_bits(lds16(slot_addr(r) + vsz_off));
            vz_r = half_from_bits(lds16(slot_addr(r) + vsz_off + 2));
        }
        if (v_r8) {
            vs_r8 = half_from_bits(lds16(slot_addr(r + 8) + vsz_off));
            vz_r8 = half_from_bits(lds16(slot_addr(r + 8) + vsz_off + 2));
        }
        // zero point plus the centre of the code range (codes enter centred)
        const float zc_r = vz_r + kCentre * vs_r;
        const float zc_r8 = vz_r8 + kCentre * vs_r8;
        z_acc[0] += pr[0] * zc_r + pr[2] * zc_r8;
        z_acc[1] += pr[1] * zc_r + pr[3] * zc_r8;
        const uint32_t pb0 = movmatrix_trans(pack_half2(pr[0] * vs_r, pr[1] * vs_r));
        const uint32_t pb1 = movmatrix_trans(pack_half2(pr[2] * vs_r8, pr[3] * vs_r8));

        // ---- P.V ------------------------------------------------------------------
        {
            uint32_t w0[G::VWORDS], w1[G::VWORDS], w8[G::VWORDS], w9[G::VWORDS];
            const uint32_t voff = S::kKeyBytes + (r * (D / 8) * VB) / 8;
            lds_words(slot_addr(2 * cc) + voff, w0);
            lds_words(slot_addr(2 * cc + 1) + voff, w1);
            lds_words(slot_addr(2 * cc + 8) + voff, w8);
            lds_words(slot_addr(2 * cc + 9) + voff, w9);
#pragma unroll
            for (int mt = 0; mt < G::MTILES; ++mt) {
                uint32_t vf[4];
                vf[0] = value_pair<VB>(w0, w1, 2 * mt);
                vf[1] = value_pair<VB>(w0, w1, 2 * mt + 1);
                vf[2] = value_pair<VB>(w8, w9, 2 * mt);
                vf[3] = value_pair<VB>(w8, w9, 2 * mt + 1);
                mma16816(o[mt], vf, pb0, pb1);
            }
            mma16816(ob, a_bias, pb0, pb1);
        }
    }
    cp_async_wait<0>();

    // ---- partial state ------------------------------------------------------------------
#pragma unroll
    for (int m = 4; m < 32; m <<= 1) {
        l_acc[0] += __shfl_xor_sync(kFull, l_acc[0], m);
        l_acc[1] += __shfl_xor_sync(kFull, l_acc[1], m);
        z_acc[0] += __shfl_xor_sync(kFull, z_acc[0], m);
        z_acc[1] += __shfl_xor_sync(kFull, z_acc[1], m);
    }
    const float bias0 = __shfl_sync(kFull, ob[0], cc);
    const float bias1 = __shfl_sync(kFull, ob[1], cc);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int q = 2 * cc + e;
        if (q >= Gq) continue;
        const int hq = h * Gq + q;
        float* part = a.partials + ((static_cast<int64_t>(s) * Hq + hq) * a.num_splits + split) * (D + 2);
        if (r == 0) {
            part[0] = m_ref[e];
            part[1] = l_acc[e];
        }
        const float bias = e ? bias1 : bias0;
        const float z = z_acc[e];
#pragma unroll
        for (int mt = 0; mt < G::MTILES; ++mt) {
            const int d0 = r * (D / 8) + 2 * mt;
            // sum P'(code - centre) = 2^VB (o - bias) - centre * bias
            part[2 + d0] = (o[mt][e] - bias) * kValW - kCentre * bias + z;
            part[2 + d0 + 1] = (o[mt][2 + e] - bias) * kValW - kCentre * bias + z;
        }
    }
}

template <int D, int KB, int VB, bool NC>
cudaError_t launch_t(const LayerParams& p, const CacheGeom& c, const MmaArgs& a, int num_seqs, float* out,
                     cudaStream_t stream) {
    constexpr int NS = D >= 256 ? 2 : 3;
    const MmaSmem<D, KB, VB, NS> lay(c.num_kv_heads, a.num_q_heads);
    auto kern = decode_mma_kernel<D, KB, VB, NC, NS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, lay.total);
    if (e != cudaSuccess) return e;
    dim3 grid(static_cast<unsigned>(a.num_splits), static_cast<unsigned>(num_seqs));
    kern<<<grid, 32 * c.num_kv_heads, lay.total, stream>>>(p, c, a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_combine(a.partials, out, num_seqs, a.num_q_heads, D, a.num_splits, stream);
}

template <int D, int KB, int VB>
cudaError_t dispatch_nc(const LayerParams& p, const CacheGeom& c, const MmaArgs& a, int ns, float* out,
                        cudaStream_t st) {
    if (KB != 8 && p.nc) return launch_t<D, KB, VB, true>(p, c, a, ns, out, st);
    return launch_t<D, KB, VB, false>(p, c, a, ns, out, st);
}

template <int D>
cudaError_t dispatch_bits(const LayerParams& p, const CacheGeom& c, const MmaArgs& a, int ns, float* out,
                          cudaStream_t st) {
    const int kb = p.kbits, vb = p.vbits;
    if (kb == 3 && vb == 3) return dispatch_nc<D, 3, 3>(p, c, a, ns, out, st);
    if (kb == 3 && vb == 4) return dispatch_nc<D, 3, 4>(p, c, a, ns, out, st);
    if (kb == 4 && vb == 3) return dispatch_nc<D, 4, 3>(p, c, a, ns, out, st);
    if (kb == 4 && vb == 4) return dispatch_nc<D, 4, 4>(p, c, a, ns, out, st);
    if (kb == 8 && vb == 3) return dispatch_nc<D, 8, 3>(p, c, a, ns, out, st);
    if (kb == 8 && vb == 4) return dispatch_nc<D, 8, 4>(p, c, a, ns, out, st);
    return cudaErrorInvalidValue;
}

// Round to the nearest fp16 value (ties to even), on the host.
float round_half(float x) { return __half2float(__float2half_rn(x)); }

// A factor gamma in [1, 2) for which the centroids, in units of 1/sqrt(d)
// and multiplied by gamma, have the smallest worst-case fp16 rounding error
// (searched on a 2^16 grid once per codebook width).  Any gamma gives the
// same attention; this one makes the fp16 table values nearly exact.
float table_gamma(const LayerParams& p) {
    static float cache[9] = {0.f};
    static std::mutex mu;
    if (p.key_fp8) return 1.0f;
    std::lock_guard<std::mutex> lock(mu);
    float& g = cache[p.mse_bits];
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

}  // namespace

bool decode_mma_supported(const LayerParams& p, int num_kv_heads, int num_q_heads) {
    const int h = num_kv_heads;
    if (!(h == 1 || h == 2 || h == 4 || h == 8)) return false;
    if (num_q_heads % h != 0 || num_q_heads / h > 8) return false;
    return p.d == 64 || p.d == 128 || p.d == 256;
}

cudaError_t launch_decode_mma(const LayerParams& p, const CacheGeom& c, const uint16_t* q, int num_seqs,
                              int num_q_heads, const int32_t* block_table, int max_blocks_per_seq,
                              const int32_t* seq_lens, int max_seq_len, float sm_scale, const DecodePlan& plan,
                              float* out, void* workspace, cudaStream_t stream) {
    MmaArgs a{};
    a.q = q;
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.partials = static_cast<float*>(workspace);
    a.num_q_heads = num_q_heads;
    a.max_blocks = max_blocks_per_seq;
    a.max_seq_len = max_seq_len;
    a.chunks_per_split = plan.chunks_per_split;
    a.num_splits = plan.num_splits;
    a.qscale = sm_scale * kLog2e;
    a.lut_scale = table_gamma(p) * sqrtf(static_cast<float>(p.d));
    switch (p.d) {
        case 64: return dispatch_bits<64>(p, c, a, num_seqs, out, stream);
        case 128: return dispatch_bits<128>(p, c, a, num_seqs, out, stream);
        case 256: return dispatch_bits<256>(p, c, a, num_seqs, out, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace tq
