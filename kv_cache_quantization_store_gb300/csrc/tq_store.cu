// Store path: quantise new keys/values and scatter their packed slots into
// the paged cache.
//
// [TQC] TurboQuantConfig (vLLM API docs, quantization.turboquant): slot layout
// [key_packed | value_packed]; key_packed = MSE indices + fp16 vec_norm, or d
// FP8 bytes; value_packed = codes + fp16 scale + fp16 zero.  Key transform:
// random-sign Walsh-Hadamard rotation then Lloyd-Max scalar quantisation.
//
// Work decomposition: one (token, KV head) vector is split into LPV lane
// parts of EPL = min(d, 32) consecutive elements, so one warp handles
// 32 / LPV consecutive vectors per iteration (a whole token row when
// H * d = 1024).  The rotation is an in-register FWHT over the lane's EPL
// elements followed by log2(LPV) shuffle stages.  Each warp assembles its
// slots in shared memory and copies them to the cache with 2-byte stores,
// because a slot is only 2-byte aligned.
#include "tq_device.cuh"

namespace tq {
namespace {

constexpr int kStoreWarps = 8;

// Number of the positive decision thresholds t[0] < t[1] < ... below a >= 0
// (strictly), by binary search over the 3 (3-bit) or 7 (4-bit) thresholds.
template <int NT>
__device__ __forceinline__ uint32_t count_above(float a, const float (&t)[NT]) {
    static_assert(NT == 3 || NT == 7, "3 or 7 positive thresholds");
    if constexpr (NT == 3) {
        const bool p1 = a > t[1];
        const bool p2 = a > (p1 ? t[2] : t[0]);
        return (p1 ? 2u : 0u) + (p2 ? 1u : 0u);
    } else {
        const bool p1 = a > t[3];
        const bool p2 = a > (p1 ? t[5] : t[1]);
        const float tc = p1 ? (p2 ? t[6] : t[4]) : (p2 ? t[2] : t[0]);
        const bool p3 = a > tc;
        return (p1 ? 4u : 0u) + (p2 ? 2u : 0u) + (p3 ? 1u : 0u);
    }
}

// Correctly rounded fp32 quotient a / s from y = RN(1 / s): q0 = RN(a y) is
// within one ulp of a / s, the residual a - s q0 is exact in one fma, and
// RN(q0 + r y) is the correctly rounded quotient (P. Markstein, "Computation
// of elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990), for finite a and finite non-zero s.
__device__ __forceinline__ float quotient_rn(float a, float s, float y) {
    const float q0 = __fmul_rn(a, y);
    const float r = __fmaf_rn(-s, q0, a);
    return __fmaf_rn(r, y, q0);
}

// Writes the NB low-order bytes of `bits` (NB = 3, 4 or 8) at a byte address of
// shared memory; `two_aligned` says the address is even.
template <int NB>
__device__ __forceinline__ void put_bytes(uint8_t* dst, uint64_t bits, bool two_aligned) {
    if constexpr (NB == 3) {
        dst[0] = static_cast<uint8_t>(bits);
        dst[1] = static_cast<uint8_t>(bits >> 8);
        dst[2] = static_cast<uint8_t>(bits >> 16);
    } else {
        (void)two_aligned;  // 4- and 8-byte groups start on even offsets
        uint16_t* h = reinterpret_cast<uint16_t*>(dst);
#pragma unroll
        for (int i = 0; i < NB / 2; ++i) h[i] = static_cast<uint16_t>(bits >> (16 * i));
    }
}

// Packs 8 codes of B bits LSB-first.
template <int B>
__device__ __forceinline__ uint64_t pack8(const uint32_t* code) {
    uint64_t w = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) w |= static_cast<uint64_t>(code[e]) << (B * e);
    return w;
}

template <int D, int KB, int VB>
__global__ void __launch_bounds__(kStoreWarps * 32)
store_kernel(const LayerParams p, const CacheGeom c, const uint16_t* __restrict__ k,
             const uint16_t* __restrict__ v, const int64_t num_tokens,
             const int64_t* __restrict__ slot_mapping) {
    using S = Slot<D, KB, VB>;
    using LS = LaneSplit<D>;
    constexpr int EPL = LS::kEPL, LPV = LS::kLPV, VPW = LS::kVPW;
    constexpr int SA = S::kAligned;
    constexpr int kTopV = (1 << VB) - 1;
    constexpr int kHalf = KB == 8 ? 2 : (1 << KB) / 2;  // levels per sign
    constexpr int kSpan = VPW * D;                      // bf16 elements of one warp step (K or V)
    // MSE keys (arithmetic-heavy) stage the next step's K and V rows in
    // shared memory by bulk copies; FP8 keys (little arithmetic) read them
    // straight from global memory, coalesced 128 bytes per quarter-warp.
    constexpr bool kPrefetch = KB != 8;

    // Element layout: lane part p of a vector owns elements 8 (p + LPV j) + e
    // (j < EPL / 8, e < 8) as x[8 j + e].  The Walsh-Hadamard transform
    // factors over the index bits, so the in-register stages cover bits
    // 0-2 and the bits above the lane bits, and the shuffle stages the lane
    // bits.  Each 8-element group is 16 contiguous bf16 bytes (the 8 lanes of
    // a quarter-warp read 128 contiguous bytes) and packs to whole bytes.
    __shared__ __align__(16) uint8_t stage_all[kStoreWarps][VPW * SA + 2];
    // per lane part: XOR masks that flip the sign bits of the bf16 pairs the
    // random signs negate, word w of group j at [4 j + w]
    __shared__ __align__(16) uint32_t sign_mask[LPV][EPL / 2];
    // K and V rows of the warp's next step, prefetched by bulk copies
    extern __shared__ __align__(16) uint8_t kv_ring[];  // [warp][slot][K | V][kSpan] bf16
    __shared__ __align__(8) uint64_t kv_full[kStoreWarps][2];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    uint8_t* stage = stage_all[warp];
    const int part = lane % LPV;
    const int vin = lane / LPV;
    const int H = c.num_kv_heads;
    const int64_t num_vecs = num_tokens * H;

    // Sign masks, and the positive-half decision thresholds (the grid is
    // symmetric about 0 and the middle boundary is 0).
    float pos_b[kHalf - 1];
    if constexpr (KB != 8) {
        for (int i = threadIdx.x; i < LPV * EPL / 2; i += kStoreWarps * 32) {
            const int pp = i / (EPL / 2), jw = i % (EPL / 2);
            const int e = 8 * (pp + LPV * (jw / 4)) + 2 * (jw % 4);
            const uint32_t b0 = (p.sign_mask[e / 32] >> (e % 32)) & 1u;
            const uint32_t b1 = (p.sign_mask[(e + 1) / 32] >> ((e + 1) % 32)) & 1u;
            sign_mask[pp][jw] = (b0 << 15) | (b1 << 31);
        }
#pragma unroll
        for (int j = 0; j < kHalf - 1; ++j) pos_b[j] = p.boundaries[kHalf + j];
    }
    if (kPrefetch && threadIdx.x == 0) {
        for (int w = 0; w < kStoreWarps; ++w) {
            mbar_init(static_cast<uint32_t>(__cvta_generic_to_shared(&kv_full[w][0])), 1u);
            mbar_init(static_cast<uint32_t>(__cvta_generic_to_shared(&kv_full[w][1])), 1u);
        }
        fence_mbar_init();
    }
    __syncthreads();
    const float sqrt_d = sqrtf(static_cast<float>(D));

    const uint16_t* ring = reinterpret_cast<const uint16_t*>(kv_ring) + warp * 4 * kSpan;
    const uint32_t ring_sh = static_cast<uint32_t>(__cvta_generic_to_shared(ring));
    const uint32_t full_sh = static_cast<uint32_t>(__cvta_generic_to_shared(&kv_full[warp][0]));
    // lane 0: stage the K and V rows of the VPW vectors from `b` into slot sl
    auto issue = [&](int64_t b, int sl) {
        const int64_t n = num_vecs - b < VPW ? num_vecs - b : VPW;
        const uint32_t bytes = static_cast<uint32_t>(n) * D * 2;
        mbar_arrive_tx(full_sh + 8u * sl, 2u * bytes);
        bulk_copy(ring_sh + static_cast<uint32_t>(2 * sl) * kSpan * 2, k + b * D, bytes, full_sh + 8u * sl);
        bulk_copy(ring_sh + static_cast<uint32_t>(2 * sl + 1) * kSpan * 2, v + b * D, bytes, full_sh + 8u * sl);
    };

    const int64_t step = static_cast<int64_t>(gridDim.x) * kStoreWarps * VPW;
    int64_t base = (static_cast<int64_t>(blockIdx.x) * kStoreWarps + warp) * VPW;
    if (kPrefetch && lane == 0 && base < num_vecs) issue(base, 0);
    bool timed_out = false;
    int it = 0;
    for (; base < num_vecs; base += step, ++it) {
        const int sl = it & 1;
        if constexpr (kPrefetch) {
            if (lane == 0 && base + step < num_vecs) {
                fence_proxy_async();  // the other slot was read through the generic proxy
                issue(base + step, sl ^ 1);
            }
            if (!mbar_wait(full_sh + 8u * sl, static_cast<uint32_t>((it >> 1) & 1))) {
                timed_out = true;
                break;
            }
        }
        const int64_t vi = base + vin;
        const bool valid = vi < num_vecs;
        const int64_t vsafe = valid ? vi : num_vecs - 1;
        uint8_t* my_slot = stage + vin * SA;
        // this lane's groups: 16 bytes at element 8 (part + LPV j) of its vector
        const uint4* ksrc = kPrefetch ? reinterpret_cast<const uint4*>(ring + 2 * sl * kSpan + vin * D) + part
                                      : reinterpret_cast<const uint4*>(k + vsafe * D) + part;
        const uint4* vsrc = kPrefetch ? reinterpret_cast<const uint4*>(ring + (2 * sl + 1) * kSpan + vin * D) + part
                                      : reinterpret_cast<const uint4*>(v + vsafe * D) + part;
        // 16-byte group j of K or V: shared memory (staged) or read-only global
        auto ld16 = [&](const uint4* src, int j) -> uint4 { return kPrefetch ? src[LPV * j] : __ldg(src + LPV * j); };

        // ---- key -----------------------------------------------------------
        {
            float x[EPL];
            if constexpr (KB == 8) {
#pragma unroll
                for (int j = 0; j < EPL / 8; ++j) {
                    const uint4 u = ld16(ksrc, j);
                    // FP8 e4m3, round to nearest even, saturating finite
                    const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
                    uint32_t f[2];
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const uint32_t lo = __nv_cvt_float2_to_fp8x2(
                            make_float2(bf16_lo(w4[2 * q]), bf16_hi(w4[2 * q])), __NV_SATFINITE, __NV_E4M3);
                        const uint32_t hi = __nv_cvt_float2_to_fp8x2(
                            make_float2(bf16_lo(w4[2 * q + 1]), bf16_hi(w4[2 * q + 1])), __NV_SATFINITE, __NV_E4M3);
                        f[q] = (lo & 0xffffu) | (hi << 16);
                    }
                    put_bytes<8>(my_slot + 8 * (part + LPV * j), (static_cast<uint64_t>(f[1]) << 32) | f[0], true);
                }
            } else {
                // bf16 pairs with the random signs applied to the raw sign bits
                const uint4* msk = reinterpret_cast<const uint4*>(sign_mask[part]);
#pragma unroll
                for (int j = 0; j < EPL / 8; ++j) {
                    const uint4 u = ld16(ksrc, j);
                    const uint4 m = msk[j];
                    const uint32_t w[4] = {u.x ^ m.x, u.y ^ m.y, u.z ^ m.z, u.w ^ m.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        x[8 * j + 2 * q] = bf16_lo(w[q]);
                        x[8 * j + 2 * q + 1] = bf16_hi(w[q]);
                    }
                }
                float ss = 0.f;  // the signs do not change the squares
#pragma unroll
                for (int i = 0; i < EPL; ++i) ss = fmaf(x[i], x[i], ss);
                ss = sum_lanes<LPV>(ss);
                const float n = sqrtf(ss);
                fwht_local<EPL>(x);
                fwht_lanes_fma<EPL, LPV>(x, part);
                // x = sqrt(d) * n * y with y = Pi k / n; compare against the
                // boundaries scaled the same way.
                const float u = n * sqrt_d;
                float t[kHalf - 1];
#pragma unroll
                for (int j = 0; j < kHalf - 1; ++j) t[j] = pos_b[j] * u;
#pragma unroll
                for (int j = 0; j < EPL / 8; ++j) {
                    uint32_t code[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float xe = x[8 * j + e];
                        const uint32_t cnt = count_above(fabsf(xe), t);
                        code[e] = xe > 0.f ? kHalf + cnt : kHalf - 1 - cnt;
                    }
                    put_bytes<KB>(my_slot + KB * (part + LPV * j), pack8<KB>(code), false);
                }
                if (part == 0)
                    *reinterpret_cast<uint16_t*>(my_slot + S::kKeyIdxBytes) = half_bits(n);
            }
        }

        // ---- value ---------------------------------------------------------
        {
            float x[EPL];
#pragma unroll
            for (int j = 0; j < EPL / 8; ++j) {
                const uint4 u = ld16(vsrc, j);
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    x[8 * j + 2 * q] = bf16_lo(w[q]);
                    x[8 * j + 2 * q + 1] = bf16_hi(w[q]);
                }
            }
            float mn = x[0], mx = x[0];
#pragma unroll
            for (int i = 1; i < EPL; ++i) {
                mn = fminf(mn, x[i]);
                mx = fmaxf(mx, x[i]);
            }
            mn = min_lanes<LPV>(mn);
            mx = max_lanes<LPV>(mx);
            const uint16_t sb = half_bits(__fdiv_rn(__fsub_rn(mx, mn), static_cast<float>(kTopV)));
            const uint16_t zb = half_bits(mn);
            const float s = half_from_bits(sb);
            const float z = half_from_bits(zb);
            uint32_t code[EPL];
            if (isfinite(mn) && isfinite(mx) && isfinite(z) && isfinite(s)) {
                // y = 0 for a zero scale gives quotient 0, i.e. code 0
                const float y = (s == 0.f) ? 0.f : __frcp_rn(s);
#pragma unroll
                for (int i = 0; i < EPL; ++i) {
                    const float qv = quotient_rn(__fsub_rn(x[i], z), s, y);
                    // clamp, then round half to even by the 1.5 * 2^23 addition
                    const float cl = fminf(fmaxf(qv, 0.f), static_cast<float>(kTopV));
                    code[i] = __float_as_uint(__fadd_rn(cl, 12582912.f)) & static_cast<uint32_t>(kTopV);
                }
            } else {
#pragma unroll
                for (int i = 0; i < EPL; ++i) {
                    const float qv = __fdiv_rn(__fsub_rn(x[i], z), s);
                    const float r = fminf(fmaxf(rintf(qv), 0.f), static_cast<float>(kTopV));
                    code[i] = (s == 0.f) ? 0u : static_cast<uint32_t>(r);
                }
            }
#pragma unroll
            for (int j = 0; j < EPL / 8; ++j)
                put_bytes<VB>(my_slot + S::kKeyBytes + VB * (part + LPV * j), pack8<VB>(code + 8 * j), false);
            if (part == 0) {
                uint16_t* sz = reinterpret_cast<uint16_t*>(my_slot + S::kKeyBytes + S::kValCodeBytes);
                sz[0] = sb;
                sz[1] = zb;
                if constexpr (SA > S::kBytes) my_slot[S::kBytes] = 0;
            }
        }
        __syncwarp();

        // ---- scatter the warp's slots ---------------------------------------
        uint64_t dst = 0;
        if (valid && part == 0) {
            const int64_t t = vi / H;
            const int h = static_cast<int>(vi - t * H);
            const int64_t slot = slot_mapping[t];
            if (slot >= 0) {
                const int64_t blk = slot / c.block_size;
                const int64_t pos = slot - blk * c.block_size;
                if (blk < c.num_blocks)
                    dst = reinterpret_cast<uint64_t>(c.data + blk * c.block_stride + (pos * H + h) * SA);
                else
                    set_flag(c.flags, kFlagSlot);
            }
        }
        constexpr int kUnits = VPW * SA / 2;
        constexpr int kPerSlot = SA / 2;
#pragma unroll 1
        for (int u = lane; u < (kUnits + 31) / 32 * 32; u += 32) {
            const int vv = min(u / kPerSlot, VPW - 1);
            const uint64_t d = __shfl_sync(kFull, dst, vv * LPV);
            if (u < kUnits && d != 0)
                reinterpret_cast<uint16_t*>(d)[u - vv * kPerSlot] = reinterpret_cast<const uint16_t*>(stage)[u];
        }
        __syncwarp();
    }
    if (timed_out) {
        if (lane == 0) {
            set_flag(c.flags, kFlagWait);
            // the other slot may still be filling: wait for it (bounded) before exiting
            if (base + step < num_vecs) mbar_wait(full_sh + 8u * ((it & 1) ^ 1), static_cast<uint32_t>(((it + 1) >> 1) & 1));
        }
    }
}

template <int D, int KB, int VB>
cudaError_t launch(const LayerParams& p, const CacheGeom& c, const uint16_t* k, const uint16_t* v,
                   int64_t num_tokens, const int64_t* slot_mapping, int sm_count, cudaStream_t stream) {
    constexpr int VPW = LaneSplit<D>::kVPW;
    const int64_t vecs = num_tokens * c.num_kv_heads;
    const int64_t warps = (vecs + VPW - 1) / VPW;
    const int64_t want = (warps + kStoreWarps - 1) / kStoreWarps;
    const int64_t cap = static_cast<int64_t>(sm_count) * 8;
    const int grid = static_cast<int>(want < cap ? want : cap);
    const int ring_bytes = KB != 8 ? kStoreWarps * 4 * VPW * D * 2 : 0;
    auto kern = store_kernel<D, KB, VB>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, ring_bytes);
    if (e != cudaSuccess) return e;
    kern<<<grid, kStoreWarps * 32, ring_bytes, stream>>>(p, c, k, v, num_tokens, slot_mapping);
    return cudaGetLastError();
}

template <int D>
cudaError_t dispatch_bits(const LayerParams& p, const CacheGeom& c, const uint16_t* k, const uint16_t* v,
                          int64_t n, const int64_t* sm, int sms, cudaStream_t st) {
    const int kb = p.kbits, vb = p.vbits;
    if (kb == 3 && vb == 3) return launch<D, 3, 3>(p, c, k, v, n, sm, sms, st);
    if (kb == 3 && vb == 4) return launch<D, 3, 4>(p, c, k, v, n, sm, sms, st);
    if (kb == 4 && vb == 3) return launch<D, 4, 3>(p, c, k, v, n, sm, sms, st);
    if (kb == 4 && vb == 4) return launch<D, 4, 4>(p, c, k, v, n, sm, sms, st);
    if (kb == 8 && vb == 3) return launch<D, 8, 3>(p, c, k, v, n, sm, sms, st);
    if (kb == 8 && vb == 4) return launch<D, 8, 4>(p, c, k, v, n, sm, sms, st);
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_store(const LayerParams& p, const CacheGeom& c, const uint16_t* k, const uint16_t* v,
                         int64_t num_tokens, const int64_t* slot_mapping, int sm_count,
                         cudaStream_t stream) {
    switch (p.d) {
        case 16: return dispatch_bits<16>(p, c, k, v, num_tokens, slot_mapping, sm_count, stream);
        case 32: return dispatch_bits<32>(p, c, k, v, num_tokens, slot_mapping, sm_count, stream);
        case 64: return dispatch_bits<64>(p, c, k, v, num_tokens, slot_mapping, sm_count, stream);
        case 128: return dispatch_bits<128>(p, c, k, v, num_tokens, slot_mapping, sm_count, stream);
        case 256: return dispatch_bits<256>(p, c, k, v, num_tokens, slot_mapping, sm_count, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace tq
