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

// Key index by table lookup.  A monotone map of the unit-vector coordinate
// y in [-1, 1] onto 256 buckets, g(y) = RN(127 y + 128 + 1.5 * 2^23) & 0xFF
// (one fma; the 1.5 * 2^23 puts the rounded integer in the low mantissa
// bits), is applied to the boundaries and to every coordinate alike.
// Because g is non-decreasing, a boundary whose bucket is below g(y) lies
// below y, and one whose bucket is above lies above; so with at most one
// boundary per bucket (the Lloyd-Max boundaries are at least 0.25 sigma
// apart, two or more buckets at d <= 256) the count of boundaries strictly
// below y is base[g(y)] + (y > thr[g(y)]), where base[b] counts the
// boundaries in buckets below b and thr[b] is the boundary in bucket b
// (+inf if none).  The table is built on the device from the fp32
// boundaries with the same fma, so both sides round alike.
//
// An entry is one 32-bit word: the threshold's fp32 bits with base in the
// low 4 mantissa bits.  Compared as a float, that word differs from the
// threshold by at most 15 ulp (3.6e-6 relative; a tiny subnormal for the
// boundary at 0; a NaN, which compares false like +inf, for no boundary),
// so a key index can change only for coordinates that close to a
// boundary, inside the near-boundary window where the stored index is not
// pinned to the oracle's.  One word per lookup keeps the table at 1 KB and
// its reads at one 4-byte load.
constexpr int kBuckets = 256;
constexpr float kBucketScale = 127.f;
constexpr float kBucketMagic = 12583040.f;  // 128 + 1.5 * 2^23

__device__ __forceinline__ uint32_t bucket_of(float y) {
    return __float_as_uint(__fmaf_rn(y, kBucketScale, kBucketMagic)) & (kBuckets - 1);
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

// Packs 8 codes of B bits LSB-first (B <= 4: one 32-bit word).
template <int B>
__device__ __forceinline__ uint64_t pack8(const uint32_t* code) {
    if constexpr (B <= 4) {
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            lo |= code[e] << (B * e);
            hi |= code[4 + e] << (B * e);
        }
        return static_cast<uint64_t>(lo | (hi << (4 * B)));
    } else {
        uint64_t w = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) w |= static_cast<uint64_t>(code[e]) << (B * e);
        return w;
    }
}

// Token map of a ring append ([ART] hnwysp.cn article, "full_tq
// zero-allocation mode", item 3: new tokens wait in an exact bf16 ring and a
// ring block is compressed once it is whole).  Sequence s packs the
// positions [R floor(L/R), R floor((L + N)/R)) (L = seq_lens[s] tokens before
// the call, N new ones); token t of the append list is position
// R floor(L/R) + t - off[s] of the sequence with off[s] <= t < off[s + 1],
// read from ring row p mod R (p < L) or from new row cu_new[s] + p - L.
//
// Step mode (one new token per sequence, row s of k / v): the list is the
// fixed space of num_seqs x R ring rows.  Row i of sequence s is packed
// when the new token completes its ring block ((L + 1) mod R = 0; row R - 1
// is the new token itself); otherwise the new token is copied into ring row
// L mod R.  A warp whose rows have neither job skips them.
struct RingMap {
    const int64_t* off;  // [num_seqs + 1]: exclusive scan of the packed counts (list mode)
    const int32_t* seq_lens;
    const int32_t* cu_new;
    const int32_t* block_table;
    const uint16_t* ring_k;
    const uint16_t* ring_v;
    uint16_t* ring_k_w;  // step mode: the ring rows new tokens are copied into
    uint16_t* ring_v_w;
    int num_seqs;
    int ring_tokens;
    int max_blocks;
    int cap;    // tokens the block table can hold
    int step;   // 1: step mode
    int parts;  // step mode: CTAs sharing one sequence's ring block
};

// Validity and packed-token count of a sequence's append: L + N must fit the
// block table (cap tokens) and the new rows the input; otherwise the
// sequence takes no tokens.
__device__ __forceinline__ bool ring_seq_ok(int L, int a, int b, int64_t num_tokens, int cap) {
    return L >= 0 && a >= 0 && b >= a && b <= num_tokens && static_cast<int64_t>(L) + (b - a) <= cap;
}

template <int D, int KB, int VB, bool RING>
__global__ void __launch_bounds__(kStoreWarps * 32)
store_kernel(const LayerParams p, const CacheGeom c, const uint16_t* __restrict__ k,
             const uint16_t* __restrict__ v, int64_t num_tokens,
             const int64_t* __restrict__ slot_mapping, const RingMap rm, const FastDiv div_h,
             const FastDiv div_bs, const int narrow, const int row_unit) {
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
    // A ring append's tokens come from two places; they are read directly.
    constexpr bool kPrefetch = KB != 8 && !RING;

    // Element layout: lane part p of a vector owns elements 8 (p + LPV j) + e
    // (j < EPL / 8, e < 8) as x[8 j + e].  The Walsh-Hadamard transform
    // factors over the index bits, so the in-register stages cover bits
    // 0-2 and the bits above the lane bits, and the shuffle stages the lane
    // bits.  Each 8-element group is 16 contiguous bf16 bytes (the 8 lanes of
    // a quarter-warp read 128 contiguous bytes) and packs to whole bytes.
    // (rows padded to 16 bytes, so that every warp's stage is 16-byte aligned)
    __shared__ __align__(16) uint8_t stage_all[kStoreWarps][(VPW * SA + 2 + 15) / 16 * 16];
    // per lane part: XOR masks that flip the sign bits of the bf16 pairs the
    // random signs negate, word w of group j at [4 j + w]
    __shared__ __align__(16) uint32_t sign_mask[LPV][EPL / 2];
    // K and V rows of the warp's next step, prefetched by bulk copies
    extern __shared__ __align__(16) uint8_t kv_ring[];  // [warp][slot][K | V][kSpan] bf16
    __shared__ __align__(8) uint64_t kv_full[kStoreWarps][2];
    // key-index buckets: {threshold bits, boundaries below the bucket}
    __shared__ uint32_t bucket_tab[KB == 8 ? 1 : kBuckets];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    uint8_t* stage = stage_all[warp];
    const int part = lane % LPV;
    const int vin = lane / LPV;
    const int H = c.num_kv_heads;
    if constexpr (RING) {
        if (!rm.step) {
            const int64_t listed = rm.off[rm.num_seqs];  // num_tokens: the host's bound
            num_tokens = listed < num_tokens ? listed : num_tokens;
        }
    }
    const int64_t num_vecs = num_tokens * H;

    // Sign masks and the bucket table of the decision boundaries.
    if constexpr (KB != 8) {
        for (int bk = threadIdx.x; bk < kBuckets; bk += kStoreWarps * 32) {
            uint32_t thr = 0x7F800000u, below = 0;  // +inf: no boundary in this bucket
#pragma unroll
            for (int j = 0; j < 2 * kHalf - 1; ++j) {
                const uint32_t bj = bucket_of(p.boundaries[j]);
                below += bj < static_cast<uint32_t>(bk) ? 1u : 0u;
                if (bj == static_cast<uint32_t>(bk)) thr = __float_as_uint(p.boundaries[j]);
            }
            bucket_tab[bk] = (thr & ~0xFu) | below;
        }
        for (int i = threadIdx.x; i < LPV * EPL / 2; i += kStoreWarps * 32) {
            const int pp = i / (EPL / 2), jw = i % (EPL / 2);
            const int e = 8 * (pp + LPV * (jw / 4)) + 2 * (jw % 4);
            const uint32_t b0 = (p.sign_mask[e / 32] >> (e % 32)) & 1u;
            const uint32_t b1 = (p.sign_mask[(e + 1) / 32] >> ((e + 1) % 32)) & 1u;
            sign_mask[pp][jw] = (b0 << 15) | (b1 << 31);
        }
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

    // ---- one warp step: the VPW vectors from `base` (staged in slot sl) --------
    auto warp_step = [&](const int64_t base, const int sl) {
        const int64_t vi = base + vin;
        const bool valid = vi < num_vecs;
        const int64_t vsafe = valid ? vi : num_vecs - 1;
        uint8_t* my_slot = stage + vin * SA;
        // the vector's K and V rows and its cache slot (-1: none)
        const uint16_t* krow = k + vsafe * D;
        const uint16_t* vrow = v + vsafe * D;
        int64_t slot_id = -1;
        int64_t copy_row = -1;  // step mode: ring row the new token goes to
        bool skip = false;      // step mode: neither job for this vector
        if constexpr (RING) {
          if (rm.step) {
            const int64_t t = vsafe / H;
            const int h = static_cast<int>(vsafe - t * H);
            const int R = rm.ring_tokens;
            const int s_ = static_cast<int>(t / R);
            const int i = static_cast<int>(t - static_cast<int64_t>(s_) * R);
            const int L = rm.seq_lens[s_];
            const bool ok = L >= 0 && L < rm.cap;
            if (L >= rm.cap && valid && part == 0 && i == 0 && h == 0) set_flag(c.flags, kFlagSeq);
            const int64_t new_row = static_cast<int64_t>(s_) * H + h;
            if (ok && (L + 1) % R == 0) {
                const int pos = L + 1 - R + i;
                const int64_t r = (static_cast<int64_t>(s_) * R + i) * H + h;
                krow = i < R - 1 ? rm.ring_k + r * D : k + new_row * D;
                vrow = i < R - 1 ? rm.ring_v + r * D : v + new_row * D;
                const int b = rm.block_table[static_cast<int64_t>(s_) * rm.max_blocks + pos / c.block_size];
                if (b >= 0 && b < c.num_blocks) slot_id = static_cast<int64_t>(b) * c.block_size + pos % c.block_size;
                else if (valid && part == 0) set_flag(c.flags, kFlagBlock);
            } else if (ok && i == L % R) {
                krow = k + new_row * D;
                vrow = v + new_row * D;
                copy_row = (static_cast<int64_t>(s_) * R + i) * H + h;
            } else {
                skip = true;
            }
            skip = skip || !valid;
          } else {
            const int64_t t = vsafe / H;
            const int h = static_cast<int>(vsafe - t * H);
            int lo = 0, hi = rm.num_seqs;  // off[lo] <= t < off[hi]
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (rm.off[mid] <= t) lo = mid;
                else hi = mid;
            }
            const int s_ = lo;
            const int L = rm.seq_lens[s_];
            const int R = rm.ring_tokens;
            const int pos = (L / R) * R + static_cast<int>(t - rm.off[s_]);
            if (pos < L) {
                const int64_t r = (static_cast<int64_t>(s_) * R + pos % R) * H + h;
                krow = rm.ring_k + r * D;
                vrow = rm.ring_v + r * D;
            } else {
                const int64_t r = (static_cast<int64_t>(rm.cu_new[s_]) + (pos - L)) * H + h;
                krow = k + r * D;
                vrow = v + r * D;
            }
            const int b = rm.block_table[static_cast<int64_t>(s_) * rm.max_blocks + pos / c.block_size];
            if (b >= 0 && b < c.num_blocks) slot_id = static_cast<int64_t>(b) * c.block_size + pos % c.block_size;
            else if (valid && part == 0 && h == 0) set_flag(c.flags, kFlagBlock);
          }
        } else {
            if (valid) {
                // narrow: every vector index fits 32 bits (host-checked)
                const int64_t t = narrow ? static_cast<int64_t>(fast_div(static_cast<uint32_t>(vsafe), div_h))
                                         : vsafe / H;
                slot_id = slot_mapping[t];
            }
        }
        // this lane's groups: 16 bytes at element 8 (part + LPV j) of its vector
        const uint4* ksrc = kPrefetch ? reinterpret_cast<const uint4*>(ring + 2 * sl * kSpan + vin * D) + part
                                      : reinterpret_cast<const uint4*>(krow) + part;
        const uint4* vsrc = kPrefetch ? reinterpret_cast<const uint4*>(ring + (2 * sl + 1) * kSpan + vin * D) + part
                                      : reinterpret_cast<const uint4*>(vrow) + part;
        // 16-byte group j of K or V: shared memory (staged) or read-only global
        auto ld16 = [&](const uint4* src, int j) -> uint4 { return kPrefetch ? src[LPV * j] : __ldg(src + LPV * j); };
        if constexpr (RING) {
            if (rm.step) {
                if (copy_row >= 0 && valid) {
                    uint4* kd = reinterpret_cast<uint4*>(rm.ring_k_w + copy_row * D) + part;
                    uint4* vd = reinterpret_cast<uint4*>(rm.ring_v_w + copy_row * D) + part;
#pragma unroll
                    for (int j = 0; j < EPL / 8; ++j) {
                        kd[LPV * j] = ksrc[LPV * j];
                        vd[LPV * j] = vsrc[LPV * j];
                    }
                }
                // nothing to pack in this warp step (the copies are done)
                if (!__any_sync(kFull, !skip && copy_row < 0)) return;
            }
        }

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
                float2 x2[EPL / 2];
                const uint4* msk = reinterpret_cast<const uint4*>(sign_mask[part]);
#pragma unroll
                for (int j = 0; j < EPL / 8; ++j) {
                    const uint4 u = ld16(ksrc, j);
                    const uint4 m = msk[j];
                    const uint32_t w[4] = {u.x ^ m.x, u.y ^ m.y, u.z ^ m.z, u.w ^ m.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) x2[4 * j + q] = make_float2(bf16_lo(w[q]), bf16_hi(w[q]));
                }
                float2 ss2 = make_float2(0.f, 0.f);  // the signs do not change the squares
#pragma unroll
                for (int i = 0; i < EPL / 2; ++i) ss2 = __ffma2_rn(x2[i], x2[i], ss2);
                const float ss = sum_lanes<LPV>(ss2.x + ss2.y);
                const float n = sqrtf(ss);
                fwht_local2<EPL / 2>(x2);
                fwht_lanes2<EPL / 2, LPV>(x2, part);
                // x = sqrt(d) n y with y = Pi k / n: y = x / (n sqrt(d)), then the
                // bucket table (a zero key gives y = 0, the lower middle cell)
                const float un = n * sqrt_d;
                const float inv_u = un > 0.f ? __frcp_rn(un) : 0.f;
                const float2 inv2 = make_float2(inv_u, inv_u);
                const float2 sc2 = make_float2(kBucketScale, kBucketScale);
                const float2 mg2 = make_float2(kBucketMagic, kBucketMagic);
#pragma unroll
                for (int j = 0; j < EPL / 8; ++j) {
                    uint32_t code[8];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 y2 = __fmul2_rn(x2[4 * j + e], inv2);
                        const float2 g2 = __ffma2_rn(y2, sc2, mg2);
                        const uint32_t t0 = bucket_tab[__float_as_uint(g2.x) & (kBuckets - 1)];
                        const uint32_t t1 = bucket_tab[__float_as_uint(g2.y) & (kBuckets - 1)];
                        code[2 * e] = (t0 & 0xFu) + (y2.x > __uint_as_float(t0) ? 1u : 0u);
                        code[2 * e + 1] = (t1 & 0xFu) + (y2.y > __uint_as_float(t1) ? 1u : 0u);
                    }
                    put_bytes<KB>(my_slot + KB * (part + LPV * j), pack8<KB>(code), false);
                }
                if (part == 0)
                    *reinterpret_cast<uint16_t*>(my_slot + S::kKeyIdxBytes) = half_bits(n);
            }
        }

        // ---- value ---------------------------------------------------------
        {
            float2 x2[EPL / 2];
            // min and max on the bf16 pairs (packed min/max, the same choices
            // as on the fp32 values: NaN loses to a number, -0 below +0)
            __nv_bfloat162 mn2, mx2;
#pragma unroll
            for (int j = 0; j < EPL / 8; ++j) {
                const uint4 u = ld16(vsrc, j);
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    x2[4 * j + q] = make_float2(bf16_lo(w[q]), bf16_hi(w[q]));
                    const __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162*>(&w[q]);
                    if (j == 0 && q == 0) {
                        mn2 = b2;
                        mx2 = b2;
                    } else {
                        mn2 = __hmin2(mn2, b2);
                        mx2 = __hmax2(mx2, b2);
                    }
                }
            }
            float mn = fminf(__low2float(mn2), __high2float(mn2));
            float mx = fmaxf(__low2float(mx2), __high2float(mx2));
            mn = min_lanes<LPV>(mn);
            mx = max_lanes<LPV>(mx);
            const uint16_t sb = half_bits(__fdiv_rn(__fsub_rn(mx, mn), static_cast<float>(kTopV)));
            const uint16_t zb = half_bits(mn);
            const float s = half_from_bits(sb);
            const float z = half_from_bits(zb);
            uint32_t code[EPL];
            if (isfinite(mn) && isfinite(mx) && isfinite(z) && isfinite(s)) {
                // y = 0 for a zero scale gives quotient 0, i.e. code 0.  Two
                // elements per packed op; each keeps its own rounding: RN(v - z),
                // then the correctly rounded quotient (see quotient_rn).
                const float y = (s == 0.f) ? 0.f : __frcp_rn(s);
                const float2 y2 = make_float2(y, y), ns2 = make_float2(-s, -s), nz2 = make_float2(-z, -z);
                const float2 magic2 = make_float2(12582912.f, 12582912.f);
                if constexpr (KB == 8) {
                    // FP8 keys leave the store bound by memory, where the
                    // scalar form measured faster than the packed one
#pragma unroll
                    for (int i = 0; i < EPL; ++i) {
                        const float xi = (i & 1) ? x2[i / 2].y : x2[i / 2].x;
                        const float qv = quotient_rn(__fsub_rn(xi, z), s, y);
                        const float cl = fminf(fmaxf(qv, 0.f), static_cast<float>(kTopV));
                        code[i] = __float_as_uint(__fadd_rn(cl, 12582912.f)) & static_cast<uint32_t>(kTopV);
                    }
                } else {
#pragma unroll
                for (int i = 0; i < EPL / 2; ++i) {
                    const float2 a2 = __fadd2_rn(x2[i], nz2);
                    const float2 q0 = __fmul2_rn(a2, y2);
                    const float2 r2 = __ffma2_rn(ns2, q0, a2);
                    const float2 qv = __ffma2_rn(r2, y2, q0);
                    // clamp, then round half to even by the 1.5 * 2^23 addition
                    const float2 cl = make_float2(fminf(fmaxf(qv.x, 0.f), static_cast<float>(kTopV)),
                                                  fminf(fmaxf(qv.y, 0.f), static_cast<float>(kTopV)));
                    const float2 rr = __fadd2_rn(cl, magic2);
                    code[2 * i] = __float_as_uint(rr.x) & static_cast<uint32_t>(kTopV);
                    code[2 * i + 1] = __float_as_uint(rr.y) & static_cast<uint32_t>(kTopV);
                }
                }
            } else {
#pragma unroll
                for (int i = 0; i < EPL; ++i) {
                    const float xi = (i & 1) ? x2[i / 2].y : x2[i / 2].x;
                    const float qv = __fdiv_rn(__fsub_rn(xi, z), s);
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
            const int64_t t = narrow ? static_cast<int64_t>(fast_div(static_cast<uint32_t>(vi), div_h)) : vi / H;
            const int h = static_cast<int>(vi - t * H);
            const int64_t slot = slot_id;
            if (slot >= 0) {
                const int64_t blk = narrow && slot < (int64_t{1} << 32)
                                        ? static_cast<int64_t>(fast_div(static_cast<uint32_t>(slot), div_bs))
                                        : slot / c.block_size;
                const int64_t pos = slot - blk * c.block_size;
                if (blk < c.num_blocks)
                    dst = reinterpret_cast<uint64_t>(c.data + blk * c.block_stride + (pos * H + h) * SA);
                else
                    set_flag(c.flags, kFlagSlot);
            }
        }
        if (row_unit != 0) {
            // The warp step covers whole tokens (VPW a multiple of H): a
            // token's H slots are one contiguous row of the cache, copied in
            // row_unit-byte units (the host checked the alignment of the
            // rows, the cache and the block stride).
            const int rows = VPW / H;
            const int row_bytes = H * SA;
#pragma unroll 1
            for (int tl = 0; tl < rows; ++tl) {
                const uint64_t d = __shfl_sync(kFull, dst, tl * H * LPV);  // head 0 of token tl
                if (d == 0) continue;
                const uint8_t* src = stage + tl * row_bytes;
                if (row_unit == 16) {
                    for (int u = lane; u < row_bytes / 16; u += 32)
                        reinterpret_cast<uint4*>(d)[u] = reinterpret_cast<const uint4*>(src)[u];
                } else if (row_unit == 8) {
                    for (int u = lane; u < row_bytes / 8; u += 32)
                        reinterpret_cast<uint2*>(d)[u] = reinterpret_cast<const uint2*>(src)[u];
                } else {
                    for (int u = lane; u < row_bytes / 4; u += 32)
                        reinterpret_cast<uint32_t*>(d)[u] = reinterpret_cast<const uint32_t*>(src)[u];
                }
            }
        } else {
            constexpr int kUnits = VPW * SA / 2;
            constexpr int kPerSlot = SA / 2;
#pragma unroll 1
            for (int u = lane; u < (kUnits + 31) / 32 * 32; u += 32) {
                const int vv = min(u / kPerSlot, VPW - 1);
                const uint64_t d = __shfl_sync(kFull, dst, vv * LPV);
                if (u < kUnits && d != 0)
                    reinterpret_cast<uint16_t*>(d)[u - vv * kPerSlot] = reinterpret_cast<const uint16_t*>(stage)[u];
            }
        }
        __syncwarp();
    };

    if constexpr (RING) {
        if (rm.step) {
            // Step mode: `parts` CTAs per sequence.  They pack the ring block
            // the new token completes (R x H vectors, interleaved by warp
            // step), or the first copies the token into its ring row.
            const int R = rm.ring_tokens;
            const int parts = rm.parts;
            const int64_t per_seq = static_cast<int64_t>(R) * H;
            for (int idx = blockIdx.x; idx < rm.num_seqs * parts; idx += gridDim.x) {
                const int s_ = idx / parts, part_ = idx - s_ * parts;
                const int L = rm.seq_lens[s_];
                if (L >= rm.cap && threadIdx.x == 0 && part_ == 0) set_flag(c.flags, kFlagSeq);
                if (L < 0 || L >= rm.cap) continue;
                if ((L + 1) % R == 0) {
                    for (int64_t b0 = s_ * per_seq + (static_cast<int64_t>(part_) * kStoreWarps + warp) * VPW;
                         b0 < (s_ + 1) * per_seq; b0 += static_cast<int64_t>(parts) * kStoreWarps * VPW)
                        warp_step(b0, 0);
                } else if (part_ == 0) {
                    const int units = H * D / 8;  // 16-byte units of the token's H rows
                    const uint4* ks = reinterpret_cast<const uint4*>(k + static_cast<int64_t>(s_) * H * D);
                    const uint4* vs = reinterpret_cast<const uint4*>(v + static_cast<int64_t>(s_) * H * D);
                    const int64_t row = (static_cast<int64_t>(s_) * R + L % R) * H * D;
                    uint4* kd = reinterpret_cast<uint4*>(rm.ring_k_w + row);
                    uint4* vd = reinterpret_cast<uint4*>(rm.ring_v_w + row);
                    for (int u = threadIdx.x; u < units; u += blockDim.x) {
                        kd[u] = __ldg(ks + u);
                        vd[u] = __ldg(vs + u);
                    }
                }
            }
            return;
        }
    }

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
        warp_step(base, sl);
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
                   int64_t num_tokens, const int64_t* slot_mapping, const RingMap* rm, int sm_count,
                   cudaStream_t stream) {
    constexpr int VPW = LaneSplit<D>::kVPW;
    const int64_t vecs = num_tokens * c.num_kv_heads;
    const int64_t warps = (vecs + VPW - 1) / VPW;
    const int64_t want = (warps + kStoreWarps - 1) / kStoreWarps;
    const int64_t cap = static_cast<int64_t>(sm_count) * 8;
    const int grid = static_cast<int>(want < cap ? want : cap);
    const FastDiv div_h = make_fast_div(static_cast<uint32_t>(c.num_kv_heads));
    const FastDiv div_bs = make_fast_div(static_cast<uint32_t>(c.block_size));
    const int narrow = vecs < (int64_t{1} << 32) ? 1 : 0;
    // whole-token rows: the widest unit that the row size, the cache base and
    // the block stride allow (0: the 2-byte scatter)
    int row_unit = 0;
    if (VPW % c.num_kv_heads == 0) {
        const int64_t row = static_cast<int64_t>(c.num_kv_heads) * Slot<D, KB, VB>::kAligned;
        const uint64_t base = reinterpret_cast<uint64_t>(c.data);
        for (int u : {16, 8, 4}) {
            if (row % u == 0 && base % u == 0 && c.block_stride % u == 0) {
                row_unit = u;
                break;
            }
        }
    }
    if (rm != nullptr) {
        RingMap r = *rm;
        int g = grid;
        if (r.step) {
            // step mode: enough CTAs per sequence that a block completed by
            // few sequences still spreads over about one CTA per SM
            const int per_seq_steps = (r.ring_tokens * c.num_kv_heads + VPW - 1) / VPW;
            const int max_parts = (per_seq_steps + kStoreWarps - 1) / kStoreWarps;
            int parts = (sm_count + r.num_seqs - 1) / r.num_seqs;
            parts = parts < 1 ? 1 : (parts > max_parts ? max_parts : parts);
            r.parts = parts;
            const int64_t want_step = static_cast<int64_t>(r.num_seqs) * parts;
            g = static_cast<int>(want_step < cap ? want_step : cap);
        }
        store_kernel<D, KB, VB, true><<<g, kStoreWarps * 32, 0, stream>>>(p, c, k, v, num_tokens, nullptr, r, div_h,
                                                                          div_bs, narrow, row_unit);
        return cudaGetLastError();
    }
    const int ring_bytes = KB != 8 ? kStoreWarps * 4 * VPW * D * 2 : 0;
    auto kern = store_kernel<D, KB, VB, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, ring_bytes);
    if (e != cudaSuccess) return e;
    kern<<<grid, kStoreWarps * 32, ring_bytes, stream>>>(p, c, k, v, num_tokens, slot_mapping, RingMap{}, div_h,
                                                         div_bs, narrow, row_unit);
    return cudaGetLastError();
}

template <int D>
cudaError_t dispatch_bits(const LayerParams& p, const CacheGeom& c, const uint16_t* k, const uint16_t* v,
                          int64_t n, const int64_t* sm, const RingMap* rm, int sms, cudaStream_t st) {
    const int kb = p.kbits, vb = p.vbits;
    if (kb == 3 && vb == 3) return launch<D, 3, 3>(p, c, k, v, n, sm, rm, sms, st);
    if (kb == 3 && vb == 4) return launch<D, 3, 4>(p, c, k, v, n, sm, rm, sms, st);
    if (kb == 4 && vb == 3) return launch<D, 4, 3>(p, c, k, v, n, sm, rm, sms, st);
    if (kb == 4 && vb == 4) return launch<D, 4, 4>(p, c, k, v, n, sm, rm, sms, st);
    if (kb == 8 && vb == 3) return launch<D, 8, 3>(p, c, k, v, n, sm, rm, sms, st);
    if (kb == 8 && vb == 4) return launch<D, 8, 4>(p, c, k, v, n, sm, rm, sms, st);
    return cudaErrorInvalidValue;
}

cudaError_t dispatch_d(const LayerParams& p, const CacheGeom& c, const uint16_t* k, const uint16_t* v,
                       int64_t num_tokens, const int64_t* slot_mapping, const RingMap* rm, int sm_count,
                       cudaStream_t stream) {
    switch (p.d) {
        case 16: return dispatch_bits<16>(p, c, k, v, num_tokens, slot_mapping, rm, sm_count, stream);
        case 32: return dispatch_bits<32>(p, c, k, v, num_tokens, slot_mapping, rm, sm_count, stream);
        case 64: return dispatch_bits<64>(p, c, k, v, num_tokens, slot_mapping, rm, sm_count, stream);
        case 128: return dispatch_bits<128>(p, c, k, v, num_tokens, slot_mapping, rm, sm_count, stream);
        case 256: return dispatch_bits<256>(p, c, k, v, num_tokens, slot_mapping, rm, sm_count, stream);
        default: return cudaErrorInvalidValue;
    }
}

// ---- ring append: plan and tail copy ------------------------------------------------------
constexpr int kPlanThreads = 1024;

// One CTA: off[s] = sum over earlier sequences of the positions their
// append packs (an exclusive scan in chunks of kPlanThreads sequences).
__global__ void __launch_bounds__(kPlanThreads)
ring_plan_kernel(const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ cu_new, int num_seqs,
                 int64_t num_tokens, int R, int cap, int64_t* __restrict__ off, uint32_t* flags) {
    __shared__ int64_t warp_sum[kPlanThreads / 32];
    __shared__ int64_t carry;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    for (int c0 = 0; c0 < num_seqs; c0 += kPlanThreads) {
        const int s = c0 + threadIdx.x;
        int64_t cnt = 0;
        if (s < num_seqs) {
            const int L = seq_lens[s];
            const int a = cu_new[s], b = cu_new[s + 1];
            if (ring_seq_ok(L, a, b, num_tokens, cap)) {
                cnt = static_cast<int64_t>(R) * ((L + (b - a)) / R - L / R);
            } else if (L >= 0) {
                set_flag(flags, kFlagSeq);
            }
        }
        // inclusive scan within the warp, then across the warps
        int64_t x = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t y = __shfl_up_sync(kFull, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_sum[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int64_t w = warp_sum[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int64_t y = __shfl_up_sync(kFull, w, o);
                if (lane >= o) w += y;
            }
            warp_sum[lane] = w;  // inclusive over the warps
        }
        __syncthreads();
        const int64_t before = carry + (warp > 0 ? warp_sum[warp - 1] : 0) + (x - cnt);
        if (s < num_seqs) off[s] = before;
        __syncthreads();
        if (threadIdx.x == kPlanThreads - 1) carry = before + cnt;
        __syncthreads();
    }
    if (threadIdx.x == 0) off[num_seqs] = carry;
}

// Copies the new tokens that stay in the ring (positions from R floor((L +
// N)/R) on) into ring row p mod R; one warp per new token, 16-byte units.
__global__ void __launch_bounds__(256)
ring_tail_kernel(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v, int64_t num_tokens,
                 const int32_t* __restrict__ cu_new, int num_seqs, const int32_t* __restrict__ seq_lens, int R,
                 int cap, int row_elems, uint16_t* __restrict__ ring_k, uint16_t* __restrict__ ring_v) {
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    const int units = row_elems / 8;  // 16-byte units of one row
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); i < num_tokens;
         i += nwarps) {
        // the sequence whose new rows hold row i: cu_new[lo] <= i < cu_new[hi]
        int lo = 0, hi = num_seqs;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (cu_new[mid] <= i) lo = mid;
            else hi = mid;
        }
        const int L = seq_lens[lo];
        const int a = cu_new[lo], b = cu_new[lo + 1];
        if (!ring_seq_ok(L, a, b, num_tokens, cap) || i < a || i >= b) continue;
        const int pos = L + static_cast<int>(i - a);
        if (pos < ((L + (b - a)) / R) * R) continue;  // packed by the store
        const int64_t dst = (static_cast<int64_t>(lo) * R + pos % R) * row_elems;
        const uint4* ks = reinterpret_cast<const uint4*>(k + i * row_elems);
        const uint4* vs = reinterpret_cast<const uint4*>(v + i * row_elems);
        uint4* kd = reinterpret_cast<uint4*>(ring_k + dst);
        uint4* vd = reinterpret_cast<uint4*>(ring_v + dst);
        for (int u = lane; u < units; u += 32) {
            kd[u] = ks[u];
            vd[u] = vs[u];
        }
    }
}

}  // namespace

cudaError_t launch_store(const LayerParams& p, const CacheGeom& c, const uint16_t* k, const uint16_t* v,
                         int64_t num_tokens, const int64_t* slot_mapping, int sm_count,
                         cudaStream_t stream) {
    return dispatch_d(p, c, k, v, num_tokens, slot_mapping, nullptr, sm_count, stream);
}

cudaError_t launch_ring_step(const LayerParams& p, const CacheGeom& c, const uint16_t* k, const uint16_t* v,
                             int num_seqs, const int32_t* seq_lens, uint16_t* ring_k, uint16_t* ring_v,
                             int ring_tokens, const int32_t* block_table, int max_blocks_per_seq, int sm_count,
                             cudaStream_t stream) {
    if (num_seqs <= 0) return cudaSuccess;
    RingMap rm{nullptr, seq_lens, nullptr, block_table, ring_k, ring_v, ring_k, ring_v, num_seqs, ring_tokens,
               max_blocks_per_seq, max_blocks_per_seq * c.block_size, 1, 1};
    return dispatch_d(p, c, k, v, static_cast<int64_t>(num_seqs) * ring_tokens, nullptr, &rm, sm_count, stream);
}

size_t ring_workspace_bytes(int num_seqs) {
    return (static_cast<size_t>(num_seqs > 0 ? num_seqs : 0) + 1) * sizeof(int64_t) + 256;
}

cudaError_t launch_ring_append(const LayerParams& p, const CacheGeom& c, const uint16_t* k, const uint16_t* v,
                               int64_t num_tokens, const int32_t* cu_new, int num_seqs, const int32_t* seq_lens,
                               uint16_t* ring_k, uint16_t* ring_v, int ring_tokens, const int32_t* block_table,
                               int max_blocks_per_seq, void* workspace, int sm_count, cudaStream_t stream) {
    if (num_seqs <= 0) return cudaSuccess;
    const int cap = max_blocks_per_seq * c.block_size;
    int64_t* off = static_cast<int64_t*>(workspace);
    ring_plan_kernel<<<1, kPlanThreads, 0, stream>>>(seq_lens, cu_new, num_seqs, num_tokens, ring_tokens, cap, off,
                                                     c.flags);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // every packed position is an old ring row or a new token: at most
    // num_tokens + num_seqs (R - 1) of them
    RingMap rm{off, seq_lens, cu_new, block_table, ring_k, ring_v, ring_k, ring_v, num_seqs, ring_tokens,
               max_blocks_per_seq, cap, 0, 1};
    const int64_t bound = num_tokens + static_cast<int64_t>(num_seqs) * (ring_tokens - 1);
    e = dispatch_d(p, c, k, v, bound, nullptr, &rm, sm_count, stream);
    if (e != cudaSuccess) return e;
    if (num_tokens > 0) {
        const int64_t want = (num_tokens + 7) / 8;
        const int64_t cap_ctas = static_cast<int64_t>(sm_count > 0 ? sm_count : 1) * 8;
        const int grid = static_cast<int>(want < cap_ctas ? want : cap_ctas);
        ring_tail_kernel<<<grid, 256, 0, stream>>>(k, v, num_tokens, cu_new, num_seqs, seq_lens, ring_tokens, cap,
                                                   c.num_kv_heads * p.d, ring_k, ring_v);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace tq
