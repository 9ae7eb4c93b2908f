// Continuation-prefill dequant: packed cache -> bf16 K and V (varlen rows).
//
// [TQC] TurboQuantConfig.mse_bits docstring: the centroids also serve the
// continuation-prefill dequant.  Keys: k_hat = vec_norm * Pi^T c~, with c~
// divided by ||c~|| under norm correction ([TQC] docstring, norm_correction);
// Pi^T = diag(s) H / sqrt(d), so the FWHT runs first and the signs after
// (a sign flip commutes with the rounding to bf16, so it is applied to the
// packed bf16 bits).
// FP8 keys decode their e4m3 bytes.  Values: scale * code + zero.
//
// Same lane decomposition as the store: a vector is LPV lane parts of
// EPL = min(d, 32) elements, part p owning the 8-element groups
// 8 (p + LPV j) + e, so that a quarter-warp writes 128 contiguous bytes of
// bf16 and reads whole bytes of codes per group.
#include "tq_device.cuh"

namespace tq {
namespace {

constexpr int kDqWarps = 8;
// Grid sizing: with MSE keys a block's warps take up to kDqIters grid-stride
// steps each, so that fewer, longer-lived blocks share the cost of the
// per-block table set-up, while the grid still spans kDqMinWaves waves of
// kDqBlocksPerSm resident blocks (256 threads at up to 64 registers).  FP8
// keys have no set-up to share and keep one step per warp.
constexpr int kDqIters = 4;
constexpr int kDqBlocksPerSm = 4;
constexpr int kDqMinWaves = 4;

// Reads NB bytes (3, 4 or 8) at a 2-byte aligned global address + byte offset
// `off` (even for NB = 4 and 8) as the low-order bytes of a 64-bit word.
template <int NB>
__device__ __forceinline__ uint64_t get_bytes(const uint8_t* p) {
    if constexpr (NB == 3) {
        return static_cast<uint64_t>(p[0]) | (static_cast<uint64_t>(p[1]) << 8) | (static_cast<uint64_t>(p[2]) << 16);
    } else {
        const uint16_t* h = reinterpret_cast<const uint16_t*>(p);
        uint64_t w = 0;
#pragma unroll
        for (int i = 0; i < NB / 2; ++i) w |= static_cast<uint64_t>(h[i]) << (16 * i);
        return w;
    }
}

// Two floats -> bf16x2 (round to nearest even; lo in the low half).
__device__ __forceinline__ uint32_t bf16_pair(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two e4m3 codes (the low 16 bits of w; byte 0 -> low half) -> bf16x2.  The
// e4m3 values are exact in f16, f32 and bf16, so no step rounds.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t w) {
    uint32_t r;
    asm("{\n .reg .b16 p, l, h;\n .reg .b32 hx;\n .reg .f32 fl, fh;\n"
        " cvt.u16.u32 p, %1;\n"
        " cvt.rn.f16x2.e4m3x2 hx, p;\n"
        " mov.b32 {l, h}, hx;\n"
        " cvt.f32.f16 fl, l;\n"
        " cvt.f32.f16 fh, h;\n"
        " cvt.rn.bf16x2.f32 %0, fh, fl;\n}\n"
        : "=r"(r)
        : "r"(w));
    return r;
}

// One (token, head) vector: this lane's EPL elements of the key and the value
// read from `slot` (global or shared memory) and written as bf16 to kdst /
// vdst (16-byte groups LPV apart) when `ok`.
//
// jx < EPL / 8 sets the order in which the lane visits its 8-element groups:
// step j reads group j ^ jx.  Lanes of different vectors then read different
// groups at the same time, which spreads the reads of neighbouring slots in
// shared memory over more banks.  Values and FP8 keys are written to the
// group they were read from.  MSE keys keep group j ^ jx in registers 8 j ..
// 8 j + 7 through the Walsh-Hadamard transform: relabelling the inputs by
// XOR with 8 jx multiplies output 8 j + e by (-1)^popcount(jx & j) and
// changes nothing else (each butterfly adds or subtracts the same two
// values, possibly in swapped order, and rounding is symmetric under
// negation), so that sign joins the random-sign mask of output group j.
template <int D, int KB, int VB>
__device__ __forceinline__ void dequant_vector(const uint8_t* slot, bool ok, uint4* kdst, uint4* vdst, int part,
                                               int jx, const float* cent, const uint32_t* sign_mask_part, bool nc,
                                               float inv_sqrt_d) {
    using S = Slot<D, KB, VB>;
    using LS = LaneSplit<D>;
    constexpr int EPL = LS::kEPL, LPV = LS::kLPV;
    constexpr int NG = EPL / 8;
    static_assert(NG == 1 || NG == 2 || NG == 4, "8-element groups per lane");
    // ---- key -----------------------------------------------------------
    if constexpr (KB == 8) {
#pragma unroll
        for (int j = 0; j < NG; ++j) {
            const int g = j ^ jx;
            const uint64_t b = get_bytes<8>(slot + 8 * (part + LPV * g));
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) w[q] = e4m3x2_to_bf16x2(static_cast<uint32_t>(b >> (16 * q)));
            if (ok) kdst[LPV * g] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    } else {
        float x[EPL];
        float ng[NG];  // sum of squares of each group; added in an XOR-invariant order
#pragma unroll
        for (int j = 0; j < NG; ++j) {
            const uint64_t b = get_bytes<KB>(slot + KB * (part + LPV * (j ^ jx)));
            ng[j] = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                x[8 * j + e] = cent[static_cast<uint32_t>(b >> (KB * e)) & ((1u << KB) - 1u)];
                ng[j] = fmaf(x[8 * j + e], x[8 * j + e], ng[j]);
            }
        }
        float nsq = ng[0];
        if constexpr (NG == 2) nsq = ng[0] + ng[1];
        if constexpr (NG == 4) nsq = (ng[0] + ng[1]) + (ng[2] + ng[3]);
        nsq = sum_lanes<LPV>(nsq);
        const float vec_norm = half_from_bits(*reinterpret_cast<const uint16_t*>(slot + S::kKeyIdxBytes));
        float f = vec_norm * inv_sqrt_d;
        if (nc) f = f / sqrtf(nsq);
        fwht_local<EPL>(x);
        fwht_lanes_fma<EPL, LPV>(x, part);
        const uint4* msk = reinterpret_cast<const uint4*>(sign_mask_part);
#pragma unroll
        for (int j = 0; j < NG; ++j) {
            const uint4 m = msk[j];
            const uint32_t flip = (__popc(jx & j) & 1) ? 0x80008000u : 0u;
            const uint32_t mw[4] = {m.x ^ flip, m.y ^ flip, m.z ^ flip, m.w ^ flip};
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) w[q] = bf16_pair(x[8 * j + 2 * q] * f, x[8 * j + 2 * q + 1] * f) ^ mw[q];
            if (ok) kdst[LPV * j] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }

    // ---- value ---------------------------------------------------------
    {
        const uint16_t* sz = reinterpret_cast<const uint16_t*>(slot + S::kKeyBytes + S::kValCodeBytes);
        const float sc = half_from_bits(sz[0]);
        const float z = half_from_bits(sz[1]);
#pragma unroll
        for (int j = 0; j < NG; ++j) {
            const int g = j ^ jx;
            const uint64_t b = get_bytes<VB>(slot + S::kKeyBytes + VB * (part + LPV * g));
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float c0 = static_cast<float>(static_cast<uint32_t>(b >> (VB * 2 * q)) & ((1u << VB) - 1u));
                const float c1 = static_cast<float>(static_cast<uint32_t>(b >> (VB * (2 * q + 1))) & ((1u << VB) - 1u));
                w[q] = bf16_pair(fmaf(sc, c0, z), fmaf(sc, c1, z));
            }
            if (ok) vdst[LPV * g] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

template <int D, int KB, int VB>
__global__ void __launch_bounds__(kDqWarps * 32)
dequant_kernel(const LayerParams p, const CacheGeom c, const int32_t* __restrict__ block_table,
               const int max_blocks, const int32_t* __restrict__ cu_seqlens, const int max_seq_len,
               uint16_t* __restrict__ k_out, uint16_t* __restrict__ v_out, const FastDiv div_h,
               const FastDiv div_bs, const int narrow) {
    using S = Slot<D, KB, VB>;
    using LS = LaneSplit<D>;
    constexpr int EPL = LS::kEPL, LPV = LS::kLPV, VPW = LS::kVPW;
    constexpr int SA = S::kAligned;
    // centroid table and, per lane part, XOR masks that apply the random
    // signs to the packed bf16 pairs of the output (word w of group j at 4 j + w)
    __shared__ float cent[16];
    __shared__ __align__(16) uint32_t sign_mask[LPV][EPL / 2];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int part = lane % LPV;
    const int vin = lane / LPV;
    const int H = c.num_kv_heads;
    const int s = blockIdx.y;
    const int64_t row0 = cu_seqlens[s];
    int n = cu_seqlens[s + 1] - cu_seqlens[s];
    const int cap = min(max_seq_len, max_blocks * c.block_size);
    if (n > cap || n < 0) {
        if (threadIdx.x == 0 && blockIdx.x == 0) set_flag(c.flags, kFlagSeq);
        n = n < 0 ? 0 : cap;
    }
    const int64_t num_vecs = static_cast<int64_t>(n) * H;
    if constexpr (KB != 8) {
        if (threadIdx.x < 16) cent[threadIdx.x] = p.centroids[threadIdx.x < p.n_centroids ? threadIdx.x : 0];
        for (int i = threadIdx.x; i < LPV * EPL / 2; i += kDqWarps * 32) {
            const int pp = i / (EPL / 2), jw = i % (EPL / 2);
            const int e = 8 * (pp + LPV * (jw / 4)) + 2 * (jw % 4);
            const uint32_t b0 = (p.sign_mask[e / 32] >> (e % 32)) & 1u;
            const uint32_t b1 = (p.sign_mask[(e + 1) / 32] >> ((e + 1) % 32)) & 1u;
            sign_mask[pp][jw] = (b0 << 15) | (b1 << 31);
        }
        __syncthreads();
    }
    const float inv_sqrt_d = 1.0f / sqrtf(static_cast<float>(D));

    const int64_t step = static_cast<int64_t>(gridDim.x) * kDqWarps * VPW;
    for (int64_t base = (static_cast<int64_t>(blockIdx.x) * kDqWarps + warp) * VPW; base < num_vecs;
         base += step) {
        const int64_t vi = base + vin;
        const bool valid = vi < num_vecs;
        // narrow: vector indices fit 32 bits (host-checked); positions always do
        const int pos = valid ? (narrow ? static_cast<int>(fast_div(static_cast<uint32_t>(vi), div_h))
                                        : static_cast<int>(vi / H))
                              : 0;
        const int h = valid ? static_cast<int>(vi - static_cast<int64_t>(pos) * H) : 0;
        const int col = static_cast<int>(fast_div(static_cast<uint32_t>(pos), div_bs));  // pos / block_size
        const int blk = valid ? block_table[static_cast<int64_t>(s) * max_blocks + col] : 0;
        const bool ok = valid && blk >= 0 && blk < c.num_blocks;
        if (valid && !ok && part == 0) set_flag(c.flags, kFlagBlock);
        const uint8_t* slot = c.data + static_cast<int64_t>(ok ? blk : 0) * c.block_stride +
                              (static_cast<int64_t>(pos - col * c.block_size) * H + h) * SA;
        uint4* kdst = reinterpret_cast<uint4*>(k_out + ((row0 + pos) * H + h) * D) + part;
        uint4* vdst = reinterpret_cast<uint4*>(v_out + ((row0 + pos) * H + h) * D) + part;

        dequant_vector<D, KB, VB>(slot, ok, kdst, vdst, part, 0, cent, sign_mask[part], p.nc != 0, inv_sqrt_d);
    }
}

// Staged variant: each warp walks whole token steps (ts consecutive
// positions of one block, ts * H * slot bytes, a multiple of 16 that starts
// 16-byte aligned) and has a 2-slot ring in shared memory.  Lane 0 copies
// the next step's rows with one bulk copy (cp.async.bulk, completing the
// slot's mbarrier) while the warp expands the current one, so the slot
// bytes come from shared memory instead of many small dependent global
// loads.  The block-table entry of a step is read when its copy is issued,
// one step ahead of its use.
template <int D, int KB, int VB>
__global__ void __launch_bounds__(kDqWarps * 32, 3)
dequant_staged_kernel(const LayerParams p, const CacheGeom c, const int32_t* __restrict__ block_table,
                      const int max_blocks, const int32_t* __restrict__ cu_seqlens, const int max_seq_len,
                      uint16_t* __restrict__ k_out, uint16_t* __restrict__ v_out, const FastDiv div_h,
                      const FastDiv div_bs, const int ts, const int step_bytes, const uint32_t order) {
    using S = Slot<D, KB, VB>;
    using LS = LaneSplit<D>;
    constexpr int EPL = LS::kEPL, LPV = LS::kLPV, VPW = LS::kVPW;
    constexpr int SA = S::kAligned;
    __shared__ float cent[16];
    __shared__ __align__(16) uint32_t sign_mask[LPV][EPL / 2];
    __shared__ __align__(8) uint64_t full[kDqWarps][2];
    extern __shared__ __align__(16) uint8_t dq_ring[];  // [warp][slot][step_bytes]
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int part = lane % LPV;
    const int vin = lane / LPV;
    // group order of this lane's vectors: j ^ jx, jx = (a vin + b (vin >> 2) + c (vin >> 3)) mod groups
    // (d < 64: one vector per lane or one group, the natural order)
    const int jx = D < 64 ? 0
                          : static_cast<int>(((order & 3u) * vin + ((order >> 2) & 3u) * (vin >> 2) +
                                              ((order >> 4) & 3u) * (vin >> 3)) % static_cast<uint32_t>(EPL / 8));
    const int H = c.num_kv_heads;
    const int s = blockIdx.y;
    const int64_t row0 = cu_seqlens[s];
    int n = cu_seqlens[s + 1] - cu_seqlens[s];
    const int cap = min(max_seq_len, max_blocks * c.block_size);
    if (n > cap || n < 0) {
        if (threadIdx.x == 0 && blockIdx.x == 0) set_flag(c.flags, kFlagSeq);
        n = n < 0 ? 0 : cap;
    }
    if constexpr (KB != 8) {
        if (threadIdx.x < 16) cent[threadIdx.x] = p.centroids[threadIdx.x < p.n_centroids ? threadIdx.x : 0];
        for (int i = threadIdx.x; i < LPV * EPL / 2; i += kDqWarps * 32) {
            const int pp = i / (EPL / 2), jw = i % (EPL / 2);
            const int e = 8 * (pp + LPV * (jw / 4)) + 2 * (jw % 4);
            const uint32_t b0 = (p.sign_mask[e / 32] >> (e % 32)) & 1u;
            const uint32_t b1 = (p.sign_mask[(e + 1) / 32] >> ((e + 1) % 32)) & 1u;
            sign_mask[pp][jw] = (b0 << 15) | (b1 << 31);
        }
    }
    if (threadIdx.x == 0) {
        for (int w = 0; w < kDqWarps; ++w) {
            mbar_init(static_cast<uint32_t>(__cvta_generic_to_shared(&full[w][0])), 1u);
            mbar_init(static_cast<uint32_t>(__cvta_generic_to_shared(&full[w][1])), 1u);
        }
        fence_mbar_init();
    }
    __syncthreads();
    const float inv_sqrt_d = 1.0f / sqrtf(static_cast<float>(D));

    uint8_t* const ring = dq_ring + static_cast<int64_t>(warp) * 2 * step_bytes;
    const uint32_t ring_sh = static_cast<uint32_t>(__cvta_generic_to_shared(ring));
    const uint32_t full_sh = static_cast<uint32_t>(__cvta_generic_to_shared(&full[warp][0]));
    const int row_bytes = H * SA;
    // lane 0: stage step kk (positions kk * ts ...) into slot sl; returns its block id (-1: none)
    auto issue = [&](int kk, int sl) -> int {
        const int pos = kk * ts;
        const int col = static_cast<int>(fast_div(static_cast<uint32_t>(pos), div_bs));
        const int b = block_table[static_cast<int64_t>(s) * max_blocks + col];
        if (b >= 0 && b < c.num_blocks) {
            const uint8_t* src = c.data + static_cast<int64_t>(b) * c.block_stride +
                                 static_cast<int64_t>(pos - col * c.block_size) * row_bytes;
            mbar_arrive_tx(full_sh + 8u * sl, static_cast<uint32_t>(step_bytes));
            bulk_copy(ring_sh + static_cast<uint32_t>(sl * step_bytes), src, static_cast<uint32_t>(step_bytes),
                      full_sh + 8u * sl);
            return b;
        }
        mbar_arrive(full_sh + 8u * sl);
        return -1;
    };
    const int steps_n = (n + ts - 1) / ts;
    const int gstride = gridDim.x * kDqWarps;
    int k = blockIdx.x * kDqWarps + warp;
    int blk_cur = -1, blk_next = -1;
    if (lane == 0 && k < steps_n) blk_cur = issue(k, 0);
    bool timed_out = false;
    int it = 0;
    for (; k < steps_n; k += gstride, ++it) {
        const int sl = it & 1;
        __syncwarp();  // every lane is done with the other slot (the previous step)
        if (lane == 0 && k + gstride < steps_n) {
            fence_proxy_async();  // that slot was read through the generic proxy
            blk_next = issue(k + gstride, sl ^ 1);
        }
        const int blk = __shfl_sync(kFull, blk_cur, 0);
        if (!mbar_wait(full_sh + 8u * sl, static_cast<uint32_t>((it >> 1) & 1))) {
            timed_out = true;
            break;
        }
        const int pos0 = k * ts;
        const uint8_t* stage = ring + sl * step_bytes;
        for (int v0 = 0; v0 < ts * H; v0 += VPW) {
            const int vl = v0 + vin;  // vector of the step: token vl / H, head vl % H
            const int tl = static_cast<int>(fast_div(static_cast<uint32_t>(vl), div_h));
            const int h = vl - tl * H;
            const int pos = pos0 + tl;
            const bool valid = vl < ts * H && pos < n;
            const bool ok = valid && blk >= 0;
            if (valid && blk < 0 && part == 0) set_flag(c.flags, kFlagBlock);
            const uint8_t* slot = stage + (valid ? vl * SA : 0);
            uint4* kdst = reinterpret_cast<uint4*>(k_out + ((row0 + pos) * H + h) * D) + part;
            uint4* vdst = reinterpret_cast<uint4*>(v_out + ((row0 + pos) * H + h) * D) + part;
            dequant_vector<D, KB, VB>(slot, ok, kdst, vdst, part, jx, cent, sign_mask[part], p.nc != 0,
                                      inv_sqrt_d);
        }
        blk_cur = blk_next;
    }
    if (timed_out && lane == 0) {
        set_flag(c.flags, kFlagWait);
        // the other slot may still be filling: wait for it (bounded) before exiting
        if (k + gstride < steps_n) mbar_wait(full_sh + 8u * ((it & 1) ^ 1), static_cast<uint32_t>(((it + 1) >> 1) & 1));
    }
}

// Shared-memory wavefronts of the staged kernel's slot reads under one group
// order (see dequant_vector): for 8 consecutive warp steps over a staged
// run of slots, each load instruction costs the largest number of distinct
// 4-byte words that one of the 32 banks has to serve.
template <int D, int KB, int VB>
long slot_read_wavefronts(uint32_t order) {
    using S = Slot<D, KB, VB>;
    using LS = LaneSplit<D>;
    constexpr int EPL = LS::kEPL, LPV = LS::kLPV, VPW = LS::kVPW, NG = EPL / 8;
    // one entry per load instruction of a lane: (field start, bytes per group, byte in the group)
    struct Load {
        int base, unit, off;
        bool per_group;
    };
    Load loads[2 * NG * 4 + 3];
    int nl = 0;
    const int kstep = KB == 8 ? 2 : (KB == 4 ? 2 : 1), kn = KB == 8 ? 4 : (KB == 4 ? 2 : 3);
    for (int i = 0; i < kn; ++i) loads[nl++] = {0, KB, i * kstep, true};
    if (KB != 8) loads[nl++] = {S::kKeyIdxBytes, 0, 0, false};
    const int vstep = VB == 4 ? 2 : 1, vn = VB == 4 ? 2 : 3;
    for (int i = 0; i < vn; ++i) loads[nl++] = {S::kKeyBytes, VB, i * vstep, true};
    loads[nl++] = {S::kKeyBytes + S::kValCodeBytes, 0, 0, false};
    loads[nl++] = {S::kKeyBytes + S::kValCodeBytes + 2, 0, 0, false};
    long total = 0;
    for (int st = 0; st < 8; ++st) {
        for (int li = 0; li < nl; ++li) {
            const Load& ld = loads[li];
            for (int j = 0; j < (ld.per_group ? NG : 1); ++j) {
                long words[32];
                int bank_n[32] = {0};
                for (int lane = 0; lane < 32; ++lane) {
                    const int vin = lane / LPV, part = lane % LPV;
                    const int jx = static_cast<int>(((order & 3u) * vin + ((order >> 2) & 3u) * (vin >> 2) +
                                                     ((order >> 4) & 3u) * (vin >> 3)) % NG);
                    const long addr = static_cast<long>(st * VPW + vin) * S::kAligned + ld.base +
                                      (ld.per_group ? ld.unit * (part + LPV * (j ^ jx)) + ld.off : 0);
                    words[lane] = addr / 4;
                    bool seen = false;
                    for (int o = 0; o < lane && !seen; ++o) seen = words[o] == words[lane];
                    if (!seen) ++bank_n[words[lane] % 32];
                }
                int most = 0;
                for (int bk = 0; bk < 32; ++bk) most = bank_n[bk] > most ? bank_n[bk] : most;
                total += most;
            }
        }
    }
    return total;
}

// The group order with the fewest wavefronts among jx = (a vin + b (vin >> 2)
// + c (vin >> 3)) mod groups, packed as a | b << 2 | c << 4 (0: the natural order).
template <int D, int KB, int VB>
uint32_t best_group_order() {
    if (D < 64) return 0u;
    // b matters only with more than 4 vectors per warp, c with more than 8
    constexpr int VPW = LaneSplit<D>::kVPW;
    const uint32_t nb = VPW > 4 ? 4u : 1u, nc = VPW > 8 ? 4u : 1u;
    uint32_t best = 0u;
    long best_w = slot_read_wavefronts<D, KB, VB>(0u);
    for (uint32_t c = 0; c < nc; ++c) {
        for (uint32_t b = 0; b < nb; ++b) {
            for (uint32_t a = 0; a < 4; ++a) {
                const uint32_t code = a | (b << 2) | (c << 4);
                if (code == 0u) continue;
                const long w = slot_read_wavefronts<D, KB, VB>(code);
                if (w < best_w) {
                    best_w = w;
                    best = code;
                }
            }
        }
    }
    return best;
}

template <int D, int KB, int VB>
cudaError_t launch(const LayerParams& p, const CacheGeom& c, const int32_t* bt, int max_blocks,
                   const int32_t* cu, int num_seqs, int max_seq_len, uint16_t* k_out, uint16_t* v_out,
                   int sm_count, cudaStream_t stream) {
    constexpr int VPW = LaneSplit<D>::kVPW;
    const FastDiv div_h = make_fast_div(static_cast<uint32_t>(c.num_kv_heads));
    const FastDiv div_bs = make_fast_div(static_cast<uint32_t>(c.block_size));
    // Staged kernel: token steps of ts rows whose bytes are a multiple of 16
    // (ts = 16 / gcd(row, 16)) inside one block, a 16-byte aligned cache and
    // block stride, and a ring that fits the shared memory.
    {
        const int64_t row = static_cast<int64_t>(c.num_kv_heads) * Slot<D, KB, VB>::kAligned;
        int64_t g = row, m = 16;
        while (m != 0) {
            const int64_t r = g % m;
            g = m;
            m = r;
        }
        const int ts = static_cast<int>(16 / g);
        const int64_t step_bytes = ts * row;
        const size_t ring = static_cast<size_t>(kDqWarps) * 2 * static_cast<size_t>(step_bytes);
        if (c.block_size % ts == 0 && c.block_stride % 16 == 0 && reinterpret_cast<uintptr_t>(c.data) % 16 == 0 &&
            ring <= 160 * 1024) {
            auto fn = dequant_staged_kernel<D, KB, VB>;
            cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(ring));
            if (e != cudaSuccess) return e;
            // about two waves of 4 CTAs per SM over all sequences, at most one
            // step per warp per CTA column
            const int64_t steps = (static_cast<int64_t>(max_seq_len) + ts - 1) / ts;
            const int64_t target = static_cast<int64_t>(sm_count > 0 ? sm_count : 1) * 8;
            int64_t gx = (target + num_seqs - 1) / (num_seqs > 0 ? num_seqs : 1);
            const int64_t most = (steps + kDqWarps - 1) / kDqWarps;
            if (gx > most) gx = most;
            if (gx > 65535) gx = 65535;
            if (gx < 1) gx = 1;
            dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(num_seqs));
            static const uint32_t order = best_group_order<D, KB, VB>();
            fn<<<grid, kDqWarps * 32, ring, stream>>>(p, c, bt, max_blocks, cu, max_seq_len, k_out, v_out, div_h,
                                                      div_bs, ts, static_cast<int>(step_bytes), order);
            return cudaGetLastError();
        }
    }
    const int64_t vecs = static_cast<int64_t>(max_seq_len) * c.num_kv_heads;
    int64_t gx = (vecs + VPW * kDqWarps - 1) / (VPW * kDqWarps);
    const int64_t wave_blocks = static_cast<int64_t>(sm_count > 0 ? sm_count : 1) * kDqBlocksPerSm * kDqMinWaves;
    int64_t iters = gx * num_seqs / wave_blocks;
    constexpr int64_t kMaxIters = KB == 8 ? 1 : kDqIters;
    iters = iters < 1 ? 1 : (iters > kMaxIters ? kMaxIters : iters);
    gx = (gx + iters - 1) / iters;
    if (gx > 1024) gx = 1024;
    if (gx < 1) gx = 1;
    dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(num_seqs));
    const int narrow = vecs < (int64_t{1} << 32) ? 1 : 0;
    dequant_kernel<D, KB, VB><<<grid, kDqWarps * 32, 0, stream>>>(p, c, bt, max_blocks, cu, max_seq_len,
                                                                   k_out, v_out, div_h, div_bs, narrow);
    return cudaGetLastError();
}

template <int D>
cudaError_t dispatch_bits(const LayerParams& p, const CacheGeom& c, const int32_t* bt, int mb,
                          const int32_t* cu, int ns, int msl, uint16_t* ko, uint16_t* vo, int sms, cudaStream_t st) {
    const int kb = p.kbits, vb = p.vbits;
    if (kb == 3 && vb == 3) return launch<D, 3, 3>(p, c, bt, mb, cu, ns, msl, ko, vo, sms, st);
    if (kb == 3 && vb == 4) return launch<D, 3, 4>(p, c, bt, mb, cu, ns, msl, ko, vo, sms, st);
    if (kb == 4 && vb == 3) return launch<D, 4, 3>(p, c, bt, mb, cu, ns, msl, ko, vo, sms, st);
    if (kb == 4 && vb == 4) return launch<D, 4, 4>(p, c, bt, mb, cu, ns, msl, ko, vo, sms, st);
    if (kb == 8 && vb == 3) return launch<D, 8, 3>(p, c, bt, mb, cu, ns, msl, ko, vo, sms, st);
    if (kb == 8 && vb == 4) return launch<D, 8, 4>(p, c, bt, mb, cu, ns, msl, ko, vo, sms, st);
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_dequant(const LayerParams& p, const CacheGeom& c, const int32_t* block_table,
                           int max_blocks_per_seq, const int32_t* cu_seqlens, int num_seqs, int max_seq_len,
                           uint16_t* k_out, uint16_t* v_out, int sm_count, cudaStream_t stream) {
    switch (p.d) {
        case 16: return dispatch_bits<16>(p, c, block_table, max_blocks_per_seq, cu_seqlens, num_seqs, max_seq_len, k_out, v_out, sm_count, stream);
        case 32: return dispatch_bits<32>(p, c, block_table, max_blocks_per_seq, cu_seqlens, num_seqs, max_seq_len, k_out, v_out, sm_count, stream);
        case 64: return dispatch_bits<64>(p, c, block_table, max_blocks_per_seq, cu_seqlens, num_seqs, max_seq_len, k_out, v_out, sm_count, stream);
        case 128: return dispatch_bits<128>(p, c, block_table, max_blocks_per_seq, cu_seqlens, num_seqs, max_seq_len, k_out, v_out, sm_count, stream);
        case 256: return dispatch_bits<256>(p, c, block_table, max_blocks_per_seq, cu_seqlens, num_seqs, max_seq_len, k_out, v_out, sm_count, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace tq
