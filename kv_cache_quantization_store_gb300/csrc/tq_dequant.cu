// Continuation-prefill dequant: packed cache -> bf16 K and V (varlen rows).
//
// [TQC] TurboQuantConfig.mse_bits docstring: the centroids also serve the
// continuation-prefill dequant.  Keys: k_hat = vec_norm * Pi^T c~, with c~
// divided by ||c~|| under norm correction ([TQC] docstring, norm_correction);
// Pi^T = diag(s) H / sqrt(d), so the FWHT runs first and the signs after.
// FP8 keys decode their e4m3 bytes.  Values: scale * code + zero.
//
// Same lane decomposition as the store: a vector is LPV lane parts of
// EPL = min(d, 32) elements; each lane writes its part as 16-byte stores.
#include "tq_device.cuh"

namespace tq {
namespace {

constexpr int kDqWarps = 8;

template <int N>
__device__ __forceinline__ void store_bf16(uint16_t* dst, const float (&x)[N]) {
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int j = 0; j < N / 8; ++j) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(x[8 * j + 2 * e]));
            const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(x[8 * j + 2 * e + 1]));
            w[e] = lo | (hi << 16);
        }
        d[j] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

template <int D, int KB, int VB>
__global__ void __launch_bounds__(kDqWarps * 32)
dequant_kernel(const LayerParams p, const CacheGeom c, const int32_t* __restrict__ block_table,
               const int max_blocks, const int32_t* __restrict__ cu_seqlens, const int max_seq_len,
               uint16_t* __restrict__ k_out, uint16_t* __restrict__ v_out) {
    using S = Slot<D, KB, VB>;
    using LS = LaneSplit<D>;
    constexpr int EPL = LS::kEPL, LPV = LS::kLPV, VPW = LS::kVPW;
    constexpr int SA = S::kAligned;
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

    uint32_t signs = 0;
    if constexpr (KB != 8) {
        const int first = part * EPL;
        signs = p.sign_mask[first / 32] >> (first % 32);
    }
    const float inv_sqrt_d = 1.0f / sqrtf(static_cast<float>(D));

    const int64_t step = static_cast<int64_t>(gridDim.x) * kDqWarps * VPW;
    for (int64_t base = (static_cast<int64_t>(blockIdx.x) * kDqWarps + warp) * VPW; base < num_vecs;
         base += step) {
        const int64_t vi = base + vin;
        const bool valid = vi < num_vecs;
        const int pos = valid ? static_cast<int>(vi / H) : 0;
        const int h = valid ? static_cast<int>(vi - static_cast<int64_t>(pos) * H) : 0;
        const int blk = valid ? block_table[static_cast<int64_t>(s) * max_blocks + pos / c.block_size] : 0;
        const bool ok = valid && blk >= 0 && blk < c.num_blocks;
        if (valid && !ok && part == 0) set_flag(c.flags, kFlagBlock);
        const uint8_t* slot = c.data + static_cast<int64_t>(ok ? blk : 0) * c.block_stride +
                              (static_cast<int64_t>(pos % c.block_size) * H + h) * SA;
        const int64_t out_off = ((row0 + pos) * H + h) * D + part * EPL;

        // ---- key -----------------------------------------------------------
        float x[EPL];
        if constexpr (KB == 8) {
            uint32_t w[EPL / 4];
            read_u16_words(slot + part * EPL, EPL, w);
#pragma unroll
            for (int i = 0; i < EPL; ++i) x[i] = e4m3_to_float((w[i / 4] >> (8 * (i % 4))) & 0xffu);
        } else {
            constexpr int NW = (EPL * KB + 31) / 32;
            uint32_t w[NW];
            read_u16_words(slot + part * (EPL * KB / 8), EPL * KB / 8, w);
            float nsq = 0.f;
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                x[i] = p.centroids[unpack_code<KB, NW>(w, i)];
                nsq = fmaf(x[i], x[i], nsq);
            }
            nsq = sum_lanes<LPV>(nsq);
            const float vec_norm = half_from_bits(*reinterpret_cast<const uint16_t*>(slot + S::kKeyIdxBytes));
            float f = vec_norm * inv_sqrt_d;
            if (p.nc) f = f / sqrtf(nsq);
            fwht_local<EPL>(x);
            fwht_lanes<EPL, LPV>(x, part);
#pragma unroll
            for (int i = 0; i < EPL; ++i) x[i] = ((signs >> i) & 1u) ? -x[i] * f : x[i] * f;
        }
        if (ok) store_bf16<EPL>(k_out + out_off, x);

        // ---- value ---------------------------------------------------------
        {
            constexpr int NW = (EPL * VB + 31) / 32;
            uint32_t w[NW];
            read_u16_words(slot + S::kKeyBytes + part * (EPL * VB / 8), EPL * VB / 8, w);
            const uint16_t* sz = reinterpret_cast<const uint16_t*>(slot + S::kKeyBytes + S::kValCodeBytes);
            const float sc = half_from_bits(sz[0]);
            const float z = half_from_bits(sz[1]);
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                x[i] = fmaf(sc, static_cast<float>(unpack_code<VB, NW>(w, i)), z);
        }
        if (ok) store_bf16<EPL>(v_out + out_off, x);
    }
}

template <int D, int KB, int VB>
cudaError_t launch(const LayerParams& p, const CacheGeom& c, const int32_t* bt, int max_blocks,
                   const int32_t* cu, int num_seqs, int max_seq_len, uint16_t* k_out, uint16_t* v_out,
                   cudaStream_t stream) {
    constexpr int VPW = LaneSplit<D>::kVPW;
    const int64_t vecs = static_cast<int64_t>(max_seq_len) * c.num_kv_heads;
    int64_t gx = (vecs + VPW * kDqWarps - 1) / (VPW * kDqWarps);
    if (gx > 1024) gx = 1024;
    if (gx < 1) gx = 1;
    dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(num_seqs));
    dequant_kernel<D, KB, VB><<<grid, kDqWarps * 32, 0, stream>>>(p, c, bt, max_blocks, cu, max_seq_len,
                                                                   k_out, v_out);
    return cudaGetLastError();
}

template <int D>
cudaError_t dispatch_bits(const LayerParams& p, const CacheGeom& c, const int32_t* bt, int mb,
                          const int32_t* cu, int ns, int msl, uint16_t* ko, uint16_t* vo, cudaStream_t st) {
    const int kb = p.kbits, vb = p.vbits;
    if (kb == 3 && vb == 3) return launch<D, 3, 3>(p, c, bt, mb, cu, ns, msl, ko, vo, st);
    if (kb == 3 && vb == 4) return launch<D, 3, 4>(p, c, bt, mb, cu, ns, msl, ko, vo, st);
    if (kb == 4 && vb == 3) return launch<D, 4, 3>(p, c, bt, mb, cu, ns, msl, ko, vo, st);
    if (kb == 4 && vb == 4) return launch<D, 4, 4>(p, c, bt, mb, cu, ns, msl, ko, vo, st);
    if (kb == 8 && vb == 3) return launch<D, 8, 3>(p, c, bt, mb, cu, ns, msl, ko, vo, st);
    if (kb == 8 && vb == 4) return launch<D, 8, 4>(p, c, bt, mb, cu, ns, msl, ko, vo, st);
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_dequant(const LayerParams& p, const CacheGeom& c, const int32_t* block_table,
                           int max_blocks_per_seq, const int32_t* cu_seqlens, int num_seqs, int max_seq_len,
                           uint16_t* k_out, uint16_t* v_out, cudaStream_t stream) {
    switch (p.d) {
        case 16: return dispatch_bits<16>(p, c, block_table, max_blocks_per_seq, cu_seqlens, num_seqs, max_seq_len, k_out, v_out, stream);
        case 32: return dispatch_bits<32>(p, c, block_table, max_blocks_per_seq, cu_seqlens, num_seqs, max_seq_len, k_out, v_out, stream);
        case 64: return dispatch_bits<64>(p, c, block_table, max_blocks_per_seq, cu_seqlens, num_seqs, max_seq_len, k_out, v_out, stream);
        case 128: return dispatch_bits<128>(p, c, block_table, max_blocks_per_seq, cu_seqlens, num_seqs, max_seq_len, k_out, v_out, stream);
        case 256: return dispatch_bits<256>(p, c, block_table, max_blocks_per_seq, cu_seqlens, num_seqs, max_seq_len, k_out, v_out, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace tq
