// Device helpers shared by the store, dequant and decode kernels.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "tq_internal.h"

namespace tq {

constexpr unsigned kFull = 0xffffffffu;

// Compile-time slot geometry ([TQC] key_packed_size / value_packed_size /
// slot_size_aligned).
template <int D, int KB, int VB>
struct Slot {
    static constexpr int kKeyIdxBytes = KB == 8 ? D : (D * KB + 7) / 8;
    static constexpr int kKeyBytes = KB == 8 ? D : kKeyIdxBytes + 2;
    static constexpr int kValCodeBytes = (D * VB + 7) / 8;
    static constexpr int kValBytes = kValCodeBytes + 4;
    static constexpr int kBytes = kKeyBytes + kValBytes;
    static constexpr int kAligned = kBytes + (kBytes & 1);
};

// Lane decomposition used by the per-vector kernels: a d-vector is split
// into LPV lane parts of EPL consecutive elements.
template <int D>
struct LaneSplit {
    static constexpr int kEPL = D < 32 ? D : 32;
    static constexpr int kLPV = D / kEPL;
    static constexpr int kVPW = 32 / kLPV;
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Loads N bf16 values (N a multiple of 8, 16-byte aligned) as fp32.
template <int N>
__device__ __forceinline__ void load_bf16(const uint16_t* __restrict__ src, float (&x)[N]) {
    static_assert(N % 8 == 0, "bf16 loads come in 16-byte units");
    const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int j = 0; j < N / 8; ++j) {
        uint4 u = __ldg(s + j);
        x[8 * j + 0] = bf16_lo(u.x);
        x[8 * j + 1] = bf16_hi(u.x);
        x[8 * j + 2] = bf16_lo(u.y);
        x[8 * j + 3] = bf16_hi(u.y);
        x[8 * j + 4] = bf16_lo(u.z);
        x[8 * j + 5] = bf16_hi(u.z);
        x[8 * j + 6] = bf16_lo(u.w);
        x[8 * j + 7] = bf16_hi(u.w);
    }
}

// In-register Walsh-Hadamard butterflies over the low log2(N) index bits
// (natural Sylvester order: stage s pairs i and i + s).
template <int N>
__device__ __forceinline__ void fwht_local(float (&x)[N]) {
#pragma unroll
    for (int s = 1; s < N; s <<= 1) {
#pragma unroll
        for (int i = 0; i < N; ++i) {
            if ((i & s) == 0) {
                const float a = x[i], b = x[i + s];
                x[i] = a + b;
                x[i + s] = a - b;
            }
        }
    }
}

// Butterflies across the LPV lanes of one vector (index bits above the
// lane-local ones); `part` is this lane's position within the vector.
template <int N, int LPV>
__device__ __forceinline__ void fwht_lanes(float (&x)[N], int part) {
#pragma unroll
    for (int m = 1; m < LPV; m <<= 1) {
        const bool upper = (part & m) != 0;
#pragma unroll
        for (int i = 0; i < N; ++i) {
            const float o = __shfl_xor_sync(kFull, x[i], m);
            x[i] = upper ? (o - x[i]) : (x[i] + o);
        }
    }
}

template <int LPV>
__device__ __forceinline__ float sum_lanes(float v) {
#pragma unroll
    for (int m = 1; m < LPV; m <<= 1) v += __shfl_xor_sync(kFull, v, m);
    return v;
}

template <int LPV>
__device__ __forceinline__ float min_lanes(float v) {
#pragma unroll
    for (int m = 1; m < LPV; m <<= 1) v = fminf(v, __shfl_xor_sync(kFull, v, m));
    return v;
}

template <int LPV>
__device__ __forceinline__ float max_lanes(float v) {
#pragma unroll
    for (int m = 1; m < LPV; m <<= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, m));
    return v;
}

// Packs N codes of B bits into an LSB-first bitstream held in 32-bit words.
template <int N, int B>
__device__ __forceinline__ void pack_codes(const uint32_t (&code)[N], uint32_t (&w)[(N * B + 31) / 32]) {
#pragma unroll
    for (int j = 0; j < (N * B + 31) / 32; ++j) w[j] = 0u;
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const int bit = i * B;
        w[bit / 32] |= code[i] << (bit % 32);
        if (bit % 32 + B > 32) w[bit / 32 + 1] |= code[i] >> (32 - bit % 32);
    }
}

// Extracts code i (B bits) of an LSB-first bitstream given as 32-bit words.
template <int B, int NW>
__device__ __forceinline__ uint32_t unpack_code(const uint32_t (&w)[NW], int i) {
    const int bit = i * B;
    uint32_t v = w[bit / 32] >> (bit % 32);
    if (bit % 32 + B > 32) v |= w[bit / 32 + 1] << (32 - bit % 32);
    return v & ((1u << B) - 1u);
}

// Reads `nbytes` (even) bytes at a 2-byte aligned shared/global address into
// little-endian 32-bit words.
template <int NW>
__device__ __forceinline__ void read_u16_words(const uint8_t* p, int nbytes, uint32_t (&w)[NW]) {
    const uint16_t* h = reinterpret_cast<const uint16_t*>(p);
#pragma unroll
    for (int j = 0; j < NW; ++j) {
        const uint32_t lo = (4 * j < nbytes) ? h[2 * j] : 0u;
        const uint32_t hi = (4 * j + 2 < nbytes) ? h[2 * j + 1] : 0u;
        w[j] = lo | (hi << 16);
    }
}

template <int NW>
__device__ __forceinline__ void write_u16_words(uint8_t* p, int nbytes, const uint32_t (&w)[NW]) {
    uint16_t* h = reinterpret_cast<uint16_t*>(p);
#pragma unroll
    for (int j = 0; j < NW; ++j) {
        if (4 * j < nbytes) h[2 * j] = static_cast<uint16_t>(w[j] & 0xffffu);
        if (4 * j + 2 < nbytes) h[2 * j + 1] = static_cast<uint16_t>(w[j] >> 16);
    }
}

__device__ __forceinline__ float e4m3_to_float(uint32_t byte) {
    const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(byte), __NV_E4M3);
    return __half2float(__half(h));
}

__device__ __forceinline__ uint16_t half_bits(float x) {
    return __half_as_ushort(__float2half_rn(x));
}

__device__ __forceinline__ float half_from_bits(uint32_t b) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(b)));
}

__device__ __forceinline__ void set_flag(uint32_t* flags, uint32_t bit) {
    if (flags != nullptr) atomicOr(flags, bit);
}

// ---- bulk copies and mbarriers (sm_90+ asynchronous copy engine) ----------------
// One-dimensional bulk copy global -> shared that signals completion on an
// mbarrier of this CTA (complete_tx of `bytes`).
__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src, uint32_t bytes, uint32_t mbar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(mbar)
        : "memory");
}
__device__ __forceinline__ void mbar_init(uint32_t mbar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(mbar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t mbar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(mbar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t mbar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(mbar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t mbar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(mbar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Waits for phase `parity` of an mbarrier, giving up after about a second.
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity) {
    if (mbar_try_wait(mbar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(mbar, parity))
        if (clock64() - t0 > (1ll << 31)) return false;
    return true;
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }
// Makes mbarrier initialisations visible to the bulk-copy engine.
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory"); }
// Shared-memory counter increment with acquire-release ordering; returns the old value.
__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t addr, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;\n" : "=r"(old) : "r"(addr), "r"(v) : "memory");
    return old;
}


}  // namespace tq
