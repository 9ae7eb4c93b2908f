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

// Butterflies across the LPV lanes of one vector as fma(+-1, x, partner):
// the same single rounding as the add or the subtract it stands for.
template <int N, int LPV>
__device__ __forceinline__ void fwht_lanes_fma(float (&x)[N], int part) {
#pragma unroll
    for (int m = 1; m < LPV; m <<= 1) {
        const float sg = (part & m) ? -1.f : 1.f;
#pragma unroll
        for (int i = 0; i < N; ++i) x[i] = fmaf(sg, x[i], __shfl_xor_sync(kFull, x[i], m));
    }
}

// The same transforms on float2 pairs (x[m] = elements 2m, 2m + 1), with
// Blackwell's packed FADD2 / FFMA2 doing two butterflies per instruction
// from the second stage on; each element is still rounded once per stage,
// so the results equal the scalar versions bit for bit.
template <int N2>
__device__ __forceinline__ void fwht_local2(float2 (&x)[N2]) {
#pragma unroll
    for (int m = 0; m < N2; ++m) {
        const float a = x[m].x, b = x[m].y;
        x[m] = make_float2(a + b, a - b);
    }
    const float2 neg1 = make_float2(-1.f, -1.f);
#pragma unroll
    for (int s = 1; s < N2; s <<= 1) {
#pragma unroll
        for (int m = 0; m < N2; ++m) {
            if ((m & s) == 0) {
                const float2 a = x[m], b = x[m + s];
                x[m] = __fadd2_rn(a, b);
                x[m + s] = __ffma2_rn(b, neg1, a);
            }
        }
    }
}

template <int N2, int LPV>
__device__ __forceinline__ void fwht_lanes2(float2 (&x)[N2], int part) {
#pragma unroll
    for (int m = 1; m < LPV; m <<= 1) {
        const float sg = (part & m) ? -1.f : 1.f;
        const float2 sg2 = make_float2(sg, sg);
#pragma unroll
        for (int i = 0; i < N2; ++i) {
            const float2 o = make_float2(__shfl_xor_sync(kFull, x[i].x, m), __shfl_xor_sync(kFull, x[i].y, m));
            x[i] = __ffma2_rn(sg2, x[i], o);
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

// Unsigned 32-bit division by an invariant divisor d >= 1 with one
// multiply-high (T. Granlund and P. Montgomery, "Division by invariant
// integers using multiplication", PLDI 1994, the round-up method):
// l = ceil(log2 d), m = floor(2^32 (2^l - d) / d) + 1, and
// n / d = (t + ((n - t) >> min(l, 1))) >> max(l - 1, 0) with t = mulhi(m, n).
struct FastDiv {
    uint32_t m, s1, s2;
};

inline FastDiv make_fast_div(uint32_t d) {
    uint32_t l = 0;
    while (l < 32 && (1ull << l) < d) ++l;
    const uint64_t m = ((1ull << 32) * ((1ull << l) - d)) / d + 1;
    return FastDiv{static_cast<uint32_t>(m), l < 1 ? l : 1u, l > 1 ? l - 1 : 0u};
}

__device__ __forceinline__ uint32_t fast_div(uint32_t n, const FastDiv& d) {
    const uint32_t t = __umulhi(d.m, n);
    return (t + ((n - t) >> d.s1)) >> d.s2;
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
// Programmatic dependent launch (sm_90+): a kernel lets the next kernel of
// its stream, launched with programmatic stream serialisation, start
// early; the dependent waits for this grid's completion (and its memory)
// before reading what it wrote.
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
// Makes mbarrier initialisations visible to the bulk-copy engine.
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory"); }
// Shared-memory counter increment with acquire-release ordering; returns the old value.
__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t addr, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;\n" : "=r"(old) : "r"(addr), "r"(v) : "memory");
    return old;
}


}  // namespace tq
