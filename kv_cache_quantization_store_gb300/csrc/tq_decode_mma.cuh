// Fused decode attention on the packed cache with tensor-core QK and P.V
// (mma.sync m16n8k16, f16 operands, f32 accumulation).  Kernel template;
// tq_decode_mma_d{64,128,256}.cu instantiate it per head size.
//
// [ART] hnwysp.cn TurboQuant article, "Direction 1": rotate the query once
// (q' = Pi q) and score it against the compressed keys; run an online
// softmax block by block; never materialise fp16 K or V.  [TQC]
// TurboQuantConfig docstring, norm_correction: divide each score by the
// norm of its centroid vector.
//
// Work decomposition.  A CTA owns one sequence's split (a range of 16-token
// chunks) and has WPH warps per KV head (H heads, compile-time).  Each chunk
// -- 16 consecutive tokens of every head, contiguous and 16-byte aligned in a
// paged block -- is staged into shared memory by one bulk copy
// (cp.async.bulk) that completes the stage's mbarrier, through an NS-deep
// ring whose stage slots and per-thread offsets are compile-time constants.
// A warp releases a stage once its data is in registers; the last warp to
// release it refills it.  The WPH warps of a head split its dims: each
// computes a partial QK over its share, the partials are added through
// shared memory, and each computes P.V for its share of the output.
//
// Prologue: the first chunks are in flight while the query rotation runs
// in the ring's last stages (one warp per query row: shuffles and register
// butterflies), then the pair table and the query fragments are built.
//
//   QK   S[16 tok x 8 cols] = Khat[16 x d] * Q'^T[d x 8]
//        Thread (r = lane/4, c = lane%4) feeds key dims of tokens r and
//        r+8; each A register is one pair of consecutive dims, looked up
//        from a pair table of half2 centroids in shared memory (3-bit: 64
//        entries, 4-bit: 256), or converted from two FP8 bytes.  The table
//        has one copy per lane (32), or 16 copies shared by lanes l and
//        l + 16 when three CTAs share an SM (a 4-bit table of 32 KB would not
//        fit three times).  Q' is permuted to the same dim order and split into fp16 hi
//        + lo parts: with G <= 4 columns 0-3 carry the hi and 4-7 the lo
//        parts (one MMA and a shuffle), else two MMAs.  The table holds the
//        centroids times a scale chosen so that their fp16 rounding error is
//        small; together this keeps the scores near fp32 accuracy.
//   norm (norm correction) Khat*Khat (HMUL2) against a ones column, one
//        extra MMA per k-step.
//   softmax  per query column, lazily rescaled (only when the running max
//        grows by more than 2^8).
//   PV   O^T[d x 8 q] += V^T[d x 16 tok] * P'[16 tok x 8 q], P' = p * scale_t.
//        Thread r feeds value dims of tokens 2c, 2c+1, 2c+8, 2c+9 as fp16
//        subnormals code * 2^(pos - 24), masked in place from their bytes; a
//        per-dim power of two restores them at the end.  An extra M-tile whose
//        row 0 is all ones accumulates sum P', which re-centres the codes on
//        the middle of their range.  P moves into the B layout with
//        movmatrix.  The zero points enter as sum p * (zero_t + centre *
//        scale_t) in fp32.
//
// Each warp writes its dims of a partial (m, l, o) per query head; the
// merge kernel (tq_decode.cu) combines the splits by log-sum-exp and waits
// for this grid through programmatic dependent launch.  Every call writes
// every partial it reads, so the workspace needs no clearing between calls.
#pragma once

#include <atomic>
#include <cmath>
#include <type_traits>

#include "tq_device.cuh"

namespace tq {
namespace mma {

constexpr int kTok = 16;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct Args {
    const uint16_t* q;
    const int32_t* block_table;
    const int32_t* seq_lens;
    float* partials;
    int num_q_heads;
    int max_blocks;
    int max_seq_len;
    int chunks_per_split;
    int num_splits;
    int slot_stride;  // partial slots per (sequence, query head)
    int ring_tokens;  // > 0: the last L mod ring_tokens tokens are in an exact ring, not in the cache
    float qscale;     // sm_scale * log2(e)
    float lut_scale;  // table value = centroid * lut_scale (= gamma * sqrt(d))
    int tok_eo;       // token order of the chunk rows: 0 natural, 1 even tokens then odd tokens
};

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Four e4m3 codes (a 32-bit word) -> two f16x2: lo from bytes 0-1, hi from bytes 2-3.
__device__ __forceinline__ void e4m3x4_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    asm("{\n .reg .b16 l16, h16;\n mov.b32 {l16, h16}, %2;\n cvt.rn.f16x2.e4m3x2 %0, l16;\n"
        " cvt.rn.f16x2.e4m3x2 %1, h16;\n}\n"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
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

__device__ __forceinline__ void group_barrier(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(nthreads) : "memory");
}

// Shared-memory loads through generic pointers into the dynamic shared array.
__device__ __forceinline__ uint32_t ld32(const uint8_t* p) { return *reinterpret_cast<const uint32_t*>(p); }
__device__ __forceinline__ uint16_t ld16(const uint8_t* p) { return *reinterpret_cast<const uint16_t*>(p); }

// NW consecutive little-endian words starting at byte `off` of a 4-byte
// aligned shared buffer (reads one aligned word past the range; the ring
// carries padding).  Plain pointer arithmetic on the shared buffer keeps the
// loads in the shared state space.
template <int NW>
__device__ __forceinline__ void ld_words(const uint8_t* base, int off, uint32_t (&w)[NW]) {
    const uint32_t* p = reinterpret_cast<const uint32_t*>(base + (off & ~3));
    const uint32_t sh = static_cast<uint32_t>(off & 3) * 8u;
    uint32_t raw[NW + 1];
#pragma unroll
    for (int i = 0; i <= NW; ++i) raw[i] = p[i];
#pragma unroll
    for (int i = 0; i < NW; ++i) w[i] = __funnelshift_r(raw[i], raw[i + 1], sh);
}

// One code unit of U bytes (2 or 4) from shared memory, zero-extended.
template <int U>
__device__ __forceinline__ uint32_t ld_unit(const uint8_t* p) {
    if constexpr (U == 4) return *reinterpret_cast<const uint32_t*>(p);
    else return *reinterpret_cast<const uint16_t*>(p);
}

// 4-bit value codes of two tokens' units (token a in the low half, token b in
// the high half) as fp16 subnormals: the code of dim w of the unit stays in
// place inside byte w / 2, i.e. code * 2^(4 (w % 2) - 24).
__device__ __forceinline__ uint32_t value_unit_sub(uint32_t ua, uint32_t ub, int w) {
    const int b = w / 2, pos = 4 * (w % 2);
    const uint32_t win = prmt(ua, ub, b | (b << 4) | ((b + 4) << 8) | ((b + 4) << 12));
    return win & ((0xFu << pos) * 0x00010001u);
}

// Value code of local dim n for two tokens as an fp16 subnormal pair
// (token a in the low half, token b in the high half): the code's bits are
// masked in place inside a 16-bit window that starts on the byte holding the
// code's first bit, so the half is code * 2^(pos - 24) with pos = (n VB) mod 8
// (pos + VB <= 10: the field never reaches the exponent bits).
template <int VB, int NW>
__device__ __forceinline__ uint32_t value_sub(const uint32_t (&wa)[NW], const uint32_t (&wb)[NW], int n) {
    const int bit = n * VB;
    const int b0 = bit / 8, pos = bit % 8;
    const int w = b0 / 4, o = b0 % 4;
    uint32_t win;
    if (o <= 2) {
        // bytes b0, b0 + 1 of both tokens (one selector per byte, shared by its codes)
        win = prmt(wa[w], wb[w], o | ((o + 1) << 4) | ((o + 4) << 8) | ((o + 5) << 12));
    } else if (pos + VB <= 8) {
        win = prmt(wa[w], wb[w], 3 | (3 << 4) | (7 << 8) | (7 << 12));
    } else {
        const uint32_t fa = __funnelshift_r(wa[w], wa[w + 1], 24);
        const uint32_t fb = __funnelshift_r(wb[w], wb[w + 1], 24);
        win = prmt(fa, fb, 0x5410);
    }
    constexpr uint32_t kField = (1u << VB) - 1u;
    return win & ((kField << pos) * 0x00010001u);
}

// 2^(24 - pos): turns the accumulated subnormal products of local dim n back
// into code units.
template <int VB>
__device__ __forceinline__ constexpr float value_weight(int n) {
    return static_cast<float>(1u << (24 - (n * VB) % 8));
}

// Compile-time geometry of one kernel instantiation.  Shared memory:
// [pair table][score exchange x2][control][16 zero bytes][stage ring][Q' fragments].
template <int D, int KB, int VB, int H, int WPH, int NS, bool PACKQ, int LREP = 32>
struct Geo {
    using S = Slot<D, KB, VB>;
    static constexpr int SA = S::kAligned;
    static constexpr int ROW = H * SA;        // one token, all heads
    static constexpr int CHUNK = kTok * ROW;  // one stage
    static constexpr int STAGE = (CHUNK + 15) & ~15;
    static constexpr int NWARPS = H * WPH;
    static constexpr int NT = 32 * NWARPS;
    static constexpr int KSTEPS = D / 16 / WPH;  // k-steps of one warp
    static constexpr int MTILES = D / 16 / WPH;  // M-tiles of one warp
    static constexpr int KBYTES = (D / 4) * KB / 8;  // key code bytes of one thread, one token
    static constexpr int KBYTES_W = KBYTES / WPH;    // ... of which one warp reads
    static constexpr int KWORDS = (KBYTES_W + 3) / 4;
    static constexpr int VBITS_W = (D / 8 / WPH) * VB;  // value code bits of one thread, token and warp
    static constexpr int VWORDS = (VBITS_W + 31) / 32;
    // Lane layout of the code loads.  Unit layouts: lane c (keys) or r
    // (values) reads units c + 4m or r + 8m of its warp's contiguous share of
    // the slot, so that neighbouring lanes hit neighbouring banks; a unit is 4
    // bytes where every share starts 4-byte aligned, else 2.  3-bit codes keep
    // one contiguous block per lane.
    static constexpr bool KUNITS = KB != 3;
    static constexpr int KUNIT = KB == 8 ? 4 : 2;   // bytes: the 4 dims of one k-step
    static constexpr int KSH = (D / WPH) * KB / 8;  // key code bytes of a warp's share
    static constexpr bool VUNITS = VB == 4;
    static constexpr int VSH = (D / WPH) * VB / 8;  // value code bytes of a warp's share
    static constexpr int VUNIT = (SA % 4 == 0 && S::kKeyBytes % 4 == 0 && VSH % 32 == 0) ? 4 : 2;
    static constexpr int VDPU = 2 * VUNIT;          // 4-bit value dims per unit
    static constexpr int VNU = VSH / (8 * VUNIT);   // value units of one lane and token
    static constexpr int VREGS = VUNITS ? VNU : VWORDS;
    static constexpr int LUT_ENTRIES = KB == 3 ? 64 : (KB == 4 ? 256 : 0);
    static constexpr int LUT_REP = LREP;                    // copies of the table (lanes l and l + LREP share one)
    static constexpr int LUT_SHIFT = LREP == 32 ? 7 : 6;    // log2 of an entry's stride (LREP x 4 bytes)
    static constexpr int LUT_BYTES = LUT_ENTRIES * LREP * 4;  // half2 per entry and copy
    // 4-bit keys of packed-query kernels at 3 CTAs per SM (the 16-copy table):
    // key codes held as 32-bit words of two k-steps, read as 4-byte units by
    // warps whose share is 4-byte aligned
    static constexpr bool PAIR_K = KB == 4 && PACKQ && LREP == 16 && KSTEPS % 2 == 0;
    static constexpr int XCH_W = WPH > 1 ? 32 * 6 * 4 : 0;  // per warp and buffer: 32 x {4 scores, 2 norms}
    static constexpr int X_OFF = LUT_BYTES;
    // control block: full mbarrier, release counter, block id per stage; error word
    static constexpr int CTRL_OFF = X_OFF + 2 * NWARPS * XCH_W;
    static constexpr int CTRL_BYTES = (16 * NS + 16 + 15) & ~15;
    // the split's block-table entries (the first BT_MAX; later ones are read from global)
    static constexpr int BT_MAX = 512;
    static constexpr int BT_OFF = CTRL_OFF + CTRL_BYTES;
    static constexpr int ZERO_OFF = BT_OFF + 4 * BT_MAX;
    static constexpr int RING_OFF = ZERO_OFF + 16;
    static constexpr int RING = NS * STAGE + 16;
    // Q' fragments follow the ring.  PACKQ (G <= 4): per warp and k-step one
    // {b0, b1} per lane, columns 0-3 the hi parts and 4-7 the lo parts of the
    // queries (d * 16 bytes per KV head).  Otherwise per warp, k-step and
    // query row r < G, 4 lanes x {hi0, hi1, lo0, lo1} (G * d * 4 bytes per KV head).
    __host__ __device__ static int q_off(int hq) {
        const int qrot = hq * D * 4;  // the ring also holds the fp32 query rotation
        return RING_OFF + (RING > qrot ? RING : qrot);
    }
    __host__ __device__ static int q_bytes(int hq) { return PACKQ ? H * D * 16 : hq * D * 4; }
    __host__ __device__ static int smem_bytes(int hq) { return q_off(hq) + q_bytes(hq); }
};

template <int D, int KB, int VB, bool NC, int H, int WPH, int NS, int MINB, bool PACKQ>
__global__ void __launch_bounds__(32 * H * WPH, MINB)
decode_kernel(const LayerParams p, const CacheGeom c, const Args a) {
    using G = Geo<D, KB, VB, H, WPH, NS, PACKQ, (MINB >= 3 ? 16 : 32)>;
    using S = typename G::S;
    static_assert(((D / 4 / WPH) * KB) % 8 == 0 && ((D / 8 / WPH) * VB) % 8 == 0,
                  "a warp's share of the codes must start on a byte");
    constexpr int SA = G::SA;
    constexpr int ROW = G::ROW;
    constexpr int NT = G::NT;
    constexpr float kCentre = 0.5f * static_cast<float>((1 << VB) - 1);
    extern __shared__ __align__(16) uint8_t smem[];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int r = lane >> 2;
    const int cc = lane & 3;
    const int Hq = a.num_q_heads;
    const int Gq = Hq / H;
    const int h = warp / WPH;     // KV head of this warp
    const int part = warp % WPH;  // its share of the head's dims
    const int split = blockIdx.x;
    const int s = blockIdx.y;
    uint8_t* const ring = smem + G::RING_OFF;
    const uint32_t ring_sh = static_cast<uint32_t>(__cvta_generic_to_shared(ring));

    // ---- sequence range ------------------------------------------------------
    int L = a.seq_lens[s];
    if (a.ring_tokens > 0 && L > 0) L -= L % a.ring_tokens;  // packed positions: the whole ring blocks
    const int cap = min(a.max_seq_len, a.max_blocks * c.block_size);
    if (L > cap || L < 0) {
        if (threadIdx.x == 0 && split == 0) set_flag(c.flags, kFlagSeq);
        L = L < 0 ? 0 : cap;
    }
    const int n_chunks = (L + kTok - 1) / kTok;
    const int c0 = split * a.chunks_per_split;
    const int c1 = min(c0 + a.chunks_per_split, n_chunks);

    // ---- this split's block-table entries, staged once -------------------------------
    {
        const int cpb_ = c.block_size / kTok;
        const int first = c0 / cpb_;
        const int n_bt = c1 > c0 ? min((c1 - 1) / cpb_ - first + 1, G::BT_MAX) : 0;
        const int32_t* row = a.block_table + static_cast<int64_t>(s) * a.max_blocks + first;
        int* dst = reinterpret_cast<int*>(smem + G::BT_OFF);
        for (int i = threadIdx.x; i < n_bt; i += NT) dst[i] = row[i];
    }

    // ---- control block: stage mbarriers and counters ------------------------------
    if (threadIdx.x == 0) {
        uint8_t* ctl = smem + G::CTRL_OFF;
        const uint32_t ctl_sh = static_cast<uint32_t>(__cvta_generic_to_shared(ctl));
        for (int st = 0; st < NS; ++st) {
            mbar_init(ctl_sh + 8u * st, 1u);
            reinterpret_cast<uint32_t*>(ctl + 8 * NS)[st] = 0u;
            reinterpret_cast<int*>(ctl + 12 * NS)[st] = -1;
        }
        *reinterpret_cast<int*>(ctl + 16 * NS) = 0;
        fence_mbar_init();
    }

    __syncthreads();  // block ids and mbarriers ready

    // ---- chunk staging.  Chunk it (of this split) lives in stage it % NS; one
    // thread copies all of it (16 token rows of every head, contiguous in the
    // paged block) with one bulk copy that completes the stage's mbarrier.  A
    // warp releases a stage once its data is in registers; the last warp to
    // release it refills it with chunk it + NS.  No CTA-wide barrier in the loop.
    uint8_t* const ctrl = smem + G::CTRL_OFF;
    const uint32_t ctrl_sh = static_cast<uint32_t>(__cvta_generic_to_shared(ctrl));
    auto full_bar = [&](int slot) -> uint32_t { return ctrl_sh + 8u * slot; };
    auto cnt_addr = [&](int slot) -> uint32_t { return ctrl_sh + 8u * NS + 4u * slot; };
    int* const stage_blk = reinterpret_cast<int*>(ctrl + 12 * NS);  // block id of the staged chunk, -1: none
    int* const err_word = reinterpret_cast<int*>(ctrl + 16 * NS);
    const int cpb = c.block_size / kTok;  // 16-token chunks per paged block
    const int32_t* bt_row = a.block_table + static_cast<int64_t>(s) * a.max_blocks;
    const int nch = c1 - c0;
    const int col0 = c0 / cpb;
    const int* bt_sm = reinterpret_cast<const int*>(smem + G::BT_OFF);
    auto issue = [&](int it) {  // one thread
        const int slot = it % NS;
        const int cg = c0 + it;
        const int col = cg / cpb;
        int b = col - col0 < G::BT_MAX ? bt_sm[col - col0] : bt_row[col];
        b = (b >= 0 && b < c.num_blocks) ? b : -1;
        stage_blk[slot] = b;
        if (b >= 0) {
            const uint8_t* src =
                c.data + static_cast<int64_t>(b) * c.block_stride + static_cast<int64_t>(cg - col * cpb) * G::CHUNK;
            mbar_arrive_tx(full_bar(slot), G::CHUNK);
            bulk_copy(ring_sh + slot * G::STAGE, src, G::CHUNK, full_bar(slot));
        } else {
            mbar_arrive(full_bar(slot));
        }
    };
    // The query rotation borrows the ring's last nq stages as scratch; the
    // first chunks go into the others before it starts.
    const int nq = (Hq * D * 4 + G::STAGE - 1) / G::STAGE;
    const int early = NS - nq > 0 ? NS - nq : 0;
    if (threadIdx.x == 0) {
        for (int it = 0; it < early && it < nch; ++it) issue(it);
    }

    // ---- pair lookup table: centroids * lut_scale as fp16 (lane l reads copy l % LUT_REP) --
    const float ls = a.lut_scale;
    if constexpr (KB == 3 || KB == 4) {
        // entry e = codes (e & mask, e >> bits) of a dim pair, LUT_REP copies x 4 bytes;
        // one 16-byte store writes four lanes' copies
        constexpr int kBits = KB, kMask = (1 << KB) - 1;
        for (int i = threadIdx.x; i < G::LUT_ENTRIES * (G::LUT_REP / 4); i += NT) {
            const int e = i / (G::LUT_REP / 4);
            const uint32_t hv = pack_half2(p.centroids[e & kMask] * ls, p.centroids[e >> kBits] * ls);
            reinterpret_cast<uint4*>(smem)[i] = make_uint4(hv, hv, hv, hv);
        }
    }

    // 4-bit keys: a warp whose share of every token's key codes starts on a
    // 4-byte boundary reads 4-byte units (two k-steps each, lane c taking
    // units c + 4m), the others 2-byte units (one k-step, units c + 4j) that
    // it pairs into the same 32-bit form.
    const int hs = h * SA;
    constexpr bool kPairK = G::PAIR_K;
    const bool ku4 = kPairK && ROW % 4 == 0 && (hs + part * G::KSH) % 4 == 0;
    // First of the 4 consecutive key dims lane c of warp part covers at local
    // k-step jl (the lane layout of the key loads).
    auto key_dim0 = [&](int c_, int part_, int jl) -> int {
        if constexpr (G::KUNITS) {
            if (kPairK && ku4) return part_ * (D / WPH) + 8 * (c_ + 4 * (jl / 2)) + 4 * (jl % 2);
            return part_ * (D / WPH) + 4 * (c_ + 4 * jl);
        } else {
            return c_ * (D / 4) + part_ * (D / (4 * WPH)) + 4 * jl;
        }
    };

    // ---- queries: q' = Pi q (MSE keys), scaled, into B fragments ---------------
    {
        float* qs = reinterpret_cast<float*>(ring + early * G::STAGE);
        const uint16_t* qg = a.q + static_cast<int64_t>(s) * Hq * D;
        for (int i = threadIdx.x; i < Hq * D; i += NT) {
            float x = __uint_as_float(static_cast<uint32_t>(qg[i]) << 16);
            if constexpr (KB != 8) {
                const int dim = i % D;
                if ((p.sign_mask[dim >> 5] >> (dim & 31)) & 1u) x = -x;
            }
            qs[i] = x;
        }
        if constexpr (KB != 8) {
            // Walsh-Hadamard butterflies of each query row in one warp: lane
            // holds elements lane + 32 j, so the stages 1 .. 16 pair lanes
            // (shuffles) and 32 .. D/2 pair registers, in the natural stage
            // order and with the one rounding of each add or subtract.
            constexpr int E = D / 32;
            __syncthreads();
            for (int row = warp; row < Hq; row += G::NWARPS) {
                float* rw = qs + row * D;
                float x[E];
#pragma unroll
                for (int j = 0; j < E; ++j) x[j] = rw[lane + 32 * j];
#pragma unroll
                for (int st = 1; st < 32; st <<= 1) {
#pragma unroll
                    for (int j = 0; j < E; ++j) {
                        const float o = __shfl_xor_sync(kFull, x[j], st);
                        x[j] = (lane & st) ? o - x[j] : x[j] + o;
                    }
                }
#pragma unroll
                for (int st = 1; st < E; st <<= 1) {
#pragma unroll
                    for (int j = 0; j < E; ++j) {
                        if ((j & st) == 0) {
                            const float x0 = x[j], x1 = x[j + st];
                            x[j] = x0 + x1;
                            x[j + st] = x0 - x1;
                        }
                    }
                }
#pragma unroll
                for (int j = 0; j < E; ++j) rw[lane + 32 * j] = x[j];
            }
        }
        __syncthreads();
        // Scores come out in log2 units.  MSE keys: the table holds
        // c * lut_scale and Pi carries 1/sqrt(d); without NC the table scale
        // is divided out here (with NC it cancels in c / ||c||).
        float f = a.qscale;
        if constexpr (KB != 8) f *= rsqrtf(static_cast<float>(D)) * (NC ? 1.0f : 1.0f / ls);
        if constexpr (PACKQ) {
            // column r of the B operand: query r & 3 of this head, hi part for
            // r < 4 and lo part for r >= 4; zero past the G queries
            const int qi = r & 3;
            const bool real = qi < Gq;
            const float* qrow = qs + (h * Gq + (real ? qi : 0)) * D;
            uint2* dst = reinterpret_cast<uint2*>(smem + G::q_off(Hq)) + warp * G::KSTEPS * 32;
            for (int jl = 0; jl < G::KSTEPS; ++jl) {
                const int dm = key_dim0(cc, part, jl);  // b0: dims dm, dm + 1; b1: dm + 2, dm + 3
                const float x0 = qrow[dm] * f, x1 = qrow[dm + 1] * f;
                const float x2 = qrow[dm + 2] * f, x3 = qrow[dm + 3] * f;
                const uint32_t hi0 = pack_half2(x0, x1);
                const uint32_t hi1 = pack_half2(x2, x3);
                const __half2 h0 = *reinterpret_cast<const __half2*>(&hi0);
                const __half2 h1 = *reinterpret_cast<const __half2*>(&hi1);
                const uint32_t lo0 = pack_half2(x0 - __low2float(h0), x1 - __high2float(h0));
                const uint32_t lo1 = pack_half2(x2 - __low2float(h1), x3 - __high2float(h1));
                uint2 v = r < 4 ? make_uint2(hi0, hi1) : make_uint2(lo0, lo1);
                if (!real) v = make_uint2(0u, 0u);
                dst[jl * 32 + lane] = v;
            }
        } else {
            const float* qrow = qs + (h * Gq + r) * D;
            // fragments of this warp: [k-step][query row r < G][lane c]
            uint4* dst = reinterpret_cast<uint4*>(smem + G::q_off(Hq)) + warp * G::KSTEPS * Gq * 4;
            for (int jl = 0; jl < G::KSTEPS && r < Gq; ++jl) {
                const int dm = key_dim0(cc, part, jl);  // b0: dims dm, dm + 1; b1: dm + 2, dm + 3
                const float x0 = qrow[dm] * f, x1 = qrow[dm + 1] * f;
                const float x2 = qrow[dm + 2] * f, x3 = qrow[dm + 3] * f;
                const uint32_t hi0 = pack_half2(x0, x1);
                const uint32_t hi1 = pack_half2(x2, x3);
                const __half2 h0 = *reinterpret_cast<const __half2*>(&hi0);
                const __half2 h1 = *reinterpret_cast<const __half2*>(&hi1);
                const uint32_t lo0 = pack_half2(x0 - __low2float(h0), x1 - __high2float(h0));
                const uint32_t lo1 = pack_half2(x2 - __low2float(h1), x3 - __high2float(h1));
                dst[(jl * Gq + r) * 4 + cc] = make_uint4(hi0, hi1, lo0, lo1);
            }
        }
        if (threadIdx.x == 0) *reinterpret_cast<uint4*>(smem + G::ZERO_OFF) = make_uint4(0u, 0u, 0u, 0u);
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        fence_proxy_async();  // the borrowed stages held the rotation (generic proxy writes)
        for (int it = early; it < NS && it < nch; ++it) issue(it);
    }
    // lanes of padded query rows (r >= G) read the zero block at every k-step
    const bool q_real = r < Gq;
    const uint4* qfrag = q_real ? reinterpret_cast<const uint4*>(smem + G::q_off(Hq)) + warp * G::KSTEPS * Gq * 4 +
                                      r * 4 + cc
                                : reinterpret_cast<const uint4*>(smem + G::ZERO_OFF);
    const int qstride = q_real ? Gq * 4 : 0;
    const uint2* qfrag2 = reinterpret_cast<const uint2*>(smem + G::q_off(Hq)) + warp * G::KSTEPS * 32 + lane;

    // every CTA of the grid is resident: the merge kernel may be scheduled
    grid_launch_dependents();

    // ---- per-thread constant offsets inside a stage.  Row k of the MMA tiles
    // holds token sig(k) of the chunk; the order is chosen on the host to
    // spread each warp's loads over the shared-memory banks. -------------------
    auto sig = [&](int k) -> int { return a.tok_eo ? (k < 8 ? 2 * k : 2 * (k - 8) + 1) : k; };
    const int tq0 = sig(r), tq1 = sig(r + 8);  // QK rows r, r + 8
    const int kbase = G::KUNITS ? hs + part * G::KSH + (ku4 ? 4 : G::KUNIT) * cc
                                : hs + cc * G::KBYTES + part * G::KBYTES_W;
    const int k_off0 = tq0 * ROW + kbase, k_off1 = tq1 * ROW + kbase;
    const int n_off0 = tq0 * ROW + hs + S::kKeyIdxBytes, n_off1 = tq1 * ROW + hs + S::kKeyIdxBytes;
    const int z_off0 = tq0 * ROW + hs + S::kKeyBytes + S::kValCodeBytes;
    const int z_off1 = tq1 * ROW + hs + S::kKeyBytes + S::kValCodeBytes;
    const int vbase = G::VUNITS ? hs + S::kKeyBytes + part * G::VSH + G::VUNIT * r
                                : hs + S::kKeyBytes + (r * (D / 8) * VB + part * G::VBITS_W) / 8;
    // P.V k-columns 2c, 2c + 1, 2c + 8, 2c + 9
    const int v_off0 = sig(2 * cc) * ROW + vbase, v_off1 = sig(2 * cc + 1) * ROW + vbase;
    const int v_off8 = sig(2 * cc + 8) * ROW + vbase, v_off9 = sig(2 * cc + 9) * ROW + vbase;
    const uint8_t* lut = smem;
    const uint32_t lane4 = static_cast<uint32_t>(lane & (G::LUT_REP - 1)) << 2;
    float* xch = reinterpret_cast<float*>(smem + G::X_OFF);  // [buffer][warp][32 float4 | 32 float2]

    // ---- QK of one staged chunk: log2-domain scores of tokens r, r + 8 for
    // query columns 2c, 2c + 1, -inf past the sequence end ---------------------------
    auto qk = [&](const uint8_t* stage, int tok0, bool ok, int buf, float (&sc)[4]) {
        float qacc[2][4];  // hi and lo query parts (PACKQ: even and odd k-steps)
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e) qacc[i][e] = 0.f;
        float nacc[4] = {0.f, 0.f, 0.f, 0.f};
        constexpr int KREGS = kPairK ? G::KSTEPS / 2 : (G::KUNITS ? G::KSTEPS : G::KWORDS);
        uint32_t kw0[KREGS], kw1[KREGS];
        if constexpr (kPairK) {
            // word m: k-step 2m in the low half, 2m + 1 in the high half
            if (ku4) {
#pragma unroll
                for (int m = 0; m < KREGS; ++m) {
                    kw0[m] = ld32(stage + k_off0 + 16 * m);
                    kw1[m] = ld32(stage + k_off1 + 16 * m);
                }
            } else {
#pragma unroll
                for (int m = 0; m < KREGS; ++m) {
                    kw0[m] = prmt(ld_unit<2>(stage + k_off0 + 16 * m), ld_unit<2>(stage + k_off0 + 16 * m + 8), 0x5410u);
                    kw1[m] = prmt(ld_unit<2>(stage + k_off1 + 16 * m), ld_unit<2>(stage + k_off1 + 16 * m + 8), 0x5410u);
                }
            }
        } else if constexpr (G::KUNITS) {
#pragma unroll
            for (int m = 0; m < KREGS; ++m) {
                kw0[m] = ld_unit<G::KUNIT>(stage + k_off0 + 4 * G::KUNIT * m);
                kw1[m] = ld_unit<G::KUNIT>(stage + k_off1 + 4 * G::KUNIT * m);
            }
        } else {
            ld_words(stage, k_off0, kw0);
            ld_words(stage, k_off1, kw1);
        }
#pragma unroll
        for (int j = 0; j < G::KSTEPS; ++j) {
            // a = {row r dims 0-1, row r+8 dims 0-1, row r dims 2-3, row r+8 dims 2-3}
            // of the 4 dims this lane covers at k-step j
            uint32_t af[4];
            if constexpr (KB == 8) {
                // unit j: 4 FP8 codes; each 16-bit half is one e4m3 pair -> f16x2
                e4m3x4_to_f16x2(kw0[j], af[0], af[2]);
                e4m3x4_to_f16x2(kw1[j], af[1], af[3]);
            } else if constexpr (kPairK) {
                // k-step j: two pair codes, bytes 2 (j % 2) and 2 (j % 2) + 1 of
                // word j / 2, moved to the table's entry stride
                constexpr int kS = G::LUT_SHIFT;
                constexpr uint32_t kM = 0xFFu << kS;
                const uint32_t w0 = kw0[j >> 1], w1 = kw1[j >> 1];
                const bool hi = (j & 1) != 0;  // a constant once the loop is unrolled
                const uint32_t p0 = hi ? (w0 >> (16 - kS)) : (w0 << kS);
                const uint32_t p1 = hi ? (w1 >> (16 - kS)) : (w1 << kS);
                const uint32_t q0 = hi ? (w0 >> (24 - kS)) : (w0 >> (8 - kS));
                const uint32_t q1 = hi ? (w1 >> (24 - kS)) : (w1 >> (8 - kS));
                af[0] = ld32(lut + ((p0 & kM) | lane4));
                af[1] = ld32(lut + ((p1 & kM) | lane4));
                af[2] = ld32(lut + ((q0 & kM) | lane4));
                af[3] = ld32(lut + ((q1 & kM) | lane4));
            } else if constexpr (KB == 4) {
                // unit j: two pair codes, one per byte, moved to the table's entry stride
                constexpr int kS = G::LUT_SHIFT;
                constexpr uint32_t kM = 0xFFu << kS;
                af[0] = ld32(lut + (((kw0[j] << kS) & kM) | lane4));
                af[1] = ld32(lut + (((kw1[j] << kS) & kM) | lane4));
                af[2] = ld32(lut + (((kw0[j] >> (8 - kS)) & kM) | lane4));
                af[3] = ld32(lut + (((kw1[j] >> (8 - kS)) & kM) | lane4));
            } else {
                // 6-bit pair codes at bit 6 * pair of the lane's block, moved to bit 7
                constexpr int kS = G::LUT_SHIFT;
                constexpr uint32_t kIdx = 0x3Fu << kS;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int bit = 6 * (2 * j + e);
                    const int wi = bit / 32, off = bit % 32;
                    uint32_t x0, x1;
                    if (off + 6 <= 32) {
                        x0 = off <= kS ? (kw0[wi] << (kS - off)) : (kw0[wi] >> (off - kS));
                        x1 = off <= kS ? (kw1[wi] << (kS - off)) : (kw1[wi] >> (off - kS));
                    } else {
                        x0 = __funnelshift_r(kw0[wi], kw0[wi + 1], off - kS);
                        x1 = __funnelshift_r(kw1[wi], kw1[wi + 1], off - kS);
                    }
                    af[2 * e] = ld32(lut + ((x0 & kIdx) | lane4));
                    af[2 * e + 1] = ld32(lut + ((x1 & kIdx) | lane4));
                }
            }
            const uint32_t afrag[4] = {af[0], af[1], af[2], af[3]};
            if constexpr (PACKQ) {
                const uint2 qb = qfrag2[j * 32];
                mma16816(qacc[j & 1], afrag, qb.x, qb.y);
            } else {
                const uint4 qb = qfrag[j * qstride];
                mma16816(qacc[0], afrag, qb.x, qb.y);
                mma16816(qacc[1], afrag, qb.z, qb.w);
            }
            if constexpr (NC) {
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
        float sacc[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[e] = qacc[0][e] + qacc[1][e];
        if constexpr (PACKQ) {
            // column n + 4 holds the lo part of column n: lanes c and c ^ 2 swap
            // them, so columns n and n + 4 both end with the full score
#pragma unroll
            for (int e = 0; e < 4; ++e) sacc[e] += __shfl_xor_sync(kFull, sacc[e], 2);
        }
        float n0 = 0.f, n1 = 0.f;  // ||c~||^2 of rows r, r + 8 (this warp's share)
        if constexpr (NC) {
            n0 = nacc[0];
            n1 = nacc[2];
        }
        if constexpr (WPH > 1) {
            // add the other warps' shares of the dims
            float* xb = xch + buf * (G::NWARPS * 32 * 6);  // alternate buffers: no overwrite before it is read
            reinterpret_cast<float4*>(xb + warp * 192)[lane] = make_float4(sacc[0], sacc[1], sacc[2], sacc[3]);
            if constexpr (NC) reinterpret_cast<float2*>(xb + warp * 192 + 128)[lane] = make_float2(n0, n1);
            group_barrier(1 + h, 32 * WPH);
#pragma unroll
            for (int w = 1; w < WPH; ++w) {
                const int ow = h * WPH + (part + w) % WPH;
                const float4 os = reinterpret_cast<const float4*>(xb + ow * 192)[lane];
                sacc[0] += os.x;
                sacc[1] += os.y;
                sacc[2] += os.z;
                sacc[3] += os.w;
                if constexpr (NC) {
                    const float2 on = reinterpret_cast<const float2*>(xb + ow * 192 + 128)[lane];
                    n0 += on.x;
                    n1 += on.y;
                }
            }
        }
        // per-token factors: vec_norm, norm correction
        float f_r = 1.f, f_r8 = 1.f;
        if constexpr (KB != 8) {
            f_r = half_from_bits(ld16(stage + n_off0));
            f_r8 = half_from_bits(ld16(stage + n_off1));
            if constexpr (NC) {
                f_r *= rsqrtf(n0);
                f_r8 *= rsqrtf(n1);
            }
        }
        const bool v_r = ok && tok0 + tq0 < L;
        const bool v_r8 = ok && tok0 + tq1 < L;
        sc[0] = v_r ? sacc[0] * f_r : -INFINITY;
        sc[1] = v_r ? sacc[1] * f_r : -INFINITY;
        sc[2] = v_r8 ? sacc[2] * f_r8 : -INFINITY;
        sc[3] = v_r8 ? sacc[3] * f_r8 : -INFINITY;
    };

    // ---- value codes and (scale, zero) of one staged chunk, kept in registers
    // until the chunk's P.V one step later ------------------------------------------
    // 2-byte value units of two tokens share one register (token 2c or 2c + 8
    // in the low half, 2c + 1 or 2c + 9 in the high half): half the registers
    // a chunk's values take while they wait for its P.V.
    constexpr bool kPackV = G::VUNITS && G::VUNIT == 2;
    constexpr int kVR2 = kPackV ? 1 : G::VREGS;
    struct VRegs {
        uint32_t w0[G::VREGS], w1[kVR2], w8[G::VREGS], w9[kVR2];  // k-columns 2c, 2c+1, 2c+8, 2c+9
        uint32_t sz0, sz1;  // half2 (scale, zero) of rows r, r + 8
    };
    auto load_v = [&](const uint8_t* stage, VRegs& vr) {
        if constexpr (kPackV) {
#pragma unroll
            for (int m = 0; m < G::VNU; ++m) {
                vr.w0[m] = prmt(ld_unit<2>(stage + v_off0 + 16 * m), ld_unit<2>(stage + v_off1 + 16 * m), 0x5410u);
                vr.w8[m] = prmt(ld_unit<2>(stage + v_off8 + 16 * m), ld_unit<2>(stage + v_off9 + 16 * m), 0x5410u);
            }
        } else if constexpr (G::VUNITS) {
#pragma unroll
            for (int m = 0; m < G::VNU; ++m) {
                vr.w0[m] = ld_unit<G::VUNIT>(stage + v_off0 + 8 * G::VUNIT * m);
                vr.w1[m] = ld_unit<G::VUNIT>(stage + v_off1 + 8 * G::VUNIT * m);
                vr.w8[m] = ld_unit<G::VUNIT>(stage + v_off8 + 8 * G::VUNIT * m);
                vr.w9[m] = ld_unit<G::VUNIT>(stage + v_off9 + 8 * G::VUNIT * m);
            }
        } else {
            ld_words(stage, v_off0, vr.w0);
            ld_words(stage, v_off1, vr.w1);
            ld_words(stage, v_off8, vr.w8);
            ld_words(stage, v_off9, vr.w9);
        }
        vr.sz0 = static_cast<uint32_t>(ld16(stage + z_off0)) | (static_cast<uint32_t>(ld16(stage + z_off0 + 2)) << 16);
        vr.sz1 = static_cast<uint32_t>(ld16(stage + z_off1)) | (static_cast<uint32_t>(ld16(stage + z_off1 + 2)) << 16);
    };

    // ---- running state ---------------------------------------------------------------
    float o[G::MTILES][4];
#pragma unroll
    for (int mt = 0; mt < G::MTILES; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[mt][e] = 0.f;
    float ob[4] = {0.f, 0.f, 0.f, 0.f};  // row 0: sum of P' per query column
    // A finite start (far below any score) keeps every exponent and rescale
    // factor finite: the first chunk always raises it to the real maximum.
    constexpr float kMinRef = -1e30f;
    float m_ref[2] = {kMinRef, kMinRef};
    float l_acc[2] = {0.f, 0.f};
    float z_acc[2] = {0.f, 0.f};
    const uint32_t bias_a = (r == 0) ? 0x3C003C00u : 0u;
    const uint32_t a_bias[4] = {bias_a, 0u, bias_a, 0u};

    // ---- online softmax and P.V of one chunk (scores sc, values vr) -------------
    auto rescale = [&](const float (&sc)[4]) {
        // lazy rescale: the reference max moves only when a score passes it by
        // more than 2^8; a per-lane test, reduced across the warp only then
        const bool grow = (sc[0] > m_ref[0] + kRescaleThreshold) || (sc[2] > m_ref[0] + kRescaleThreshold) ||
                          (sc[1] > m_ref[1] + kRescaleThreshold) || (sc[3] > m_ref[1] + kRescaleThreshold);
        if (__any_sync(kFull, grow)) {
            float mx0 = fmaxf(sc[0], sc[2]);
            float mx1 = fmaxf(sc[1], sc[3]);
#pragma unroll
            for (int m = 4; m < 32; m <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, m));
                mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, m));
            }
            const float n0m = fmaxf(m_ref[0], mx0);
            const float n1m = fmaxf(m_ref[1], mx1);
            const float al0 = fast_exp2(m_ref[0] - n0m);
            const float al1 = fast_exp2(m_ref[1] - n1m);
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
            m_ref[0] = n0m;
            m_ref[1] = n1m;
        }
    };
    auto softmax_pv = [&](const float (&sc)[4], const VRegs& vr, int tok0, bool ok) {
        // After the rescale test every finite score is at most 2^8 above its
        // column's reference; exp2(-inf) = 0 masks past-the-end tokens.
        float pr[4];
        pr[0] = fast_exp2(sc[0] - m_ref[0]);
        pr[1] = fast_exp2(sc[1] - m_ref[1]);
        pr[2] = fast_exp2(sc[2] - m_ref[0]);
        pr[3] = fast_exp2(sc[3] - m_ref[1]);
        l_acc[0] += pr[0] + pr[2];
        l_acc[1] += pr[1] + pr[3];

        // value scale / zero of tokens r and r + 8 (0 past the end)
        const bool v_r = ok && tok0 + tq0 < L;
        const bool v_r8 = ok && tok0 + tq1 < L;
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&vr.sz0));
        const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&vr.sz1));
        const float vs_r = v_r ? f0.x : 0.f, vz_r = v_r ? f0.y : 0.f;
        const float vs_r8 = v_r8 ? f1.x : 0.f, vz_r8 = v_r8 ? f1.y : 0.f;
        // zero point plus the centre of the code range (codes enter centred)
        const float zc_r = fmaf(kCentre, vs_r, vz_r);
        const float zc_r8 = fmaf(kCentre, vs_r8, vz_r8);
        z_acc[0] = fmaf(pr[0], zc_r, fmaf(pr[2], zc_r8, z_acc[0]));
        z_acc[1] = fmaf(pr[1], zc_r, fmaf(pr[3], zc_r8, z_acc[1]));
        const uint32_t pb0 = movmatrix_trans(pack_half2(pr[0] * vs_r, pr[1] * vs_r));
        const uint32_t pb1 = movmatrix_trans(pack_half2(pr[2] * vs_r8, pr[3] * vs_r8));

        // P.V over this warp's share of the dims: codes enter as fp16
        // subnormals code * 2^(pos - 24), masked in place
#pragma unroll
        for (int mt = 0; mt < G::MTILES; ++mt) {
            uint32_t vf[4];
            if constexpr (kPackV) {
                // local dims 2mt, 2mt + 1 share byte b of unit m.  One PRMT
                // gives both tokens' byte b (bytes b and b + 2 of the packed
                // pair) with a zero byte above each: the odd dim enters as the
                // whole byte (16 hi + lo) and the epilogue subtracts the even
                // dim's sum (lo), which the same MMA produces.
                const int m = (2 * mt) / G::VDPU, b = ((2 * mt) % G::VDPU) / 2;
                const uint32_t sel = b | (4 << 4) | ((b + 2) << 8) | (4 << 12);
                const uint32_t win0 = prmt(vr.w0[m], 0u, sel);
                const uint32_t win8 = prmt(vr.w8[m], 0u, sel);
                vf[0] = win0 & 0x000F000Fu;
                vf[1] = win0;
                vf[2] = win8 & 0x000F000Fu;
                vf[3] = win8;
            } else if constexpr (G::VUNITS) {
                // local dims 2mt, 2mt + 1 share one byte of unit m
                const int m = (2 * mt) / G::VDPU, w = (2 * mt) % G::VDPU;
                vf[0] = value_unit_sub(vr.w0[m], vr.w1[m], w);
                vf[1] = value_unit_sub(vr.w0[m], vr.w1[m], w + 1);
                vf[2] = value_unit_sub(vr.w8[m], vr.w9[m], w);
                vf[3] = value_unit_sub(vr.w8[m], vr.w9[m], w + 1);
            } else {
                vf[0] = value_sub<VB>(vr.w0, vr.w1, 2 * mt);
                vf[1] = value_sub<VB>(vr.w0, vr.w1, 2 * mt + 1);
                vf[2] = value_sub<VB>(vr.w8, vr.w9, 2 * mt);
                vf[3] = value_sub<VB>(vr.w8, vr.w9, 2 * mt + 1);
            }
            mma16816(o[mt], vf, pb0, pb1);
        }
        mma16816(ob, a_bias, pb0, pb1);
    };

    // ---- main loop: QK of chunk it and the softmax and P.V of chunk it - 1 form
    // one straight-line block; waits and the rare rescale sit outside it -------
    // After a wait gives up, the warp stops waiting and runs on with every
    // chunk masked, so that warps sharing a head still meet at each exchange.
    bool timed_out = false;
    auto acquire = [&](int it, int& blk) -> const uint8_t* {
        const int slot = it % NS;
        blk = -1;
        if (!timed_out) {
            if (mbar_wait(full_bar(slot), static_cast<uint32_t>((it / NS) & 1))) blk = stage_blk[slot];
            else timed_out = true;
        }
        return ring + slot * G::STAGE;
    };
    auto release = [&](int it) {
        __syncwarp();
        if (lane == 0) {
            const int slot = it % NS;
            if (atom_add_acq_rel(cnt_addr(slot), 1u) == static_cast<uint32_t>(G::NWARPS - 1)) {
                *reinterpret_cast<volatile uint32_t*>(ctrl + 8 * NS + 4 * slot) = 0u;
                if (it + NS < nch) {
                    fence_proxy_async();
                    issue(it + NS);
                }
            }
        }
    };
    // With a deep ring the stage of chunk it - 1 stays resident until its P.V
    // (value codes re-read from shared memory); with a shallow one the codes
    // ride in registers and the stage is released right after its QK.
    constexpr bool kCarry = NS <= 3;
    float sc_prev[4];
    VRegs v_prev;
    bool ok_prev = false;
    const uint8_t* stage_prev = ring;
    if (nch > 0) {
        int blk = -1;
        stage_prev = acquire(0, blk);
        ok_prev = blk >= 0;
        qk(stage_prev, c0 * kTok, ok_prev, 0, sc_prev);
        if constexpr (kCarry) {
            load_v(stage_prev, v_prev);
            release(0);
        }
    }
#pragma unroll 1
    for (int it = 1; it < nch; ++it) {
        int blk = -1;
        const uint8_t* stage = acquire(it, blk);
        if (!ok_prev && !timed_out && lane == 0 && warp == 0) set_flag(c.flags, kFlagBlock);
        rescale(sc_prev);
        const bool ok = blk >= 0;
        float sc_cur[4];
        qk(stage, (c0 + it) * kTok, ok, it & 1, sc_cur);
        if constexpr (kCarry) {
            VRegs v_cur;
            load_v(stage, v_cur);
            softmax_pv(sc_prev, v_prev, (c0 + it - 1) * kTok, ok_prev);
            release(it);
            v_prev = v_cur;
        } else {
            load_v(stage_prev, v_prev);
            softmax_pv(sc_prev, v_prev, (c0 + it - 1) * kTok, ok_prev);
            release(it - 1);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) sc_prev[e] = sc_cur[e];
        ok_prev = ok;
        stage_prev = stage;
    }
    if (nch > 0) {
        if (!ok_prev && !timed_out && lane == 0 && warp == 0) set_flag(c.flags, kFlagBlock);
        rescale(sc_prev);
        if constexpr (!kCarry) load_v(stage_prev, v_prev);
        softmax_pv(sc_prev, v_prev, (c1 - 1) * kTok, ok_prev);
        if constexpr (!kCarry) release(nch - 1);
    }
    if (timed_out) {
        if (lane == 0) {
            set_flag(c.flags, kFlagWait);
            atomicExch(err_word, 1);
        }
    }
    // A CTA must not exit with bulk copies into its shared memory in flight.
    // Normally every issued chunk has been consumed; after a timed-out wait,
    // thread 0 waits (bounded) for the stages' last phases.
    __syncthreads();
    if (threadIdx.x == 0 && *reinterpret_cast<volatile int*>(err_word) != 0) {
        for (int it = nch - 1; it >= 0 && it >= nch - NS; --it)
            mbar_wait(full_bar(it % NS), static_cast<uint32_t>((it / NS) & 1));
    }
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
        float* part_out = a.partials + ((static_cast<int64_t>(s) * Hq + hq) * a.slot_stride + split) * (D + 2);
        if (r == 0 && part == 0) {
            part_out[0] = m_ref[e];
            part_out[1] = l_acc[e];
        }
        const float cb = kCentre * (e ? bias1 : bias0);
        const float z = z_acc[e];
#pragma unroll
        for (int mt = 0; mt < G::MTILES; ++mt) {
            // sum P'(code - centre) = o * 2^(24 - pos) - centre * bias
            int d0;
            float w0, w1;
            if constexpr (G::VUNITS) {
                const int m = (2 * mt) / G::VDPU, w = (2 * mt) % G::VDPU;
                d0 = part * (D / WPH) + G::VDPU * (r + 8 * m) + w;
                w0 = 16777216.f;  // even dim of the pair: low nibble
                w1 = 1048576.f;   // odd dim: high nibble
            } else {
                d0 = r * (D / 8) + 2 * (part * G::MTILES + mt);
                w0 = value_weight<VB>(2 * mt);
                w1 = value_weight<VB>(2 * mt + 1);
            }
            // (2-byte value units: row r + 8 holds 16 hi + lo, row r holds lo)
            const float odd = (G::VUNITS && G::VUNIT == 2) ? o[mt][2 + e] - o[mt][e] : o[mt][2 + e];
            part_out[2 + d0] = fmaf(o[mt][e], w0, -cb) + z;
            part_out[2 + d0 + 1] = fmaf(odd, w1, -cb) + z;
        }
    }
}

template <int D, int KB, int VB>
constexpr bool share_aligned(int wph) {
    // each warp's share of a thread's key and value codes starts on a byte
    return ((D / 4 / wph) * KB) % 8 == 0 && ((D / 8 / wph) * VB) % 8 == 0 && (D / 16) % wph == 0;
}

template <int D, int KB, int VB>
constexpr int pick_wph(int want) {
    int w = want;
    while (w > 1 && !share_aligned<D, KB, VB>(w)) w /= 2;
    return w;
}

// Launch policy per shape: warps per head, resident CTAs per SM aimed for,
// and the deepest stage ring that fits the shared memory that leaves.
// About four warps per CTA: with up to four KV heads each warp takes a whole
// head (no split dims, so no score exchange and no duplicated softmax) and
// three CTAs share an SM (registers allow ~170 per thread; shared memory
// then takes the 16-copy table and a 2-stage ring).  At d = 256, 4 KV heads
// this measured 173.6 us per decode of 256 x 2048 tokens against 190.7 us
// with two warps per head and two CTAs per SM.  Eight KV heads keep one warp
// per head in 256-thread CTAs, two per SM.
template <int D, int KB, int VB, int H, bool PACKQ>
struct Policy {
    static constexpr int kWarpsTarget = 4;
    static constexpr int kWphRaw = kWarpsTarget / H;
    static constexpr int kWphMax = D / 32;  // at least two k-steps per warp
    static constexpr int WPH = pick_wph<D, KB, VB>(kWphRaw < 1 ? 1 : (kWphRaw > kWphMax ? kWphMax : kWphRaw));
    static constexpr int MINB = 32 * H * WPH > 256 ? 1 : (32 * H * WPH > 128 ? 2 : 3);
    // per-CTA shared memory: 228 KB per SM, less 1 KB reserved per CTA
    static constexpr int kBudget = MINB == 1 ? 227 * 1024 : (MINB == 2 ? 113 * 1024 : 74 * 1024);
    using G1 = Geo<D, KB, VB, H, WPH, 8, PACKQ, (MINB >= 3 ? 16 : 32)>;
    // fixed part plus the query fragments (unpacked: up to 5 query heads per KV head)
    static constexpr int kFixed = G1::RING_OFF + 16 + (PACKQ ? H * D * 16 : H * 5 * D * 4);
    static constexpr int kNs = (kBudget - kFixed) / G1::STAGE;
    static constexpr int NS = kNs < 2 ? 2 : (kNs > 8 ? 8 : kNs);
};

// Shared-memory wavefronts one warp-wide load takes: the largest number of
// distinct 4-byte words any bank is asked for (at least bytes / 128).
inline int bank_wavefronts(const int (&addr)[32], int width) {
    int words[32][8];
    int count[32] = {};
    int deg = 1;
    for (int l = 0; l < 32; ++l) {
        for (int wd = addr[l] / 4; wd <= (addr[l] + width - 1) / 4; ++wd) {
            const int b = wd % 32;
            bool seen = false;
            for (int i = 0; i < count[b]; ++i) seen = seen || words[b][i] == wd;
            if (!seen && count[b] < 8) words[b][count[b]++] = wd;
            deg = count[b] > deg ? count[b] : deg;
        }
    }
    const int floor = (width * 32 + 127) / 128;
    return deg > floor ? deg : floor;
}

// Wavefronts of the code loads of one chunk, summed over the warps, under a
// token order (eo: rows 0-7 take the even tokens and rows 8-15 the odd ones).
// It mirrors the kernel's per-lane offsets.
template <class G, int D, int KB, int VB, int H, int WPH>
int load_wavefronts(bool eo) {
    using S = typename G::S;
    auto sig = [&](int k) { return eo ? (k < 8 ? 2 * k : 2 * (k - 8) + 1) : k; };
    int total = 0;
    int addr[32];
    for (int h = 0; h < H; ++h) {
        const int hs = h * G::SA;
        for (int part = 0; part < WPH; ++part) {
            for (int k = 0; k < 16; k += 8) {
                const bool u4 = G::PAIR_K && G::ROW % 4 == 0 && (hs + part * G::KSH) % 4 == 0;
                for (int l = 0; l < 32; ++l) {
                    const int r = l / 4, c = l % 4;
                    const int base = G::KUNITS ? hs + part * G::KSH + (u4 ? 4 : G::KUNIT) * c
                                               : hs + c * G::KBYTES + part * G::KBYTES_W;
                    addr[l] = sig(r + k) * G::ROW + base;
                    if (!G::KUNITS) addr[l] &= ~3;
                }
                total += !G::KUNITS ? bank_wavefronts(addr, 4) * (G::KWORDS + 1)
                                    : (u4 ? bank_wavefronts(addr, 4) * (G::KSTEPS / 2)
                                          : bank_wavefronts(addr, G::KUNIT) * G::KSTEPS);
            }
            const int kcols[4] = {0, 1, 8, 9};
            for (int kc : kcols) {
                for (int l = 0; l < 32; ++l) {
                    const int r = l / 4, c = l % 4;
                    const int base = G::VUNITS ? hs + S::kKeyBytes + part * G::VSH + G::VUNIT * r
                                               : hs + S::kKeyBytes + (r * (D / 8) * VB + part * G::VBITS_W) / 8;
                    addr[l] = sig(2 * c + kc) * G::ROW + base;
                    if (!G::VUNITS) addr[l] &= ~3;
                }
                total += G::VUNITS ? bank_wavefronts(addr, G::VUNIT) * G::VNU
                                   : bank_wavefronts(addr, 4) * (G::VWORDS + 1);
            }
        }
    }
    return total;
}

template <int D, int KB, int VB, bool NC, int H, bool PACKQ>
struct Kernel {
    using P = Policy<D, KB, VB, H, PACKQ>;
    using G = Geo<D, KB, VB, H, P::WPH, P::NS, PACKQ, (P::MINB >= 3 ? 16 : 32)>;
    static constexpr auto fn = decode_kernel<D, KB, VB, NC, H, P::WPH, P::NS, P::MINB, PACKQ>;

    // Per device (function attributes belong to a device's context): the
    // largest dynamic shared memory granted so far, and the resident CTAs per
    // SM per query-head count, so that repeated calls skip the driver queries.
    static constexpr int kDevs = 16;
    static inline std::atomic<int> granted[kDevs] = {};
    static inline std::atomic<int> ctas_cache[kDevs][65] = {};
    static int device() {
        int dev = -1;
        return cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kDevs ? dev : -1;
    }
    static cudaError_t prepare(int hq, int* smem) {
        *smem = G::smem_bytes(hq);
        const int dev = device();
        if (dev >= 0 && *smem <= granted[dev].load(std::memory_order_relaxed)) return cudaSuccess;
        const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, *smem);
        if (e == cudaSuccess && dev >= 0) {
            int cur = granted[dev].load(std::memory_order_relaxed);
            while (cur < *smem && !granted[dev].compare_exchange_weak(cur, *smem)) {
            }
        }
        return e;
    }
    static cudaError_t occupancy(int hq, int* ctas) {
        const int dev = device();
        const bool cacheable = dev >= 0 && hq >= 0 && hq <= 64;
        if (cacheable) {
            const int v = ctas_cache[dev][hq].load(std::memory_order_relaxed);
            if (v > 0) {
                *ctas = v;
                return cudaSuccess;
            }
        }
        int smem = 0;
        cudaError_t e = prepare(hq, &smem);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, fn, G::NT, smem);
        if (e == cudaSuccess && cacheable) ctas_cache[dev][hq].store(*ctas, std::memory_order_relaxed);
        return e;
    }
    static cudaError_t launch(const LayerParams& p, const CacheGeom& c, const Args& a, int num_seqs,
                              cudaStream_t stream) {
        int smem = 0;
        const cudaError_t e = prepare(a.num_q_heads, &smem);
        if (e != cudaSuccess) return e;
        static const int tok_eo =
            load_wavefronts<G, D, KB, VB, H, P::WPH>(true) < load_wavefronts<G, D, KB, VB, H, P::WPH>(false) ? 1 : 0;
        Args args = a;
        args.tok_eo = tok_eo;
        dim3 grid(static_cast<unsigned>(a.num_splits), static_cast<unsigned>(num_seqs));
        fn<<<grid, G::NT, smem, stream>>>(p, c, args);
        return cudaGetLastError();
    }
};

// One entry per head size: occupancy query (ctas != nullptr) or launch.
template <int D>
cudaError_t run(const LayerParams& p, const CacheGeom& c, const Args& a, int num_seqs, int num_kv_heads,
                cudaStream_t stream, int* ctas) {
    auto go = [&](auto kern) -> cudaError_t {
        using K = decltype(kern);
        if (ctas != nullptr) return K::occupancy(a.num_q_heads, ctas);
        return K::launch(p, c, a, num_seqs, stream);
    };
    // up to 4 query heads per KV head: hi and lo query parts share one MMA
    const bool packq = num_kv_heads > 0 && a.num_q_heads / num_kv_heads <= 4;
    auto by_h = [&](auto kb, auto vb, auto nc) -> cudaError_t {
        constexpr int KB = decltype(kb)::value, VB = decltype(vb)::value;
        constexpr bool NC = decltype(nc)::value;
        auto by_q = [&](auto h) -> cudaError_t {
            constexpr int HH = decltype(h)::value;
            if (packq) return go(Kernel<D, KB, VB, NC, HH, true>{});
            return go(Kernel<D, KB, VB, NC, HH, false>{});
        };
        switch (num_kv_heads) {
            case 1: return by_q(std::integral_constant<int, 1>{});
            case 2: return by_q(std::integral_constant<int, 2>{});
            case 4: return by_q(std::integral_constant<int, 4>{});
            case 8: return by_q(std::integral_constant<int, 8>{});
            default: return cudaErrorInvalidValue;
        }
    };
    auto by_nc = [&](auto kb, auto vb) -> cudaError_t {
        if constexpr (decltype(kb)::value != 8) {
            if (p.nc) return by_h(kb, vb, std::true_type{});
        }
        return by_h(kb, vb, std::false_type{});
    };
    using I3 = std::integral_constant<int, 3>;
    using I4 = std::integral_constant<int, 4>;
    using I8 = std::integral_constant<int, 8>;
    const int kb = p.kbits, vb = p.vbits;
    if (kb == 3 && vb == 3) return by_nc(I3{}, I3{});
    if (kb == 3 && vb == 4) return by_nc(I3{}, I4{});
    if (kb == 4 && vb == 3) return by_nc(I4{}, I3{});
    if (kb == 4 && vb == 4) return by_nc(I4{}, I4{});
    if (kb == 8 && vb == 3) return by_nc(I8{}, I3{});
    if (kb == 8 && vb == 4) return by_nc(I8{}, I4{});
    return cudaErrorInvalidValue;
}

}  // namespace mma
}  // namespace tq

namespace tq {
// One translation unit per head size (tq_decode_mma_d{64,128,256}.cu).
// ctas != nullptr: report resident CTAs per SM instead of launching.
cudaError_t decode_mma_run_d64(const LayerParams& p, const CacheGeom& c, const mma::Args& a, int num_seqs,
                               int num_kv_heads, cudaStream_t stream, int* ctas);
cudaError_t decode_mma_run_d128(const LayerParams& p, const CacheGeom& c, const mma::Args& a, int num_seqs,
                                int num_kv_heads, cudaStream_t stream, int* ctas);
cudaError_t decode_mma_run_d256(const LayerParams& p, const CacheGeom& c, const mma::Args& a, int num_seqs,
                                int num_kv_heads, cudaStream_t stream, int* ctas);
}  // namespace tq
