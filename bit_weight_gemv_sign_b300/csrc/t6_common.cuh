// Device helpers shared by the 6-bit-table GEMV kernels: TMA / mbarrier
// wrappers, the table builder and the table lookup.  See gemv_t6.cu for the
// method and the numerical argument.
#pragma once

#include <cuda.h>

#include <utility>

#include "common.cuh"

namespace bit1 {

constexpr int kT6Fields = 22;                     // 21 six-bit + 1 two-bit field per group
constexpr int kT6TableBytes = 128;                // 64 fp16 entries
constexpr int kT6GroupBytes = kT6Fields * kT6TableBytes;  // 2816


// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// Bounded wait on an mbarrier phase: false if it did not complete within
// `polls` suspending try_waits.
__device__ __forceinline__ bool mbar_wait_polls(uint32_t bar, uint32_t parity, uint32_t polls) {
    for (uint32_t i = 0; i < polls; ++i) {
        uint32_t done;
        asm volatile("{.reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p;}"
                     : "=r"(done) : "r"(bar), "r"(parity) : "memory");
        if (done) return true;
    }
    return false;
}
// The kernels' bound: 2^22 polls (about 16 s on B300), far beyond any copy.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    return mbar_wait_polls(bar, parity, 1u << 22);
}
__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
                 ::"r"(dst), "l"(map), "r"(c0), "r"(c1), "r"(bar) : "memory");
}
// 1-D bulk copy global -> shared, completion on an mbarrier (sizes and both
// addresses multiples of 16 bytes).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t local_addr, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

// ---------------------------------------------------------------- tables
// Two 16-byte chunks (entries 8c..8c+7 for c = h and c = h+4) of the table of
// field f of one group, from the group's 128 activations (bf16, shared memory)
// times the group's power-of-two prescale finv (exact): six of them (f < 21)
// or the last two (f = 21: an 8-byte table, written by h = 0).  Entry e sits at byte 2e; complementary indices
// hold exact negatives (every sum is formed symmetrically).  Four threads
// build one table; the thread with odd `flip` writes its upper chunk first,
// so the eight threads of a quarter warp (two tables) store to eight
// different bank quads at each store (no conflicts).
__device__ __forceinline__ void t6_build_pair(uint8_t* tab, const uint16_t* xg, float finv, int f, int h,
                                              int flip) {
    if (f < 21) {
        const uint16_t* xs = xg + 6 * f;   // bf16, 4-byte aligned (6f elements)
        const uint32_t p01 = *reinterpret_cast<const uint32_t*>(xs);
        const uint32_t p23 = *reinterpret_cast<const uint32_t*>(xs + 2);
        const uint32_t p45 = *reinterpret_cast<const uint32_t*>(xs + 4);
        const float v0 = bf16_bits_to_f32(p01 & 0xffffu) * finv, v1 = bf16_bits_to_f32(p01 >> 16) * finv;
        const float v2 = bf16_bits_to_f32(p23 & 0xffffu) * finv, v3 = bf16_bits_to_f32(p23 >> 16) * finv;
        const float v4 = bf16_bits_to_f32(p45 & 0xffffu) * finv, v5 = bf16_bits_to_f32(p45 >> 16) * finv;
        const float a = v0 + v1, b = v0 - v1;
        const float lo[8] = {-a - v2, b - v2, -b - v2, a - v2, -a + v2, b + v2, -b + v2, a + v2};
        const float s3 = (h & 1) ? v3 : -v3, s4 = (h & 2) ? v4 : -v4;
        const float h34 = s3 + s4;                   // +-v3 +-v4 of chunk h (and of h+4)
        const float hc0 = h34 - v5, hc1 = h34 + v5;  // chunk h (bit 5 clear) and h+4 (set)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int which = r ^ flip;              // 0: chunk h, 1: chunk h+4
            const float hc = which ? hc1 : hc0;
            uint32_t wd[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const __half2 q = __floats2half2_rn(lo[2 * j] + hc, lo[2 * j + 1] + hc);
                wd[j] = *reinterpret_cast<const uint32_t*>(&q);
            }
            reinterpret_cast<uint4*>(tab)[h + 4 * which] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
        }
    } else if (h == 0) {
        const uint32_t p = *reinterpret_cast<const uint32_t*>(xg + 126);
        const float v0 = bf16_bits_to_f32(p & 0xffffu) * finv, v1 = bf16_bits_to_f32(p >> 16) * finv;
        const __half2 h0 = __floats2half2_rn(-v0 - v1, v0 - v1);
        const __half2 h1 = __floats2half2_rn(-v0 + v1, v0 + v1);
        *reinterpret_cast<uint2*>(tab) = make_uint2(*reinterpret_cast<const uint32_t*>(&h0),
                                                    *reinterpret_cast<const uint32_t*>(&h1));
    }
}

// Field F of the 128-bit group w[0..3]: its value times 2 (byte offset of the
// fp16 entry), or'ed into the 128-byte aligned table base of the group; the
// entry is loaded here and added by t6_add.  The load is an ordinary
// (non-volatile) shared load so that the compiler can issue the 22 loads of a
// group back to back; its address depends on w, which is only read after the
// stage's mbarrier completed, which orders it after the table build.
template <int F>
__device__ __forceinline__ unsigned short t6_ld(const uint32_t (&w)[4], uint32_t tg) {
    constexpr int O = 6 * F, QW = O >> 5, S = O & 31;
    uint32_t v;
    if constexpr (F == 21) v = (w[3] >> 29) & 0x6u;
    else if constexpr (S == 0) v = (w[QW] << 1) & 0x7Eu;
    else if constexpr (S + 6 <= 32) v = (w[QW] >> (S - 1)) & 0x7Eu;
    else v = __funnelshift_r(w[QW], w[QW + 1], S - 1) & 0x7Eu;
    unsigned short t;
    asm("ld.shared.b16 %0, [%1+%2];" : "=h"(t) : "r"(v | tg), "n"(F * kT6TableBytes));
    return t;
}

// acc + (fp32) t, the fp16 -> fp32 widening exact, in one mixed-precision add
// (one rounding, in fp32).
__device__ __forceinline__ float t6_add(unsigned short t, float acc) {
    asm("add.rn.f32.f16 %0, %1, %0;" : "+f"(acc) : "h"(t));
    return acc;
}

template <size_t... F>
__device__ __forceinline__ float t6_group(const uint32_t (&w)[4], uint32_t tg, std::index_sequence<F...>) {
    unsigned short t[sizeof...(F)];
    ((t[F] = t6_ld<(int)F>(w, tg)), ...);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    ((acc[F & 3] = t6_add(t[F], acc[F & 3])), ...);
    return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

// ---------------------------------------------------------------- layouts
// Sign bits of a 128-input group as stored in memory: 16 bytes = 4 words.
//  * Layout 0 (canonical): input k of the group is bit k % 32 of word k / 32
//    (row-major, least significant bit first).  Field F (inputs 6F..6F+5) is
//    extracted with a shift and a mask.
//  * Layout 1 ("g128x", a permutation of the bits within each group, so that
//    a whole-row XOR still flips exactly that row): words 0-2 hold fields
//    0..11 at bits 1-6 of their bytes (field F in byte F of the 12; input
//    6F + i at bit 8F + 1 + i), and bits 0 and 7 of those 12 bytes hold the
//    24 inputs of fields 12..15: input 72 + 6j + i (j = 0..3, i = 0..5) sits
//    in word i / 2, at bit 7 of byte j if i is even, else at bit 0 of byte
//    (j + 1) % 4.  Word 3 is as in layout 0 (fields 16..20 and the last two
//    inputs).  Then one mask per word and one byte permute per field give
//    fields 0..11, three rotations and three and-ors gather fields 12..15
//    into the bytes of one word (rotating word q right by 6 - 2q brings its
//    bit 7 of byte j and bit 0 of byte j + 1 to bits 8j + 1 + 2q and 8j + 2 + 2q),
//    and a byte permute gives each of them: 37 integer operations per group
//    instead of 44.  The fields cover the same inputs as in layout 0, so the
//    tables are the same.
constexpr int kLayoutCanonical = BIT1_LAYOUT_CANONICAL;
constexpr int kLayoutG128x = BIT1_LAYOUT_G128X;

// Field F of group w[0..3] in layout L, times 2 (the byte offset of its fp16
// entry), in the low byte of a copy of tg0 (a 256-byte aligned table base).
template <int L, int F>
__device__ __forceinline__ uint32_t t6_addr(const uint32_t (&w)[4], uint32_t tg0) {
    constexpr int O = 6 * F, QW = O >> 5, S = O & 31;
    if constexpr (L == kLayoutG128x && F < 12) {
        const uint32_t m = w[F >> 2] & 0x7E7E7E7Eu;                     // shared by four fields
        return __byte_perm(m, tg0, 0x7650u | (uint32_t)(F & 3));
    } else if constexpr (L == kLayoutG128x && F < 16) {
        const uint32_t v = (__funnelshift_r(w[0], w[0], 6) & 0x06060606u) |
                           (__funnelshift_r(w[1], w[1], 4) & 0x18181818u) |
                           (__funnelshift_r(w[2], w[2], 2) & 0x60606060u);   // shared by four fields
        return __byte_perm(v, tg0, 0x7650u | (uint32_t)(F - 12));
    } else {
        uint32_t v;
        if constexpr (F == 21) v = (w[3] >> 29) & 0x6u;
        else if constexpr (S == 0) v = (w[QW] << 1) & 0x7Eu;
        else if constexpr (S + 6 <= 32) v = (w[QW] >> (S - 1)) & 0x7Eu;
        else v = __funnelshift_r(w[QW], w[QW + 1], S - 1) & 0x7Eu;
        return v | tg0;
    }
}

// The lookup for group JJ of a run of consecutive groups whose tables start
// at the 256-byte aligned address tg0: the group's offset JJ * 2816 and the
// field's F * 128 both ride in the load's immediate, so forming the address
// costs only the field extraction.
template <int L, int F, int JJ>
__device__ __forceinline__ unsigned short t6_ldj(const uint32_t (&w)[4], uint32_t tg0) {
    unsigned short t;
    asm("ld.shared.b16 %0, [%1+%2];" : "=h"(t) : "r"(t6_addr<L, F>(w, tg0)), "n"(JJ * kT6GroupBytes + F * kT6TableBytes));
    return t;
}

// Sum of the 22 entries of group JJ (relative to tg0) in two interleaved fp32
// chains: one widening add per entry and a single add to join the chains.
template <int L, int JJ, size_t... F>
__device__ __forceinline__ float t6_groupj(const uint32_t (&w)[4], uint32_t tg0, std::index_sequence<F...>) {
    unsigned short t[sizeof...(F)];
    ((t[F] = t6_ldj<L, (int)F, JJ>(w, tg0)), ...);
    float acc[2] = {0.f, 0.f};
    ((acc[F & 1] = t6_add(t[F], acc[F & 1])), ...);
    return acc[0] + acc[1];
}

// Layout-aware form of t6_group (tg: the group's 256-byte aligned tables).
template <int L>
struct T6GroupL {
    template <size_t... F>
    static __device__ __forceinline__ float run(const uint32_t (&w)[4], uint32_t tg, std::index_sequence<F...>) {
        unsigned short t[sizeof...(F)];
        ((t[F] = t6_ldj<L, (int)F, 0>(w, tg)), ...);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        ((acc[F & 3] = t6_add(t[F], acc[F & 3])), ...);
        return (acc[0] + acc[1]) + (acc[2] + acc[3]);
    }
};

}  // namespace bit1
