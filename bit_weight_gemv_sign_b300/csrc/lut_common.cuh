// Nibble-table helpers shared by the batch-1 table kernel (gemv_lut.cu) and
// the persistent chain kernel (chain.cu): the fp32 tables of 16 signed sums
// per four inputs, their conflict-free layout (a table lives in the bank of
// the lane that reads it), the row loads and the per-row lookup sum.  The
// method: packed sign bits with one fp16 scale per 128 inputs (web page
// "Bonsai 27B: 노트북과 폰에서 실행되는 27B급 이진 및 삼진 저비트 LLM", section
// "이진(Binary) 가중치 형식"); four weights per lookup, no multiply per weight.
#pragma once

#include <utility>

#include "common.cuh"

namespace bit1 {

constexpr int kLutMaxM = 13;            // fp32 tables: 16 KB per 1024 of K
constexpr int kLutThreads = 512;

template <int IMM>
__device__ __forceinline__ float lds_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1+%2];" : "=f"(v) : "r"(addr), "n"(IMM));
    return v;
}

// Sum of the 8 table entries selected by the 8 nibbles of word w, whose
// tables sit in slots 8J..8J+7 of this lane.  lb = 2 KB-aligned table base +
// 4*lane, so (e*128) | lb is the entry address without an add.
template <int J>
__device__ __forceinline__ float lut_word(uint32_t w, uint32_t lb) {
    constexpr int S = 8 * J * 2048;
    const float v0 = lds_f32<S + 0 * 2048>(((w << 7) & 0x780u) | lb);
    const float v1 = lds_f32<S + 1 * 2048>(((w << 3) & 0x780u) | lb);
    const float v2 = lds_f32<S + 2 * 2048>(((w >> 1) & 0x780u) | lb);
    const float v3 = lds_f32<S + 3 * 2048>(((w >> 5) & 0x780u) | lb);
    const float v4 = lds_f32<S + 4 * 2048>(((w >> 9) & 0x780u) | lb);
    const float v5 = lds_f32<S + 5 * 2048>(((w >> 13) & 0x780u) | lb);
    const float v6 = lds_f32<S + 6 * 2048>(((w >> 17) & 0x780u) | lb);
    const float v7 = lds_f32<S + 7 * 2048>(((w >> 21) & 0x780u) | lb);
    return ((v0 + v1) + (v2 + v3)) + ((v4 + v5) + (v6 + v7));
}

template <int M, size_t... J>
__device__ __forceinline__ void lut_words(const uint32_t (&w)[M], uint32_t lb, float (&ws)[M],
                                          std::index_sequence<J...>) {
    ((ws[J] = lut_word<(int)J>(w[J], lb)), ...);
}

template <int M>
struct LutCfg {
    static constexpr int NS = (M % 4 == 0) ? M / 4 : (M + 6) / 4;  // scales per lane per row
    static constexpr int D = (16 / M) < 2 ? 2 : ((16 / M) > 8 ? 8 : 16 / M);  // rows in flight
    static constexpr int VEC = (M % 4 == 0) ? 4 : ((M % 2 == 0) ? 2 : 1);
    static constexpr size_t smem = (size_t)16384 * M + 2048;
};

template <int M>
__device__ __forceinline__ void load_row(const uint8_t* __restrict__ bits,
                                         const uint16_t* __restrict__ scales, int64_t row,
                                         int lane, uint32_t (&w)[M],
                                         uint32_t (&s)[LutCfg<M>::NS]) {
    constexpr int K = 1024 * M, G = K / 128;
    const uint8_t* p = bits + row * (K / 8) + (size_t)lane * M * 4;
    if constexpr (LutCfg<M>::VEC == 4) {
#pragma unroll
        for (int v = 0; v < M / 4; ++v) {
            const uint4 t = ldg_stream_v4(p + 16 * v);
            w[4 * v] = t.x; w[4 * v + 1] = t.y; w[4 * v + 2] = t.z; w[4 * v + 3] = t.w;
        }
    } else if constexpr (LutCfg<M>::VEC == 2) {
#pragma unroll
        for (int v = 0; v < M / 2; ++v) {
            const uint2 t = ldg_stream_v2(p + 8 * v);
            w[2 * v] = t.x; w[2 * v + 1] = t.y;
        }
    } else {
#pragma unroll
        for (int v = 0; v < M; ++v) w[v] = ldg_stream_u32(p + 4 * v);
    }
    const int g0 = (lane * M) >> 2;
    const uint16_t* sp = scales + row * G;
#pragma unroll
    for (int i = 0; i < LutCfg<M>::NS; ++i) {
        const int g = g0 + i;
        s[i] = (g < G) ? (uint32_t)__ldg(sp + g) : 0u;
    }
}

// Sum of one row over this lane's words (the caller then reduces the warp):
// table lookups, then the group scales, issuing `next` (the prefetch of a
// later row into the same registers) between the two.
template <int M, typename Next>
__device__ __forceinline__ float lut_row(uint32_t (&w)[M], uint32_t (&sv)[LutCfg<M>::NS], uint32_t lb, int o,
                                         Next&& next) {
    constexpr int NS = LutCfg<M>::NS;
    float ws[M];
    lut_words<M>(w, lb, ws, std::make_index_sequence<M>{});
    float sc[NS];
#pragma unroll
    for (int i = 0; i < NS; ++i) sc[i] = f16_bits_to_f32((uint16_t)sv[i]);
    next();
    float acc = 0.f;
    if constexpr (M % 4 == 0) {
#pragma unroll
        for (int q = 0; q < M / 4; ++q)
            acc = fmaf((ws[4 * q] + ws[4 * q + 1]) + (ws[4 * q + 2] + ws[4 * q + 3]), sc[q], acc);
    } else {
        float part = 0.f;
        float s0 = sc[0];
#pragma unroll
        for (int j = 0; j < M; ++j) {
            if (j > 0 && ((o + j) & 3) == 0) {
                acc = fmaf(part, s0, acc);
                part = 0.f;
#pragma unroll
                for (int i = 0; i + 1 < NS; ++i) sc[i] = sc[i + 1];
                s0 = sc[0];
            }
            part += ws[j];
        }
        acc = fmaf(part, s0, acc);
    }
    return warp_sum(acc);
}

// Tables of x (bf16 [1024 M]) into `tab`: for every nibble position p the 16
// sums T_p[e] = sum_{t<4} (bit t of e ? +x[4p+t] : -x[4p+t]); all threads of
// the CTA take part.  COHERENT reads x through L2 (ld.global.cg), for inputs
// that other CTAs of the same grid wrote.
template <int M, bool COHERENT>
__device__ __forceinline__ void lut_build(const uint16_t* x, float* tab) {
    constexpr int K = 1024 * M;
    for (int q = threadIdx.x; q < K / 4; q += blockDim.x) {
        const int l = q & 31, slot = q >> 5;            // consecutive threads -> consecutive banks
        const int p = l * 8 * M + slot;                 // nibble position within the row
        uint2 xv;
        if constexpr (COHERENT) xv = __ldcg(reinterpret_cast<const uint2*>(x + 4 * p));
        else xv = *reinterpret_cast<const uint2*>(x + 4 * p);
        const float x0 = bf16_bits_to_f32(xv.x & 0xffffu), x1 = bf16_bits_to_f32(xv.x >> 16);
        const float x2 = bf16_bits_to_f32(xv.y & 0xffffu), x3 = bf16_bits_to_f32(xv.y >> 16);
        const float a = x0 + x1, b = x0 - x1, c = x2 + x3, d = x2 - x3;
        const float lo[4] = {-a, b, -b, a};   // index bits (t0, t1) -> +-x0 +-x1
        const float hi[4] = {-c, d, -d, c};   // index bits (t2, t3) -> +-x2 +-x3
        float* tp = tab + (size_t)slot * 16 * 32 + l;
#pragma unroll
        for (int e = 0; e < 16; ++e) tp[e * 32] = lo[e & 3] + hi[e >> 2];
    }
}

}  // namespace bit1
