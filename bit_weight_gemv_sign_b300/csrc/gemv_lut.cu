// Batch-1 GEMV over packed sign bits by table lookup (CUDA cores, sm_103a).
//
// What it computes: y[n] = sum_g s[n][g] * sum_{k in g} (bit(n,k) ? x[k] : -x[k]),
// the binary weight format of the web page "Bonsai 27B: 노트북과 폰에서 실행되는
// 27B급 이진 및 삼진 저비트 LLM" (section "이진(Binary) 가중치 형식"), with the
// group scale applied inside the product and fp32 accumulation (section
// "하이브리드 어텐션을 위한 저비트 커널").  No multiply per weight: every
// four weights cost one table lookup and one add (the multiply-free property
// of ±1 weights, page "PrismML Bonsai — 1.15GB짜리 8B 모델이 말이 되나?",
// section "1-bit이 뭔지부터").
//
// Design:
//  * K = 1024*M.  Lane l of every warp owns the M consecutive 32-bit words
//    [l*M, l*M+M) of each row, i.e. nibble positions [8*M*l, 8*M*l + 8*M).
//  * For every nibble position p the CTA builds, once, the 16 sums
//    T_p[e] = sum_{t<4} (bit t of e ? +x[4p+t] : -x[4p+t]) in fp32 shared
//    memory.  T_p lives entirely in bank (p / 8M) = the owning lane, entry e at
//    word ((slot*16 + e)*32 + lane), slot = p % 8M: all 32 lanes of a warp
//    always hit 32 different banks, whatever their nibble values.
//  * A word of weights (32 weights, 8 nibbles) costs 8 x (shift, mask|or,
//    LDS, FADD).  The lane's group partial sums are multiplied by the fp16
//    scale once per group and the row is reduced with warp shuffles.
//  * One CTA per SM; each CTA takes a contiguous block of rows; warps
//    interleave over its rows with a D-deep register prefetch of the next
//    rows' bits and scales, issued before griddepcontrol.wait so that under
//    programmatic dependent launch the weight stream starts while the previous
//    kernel finishes.
//  * SwiGLU epilogue (rows interleaved as gate/up pairs of a SwiGLU MLP, the
//    base model's MLP on the Bonsai 27B page, section "Bonsai 27B의 표현
//    방식"): CTAs and warps take whole pairs, a warp runs a pair's gate row
//    then its up row, keeps the gate sum and writes h = silu(g) * u.
#include <utility>

#include "common.cuh"
#include "internal.h"

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

template <int M, bool SWIGLU>
__global__ void __launch_bounds__(kLutThreads, 1)
k_gemv_lut(const uint8_t* __restrict__ bits, const uint16_t* __restrict__ scales,
           const uint16_t* __restrict__ x, int64_t N, void* __restrict__ y, int y_bf16) {
    using C = LutCfg<M>;
    constexpr int K = 1024 * M;
    constexpr int D = C::D, NS = C::NS;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t sraw = (uint32_t)__cvta_generic_to_shared(smem_raw);
    const uint32_t tbase = (sraw + 2047u) & ~2047u;
    float* tab = reinterpret_cast<float*>(smem_raw + (tbase - sraw));

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    // Units: rows, or (gate, up) row pairs with the SwiGLU epilogue.  The
    // CTA takes units [n0, n1); this warp units n0 + warp + j * nw.  With
    // pairs its t-th row is row t & 1 of its unit t >> 1.
    const int64_t U = SWIGLU ? N / 2 : N;
    const int64_t n0 = U * blockIdx.x / gridDim.x, n1 = U * (blockIdx.x + 1) / gridDim.x;
    const int64_t mine = n1 - n0 > warp ? (n1 - n0 - warp + nw - 1) / nw : 0;
    auto pair_row = [&](int64_t t) -> int64_t { return 2 * (n0 + warp + (t >> 1) * nw) + (t & 1); };

    uint32_t wb[D][M];
    uint32_t sb[D][NS];
#pragma unroll
    for (int d = 0; d < D; ++d) {
        if constexpr (SWIGLU) {
            if (d < 2 * mine) load_row<M>(bits, scales, pair_row(d), lane, wb[d], sb[d]);
        } else {
            const int64_t row = n0 + warp + (int64_t)d * nw;
            if (row < n1) load_row<M>(bits, scales, row, lane, wb[d], sb[d]);
        }
    }

    // x is produced by the preceding kernel in a decode step: wait for it here,
    // after the weight prefetch is in flight.
    pdl_wait();
    for (int q = threadIdx.x; q < K / 4; q += blockDim.x) {
        const int l = q & 31, slot = q >> 5;            // consecutive threads -> consecutive banks
        const int p = l * 8 * M + slot;                 // nibble position within the row
        const uint2 xv = *reinterpret_cast<const uint2*>(x + 4 * p);
        const float x0 = bf16_bits_to_f32(xv.x & 0xffffu), x1 = bf16_bits_to_f32(xv.x >> 16);
        const float x2 = bf16_bits_to_f32(xv.y & 0xffffu), x3 = bf16_bits_to_f32(xv.y >> 16);
        const float a = x0 + x1, b = x0 - x1, c = x2 + x3, d = x2 - x3;
        const float lo[4] = {-a, b, -b, a};   // index bits (t0, t1) -> +-x0 +-x1
        const float hi[4] = {-c, d, -d, c};   // index bits (t2, t3) -> +-x2 +-x3
        float* tp = tab + (size_t)slot * 16 * 32 + l;
#pragma unroll
        for (int e = 0; e < 16; ++e) tp[e * 32] = lo[e & 3] + hi[e >> 2];
    }
    __syncthreads();
    pdl_launch_dependents();

    const uint32_t lb = tbase + 4u * (uint32_t)lane;
    const int o = (M % 4 == 0) ? 0 : ((lane * M) & 3);  // offset of the lane's first word in its group
    if constexpr (SWIGLU) {
        // Gate row then up row of each pair; h = silu(g) * u from the kept gate sum.
        const int64_t R = 2 * mine;
        float gate = 0.f;
        for (int64_t base = 0; base < R; base += D) {
#pragma unroll
            for (int d = 0; d < D; ++d) {
                const int64_t t = base + d;
                if (t >= R) break;
                const float acc = lut_row<M>(wb[d], sb[d], lb, o, [&] {
                    if (t + D < R) load_row<M>(bits, scales, pair_row(t + D), lane, wb[d], sb[d]);
                });
                if (!(t & 1)) {
                    gate = acc;
                    continue;
                }
                const float h = gate / (1.f + expf(-gate)) * acc;
                const int64_t u = pair_row(t) >> 1;
                if (lane == 0) {
                    if (y_bf16)
                        reinterpret_cast<uint16_t*>(y)[u] = f32_to_bf16_bits(h);
                    else
                        reinterpret_cast<float*>(y)[u] = h;
                }
            }
        }
    } else {
        for (int64_t base = n0 + warp; base < n1; base += (int64_t)D * nw) {
#pragma unroll
            for (int d = 0; d < D; ++d) {
                const int64_t row = base + (int64_t)d * nw;
                if (row >= n1) break;
                const float acc = lut_row<M>(wb[d], sb[d], lb, o, [&] {
                    const int64_t nrow = row + (int64_t)D * nw;
                    if (nrow < n1) load_row<M>(bits, scales, nrow, lane, wb[d], sb[d]);
                });
                if (lane == 0) {
                    if (y_bf16)
                        reinterpret_cast<uint16_t*>(y)[row] = f32_to_bf16_bits(acc);
                    else
                        reinterpret_cast<float*>(y)[row] = acc;
                }
            }
        }
    }
}

template <int M, bool SWIGLU>
static cudaError_t launch_lut_ms(const GemvArgs& a) {
    const size_t smem = LutCfg<M>::smem;
    const cudaError_t e = func_attrs((const void*)k_gemv_lut<M, SWIGLU>, (int)smem, false);
    if (e != cudaSuccess) return e;
    const int sms = sm_count();
    const int64_t units = a.swiglu ? a.N / 2 : a.N;
    const int64_t grid = units < sms ? units : sms;
    const uint8_t* bits = a.bits;
    const uint16_t* scales = a.scales;
    const uint16_t* x = a.x;
    int64_t N = a.N;
    void* y = a.y;
    int yb = a.y_bf16;
    void* args[] = {&bits, &scales, &x, &N, &y, &yb};
    return launch((const void*)k_gemv_lut<M, SWIGLU>, dim3((unsigned)grid), dim3(kLutThreads), smem,
                  a.stream, a.pdl, args);
}

template <int M>
static cudaError_t launch_lut_m(const GemvArgs& a) {
    return a.swiglu ? launch_lut_ms<M, true>(a) : launch_lut_ms<M, false>(a);
}

bool lut_supported(int64_t B, int64_t N, int64_t K) {
    return B == 1 && N >= 1 && K % 1024 == 0 && K / 1024 >= 1 && K / 1024 <= kLutMaxM;
}

cudaError_t launch_gemv_lut(const GemvArgs& a) {
    if (!lut_supported(a.B, a.N, a.K)) return cudaErrorNotSupported;
    switch (a.K / 1024) {
        case 1: return launch_lut_m<1>(a);
        case 2: return launch_lut_m<2>(a);
        case 3: return launch_lut_m<3>(a);
        case 4: return launch_lut_m<4>(a);
        case 5: return launch_lut_m<5>(a);
        case 6: return launch_lut_m<6>(a);
        case 7: return launch_lut_m<7>(a);
        case 8: return launch_lut_m<8>(a);
        case 9: return launch_lut_m<9>(a);
        case 10: return launch_lut_m<10>(a);
        case 11: return launch_lut_m<11>(a);
        case 12: return launch_lut_m<12>(a);
        case 13: return launch_lut_m<13>(a);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace bit1
