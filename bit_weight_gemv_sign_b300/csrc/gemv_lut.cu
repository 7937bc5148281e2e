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
#include "lut_common.cuh"

namespace bit1 {

template <int M, bool SWIGLU>
__global__ void __launch_bounds__(kLutThreads, 1)
k_gemv_lut(const uint8_t* __restrict__ bits, const uint16_t* __restrict__ scales,
           const uint16_t* __restrict__ x, int64_t N, void* __restrict__ y, int y_bf16) {
    using C = LutCfg<M>;
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
    lut_build<M, false>(x, tab);
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
    static bool configured = false;  // per-instantiation attribute (idempotent, benign race)
    const size_t smem = LutCfg<M>::smem;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute((const void*)k_gemv_lut<M, SWIGLU>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
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
