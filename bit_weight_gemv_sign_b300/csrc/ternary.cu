// Ternary weights in 2-bit slots.
//
// Format: web page "Bonsai 27B: 노트북과 폰에서 실행되는 27B급 이진 및 삼진 저비트
// LLM", section "삼진(Ternary) 가중치 형식": w = s_g * t, t in {-1, 0, +1}, one
// fp16 scale per 128 consecutive input weights; section "저장 공간과 실제 배포
// 크기": today's kernels keep one ternary value in a 2-bit slot.  The slot is
// read here as two sign planes a, b in the binary layout (bit 1 -> +1) with
// t = (a + b) / 2, so a ternary product is the mean of two binary products
// that share the scales and the activations:
//     y = ( sum_g s_g sum_k a_k x_k  +  sum_g s_g sum_k b_k x_k ) / 2.
// The binary kernels compute both halves into fp32 scratch; k_ternary_combine
// forms the mean and the output type (k_ternary_combine_swiglu: the means of
// a gate/up pair and h = silu(g) * u).
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace bit1 {

// ---------------------------------------------------------------- codes -> planes
// One thread per 32 consecutive codes of a row (one little-endian 32-bit word
// of each plane): a = (t >= 0), b = (t > 0).  A code outside {-1, 0, +1} sets
// bit 2 of *flags; its bits are then unspecified.
__global__ void __launch_bounds__(256) k_ternary_planes(const int8_t* __restrict__ codes, int64_t words,
                                                        uint32_t* __restrict__ pa, uint32_t* __restrict__ pb,
                                                        uint32_t* __restrict__ flags) {
    bool bad = false;
    for (int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; w < words;
         w += (int64_t)gridDim.x * blockDim.x) {
        const uint4* src = reinterpret_cast<const uint4*>(codes + 32 * w);
        uint32_t q[8];
        uint4 lo = __ldg(src), hi = __ldg(src + 1);
        q[0] = lo.x; q[1] = lo.y; q[2] = lo.z; q[3] = lo.w;
        q[4] = hi.x; q[5] = hi.y; q[6] = hi.z; q[7] = hi.w;
        uint32_t a = 0, b = 0;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int v = (int8_t)(q[j >> 2] >> (8 * (j & 3)));
            bad |= (v < -1) | (v > 1);
            a |= (uint32_t)(v >= 0) << j;
            b |= (uint32_t)(v > 0) << j;
        }
        pa[w] = a;
        pb[w] = b;
    }
    if (bad && flags) atomicOr(flags, 4u);
}

cudaError_t launch_ternary_planes(const int8_t* codes, int64_t N, int64_t K, uint8_t* a, uint8_t* b,
                                  uint32_t* flags, cudaStream_t stream) {
    if (flags) {
        cudaError_t e = cudaMemsetAsync(flags, 0, sizeof(uint32_t), stream);
        if (e != cudaSuccess) return e;
    }
    const int64_t words = N * (K / 32);
    const int threads = 256;
    const int64_t want = (words + threads - 1) / threads;
    const unsigned blocks = (unsigned)std::min<int64_t>(want, (int64_t)sm_count() * 16);
    k_ternary_planes<<<blocks, threads, 0, stream>>>(codes, words, reinterpret_cast<uint32_t*>(a),
                                                     reinterpret_cast<uint32_t*>(b), flags);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- combine
// y[i] = (ya[i] + yb[i]) / 2 in fp32 (the halving is exact), then the output
// type (bf16: round to nearest even).  Four elements per thread step.
template <bool BF16>
__global__ void __launch_bounds__(256) k_ternary_combine(const float* __restrict__ ya,
                                                         const float* __restrict__ yb, int64_t n,
                                                         void* __restrict__ y) {
    const int64_t quads = n / 4;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < quads; i += stride) {
        const float4 u = __ldg(reinterpret_cast<const float4*>(ya) + i);
        const float4 v = __ldg(reinterpret_cast<const float4*>(yb) + i);
        const float r0 = 0.5f * (u.x + v.x), r1 = 0.5f * (u.y + v.y);
        const float r2 = 0.5f * (u.z + v.z), r3 = 0.5f * (u.w + v.w);
        if (BF16) {
            uint2 o;
            o.x = (uint32_t)f32_to_bf16_bits(r0) | ((uint32_t)f32_to_bf16_bits(r1) << 16);
            o.y = (uint32_t)f32_to_bf16_bits(r2) | ((uint32_t)f32_to_bf16_bits(r3) << 16);
            reinterpret_cast<uint2*>(y)[i] = o;
        } else {
            reinterpret_cast<float4*>(y)[i] = make_float4(r0, r1, r2, r3);
        }
    }
    for (int64_t i = 4 * quads + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const float r = 0.5f * (ya[i] + yb[i]);
        if (BF16)
            reinterpret_cast<uint16_t*>(y)[i] = f32_to_bf16_bits(r);
        else
            reinterpret_cast<float*>(y)[i] = r;
    }
}

// SwiGLU pairs (rows interleaved as gate, up; the Bonsai 27B page, section
// "Bonsai 27B의 표현 방식": the base model's MLP is SwiGLU): element 2i of the
// flat [B][N] halves is a gate, 2i+1 its up (N even, so pairs never cross batch
// rows); y[i] = silu(g) * u with g, u the two means.
template <bool BF16>
__global__ void __launch_bounds__(256) k_ternary_combine_swiglu(const float2* __restrict__ ya,
                                                                const float2* __restrict__ yb, int64_t pairs,
                                                                void* __restrict__ y) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < pairs; i += stride) {
        const float2 u = __ldg(ya + i), v = __ldg(yb + i);
        const float g = 0.5f * (u.x + v.x), up = 0.5f * (u.y + v.y);
        const float h = g / (1.f + expf(-g)) * up;
        if (BF16)
            reinterpret_cast<uint16_t*>(y)[i] = f32_to_bf16_bits(h);
        else
            reinterpret_cast<float*>(y)[i] = h;
    }
}

cudaError_t launch_ternary_combine(const float* ya, const float* yb, int64_t n, void* y, bool y_bf16,
                                   cudaStream_t stream, bool swiglu) {
    const int threads = 256;
    if (swiglu) {
        const int64_t pairs = n / 2;
        const int64_t want = (pairs + threads - 1) / threads;
        const unsigned blocks = (unsigned)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)sm_count() * 8));
        const float2* a2 = reinterpret_cast<const float2*>(ya);
        const float2* b2 = reinterpret_cast<const float2*>(yb);
        if (y_bf16)
            k_ternary_combine_swiglu<true><<<blocks, threads, 0, stream>>>(a2, b2, pairs, y);
        else
            k_ternary_combine_swiglu<false><<<blocks, threads, 0, stream>>>(a2, b2, pairs, y);
        return cudaGetLastError();
    }
    const int64_t want = (n / 4 + threads) / threads;
    const unsigned blocks = (unsigned)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)sm_count() * 8));
    if (y_bf16)
        k_ternary_combine<true><<<blocks, threads, 0, stream>>>(ya, yb, n, y);
    else
        k_ternary_combine<false><<<blocks, threads, 0, stream>>>(ya, yb, n, y);
    return cudaGetLastError();
}

}  // namespace bit1
