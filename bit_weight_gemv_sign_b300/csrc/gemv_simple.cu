// Reference-quality GEMV over packed sign bits: any B >= 1, any K multiple of
// 128.  One warp per output row; lane l takes groups l, l+32, ... of the row;
// per group it loads the 16 sign bytes (one 128-bit load) and the fp16 scale,
// adds or subtracts each activation by its bit, multiplies the group's fp32
// partial sum by the scale, and the warp reduces the row with shuffles.
//
// Product definition: web page "Bonsai 27B: 노트북과 폰에서 실행되는 27B급 이진
// 및 삼진 저비트 LLM", sections "이진(Binary) 가중치 형식" (w = s_g * b) and
// "하이브리드 어텐션을 위한 저비트 커널" (scale applied inside the product,
// high-precision accumulation).
#include "common.cuh"
#include "internal.h"

namespace bit1 {

constexpr int kSimpleBatch = 4;  // batch rows per pass over the weights

__global__ void __launch_bounds__(256) k_gemv_simple(const uint8_t* __restrict__ bits,
                                                     const uint16_t* __restrict__ scales,
                                                     const uint16_t* __restrict__ x,
                                                     int64_t B, int64_t N, int64_t K,
                                                     void* __restrict__ y, int y_bf16) {
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    pdl_wait();
    pdl_launch_dependents();
    if (row >= N) return;
    const int64_t G = K / 128;
    const uint8_t* rbits = bits + row * (K / 8);
    for (int64_t b0 = 0; b0 < B; b0 += kSimpleBatch) {
        float acc[kSimpleBatch];
#pragma unroll
        for (int i = 0; i < kSimpleBatch; ++i) acc[i] = 0.f;
        for (int64_t g = lane; g < G; g += 32) {
            const uint4 wv = *reinterpret_cast<const uint4*>(rbits + g * 16);
            const uint32_t wq[4] = {wv.x, wv.y, wv.z, wv.w};
            const float s = f16_bits_to_f32(scales[row * G + g]);
#pragma unroll
            for (int i = 0; i < kSimpleBatch; ++i) {
                const int64_t b = b0 + i;
                if (b >= B) break;
                const uint16_t* xg = x + b * K + g * 128;
                float part = 0.f;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
#pragma unroll 8
                    for (int t = 0; t < 32; ++t) {
                        const float xv = bf16_bits_to_f32(__ldg(xg + q * 32 + t));
                        part += ((wq[q] >> t) & 1u) ? xv : -xv;
                    }
                }
                acc[i] = fmaf(s, part, acc[i]);
            }
        }
#pragma unroll
        for (int i = 0; i < kSimpleBatch; ++i) {
            const int64_t b = b0 + i;
            const float v = warp_sum(acc[i]);
            if (lane == 0 && b < B) {
                if (y_bf16)
                    reinterpret_cast<uint16_t*>(y)[b * N + row] = f32_to_bf16_bits(v);
                else
                    reinterpret_cast<float*>(y)[b * N + row] = v;
            }
        }
    }
}

cudaError_t launch_gemv_simple(const GemvArgs& a) {
    const int warps = 8;
    const int64_t blocks = (a.N + warps - 1) / warps;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    const uint8_t* bits = a.bits;
    const uint16_t* scales = a.scales;
    const uint16_t* x = a.x;
    int64_t B = a.B, N = a.N, K = a.K;
    void* y = a.y;
    int yb = a.y_bf16;
    void* args[] = {&bits, &scales, &x, &B, &N, &K, &y, &yb};
    return launch((const void*)k_gemv_simple, dim3((unsigned)blocks), dim3(warps * 32), 0, a.stream,
                  a.pdl, args);
}

}  // namespace bit1
