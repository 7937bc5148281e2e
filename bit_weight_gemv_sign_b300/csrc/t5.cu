// Ternary codes packed five per byte (1.75 bits/weight with the fp16 scales).
//
// Format: web page "Bonsai 27B: 노트북과 폰에서 실행되는 27B급 이진 및 삼진 저비트
// LLM", section "삼진(Ternary) 가중치 형식" (w = s_g * t, t in {-1, 0, +1}, one
// fp16 scale per 128 weights, ideal cost log2(3) + 16/128 bits); section "저장
// 공간과 실제 배포 크기": 2-bit slots exceed that minimum until native ternary
// kernels exist.  This library's packing: each group of 128 codes of a row is
// 26 bytes; byte j < 25 holds codes 5j .. 5j+4 and byte 25 codes 125 .. 127,
// each byte the base-3 number v = sum_i (t_i + 1) 3^i, lowest k first.
//
// Three kernels:
//  * k_t5_pack      codes -> bytes (one thread per output byte);
//  * k_t5_planes    bytes -> the two sign planes of the 2-bit-slot layout
//                   (a = t >= 0, b = t > 0), so that a matrix kept in the
//                   compact packing runs on the slot kernels;
//  * k_gemv_t5      the product straight from the bytes for the shapes the
//                   batch-1 table kernel (t5lut.cu) does not take: one warp
//                   per row, lanes over the row's bytes, a 256-entry shared
//                   table that turns a byte into its five digits, fp32
//                   accumulation, up to 8 batch rows per launch.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace bit1 {

namespace {

// Digits of byte v (v < 243) as five 2-bit fields d_i = t_i + 1; bytes 243 ..
// 255 are not codes: bit 15 marks them.
__device__ __forceinline__ uint32_t t5_digits(uint32_t v) {
    if (v > 242u) return 0x8000u;
    uint32_t r = 0;
#pragma unroll
    for (int i = 0; i < 5; ++i) {
        r |= (v % 3u) << (2 * i);
        v /= 3u;
    }
    return r;
}

}  // namespace

// ---------------------------------------------------------------- codes -> bytes
__global__ void __launch_bounds__(256) k_t5_pack(const int8_t* __restrict__ codes, int64_t K, int64_t total,
                                                 uint8_t* __restrict__ out, uint32_t* __restrict__ flags) {
    bool bad = false;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t grp = i / 26, j = i - grp * 26;
        const int64_t G = K / 128, n = grp / G, g = grp - n * G;
        const int8_t* c = codes + n * K + 128 * g + 5 * j;
        const int nd = j < 25 ? 5 : 3;
        uint32_t v = 0, p = 1;
        for (int d = 0; d < nd; ++d) {
            const int t = c[d];
            bad |= (t < -1) | (t > 1);
            v += (uint32_t)(t + 1) * p;
            p *= 3u;
        }
        out[i] = (uint8_t)v;
    }
    if (bad && flags) atomicOr(flags, 4u);
}

// ---------------------------------------------------------------- bytes -> planes
// One thread per (row, group): 26 bytes in, 16 bytes of each plane out.
__global__ void __launch_bounds__(256) k_t5_planes(const uint8_t* __restrict__ packed, int64_t groups,
                                                   uint4* __restrict__ pa, uint4* __restrict__ pb,
                                                   uint32_t* __restrict__ flags) {
    __shared__ uint16_t dig[256];
    for (int v = threadIdx.x; v < 256; v += blockDim.x) dig[v] = (uint16_t)t5_digits((uint32_t)v);
    __syncthreads();
    bool bad = false;
    for (int64_t gi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; gi < groups;
         gi += (int64_t)gridDim.x * blockDim.x) {
        const uint8_t* src = packed + gi * 26;
        uint32_t a[4] = {0, 0, 0, 0}, b[4] = {0, 0, 0, 0};
#pragma unroll
        for (int j = 0; j < 26; ++j) {
            const uint32_t v = src[j];
            const uint32_t d = dig[v];
            const int nd = j < 25 ? 5 : 3;
            bad |= (d & 0x8000u) != 0 || (j == 25 && v > 26u);
#pragma unroll
            for (int i = 0; i < nd; ++i) {
                const int k = 5 * j + i;
                const uint32_t di = (d >> (2 * i)) & 3u;   // t + 1
                a[k >> 5] |= (uint32_t)(di >= 1u) << (k & 31);
                b[k >> 5] |= (uint32_t)(di == 2u) << (k & 31);
            }
        }
        pa[gi] = make_uint4(a[0], a[1], a[2], a[3]);
        pb[gi] = make_uint4(b[0], b[1], b[2], b[3]);
    }
    if (bad && flags) atomicOr(flags, 8u);
}

// ---------------------------------------------------------------- direct product
// Warp w of the grid takes rows w, w + warps, ...; lane l takes bytes l, l+32,
// ... of the row (G*26 bytes).  For each byte it reads the digits from the
// shared table, adds the five +-x / 0 terms in fp32, multiplies the byte's
// partial by its group scale and accumulates; the lanes' sums are added by a
// butterfly.  Up to 8 batch rows per launch share each decoded byte.
template <int NB>
__global__ void __launch_bounds__(256) k_gemv_t5(const uint8_t* __restrict__ packed,
                                                 const uint16_t* __restrict__ scales,
                                                 const uint16_t* __restrict__ x, int64_t N, int64_t K,
                                                 void* __restrict__ y, int64_t ystride, int y_bf16) {
    __shared__ uint16_t dig[256];
    for (int v = threadIdx.x; v < 256; v += blockDim.x) dig[v] = (uint16_t)(t5_digits((uint32_t)v) & 0x3ffu);
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t G = K / 128, row_bytes = G * 26;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t n = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); n < N; n += warps) {
        const uint8_t* prow = packed + n * row_bytes;
        float acc[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) acc[b] = 0.f;
        for (int64_t j = lane; j < row_bytes; j += 32) {
            const int64_t g = j / 26, jj = j - g * 26;
            const uint32_t d = dig[__ldg(prow + j)];
            const float s = f16_bits_to_f32(__ldg(scales + n * G + g));
            const int64_t k0 = 128 * g + 5 * jj;
            const int nd = jj < 25 ? 5 : 3;
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const uint16_t* xb = x + (int64_t)b * K + k0;
                float part = 0.f;
                for (int i = 0; i < nd; ++i) {
                    const uint32_t di = (d >> (2 * i)) & 3u;
                    const float xv = bf16_bits_to_f32(__ldg(xb + i));
                    part += di == 2u ? xv : (di == 0u ? -xv : 0.f);
                }
                acc[b] = fmaf(s, part, acc[b]);
            }
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const float v = warp_sum(acc[b]);
            if (lane == 0) {
                if (y_bf16) reinterpret_cast<uint16_t*>(y)[b * ystride + n] = f32_to_bf16_bits(v);
                else reinterpret_cast<float*>(y)[b * ystride + n] = v;
            }
        }
    }
}

namespace {

unsigned grid_for(int64_t items, int threads, int per_sm) {
    const int64_t want = (items + threads - 1) / threads;
    return (unsigned)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)sm_count() * per_sm));
}

}  // namespace

cudaError_t launch_t5_pack(const int8_t* codes, int64_t N, int64_t K, uint8_t* out, uint32_t* flags,
                           cudaStream_t stream) {
    if (flags) {
        cudaError_t e = cudaMemsetAsync(flags, 0, sizeof(uint32_t), stream);
        if (e != cudaSuccess) return e;
    }
    const int64_t total = N * (K / 128) * 26;
    k_t5_pack<<<grid_for(total, 256, 16), 256, 0, stream>>>(codes, K, total, out, flags);
    return cudaGetLastError();
}

cudaError_t launch_t5_planes(const uint8_t* packed, int64_t N, int64_t K, uint8_t* a, uint8_t* b,
                             uint32_t* flags, cudaStream_t stream) {
    if (flags) {
        cudaError_t e = cudaMemsetAsync(flags, 0, sizeof(uint32_t), stream);
        if (e != cudaSuccess) return e;
    }
    const int64_t groups = N * (K / 128);
    k_t5_planes<<<grid_for(groups, 256, 16), 256, 0, stream>>>(packed, groups, reinterpret_cast<uint4*>(a),
                                                               reinterpret_cast<uint4*>(b), flags);
    return cudaGetLastError();
}

cudaError_t launch_gemv_t5(const uint8_t* packed, const uint16_t* scales, const uint16_t* x, int64_t B,
                           int64_t N, int64_t K, void* y, bool y_bf16, cudaStream_t stream) {
    const int threads = 256;
    const unsigned blocks = grid_for(N * 32, threads, 8);
    const size_t ysz = y_bf16 ? 2 : 4;
    for (int64_t b0 = 0; b0 < B; b0 += 8) {
        const int nb = (int)std::min<int64_t>(8, B - b0);
        const uint16_t* xb = x + b0 * K;
        void* yb = static_cast<uint8_t*>(y) + b0 * N * ysz;
        switch (nb) {
            case 1: k_gemv_t5<1><<<blocks, threads, 0, stream>>>(packed, scales, xb, N, K, yb, N, y_bf16); break;
            case 2: k_gemv_t5<2><<<blocks, threads, 0, stream>>>(packed, scales, xb, N, K, yb, N, y_bf16); break;
            case 3: k_gemv_t5<3><<<blocks, threads, 0, stream>>>(packed, scales, xb, N, K, yb, N, y_bf16); break;
            case 4: k_gemv_t5<4><<<blocks, threads, 0, stream>>>(packed, scales, xb, N, K, yb, N, y_bf16); break;
            case 5: k_gemv_t5<5><<<blocks, threads, 0, stream>>>(packed, scales, xb, N, K, yb, N, y_bf16); break;
            case 6: k_gemv_t5<6><<<blocks, threads, 0, stream>>>(packed, scales, xb, N, K, yb, N, y_bf16); break;
            case 7: k_gemv_t5<7><<<blocks, threads, 0, stream>>>(packed, scales, xb, N, K, yb, N, y_bf16); break;
            default: k_gemv_t5<8><<<blocks, threads, 0, stream>>>(packed, scales, xb, N, K, yb, N, y_bf16); break;
        }
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

int t5_launch_count(int64_t B) { return (int)((B + 7) / 8); }

}  // namespace bit1
