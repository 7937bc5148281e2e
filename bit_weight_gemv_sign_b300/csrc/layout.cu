// Conversion of packed sign bits between the canonical layout and the g128x
// layout that the grouped kernels can read (t6_common.cuh describes both).
// A within-group permutation: every row keeps its own bits, so the row-wise
// XOR patch of the web page "LocalLLaMA, true 1-bit LLM용 XOR patch 방식
// "Bankai" 실험에 주목" (section "LocalLLaMA가 본 핵심 포인트") flips exactly
// the same rows in either layout, and the scales are unchanged.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace bit1 {
namespace {

// Bit of the 128-bit group (word k / 32 of four, bit k % 32) holding input k
// of the group in the g128x layout.
__host__ __device__ constexpr int g128x_bit(int k) {
    if (k < 72) return 8 * (k / 6) + 1 + k % 6;               // fields 0..11: bits 1-6 of bytes 0..11
    if (k < 96) {                                              // fields 12..15: bits 0 and 7 of those bytes
        const int j = (k - 72) / 6, i = (k - 72) % 6;
        const int byte = (i % 2 == 0) ? j : (j + 1) % 4;
        return 32 * (i / 2) + 8 * byte + ((i % 2 == 0) ? 7 : 0);
    }
    return k;                                                  // word 3 as in the canonical layout
}

// dir 0: canonical -> g128x (input k moves from bit k to bit g128x_bit(k));
// dir 1: the inverse.  One thread per 16-byte group; in place is allowed.
template <int DIR>
__global__ void __launch_bounds__(256) k_relayout(const uint4* in, uint4* out, int64_t groups) {
    for (int64_t gi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; gi < groups;
         gi += (int64_t)gridDim.x * blockDim.x) {
        const uint4 v = in[gi];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int k = 0; k < 128; ++k) {
            const int src = DIR == 0 ? k : g128x_bit(k);
            const int dst = DIR == 0 ? g128x_bit(k) : k;
            o[dst >> 5] |= ((w[src >> 5] >> (src & 31)) & 1u) << (dst & 31);
        }
        out[gi] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

}  // namespace

cudaError_t launch_relayout(const uint8_t* in, uint8_t* out, int64_t N, int64_t K, bool to_g128x,
                            cudaStream_t stream) {
    const int64_t groups = N * (K / 128);
    const int threads = 256;
    const int64_t want = (groups + threads - 1) / threads;
    const unsigned grid = (unsigned)std::min<int64_t>(want, (int64_t)sm_count() * 16);
    const uint4* i4 = reinterpret_cast<const uint4*>(in);
    uint4* o4 = reinterpret_cast<uint4*>(out);
    if (to_g128x) k_relayout<0><<<grid, threads, 0, stream>>>(i4, o4, groups);
    else k_relayout<1><<<grid, threads, 0, stream>>>(i4, o4, groups);
    return cudaGetLastError();
}

}  // namespace bit1
