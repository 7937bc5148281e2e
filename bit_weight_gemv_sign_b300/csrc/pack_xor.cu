// Packing (fp weights -> sign bits + fp16 group scales) and the row-wise XOR
// sign-flip patch.
//
// Weight format: web page "Bonsai 27B: 노트북과 폰에서 실행되는 27B급 이진 및 삼진
// 저비트 LLM", section "이진(Binary) 가중치 형식": w = s_g * b, b in {-1,+1},
// one fp16 scale per 128 consecutive input weights.
// Patch: page "LocalLLaMA, true 1-bit LLM용 XOR patch 방식 \"Bankai\" 실험에
// 주목", section "LocalLLaMA가 본 핵심 포인트": listed rows have their binary
// weights flipped; the same XOR removes the patch.
#include <algorithm>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace bit1 {

// ---------------------------------------------------------------- pack
// One thread per (row, group).  The 128 magnitudes are summed in fp64 in
// ascending k order (the library's stated definition of the scale), the mean
// is rounded once to fp16 (round to nearest even, straight from fp64), and the
// sign bits bit = !(w < 0) are assembled into four little-endian words, which
// are exactly the 16 bytes of the group in the packed layout.
template <int DT>
__device__ __forceinline__ double load_weight(const void* w, int64_t i) {
    if (DT == BIT1_F32) return (double)__ldg(reinterpret_cast<const float*>(w) + i);
    uint16_t h = __ldg(reinterpret_cast<const unsigned short*>(w) + i);
    if (DT == BIT1_BF16) return (double)__uint_as_float((uint32_t)h << 16);
    return (double)__half2float(__ushort_as_half(h));
}

template <int DT>
__global__ void __launch_bounds__(256) k_pack(const void* __restrict__ w, int64_t N, int64_t K,
                                              uint8_t* __restrict__ bits,
                                              uint16_t* __restrict__ scales,
                                              uint32_t* __restrict__ flags) {
    const int64_t G = K / 128;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= N * G) return;
    const int64_t n = idx / G, g = idx - n * G;
    const int64_t base = n * K + g * 128;
    double sum = 0.0;
    uint32_t words[4] = {0u, 0u, 0u, 0u};
    bool nan_seen = false;
#pragma unroll 4
    for (int k = 0; k < 128; ++k) {
        const double v = load_weight<DT>(w, base + k);
        nan_seen |= (v != v);
        if (!(v < 0.0)) words[k >> 5] |= 1u << (k & 31);
        sum = __dadd_rn(sum, fabs(v));  // no contraction: plain sequential fp64 sum
    }
    const double mean = sum * 0.0078125;  // /128, exact
    const __half h = __double2half(mean); // single rounding fp64 -> fp16, nearest even
    const uint16_t hb = __half_as_ushort(h);
    uint4 out;
    out.x = words[0]; out.y = words[1]; out.z = words[2]; out.w = words[3];
    *reinterpret_cast<uint4*>(bits + n * (K / 8) + g * 16) = out;
    scales[idx] = hb;
    if (flags) {
        if (nan_seen) atomicOr(flags, 1u);
        if ((hb & 0x7c00u) == 0x7c00u) atomicOr(flags, 2u);
    }
}

cudaError_t launch_pack(const void* w, int dtype, int64_t N, int64_t K, uint8_t* bits,
                        uint16_t* scales, uint32_t* flags, cudaStream_t stream) {
    if (flags) {
        cudaError_t e = cudaMemsetAsync(flags, 0, sizeof(uint32_t), stream);
        if (e != cudaSuccess) return e;
    }
    const int64_t units = N * (K / 128);
    const int threads = 256;
    const int64_t blocks = (units + threads - 1) / threads;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    switch (dtype) {
        case BIT1_F32: k_pack<BIT1_F32><<<(unsigned)blocks, threads, 0, stream>>>(w, N, K, bits, scales, flags); break;
        case BIT1_BF16: k_pack<BIT1_BF16><<<(unsigned)blocks, threads, 0, stream>>>(w, N, K, bits, scales, flags); break;
        default: k_pack<BIT1_F16><<<(unsigned)blocks, threads, 0, stream>>>(w, N, K, bits, scales, flags); break;
    }
    return cudaGetLastError();
}

// ---------------------------------------------------------------- XOR patch
// The row list travels in the kernel's parameter block (no device copy, no
// allocation).  Rows inside one launch are distinct (the host reduces the
// list to the rows listed an odd number of times), so plain XOR stores never
// race.  Grid: x = 16-byte chunks of a row, y = list entry.
constexpr int kXorRowsPerLaunch = 900;  // 3.6 KB of parameters

struct XorRows {
    int32_t count;
    int32_t rows[kXorRowsPerLaunch];
};

__global__ void __launch_bounds__(256) k_xor_patch(uint8_t* __restrict__ bits, int64_t row_bytes,
                                                   const __grid_constant__ XorRows list) {
    const int entry = blockIdx.y;
    if (entry >= list.count) return;
    const int64_t chunk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // 16-byte chunk
    if (chunk * 16 >= row_bytes) return;
    uint4* p = reinterpret_cast<uint4*>(bits + (int64_t)list.rows[entry] * row_bytes) + chunk;
    uint4 v = *p;
    v.x = ~v.x; v.y = ~v.y; v.z = ~v.z; v.w = ~v.w;
    *p = v;
}

cudaError_t launch_xor_patch(uint8_t* bits, int64_t N, int64_t K, const int32_t* rows,
                             int64_t n_rows, cudaStream_t stream) {
    // Keep the rows listed an odd number of times (pairs cancel), sorted.
    std::vector<int32_t> r(rows, rows + n_rows);
    std::sort(r.begin(), r.end());
    std::vector<int32_t> odd;
    for (size_t i = 0; i < r.size();) {
        size_t j = i;
        while (j < r.size() && r[j] == r[i]) ++j;
        if ((j - i) & 1) odd.push_back(r[i]);
        i = j;
    }
    (void)N;
    const int64_t row_bytes = K / 8;
    const int64_t chunks = row_bytes / 16;
    const int threads = 256;
    const unsigned gx = (unsigned)((chunks + threads - 1) / threads);
    for (size_t off = 0; off < odd.size(); off += kXorRowsPerLaunch) {
        XorRows list;
        list.count = (int32_t)std::min<size_t>(kXorRowsPerLaunch, odd.size() - off);
        for (int i = 0; i < list.count; ++i) list.rows[i] = odd[off + i];
        k_xor_patch<<<dim3(gx, (unsigned)list.count), threads, 0, stream>>>(bits, row_bytes, list);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace bit1
