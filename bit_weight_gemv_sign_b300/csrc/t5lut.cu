// Batch-1 product straight from ternary codes packed five per byte, by table
// lookup (CUDA cores, sm_103a).
//
// Format: web page "Bonsai 27B: 노트북과 폰에서 실행되는 27B급 이진 및 삼진 저비트
// LLM", section "삼진(Ternary) 가중치 형식" (w = s_g * t, t in {-1, 0, +1}, one
// fp16 scale per 128 weights); this library's five-per-byte packing (26 bytes
// per group of 128 codes; byte j < 25 holds codes 5j .. 5j+4, byte 25 codes
// 125 .. 127, v = sum_i (t_i + 1) 3^i).  Section "저장 공간과 실제 배포 크기"
// notes that native ternary kernels are still to come; this is one.
//
// Method: a byte v splits into r = v mod 27 (its first three codes) and
// q = v / 27 (the last two), q = (v * 19) >> 9 exactly for every v < 243.
// For every byte position the CTA builds two tables of partial sums of the
// (power-of-two prescaled) activations: A[r] over the three codes (27
// entries) and B[q] over the two (9 entries and a zero for the invalid
// bytes' q = 9).  A byte then costs two table lookups and two adds.  A
// 27-entry fp16 table spans 14 words, so the 32 lanes of a warp, which look
// up the same byte position of 32 different rows, hit distinct banks or the
// same word: no bank conflicts, unlike a single 243-entry table per byte.
// Entries are formed with selects (no 0 * x), rounded once to fp16: within
// 2^-11 of the sum of their inputs' magnitudes, inside the 1e-3 budget.
//
// Layout of the work: one CTA per SM owns a contiguous range of 32-row
// blocks.  For each chunk of up to 32 groups (4096 inputs) it builds the
// chunk's tables, then its 16 warps take work items (one 32-row block x two
// groups): a warp stages the 32 rows' 52 bytes in shared memory from
// coalesced 4-byte loads issued one item ahead (row pitch 60 bytes, 15 words,
// so each lane's word reads are conflict-free), then lane l runs row l.  Each item's partial goes
// to its own slot; the slots are summed in a fixed order, so the result is
// deterministic.
#include <algorithm>
#include <utility>

#include "common.cuh"
#include "internal.h"

namespace bit1 {

namespace {

constexpr int kL5Warps = 16;
constexpr int kL5Threads = kL5Warps * 32;
constexpr int kL5CG = 32;                     // groups per table chunk
constexpr int kL5SG = 2;                      // groups per work item (52 bytes of a row)
constexpr int kL5Words = 13;                  // 4-byte words of a row per item
constexpr int kL5Pitch = 60;                  // staged row pitch: 15 words (odd: conflict-free)
constexpr int kL5PosBytes = 80;               // one byte position: A (27 halves), B (10), pad (3)
constexpr int kL5GroupBytes = 26 * kL5PosBytes;
constexpr int kL5Subs = kL5CG / kL5SG;        // items of a block per chunk

struct L5Params {
    const uint8_t* packed;    // [N][G*26]
    const uint16_t* scales;   // [N][G] fp16
    const uint16_t* x;        // [K] bf16
    void* y;                  // [N]
    int N, K, G, RB, bpc, y_bf16;
    uint32_t off_fac, off_stage, off_part, off_acc;
};

__device__ __forceinline__ float l5_sel(int d, float v) {   // (d - 1) * v without a multiply
    return d == 2 ? v : (d == 0 ? -v : 0.f);
}

__device__ __forceinline__ float l5_add(unsigned short t, float acc) {
    asm("add.rn.f32.f16 %0, %1, %0;" : "+f"(acc) : "h"(t));
    return acc;
}

// The two lookups of byte v at position offset P (bytes) from the group table
// base tg: A[v mod 27] + B[v / 27], accumulated into a and b.
template <int P>
__device__ __forceinline__ void l5_byte(uint32_t v, uint32_t tg, float& a, float& b) {
    const uint32_t q = __umulhi(v, 19u << 23);
    const uint32_t r = v - 27u * q;
    unsigned short ta, tb;
    asm("ld.shared.b16 %0, [%1+%2];" : "=h"(ta) : "r"(tg + 2u * r), "n"(P));
    asm("ld.shared.b16 %0, [%1+%2];" : "=h"(tb) : "r"(tg + 2u * q), "n"(P + 54));
    a = l5_add(ta, a);
    b = l5_add(tb, b);
}

// The 26 bytes of one group of the staged row (words w, group gg of the item).
template <int GG, size_t... J>
__device__ __forceinline__ float l5_group(const uint32_t (&w)[kL5Words], uint32_t tg, std::index_sequence<J...>) {
    float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
    (((J & 1) ? l5_byte<(int)J * kL5PosBytes>((w[(26 * GG + J) >> 2] >> (8 * ((26 * GG + J) & 3))) & 0xffu,
                                              tg, a1, b1)
              : l5_byte<(int)J * kL5PosBytes>((w[(26 * GG + J) >> 2] >> (8 * ((26 * GG + J) & 3))) & 0xffu,
                                              tg, a0, b0)), ...);
    return (a0 + a1) + (b0 + b1);
}

template <size_t... GG>
__device__ __forceinline__ float l5_item(const uint32_t (&w)[kL5Words], uint32_t tg0, const float (&f)[kL5SG],
                                         std::index_sequence<GG...>) {
    float acc = 0.f;
    ((acc = fmaf(l5_group<(int)GG>(w, tg0 + (uint32_t)GG * kL5GroupBytes, std::make_index_sequence<26>{}),
                 f[GG], acc)), ...);
    return acc;
}

}  // namespace

__global__ void __launch_bounds__(kL5Threads, 1) k_gemv_t5lut(const __grid_constant__ L5Params p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = (uint32_t)__cvta_generic_to_shared(smem_raw);
    const uint32_t base = (raw + 127u) & ~127u;
    uint8_t* sm = smem_raw + (base - raw);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int rb0 = (int)((int64_t)p.RB * blockIdx.x / gridDim.x);
    const int rb1 = (int)((int64_t)p.RB * (blockIdx.x + 1) / gridDim.x);
    const int nb = rb1 - rb0;
    const int64_t row_bytes = (int64_t)p.G * 26;

    float* fac = reinterpret_cast<float*>(sm + p.off_fac);        // [2][kL5CG]: 2^m, 2^-m
    float* part = reinterpret_cast<float*>(sm + p.off_part);      // [bpc][kL5Subs][32]
    float* racc = reinterpret_cast<float*>(sm + p.off_acc);       // [bpc][32]
    const uint32_t tab = base;                                     // [kL5CG][26 positions][80 B]
    const uint32_t stage = base + p.off_stage + (uint32_t)warp * 32u * kL5Pitch;
    for (int i = threadIdx.x; i < nb * 32; i += kL5Threads) racc[i] = 0.f;

    pdl_wait();
    for (int c0 = 0; c0 < p.G; c0 += kL5CG) {
        const int cg = min(kL5CG, p.G - c0);
        __syncthreads();                                           // previous chunk's tables no longer read
        // power-of-two prescale of each group: max |x'| < 2^12
        for (int g = warp; g < cg; g += kL5Warps) {
            const uint2 xv = *reinterpret_cast<const uint2*>(p.x + (size_t)(c0 + g) * 128 + 4 * lane);
            float m = fmaxf(fmaxf(fabsf(bf16_bits_to_f32(xv.x & 0xffffu)), fabsf(bf16_bits_to_f32(xv.x >> 16))),
                            fmaxf(fabsf(bf16_bits_to_f32(xv.y & 0xffffu)), fabsf(bf16_bits_to_f32(xv.y >> 16))));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            int mg = 0;
            if (m > 0.f) {
                const int e = (int)((__float_as_uint(m) >> 23) & 0xffu) - 127;
                mg = min(max(e - 11, -126), 127);
            }
            if (lane == 0) {
                fac[g] = __uint_as_float((uint32_t)(mg + 127) << 23);
                fac[kL5CG + g] = __uint_as_float((uint32_t)(127 - mg) << 23);
            }
        }
        __syncthreads();
        // tables: one thread per (group, byte position)
        for (int t = threadIdx.x; t < cg * 26; t += kL5Threads) {
            const int g = t / 26, j = t - g * 26;
            const float finv = fac[kL5CG + g];
            const uint16_t* xs = p.x + (size_t)(c0 + g) * 128 + 5 * j;
            float xv[5];
#pragma unroll
            for (int i = 0; i < 5; ++i)
                xv[i] = (j < 25 || i < 3) ? bf16_bits_to_f32(__ldg(xs + i)) * finv : 0.f;
            uint32_t* out = reinterpret_cast<uint32_t*>(sm + g * kL5GroupBytes + j * kL5PosBytes);
            uint32_t hw[20];
#pragma unroll
            for (int e = 0; e < 40; ++e) {
                float v = 0.f;
                if (e < 27) {
                    v = l5_sel(e % 3, xv[0]) + l5_sel((e / 3) % 3, xv[1]) + l5_sel(e / 9, xv[2]);
                } else if (e < 36 && j < 25) {
                    const int qq = e - 27;
                    v = l5_sel(qq % 3, xv[3]) + l5_sel(qq / 3, xv[4]);
                }
                const uint32_t h = __half_as_ushort(__float2half_rn(v));
                if (e & 1) hw[e >> 1] |= h << 16;
                else hw[e >> 1] = h;
            }
#pragma unroll
            for (int i = 0; i < 20; ++i) out[i] = hw[i];
        }
        __syncthreads();
        if (c0 == 0) pdl_launch_dependents();

        // work items: (block, two groups of this chunk).  The next item's bytes
        // and scales are loaded into registers while the current one runs.
        const int subs = cg / kL5SG, total = nb * subs;
        uint32_t nxt[kL5Words], scn = 0u;
        auto fetch = [&](int it) {
            const int b = it / subs, sj = it - b * subs;
            const int g0 = c0 + kL5SG * sj, rowb = (rb0 + b) * 32;
#pragma unroll
            for (int k = 0; k < kL5Words; ++k) {
                const int i = lane + 32 * k, r = i / kL5Words, piece = i - r * kL5Words;
                nxt[k] = rowb + r < p.N
                             ? __ldg(reinterpret_cast<const uint32_t*>(p.packed + (int64_t)(rowb + r) * row_bytes +
                                                                       (int64_t)g0 * 26) + piece)
                             : 0u;
            }
            const int row = rowb + lane;
            scn = row < p.N ? __ldg(reinterpret_cast<const uint32_t*>(p.scales + (int64_t)row * p.G + g0)) : 0u;
        };
        uint32_t* stw = reinterpret_cast<uint32_t*>(sm + p.off_stage + (size_t)warp * 32 * kL5Pitch);
        if (warp < total) fetch(warp);
        for (int it = warp; it < total; it += kL5Warps) {
            const int b = it / subs, sj = it - b * subs;
            const int g0 = c0 + kL5SG * sj;
#pragma unroll
            for (int k = 0; k < kL5Words; ++k) {
                const int i = lane + 32 * k, r = i / kL5Words, piece = i - r * kL5Words;
                stw[r * (kL5Pitch / 4) + piece] = nxt[k];
            }
            const uint32_t sc2 = scn;
            __syncwarp();
            uint32_t w[kL5Words];
#pragma unroll
            for (int i = 0; i < kL5Words; ++i) {
                uint32_t v;
                asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(stage + (uint32_t)lane * kL5Pitch + 4u * i));
                w[i] = v;
            }
            __syncwarp();                                          // the stage is free for the next item
            if (it + kL5Warps < total) fetch(it + kL5Warps);
            float f[kL5SG];
            f[0] = f16_bits_to_f32((uint16_t)(sc2 & 0xffffu)) * fac[g0 - c0];
            f[1] = f16_bits_to_f32((uint16_t)(sc2 >> 16)) * fac[g0 - c0 + 1];
            const float acc = l5_item(w, tab + (uint32_t)(g0 - c0) * kL5GroupBytes, f,
                                      std::make_index_sequence<kL5SG>{});
            part[(b * kL5Subs + sj) * 32 + lane] = acc;
        }
        __syncthreads();
        // this chunk's item partials, in a fixed order, onto the rows
        for (int i = threadIdx.x; i < nb * 32; i += kL5Threads) {
            const int b = i >> 5, l = i & 31;
            float v = racc[i];
            for (int sj = 0; sj < subs; ++sj) v += part[(b * kL5Subs + sj) * 32 + l];
            racc[i] = v;
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < nb * 32; i += kL5Threads) {
        const int row = rb0 * 32 + i;
        if (row < p.N) {
            if (p.y_bf16) reinterpret_cast<uint16_t*>(p.y)[row] = f32_to_bf16_bits(racc[i]);
            else reinterpret_cast<float*>(p.y)[row] = racc[i];
        }
    }
}

bool t5lut_supported(int64_t B, int64_t N, int64_t K) {
    return B == 1 && N >= 1 && N <= (1LL << 30) && K >= 1024 && K % 1024 == 0 && K <= (1LL << 20);
}

cudaError_t launch_gemv_t5lut(const uint8_t* packed, const uint16_t* scales, const uint16_t* x, int64_t N,
                              int64_t K, void* y, bool y_bf16, cudaStream_t stream) {
    if (!t5lut_supported(1, N, K)) return cudaErrorNotSupported;
    L5Params prm{};
    prm.packed = packed;
    prm.scales = scales;
    prm.x = x;
    prm.y = y;
    prm.N = (int)N;
    prm.K = (int)K;
    prm.G = (int)(K / 128);
    prm.RB = (int)((N + 31) / 32);
    const int grid = std::max(1, std::min(sm_count(), prm.RB));
    prm.bpc = (prm.RB + grid - 1) / grid;
    prm.y_bf16 = y_bf16 ? 1 : 0;
    uint32_t off = (uint32_t)(kL5CG * kL5GroupBytes);              // tables
    prm.off_fac = off;    off += 2 * kL5CG * 4;
    prm.off_stage = off;  off += (uint32_t)(kL5Warps * 32 * kL5Pitch);
    off = (off + 15u) & ~15u;
    prm.off_part = off;   off += (uint32_t)(prm.bpc * kL5Subs * 32 * 4);
    prm.off_acc = off;    off += (uint32_t)(prm.bpc * 32 * 4);
    const size_t smem = 128 + (size_t)off;
    if (smem > 227 * 1024) return cudaErrorNotSupported;
    const cudaError_t e = func_attrs((const void*)k_gemv_t5lut, 227 * 1024, false);
    if (e != cudaSuccess) return e;
    void* args[] = {(void*)&prm};
    return launch((const void*)k_gemv_t5lut, dim3((unsigned)grid), dim3(kL5Threads), smem, stream, false, args);
}

}  // namespace bit1
