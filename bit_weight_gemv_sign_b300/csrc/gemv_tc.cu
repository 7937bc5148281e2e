// Batched GEMM over packed sign bits on the 5th-generation tensor cores
// (tcgen05, sm_103a), for batch >= 16 where the product is a real dense
// contraction: Y[b][n] = sum_k X[b][k] * W[n][k], W[n][k] = s[n][k/128] * (+-1).
//
// Format and semantics: web page "Bonsai 27B: 노트북과 폰에서 실행되는 27B급
// 이진 및 삼진 저비트 LLM", section "이진(Binary) 가중치 형식" (w = s_g * b) and
// section "하이브리드 어텐션을 위한 저비트 커널" (packed codes decoded inside the
// fused product, never a dense fp16 weight matrix in memory, high-precision
// accumulation; prompt processing is the compute-heavy regime).
//
// Design (one CTA = 256 weight rows x one K range):
//  * A (weights): two M = 128 operands per K step, held in tensor memory.
//    Thread t of warps 0-7 owns one row: per 128-input step it reads the row's
//    16 sign bytes from a TMA-filled shared-memory ring, forms +-s exactly in
//    fp16 and writes the 64 fp16x2 words with tcgen05.st.  Inside every
//    32-bit sign word, inputs k and k+16 share one fp16x2 register (sign bits
//    15 and 31), so one shift and one LOP3 produce two weights; the
//    activations are stored in the same permuted K order, so the contraction
//    is unchanged.  No dense weight tile ever exists in shared memory or HBM.
//  * B (activations): a prep kernel converts x (bf16) to fp16 with an exact
//    per-batch-row power-of-two prescale (a bf16 significand fits fp16's),
//    permuted as above, into the workspace; TMA stages 64-wide K boxes with
//    128-byte swizzle (the canonical K-major operand layout).
//  * fp32 accumulators in tensor memory (N = batch rounded up to 16; two
//    accumulators, one per 128-row half), read back with tcgen05.ld; the
//    prescale is undone in the epilogue.
//  * Warps 0-7 unpack and run the epilogue, warp 8 streams sign bits, warp 9
//    streams activations, warp 10 issues the MMAs; every mbarrier wait is
//    bounded.  When the row tiles alone cannot fill the SMs, K is split over
//    CTAs and a second kernel sums the fp32 partials in a fixed order.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "t6_common.cuh"

namespace bit1 {

__device__ unsigned int g_tc_wait_timeouts = 0;

constexpr int kTcRows = 256;              // weight rows per CTA (two M = 128 MMAs)
constexpr int kTcStepK = 128;             // inputs per pipeline step (one scale group)
constexpr int kTcStages = 3;              // A (tensor memory) / B (shared memory) stages
constexpr int kTcWSlots = 8;              // sign-bit ring slots (4 KB each)
constexpr int kTcMaxB = 64;               // batch rows per launch (accumulators: 2 x 64 columns)
constexpr int kTcUnpackWarps = 8;
constexpr int kTcThreads = 32 * (kTcUnpackWarps + 3);
constexpr uint32_t kTcWSlotBytes = kTcRows * 16;

struct TcParams {
    const uint16_t* scales;
    const float* xscale;      // [Bp] 2^m_b (undo the prescale)
    float* partial;           // [Ks][Bp][N] fp32 when Ks > 1, else null
    void* y;                  // [B][N]
    int N, K, B, Bp, Ks, steps, y_bf16;
};

// ---------------------------------------------------------------- helpers
__device__ __forceinline__ void tc_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle (8-row x
// 128-byte atoms, consecutive atoms 1024 bytes apart), descriptor version 1.
__device__ __forceinline__ uint64_t tc_desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}
__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// ---------------------------------------------------------------- prep
// One CTA per padded batch row b: xp[b][32q + 2j + h] = fp16(x[b][32q + j + 16h]
// * 2^-m_b) and xscale[b] = 2^m_b, with m_b chosen so that max|x * 2^-m_b| lies
// in [2^14, 2^15) (exact: bf16 keeps 8 significant bits, fp16 11).  Rows b >= B
// are zero.
__global__ void __launch_bounds__(256) k_tc_prep(const uint16_t* __restrict__ x, int B, int K,
                                                 uint16_t* __restrict__ xp, float* __restrict__ xscale) {
    pdl_wait();
    const int b = blockIdx.x;
    __shared__ uint32_t red[8];
    uint16_t* out = xp + (size_t)b * K;
    if (b >= B) {
        for (int i = threadIdx.x; i < K / 8; i += blockDim.x) reinterpret_cast<uint4*>(out)[i] = make_uint4(0, 0, 0, 0);
        if (threadIdx.x == 0) xscale[b] = 1.f;
        return;
    }
    const uint16_t* in = x + (size_t)b * K;
    uint32_t m = 0;                                   // max |x| as bf16 magnitude bits (monotone)
    for (int i = threadIdx.x; i < K; i += blockDim.x) {
        const uint32_t v = in[i] & 0x7fffu;
        m = max(m, v > 0x7f80u ? 0u : v);             // NaN does not set the scale
    }
    m = __reduce_max_sync(0xffffffffu, m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    m = red[0];
    for (int i = 1; i < (int)(blockDim.x >> 5); ++i) m = max(m, red[i]);
    int mb = 0;
    if (m != 0) {
        const int e = (int)(m >> 7) - 127;            // exponent of max|x| (subnormal -> -127)
        mb = min(max(e - 14, -126), 126);
    }
    const float finv = __uint_as_float((uint32_t)(127 - mb) << 23);
    if (threadIdx.x == 0) xscale[b] = __uint_as_float((uint32_t)(mb + 127) << 23);
    for (int i = threadIdx.x; i < K / 2; i += blockDim.x) {   // output pair i = (32q + 2j, 32q + 2j + 1)
        const int q = i >> 4, j = i & 15;
        const float lo = bf16_bits_to_f32(in[32 * q + j]) * finv;
        const float hi = bf16_bits_to_f32(in[32 * q + j + 16]) * finv;
        const __half2 h = __floats2half2_rn(lo, hi);
        reinterpret_cast<uint32_t*>(out)[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
}

// ---------------------------------------------------------------- reduce
// y[b][n] = xscale[b] * sum over s = 0 .. Ks-1 (in order) of partial[s][b][n].
__global__ void __launch_bounds__(256) k_tc_reduce(const float* __restrict__ partial, const float* __restrict__ xscale,
                                                   int Ks, int B, int Bp, int N, void* __restrict__ y, int y_bf16) {
    pdl_wait();
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)B * N) return;
    const int b = (int)(i / N), n = (int)(i - (int64_t)b * N);
    float v = 0.f;
    for (int s = 0; s < Ks; ++s) v += partial[((int64_t)s * Bp + b) * N + n];
    v *= xscale[b];
    if (y_bf16) reinterpret_cast<uint16_t*>(y)[i] = f32_to_bf16_bits(v);
    else reinterpret_cast<float*>(y)[i] = v;
}

// ---------------------------------------------------------------- main kernel
// Grid: (row tiles) x Ks.  Shared memory: [sign-bit ring 8 x 4 KB][B ring 3 x
// Bp*256 B][mbarriers][tensor-memory slot].
__global__ void __launch_bounds__(kTcThreads, 1)
k_gemv_tc(const __grid_constant__ CUtensorMap tm_bits, const __grid_constant__ CUtensorMap tm_x,
          const __grid_constant__ TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = (uint32_t)__cvta_generic_to_shared(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int Mt = (p.N + kTcRows - 1) / kTcRows;
    const int mt = blockIdx.x % Mt, ks = blockIdx.x / Mt;
    const int s0 = (int)((int64_t)p.steps * ks / p.Ks), s1 = (int)((int64_t)p.steps * (ks + 1) / p.Ks);
    const int nst = s1 - s0;
    const uint32_t btile = (uint32_t)p.Bp * 128u;          // one 64-wide K box of B
    const uint32_t bstage = 2u * btile;                     // one step (128 K)
    const uint32_t wring = base;
    const uint32_t bring = base + kTcWSlots * kTcWSlotBytes;
    const uint32_t bar0 = bring + kTcStages * bstage;
    const uint32_t wfull = bar0, wempty = bar0 + 8 * kTcWSlots;
    const uint32_t afull = bar0 + 16 * kTcWSlots, bfull = afull + 8 * kTcStages, freed = bfull + 8 * kTcStages;
    const uint32_t d_done = freed + 8 * kTcStages;
    const uint32_t tslot_s = d_done + 8;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem_raw + (tslot_s - raw));

    if (threadIdx.x == 0) {
        for (int i = 0; i < kTcWSlots; ++i) {
            mbar_init(wfull + 8 * i, 1);
            mbar_init(wempty + 8 * i, kTcUnpackWarps);
        }
        for (int s = 0; s < kTcStages; ++s) {
            mbar_init(afull + 8 * s, kTcUnpackWarps);
            mbar_init(bfull + 8 * s, 1);
            mbar_init(freed + 8 * s, 1);
        }
        mbar_init(d_done, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(tslot_s) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;");
    // Tensor memory: D half h at columns [h*Bp, h*Bp + Bp); A stage st, half h
    // at columns 128 + 128*st + 64*h (64 columns = 128 fp16 inputs).
    const uint32_t tmem = *tslot;
    pdl_wait();

    if (warp < kTcUnpackWarps) {
        const int quad = warp & 3, h = warp >> 2;
        const int r = 128 * h + 32 * quad + lane;          // row within the tile
        const int row = mt * kTcRows + r;
        const bool live = row < p.N;
        const int G = p.K / 128;
        const uint16_t* rs = p.scales + (size_t)(live ? row : 0) * G;
        const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
        bool ok = true;
        // fp16 scales of this row, 8 groups (16 bytes) per window, one window ahead
        uint4 sc_cur = make_uint4(0, 0, 0, 0), sc_nxt = sc_cur;
        if (live && nst > 0) {
            sc_cur = ldg_nc_v4(rs + (s0 & ~7));
            if ((s0 >> 3) + 1 < G / 8) sc_nxt = ldg_nc_v4(rs + (s0 & ~7) + 8);
        }
        for (int s = 0; s < nst; ++s) {
            const int step = s0 + s;
            if ((step & 7) == 0 && s > 0) {
                sc_cur = sc_nxt;
                if (live && (step >> 3) + 1 < G / 8) sc_nxt = ldg_nc_v4(rs + step + 8);
            }
            const int st = s % kTcStages, ws = s % kTcWSlots;
            if (s >= kTcStages && !warp_wait(freed + 8 * st, (uint32_t)(s / kTcStages - 1) & 1u)) { ok = false; break; }
            if (!warp_wait(wfull + 8 * ws, (uint32_t)(s / kTcWSlots) & 1u)) { ok = false; break; }
            asm volatile("tcgen05.fence::after_thread_sync;");
            const uint4 w = lds128(wring + ws * kTcWSlotBytes + 16u * r);
            __syncwarp();
            if (lane == 0) tc_arrive(wempty + 8 * ws);
            const uint32_t wsel = (step & 4) ? ((step & 2) ? sc_cur.w : sc_cur.z) : ((step & 2) ? sc_cur.y : sc_cur.x);
            const uint32_t s16 = (step & 1) ? (wsel >> 16) : (wsel & 0xffffu);
            const uint32_t s2 = live ? (s16 | (s16 << 16)) : 0u;
            const uint32_t words[4] = {~w.x, ~w.y, ~w.z, ~w.w};
            const uint32_t col0 = 128u + 128u * st + 64u * h;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t v[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = ((words[q] << (15 - j)) & 0x80008000u) | s2;  // bit 1 -> +s
                asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                             ::"r"(tmem + lane_base + col0 + 16u * q), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]),
                               "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]),
                               "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]) : "memory");
            }
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            asm volatile("tcgen05.fence::before_thread_sync;");
            __syncwarp();
            if (lane == 0) tc_arrive(afull + 8 * st);
        }
        // ---- epilogue: accumulator half h, row r
        if (ok) ok = warp_wait(d_done, 0);
        if (!ok) {
            if (lane == 0) atomicOr(&g_tc_wait_timeouts, 1u);
        } else if (nst > 0) {
            asm volatile("tcgen05.fence::after_thread_sync;");
            for (int c0 = 0; c0 < p.Bp; c0 += 16) {
                uint32_t d[16];
                asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                             : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3]), "=r"(d[4]), "=r"(d[5]), "=r"(d[6]),
                               "=r"(d[7]), "=r"(d[8]), "=r"(d[9]), "=r"(d[10]), "=r"(d[11]), "=r"(d[12]), "=r"(d[13]),
                               "=r"(d[14]), "=r"(d[15])
                             : "r"(tmem + lane_base + (uint32_t)(h * p.Bp + c0)) : "memory");
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                if (live) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int b = c0 + i;
                        const float v = __uint_as_float(d[i]);
                        if (p.partial) {
                            p.partial[((int64_t)ks * p.Bp + b) * p.N + row] = v;
                        } else if (b < p.B) {
                            const float yv = v * p.xscale[b];
                            if (p.y_bf16) reinterpret_cast<uint16_t*>(p.y)[(int64_t)b * p.N + row] = f32_to_bf16_bits(yv);
                            else reinterpret_cast<float*>(p.y)[(int64_t)b * p.N + row] = yv;
                        }
                    }
                }
            }
        }
    } else if (warp == kTcUnpackWarps) {
        // ---- sign-bit producer: one 256-row x 16-byte box per step
        if (lane == 0) {
            int issued = 0;
            for (int s = 0; s < nst; ++s) {
                const int ws = s % kTcWSlots;
                if (s >= kTcWSlots && !mbar_wait(wempty + 8 * ws, (uint32_t)(s / kTcWSlots - 1) & 1u)) {
                    atomicOr(&g_tc_wait_timeouts, 2u);
                    break;
                }
                mbar_expect_tx(wfull + 8 * ws, kTcWSlotBytes);
                tma_2d(wring + ws * kTcWSlotBytes, &tm_bits, 16 * (s0 + s), mt * kTcRows, wfull + 8 * ws);
                ++issued;
            }
            // every issued copy has landed before the CTA may exit
            for (int s = std::max(0, issued - kTcWSlots); s < issued; ++s)
                if (!mbar_wait(wfull + 8 * (s % kTcWSlots), (uint32_t)(s / kTcWSlots) & 1u)) atomicOr(&g_tc_wait_timeouts, 2u);
        }
    } else if (warp == kTcUnpackWarps + 1) {
        // ---- activation producer: two 64-input boxes per step
        if (lane == 0) {
            int issued = 0;
            for (int s = 0; s < nst; ++s) {
                const int st = s % kTcStages;
                if (s >= kTcStages && !mbar_wait(freed + 8 * st, (uint32_t)(s / kTcStages - 1) & 1u)) {
                    atomicOr(&g_tc_wait_timeouts, 4u);
                    break;
                }
                const uint32_t dst = bring + st * bstage;
                mbar_expect_tx(bfull + 8 * st, bstage);
                const int k = (s0 + s) * kTcStepK;
                tma_2d(dst, &tm_x, k, 0, bfull + 8 * st);
                tma_2d(dst + btile, &tm_x, k + 64, 0, bfull + 8 * st);
                ++issued;
            }
            for (int s = std::max(0, issued - kTcStages); s < issued; ++s)
                if (!mbar_wait(bfull + 8 * (s % kTcStages), (uint32_t)(s / kTcStages) & 1u)) atomicOr(&g_tc_wait_timeouts, 4u);
        }
    } else {
        // ---- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = (1u << 4)                         // D: fp32
                                   | (0u << 7) | (0u << 10)          // A, B: fp16
                                   | ((uint32_t)(p.Bp >> 3) << 17)   // N
                                   | ((uint32_t)(128 >> 4) << 24);   // M
            for (int s = 0; s < nst; ++s) {
                const int st = s % kTcStages;
                const uint32_t par = (uint32_t)(s / kTcStages) & 1u;
                if (!mbar_wait(afull + 8 * st, par) || !mbar_wait(bfull + 8 * st, par)) {
                    atomicOr(&g_tc_wait_timeouts, 8u);
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;");
                const uint32_t bst = bring + st * bstage;
#pragma unroll
                for (int kk = 0; kk < kTcStepK / 16; ++kk) {
                    const uint64_t bdesc = tc_desc_sw128(bst + (kk >> 2) * btile + (kk & 3) * 32);
                    const uint32_t acc = (s > 0 || kk > 0) ? 1u : 0u;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t a_addr = tmem + 128u + 128u * st + 64u * h + 8u * kk;
                        const uint32_t d_addr = tmem + (uint32_t)(h * p.Bp);
                        asm volatile("{.reg .pred pa; setp.ne.b32 pa, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, pa;}"
                                     ::"r"(d_addr), "r"(a_addr), "l"(bdesc), "r"(idesc), "r"(acc) : "memory");
                    }
                }
                asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                             ::"r"(freed + 8 * st) : "memory");
            }
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                         ::"r"(d_done) : "memory");
            // no MMA may still be running when the tensor memory is released
            if (!mbar_wait(d_done, 0)) atomicOr(&g_tc_wait_timeouts, 8u);
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
}

// ---------------------------------------------------------------- host
namespace {

PFN_cuTensorMapEncodeTiled_v12000 tc_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void* f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

struct TcPlan {
    int Bp, Mt, Ks, steps;
    size_t smem, ws_xp, ws_scale, ws_part, ws_total, off_part;
};

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

TcPlan tc_plan(int64_t B, int64_t N, int64_t K) {
    TcPlan pl{};
    const int64_t Bc = std::min<int64_t>(B, kTcMaxB);
    pl.Bp = (int)((Bc + 15) / 16 * 16);
    pl.Mt = (int)((N + kTcRows - 1) / kTcRows);
    pl.steps = (int)(K / kTcStepK);
    // Split K until the CTAs fill the SMs once (one CTA per SM: it holds all
    // 512 tensor-memory columns); every slice keeps at least 8 steps.
    const int sms = sm_count();
    int ks = 1;
    while (pl.Mt * (ks + 1) <= sms && pl.steps / (ks + 1) >= 8) ++ks;
    pl.Ks = ks;
    const size_t need = 1024 + (size_t)kTcWSlots * kTcWSlotBytes + (size_t)kTcStages * 2 * 128 * pl.Bp +
                        8 * (2 * kTcWSlots + 3 * kTcStages + 1) + 16;
    pl.smem = std::max<size_t>(need, 120 * 1024);   // keeps a second CTA off the SM
    pl.ws_xp = align256((size_t)pl.Bp * K * 2);
    pl.ws_scale = 256;
    pl.off_part = pl.ws_xp + pl.ws_scale;
    pl.ws_part = pl.Ks > 1 ? align256((size_t)pl.Ks * pl.Bp * N * 4) : 0;
    pl.ws_total = pl.off_part + pl.ws_part;
    return pl;
}

}  // namespace

bool tc_supported(int64_t B, int64_t N, int64_t K) {
    return B >= 1 && N >= 1 && N <= (1LL << 30) && K >= 1024 && K % 1024 == 0 && K <= (1LL << 20) &&
           (int64_t)N * (K / 8) < (1LL << 40);
}

size_t tc_workspace_bytes(int64_t B, int64_t N, int64_t K) {
    if (!tc_supported(B, N, K)) return 0;
    return tc_plan(B, N, K).ws_total;
}

int tc_launch_count(int64_t B, int64_t N, int64_t K) {
    if (!tc_supported(B, N, K)) return 0;
    const TcPlan pl = tc_plan(B, N, K);
    const int64_t chunks = (B + kTcMaxB - 1) / kTcMaxB;
    return (int)(chunks * (2 + (pl.Ks > 1 ? 1 : 0)));
}

cudaError_t launch_gemv_tc(const GemvArgs& a) {
    if (!tc_supported(a.B, a.N, a.K)) return cudaErrorNotSupported;
    const TcPlan pl = tc_plan(a.B, a.N, a.K);
    if (!a.workspace || a.ws_bytes < pl.ws_total) return cudaErrorInvalidValue;
    auto enc = tc_encode();
    if (!enc) return cudaErrorNotSupported;
    uint8_t* ws = static_cast<uint8_t*>(a.workspace);
    uint16_t* xp = reinterpret_cast<uint16_t*>(ws);
    float* xscale = reinterpret_cast<float*>(ws + pl.ws_xp);
    float* partial = pl.Ks > 1 ? reinterpret_cast<float*>(ws + pl.off_part) : nullptr;
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute((const void*)k_gemv_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    });
    if (attr_err != cudaSuccess) return attr_err;

    CUtensorMap tm_bits;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)(a.K / 8), (cuuint64_t)a.N};
        const cuuint64_t strides[1] = {(cuuint64_t)(a.K / 8)};
        const cuuint32_t box[2] = {16, (cuuint32_t)kTcRows};
        const cuuint32_t es[2] = {1, 1};
        if (enc(&tm_bits, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, (void*)a.bits, dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const size_t ysz = a.y_bf16 ? 2 : 4;
    for (int64_t b0 = 0; b0 < a.B; b0 += kTcMaxB) {
        const int Bc = (int)std::min<int64_t>(kTcMaxB, a.B - b0);
        const int Bp = (Bc + 15) / 16 * 16;
        const uint16_t* xin = a.x + b0 * a.K;
        int Bci = Bc, Ki = (int)a.K;
        void* prep_args[] = {(void*)&xin, (void*)&Bci, (void*)&Ki, (void*)&xp, (void*)&xscale};
        cudaError_t e = launch((const void*)k_tc_prep, dim3((unsigned)Bp), dim3(256), 0, a.stream, a.pdl || b0 > 0,
                               prep_args);
        if (e != cudaSuccess) return e;
        CUtensorMap tm_x;
        {
            const cuuint64_t dims[2] = {(cuuint64_t)a.K, (cuuint64_t)Bp};
            const cuuint64_t strides[1] = {(cuuint64_t)(a.K * 2)};
            const cuuint32_t box[2] = {64, (cuuint32_t)Bp};
            const cuuint32_t es[2] = {1, 1};
            if (enc(&tm_x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, (void*)xp, dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return cudaErrorInvalidValue;
        }
        TcParams prm;
        prm.scales = a.scales;
        prm.xscale = xscale;
        prm.partial = partial;
        prm.y = static_cast<uint8_t*>(a.y) + b0 * a.N * ysz;
        prm.N = (int)a.N;
        prm.K = (int)a.K;
        prm.B = Bc;
        prm.Bp = Bp;
        prm.Ks = pl.Ks;
        prm.steps = pl.steps;
        prm.y_bf16 = a.y_bf16;
        void* args[] = {(void*)&tm_bits, (void*)&tm_x, (void*)&prm};
        e = launch((const void*)k_gemv_tc, dim3((unsigned)(pl.Mt * pl.Ks)), dim3(kTcThreads), pl.smem, a.stream, true,
                   args);
        if (e != cudaSuccess) return e;
        if (pl.Ks > 1) {
            const int64_t total = (int64_t)Bc * a.N;
            const float* pc = partial;
            const float* xs = xscale;
            int Ksi = pl.Ks, Bpi = Bp, Ni = (int)a.N, yb = a.y_bf16;
            void* yp = prm.y;
            void* rargs[] = {(void*)&pc, (void*)&xs, (void*)&Ksi, (void*)&Bci, (void*)&Bpi, (void*)&Ni, (void*)&yp, (void*)&yb};
            e = launch((const void*)k_tc_reduce, dim3((unsigned)((total + 255) / 256)), dim3(256), 0, a.stream, true, rargs);
            if (e != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

unsigned int tc_take_timeouts() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_tc_wait_timeouts, sizeof(v)) != cudaSuccess) return 0xffffffffu;
    if (v) cudaMemcpyToSymbol(g_tc_wait_timeouts, &zero, sizeof(zero));
    return v;
}

}  // namespace bit1
