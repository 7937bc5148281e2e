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
//    16 sign bytes from a shared-memory ring (TMA boxes of 64 bytes x 256 rows,
//    four steps, 64-byte swizzle), forms +-s exactly in fp16 and writes the 64
//    fp16x2 words with tcgen05.st.  Inside every
//    32-bit sign word, inputs k and k+16 share one fp16x2 register (sign bits
//    15 and 31), so one shift and one LOP3 produce two weights; the
//    activations are stored in the same permuted K order, so the contraction
//    is unchanged.  No dense weight tile ever exists in shared memory or HBM.
//  * B (activations): a prep kernel converts x (bf16) to fp16 with an exact
//    per-batch-row power-of-two prescale (a bf16 significand fits fp16's),
//    permuted as above, into the workspace; one 3-D TMA box per step stages
//    two 64-wide K slabs with 128-byte swizzle (the canonical K-major layout).
//  * fp32 accumulators in tensor memory (N = batch rounded up to 16; four
//    accumulators: two per 128-row half, for the even and the odd 16-input
//    slices of each step, summed in that order in the epilogue), read back
//    with tcgen05.ld; the prescale is undone in the epilogue.
//  * Warps 0-7 unpack and run the epilogue, warp 8 streams sign bits (one
//    issuing lane per ring slot), warp 9 streams activations (one lane per
//    stage), warps 10-13 issue the MMAs, one warp per accumulator (one thread
//    issues a tcgen05.mma about every 54 cycles, so a single issuer would
//    bound the kernel at small batch); every mbarrier wait is bounded.
//  * Sign bits and scales do not depend on the preceding kernel (the prep
//    kernel lets this one start only after its own wait on its predecessor),
//    so they stream and unpack before griddepcontrol.wait; only the
//    activation loads, the MMAs and the epilogue wait.
//  * When the row tiles alone cannot fill the SMs, K is split over the Ks CTAs
//    of a thread-block cluster in whole 4-step chunks.  Each CTA stages its
//    fp32 accumulators in its own shared memory; after a cluster barrier, CTA
//    j sums rows [64j/Ks, 64(j+1)/Ks) x 4 of every CTA's tile through
//    distributed shared memory in rank order (deterministic) and writes y.
//  * SwiGLU epilogue (rows interleaved as the gate/up pairs of a SwiGLU MLP,
//    the base model's MLP on the same page, section "Bonsai 27B의 표현
//    방식"): the two epilogue lanes of a pair exchange one value per two batch
//    columns and each writes h = silu(g) * u for one of them; the split-K
//    reduction sums four consecutive rows, i.e. two whole pairs.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <map>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "t6_common.cuh"
#include "tc_common.cuh"

namespace bit1 {

__device__ unsigned int g_tc_wait_timeouts = 0;

constexpr int kTcRows = 256;              // weight rows per CTA (two M = 128 MMAs)
constexpr int kTcStages = 3;              // max A (tensor memory) / B (shared memory) stages
constexpr int kTcWSlots = 4;              // sign-bit ring slots
constexpr uint32_t kTcWSlotBytes = kTcRows * 16 * kTcChunkSteps;   // 16 KB
constexpr int kTcMaxB = 64;               // batch rows per chunk with two accumulators per half
constexpr int kTcWideB = 128;             // rows per chunk with one accumulator per half (wide mode)
constexpr int kTcUnpackWarps = 8;
constexpr int kTcMmaWarps = 4;
constexpr int kTcThreads = 32 * (kTcUnpackWarps + 2 + kTcMmaWarps);

struct TcParams {
    const uint16_t* scales;
    const float* xscale;      // [Bp] 2^m_b (undo the prescale)
    void* y;                  // [B][N]
    int N, K, B, Bp, Ks, chunks, y_bf16;   // B: valid batch rows of all batch chunks of the launch
    int stages;               // A/B stages: 3 when the accumulators fit 128 columns (Bp <= 32), else 2
    int swiglu;               // rows are (gate, up) pairs; y is h = silu(gate) * up, [B][N/2]
    // Wide mode (Bp > 64): one accumulator per 128-row half (columns h*Bp), two
    // MMA issuers each issuing all eight 16-input slices of a step; Ks = 1.
};

// ---------------------------------------------------------------- helpers
__device__ __forceinline__ float4 ld_cluster_v4(uint32_t remote_addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(remote_addr) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t map_rank(uint32_t local_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void store_y(const TcParams& p, int b, int row, float v) {
    if (p.y_bf16) reinterpret_cast<uint16_t*>(p.y)[(int64_t)b * p.N + row] = f32_to_bf16_bits(v);
    else reinterpret_cast<float*>(p.y)[(int64_t)b * p.N + row] = v;
}
// SwiGLU output of hidden unit `unit` (rows 2 unit, 2 unit + 1): h = silu(g) * u.
__device__ __forceinline__ void put_h(const TcParams& p, int b, int unit, float h) {
    const int64_t o = (int64_t)b * (p.N >> 1) + unit;
    if (p.y_bf16) reinterpret_cast<uint16_t*>(p.y)[o] = f32_to_bf16_bits(h);
    else reinterpret_cast<float*>(p.y)[o] = h;
}
__device__ __forceinline__ void store_h(const TcParams& p, int b, int unit, float g, float u) {
    put_h(p, b, unit, g / (1.f + expf(-g)) * u);
}
// The same with the hardware exponential and reciprocal (a few ulps of h,
// far inside the products' own tolerance): the direct-store epilogue runs
// once per batch column of every row, on the CTA's critical path.
__device__ __forceinline__ void store_h_fast(const TcParams& p, int b, int unit, float g, float u) {
    put_h(p, b, unit, __fdividef(g, 1.f + __expf(-g)) * u);
}
// ---------------------------------------------------------------- prep
// One CTA per padded batch row b (tc_prep_row): xp[b] = the permuted,
// prescaled fp16 copy of x[b], xscale[b] = 2^m_b; rows b >= B are zero.
__global__ void __launch_bounds__(kTcPrepThreads) k_tc_prep(const uint16_t* __restrict__ x, int B, int K,
                                                            uint16_t* __restrict__ xp, float* __restrict__ xscale) {
    pdl_wait();
    pdl_launch_dependents();   // the main kernel may start: everything before this one has completed
    const int b = blockIdx.x;
    __shared__ uint32_t red[kTcPrepThreads / 32];
    tc_prep_row(b < B ? x + (size_t)b * K : nullptr, K, xp + (size_t)b * K, xscale + b, red);
}

// ---------------------------------------------------------------- main kernel
// Grid: Ks x (row tiles), clusters of Ks along x.  Shared memory: [sign-bit
// ring 4 x 16 KB, reused as the fp32 accumulator staging [Bp][256]][B ring 3 x
// Bp*256 B][mbarriers][tensor-memory slot].
__global__ void __launch_bounds__(kTcThreads, 1)
k_gemv_tc(const __grid_constant__ CUtensorMap tm_bits, const __grid_constant__ CUtensorMap tm_x,
          const __grid_constant__ TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = (uint32_t)__cvta_generic_to_shared(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int mt = blockIdx.x / p.Ks, ks = blockIdx.x % p.Ks;   // ks = rank in the cluster
    // Batch chunk: rows [cb0, cb0 + Bp) of x' and y (several chunks run as one
    // launch along grid y when the workspace holds all of them).
    const int cb0 = (int)blockIdx.y * p.Bp, bvalid = min(p.Bp, p.B - cb0);
    const int c0 = (int)((int64_t)p.chunks * ks / p.Ks), c1 = (int)((int64_t)p.chunks * (ks + 1) / p.Ks);
    const int nch = c1 - c0, s0 = c0 * kTcChunkSteps, nst = nch * kTcChunkSteps;
    const uint32_t btile = (uint32_t)p.Bp * 128u;          // one 64-wide K slab of B
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
            mbar_init(freed + 8 * s, p.Bp > kTcMaxB ? 2 : kTcMmaWarps);    // one commit per MMA issuer
        }
        mbar_init(d_done, p.Bp > kTcMaxB ? 2 : kTcMmaWarps);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(tslot_s) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;");
    // Tensor memory: accumulator (half h, slice parity q) at columns
    // (2h + q)*Bp; A stage st, half h at columns abase + 128*st + 64*h (64
    // columns = 128 fp16 inputs), abase = 4*Bp rounded up to 128.
    const uint32_t tmem = *tslot;
    const int nstg = p.stages;
    const bool wide = p.Bp > kTcMaxB;
    const uint32_t abase = (uint32_t)(((wide ? 2 : 4) * p.Bp + 127) / 128 * 128);

    if (warp < kTcUnpackWarps) {
        const int quad = warp & 3, h = warp >> 2;
        const int r = 128 * h + 32 * quad + lane;          // row within the tile
        const int row = mt * kTcRows + r;
        const bool live = row < p.N;
        const int G = p.K / 128;
        const uint16_t* rs = p.scales + (size_t)(live ? row : 0) * G;
        const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
        const uint32_t rsw = (uint32_t)(r >> 1) & 3u;      // 64-byte swizzle of this row
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
            const int st = s % nstg, c = s >> 2, i = s & 3, ws = c % kTcWSlots;
            if (s >= nstg && !warp_wait(freed + 8 * st, (uint32_t)(s / nstg - 1) & 1u)) { ok = false; break; }
            if (i == 0 && !warp_wait(wfull + 8 * ws, (uint32_t)(c / kTcWSlots) & 1u)) { ok = false; break; }
            asm volatile("tcgen05.fence::after_thread_sync;");
            const uint4 w = lds128(wring + ws * kTcWSlotBytes + 64u * r + 16u * ((uint32_t)i ^ rsw));
            if (i == kTcChunkSteps - 1) {
                __syncwarp();
                if (lane == 0) tc_arrive(wempty + 8 * ws);
            }
            const uint32_t wsel = (step & 4) ? ((step & 2) ? sc_cur.w : sc_cur.z) : ((step & 2) ? sc_cur.y : sc_cur.x);
            const uint32_t s16 = (step & 1) ? (wsel >> 16) : (wsel & 0xffffu);
            const uint32_t s2 = live ? (s16 | (s16 << 16)) : 0u;
            tc_unpack_step(w, s2, tmem + lane_base + abase + 128u * st + 64u * h);
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            asm volatile("tcgen05.fence::before_thread_sync;");
            __syncwarp();
            if (lane == 0) tc_arrive(afull + 8 * st);
        }
        // ---- epilogue: accumulators of half h, row r
        pdl_wait();
        if (ok) ok = warp_wait(d_done, 0);
        if (!ok) {
            if (lane == 0) atomicOr(&g_tc_wait_timeouts, 1u);
        } else {
            asm volatile("tcgen05.fence::after_thread_sync;");
            for (int cb = 0; cb < p.Bp; cb += 16) {
                uint32_t d[16], e[16];
                tc_ld16(tmem + lane_base + (uint32_t)((wide ? h : 2 * h) * p.Bp + cb), d);
                if (!wide) tc_ld16(tmem + lane_base + (uint32_t)((2 * h + 1) * p.Bp + cb), e);
                tc_wait_ld();
                if (!wide) {
#pragma unroll
                    for (int k = 0; k < 16; ++k) d[k] = __float_as_uint(__uint_as_float(d[k]) + __uint_as_float(e[k]));
                }
                if (p.Ks > 1) {
                    // stage [b][r] in the (drained) sign-bit ring for the cluster reduction
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        asm volatile("st.shared.u32 [%0], %1;" ::"r"(wring + 4u * (uint32_t)((cb + k) * kTcRows + r)), "r"(d[k]) : "memory");
                } else if (p.swiglu) {
                    // Lane 2m holds the gate row and lane 2m+1 the up row of unit
                    // row/2.  The pair splits the batch columns: the even lane forms h
                    // for column 2j, the odd lane for column 2j+1, after one exchange.
                    const bool odd = lane & 1;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int c0 = cb + 2 * j;
                        const float v0 = c0 < bvalid ? __uint_as_float(d[2 * j]) * p.xscale[cb0 + c0] : 0.f;
                        const float v1 = c0 + 1 < bvalid ? __uint_as_float(d[2 * j + 1]) * p.xscale[cb0 + c0 + 1] : 0.f;
                        const float w = __shfl_xor_sync(0xffffffffu, odd ? v0 : v1, 1);
                        const float g = odd ? w : v0, u = odd ? v1 : w;
                        const int c = c0 + (odd ? 1 : 0);
                        if (live && c < bvalid) store_h_fast(p, cb0 + c, row >> 1, g, u);
                    }
                } else if (live) {
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        if (cb + k < bvalid)
                            store_y(p, cb0 + cb + k, row, __uint_as_float(d[k]) * p.xscale[cb0 + cb + k]);
                }
            }
        }
    } else if (warp == kTcUnpackWarps) {
        // ---- sign-bit producer: lane L owns ring slot L (chunks L, L+4, ...)
        if (lane < kTcWSlots) {
            const uint32_t full = wfull + 8 * lane, empty = wempty + 8 * lane, dst = wring + lane * kTcWSlotBytes;
            int issued = 0;
            for (int c = lane; c < nch; c += kTcWSlots, ++issued) {
                if (issued > 0 && !mbar_wait(empty, (uint32_t)(issued - 1) & 1u)) {
                    atomicOr(&g_tc_wait_timeouts, 2u);
                    break;
                }
                mbar_expect_tx(full, kTcWSlotBytes);
                tma_2d(dst, &tm_bits, 16 * (s0 + kTcChunkSteps * c), mt * kTcRows, full);
            }
            // the last issued copy has landed before the CTA may exit
            if (issued > 0 && !mbar_wait(full, (uint32_t)(issued - 1) & 1u)) atomicOr(&g_tc_wait_timeouts, 2u);
        }
    } else if (warp == kTcUnpackWarps + 1) {
        // ---- activation producer: lane st owns stage st (steps st, st+nstg, ...)
        pdl_wait();
        if (lane < nstg) {
            const uint32_t full = bfull + 8 * lane, dst = bring + lane * bstage;
            int issued = 0;
            for (int s = lane; s < nst; s += nstg, ++issued) {
                if (issued > 0 && !mbar_wait(freed + 8 * lane, (uint32_t)(issued - 1) & 1u)) {
                    atomicOr(&g_tc_wait_timeouts, 4u);
                    break;
                }
                mbar_expect_tx(full, bstage);
                tma_3d(dst, &tm_x, 0, cb0, 2 * (s0 + s), full);
            }
            if (issued > 0 && !mbar_wait(full, (uint32_t)(issued - 1) & 1u)) atomicOr(&g_tc_wait_timeouts, 4u);
        }
    } else {
        // ---- MMA issuers: warp 10 + 2h + q accumulates half h, 16-input slices of parity q
        const int mw = warp - (kTcUnpackWarps + 2), h = mw >> 1, q = mw & 1;
        pdl_wait();
        // wide mode: warp (h, 0) issues every slice into the one accumulator of half h
        const int kk0 = wide ? 0 : q, kkd = wide ? 1 : 2;
        if (lane == 0 && !(wide && q == 1)) {
            const uint32_t idesc = tc_idesc_f16(p.Bp);
            const uint32_t d_addr = tmem + (uint32_t)((wide ? h : 2 * h + q) * p.Bp);
            for (int s = 0; s < nst; ++s) {
                const int st = s % nstg;
                const uint32_t par = (uint32_t)(s / nstg) & 1u;
                if (!mbar_wait(afull + 8 * st, par) || !mbar_wait(bfull + 8 * st, par)) {
                    atomicOr(&g_tc_wait_timeouts, 8u);
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;");
                const uint32_t bst = bring + st * bstage;
                const uint32_t a0 = tmem + abase + 128u * st + 64u * h;
                tc_mma_step(d_addr, a0, bst, btile, idesc, kk0, kkd, s == 0);
                tc_commit(freed + 8 * st);
            }
            tc_commit(d_done);
            // no MMA may still be running when the tensor memory is released
            if (!mbar_wait(d_done, 0)) atomicOr(&g_tc_wait_timeouts, 8u);
        }
    }
    if (p.Ks > 1) {
        // ---- split-K: sum the cluster's staged tiles in rank order (all threads
        // take part in both cluster barriers; the second keeps every CTA's
        // shared memory alive until all remote reads are done)
        cluster_sync();
        if (warp < kTcUnpackWarps) {
            const int q0 = 64 * ks / p.Ks, q1 = 64 * (ks + 1) / p.Ks, nq = q1 - q0;
            for (int it = threadIdx.x; it < nq * bvalid; it += kTcUnpackWarps * 32) {
                const int b = it / nq, r0 = 4 * (q0 + it % nq);
                const uint32_t off = wring + 4u * (uint32_t)(b * kTcRows + r0);
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
                for (int k = 0; k < p.Ks; ++k) {
                    const float4 v = ld_cluster_v4(map_rank(off, (uint32_t)k));
                    acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
                }
                const float xs = p.xscale[cb0 + b];
                const int row = mt * kTcRows + r0;
                if (p.swiglu) {          // rows r0, r0 + 1 and r0 + 2, r0 + 3 are two (gate, up) pairs
                    if (row + 0 < p.N) store_h(p, cb0 + b, (row >> 1) + 0, acc.x * xs, acc.y * xs);
                    if (row + 2 < p.N) store_h(p, cb0 + b, (row >> 1) + 1, acc.z * xs, acc.w * xs);
                } else {
                    if (row + 0 < p.N) store_y(p, cb0 + b, row + 0, acc.x * xs);
                    if (row + 1 < p.N) store_y(p, cb0 + b, row + 1, acc.y * xs);
                    if (row + 2 < p.N) store_y(p, cb0 + b, row + 2, acc.z * xs);
                    if (row + 3 < p.N) store_y(p, cb0 + b, row + 3, acc.w * xs);
                }
            }
        }
        cluster_sync();
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
    int Bp, Mt, Ks, chunks;
    size_t smem, off_scale, ws_total;   // one chunk of <= 64 rows at a time (the minimum scratch)
    // Every chunk staged at once, one launch pair for the whole batch: chunks
    // of 64 rows (narrow) or of 128 (wide mode); the scratch covers both.
    int nbc_n, Bp_n, nbc_w, Bp_w;
    size_t ws_all;
};

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

size_t tc_smem(int Bp) {
    const size_t need = 1024 + (size_t)kTcWSlots * kTcWSlotBytes + (size_t)kTcStages * 2 * 128 * Bp +
                        8 * (2 * kTcWSlots + 3 * kTcStages + 1) + 16;
    return std::max<size_t>(need, 120 * 1024);      // keeps a second CTA off the SM
}

void tc_set_attrs(cudaError_t* err) { *err = func_attrs((const void*)k_gemv_tc, 227 * 1024, true); }

// Co-resident clusters of size ks for this kernel (0 when the query fails).
int tc_max_clusters(int ks, size_t smem) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(ks * 256));
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (const void*)k_gemv_tc, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

// K split: the cluster size that minimises (waves of clusters) x (chunks per
// CTA + one chunk of fixed cost); every CTA keeps at least two chunks.
int tc_pick_ks(int Mt, int chunks, size_t smem) {
    static std::mutex mu;
    static std::map<std::pair<int, int>, int> memo;   // (Mt, chunks) per smem class
    const int key_smem = (int)(smem >> 10);
    std::lock_guard<std::mutex> lk(mu);
    auto key = std::make_pair(Mt * 4096 + key_smem, chunks);
    auto it = memo.find(key);
    if (it != memo.end()) return it->second;
    const int sms = sm_count();
    int best = 1;
    double best_cost = (double)((Mt + sms - 1) / sms) * (chunks + 1);
    for (int ks = 2; ks <= 16 && chunks / ks >= 2; ++ks) {
        const int mc = tc_max_clusters(ks, smem);
        if (mc <= 0) continue;
        const double cost = (double)((Mt + mc - 1) / mc) * ((chunks + ks - 1) / ks + 1);
        if (cost < best_cost - 1e-9) { best_cost = cost; best = ks; }
    }
    memo[key] = best;
    return best;
}

TcPlan tc_plan(int64_t B, int64_t N, int64_t K) {
    TcPlan pl{};
    const int64_t Bc = std::min<int64_t>(B, kTcMaxB);
    pl.Bp = (int)((Bc + 15) / 16 * 16);
    pl.Mt = (int)((N + kTcRows - 1) / kTcRows);
    pl.chunks = (int)(K / (kTcStepK * kTcChunkSteps));
    pl.smem = tc_smem(pl.Bp);
    pl.Ks = 1;
    pl.off_scale = align256((size_t)pl.Bp * K * 2);
    pl.ws_total = pl.off_scale + 256;
    pl.nbc_n = (int)((B + kTcMaxB - 1) / kTcMaxB);
    pl.Bp_n = pl.nbc_n == 1 ? pl.Bp : kTcMaxB;
    pl.nbc_w = (int)((B + kTcWideB - 1) / kTcWideB);
    pl.Bp_w = B <= kTcMaxB ? pl.Bp_n : (pl.nbc_w == 1 ? (int)((B + 15) / 16 * 16) : kTcWideB);
    const size_t rows = (size_t)std::max(pl.nbc_n * pl.Bp_n, pl.nbc_w * pl.Bp_w);
    pl.ws_all = align256(rows * K * 2) + align256(rows * 4);
    return pl;
}

}  // namespace

bool tc_supported(int64_t B, int64_t N, int64_t K) {
    return B >= 1 && N >= 1 && N <= (1LL << 30) && K >= 1024 && K % 1024 == 0 && K <= (1LL << 20) &&
           (int64_t)N * (K / 8) < (1LL << 40);
}

size_t tc_workspace_bytes(int64_t B, int64_t N, int64_t K) {
    if (!tc_supported(B, N, K)) return 0;
    return tc_plan(B, N, K).ws_all;
}

size_t tc_min_workspace_bytes(int64_t B, int64_t N, int64_t K) {
    if (!tc_supported(B, N, K)) return 0;
    return tc_plan(B, N, K).ws_total;
}

int tc_launch_count(int64_t B, int64_t N, int64_t K) {
    if (!tc_supported(B, N, K)) return 0;
    return 2;   // with tc_workspace_bytes() of scratch; less scratch: two per 64-row chunk
}

namespace {

cudaError_t launch_tc_main(const CUtensorMap& tm_bits, const CUtensorMap& tm_x, const TcParams& prm, int Mt,
                           int nbc, size_t smem, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(Mt * prm.Ks), (unsigned)nbc);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)prm.Ks;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    void* args[] = {(void*)&tm_bits, (void*)&tm_x, (void*)&prm};
    return cudaLaunchKernelExC(&cfg, (const void*)k_gemv_tc, args);
}

}  // namespace

cudaError_t launch_gemv_tc(const GemvArgs& a) {
    if (!tc_supported(a.B, a.N, a.K)) return cudaErrorNotSupported;
    TcPlan pl = tc_plan(a.B, a.N, a.K);
    if (!a.workspace || a.ws_bytes < pl.ws_total) return cudaErrorInvalidValue;
    auto enc = tc_encode();
    if (!enc) return cudaErrorNotSupported;
    cudaError_t e;
    tc_set_attrs(&e);
    if (e != cudaSuccess) return e;
    // All batch chunks in one launch pair when the scratch holds them.  Narrow
    // (64-row chunks, K split over a cluster) or wide (128-row chunks: each
    // weight tile unpacked once for 128 rows, but no K split, since the
    // cluster reduction stages at most 64 rows): the smaller estimate of waves
    // x chunks per CTA, a wide chunk step costing about 1.4 narrow ones
    // (measured).
    const bool one = a.B > kTcMaxB && a.ws_bytes >= pl.ws_all;
    int nbc = 1;
    if (one) {
        const int sms = std::max(1, sm_count());
        const int ks_n = tc_pick_ks(pl.Mt * pl.nbc_n, pl.chunks, tc_smem(pl.Bp_n));
        const double cost_n = (double)((pl.Mt * pl.nbc_n * ks_n + sms - 1) / sms) *
                              ((pl.chunks + ks_n - 1) / ks_n + 1);
        const double cost_w = 1.4 * (double)((pl.Mt * pl.nbc_w + sms - 1) / sms) * (pl.chunks + 1);
        const bool wide = cost_w < cost_n;
        nbc = wide ? pl.nbc_w : pl.nbc_n;
        pl.Bp = wide ? pl.Bp_w : pl.Bp_n;
        pl.smem = tc_smem(pl.Bp);
        pl.Ks = wide ? 1 : ks_n;
    } else {
        pl.Ks = tc_pick_ks(pl.Mt, pl.chunks, pl.smem);
    }
    uint8_t* ws = static_cast<uint8_t*>(a.workspace);
    uint16_t* xp = reinterpret_cast<uint16_t*>(ws);
    float* xscale = reinterpret_cast<float*>(ws + pl.off_scale);

    CUtensorMap tm_bits;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)(a.K / 8), (cuuint64_t)a.N};
        const cuuint64_t strides[1] = {(cuuint64_t)(a.K / 8)};
        const cuuint32_t box[2] = {16 * kTcChunkSteps, (cuuint32_t)kTcRows};
        const cuuint32_t es[2] = {1, 1};
        if (enc(&tm_bits, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, (void*)a.bits, dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const size_t ysz = a.y_bf16 ? 2 : 4;
    // All batch chunks in one prep + one main launch (grid y = chunk) when the
    // scratch holds every chunk's activations; else one pair per 64-row chunk.
    const int nbc_launch = nbc;
    if (one) xscale = reinterpret_cast<float*>(ws + align256((size_t)nbc * pl.Bp * a.K * 2));
    for (int64_t b0 = 0; b0 < a.B; b0 += one ? a.B : (int64_t)kTcMaxB) {
        const int Bc = (int)std::min<int64_t>(kTcMaxB, a.B - b0);
        const int Bp = one ? pl.Bp : (Bc + 15) / 16 * 16;
        const int rows = Bp * nbc_launch;                  // x' rows this launch pair stages
        const uint16_t* xin = a.x + b0 * a.K;
        int Bci = (int)std::min<int64_t>(a.B - b0, (int64_t)rows), Ki = (int)a.K;
        void* prep_args[] = {(void*)&xin, (void*)&Bci, (void*)&Ki, (void*)&xp, (void*)&xscale};
        e = launch((const void*)k_tc_prep, dim3((unsigned)rows), dim3(kTcPrepThreads), 0, a.stream, a.pdl || b0 > 0,
                   prep_args);
        if (e != cudaSuccess) return e;
        // activations: [K/64 slabs][rows][64 inputs], one box = 2 slabs x Bp rows
        CUtensorMap tm_x;
        {
            const cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(a.K / 64)};
            const cuuint64_t strides[2] = {(cuuint64_t)(a.K * 2), 128};
            const cuuint32_t box[3] = {64, (cuuint32_t)Bp, 2};
            const cuuint32_t es[3] = {1, 1, 1};
            if (enc(&tm_x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, (void*)xp, dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return cudaErrorInvalidValue;
        }
        TcParams prm;
        prm.scales = a.scales;
        prm.xscale = xscale;
        prm.y = static_cast<uint8_t*>(a.y) + b0 * (a.swiglu ? a.N / 2 : a.N) * ysz;
        prm.N = (int)a.N;
        prm.K = (int)a.K;
        prm.B = Bci;
        prm.Bp = Bp;
        prm.Ks = pl.Ks;
        prm.chunks = pl.chunks;
        prm.y_bf16 = a.y_bf16;
        prm.stages = 4 * Bp <= 128 ? 3 : 2;
        prm.swiglu = a.swiglu ? 1 : 0;
        e = launch_tc_main(tm_bits, tm_x, prm, pl.Mt, nbc_launch, pl.smem, a.stream);
        if (e != cudaSuccess) return e;
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
