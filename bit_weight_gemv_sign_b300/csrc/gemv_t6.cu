// GEMV / skinny GEMM over packed sign bits with 6-bit fp16 lookup tables, one
// row per lane, TMA-staged weights and split-K over a thread-block cluster
// (CUDA cores, sm_103a); NB = 1..8 batch rows per launch.
//
// What it computes: y[b][n] = sum_g s[n][g] * sum_{k in g} (bit(n,k) ? x[b][k] : -x[b][k])
// (web page "Bonsai 27B: 노트북과 폰에서 실행되는 27B급 이진 및 삼진 저비트 LLM",
// section "이진(Binary) 가중치 형식"), the fp16 group scale applied inside the
// product and fp32 accumulation (section "하이브리드 어텐션을 위한 저비트 커널").
// No multiply per weight: six weights cost one table lookup and one add (the
// ±1 weights of "PrismML Bonsai — 1.15GB짜리 8B 모델이 말이 되나?", section
// "1-bit이 뭔지부터", turn the product into additions and subtractions).
//
// Design (B300: LDS serves 32 lanes per clock per SM, integer ALU ops issue at
// half rate, so a per-weight instruction is unaffordable at HBM speed):
//  * A group of 128 weights is cut into 21 six-bit fields and one two-bit
//    field.  For every field the CTA precomputes the 64 sums
//    T[e] = sum_t (bit t of e ? +x'_t : -x'_t) once, rounded to fp16 and packed
//    two per word: a table is 128 contiguous bytes = the 32 banks, so a warp
//    whose lanes pick any 32 entries of the same table is conflict-free.
//  * Lane l of a warp owns row 32*b + l; all lanes walk the same fields in
//    lockstep, so one shared table serves the whole warp and every CTA.
//  * Batch rows: every batch row has its own tables; a lane reads its 16
//    bytes of sign bits once per group and looks them up in each batch row's
//    tables (the lookups, not the weight reads, grow with the batch).
//  * x' = x * 2^-m_g per group (exact power-of-two prescale) keeps every entry
//    within fp16 range; the entry rounding error is <= 2^-11 of the sum of the
//    six |x'| (round to nearest, 11 significant bits), i.e. a relative 4.9e-4
//    of sum|s x| at most, inside the 1e-3 budget.  The group's fp32 partial
//    is multiplied by s_g and 2^m_g.
//  * Weights and scales of 32-row blocks are copied by TMA into per-warp
//    rings (mbarrier completion, bounded waits).  Bits arrive as 2-D boxes of
//    [32 rows][128 B] (8 groups) with 128-byte swizzle: row r's 16-byte chunk
//    c lands at r*128 + ((c ^ (r % 8)) * 16), so the 32 lanes' 16-byte reads
//    of one group are bank-conflict-free.
//  * K is split over the Q CTAs of a cluster: each builds only its K/Q slice of
//    tables; the per-row partials are summed in a fixed order through
//    distributed shared memory (deterministic, so a flipped row negates
//    exactly).  When a CTA has few row blocks (short N), each block is shared
//    by KW warps that take disjoint group ranges of its slice, so the CTA
//    still runs up to 16 warps; their partials join the same fixed-order sum.
//  * The weight stream of the first stages is issued before
//    griddepcontrol.wait (programmatic dependent launch): only x depends on
//    the preceding kernel.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>
#include <utility>
#include <vector>

#include "common.cuh"
#include "internal.h"
#include "t6_common.cuh"

namespace bit1 {

constexpr int kT6MaxWarps = 16;
constexpr int kT6MaxSmem = 227 * 1024;

__device__ unsigned int g_bit1_wait_timeouts = 0;

struct T6Params {
    const uint16_t* x;        // [NB][K] bf16
    void* y;                  // [NB][N]
    int N, K, Gc, Q, S, stage_bytes, y_bf16;
    int prow;                 // rows per batch row in the partials area (32 x blocks per cluster)
    int KW;                   // warps sharing one row block, each on Gc/KW of its groups (1: no split)
    uint32_t off_tables, off_factors, off_x, off_partials, off_bars;
    int swiglu;               // rows are (gate, up) pairs; y is h = silu(gate) * up, [NB][N/2]
};

// ---------------------------------------------------------------- kernel
// One CTA per SM (its shared memory sees to that), so all registers are usable.
template <int NB, bool SPLIT>
__global__ void __launch_bounds__(kT6MaxWarps * 32, 1)
k_gemv_t6(const __grid_constant__ CUtensorMap tm_bits, const __grid_constant__ CUtensorMap tm_sc,
          const __grid_constant__ T6Params p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = (uint32_t)__cvta_generic_to_shared(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, W = blockDim.x >> 5;
    // Warp = (row-block slot wb, K part kw).  With KW > 1 the planner gives
    // every slot exactly one block, loaded once (no stage reuse), and the KW
    // warps of a slot read disjoint group ranges of the same stage.
    const int KW = SPLIT ? p.KW : 1, wb = SPLIT ? warp / KW : warp, kw = warp - wb * KW, WB = W / KW;
    uint32_t q;
    asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(q));
    const int ncl = gridDim.x / p.Q, cl = blockIdx.x / p.Q;
    const int RB = (p.N + 31) >> 5;
    const int rb0 = (int)((int64_t)RB * cl / ncl), rb1 = (int)((int64_t)RB * (cl + 1) / ncl);
    const int Gc = p.Gc, S = p.S;
    const int g0 = (int)q * Gc;
    const uint32_t bits_tile = 32u * Gc * 16u, sc_tile = 32u * Gc * 2u;
    const uint32_t bars = base + p.off_bars + (uint32_t)(wb * S) * 8u;

    auto issue = [&](int k) {  // lane 0 of K part 0: block rb0 + wb + k*WB -> stage k % S
        const int b = rb0 + wb + k * WB;
        if (b >= rb1) return;
        const uint32_t st = base + (uint32_t)(wb * S + (k % S)) * p.stage_bytes;
        const uint32_t bar = bars + 8u * (k % S);
        mbar_expect_tx(bar, bits_tile + sc_tile);
        for (int j = 0; j < Gc / 8; ++j)   // 128-byte column j of the slice: groups g0+8j .. g0+8j+7
            tma_2d(st + 4096u * j, &tm_bits, (g0 + 8 * j) * 16, b * 32, bar);
        tma_2d(st + bits_tile, &tm_sc, g0, b * 32, bar);
    };
    if (lane == 0 && kw == 0) {
        for (int s = 0; s < S; ++s) mbar_init(bars + 8u * s, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        for (int k = 0; k < S; ++k) issue(k);
    }
    __syncwarp();

    // Activations come from the preceding kernel of a decode step.
    pdl_wait();
    float* fac = reinterpret_cast<float*>(sm + p.off_factors);   // [NB][2*Gc]: 2^m_g, then 2^-m_g
    uint16_t* xs = reinterpret_cast<uint16_t*>(sm + p.off_x);     // [NB][Gc*128] bf16 activations
    for (int i = threadIdx.x; i < NB * Gc * 16; i += blockDim.x) { // 8 activations per thread
        const int b = i / (Gc * 16), j = i - b * (Gc * 16);
        reinterpret_cast<uint4*>(xs)[i] = reinterpret_cast<const uint4*>(p.x + (size_t)b * p.K + (size_t)g0 * 128)[j];
    }
    __syncthreads();
    for (int bg = warp; bg < NB * Gc; bg += W) {
        const int b = bg / Gc, g = bg - b * Gc;
        const uint2 xv = *reinterpret_cast<const uint2*>(xs + bg * 128 + 4 * lane);
        float m = fmaxf(fmaxf(fabsf(bf16_bits_to_f32(xv.x & 0xffffu)), fabsf(bf16_bits_to_f32(xv.x >> 16))),
                        fmaxf(fabsf(bf16_bits_to_f32(xv.y & 0xffffu)), fabsf(bf16_bits_to_f32(xv.y >> 16))));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        int mg = 0;
        if (m > 0.f) {
            const int e = (int)((__float_as_uint(m) >> 23) & 0xffu) - 127;  // floor(log2 m), normal m
            mg = min(max(e - 11, -126), 127);                                // max|x'| < 2^12
        }
        if (lane == 0) {
            fac[b * 2 * Gc + g] = __uint_as_float((uint32_t)(mg + 127) << 23);
            fac[b * 2 * Gc + Gc + g] = __uint_as_float((uint32_t)(127 - mg) << 23);
        }
    }
    __syncthreads();
    uint8_t* tabs = sm + p.off_tables;   // [NB][Gc][22 tables]
    for (int t = threadIdx.x; t < NB * Gc * kT6Fields * 4; t += blockDim.x) {
        const int tt = t >> 2, bg = tt / kT6Fields, f = tt - bg * kT6Fields;
        const int b = bg / Gc, g = bg - b * Gc;
        t6_build_pair(tabs + bg * kT6GroupBytes + f * kT6TableBytes, xs + bg * 128, fac[b * 2 * Gc + Gc + g], f,
                      t & 3, tt & 1);
    }
    __syncthreads();
    pdl_launch_dependents();

    float* partials = reinterpret_cast<float*>(sm + p.off_partials);
    const uint32_t tb = base + p.off_tables;
    bool ok = true;
    int k = 0;
    if constexpr (!SPLIT) {
      for (;; ++k) {
        const int b = rb0 + warp + k * W;
        if (b >= rb1) break;
        const int s = k % S;
        if (!mbar_wait(bars + 8u * s, (uint32_t)(k / S) & 1u)) {
            if (lane == 0) atomicOr(&g_bit1_wait_timeouts, 1u);
            ok = false;
            break;
        }
        const uint32_t st = base + (uint32_t)(warp * S + s) * p.stage_bytes;
        const uint32_t sts = st + bits_tile + (uint32_t)lane * Gc * 2u;
        float acc[NB];
#pragma unroll
        for (int bb = 0; bb < NB; ++bb) acc[bb] = 0.f;
        for (int g8 = 0; g8 < Gc; g8 += 8) {
            const uint4 sv = lds128(sts + 2u * g8);
            const uint32_t svw[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int g = g8 + j;
                // box g8/8 holds [32 rows][128 B]; 128-byte swizzle of chunk j in row `lane`
                const uint32_t L = ((uint32_t)g8 << 9) + (uint32_t)lane * 128u +
                                   ((uint32_t)(j ^ (lane & 7)) << 4);
                const uint4 wv = lds128(st + L);
                const uint32_t w[4] = {wv.x, wv.y, wv.z, wv.w};
                const float sc = f16_bits_to_f32((uint16_t)(svw[j >> 1] >> (16 * (j & 1))));
#pragma unroll
                for (int bb = 0; bb < NB; ++bb) {
                    const float part = t6_group(w, tb + (uint32_t)((bb * Gc + g) * kT6GroupBytes),
                                                std::make_index_sequence<kT6Fields>{});
                    acc[bb] = fmaf(part * sc, fac[bb * 2 * Gc + g], acc[bb]);
                }
            }
        }
#pragma unroll
        for (int bb = 0; bb < NB; ++bb) partials[bb * p.prow + (b - rb0) * 32 + lane] = acc[bb];
        __syncwarp();
        if (lane == 0) issue(k + S);
      }
    } else {
        // K split inside the CTA: this warp's block (one per slot, loaded once
        // into stage 0 of the slot), groups [g_lo, g_hi) of the slice.
        const int b = rb0 + wb;
        const int g_lo = kw * (Gc / KW), g_hi = g_lo + Gc / KW;
        if (b < rb1) {
            if (!mbar_wait(bars, 0u)) {
                if (lane == 0) atomicOr(&g_bit1_wait_timeouts, 1u);
                ok = false;
            } else {
                const uint32_t st = base + (uint32_t)(wb * S) * p.stage_bytes;
                const uint32_t sts = st + bits_tile + (uint32_t)lane * Gc * 2u;
                float acc[NB];
#pragma unroll
                for (int bb = 0; bb < NB; ++bb) acc[bb] = 0.f;
                for (int g = g_lo; g < g_hi; ++g) {
                    const uint32_t L = ((uint32_t)(g & ~7) << 9) + (uint32_t)lane * 128u +
                                       ((uint32_t)((g & 7) ^ (lane & 7)) << 4);
                    const uint4 wv = lds128(st + L);
                    const uint32_t w[4] = {wv.x, wv.y, wv.z, wv.w};
                    unsigned short sh;
                    asm volatile("ld.shared.b16 %0, [%1];" : "=h"(sh) : "r"(sts + 2u * (uint32_t)g));
                    const float sc = f16_bits_to_f32(sh);
#pragma unroll
                    for (int bb = 0; bb < NB; ++bb) {
                        const float part = t6_group(w, tb + (uint32_t)((bb * Gc + g) * kT6GroupBytes),
                                                    std::make_index_sequence<kT6Fields>{});
                        acc[bb] = fmaf(part * sc, fac[bb * 2 * Gc + g], acc[bb]);
                    }
                }
#pragma unroll
                for (int bb = 0; bb < NB; ++bb)
                    partials[(kw * NB + bb) * p.prow + (b - rb0) * 32 + lane] = acc[bb];
            }
        }
        k = 1;
    }
    if (!ok && lane == 0) {
        // Give copies still in flight a bounded chance to land before exit.
        for (int kk = k + 1; kk < k + S; ++kk)
            if (rb0 + wb + kk * WB < rb1) (void)mbar_wait(bars + 8u * (kk % S), (uint32_t)(kk / S) & 1u);
    }

    // Sum the Q partials of every row in a fixed order.
    __syncthreads();
    cluster_sync();
    const int R = (rb1 - rb0) * 32;
    const uint32_t part_s = base + p.off_partials;
    auto row_sum = [&](int b, int i) {
        float v = 0.f;
        for (int r = 0; r < p.Q; ++r) {
            if constexpr (SPLIT) {
                for (int j = 0; j < KW; ++j)
                    v += ld_cluster_f32(part_s + 4u * (uint32_t)((j * NB + b) * p.prow + i), (uint32_t)r);
            } else {
                v += ld_cluster_f32(part_s + 4u * (uint32_t)(b * p.prow + i), (uint32_t)r);
            }
        }
        return v;
    };
    if (p.swiglu) {
        // SwiGLU pairs (rows 2m, 2m+1 = gate, up of unit m; the Bonsai 27B
        // page, section "Bonsai 27B의 표현 방식"): the ranks split the pairs, one
        // thread sums both rows of a pair and writes h = silu(g) * u.
        const int P = R / 2;
        const int lo = (int)((int64_t)P * q / p.Q), hi = (int)((int64_t)P * (q + 1) / p.Q);
        for (int b = 0; b < NB; ++b)
        for (int m = lo + threadIdx.x; m < hi; m += blockDim.x) {
            const float g = row_sum(b, 2 * m), u = row_sum(b, 2 * m + 1);
            const int row = rb0 * 32 + 2 * m;
            if (row < p.N) {
                const float h = g / (1.f + expf(-g)) * u;
                const int64_t o = (int64_t)b * (p.N >> 1) + (row >> 1);
                if (p.y_bf16) reinterpret_cast<uint16_t*>(p.y)[o] = f32_to_bf16_bits(h);
                else reinterpret_cast<float*>(p.y)[o] = h;
            }
        }
    } else {
        const int lo = (int)((int64_t)R * q / p.Q), hi = (int)((int64_t)R * (q + 1) / p.Q);
        for (int b = 0; b < NB; ++b)
        for (int i = lo + threadIdx.x; i < hi; i += blockDim.x) {
            const float v = row_sum(b, i);
            const int row = rb0 * 32 + i;
            if (row < p.N) {
                if (p.y_bf16) reinterpret_cast<uint16_t*>(p.y)[(int64_t)b * p.N + row] = f32_to_bf16_bits(v);
                else reinterpret_cast<float*>(p.y)[(int64_t)b * p.N + row] = v;
            }
        }
    }
    cluster_sync();
}

// ---------------------------------------------------------------- host side
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

struct T6Plan {
    int Q = 0, Gc = 0, W = 0, S = 0, ncl = 0, stage_bytes = 0;
    size_t smem = 0;
    T6Params p{};
};

constexpr int kT6MaxNB = 8;

template <bool SPLIT>
const void* t6_kernel_s(int nb) {
    switch (nb) {
        case 1: return (const void*)k_gemv_t6<1, SPLIT>;
        case 2: return (const void*)k_gemv_t6<2, SPLIT>;
        case 3: return (const void*)k_gemv_t6<3, SPLIT>;
        case 4: return (const void*)k_gemv_t6<4, SPLIT>;
        case 5: return (const void*)k_gemv_t6<5, SPLIT>;
        case 6: return (const void*)k_gemv_t6<6, SPLIT>;
        case 7: return (const void*)k_gemv_t6<7, SPLIT>;
        case 8: return (const void*)k_gemv_t6<8, SPLIT>;
        default: return nullptr;
    }
}

// The kernel for nb batch rows, with (kw > 1) or without the in-CTA K split.
const void* t6_kernel(int nb, int kw) { return kw > 1 ? t6_kernel_s<true>(nb) : t6_kernel_s<false>(nb); }

// Cluster sizes that split G into slices of a multiple of 8 groups whose
// tables (NB batch rows) fit comfortably in shared memory, most preferred
// first.  Sizes above 8 are non-portable clusters (allowed on this part up to
// 16): they let several batch rows' tables fit for long K (K = 12288 at four
// rows needs slices of 8 groups, a cluster of 12).
int q_candidates(int64_t G, int nb, int* out) {
    int n = 0;
    if (G % 8 != 0) return 0;
    const int64_t u = G / 8;  // units of 8 groups
    for (int q : {4, 2, 1, 5, 3, 7, 6, 8, 12, 10, 16})
        if (u % q == 0 && (G / q) * kT6GroupBytes * nb <= 150 * 1024) out[n++] = q;
    return n;
}

cudaError_t t6_set_attrs(const void* fn) { return func_attrs(fn, kT6MaxSmem, true); }

// Clusters of size Q that can be resident at once with this kernel, block
// size and shared memory (clusters must fit inside one GPC, so this can be
// less than SMs / Q); cached per configuration.
int active_clusters(const void* fn, int Q, int threads, size_t smem) {
    struct Key { const void* fn; int Q, threads; size_t smem; int n; };
    static std::mutex mu;
    static std::vector<Key> cache;
    std::lock_guard<std::mutex> lk(mu);
    for (auto& c : cache)
        if (c.fn == fn && c.Q == Q && c.threads == threads && c.smem == smem) return c.n;
    int n = 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(Q * (sm_count() / Q)));
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)Q;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (t6_set_attrs(fn) != cudaSuccess || cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        int devices = 0;
        const bool no_device = cudaGetDeviceCount(&devices) != cudaSuccess || devices == 0;
        cudaGetLastError();
        n = no_device ? sm_count() / Q : 0;  // host-only checks: assume every SM; on a GPU: unusable
    }
    cache.push_back({fn, Q, threads, smem, n});
    return n;
}

bool plan_t6_q(int64_t N, int64_t K, int Q, int nb, T6Plan& pl) {
    const int64_t G = K / 128;
    pl.Q = Q;
    pl.Gc = (int)(G / Q);
    pl.stage_bytes = (32 * pl.Gc * 18 + 1023) & ~1023;
    const int tables = nb * pl.Gc * kT6GroupBytes;
    const int factors = nb * pl.Gc * 8;
    const int xbytes = nb * pl.Gc * 128 * 2;
    const int64_t RB = (N + 31) / 32;
    auto total = [&](int W, int S, int bpc, int KW) {
        return (size_t)1024 + (size_t)(W / KW) * S * pl.stage_bytes + tables + factors + xbytes +
               (size_t)nb * bpc * 128 * KW + (size_t)(W / KW) * S * 8 + 64;
    };
    // first guess with every SM, then shrink to the clusters that fit at once
    int ncl = sm_count() / Q;
    if (ncl < 1) return false;
    int W = 0, S = 0, bpc = 0, KW = 1;
    for (int iter = 0; iter < 3; ++iter) {
        bpc = (int)((RB + ncl - 1) / ncl);
        // Few row blocks per CTA: give each block KW warps, each on Gc/KW of
        // its groups (whole 8-group boxes or fewer than 8 groups), so that
        // the CTA still runs up to 16 warps.  Each block is then loaded once.
        KW = 1;
        for (int kw : {8, 4, 2}) {
            const int gp = pl.Gc / kw;
            if (bpc * kw <= kT6MaxWarps && pl.Gc % kw == 0 && (gp < 8 || gp % 8 == 0) &&
                total(bpc * kw, 1, bpc, kw) <= kT6MaxSmem) {
                KW = kw;
                break;
            }
        }
        if (KW > 1) {
            W = bpc * KW;
            S = 1;
        } else {
            W = bpc < kT6MaxWarps ? bpc : kT6MaxWarps;
            if (W < 4) W = 4;  // at least 4 warps: they share the table build
            S = (bpc + W - 1) / W;
            if (S > 3) S = 3;
            while (total(W, S, bpc, 1) > kT6MaxSmem && S > 1) --S;
            while (total(W, S, bpc, 1) > kT6MaxSmem && W > 4) --W;
            if (total(W, S, bpc, 1) > kT6MaxSmem) return false;
        }
        const int act = active_clusters(t6_kernel(nb, KW), Q, W * 32, total(W, S, bpc, KW));
        if (act < 1) return false;            // this cluster size cannot run here
        if (act >= ncl) break;
        ncl = act;
    }
    pl.ncl = ncl;
    pl.W = W;
    pl.S = S;
    pl.smem = total(W, S, bpc, KW);
    uint32_t off = (uint32_t)((W / KW) * S * pl.stage_bytes);
    pl.p.off_tables = off;        off += tables;           // multiple of 128 (stages are 1 KB multiples)
    pl.p.off_factors = off;       off += factors;          // 16-byte aligned (tables multiple of 128)
    off = (off + 15u) & ~15u;
    pl.p.off_x = off;             off += xbytes;
    pl.p.off_partials = off;      off += nb * bpc * 128 * KW;
    off = (off + 7u) & ~7u;
    pl.p.off_bars = off;
    pl.p.N = (int)N;
    pl.p.K = (int)K;
    pl.p.Gc = pl.Gc;
    pl.p.Q = Q;
    pl.p.S = S;
    pl.p.stage_bytes = pl.stage_bytes;
    pl.p.prow = bpc * 32;
    pl.p.KW = KW;
    return true;
}

// Relative time of a plan, in units of one warp's work on one 32-row block of
// one group: a warp runs ceil(bpc / WB) blocks of Gc / KW groups back to back
// (its dependent chain), an SM issues about eight warps' worth at once, and the
// table build (about 0.75 units per group, spread over the W warps) comes
// first.  More SMs with fewer warps each can lose: half the warps per CTA and
// twice the K per CTA doubles every warp's chain.
double t6_estimate(const T6Plan& pl) {
    const int bpc = pl.p.prow / 32, KW = pl.p.KW, WB = pl.W / KW;
    const double chain = (double)((bpc + WB - 1) / WB) * pl.Gc / KW;
    return std::max(chain, bpc * pl.Gc / 8.0) + 0.75 * pl.Gc / pl.W;
}

// Among the usable cluster sizes, take the plan with the smallest estimate
// (ties: more SMs busy).
bool plan_t6(int64_t N, int64_t K, int nb, T6Plan& best) {
    if (N < 1 || N > (1LL << 30) || nb < 1 || nb > kT6MaxNB) return false;
    int qs[16];
    const int nq = q_candidates(K / 128, nb, qs);
    bool found = false;
    double best_est = 0.0;
    for (int i = 0; i < nq; ++i) {
        T6Plan pl;
        if (!plan_t6_q(N, K, qs[i], nb, pl)) continue;
        const double est = t6_estimate(pl);
        if (!found || est < best_est - 1e-9 ||
            (est < best_est + 1e-9 && pl.ncl * pl.Q > best.ncl * best.Q)) {
            best = pl;
            best_est = est;
            found = true;
        }
    }
    return found;
}

// Largest batch rows per launch: the largest NB <= min(B, 8) that has a plan.
int t6_chunk(int64_t B, int64_t N, int64_t K) {
    for (int nb = (int)std::min<int64_t>(B, kT6MaxNB); nb >= 1; --nb) {
        T6Plan pl;
        if (plan_t6(N, K, nb, pl)) return nb;
    }
    return 0;
}

cudaError_t launch_t6_chunk(const GemvArgs& a, int nb, const uint16_t* x, void* y, bool pdl) {
    T6Plan pl;
    if (!plan_t6(a.N, a.K, nb, pl)) return cudaErrorNotSupported;
    auto enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const int64_t G = a.K / 128;
    CUtensorMap tm_bits, tm_sc;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)(a.K / 8), (cuuint64_t)a.N};
        const cuuint64_t strides[1] = {(cuuint64_t)(a.K / 8)};
        const cuuint32_t box[2] = {128, 32};
        const cuuint32_t es[2] = {1, 1};
        if (enc(&tm_bits, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, (void*)a.bits, dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[2] = {(cuuint64_t)G, (cuuint64_t)a.N};
        const cuuint64_t strides[1] = {(cuuint64_t)(G * 2)};
        const cuuint32_t box[2] = {(cuuint32_t)pl.Gc, 32};
        const cuuint32_t es[2] = {1, 1};
        if (enc(&tm_sc, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, (void*)a.scales, dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const void* fn = t6_kernel(nb, pl.p.KW);
    {
        const cudaError_t e = t6_set_attrs(fn);
        if (e != cudaSuccess) return e;
    }
    T6Params prm = pl.p;
    prm.x = x;
    prm.y = y;
    prm.y_bf16 = a.y_bf16;
    prm.swiglu = a.swiglu ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(pl.ncl * pl.Q));
    cfg.blockDim = dim3((unsigned)(pl.W * 32));
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)pl.Q;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    int na = 1;
    if (pdl) {
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        na = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    void* args[] = {(void*)&tm_bits, (void*)&tm_sc, (void*)&prm};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace

bool t6_supported(int64_t B, int64_t N, int64_t K) {
    int qs[16];
    return B >= 1 && K % 1024 == 0 && K <= (1LL << 20) && q_candidates(K / 128, 1, qs) > 0 && N >= 1 &&
           N <= (1LL << 30);
}

int t6_launch_count(int64_t B, int64_t N, int64_t K) {
    if (!t6_supported(B, N, K)) return 0;
    const int nb = t6_chunk(B, N, K);
    return nb > 0 ? (int)((B + nb - 1) / nb) : 0;
}

cudaError_t launch_gemv_t6(const GemvArgs& a) {
    if (!t6_supported(a.B, a.N, a.K)) return cudaErrorNotSupported;
    const int nb = t6_chunk(a.B, a.N, a.K);
    if (nb < 1) return cudaErrorNotSupported;
    const size_t ysz = a.y_bf16 ? 2 : 4;
    // ceil(B / nb) launches with balanced batch chunks (8 rows at nb = 6 run
    // as 4 + 4, not 6 + 2).
    const int64_t chunks = (a.B + nb - 1) / nb;
    for (int64_t i = 0, b0 = 0; i < chunks; ++i) {
        const int n = (int)(a.B / chunks + (i < a.B % chunks ? 1 : 0));
        const int64_t yrow = a.swiglu ? a.N / 2 : a.N;    // outputs per batch row
        const cudaError_t e = launch_t6_chunk(a, n, a.x + b0 * a.K, static_cast<uint8_t*>(a.y) + b0 * yrow * ysz,
                                              a.pdl || b0 > 0);
        if (e != cudaSuccess) return e;
        b0 += n;
    }
    return cudaSuccess;
}

// Self-test of the bounded wait: one thread waits on an mbarrier phase that
// nothing completes.  The wait gives up after its iteration limit, records
// the event in the timeout counter (bit 4) and the kernel returns normally:
// the failure path of every bounded wait, exercised without a fault or hang.
__global__ void __launch_bounds__(32, 1) k_wait_selftest(unsigned int* __restrict__ done) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = (uint32_t)__cvta_generic_to_shared(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        // A bound of its own, 2^12 polls (milliseconds), so that the test of
        // the failure path does not hold the GPU for the kernels' 16 s bound.
        if (!mbar_wait_polls(b, 0u, 1u << 12)) atomicOr(&g_bit1_wait_timeouts, 16u);
        *done = 1u;
    }
}

cudaError_t launch_wait_selftest(unsigned int* d_done, cudaStream_t stream) {
    k_wait_selftest<<<1, 32, 0, stream>>>(d_done);
    return cudaGetLastError();
}

unsigned int t6_take_timeouts() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_bit1_wait_timeouts, sizeof(v)) != cudaSuccess) return 0xffffffffu;
    cudaMemcpyToSymbol(g_bit1_wait_timeouts, &zero, sizeof(zero));
    return v;
}

}  // namespace bit1
