// Grouped batched GEMV on the tensor cores: many independent packed-1-bit
// problems sharing one batch size B (1..64) in one persistent tcgen05 launch
// (plus one activation-prep launch), sm_103a.
//
// Each problem is Y[b][n] = sum_k X[b][k] * W[n][k] with W in the binary g128
// format of the web page "Bonsai 27B: 노트북과 폰에서 실행되는 27B급 이진 및
// 삼진 저비트 LLM" (section "이진(Binary) 가중치 형식").  The multi-row pass
// is the verify step of speculative decoding (same page, section "DSpark:
// 추측 디코딩으로 한 번 더 가속": the target model checks the drafted tokens in
// one pass over the weights) and, at larger B, batched decode.
//
// Why a grouped tensor-core launch: at B >= 2 the lookup-table kernels do
// table work per batch row, so their time grows with B; on the tensor cores
// the per-weight work (forming +-s and writing it to tensor memory) is the
// same for every B up to the MMA's N, and one launch over all matrices pays
// the pipeline fill, the tensor-memory allocation and the drain once per SM
// instead of once per matrix.
//
// Design: the arithmetic, operand layouts and warp roles of gemv_tc.cu
// (tc_common.cuh), made persistent.  Work unit: one 256-row tile of one
// problem over its whole K.  The concatenated tiles of all problems are cut
// into one contiguous, cost-balanced range per CTA (one CTA per SM); every
// role walks the same tile sequence, and the rings (sign bits: 4 slots of 4
// steps; A in tensor memory: 2-3 steps; activations in shared memory: up to
// 32 steps) run on without draining at tile boundaries.  After a tile's last step the unpack
// warps wait for its accumulators, read them back and write y (or the SwiGLU
// output); the next tile's first MMA overwrites the accumulators only after
// that (its A operand is written after the read-back).  No split K: every
// output is produced by one accumulator, in a fixed order.
//
// Where the time goes (B300, clock counters inside a copy of this kernel, 8B
// sweep at B = 16): an A stage can be rewritten only after the MMAs that read
// it have completed, which the issuers signal with tcgen05.commit; from the
// commit to the unpack warps seeing the stage free takes 1000-1800 cycles
// (about 1000 even with no MMA in flight), and tensor memory holds three
// steps of A beside the accumulators, so a step costs about a third of that
// round trip, 600-1100 cycles, at any B up to 32.  The unpack itself (one
// shift and one LOP3 per two weights, 64 KB per step written to tensor memory
// at about 340 bytes per cycle) would allow about 300, and the tensor cores
// are mostly idle at these batch sizes.  A deeper activation ring (its copies
// come from L2) removed the waits for B.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstddef>
#include <cstring>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "internal.h"
#include "t6_common.cuh"
#include "tc_common.cuh"

namespace bit1 {

__device__ unsigned int g_tcg_wait_timeouts = 0;

constexpr int kTgRows = 256;              // weight rows per tile (two M = 128 halves)
constexpr int kTgWSlots = 4;              // sign-bit ring slots
constexpr uint32_t kTgWSlotBytes = kTgRows * 16 * kTcChunkSteps;   // 16 KB
constexpr int kTgUnpackWarps = 8;
constexpr int kTgMmaWarps = 4;
constexpr int kTgThreads = 32 * (kTgUnpackWarps + 2 + kTgMmaWarps);
constexpr int kTgMaxCtas = 160;
constexpr int kTgMaxB = 64;
constexpr int kTgMinSmem = 120 * 1024;    // keeps a second CTA (and its tensor-memory allocation) off the SM
constexpr int kTgMaxBStages = 32;         // activation ring: up to 128 KB of shared memory
constexpr uint32_t kTgBRingBytes = 128 * 1024;

struct TgHeader {            // 128 bytes; `kind` where GHeader has it
    int count, nctas, B, Bp;
    int stages, smem_bytes, ranges_off, probs_off;
    int bstages;             // activation (B operand) ring depth
    int pad0[8];
    int kind;                // kPlanKindTensor
    int pad1[14];
};
static_assert(sizeof(TgHeader) == 128, "header size");
static_assert(offsetof(TgHeader, kind) == kPlanKindOffset, "kind offset");

struct TgRange {             // tiles from (p0, t0) up to, not including, (p1, t1)
    int p0, t0, p1, t1;
};

struct alignas(128) TgProb {
    CUtensorMap tm_bits;     // 2-D [N][K/8] uint8, box {64, 256}, 64-byte swizzle
    CUtensorMap tm_x;        // 3-D x' [K/64 slabs][Bp rows][64] fp16, box {64, Bp, 2}, 128-byte swizzle
    const uint16_t* x;       // bf16 [B][K]
    uint16_t* xp;            // workspace: fp16 [Bp][K], permuted and prescaled
    float* xscale;           // workspace: [Bp] powers of two
    const uint16_t* scales;  // fp16 [N][K/128]
    void* y;                 // [B][N] (SwiGLU: [B][N/2]) of y_dtype
    int N, K, tiles, y_bf16, swiglu;
};

// ---------------------------------------------------------------- device
__global__ void __launch_bounds__(kTcPrepThreads) k_tcg_prep(const uint8_t* __restrict__ plan) {
    pdl_wait();
    pdl_launch_dependents();   // the main kernel may start: everything before this one has completed
    const TgHeader* H = reinterpret_cast<const TgHeader*>(plan);
    const TgProb* P = reinterpret_cast<const TgProb*>(plan + H->probs_off);
    const int p = (int)blockIdx.x / H->Bp, b = (int)blockIdx.x % H->Bp;
    const TgProb& q = P[p];
    __shared__ uint32_t red[kTcPrepThreads / 32];
    tc_prep_row(b < H->B ? q.x + (size_t)b * q.K : nullptr, q.K, q.xp + (size_t)b * q.K, q.xscale + b, red);
}

// Shared memory: [sign-bit ring 4 x 16 KB][B ring bstages x 2 x Bp x 128 B][mbarriers][tensor-memory slot].
// The activation ring is deeper than the A stages: its copies come from L2
// with a latency of several steps, and the A stages are bounded by tensor
// memory.
// Tensor memory: accumulator (half h, slice parity q) at columns (2h + q) Bp;
// A stage st, half h at abase + 128 st + 64 h, abase = 4 Bp rounded up to 128.
//
// MMA issue: one thread issues a tcgen05.mma about every 150-200 cycles (the
// cost is per issuing warp; warps issue in parallel), so the 16 MMAs of a
// step (2 halves x 8 slices of 16 inputs) are spread over 4 issuer warps,
// each with its own accumulator.  (Eight issuers with eight accumulators
// measured no faster: the step time is set by the stage round trip, see
// the notes at the top of this file.)
__global__ void __launch_bounds__(kTgThreads, 1) k_gemv_tc_group(const uint8_t* __restrict__ plan) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = (uint32_t)__cvta_generic_to_shared(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const TgHeader* H = reinterpret_cast<const TgHeader*>(plan);
    const TgProb* P = reinterpret_cast<const TgProb*>(plan + H->probs_off);
    const TgRange R = reinterpret_cast<const TgRange*>(plan + H->ranges_off)[blockIdx.x];
    const int Bp = H->Bp, B = H->B, nstg = H->stages, nbs = H->bstages;
    auto ts = [&](int p) { return p == R.p0 ? R.t0 : 0; };
    auto te = [&](int p) { return p == R.p1 ? R.t1 : P[p].tiles; };

    const uint32_t btile = (uint32_t)Bp * 128u;             // one 64-wide K slab of B
    const uint32_t bstage = 2u * btile;                     // one step (128 K)
    const uint32_t wring = base;
    const uint32_t bring = base + kTgWSlots * kTgWSlotBytes;
    const uint32_t bar0 = bring + (uint32_t)nbs * bstage;
    const uint32_t wfull = bar0, wempty = bar0 + 8 * kTgWSlots;
    const uint32_t afull = bar0 + 16 * kTgWSlots, freed = afull + 8 * 3;      // A stages (tensor memory)
    const uint32_t bfull = freed + 8 * 3, bfree = bfull + 8 * kTgMaxBStages;  // B stages (shared memory)
    const uint32_t d_done = bfree + 8 * kTgMaxBStages;
    const uint32_t tslot_s = d_done + 8;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem_raw + (tslot_s - raw));

    if (threadIdx.x == 0) {
        for (int i = 0; i < kTgWSlots; ++i) {
            mbar_init(wfull + 8 * i, 1);
            mbar_init(wempty + 8 * i, kTgUnpackWarps);
        }
        for (int s = 0; s < 3; ++s) {
            mbar_init(afull + 8 * s, kTgUnpackWarps);
            mbar_init(freed + 8 * s, kTgMmaWarps);          // one commit per MMA issuer
        }
        for (int s = 0; s < nbs; ++s) {
            mbar_init(bfull + 8 * s, 1);
            mbar_init(bfree + 8 * s, kTgMmaWarps);
        }
        mbar_init(d_done, kTgMmaWarps);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(tslot_s) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;");
    const uint32_t tmem = *tslot;
    const uint32_t abase = (uint32_t)((4 * Bp + 127) / 128 * 128);

    if (warp < kTgUnpackWarps) {
        // ---- unpack (A into tensor memory) and epilogue: thread = one row of the tile
        const int quad = warp & 3, h = warp >> 2;
        const int r = 128 * h + 32 * quad + lane;          // row within the tile
        const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
        const uint32_t rsw = (uint32_t)(r >> 1) & 3u;      // 64-byte swizzle of this row
        // fp16 scales of this row, 8 groups (16 bytes) per window; the next
        // window (of this tile or of the next) is loaded one window ahead
        auto window = [&](int p, int t, int wd) {
            const TgProb& q = P[p];
            const int row = t * kTgRows + r;
            if (row >= q.N) return make_uint4(0, 0, 0, 0);
            return ldg_nc_v4(q.scales + (size_t)row * (q.K / 128) + 8 * wd);
        };
        // tile after (p, t) in this CTA's range; false at the end
        auto next_tile = [&](int& p, int& t) {
            ++t;
            while (t >= te(p)) {
                if (++p > R.p1) return false;
                t = ts(p);
            }
            return true;
        };
        int gs = 0, tile_i = 0;
        int st = 0, use = 0;                               // A stage of step gs and its use count
        bool ok = true, first = true;
        uint4 sc_cur = make_uint4(0, 0, 0, 0), sc_nxt = sc_cur;
        bool pdl_done = false;
        for (int p = R.p0; p <= R.p1 && ok; ++p) {
            for (int t = ts(p); t < te(p) && ok; ++t) {
                const TgProb& pr = P[p];
                const int nst = pr.K / kTcStepK, nwin = nst / 8;
                const int row = t * kTgRows + r;
                const bool live = row < pr.N;
                if (first) {
                    sc_cur = window(p, t, 0);
                    int pn = p, tn = t;
                    sc_nxt = nwin > 1 ? window(p, t, 1) : (next_tile(pn, tn) ? window(pn, tn, 0) : sc_cur);
                    first = false;
                }
                for (int s = 0; s < nst; ++s, ++gs) {
                    if ((s & 7) == 0 && gs > 0) {
                        sc_cur = sc_nxt;
                        const int wd = s >> 3;
                        if (wd + 1 < nwin) sc_nxt = window(p, t, wd + 1);
                        else {
                            int pn = p, tn = t;
                            if (next_tile(pn, tn)) sc_nxt = window(pn, tn, 0);
                        }
                    }
                    const int c = gs >> 2, i = gs & 3, ws = c & (kTgWSlots - 1);
                    if (use > 0 && !warp_wait(freed + 8 * st, (uint32_t)(use - 1) & 1u)) { ok = false; break; }
                    if (i == 0 && !warp_wait(wfull + 8 * ws, (uint32_t)(c / kTgWSlots) & 1u)) { ok = false; break; }
                    asm volatile("tcgen05.fence::after_thread_sync;");
                    const uint4 w = lds128(wring + ws * kTgWSlotBytes + 64u * r + 16u * ((uint32_t)i ^ rsw));
                    if (i == kTcChunkSteps - 1) {
                        __syncwarp();
                        if (lane == 0) tc_arrive(wempty + 8 * ws);
                    }
                    const uint32_t wsel = (s & 4) ? ((s & 2) ? sc_cur.w : sc_cur.z) : ((s & 2) ? sc_cur.y : sc_cur.x);
                    const uint32_t s16 = (s & 1) ? (wsel >> 16) : (wsel & 0xffffu);
                    const uint32_t s2 = live ? (s16 | (s16 << 16)) : 0u;
                    tc_unpack_step(w, s2, tmem + lane_base + abase + 128u * st + 64u * h);
                    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                    asm volatile("tcgen05.fence::before_thread_sync;");
                    __syncwarp();
                    if (lane == 0) tc_arrive(afull + 8 * st);
                    if (++st == nstg) {
                        st = 0;
                        ++use;
                    }
                }
                if (!ok) break;
                // ---- epilogue of tile (p, t): accumulators of half h, row r
                if (!pdl_done) {
                    pdl_wait();          // y may still be read by the preceding kernel
                    pdl_done = true;
                }
                if (!warp_wait(d_done, (uint32_t)tile_i & 1u)) { ok = false; break; }
                ++tile_i;
                asm volatile("tcgen05.fence::after_thread_sync;");
                for (int cb = 0; cb < Bp; cb += 16) {
                    uint32_t d[16], e[16];           // even and odd slices of half h
                    const uint32_t c0 = lane_base + (uint32_t)(2 * h * Bp + cb);
                    tc_ld16(tmem + c0, d);
                    tc_ld16(tmem + c0 + (uint32_t)Bp, e);
                    tc_wait_ld();
#pragma unroll
                    for (int k = 0; k < 16; ++k) d[k] = __float_as_uint(__uint_as_float(d[k]) + __uint_as_float(e[k]));
                    if (pr.swiglu) {
                        // Lane 2m holds the gate row and lane 2m+1 the up row of unit
                        // row/2.  The pair splits the batch columns: the even lane forms h
                        // for column 2j, the odd lane for column 2j+1, after one exchange.
                        const bool odd = lane & 1;
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int c0 = cb + 2 * j;
                            const float v0 = c0 < B ? __uint_as_float(d[2 * j]) * pr.xscale[c0] : 0.f;
                            const float v1 = c0 + 1 < B ? __uint_as_float(d[2 * j + 1]) * pr.xscale[c0 + 1] : 0.f;
                            const float w = __shfl_xor_sync(0xffffffffu, odd ? v0 : v1, 1);
                            const float g = odd ? w : v0, u = odd ? v1 : w;
                            const int c = c0 + (odd ? 1 : 0);
                            if (live && c < B) {
                                const float hv = __fdividef(g, 1.f + __expf(-g)) * u;
                                const int64_t o = (int64_t)c * (pr.N >> 1) + (row >> 1);
                                if (pr.y_bf16) reinterpret_cast<uint16_t*>(pr.y)[o] = f32_to_bf16_bits(hv);
                                else reinterpret_cast<float*>(pr.y)[o] = hv;
                            }
                        }
                    } else if (live) {
#pragma unroll
                        for (int k = 0; k < 16; ++k) {
                            if (cb + k < B) {
                                const float v = __uint_as_float(d[k]) * pr.xscale[cb + k];
                                const int64_t o = (int64_t)(cb + k) * pr.N + row;
                                if (pr.y_bf16) reinterpret_cast<uint16_t*>(pr.y)[o] = f32_to_bf16_bits(v);
                                else reinterpret_cast<float*>(pr.y)[o] = v;
                            }
                        }
                    }
                }
                // the accumulators are read: the next tile's first MMA (ordered after
                // this warp's next afull arrival) may overwrite them
                asm volatile("tcgen05.fence::before_thread_sync;");
            }
        }
        if (!ok && lane == 0) atomicOr(&g_tcg_wait_timeouts, 1u);
    } else if (warp == kTgUnpackWarps) {
        // ---- sign-bit producer (one lane): 4-step chunks of every tile in order
        if (lane == 0) {
            int gc = 0;
            bool ok = true;
            for (int p = R.p0; p <= R.p1 && ok; ++p) {
                const TgProb& pr = P[p];
                const int nch = pr.K / (kTcStepK * kTcChunkSteps);
                for (int t = ts(p); t < te(p) && ok; ++t) {
                    for (int c = 0; c < nch; ++c, ++gc) {
                        const int ws = gc % kTgWSlots;
                        if (gc >= kTgWSlots && !mbar_wait_sleep(wempty + 8 * ws, (uint32_t)(gc / kTgWSlots - 1) & 1u)) {
                            ok = false;
                            break;
                        }
                        mbar_expect_tx(wfull + 8 * ws, kTgWSlotBytes);
                        tma_2d(wring + ws * kTgWSlotBytes, &pr.tm_bits, 16 * kTcChunkSteps * c, t * kTgRows,
                               wfull + 8 * ws);
                    }
                }
            }
            if (!ok) atomicOr(&g_tcg_wait_timeouts, 2u);
            // every issued copy has landed before the CTA may exit
            for (int g = max(0, gc - kTgWSlots); g < gc; ++g)
                if (!mbar_wait(wfull + 8 * (g % kTgWSlots), (uint32_t)(g / kTgWSlots) & 1u)) atomicOr(&g_tcg_wait_timeouts, 2u);
        }
    } else if (warp == kTgUnpackWarps + 1) {
        // ---- activation producer (one lane): one box of 2 x 64 inputs x Bp rows per step
        pdl_wait();
        if (lane == 0) {
            int gs = 0, st = 0, use = 0;                   // step, its B stage and that stage's use count
            bool ok = true;
            for (int p = R.p0; p <= R.p1 && ok; ++p) {
                const TgProb& pr = P[p];
                const int nst = pr.K / kTcStepK;
                for (int t = ts(p); t < te(p) && ok; ++t) {
                    for (int s = 0; s < nst; ++s, ++gs) {
                        if (use > 0 && !mbar_wait_sleep(bfree + 8 * st, (uint32_t)(use - 1) & 1u)) {
                            ok = false;
                            break;
                        }
                        mbar_expect_tx(bfull + 8 * st, bstage);
                        tma_3d(bring + (uint32_t)st * bstage, &pr.tm_x, 0, 0, 2 * s, bfull + 8 * st);
                        if (++st == nbs) {
                            st = 0;
                            ++use;
                        }
                    }
                }
            }
            if (!ok) atomicOr(&g_tcg_wait_timeouts, 4u);
            for (int g = max(0, gs - nbs); g < gs; ++g)
                if (!mbar_wait(bfull + 8 * (g % nbs), (uint32_t)(g / nbs) & 1u)) atomicOr(&g_tcg_wait_timeouts, 4u);
        }
    } else {
        // ---- MMA issuers: warp 10 + 2h + j accumulates half h, slices j, j + 2, j + 4, j + 6
        const int mw = warp - (kTgUnpackWarps + 2), h = mw >> 1, j = mw & 1;
        pdl_wait();
        if (lane == 0) {
            // The issuing thread's own instruction latency bounds its MMA rate:
            // stage indices and parities are stepped, not divided, and every
            // descriptor is the ring's base descriptor plus a 16-byte-unit
            // offset (shared-memory addresses < 256 KB: no carry out of the
            // 14-bit address field).
            const uint32_t idesc = tc_idesc_f16(Bp);
            const uint32_t d_addr = tmem + (uint32_t)((2 * h + j) * Bp);
            const uint64_t bdesc0 = tc_desc_sw128(bring);
            // slice kk: A at 8 kk columns, B at slab kk / 4, 32 (kk % 4) bytes
            const uint64_t ko0 = (uint64_t)(32u * j) >> 4, ko1 = (uint64_t)(32u * (j + 2)) >> 4;
            const uint64_t ko2 = (uint64_t)(btile + 32u * j) >> 4, ko3 = (uint64_t)(btile + 32u * (j + 2)) >> 4;
            const uint32_t a_h = tmem + abase + 64u * h + 8u * j;
            int tiles = 0;
            int st = 0, ause = 0, bs = 0, buse = 0;
            bool ok = true;
            for (int p = R.p0; p <= R.p1 && ok; ++p) {
                const int nst = P[p].K / kTcStepK;
                for (int t = ts(p); t < te(p) && ok; ++t) {
                    for (int s = 0; s < nst; ++s) {
                        if (!mbar_wait_sleep(afull + 8 * st, (uint32_t)ause & 1u) ||
                            !mbar_wait_sleep(bfull + 8 * bs, (uint32_t)buse & 1u)) {
                            ok = false;
                            break;
                        }
                        asm volatile("tcgen05.fence::after_thread_sync;");
                        const uint64_t bd = bdesc0 + (uint64_t)(((uint32_t)bs * bstage) >> 4);
                        const uint32_t a0 = a_h + 128u * (uint32_t)st;
                        tc_mma1(d_addr, a0, bd + ko0, idesc, s > 0);
                        tc_mma1(d_addr, a0 + 16u, bd + ko1, idesc, true);
                        tc_mma1(d_addr, a0 + 32u, bd + ko2, idesc, true);
                        tc_mma1(d_addr, a0 + 48u, bd + ko3, idesc, true);
                        tc_commit(freed + 8 * st);
                        tc_commit(bfree + 8 * bs);
                        if (++st == nstg) { st = 0; ++ause; }
                        if (++bs == nbs) { bs = 0; ++buse; }
                    }
                    tc_commit(d_done);
                    ++tiles;
                }
            }
            if (!ok) {
                atomicOr(&g_tcg_wait_timeouts, 8u);
                tc_commit(d_done);
                ++tiles;
            }
            // no MMA may still be running when the tensor memory is released
            if (tiles > 0 && !mbar_wait(d_done, (uint32_t)(tiles - 1) & 1u)) atomicOr(&g_tcg_wait_timeouts, 8u);
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
}

// ---------------------------------------------------------------- host
namespace {

PFN_cuTensorMapEncodeTiled_v12000 tg_encode() {
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

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }
int padded_batch(int B) { return (B + 15) / 16 * 16; }

bool tg_problem_ok(const bit1_gemv_problem& pb) {
    return pb.bits && pb.scales && pb.x && pb.y && pb.N >= 1 && pb.N <= (1LL << 30) && pb.K >= 1024 &&
           pb.K % 1024 == 0 && pb.K <= (1LL << 20) && (pb.y_dtype == BIT1_F32 || pb.y_dtype == BIT1_BF16) &&
           ((uintptr_t)pb.bits & 15) == 0 && ((uintptr_t)pb.scales & 15) == 0 && ((uintptr_t)pb.x & 15) == 0 &&
           ((uintptr_t)pb.y & 15) == 0 &&
           (pb.epilogue == BIT1_EPI_NONE || (pb.epilogue == BIT1_EPI_SWIGLU && pb.N % 2 == 0));
}

// Workspace share of one problem: x' [Bp][K] fp16 and Bp scale factors.
size_t tg_ws_share(int64_t K, int Bp) { return align256((size_t)Bp * K * 2) + align256((size_t)Bp * 4); }

// A tile costs its K steps plus a fixed share for the epilogue and the
// pipeline bubble at the tile boundary (in steps).
constexpr double kTgTileFixed = 3.0;

int tg_partition(const std::vector<TgProb>& probs, double T, std::vector<TgRange>* out) {
    const int n = (int)probs.size();
    int ctas = 1;
    double cur = 0.0;
    TgRange r{0, 0, 0, 0};
    for (int p = 0; p < n; ++p) {
        const double c = probs[p].K / (double)kTcStepK + kTgTileFixed;
        for (int t = 0; t < probs[p].tiles; ++t) {
            if (cur > 0.0 && cur + c > T) {
                if (out) { r.p1 = p; r.t1 = t; out->push_back(r); }
                r = TgRange{p, t, p, t};
                ++ctas;
                cur = 0.0;
            }
            cur += c;
        }
    }
    if (out) { r.p1 = n - 1; r.t1 = probs[n - 1].tiles; out->push_back(r); }
    return ctas;
}

cudaError_t tg_set_attrs(const void* fn) { return func_attrs(fn, 227 * 1024, false); }

}  // namespace

size_t tcg_plan_bytes(int count) {
    if (count < 1) return 0;
    const size_t ranges = sizeof(TgHeader) + (size_t)kTgMaxCtas * sizeof(TgRange);
    const size_t probs_off = (ranges + 127) & ~(size_t)127;
    return probs_off + (size_t)count * sizeof(TgProb);
}

size_t tcg_workspace_bytes(const bit1_gemv_problem* problems, int count, int B) {
    if (count < 1 || !problems || B < 1 || B > kTgMaxB) return 0;
    size_t total = 0;
    for (int i = 0; i < count; ++i) {
        if (!tg_problem_ok(problems[i])) return 0;
        total += tg_ws_share(problems[i].K, padded_batch(B));
    }
    return total;
}

bit1_status tcg_plan(const bit1_gemv_problem* problems, int count, int B, void* workspace, size_t ws_bytes,
                     void* host_plan, size_t bytes) {
    if (count < 1 || !problems || !host_plan || !workspace) return BIT1_EINVAL;
    if (B < 1 || B > kTgMaxB) return BIT1_ESHAPE;
    if (bytes < tcg_plan_bytes(count) || ((uintptr_t)host_plan & 127) || ((uintptr_t)workspace & 255))
        return BIT1_EINVAL;
    for (int i = 0; i < count; ++i)
        if (!tg_problem_ok(problems[i])) return BIT1_ESHAPE;
    if (ws_bytes < tcg_workspace_bytes(problems, count, B)) return BIT1_EINVAL;
    auto enc = tg_encode();
    if (!enc) return BIT1_ECUDA;
    const int Bp = padded_batch(B);
    std::vector<TgProb> probs(count);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    for (int i = 0; i < count; ++i) {
        const bit1_gemv_problem& pb = problems[i];
        TgProb& g = probs[i];
        std::memset(&g, 0, sizeof(g));
        g.xp = reinterpret_cast<uint16_t*>(ws);
        g.xscale = reinterpret_cast<float*>(ws + align256((size_t)Bp * pb.K * 2));
        ws += tg_ws_share(pb.K, Bp);
        {
            const cuuint64_t dims[2] = {(cuuint64_t)(pb.K / 8), (cuuint64_t)pb.N};
            const cuuint64_t strides[1] = {(cuuint64_t)(pb.K / 8)};
            const cuuint32_t box[2] = {16 * kTcChunkSteps, (cuuint32_t)kTgRows};
            const cuuint32_t es[2] = {1, 1};
            if (enc(&g.tm_bits, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, (void*)pb.bits, dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return BIT1_ECUDA;
        }
        {
            const cuuint64_t dims[3] = {64, (cuuint64_t)Bp, (cuuint64_t)(pb.K / 64)};
            const cuuint64_t strides[2] = {(cuuint64_t)(pb.K * 2), 128};
            const cuuint32_t box[3] = {64, (cuuint32_t)Bp, 2};
            const cuuint32_t es[3] = {1, 1, 1};
            if (enc(&g.tm_x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, (void*)g.xp, dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return BIT1_ECUDA;
        }
        g.x = pb.x;
        g.scales = pb.scales;
        g.y = pb.y;
        g.N = (int)pb.N;
        g.K = (int)pb.K;
        g.tiles = (int)((pb.N + kTgRows - 1) / kTgRows);
        g.y_bf16 = pb.y_dtype == BIT1_BF16;
        g.swiglu = pb.epilogue == BIT1_EPI_SWIGLU;
    }
    // contiguous tile ranges: the smallest per-CTA budget that fits nctas CTAs
    const int nctas = std::min(sm_count(), kTgMaxCtas);
    if (nctas < 1) return BIT1_ECUDA;
    double total = 0.0, biggest = 0.0;
    for (const TgProb& g : probs) {
        const double c = g.K / (double)kTcStepK + kTgTileFixed;
        total += c * g.tiles;
        biggest = std::max(biggest, c);
    }
    double lo = total / nctas, hi = total + biggest;
    for (int it = 0; it < 60 && hi - lo > 1e-4 * lo; ++it) {
        const double mid = 0.5 * (lo + hi);
        if (tg_partition(probs, mid, nullptr) <= nctas) hi = mid;
        else lo = mid;
    }
    std::vector<TgRange> ranges;
    tg_partition(probs, hi, &ranges);
    if ((int)ranges.size() > nctas) return BIT1_ESHAPE;
    while ((int)ranges.size() < nctas)            // CTAs without work
        ranges.push_back(TgRange{count - 1, probs[count - 1].tiles, count - 1, probs[count - 1].tiles});

    TgHeader h{};
    h.count = count;
    h.nctas = nctas;
    h.B = B;
    h.Bp = Bp;
    h.stages = 4 * Bp <= 128 ? 3 : 2;             // accumulators 4 Bp + stages x 128 columns <= 512
    h.bstages = std::min<int>(kTgMaxBStages, (int)(kTgBRingBytes / (256u * (uint32_t)Bp)));
    const size_t need = 1024 + (size_t)kTgWSlots * kTgWSlotBytes + (size_t)h.bstages * 2 * 128 * Bp +
                        8 * (2 * kTgWSlots + 6 + 2 * kTgMaxBStages + 1) + 16;
    h.smem_bytes = (int)std::max<size_t>(need, kTgMinSmem);
    h.kind = kPlanKindTensor;
    const size_t r_off = sizeof(TgHeader);
    const size_t p_off = (r_off + (size_t)kTgMaxCtas * sizeof(TgRange) + 127) & ~(size_t)127;
    h.ranges_off = (int)r_off;
    h.probs_off = (int)p_off;
    uint8_t* out = static_cast<uint8_t*>(host_plan);
    std::memset(out, 0, bytes);
    std::memcpy(out, &h, sizeof(h));
    std::memcpy(out + r_off, ranges.data(), ranges.size() * sizeof(TgRange));
    std::memcpy(out + p_off, probs.data(), probs.size() * sizeof(TgProb));
    return BIT1_OK;
}

cudaError_t launch_tc_group(const void* device_plan, const void* host_plan, bool pdl, cudaStream_t stream) {
    const TgHeader* h = static_cast<const TgHeader*>(host_plan);
    if (h->kind != kPlanKindTensor || h->Bp < 16 || h->Bp > kTgMaxB || h->Bp % 16 || h->B < 1 || h->B > h->Bp ||
        (h->stages != 2 && h->stages != 3) || h->bstages < 2 || h->bstages > kTgMaxBStages ||
        (4 * h->Bp + 127) / 128 * 128 + 128 * h->stages > 512 || h->nctas < 1 ||
        h->nctas > kTgMaxCtas)
        return cudaErrorInvalidValue;
    cudaError_t e = tg_set_attrs((const void*)k_gemv_tc_group);
    if (e != cudaSuccess) return e;
    const uint8_t* dp = static_cast<const uint8_t*>(device_plan);
    void* args[] = {(void*)&dp};
    e = launch((const void*)k_tcg_prep, dim3((unsigned)(h->count * h->Bp)), dim3(kTcPrepThreads), 0, stream, pdl,
               args);
    if (e != cudaSuccess) return e;
    // always programmatic: the main kernel streams weights while the prep runs
    return launch((const void*)k_gemv_tc_group, dim3((unsigned)h->nctas), dim3(kTgThreads), (size_t)h->smem_bytes,
                  stream, true, args);
}

unsigned int tcg_take_timeouts() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_tcg_wait_timeouts, sizeof(v)) != cudaSuccess) return 0xffffffffu;
    if (v) cudaMemcpyToSymbol(g_tcg_wait_timeouts, &zero, sizeof(zero));
    return v;
}

}  // namespace bit1
