// Grouped batch-1 GEMV: many independent packed-1-bit problems in one
// persistent launch (CUDA cores, sm_103a).
//
// Each problem is y = W x with W in the binary g128 format of the web page
// "Bonsai 27B: 노트북과 폰에서 실행되는 27B급 이진 및 삼진 저비트 LLM" (section
// "이진(Binary) 가중치 형식"), computed with the 6-bit fp16 tables of
// gemv_t6.cu (one row per lane, TMA-staged weights, fp32 accumulation).
//
// Why one launch: autoregressive decode reads every weight once per token and
// at batch 1 the time goes to weight traffic and to kernel launch /
// synchronisation latency (same page, sections "27B 규모에서 효율은 선택이
// 아닌 제약" and "하이브리드 어텐션을 위한 저비트 커널").  Launching every
// matrix separately pays launch, table-build and drain latency per matrix.
// Here the concatenated list of 32-row blocks of all problems is cut into
// one contiguous, cost-balanced range per CTA (one CTA per SM, no clusters,
// no split-K: every row is produced by exactly one lane, deterministically).
// A CTA builds tables only for the problems its range touches, K split into
// chunks of at most 32 groups (4096 inputs); its per-warp TMA rings run ahead
// across problem and chunk boundaries, so the weight stream does not stall
// while the next problem's tables are built.
//
// SwiGLU epilogue: a problem may be a SwiGLU MLP's gate and up projections
// with interleaved rows (same page, section "Bonsai 27B의 표현 방식": the base
// model keeps its SwiGLU MLP).  Lanes 2m and 2m+1 then hold one hidden unit's
// gate and up sums; one shuffle pairs them and the even lane writes
// h = silu(g) * u.
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

namespace bit1 {

__device__ unsigned int g_group_wait_timeouts = 0;

constexpr int kGChunkGroups = 32;            // K chunk at batch 1: 32 groups = 4096 inputs
constexpr int kGStageBytes = 5120;           // 4 KB bits box + 512 B scales box, 1 KB aligned
constexpr int kGMaxCtas = 160;
constexpr int kGWarps = 20;
constexpr int kGMaxSmem = 227 * 1024;
constexpr int kGSegBlocks = 128;             // sub-segment cap: 4096 rows of partials
constexpr int kGMaxProbsPerCta = 64;         // problems one CTA's range may touch
constexpr int kGMaxNB = 6;                   // batch rows per grouped launch (table engine)
constexpr int kGMaxNBMma = 16;               // batch rows per grouped launch (MMA engine)
constexpr int kGEngineTables = 0;            // 6-bit tables, one lookup per six inputs and batch row
constexpr int kGEngineMma = 1;               // register-sourced mma.sync, batch rows as the MMA's N

// K chunk (groups) at nb batch rows: the tables of all rows, nb * CG * 2816
// bytes, stay at about 90 KB.
__host__ __device__ constexpr int g_chunk_groups(int nb) { return nb == 1 ? 32 : nb == 2 ? 16 : 8; }
// Row blocks per sub-segment of a multi-chunk problem: nb * 32 * seg floats of
// partials stay at about 16 KB.
__host__ __device__ constexpr int g_seg_blocks(int nb) { return nb == 1 ? 128 : nb == 2 ? 64 : nb <= 4 ? 32 : 16; }

struct GHeader {            // 128 bytes
    int count, nctas, W, S;
    uint32_t off_tables;
    int nb;                 // batch rows: x is [nb][K], y is [nb][N] for every problem
    uint32_t off_fac, off_part, off_bars;
    int part_rows, smem_bytes, ranges_off, probs_off;
    int seg_blocks;         // row blocks per sub-segment of a problem with K > 4096
    uint32_t off_xraw;      // raw bf16 activations of the next phase (bulk copy target)
    uint32_t off_pinfo;     // per-problem {RB, G, nch, N} of the CTA's range
    int layout;             // sign-bit layout of every problem (kLayoutCanonical or kLayoutG128x)
    int kind;               // kPlanKindTables
    int engine;             // kGEngineTables or kGEngineMma
    int pad[13];
};
static_assert(sizeof(GHeader) == 128, "header size");
static_assert(offsetof(GHeader, kind) == kPlanKindOffset, "kind offset");

struct GRange {             // blocks from (p0, b0) up to, not including, (p1, b1)
    int p0, b0, p1, b1;
};

struct alignas(128) GProb {
    CUtensorMap tm_bits;    // 2-D [N][K/8] uint8, box {128, 32}, 128-byte swizzle
    CUtensorMap tm_sc;      // 2-D [N][G] uint16, box {8, 32}
    const uint16_t* x;
    void* y;
    int N, K, G, RB, y_bf16, nch;
    int swiglu;             // rows are (gate, up) pairs; y is h = silu(gate) * up, [nb][N/2]
};

struct GSingle {            // whole plan of a one-problem call, passed by value
    GHeader h;
    GRange r[kGMaxCtas];
    GProb p;
};

// ---------------------------------------------------------------- device
// A CTA's work is a sequence of phases: for each problem p of its range, the
// blocks [bs(p), be(p)), cut into sub-segments of at most mb(p) blocks (only
// problems with more than one K chunk are cut: their row partials live in
// shared memory between chunks); per sub-segment, chunk by chunk.  The tables
// of a phase are built by the whole CTA between two barriers, so a warp that
// runs out of work in a phase waits for the slowest one.  Within a phase of
// n blocks, warp w therefore takes blocks w, w + W, ... of the first
// q = floor(n / W) * W only (every warp the same count); with TAIL the
// r = n - qW blocks left over are cut into their 8-group slices and those
// r * nsl single-slice units go to the warps in turn (unit u to warp u % W),
// so the imbalance at the phase's end is at most one slice instead of one
// block.  The units' partial sums are added in slice order afterwards (a
// fixed order: results do not depend on timing).  Without TAIL (several
// batch rows, whose unit partials would not fit) warp w takes every W-th
// block of the phase.
struct GIter {               // position in one warp's sequence of stages
    int p, sb, c;            // phase: problem, sub-segment start block, chunk
    int b, j;                // stage: block and 8-group slice
    int k, nk;               // this warp's stage index within the phase, and its stage count
    int nsl, q, kf;          // slices per block of the chunk; full blocks per warp; q * nsl
    int g0;                  // first group of the chunk
    const CUtensorMap* tm;   // the problem's bits tensor map (its scales map follows it)
};

template <int CG, bool TAIL>
struct GCtx {
    const GProb* P;
    const int4* I;          // shared memory: {RB, G, nch, N} of problems R.p0.. (index p - R.p0)
    GRange R;
    int w, W, seg_blocks;
    __device__ __forceinline__ int4 info(int p) const { return I[p - R.p0]; }
    __device__ __forceinline__ int bs(int p) const { return p == R.p0 ? R.b0 : 0; }
    __device__ __forceinline__ int be(int p) const { return p == R.p1 ? R.b1 : info(p).x; }
    __device__ __forceinline__ int nch(int p) const { return info(p).z; }
    __device__ __forceinline__ int mb(int p) const { return nch(p) > 1 ? seg_blocks : 0x3fffffff; }
    __device__ __forceinline__ int se(int p, int sb) const { return min(be(p), sb + mb(p)); }
    __device__ __forceinline__ int slices(int p, int c) const {
        const int cg = min(CG, info(p).y - CG * c);
        return cg >> 3;
    }
    // Full blocks of warp w in a phase of n blocks.
    __device__ __forceinline__ int full_blocks(int n) const {
        return TAIL ? n / W : (w < n ? (n - 1 - w) / W + 1 : 0);
    }
    __device__ __forceinline__ bool done(const GIter& it) const { return it.p > R.p1; }
    // CTA-level phases (problem, sub-segment, chunk), in execution order.
    __device__ __forceinline__ bool next_phase(int& p, int& sb, int& c) const {
        if (++c < nch(p)) return true;
        c = 0;
        sb += mb(p);
        if (sb < be(p)) return true;
        for (++p; p <= R.p1; ++p) {
            sb = bs(p);
            if (sb < be(p)) return true;
        }
        return false;
    }
    __device__ __forceinline__ bool first_phase(int& p, int& sb, int& c) const {
        c = 0;
        for (p = R.p0; p <= R.p1; ++p) {
            sb = bs(p);
            if (sb < be(p)) return true;
        }
        return false;
    }
    // This warp's stage count in phase (it.p, it.sb, it.c).
    __device__ __forceinline__ void enter(GIter& it) const {
        const int n = se(it.p, it.sb) - it.sb;
        it.g0 = CG * it.c;
        it.tm = &P[it.p].tm_bits;
        it.nsl = slices(it.p, it.c);
        it.q = full_blocks(n);
        it.k = 0;
        it.kf = it.q * it.nsl;
        it.nk = it.kf;
        if (TAIL) {
            const int nu = (n - it.q * W) * it.nsl;
            if (w < nu) it.nk += (nu - 1 - w) / W + 1;
        }
    }
    // Block and slice of stage it.k of the phase (from scratch; next() steps
    // through the full blocks incrementally).
    __device__ __forceinline__ void pos(GIter& it) const {
        if (it.k < it.kf) {
            const int i = it.k / it.nsl;
            it.j = it.k - i * it.nsl;
            it.b = it.sb + w + W * i;
        } else {
            const int u = w + W * (it.k - it.kf);
            const int i = u / it.nsl;
            it.j = u - i * it.nsl;
            it.b = it.sb + it.q * W + i;
        }
    }
    // Move to the first stage at or after `it` (a later phase if this one is used up).
    __device__ __forceinline__ void settle(GIter& it) const {
        while (it.k >= it.nk) {
            if (!next_phase(it.p, it.sb, it.c)) {
                it.p = R.p1 + 1;
                return;
            }
            enter(it);
        }
        pos(it);
    }
    __device__ __forceinline__ GIter first() const {
        GIter it{};
        if (!first_phase(it.p, it.sb, it.c)) {
            it.p = R.p1 + 1;
            return it;
        }
        enter(it);
        settle(it);
        return it;
    }
    __device__ __forceinline__ void next(GIter& it) const {
        ++it.k;
        if (it.k < it.kf) {                 // the common case: the next slice of a full block
            if (++it.j == it.nsl) {
                it.j = 0;
                it.b += W;
            }
            return;
        }
        settle(it);
    }
};

static_assert(offsetof(GProb, tm_sc) == offsetof(GProb, tm_bits) + sizeof(CUtensorMap), "maps adjacent");

__device__ __forceinline__ void g_issue(const GIter& it, uint32_t st, uint32_t bar) {
    const int g = it.g0 + 8 * it.j;
    mbar_expect_tx(bar, 4096u + 512u);
    tma_2d(st, it.tm, g * 16, it.b * 32, bar);
    tma_2d(st + 4096u, it.tm + 1, g, it.b * 32, bar);
}

// The same, executed by the whole warp and carried out by the lanes whose
// `on` is set (one lane): a predicated block instead of a divergent branch
// around the copies, which cost the warp a reconvergence on every stage.
__device__ __forceinline__ void g_issue_pred(const GIter& it, uint32_t st, uint32_t bar, bool on) {
    const int g = it.g0 + 8 * it.j;
    asm volatile("{ .reg .pred p; setp.ne.u32 p, %0, 0;\n\t"
                 "@p mbarrier.arrive.expect_tx.shared::cta.b64 _, [%1], 4608;\n\t"
                 "@p cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%2], [%3, {%4, %5}], [%1];\n\t"
                 "@p cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%6], [%7, {%8, %5}], [%1]; }"
                 ::"r"(on ? 1u : 0u), "r"(bar), "r"(st), "l"(it.tm), "r"(g * 16), "r"(it.b * 32), "r"(st + 4096u),
                   "l"(it.tm + 1), "r"(g)
                 : "memory");
}


// Batch 1, one 8-group slice of a 32-row block: group JJ of the slice reads
// its 16 sign bytes at the swizzled offset (row r's chunk c lands at
// r*128 + ((c ^ (r % 8)) * 16); `a0` is the lane's address for chunk 0 and the
// stage is 1024-byte aligned, so chunk JJ is a0 ^ (JJ * 16)), looks them up
// in its 22 tables and adds s_g * 2^m_g times the sum to acc.
template <int L, int JJ>
__device__ __forceinline__ float g_slice1(uint32_t a0, uint32_t tg0, const uint32_t (&svw)[4],
                                          const uint32_t (&fw)[8], float acc) {
    const uint4 wv = lds128(a0 ^ (uint32_t)(JJ << 4));
    const uint32_t w4[4] = {wv.x, wv.y, wv.z, wv.w};
    const float pt = t6_groupj<L, JJ>(w4, tg0, std::make_index_sequence<kT6Fields>{});
    const float sc = f16_bits_to_f32((uint16_t)(svw[JJ >> 1] >> (16 * (JJ & 1))));
    return fmaf(pt, sc * __uint_as_float(fw[JJ]), acc);
}

template <int NB, int CG, int S, int L>
__device__ __forceinline__ void g_body(const uint8_t* plan) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = (uint32_t)__cvta_generic_to_shared(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);

    const GHeader* H = reinterpret_cast<const GHeader*>(plan);
    const int W = H->W, prows = H->part_rows;   // H->S == S (the launch picks the instantiation)
    constexpr bool TAIL = NB == 1;
    GCtx<CG, TAIL> cx;
    cx.P = reinterpret_cast<const GProb*>(plan + H->probs_off);
    cx.R = reinterpret_cast<const GRange*>(plan + H->ranges_off)[blockIdx.x];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    cx.w = warp;
    cx.W = W;
    cx.seg_blocks = H->seg_blocks;
    int4* pinfo = reinterpret_cast<int4*>(sm + H->off_pinfo);
    for (int i = threadIdx.x; i <= cx.R.p1 - cx.R.p0 && i < kGMaxProbsPerCta; i += blockDim.x) {
        const GProb& q = cx.P[cx.R.p0 + i];
        pinfo[i] = make_int4(q.RB, q.G, q.nch, q.N);
    }
    cx.I = pinfo;
    __syncthreads();
    const GProb* P = cx.P;
    const uint32_t bars = base + H->off_bars + (uint32_t)(warp * S) * 8u;
    const uint32_t stages = base + (uint32_t)(warp * S) * kGStageBytes;

    // Producer (lane 0): start the warp's weight stream before anything else.
    GIter prod = cx.first();
    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(bars + 8u * s, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        for (int s = 0; s < S && !cx.done(prod); ++s) {
            g_issue(prod, stages + (uint32_t)s * kGStageBytes, bars + 8u * s);
            cx.next(prod);
        }
    } else {
        for (int s = 0; s < S && !cx.done(prod); ++s) cx.next(prod);
    }
    __syncwarp();

    // The activations of each phase are bulk-copied into shared memory one
    // phase ahead (mbarrier xbar, one completion per phase).
    const uint32_t xbar = base + H->off_bars + (uint32_t)(W * S) * 8u;
    const uint32_t xraw = base + H->off_xraw;
    auto prefetch_x = [&](int p, int c) {   // chunk c of every batch row's x
        const GProb& q = P[p];
        const int cg = min(CG, q.G - CG * c);
        mbar_expect_tx(xbar, (uint32_t)(NB * cg) * 256u);
        for (int b = 0; b < NB; ++b)
            bulk_g2s(xraw + (uint32_t)(b * CG) * 256u, q.x + (size_t)b * q.K + (size_t)c * CG * 128,
                     (uint32_t)cg * 256u, xbar);
    };
    pdl_wait();   // inputs may come from the preceding kernel
    if (threadIdx.x == 0) {
        mbar_init(xbar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        int fp, fsb, fc;
        if (cx.first_phase(fp, fsb, fc)) prefetch_x(fp, fc);
    }
    int xphase = 0;
    const uint16_t* xr = reinterpret_cast<const uint16_t*>(sm + H->off_xraw);
    float* fac = reinterpret_cast<float*>(sm + H->off_fac);
    float* part = reinterpret_cast<float*>(sm + H->off_part);
    float* upart = part + NB * prows;          // TAIL: partial sums of the single-slice units
    uint8_t* tabs = sm + H->off_tables;
    const uint32_t tb = base + H->off_tables;
    const uint32_t fac_s = base + H->off_fac;

    int k = 0;          // stages consumed by this warp
    int sk = 0;         // k % S: ring slot of stage k
    uint32_t ph = 0;    // (k / S) & 1: its mbarrier phase parity
    int kfail = -1;     // stage whose bounded wait gave up
    bool ok = true;
    const uint32_t lane_a0 = (uint32_t)lane * 128u + ((uint32_t)(lane & 7) << 4);   // chunk 0 of row `lane`
    for (int p = cx.R.p0; p <= cx.R.p1; ++p) {
      const GProb& pr = P[p];
      const int4 pi = cx.info(p);             // RB, G, nch, N
      for (int sb = cx.bs(p); sb < cx.be(p); sb += cx.mb(p)) {
        const int be = cx.se(p, sb);
        for (int c = 0; c < pi.z; ++c) {
            const int cg = min(CG, pi.y - CG * c);
            // --- tables for (problem p, chunk c): every thread of the CTA
            __syncthreads();                                   // old tables no longer read
            if (!mbar_wait(xbar, (uint32_t)(xphase & 1))) {     // this phase's activations
                if (lane == 0) atomicOr(&g_group_wait_timeouts, 2u);
                ok = false;
            }
            ++xphase;
            for (int bg = warp; bg < NB * cg; bg += W) {       // one (row, group) per warp pass
                const int b = bg / cg, g = bg - b * cg;
                const uint2 xv = *reinterpret_cast<const uint2*>(xr + (b * CG + g) * 128 + 4 * lane);
                const float x0 = bf16_bits_to_f32(xv.x & 0xffffu), x1 = bf16_bits_to_f32(xv.x >> 16);
                const float x2 = bf16_bits_to_f32(xv.y & 0xffffu), x3 = bf16_bits_to_f32(xv.y >> 16);
                float m = fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3)));
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                int mg = 0;
                if (m > 0.f) {
                    const int e = (int)((__float_as_uint(m) >> 23) & 0xffu) - 127;
                    mg = min(max(e - 11, -126), 127);          // max|x'| < 2^12
                }
                if (lane == 0) {
                    fac[b * 2 * CG + g] = __uint_as_float((uint32_t)(mg + 127) << 23);
                    fac[b * 2 * CG + CG + g] = __uint_as_float((uint32_t)(127 - mg) << 23);
                }
            }
            __syncthreads();
            if constexpr (NB == 1) {
                // Table tt = (group g, field f) with tt = 22 g + f; thread t builds a
                // quarter of table t / 4.  The block's threads step tt by
                // blockDim.x / 4 (a multiple of 4), so (g, f) advance by a fixed
                // amount: no division per table.
                const int step = (int)blockDim.x >> 2, sg = step / kT6Fields, sf = step - sg * kT6Fields;
                int tt = (int)threadIdx.x >> 2;
                int g = tt / kT6Fields, f = tt - g * kT6Fields;
                for (; g < cg; tt += step) {
                    t6_build_pair(tabs + g * kT6GroupBytes + f * kT6TableBytes, xr + g * 128, fac[CG + g], f,
                                  threadIdx.x & 3, tt & 1);
                    g += sg;
                    f += sf;
                    if (f >= kT6Fields) {
                        f -= kT6Fields;
                        ++g;
                    }
                }
            } else {
                for (int t = threadIdx.x; t < NB * cg * kT6Fields * 4; t += blockDim.x) {
                    const int tt = t >> 2, bg = tt / kT6Fields, f = tt - bg * kT6Fields;
                    const int b = bg / cg, g = bg - b * cg;
                    t6_build_pair(tabs + (b * CG + g) * kT6GroupBytes + f * kT6TableBytes, xr + (b * CG + g) * 128,
                                  fac[b * 2 * CG + CG + g], f, t & 3, tt & 1);
                }
            }
            __syncthreads();
            if (threadIdx.x == 0) {                            // raw x consumed: fetch the next phase's
                int np = p, nsb = sb, nc = c;
                if (cx.next_phase(np, nsb, nc)) prefetch_x(np, nc);
            }
            if (p == cx.R.p0 && sb == cx.bs(p) && c == 0) pdl_launch_dependents();

            // --- this warp's work of the phase: stages (block, slice) in the
            // order the warp's ring was filled (GCtx::pos)
            const int nsl = cg >> 3;
            // One stage: wait for its copy, add its 8 groups to acc, refill the
            // ring slot with the warp's next stage.
            auto consume = [&](int j, float (&acc)[NB]) {
                if (ok && !mbar_wait(bars + 8u * sk, ph)) {
                    if (lane == 0) atomicOr(&g_group_wait_timeouts, 1u);
                    ok = false;
                    kfail = k;
                }
                // Computed even after a failed wait (the launch is then already
                // flagged; every table address stays inside the tables), so the
                // stage path has no branch around it.
                {
                    const uint32_t st = stages + (uint32_t)sk * kGStageBytes;
                    const uint4 sv = lds128(st + 4096u + 16u * lane);       // 8 scales of row `lane`
                    const uint32_t svw[4] = {sv.x, sv.y, sv.z, sv.w};
                    if constexpr (NB == 1) {
                        const uint4 fa = lds128(fac_s + 32u * j), fb = lds128(fac_s + 32u * j + 16u);
                        const uint32_t fw[8] = {fa.x, fa.y, fa.z, fa.w, fb.x, fb.y, fb.z, fb.w};
                        const uint32_t a0 = st + lane_a0;
                        const uint32_t tg0 = tb + (uint32_t)(8 * j) * kT6GroupBytes;
                        float a = acc[0];
                        a = g_slice1<L, 0>(a0, tg0, svw, fw, a);
                        a = g_slice1<L, 1>(a0, tg0, svw, fw, a);
                        a = g_slice1<L, 2>(a0, tg0, svw, fw, a);
                        a = g_slice1<L, 3>(a0, tg0, svw, fw, a);
                        a = g_slice1<L, 4>(a0, tg0, svw, fw, a);
                        a = g_slice1<L, 5>(a0, tg0, svw, fw, a);
                        a = g_slice1<L, 6>(a0, tg0, svw, fw, a);
                        a = g_slice1<L, 7>(a0, tg0, svw, fw, a);
                        acc[0] = a;
                    } else {
                        // Several batch rows: the 16 sign bytes of a group are read
                        // once and looked up in every row's tables.
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj) {
                            const uint32_t la = (uint32_t)lane * 128u + ((uint32_t)(jj ^ (lane & 7)) << 4);
                            const uint4 wv = lds128(st + la);
                            const uint32_t w4[4] = {wv.x, wv.y, wv.z, wv.w};
                            const float sc = f16_bits_to_f32((uint16_t)(svw[jj >> 1] >> (16 * (jj & 1))));
#pragma unroll
                            for (int bb = 0; bb < NB; ++bb) {
                                const int g = bb * CG + 8 * j + jj;
                                const float pt = T6GroupL<L>::run(w4, tb + (uint32_t)g * kT6GroupBytes,
                                                                  std::make_index_sequence<kT6Fields>{});
                                acc[bb] = fmaf(pt * sc, fac[bb * 2 * CG + 8 * j + jj], acc[bb]);
                            }
                        }
                    }
                }
                __syncwarp();
                g_issue_pred(prod, stages + (uint32_t)sk * kGStageBytes, bars + 8u * sk,
                             lane == 0 && ok && !cx.done(prod));
                if (!cx.done(prod)) cx.next(prod);
                ++k;
                if (++sk == S) {
                    sk = 0;
                    ph ^= 1u;
                }
            };
            // Block b's sums for chunk c: carried in `part` to the next chunk,
            // or, after the last chunk, through the epilogue into y.
            auto finish = [&](int b, float (&acc)[NB]) {
                const int row = b * 32 + lane;
                const int li = (b - sb) * 32 + lane;           // row within the sub-segment
                if (pi.z > 1) {
#pragma unroll
                    for (int bb = 0; bb < NB; ++bb) {
                        const int pl = bb * prows + li;
                        acc[bb] = (c == 0) ? acc[bb] : part[pl] + acc[bb];
                        if (c + 1 < pi.z) part[pl] = acc[bb];
                    }
                    if (c + 1 < pi.z) return;
                }
                if (pr.swiglu) {
                    // Lane 2m holds the gate row and lane 2m+1 the up row of hidden
                    // unit row/2 (N even: a pair is in range or out of it whole).
#pragma unroll
                    for (int bb = 0; bb < NB; ++bb) {
                        const float u = __shfl_down_sync(0xffffffffu, acc[bb], 1);
                        if (!(lane & 1) && row < pi.w) {
                            const float gt = acc[bb];
                            const float h = gt / (1.f + expf(-gt)) * u;
                            const int64_t o = (int64_t)bb * (pi.w >> 1) + (row >> 1);
                            if (pr.y_bf16) reinterpret_cast<uint16_t*>(pr.y)[o] = f32_to_bf16_bits(h);
                            else reinterpret_cast<float*>(pr.y)[o] = h;
                        }
                    }
                } else if (row < pi.w) {
#pragma unroll
                    for (int bb = 0; bb < NB; ++bb) {
                        const int64_t o = (int64_t)bb * pi.w + row;
                        if (pr.y_bf16) reinterpret_cast<uint16_t*>(pr.y)[o] = f32_to_bf16_bits(acc[bb]);
                        else reinterpret_cast<float*>(pr.y)[o] = acc[bb];
                    }
                }
            };
            const int n = be - sb;
            const int q = cx.full_blocks(n);
            for (int i = 0; i < q; ++i) {
                float acc[NB];
#pragma unroll
                for (int bb = 0; bb < NB; ++bb) acc[bb] = 0.f;
                for (int j = 0; j < nsl; ++j) consume(j, acc);
                finish(sb + warp + W * i, acc);
            }
            if constexpr (TAIL) {
                // The r blocks left over, one slice per unit; then, after a
                // barrier, each block's unit partials in slice order.
                const int r = n - q * W, nu = r * nsl;
                if (nu > 0) {
                    for (int u = warp; u < nu; u += W) {
                        float acc[1] = {0.f};
                        consume(u - (u / nsl) * nsl, acc);
                        upart[u * 32 + lane] = acc[0];
                    }
                    __syncthreads();
                    for (int i = warp; i < r; i += W) {
                        float acc[1] = {0.f};
                        for (int j = 0; j < nsl; ++j) acc[0] += upart[(i * nsl + j) * 32 + lane];
                        finish(sb + q * W + i, acc);
                    }
                }
            }
        }
      }
    }
    if (!ok && lane == 0) {
        // Give copies still in flight a bounded chance to land before exit.
        for (int kk = kfail + 1; kk < kfail + S; ++kk)
            (void)mbar_wait(bars + 8u * (kk % S), (uint32_t)(kk / S) & 1u);
    }
}

// ---------------------------------------------------------------- MMA engine
// Several batch rows (2..16) on register-sourced tensor-core MMAs
// (mma.sync m16n8k16, fp16 operands, fp32 accumulators).  The table engine's
// lookups grow with the batch rows; here the per-weight work (forming +-s as
// fp16 in a register: one multiply-as-shift and one LOP3 per two weights) is
// the same for every batch up to the MMA's N = 8 (NT = 1) or 16 (NT = 2).
// The A fragments never leave registers, so nothing is written to shared or
// tensor memory per weight, and each warp's MMAs depend on nothing but its own
// stage: no cross-warp hand-off per step.
//
// Within each 32-bit sign word, inputs k and k + 16 share one fp16x2
// register (sign bits 15 and 31 of s | s << 16), pair j = (k, k + 16) for
// j = 0..15.  Of a word's 16 pairs, MMA k-step h (two per word) takes pairs
// 8h..8h+7: slot pair c of the fragment (thread c = lane % 4) holds pair
// 8h + c, slot pair c + 4 holds pair 8h + c + 4.  The activations are laid
// out in the same K order, so the contraction is unchanged.  Per phase, the
// CTA converts its K chunk of activations to fp16 fragments with one
// power-of-two prescale per batch row (max |x'| in [2^14, 2^15), exact for
// every bf16 value within 2^29 of the chunk's largest), and the per-chunk
// sums are scaled back before they join the row's other chunks.  The chunk
// is read straight from global memory (L2) at the phase boundary: with 4096
// inputs per chunk a CTA has only a few phases, and the shared memory a
// staged copy would take goes to larger sub-segments instead.
__host__ __device__ constexpr int g_mma_nt(int nb) { return nb <= 8 ? 1 : 2; }
// K chunk: 4096 inputs (B <= 8) or 2048 (B > 8), 64 KB of fragments either way;
// sub-segments of multi-chunk problems: 64 KB of partials.
__host__ __device__ constexpr int g_mma_chunk_groups(int nb) { return nb <= 8 ? 32 : 16; }
__host__ __device__ constexpr int g_mma_seg_blocks(int nb) { return nb <= 4 ? 128 : nb <= 8 ? 64 : 32; }

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint2 b) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b.x), "r"(b.y));
}
// Pair j of the sign word w as an fp16x2 +-s: bits j and j + 16 moved to the
// sign positions 15 and 31 (a multiply by mul = 2^(15 - j), so the shift can
// issue on the FMA pipe; both come from real bits of w since j <= 15), then
// inverted (bit 0 -> negative) and applied to s2 = s | s << 16 in one LOP3.
__device__ __forceinline__ uint32_t g_pair(uint32_t w, uint32_t mul, uint32_t s2) {
    uint32_t t;
    asm("mul.lo.u32 %0, %1, %2;" : "=r"(t) : "r"(w), "r"(mul));
    return (~t & 0x80008000u) ^ s2;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}

template <int NT, int CG, int S>
__device__ __forceinline__ void g_body_mma(const uint8_t* plan) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = (uint32_t)__cvta_generic_to_shared(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);

    const GHeader* H = reinterpret_cast<const GHeader*>(plan);
    const int W = H->W, prows = H->part_rows, NB = H->nb;
    GCtx<CG, false> cx;
    cx.P = reinterpret_cast<const GProb*>(plan + H->probs_off);
    cx.R = reinterpret_cast<const GRange*>(plan + H->ranges_off)[blockIdx.x];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    cx.w = warp;
    cx.W = W;
    cx.seg_blocks = H->seg_blocks;
    int4* pinfo = reinterpret_cast<int4*>(sm + H->off_pinfo);
    for (int i = threadIdx.x; i <= cx.R.p1 - cx.R.p0 && i < kGMaxProbsPerCta; i += blockDim.x) {
        const GProb& q = cx.P[cx.R.p0 + i];
        pinfo[i] = make_int4(q.RB, q.G, q.nch, q.N);
    }
    cx.I = pinfo;
    __syncthreads();
    const GProb* P = cx.P;
    const uint32_t bars = base + H->off_bars + (uint32_t)(warp * S) * 8u;
    const uint32_t stages = base + (uint32_t)(warp * S) * kGStageBytes;

    GIter prod = cx.first();
    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(bars + 8u * s, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        for (int s = 0; s < S && !cx.done(prod); ++s) {
            g_issue(prod, stages + (uint32_t)s * kGStageBytes, bars + 8u * s);
            cx.next(prod);
        }
    } else {
        for (int s = 0; s < S && !cx.done(prod); ++s) cx.next(prod);
    }
    __syncwarp();

    pdl_wait();     // x may come from the preceding kernel
    float* fac = reinterpret_cast<float*>(sm + H->off_fac);     // [0, 16): 2^-m_b; [16, 32): 2^m_b
    float* part = reinterpret_cast<float*>(sm + H->off_part);
    uint2* xf = reinterpret_cast<uint2*>(sm + H->off_tables);    // [NT][CG * 8 k-steps][32 lanes]
    const uint32_t xf_s = base + H->off_tables;

    const int g = lane >> 2, c = lane & 3;
    const uint32_t mul0 = 1u << (15 - c), mul1 = 1u << (11 - c), mul2 = 1u << (7 - c), mul3 = 1u << (3 - c);
    const uint32_t swz = (uint32_t)g << 4;           // rows g, g + 8, 16 + g, 24 + g: swizzle (row % 8) = g
    int k = 0, sk = 0;
    uint32_t ph = 0;
    int kfail = -1;
    bool ok = true;
    for (int p = cx.R.p0; p <= cx.R.p1; ++p) {
      const GProb& pr = P[p];
      const int4 pi = cx.info(p);             // RB, G, nch, N
      for (int sb = cx.bs(p); sb < cx.be(p); sb += cx.mb(p)) {
        const int be = cx.se(p, sb);
        for (int ch = 0; ch < pi.z; ++ch) {
            const int cg = min(CG, pi.y - CG * ch);
            const uint16_t* xc = pr.x + (size_t)ch * CG * 128;   // this chunk of batch row 0; row b at + b K
            __syncthreads();                                   // old fragments no longer read
            // per batch row: largest finite |x| of the chunk -> prescale 2^-m
            for (int b = warp; b < NB; b += W) {
                uint32_t m = 0;
                for (int u = lane; u < cg * 16; u += 32) {     // 16-byte units of the row's chunk
                    const uint4 v = *reinterpret_cast<const uint4*>(xc + (size_t)b * pr.K + 8 * u);
                    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t lo = w4[i] & 0x7fffu, hi = (w4[i] >> 16) & 0x7fffu;
                        m = max(m, max(lo > 0x7f80u ? 0u : lo, hi > 0x7f80u ? 0u : hi));
                    }
                }
                m = __reduce_max_sync(0xffffffffu, m);
                int mb = 0;
                if (m != 0) mb = min(max((int)(m >> 7) - 127 - 14, -126), 126);
                if (lane == 0) {
                    fac[b] = __uint_as_float((uint32_t)(127 - mb) << 23);
                    fac[16 + b] = __uint_as_float((uint32_t)(127 + mb) << 23);
                }
            }
            __syncthreads();
            // fragments: entry (nt, q, l) = batch row 8 nt + l / 4, k-step q of the chunk
            {
                const int per_nt = cg * 8 * 32;
                for (int e = threadIdx.x; e < NT * per_nt; e += blockDim.x) {
                    const int nt = e / per_nt, rem = e - nt * per_nt, q = rem >> 5, l = rem & 31;
                    const int n = 8 * nt + (l >> 2), cc = l & 3;
                    uint2 v = make_uint2(0u, 0u);
                    if (n < NB) {
                        const int kb = (q >> 3) * 128 + 32 * ((q & 7) >> 1) + 8 * (q & 1) + cc;
                        const uint16_t* xs = xc + (size_t)n * pr.K + kb;
                        const float f = fac[n];
                        const __half2 h0 = __floats2half2_rn(bf16_bits_to_f32(xs[0]) * f, bf16_bits_to_f32(xs[16]) * f);
                        const __half2 h1 = __floats2half2_rn(bf16_bits_to_f32(xs[4]) * f, bf16_bits_to_f32(xs[20]) * f);
                        v.x = *reinterpret_cast<const uint32_t*>(&h0);
                        v.y = *reinterpret_cast<const uint32_t*>(&h1);
                    }
                    xf[(nt * CG * 8 + q) * 32 + l] = v;
                }
            }
            __syncthreads();
            if (p == cx.R.p0 && sb == cx.bs(p) && ch == 0) pdl_launch_dependents();

            const int nsl = cg >> 3;
            // One stage (32 rows x 8 groups): 2 row tiles x 64 k-steps of MMAs.
            auto consume = [&](int j, float (&acc)[2][NT][4]) {
                if (ok && !mbar_wait(bars + 8u * sk, ph)) {
                    if (lane == 0) atomicOr(&g_group_wait_timeouts, 1u);
                    ok = false;
                    kfail = k;
                }
                {
                    const uint32_t st = stages + (uint32_t)sk * kGStageBytes;
                    uint32_t sw[4];     // scales of groups jj, jj + 1 (jj even) of rows g, g + 8, 16 + g, 24 + g
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) {
                        uint4 w[4];
                        uint32_t s2[4];
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            w[r] = lds128(st + (uint32_t)(g + 8 * r) * 128u + (((uint32_t)jj << 4) ^ swz));
                            if (!(jj & 1)) sw[r] = lds32(st + 4096u + 16u * (uint32_t)(g + 8 * r) + 2u * (uint32_t)jj);
                            s2[r] = __byte_perm(sw[r], 0u, (jj & 1) ? 0x3232u : 0x1010u);   // s | s << 16
                        }
                        const uint32_t q0 = (uint32_t)((8 * j + jj) * 8);       // first k-step of the group in the chunk
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            uint32_t nw[4];
#pragma unroll
                            for (int r = 0; r < 4; ++r) nw[r] = i == 0 ? w[r].x : i == 1 ? w[r].y : i == 2 ? w[r].z : w[r].w;
#pragma unroll
                            for (int hh = 0; hh < 2; ++hh) {
                                const uint32_t ma = hh ? mul2 : mul0, mc = hh ? mul3 : mul1;
                                uint2 bf[NT];
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt)
                                    bf[nt] = lds64(xf_s + (((uint32_t)nt * CG * 8u + q0 + 2u * i + hh) * 32u + lane) * 8u);
#pragma unroll
                                for (int mt = 0; mt < 2; ++mt) {
                                    const int r0 = 2 * mt, r1 = 2 * mt + 1;     // rows 16 mt + g and 16 mt + g + 8
                                    const uint32_t a0 = g_pair(nw[r0], ma, s2[r0]), a1 = g_pair(nw[r1], ma, s2[r1]);
                                    const uint32_t a2 = g_pair(nw[r0], mc, s2[r0]), a3 = g_pair(nw[r1], mc, s2[r1]);
#pragma unroll
                                    for (int nt = 0; nt < NT; ++nt) mma16816(acc[mt][nt], a0, a1, a2, a3, bf[nt]);
                                }
                            }
                        }
                    }
                }
                __syncwarp();
                g_issue_pred(prod, stages + (uint32_t)sk * kGStageBytes, bars + 8u * sk,
                             lane == 0 && ok && !cx.done(prod));
                if (!cx.done(prod)) cx.next(prod);
                ++k;
                if (++sk == S) {
                    sk = 0;
                    ph ^= 1u;
                }
            };
            // Block b's sums for this chunk, scaled back by 2^m per batch row:
            // carried in `part` to the next chunk or written to y.
            auto finish = [&](int b, float (&acc)[2][NT][4]) {
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int rl = 16 * mt + g + 8 * (e >> 1);       // row within the block
                            const int bb = 8 * nt + 2 * c + (e & 1);         // batch row
                            const int row = b * 32 + rl;
                            const int li = (b - sb) * 32 + rl;
                            float v = acc[mt][nt][e] * fac[16 + (bb < NB ? bb : 0)];
                            if (pi.z > 1) {
                                const int pl = bb * prows + li;
                                if (bb < NB && ch > 0) v += part[pl];
                                if (ch + 1 < pi.z) {
                                    if (bb < NB) part[pl] = v;
                                    continue;
                                }
                            }
                            if (pr.swiglu) {
                                // rows 2u (gate) and 2u + 1 (up) sit in lanes 4 apart
                                const float u = __shfl_xor_sync(0xffffffffu, v, 4);
                                if (!(g & 1) && bb < NB && row < pi.w) {
                                    const float h = v / (1.f + expf(-v)) * u;
                                    const int64_t o = (int64_t)bb * (pi.w >> 1) + (row >> 1);
                                    if (pr.y_bf16) reinterpret_cast<uint16_t*>(pr.y)[o] = f32_to_bf16_bits(h);
                                    else reinterpret_cast<float*>(pr.y)[o] = h;
                                }
                            } else if (bb < NB && row < pi.w) {
                                const int64_t o = (int64_t)bb * pi.w + row;
                                if (pr.y_bf16) reinterpret_cast<uint16_t*>(pr.y)[o] = f32_to_bf16_bits(v);
                                else reinterpret_cast<float*>(pr.y)[o] = v;
                            }
                        }
                    }
                }
            };
            const int n = be - sb;
            const int q = cx.full_blocks(n);
            for (int i = 0; i < q; ++i) {
                float acc[2][NT][4];
#pragma unroll
                for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.f;
                for (int j = 0; j < nsl; ++j) consume(j, acc);
                finish(sb + warp + W * i, acc);
            }
        }
      }
    }
    if (!ok && lane == 0) {
        for (int kk = kfail + 1; kk < kfail + S; ++kk)
            (void)mbar_wait(bars + 8u * (kk % S), (uint32_t)(kk / S) & 1u);
    }
}

// NT: 8-column MMA tiles (1: up to 8 batch rows, 2: up to 16); canonical layout
// only; at most 16 warps, so 128 registers a thread.
template <int NT, int S>
__global__ void __launch_bounds__(16 * 32, 1) k_gemv_group_mma(const uint8_t* __restrict__ plan) {
    g_body_mma<NT, g_mma_chunk_groups(8 * NT), S>(plan);
}

// One problem on the MMA engine with its plan passed by value (bit1_gemv_ex
// with BIT1_GEMV_MMA).
template <int NT, int S>
__global__ void __launch_bounds__(16 * 32, 1) k_gemv_group1_mma(const __grid_constant__ GSingle plan) {
    g_body_mma<NT, g_mma_chunk_groups(8 * NT), S>(reinterpret_cast<const uint8_t*>(&plan));
}

// S: TMA stages per warp ring (the plan's H->S); L: the sign-bit layout (the
// plan's H->layout).  One instantiation per value the planner can choose.
template <int S, int L>
__global__ void __launch_bounds__(kGWarps * 32, 1) k_gemv_group(const uint8_t* __restrict__ plan) {
    g_body<1, g_chunk_groups(1), S, L>(plan);
}

// Several batch rows per problem: at most 16 warps, so 128 registers a thread.
template <int NB, int S, int L>
__global__ void __launch_bounds__(16 * 32, 1) k_gemv_group_b(const uint8_t* __restrict__ plan) {
    g_body<NB, g_chunk_groups(NB), S, L>(plan);
}

template <int S>
__global__ void __launch_bounds__(kGWarps * 32, 1) k_gemv_group1(const __grid_constant__ GSingle plan) {
    g_body<1, g_chunk_groups(1), S, kLayoutCanonical>(reinterpret_cast<const uint8_t*>(&plan));
}

// One problem at 2-6 batch rows (bit1_gemv_ex with BIT1_GEMV_STREAM).
template <int NB, int S>
__global__ void __launch_bounds__(16 * 32, 1) k_gemv_group1b(const __grid_constant__ GSingle plan) {
    g_body<NB, g_chunk_groups(NB), S, kLayoutCanonical>(reinterpret_cast<const uint8_t*>(&plan));
}

// ---------------------------------------------------------------- host
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode() {
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

int chunk_groups(int nb, int engine) { return engine == kGEngineMma ? g_mma_chunk_groups(nb) : g_chunk_groups(nb); }
int seg_blocks(int nb, int engine) { return engine == kGEngineMma ? g_mma_seg_blocks(nb) : g_seg_blocks(nb); }

bool encode_prob(GProb& g, const bit1_gemv_problem& pb, int nb, int engine) {
    auto enc = g_encode();
    if (!enc) return false;
    const int64_t G = pb.K / 128;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)(pb.K / 8), (cuuint64_t)pb.N};
        const cuuint64_t strides[1] = {(cuuint64_t)(pb.K / 8)};
        const cuuint32_t box[2] = {128, 32};
        const cuuint32_t es[2] = {1, 1};
        if (enc(&g.tm_bits, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, (void*)pb.bits, dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    {
        const cuuint64_t dims[2] = {(cuuint64_t)G, (cuuint64_t)pb.N};
        const cuuint64_t strides[1] = {(cuuint64_t)(G * 2)};
        const cuuint32_t box[2] = {8, 32};
        const cuuint32_t es[2] = {1, 1};
        if (enc(&g.tm_sc, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, (void*)pb.scales, dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    g.x = pb.x;
    g.y = pb.y;
    g.N = (int)pb.N;
    g.K = (int)pb.K;
    g.G = (int)G;
    g.RB = (int)((pb.N + 31) / 32);
    g.y_bf16 = pb.y_dtype == BIT1_BF16;
    g.swiglu = pb.epilogue == BIT1_EPI_SWIGLU;
    const int cg = chunk_groups(nb, engine);
    g.nch = (int)((G + cg - 1) / cg);
    return true;
}

// Contiguous block ranges, one per CTA, balanced on an estimate of each
// CTA's time: a block costs K (its bytes are proportional to K; its lookups
// to K times the batch rows) and every table build (first block of a problem
// in the CTA, and every seg-th block of a problem with several K chunks)
// costs phase_cost() per chunk.  A greedy pass packs blocks in order under a
// per-CTA budget; a binary search finds the smallest budget that fits in
// nctas CTAs.  Then the shared memory layout; false if it does not fit.
// Batch 1, fitted on one B300 so that CTA finishing times do not grow with
// their phase count (8B- and 27B-class sweeps): a phase costs about six
// 4096-wide blocks plus six more for a full chunk of tables.
constexpr double kGBuildCost = 6.0 * 4096;    // several rows: one chunk build ~ six 4096-wide blocks (measured)
constexpr double kGPhaseFixed = 6.0 * 4096;   // batch 1: a phase's barriers, activations, prescales
constexpr double kGPhaseTables = 6.0 * 4096;  // batch 1: building a full chunk's tables (32 groups)

// Cost of the table builds of one pass over all K chunks of problem p.
double phase_cost(const GProb& pr, int nb, int engine) {
    if (engine == kGEngineMma) return kGPhaseFixed * pr.nch;     // barriers, prescales, fragment build
    if (nb > 1) return kGBuildCost * pr.nch * (nb * g_chunk_groups(nb) / 32.0);
    return kGPhaseFixed * pr.nch + kGPhaseTables * (double)pr.G / g_chunk_groups(1);
}
// Cost of a 32-row block per input, relative to batch 1's table lookups.
double row_factor(int nb, int engine) {
    if (engine == kGEngineMma) return g_mma_nt(nb) == 1 ? 1.5 : 2.5;   // per weight, not per batch row
    return 1.0 + 0.8 * (nb - 1);                  // lookups grow with the batch, the weight reads do not
}

int partition(const std::vector<GProb>& probs, double T, std::vector<GRange>* out, int nb, int engine) {
    const int n = (int)probs.size();
    const int seg = seg_blocks(nb, engine);
    const double rowf = row_factor(nb, engine);
    int ctas = 1;
    double cur = 0.0;
    GRange r{0, 0, 0, 0};
    for (int p = 0; p < n; ++p) {
        int taken = 0;
        const double c = (double)probs[p].K * rowf;
        const double build = phase_cost(probs[p], nb, engine);
        for (int b = 0; b < probs[p].RB; ++b) {
            double add = c;
            if (taken == 0 || (probs[p].nch > 1 && taken % seg == 0)) add += build;
            if (cur > 0.0 && cur + add > T) {
                if (out) { r.p1 = p; r.b1 = b; out->push_back(r); }
                r = GRange{p, b, p, b};
                ++ctas;
                cur = 0.0;
                taken = 0;
                add = c + build;
            }
            cur += add;
            ++taken;
        }
    }
    if (out) { r.p1 = n - 1; r.b1 = probs[n - 1].RB; out->push_back(r); }
    return ctas;
}

bool plan_layout(const std::vector<GProb>& probs, int nctas, int nb, int engine, GHeader& h,
                 std::vector<GRange>& ranges) {
    const int n = (int)probs.size();
    const int CG = chunk_groups(nb, engine), seg = seg_blocks(nb, engine);
    const double rowf = row_factor(nb, engine);
    double total = 0.0;
    for (int p = 0; p < n; ++p)
        total += (double)probs[p].RB * probs[p].K * rowf + phase_cost(probs[p], nb, engine);
    double lo = total / nctas, hi = total + (kGBuildCost + kGPhaseFixed + kGPhaseTables) * nb * 8;
    for (int it = 0; it < 60 && hi - lo > 1e-4 * lo; ++it) {
        const double mid = 0.5 * (lo + hi);
        if (partition(probs, mid, nullptr, nb, engine) <= nctas) hi = mid;
        else lo = mid;
    }
    ranges.clear();
    partition(probs, hi, &ranges, nb, engine);
    while ((int)ranges.size() < nctas)            // CTAs without work
        ranges.push_back(GRange{n - 1, probs[n - 1].RB, n - 1, probs[n - 1].RB});
    for (const GRange& r : ranges)
        if (r.p1 - r.p0 + 1 > kGMaxProbsPerCta) return false;
    int part_rows = 0;
    for (const GRange& r : ranges)
        for (int p = r.p0; p <= r.p1 && p < n; ++p) {
            if (probs[p].nch <= 1) continue;
            const int bs = p == r.p0 ? r.b0 : 0, be = p == r.p1 ? r.b1 : probs[p].RB;
            if (be > bs) part_rows = std::max(part_rows, std::min(be - bs, seg) * 32);
        }
    h.count = n;
    h.nctas = nctas;
    h.nb = nb;
    h.part_rows = part_rows;
    h.seg_blocks = seg;
    h.engine = engine;
    // table engine: every batch row's tables; MMA engine: the chunk's activation fragments
    const int tables = engine == kGEngineMma ? g_mma_nt(nb) * CG * 8 * 32 * 8 : nb * CG * kT6GroupBytes;
    // (warps, stages per warp) in order of preference; the first that fits
    // wins.  Several batch rows: at most 16 warps (the kernel's register cap).
    static const int kCfg[][2] = {{20, 1}, {16, 1}, {12, 1}, {8, 2}, {8, 1}};
    for (const auto& cf : kCfg) {
        const int W = cf[0], S = cf[1];
        if ((nb > 1 || engine == kGEngineMma) && W > 16) continue;   // those kernels: at most 16 warps
        {
            uint32_t off = (uint32_t)(W * S * kGStageBytes);
            const uint32_t off_tables = off;  off += tables;
            const uint32_t off_fac = off;     off += std::max(nb * CG * 8, 32 * 4);   // table engine: 2^m_g and 2^-m_g per row and group; MMA engine: 2^-m_b, 2^m_b
            const uint32_t off_xraw = off;    off += engine == kGEngineMma ? 0 : nb * CG * 128 * 2;
            const uint32_t off_pinfo = off;   off += kGMaxProbsPerCta * 16;
            const uint32_t off_part = off;    off += (uint32_t)(part_rows * nb) * 4;
            if (nb == 1) off += (uint32_t)((W - 1) * (CG / 8) * 32) * 4;   // unit partials (see GCtx)
            off = (off + 7u) & ~7u;
            const uint32_t off_bars = off;    off += W * S * 8 + 8;
            const size_t smem = 1024 + (size_t)off;
            if (smem <= (size_t)kGMaxSmem) {
                h.W = W;
                h.S = S;
                h.off_tables = off_tables;
                h.off_fac = off_fac;
                h.off_xraw = off_xraw;
                h.off_pinfo = off_pinfo;
                h.off_part = off_part;
                h.off_bars = off_bars;
                h.smem_bytes = (int)smem;
                return true;
            }
        }
    }
    return false;
}

bool problem_ok(const bit1_gemv_problem& pb) {
    return pb.bits && pb.scales && pb.x && pb.y && pb.N >= 1 && pb.N <= (1LL << 30) && pb.K >= 1024 &&
           pb.K % 1024 == 0 && pb.K <= (1LL << 20) && (pb.y_dtype == BIT1_F32 || pb.y_dtype == BIT1_BF16) &&
           ((uintptr_t)pb.bits & 15) == 0 && ((uintptr_t)pb.scales & 15) == 0 && ((uintptr_t)pb.x & 15) == 0 &&
           ((uintptr_t)pb.y & 15) == 0 &&
           (pb.epilogue == BIT1_EPI_NONE || (pb.epilogue == BIT1_EPI_SWIGLU && pb.N % 2 == 0));
}

cudaError_t set_smem_attr(const void* f) {
    return func_attrs(f, kGMaxSmem, false);
}

}  // namespace

size_t group_plan_bytes(int count) {
    if (count < 1) return 0;
    const size_t ranges = sizeof(GHeader) + (size_t)kGMaxCtas * sizeof(GRange);
    const size_t probs_off = (ranges + 127) & ~(size_t)127;
    return probs_off + (size_t)count * sizeof(GProb);
}

bit1_status group_plan(const bit1_gemv_problem* problems, int count, int nb, int layout, int engine,
                       void* host_plan, size_t bytes) {
    if (count < 1 || !problems || !host_plan) return BIT1_EINVAL;
    if (engine != kGEngineTables && engine != kGEngineMma) return BIT1_EINVAL;
    if (nb < 1 || nb > (engine == kGEngineMma ? kGMaxNBMma : kGMaxNB)) return BIT1_ESHAPE;
    if (layout != kLayoutCanonical && layout != kLayoutG128x) return BIT1_EINVAL;
    if (engine == kGEngineMma && layout != kLayoutCanonical) return BIT1_EINVAL;
    if (bytes < group_plan_bytes(count) || ((uintptr_t)host_plan & 127)) return BIT1_EINVAL;
    for (int i = 0; i < count; ++i)
        if (!problem_ok(problems[i])) return BIT1_ESHAPE;
    std::vector<GProb> probs(count);
    for (int i = 0; i < count; ++i)
        if (!encode_prob(probs[i], problems[i], nb, engine)) return BIT1_ECUDA;
    GHeader h{};
    std::vector<GRange> ranges;
    const int nctas = std::min(sm_count(), kGMaxCtas);
    if (!plan_layout(probs, nctas, nb, engine, h, ranges)) return BIT1_ESHAPE;
    h.layout = layout;
    const size_t r_off = sizeof(GHeader);
    const size_t p_off = (r_off + (size_t)kGMaxCtas * sizeof(GRange) + 127) & ~(size_t)127;
    h.ranges_off = (int)r_off;
    h.probs_off = (int)p_off;
    uint8_t* out = static_cast<uint8_t*>(host_plan);
    std::memset(out, 0, bytes);
    std::memcpy(out, &h, sizeof(h));
    std::memcpy(out + r_off, ranges.data(), ranges.size() * sizeof(GRange));
    std::memcpy(out + p_off, probs.data(), probs.size() * sizeof(GProb));
    return BIT1_OK;
}

template <int L>
const void* group_kernel_s(int nb, bool s2) {
    switch (nb) {
        case 1: return s2 ? (const void*)k_gemv_group<2, L> : (const void*)k_gemv_group<1, L>;
        case 2: return s2 ? (const void*)k_gemv_group_b<2, 2, L> : (const void*)k_gemv_group_b<2, 1, L>;
        case 3: return s2 ? (const void*)k_gemv_group_b<3, 2, L> : (const void*)k_gemv_group_b<3, 1, L>;
        case 4: return s2 ? (const void*)k_gemv_group_b<4, 2, L> : (const void*)k_gemv_group_b<4, 1, L>;
        case 5: return s2 ? (const void*)k_gemv_group_b<5, 2, L> : (const void*)k_gemv_group_b<5, 1, L>;
        case 6: return s2 ? (const void*)k_gemv_group_b<6, 2, L> : (const void*)k_gemv_group_b<6, 1, L>;
        default: return nullptr;
    }
}
template <int L>
const void* group_kernel(int nb, int S) { return group_kernel_s<L>(nb, S == 2); }

cudaError_t launch_group(const void* device_plan, const void* host_plan, bool pdl, cudaStream_t stream) {
    const GHeader* h = static_cast<const GHeader*>(host_plan);
    if (h->kind != kPlanKindTables) return cudaErrorInvalidValue;
    if (h->S != 1 && h->S != 2) return cudaErrorInvalidValue;
    if (h->layout != kLayoutCanonical && h->layout != kLayoutG128x) return cudaErrorInvalidValue;
    const void* fn = nullptr;
    if (h->engine == kGEngineMma) {
        if (h->layout != kLayoutCanonical || h->nb < 1 || h->nb > kGMaxNBMma) return cudaErrorInvalidValue;
        fn = g_mma_nt(h->nb) == 1 ? (h->S == 2 ? (const void*)k_gemv_group_mma<1, 2> : (const void*)k_gemv_group_mma<1, 1>)
                                  : (h->S == 2 ? (const void*)k_gemv_group_mma<2, 2> : (const void*)k_gemv_group_mma<2, 1>);
    } else if (h->engine == kGEngineTables) {
        fn = h->layout == kLayoutG128x ? group_kernel<kLayoutG128x>(h->nb, h->S)
                                       : group_kernel<kLayoutCanonical>(h->nb, h->S);
    }
    if (!fn) return cudaErrorInvalidValue;
    cudaError_t e = set_smem_attr(fn);
    if (e != cudaSuccess) return e;
    const uint8_t* dp = static_cast<const uint8_t*>(device_plan);
    void* args[] = {(void*)&dp};
    return launch(fn, dim3((unsigned)h->nctas), dim3((unsigned)(h->W * 32)), (size_t)h->smem_bytes, stream, pdl,
                  args);
}

bool group1_supported(int64_t B, int64_t N, int64_t K) {
    return B >= 1 && N >= 1 && N <= (1LL << 30) && K >= 1024 && K % 1024 == 0 && K <= (1LL << 20);
}

int group1_launch_count(int64_t B) { return (int)((B + kGMaxNB - 1) / kGMaxNB); }

namespace {

template <int NB>
const void* group1_kernel(int S) {
    if constexpr (NB == 1) return S == 2 ? (const void*)k_gemv_group1<2> : (const void*)k_gemv_group1<1>;
    else return S == 2 ? (const void*)k_gemv_group1b<NB, 2> : (const void*)k_gemv_group1b<NB, 1>;
}

const void* group1_kernel_nb(int nb, int S) {
    switch (nb) {
        case 1: return group1_kernel<1>(S);
        case 2: return group1_kernel<2>(S);
        case 3: return group1_kernel<3>(S);
        case 4: return group1_kernel<4>(S);
        case 5: return group1_kernel<5>(S);
        case 6: return group1_kernel<6>(S);
        default: return nullptr;
    }
}

}  // namespace

// One problem as a grouped launch: B rows in ceil(B / 6) launches of balanced
// row counts (7 rows: 4 + 3), each with its plan passed by value.
cudaError_t launch_gemv_group1(const GemvArgs& a) {
    if (!group1_supported(a.B, a.N, a.K)) return cudaErrorInvalidValue;
    const int launches = group1_launch_count(a.B);
    const int64_t out_n = a.swiglu ? a.N / 2 : a.N;
    const size_t ysz = a.y_bf16 ? 2 : 4;
    static GSingle single;  // large: keep off the stack; filled and copied into each launch
    static std::mutex mu;
    std::lock_guard<std::mutex> lk(mu);
    int64_t b0 = 0;
    for (int l = 0; l < launches; ++l) {
        const int nb = (int)((a.B - b0 + (launches - l) - 1) / (launches - l));
        bit1_gemv_problem pb{};
        pb.bits = a.bits;
        pb.scales = a.scales;
        pb.x = a.x + b0 * a.K;
        pb.y = static_cast<uint8_t*>(a.y) + (size_t)b0 * (size_t)out_n * ysz;
        pb.N = a.N;
        pb.K = a.K;
        pb.y_dtype = a.y_bf16 ? BIT1_BF16 : BIT1_F32;
        pb.epilogue = a.swiglu ? BIT1_EPI_SWIGLU : BIT1_EPI_NONE;
        // y of a later launch starts b0 rows in, which need not be 16-byte
        // aligned; the kernels store y element by element, so the caller's
        // (checked) base pointer is what the shape check sees.
        void* const y_rows = pb.y;
        pb.y = a.y;
        if (!problem_ok(pb)) return cudaErrorInvalidValue;
        pb.y = y_rows;
        std::vector<GProb> probs(1);
        if (!encode_prob(probs[0], pb, nb, kGEngineTables)) return cudaErrorInvalidValue;
        std::memset(&single, 0, sizeof(single));
        std::vector<GRange> ranges;
        const int nctas = std::min(sm_count(), kGMaxCtas);
        if (!plan_layout(probs, nctas, nb, kGEngineTables, single.h, ranges)) return cudaErrorInvalidValue;
        single.h.layout = kLayoutCanonical;
        single.h.ranges_off = (int)offsetof(GSingle, r);
        single.h.probs_off = (int)offsetof(GSingle, p);
        std::memcpy(single.r, ranges.data(), ranges.size() * sizeof(GRange));
        single.p = probs[0];
        if (single.h.S != 1 && single.h.S != 2) return cudaErrorInvalidValue;
        const void* fn = group1_kernel_nb(nb, single.h.S);
        if (!fn) return cudaErrorInvalidValue;
        cudaError_t e = set_smem_attr(fn);
        if (e != cudaSuccess) return e;
        void* args[] = {(void*)&single};
        e = launch(fn, dim3((unsigned)single.h.nctas), dim3((unsigned)(single.h.W * 32)), (size_t)single.h.smem_bytes,
                   a.stream, a.pdl, args);
        if (e != cudaSuccess) return e;
        b0 += nb;
    }
    return cudaSuccess;
}

bool mma1_supported(int64_t B, int64_t N, int64_t K) { return group1_supported(B, N, K); }

int mma1_launch_count(int64_t B) { return (int)((B + kGMaxNBMma - 1) / kGMaxNBMma); }

// One problem on the MMA engine: B rows in ceil(B / 16) launches of balanced
// row counts, each with its plan passed by value.
cudaError_t launch_gemv_mma1(const GemvArgs& a) {
    if (!mma1_supported(a.B, a.N, a.K)) return cudaErrorInvalidValue;
    const int launches = mma1_launch_count(a.B);
    const int64_t out_n = a.swiglu ? a.N / 2 : a.N;
    const size_t ysz = a.y_bf16 ? 2 : 4;
    static GSingle single;  // large: keep off the stack; filled and copied into each launch
    static std::mutex mu;
    std::lock_guard<std::mutex> lk(mu);
    int64_t b0 = 0;
    for (int l = 0; l < launches; ++l) {
        const int nb = (int)((a.B - b0 + (launches - l) - 1) / (launches - l));
        bit1_gemv_problem pb{};
        pb.bits = a.bits;
        pb.scales = a.scales;
        pb.x = a.x + b0 * a.K;
        pb.y = static_cast<uint8_t*>(a.y) + (size_t)b0 * (size_t)out_n * ysz;
        pb.N = a.N;
        pb.K = a.K;
        pb.y_dtype = a.y_bf16 ? BIT1_BF16 : BIT1_F32;
        pb.epilogue = a.swiglu ? BIT1_EPI_SWIGLU : BIT1_EPI_NONE;
        // y of a later launch starts b0 rows in, which need not be 16-byte
        // aligned; the kernels store y element by element, so the caller's
        // (checked) base pointer is what the shape check sees.
        void* const y_rows = pb.y;
        pb.y = a.y;
        if (!problem_ok(pb)) return cudaErrorInvalidValue;
        pb.y = y_rows;
        std::vector<GProb> probs(1);
        if (!encode_prob(probs[0], pb, nb, kGEngineMma)) return cudaErrorInvalidValue;
        std::memset(&single, 0, sizeof(single));
        std::vector<GRange> ranges;
        const int nctas = std::min(sm_count(), kGMaxCtas);
        if (!plan_layout(probs, nctas, nb, kGEngineMma, single.h, ranges)) return cudaErrorInvalidValue;
        single.h.layout = kLayoutCanonical;
        single.h.ranges_off = (int)offsetof(GSingle, r);
        single.h.probs_off = (int)offsetof(GSingle, p);
        std::memcpy(single.r, ranges.data(), ranges.size() * sizeof(GRange));
        single.p = probs[0];
        if (single.h.S != 1 && single.h.S != 2) return cudaErrorInvalidValue;
        const bool one = g_mma_nt(nb) == 1;
        const void* fn = one ? (single.h.S == 2 ? (const void*)k_gemv_group1_mma<1, 2> : (const void*)k_gemv_group1_mma<1, 1>)
                             : (single.h.S == 2 ? (const void*)k_gemv_group1_mma<2, 2> : (const void*)k_gemv_group1_mma<2, 1>);
        cudaError_t e = set_smem_attr(fn);
        if (e != cudaSuccess) return e;
        void* args[] = {(void*)&single};
        e = launch(fn, dim3((unsigned)single.h.nctas), dim3((unsigned)(single.h.W * 32)), (size_t)single.h.smem_bytes,
                   a.stream, a.pdl, args);
        if (e != cudaSuccess) return e;
        b0 += nb;
    }
    return cudaSuccess;
}

unsigned int group_take_timeouts() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_group_wait_timeouts, sizeof(v)) != cudaSuccess) return 0xffffffffu;
    cudaMemcpyToSymbol(g_group_wait_timeouts, &zero, sizeof(zero));
    return v;
}

}  // namespace bit1
