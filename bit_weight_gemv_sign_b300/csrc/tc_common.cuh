// Device helpers of the tcgen05 kernels (gemv_tc.cu: one matrix per launch;
// gemv_tc_group.cu: many matrices in one persistent launch).  The product and
// its numerics are the ones described at the top of gemv_tc.cu: weights as
// +-s in fp16 written to tensor memory, activations as fp16 with a per-row
// power-of-two prescale in shared memory, fp32 accumulators in tensor memory.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "t6_common.cuh"

namespace bit1 {

constexpr int kTcStepK = 128;             // inputs per pipeline step (one scale group)
constexpr int kTcChunkSteps = 4;          // sign-bit box: 64 bytes of each row = 4 steps
constexpr int kTcPrepThreads = 512;
constexpr int kTcPrepUnits = 8;           // 16-byte units of x per prep thread held in registers

__device__ __forceinline__ void tc_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle (8-row x
// 128-byte atoms, consecutive atoms 1024 bytes apart), descriptor version 1.
__device__ __forceinline__ uint64_t tc_desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor of kind::f16 with fp16 A and B, fp32 D, M = 128, N = n.
__device__ __forceinline__ uint32_t tc_idesc_f16(int n) {
    return (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}
// Bounded wait for a single waiting thread that is expected to block for a
// while (a producer or an MMA issuer): each try_wait may suspend the thread
// for up to 20 us until the phase completes, so the waiting thread does not
// spend its sub-partition's issue slots on polling; 2^19 polls bound the wait
// (seconds).
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity) {
    for (uint32_t i = 0; i < (1u << 19); ++i) {
        uint32_t done;
        asm volatile("{.reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p;}"
                     : "=r"(done) : "r"(bar), "r"(parity), "r"(20000u) : "memory");
        if (done) return true;
    }
    return false;
}
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}
__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ void tma_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2, uint32_t bar) {
    asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
                 ::"r"(dst), "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(bar) : "memory");
}
__device__ __forceinline__ uint32_t bf16_mag(uint32_t v) {   // |x| bits; NaN -> 0 (does not set the scale)
    v &= 0x7fffu;
    return v > 0x7f80u ? 0u : v;
}
__device__ __forceinline__ uint32_t bf16x2_max_mag(uint32_t w) { return max(bf16_mag(w & 0xffffu), bf16_mag(w >> 16)); }
__device__ __forceinline__ uint32_t pack_h2(uint32_t lo_bf16, uint32_t hi_bf16, float finv) {
    const __half2 h = __floats2half2_rn(bf16_bits_to_f32(lo_bf16) * finv, bf16_bits_to_f32(hi_bf16) * finv);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// One batch row of the activation prep, run by a whole CTA of kTcPrepThreads
// threads: xp[32q + 2j + h] = fp16(x[32q + j + 16h] * 2^-m) and *xscale = 2^m,
// with m chosen so that max|x * 2^-m| lies in [2^14, 2^15) (exact: bf16 keeps
// 8 significant bits, fp16 11; values more than about 2^38 below the row's
// maximum fall into fp16 subnormals or zero).  x == nullptr: a padding row
// (zeros, scale 1).  `red` is kTcPrepThreads / 32 words of shared memory.
// Thread layout: 16-byte unit u = 8 consecutive inputs; the four units of a
// 32-input block sit in four consecutive lanes, and lanes p and p^2 exchange
// their units to form the (j, j+16) pairs.
__device__ __forceinline__ void tc_prep_row(const uint16_t* __restrict__ x, int K, uint16_t* __restrict__ xp,
                                            float* __restrict__ xscale, uint32_t* red) {
    uint4* out = reinterpret_cast<uint4*>(xp);
    const int units = K / 8;
    if (!x) {
        for (int i = threadIdx.x; i < units; i += blockDim.x) out[i] = make_uint4(0, 0, 0, 0);
        if (threadIdx.x == 0) *xscale = 1.f;
        return;
    }
    const uint4* in = reinterpret_cast<const uint4*>(x);
    const bool resident = units <= kTcPrepThreads * kTcPrepUnits;
    uint4 v[kTcPrepUnits];
    uint32_t m = 0;
    if (resident) {
#pragma unroll
        for (int i = 0; i < kTcPrepUnits; ++i) {
            const int u = threadIdx.x + i * kTcPrepThreads;
            v[i] = u < units ? in[u] : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < kTcPrepUnits; ++i)
            m = max(m, max(max(bf16x2_max_mag(v[i].x), bf16x2_max_mag(v[i].y)),
                           max(bf16x2_max_mag(v[i].z), bf16x2_max_mag(v[i].w))));
    } else {
        for (int u = threadIdx.x; u < units; u += blockDim.x) {
            const uint4 t = in[u];
            m = max(m, max(max(bf16x2_max_mag(t.x), bf16x2_max_mag(t.y)), max(bf16x2_max_mag(t.z), bf16x2_max_mag(t.w))));
        }
    }
    m = __reduce_max_sync(0xffffffffu, m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    m = red[0];
#pragma unroll
    for (int i = 1; i < kTcPrepThreads / 32; ++i) m = max(m, red[i]);
    int mb = 0;
    if (m != 0) {
        const int e = (int)(m >> 7) - 127;            // exponent of max|x| (subnormal -> -127)
        mb = min(max(e - 14, -126), 126);
    }
    const float finv = __uint_as_float((uint32_t)(127 - mb) << 23);
    if (threadIdx.x == 0) *xscale = __uint_as_float((uint32_t)(mb + 127) << 23);
    const int p = threadIdx.x & 3;                     // unit position within its 32-input block
    auto emit = [&](int u, uint4 own) {
        uint4 oth;
        oth.x = __shfl_xor_sync(0xffffffffu, own.x, 2);
        oth.y = __shfl_xor_sync(0xffffffffu, own.y, 2);
        oth.z = __shfl_xor_sync(0xffffffffu, own.z, 2);
        oth.w = __shfl_xor_sync(0xffffffffu, own.w, 2);
        // p = 0/1: inputs 8p..8p+7 (low of the pair) with 16+8p.. (high): pairs 8p..8p+3
        // p = 2/3: partner's low with own high: pairs 8(p-2)+4..+7
        const uint4 lo = (p < 2) ? own : oth, hi = (p < 2) ? oth : own;
        const uint32_t l0 = (p < 2) ? lo.x : lo.z, l1 = (p < 2) ? lo.y : lo.w;
        const uint32_t h0 = (p < 2) ? hi.x : hi.z, h1 = (p < 2) ? hi.y : hi.w;
        uint4 r;
        r.x = pack_h2(l0 & 0xffffu, h0 & 0xffffu, finv);
        r.y = pack_h2(l0 >> 16, h0 >> 16, finv);
        r.z = pack_h2(l1 & 0xffffu, h1 & 0xffffu, finv);
        r.w = pack_h2(l1 >> 16, h1 >> 16, finv);
        const int q = u >> 2;
        const int slot = (p == 0) ? 0 : (p == 2) ? 1 : (p == 1) ? 2 : 3;   // 16-byte slot in the block's 64 output bytes
        if (u < units) out[4 * q + slot] = r;
    };
    if (resident) {
#pragma unroll
        for (int i = 0; i < kTcPrepUnits; ++i) {
            const int u = threadIdx.x + i * kTcPrepThreads;
            if (i * kTcPrepThreads < units) emit(u, v[i]);   // warp-uniform (units is a multiple of 128)
        }
    } else {
        for (int u = threadIdx.x; u < units; u += blockDim.x) emit(u, in[u]);
    }
}

// One row's 128-input step of A: the 16 sign bytes w (bit 1 -> +s) become 64
// fp16x2 words written to tensor memory at taddr (lane base + column).
// Inside every 32-bit sign word, inputs k and k+16 share one fp16x2 register
// (sign bits 15 and 31), so one shift and one LOP3 produce two weights; the
// activations are stored in the same permuted K order.  s2 = s | s << 16.
__device__ __forceinline__ void tc_unpack_step(const uint4& w, uint32_t s2, uint32_t taddr) {
    const uint32_t words[4] = {~w.x, ~w.y, ~w.z, ~w.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            // bits j and j+16 to the fp16 sign positions 15 and 31; the shift is
            // written as a multiply so that it can issue on the FMA pipe
            uint32_t t;
            asm("mul.lo.u32 %0, %1, %2;" : "=r"(t) : "r"(words[q]), "r"(1u << (15 - j)));
            v[j] = (t & 0x80008000u) ^ s2;
        }
        asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                     ::"r"(taddr + 16u * q), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]),
                       "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]),
                       "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]) : "memory");
    }
}

// The MMAs of one 128-input step into accumulator d_addr: the 16-input slices
// kk = kk0, kk0 + kkd, ... of A (tensor memory at a0, 8 columns per slice)
// against B (shared memory at bst: two 64-wide K slabs of btile bytes, 128-byte
// swizzle).  The first slice overwrites the accumulator when `first`.
__device__ __forceinline__ void tc_mma_step(uint32_t d_addr, uint32_t a0, uint32_t bst, uint32_t btile,
                                            uint32_t idesc, int kk0, int kkd, bool first) {
#pragma unroll
    for (int kk = kk0; kk < kTcStepK / 16; kk += kkd) {
        const uint64_t bdesc = tc_desc_sw128(bst + (uint32_t)(kk >> 2) * btile + (uint32_t)(kk & 3) * 32u);
        const uint32_t acc = (!first || kk > kk0) ? 1u : 0u;
        asm volatile("{.reg .pred pa; setp.ne.b32 pa, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, pa;}"
                     ::"r"(d_addr), "r"(a0 + 8u * (uint32_t)kk), "l"(bdesc), "r"(idesc), "r"(acc) : "memory");
    }
}

// One MMA (M = 128, K = 16) into d_addr: A in tensor memory at a_tmem, B by
// descriptor; `accumulate` false overwrites the accumulator.
__device__ __forceinline__ void tc_mma1(uint32_t d_addr, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                        bool accumulate) {
    asm volatile("{.reg .pred pa; setp.ne.b32 pa, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, pa;}"
                 ::"r"(d_addr), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate ? 1u : 0u) : "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// 16 consecutive fp32 columns of this warp's 32 lanes from tensor memory
// (call tcgen05.wait::ld before using d).
__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&d)[16]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3]), "=r"(d[4]), "=r"(d[5]), "=r"(d[6]),
                   "=r"(d[7]), "=r"(d[8]), "=r"(d[9]), "=r"(d[10]), "=r"(d[11]), "=r"(d[12]), "=r"(d[13]),
                   "=r"(d[14]), "=r"(d[15])
                 : "r"(taddr) : "memory");
}
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

}  // namespace bit1
