// A dependent chain of batch-1 products in ONE persistent launch: the decode
// step's linear layers in their data order (q|k|v, o, gate|up, down, ... and
// the LM head), each stage reading -- if it wants -- the output of an earlier
// stage as its activations.
//
// Why: at batch 1 a decode step reads every weight once and the time goes to
// weight traffic and to kernel launch / synchronisation latency (web page
// "Bonsai 27B: 노트북과 폰에서 실행되는 27B급 이진 및 삼진 저비트 LLM", sections
// "27B 규모에서 효율은 선택이 아닌 제약" and "하이브리드 어텐션을 위한 저비트
// 커널").  A chain of separate launches pays a kernel turn-around per matrix
// (3-7 us each on this part, against 0.3-1.9 us of weight traffic); here a
// grid-wide barrier replaces it.
//
// Design: a cooperative launch of one 512-thread CTA per SM.  Each stage is the
// nibble-table product of gemv_lut.cu (lanes over the row's words, fp32 tables
// of 16 signed sums per four inputs, warps over rows): the CTA takes a
// contiguous range of the stage's rows (or gate/up pairs with the SwiGLU
// epilogue of the Bonsai 27B page's section "Bonsai 27B의 표현 방식").  Before
// waiting at the barrier that ends the previous stage, every warp already loads
// its first rows of this stage's weights (they do not depend on any stage), so
// the weight stream runs through the barrier; after it the CTA builds the tables
// from x through L2 (ld.global.cg: x may have been written by other CTAs in
// this launch), multiplies and writes y, then arrives at the next barrier.
// Every row is computed with the same arithmetic as the single-launch kernel,
// so the results are bit-identical to running the stages one by one with
// BIT1_GEMV_LUT.  The barrier (a count and a generation word in the plan) is
// self-resetting; every wait on it is bounded and a wait that gives up stops
// the CTA and records the event (bit1_device_wait_timeouts).
#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "internal.h"
#include "lut_common.cuh"

namespace bit1 {

__device__ unsigned int g_chain_wait_timeouts = 0;

namespace {

struct alignas(64) CStage {
    const uint8_t* bits;
    const uint16_t* scales;
    const uint16_t* x;
    void* y;
    int N, M, y_bf16, swiglu;   // M = K / 1024
};
static_assert(sizeof(CStage) == 64, "stage size");

struct CHeader {
    int count;                  // stages
    int smem;                   // dynamic shared memory of the launch (largest stage's tables)
};

constexpr size_t kChainBarOff = 128;     // {arrivals, generation}, a 128-byte line of its own
constexpr size_t kChainStagesOff = 256;
constexpr int kChainSpin = 1 << 22;      // barrier polls (with a short sleep) before giving up

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Thread 0, after the CTA's __syncthreads: publish this CTA's writes and
// arrive.  Returns the generation the CTA then waits to see change.  The
// generation cannot move before every CTA (this one included) has arrived,
// so reading it first is safe; the last arrival resets the count before it
// advances the generation, and nobody arrives again before seeing that.
__device__ __forceinline__ unsigned chain_arrive(unsigned* bar, unsigned nctas) {
    const unsigned gen = ld_acquire_gpu(bar + 1);
    __threadfence();
    if (atomicAdd(bar, 1u) == nctas - 1u) {
        atomicExch(bar, 0u);
        __threadfence();
        atomicAdd(bar + 1, 1u);
    }
    return gen;
}

__device__ __forceinline__ bool chain_wait(const unsigned* bar, unsigned gen) {
    for (int i = 0; i < kChainSpin; ++i) {
        if (ld_acquire_gpu(bar + 1) != gen) return true;
        __nanosleep(64);
    }
    return false;
}

// One stage.  sh[0]: generation to wait for (thread 0 only), sh[1]: 1 while no
// wait gave up (written by thread 0 before a __syncthreads, read by all after
// it).
template <int M, bool SWIGLU>
__device__ __forceinline__ void chain_stage(const CStage st, unsigned* bar, bool first, bool last, float* tab,
                                            uint32_t tbase, unsigned* sh) {
    using C = LutCfg<M>;
    constexpr int D = C::D, NS = C::NS;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int64_t U = SWIGLU ? st.N / 2 : st.N;
    const int64_t n0 = U * blockIdx.x / gridDim.x, n1 = U * (blockIdx.x + 1) / gridDim.x;
    const int64_t mine = n1 - n0 > warp ? (n1 - n0 - warp + nw - 1) / nw : 0;
    const int64_t R = SWIGLU ? 2 * mine : mine;             // rows this warp runs
    auto row_of = [&](int64_t t) -> int64_t {
        if constexpr (SWIGLU) return 2 * (n0 + warp + (t >> 1) * nw) + (t & 1);
        else return n0 + warp + t * nw;
    };

    uint32_t wb[D][M];
    uint32_t sb[D][NS];
#pragma unroll
    for (int d = 0; d < D; ++d)
        if (d < R) load_row<M>(st.bits, st.scales, row_of(d), lane, wb[d], sb[d]);

    if (!first) {                                           // earlier stages complete
        if (threadIdx.x == 0 && sh[1] && !chain_wait(bar, sh[0])) {
            atomicOr(&g_chain_wait_timeouts, 1u);
            sh[1] = 0;
        }
        __syncthreads();
        if (!sh[1]) return;
    }
    lut_build<M, true>(st.x, tab);
    __syncthreads();

    const uint32_t lb = tbase + 4u * (uint32_t)lane;
    const int o = (M % 4 == 0) ? 0 : ((lane * M) & 3);
    float gate = 0.f;
    for (int64_t base = 0; base < R; base += D) {
#pragma unroll
        for (int d = 0; d < D; ++d) {
            const int64_t t = base + d;
            if (t >= R) break;
            const int64_t row = row_of(t);
            float v = lut_row<M>(wb[d], sb[d], lb, o, [&] {
                if (t + D < R) load_row<M>(st.bits, st.scales, row_of(t + D), lane, wb[d], sb[d]);
            });
            int64_t out = row;
            if constexpr (SWIGLU) {
                if (!(t & 1)) {
                    gate = v;
                    continue;
                }
                v = gate / (1.f + expf(-gate)) * v;
                out = row >> 1;
            }
            if (lane == 0) {
                if (st.y_bf16) reinterpret_cast<uint16_t*>(st.y)[out] = f32_to_bf16_bits(v);
                else reinterpret_cast<float*>(st.y)[out] = v;
            }
        }
    }
    __syncthreads();                                        // the CTA's outputs are written
    if (!last && threadIdx.x == 0) sh[0] = chain_arrive(bar, gridDim.x);
}

}  // namespace

__global__ void __launch_bounds__(kLutThreads, 1) k_gemv_chain(uint8_t* plan) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ unsigned sh[2];
    const uint32_t sraw = (uint32_t)__cvta_generic_to_shared(smem_raw);
    const uint32_t tbase = (sraw + 2047u) & ~2047u;
    float* tab = reinterpret_cast<float*>(smem_raw + (tbase - sraw));
    const CHeader* H = reinterpret_cast<const CHeader*>(plan);
    const CStage* S = reinterpret_cast<const CStage*>(plan + kChainStagesOff);
    unsigned* bar = reinterpret_cast<unsigned*>(plan + kChainBarOff);
    if (threadIdx.x == 0) {
        sh[0] = 0;
        sh[1] = 1;
    }
    __syncthreads();
    const int count = H->count;
#pragma unroll 1
    for (int s = 0; s < count; ++s) {
        CStage st;
        st.bits = S[s].bits;
        st.scales = S[s].scales;
        st.x = S[s].x;
        st.y = S[s].y;
        st.N = S[s].N;
        st.M = S[s].M;
        st.y_bf16 = S[s].y_bf16;
        st.swiglu = S[s].swiglu;
        const bool first = s == 0, last = s + 1 == count;
#define BIT1_CHAIN_CASE(m)                                                              \
    case m:                                                                             \
        if (st.swiglu) chain_stage<m, true>(st, bar, first, last, tab, tbase, sh);     \
        else chain_stage<m, false>(st, bar, first, last, tab, tbase, sh);              \
        break;
        switch (st.M) {
            BIT1_CHAIN_CASE(1) BIT1_CHAIN_CASE(2) BIT1_CHAIN_CASE(3) BIT1_CHAIN_CASE(4)
            BIT1_CHAIN_CASE(5) BIT1_CHAIN_CASE(6) BIT1_CHAIN_CASE(7) BIT1_CHAIN_CASE(8)
            BIT1_CHAIN_CASE(9) BIT1_CHAIN_CASE(10) BIT1_CHAIN_CASE(11) BIT1_CHAIN_CASE(12)
            BIT1_CHAIN_CASE(13)
            default: break;
        }
#undef BIT1_CHAIN_CASE
        // No block-wide read of sh[1] here: thread 0 may already be writing it in
        // the next stage.  A stage whose wait gave up returns before its tables,
        // and so does every later one.
    }
}

// ---------------------------------------------------------------- host
namespace {

bool ranges_overlap(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
    return a0 < b0 + nb && b0 < a0 + na;
}

}  // namespace

size_t chain_plan_bytes(int count) {
    if (count < 1) return 0;
    return kChainStagesOff + (size_t)count * sizeof(CStage);
}

bit1_status chain_plan(const bit1_gemv_problem* stages, int count, void* host_plan, size_t bytes) {
    if (count < 1 || !stages || !host_plan) return BIT1_EINVAL;
    if (bytes < chain_plan_bytes(count) || ((uintptr_t)host_plan & 127)) return BIT1_EINVAL;
    int smem = 0;
    for (int i = 0; i < count; ++i) {
        const bit1_gemv_problem& p = stages[i];
        if (p.N < 1 || p.N > (1LL << 30) || p.K < 1024 || p.K % 1024 != 0 || p.K / 1024 > kLutMaxM)
            return BIT1_ESHAPE;
        if (p.epilogue != BIT1_EPI_NONE && p.epilogue != BIT1_EPI_SWIGLU) return BIT1_ESHAPE;
        if (p.epilogue == BIT1_EPI_SWIGLU && p.N % 2 != 0) return BIT1_ESHAPE;
        if (!p.bits || !p.scales || !p.x || !p.y) return BIT1_EINVAL;
        if (((uintptr_t)p.bits & 15) || ((uintptr_t)p.scales & 15) || ((uintptr_t)p.x & 15) || ((uintptr_t)p.y & 15))
            return BIT1_EINVAL;
        if (p.y_dtype != BIT1_F32 && p.y_dtype != BIT1_BF16) return BIT1_EINVAL;
        const size_t ybytes = (size_t)(p.epilogue == BIT1_EPI_SWIGLU ? p.N / 2 : p.N) * (p.y_dtype == BIT1_BF16 ? 2 : 4);
        if (ranges_overlap(p.x, (size_t)p.K * 2, p.y, ybytes)) return BIT1_EINVAL;
        smem = std::max(smem, (int)(16384 * (p.K / 1024) + 2048));
    }
    uint8_t* h = static_cast<uint8_t*>(host_plan);
    std::memset(h, 0, chain_plan_bytes(count));
    CHeader hd{count, smem};
    std::memcpy(h, &hd, sizeof(hd));
    for (int i = 0; i < count; ++i) {
        const bit1_gemv_problem& p = stages[i];
        CStage st{};
        st.bits = p.bits;
        st.scales = p.scales;
        st.x = p.x;
        st.y = p.y;
        st.N = (int)p.N;
        st.M = (int)(p.K / 1024);
        st.y_bf16 = p.y_dtype == BIT1_BF16;
        st.swiglu = p.epilogue == BIT1_EPI_SWIGLU;
        std::memcpy(h + kChainStagesOff + (size_t)i * sizeof(CStage), &st, sizeof(st));
    }
    return BIT1_OK;
}

cudaError_t launch_chain(void* device_plan, const void* host_plan, cudaStream_t stream) {
    CHeader hd;
    std::memcpy(&hd, host_plan, sizeof(hd));
    if (hd.count < 1 || hd.smem < 2048 || hd.smem > 16384 * kLutMaxM + 2048) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute((const void*)k_gemv_chain, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         16384 * kLutMaxM + 2048);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, (const void*)k_gemv_chain, kLutThreads, hd.smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)sm_count());            // one CTA per SM, all resident
    cfg.blockDim = dim3(kLutThreads);
    cfg.dynamicSmemBytes = (size_t)hd.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    uint8_t* dp = static_cast<uint8_t*>(device_plan);
    void* args[] = {(void*)&dp};
    return cudaLaunchKernelExC(&cfg, (const void*)k_gemv_chain, args);
}

unsigned int chain_take_timeouts() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_chain_wait_timeouts, sizeof(v)) != cudaSuccess) return 0xffffffffu;
    if (v) cudaMemcpyToSymbol(g_chain_wait_timeouts, &zero, sizeof(zero));
    return v;
}

}  // namespace bit1
