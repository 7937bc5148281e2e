// C ABI of the bit1 library: argument validation (on the host, before any
// CUDA call, so that a rejected call launches and modifies nothing), kernel
// selection and launch.  Declarations and their documentation: bit1.h.
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"
#include "internal.h"

namespace bit1 {

cudaError_t launch(const void* func, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                   bool pdl, void** args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelExC(&cfg, func, args);
}

cudaError_t func_attrs(const void* fn, int smem_bytes, bool nonportable_clusters) {
    static std::mutex mu;
    static std::map<std::pair<int, const void*>, int> done;   // (device, kernel) -> smem limit set
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(mu);
    auto it = done.find({dev, fn});
    if (it != done.end() && it->second >= smem_bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e == cudaSuccess && nonportable_clusters)
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();     // do not leave the failure pending for the next launch
        return e;
    }
    done[{dev, fn}] = smem_bytes;
    return cudaSuccess;
}

int sm_count() {
    static int cached[64];
    static std::once_flag once[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
    std::call_once(once[dev], [dev] {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
        cached[dev] = v;
    });
    return cached[dev];
}

}  // namespace bit1

using namespace bit1;

namespace {

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

bool shape_ok(int64_t B, int64_t N, int64_t K) {
    return B >= 1 && N >= 1 && K >= 128 && K % 128 == 0 && B <= 0x7fffffffLL &&
           N <= 0x7fffffffLL && K <= (1LL << 24);
}

bit1_status from_cuda(cudaError_t e) { return e == cudaSuccess ? BIT1_OK : BIT1_ECUDA; }

// Whether the tensor-core kernel beats the 6-bit tables at batch B, from
// per-call times measured on one B300 (graph replay, weights rotated past
// L2).  The tensor cores take 11-25 us per call almost independently of B
// (4096x4096 11 us, 12288x4096 18, 4096x12288 18, 17408x5120 21, 5120x17408
// 24); the tables grow with B.  Crossovers: 4096x4096 and 4096x12288 from
// B = 4, 17408x5120 from B = 5, 12288x4096 from B = 8.  Where the tables
// cannot take the shape (no cluster split of K, e.g. K = 17408) the rest is
// far slower (warp-per-row: 800 us at B = 2 on 5120x17408).
bool tc_beats_tables(int64_t B, int64_t N, int64_t K, bool t6_ok) {
    if (B >= 16) return true;
    if (B < 2) return false;
    if (!t6_ok || B >= 8) return true;
    if (N <= 8192) return B >= 4;
    return B >= 5 && (double)N * (double)K >= 64e6;
}

// With enough scratch, the tensor-core kernel where it is faster (above).
// Batch 1 below 65536 rows: the nibble-table kernel (one launch of it is the
// shortest for the projection sizes of 8B-27B models: less set-up than the
// cluster kernel); otherwise the 6-bit-table kernel (up to 8 batch rows per
// launch), or the register-MMA engine with the one problem from 12 rows at
// K <= 4096; shapes the 6-bit kernel cannot split (K = 17408): the grouped
// kernel with the one problem, on the register-MMA engine from 3 rows and on
// tables below; what none of them takes: one warp per row (per-call times
// measured on one B300).
int pick_variant(int64_t B, int64_t N, int64_t K, size_t ws_bytes) {
    const bool t6_ok = t6_supported(B, N, K);
    if (tc_supported(B, N, K) && ws_bytes >= tc_min_workspace_bytes(B, N, K) && tc_beats_tables(B, N, K, t6_ok))
        return BIT1_GEMV_TC;
    if (B == 1 && N < 65536 && lut_supported(B, N, K)) return BIT1_GEMV_LUT;
    // Without the tensor cores, the register-MMA engine from 12 rows at
    // K <= 4096 (its work per weight does not grow with the rows; the tables'
    // does), and from 3 rows where the 6-bit tables cannot split K.
    if (t6_ok) return (B >= 12 && K <= 4096 && mma1_supported(B, N, K)) ? BIT1_GEMV_MMA : BIT1_GEMV_LUT6;
    if (B >= 3 && mma1_supported(B, N, K)) return BIT1_GEMV_MMA;
    if (group1_supported(B, N, K)) return BIT1_GEMV_STREAM;
    if (lut_supported(B, N, K)) return BIT1_GEMV_LUT;
    return BIT1_GEMV_SIMPLE;
}

}  // namespace

extern "C" {

bit1_status bit1_pack(const void* w, int w_dtype, int64_t N, int64_t K, uint8_t* bits,
                      uint16_t* scales, uint32_t* d_flags, bit1_stream_t stream) {
    if (!shape_ok(1, N, K)) return BIT1_ESHAPE;
    if (!w || !bits || !scales) return BIT1_EINVAL;
    if (w_dtype != BIT1_F32 && w_dtype != BIT1_BF16 && w_dtype != BIT1_F16) return BIT1_EINVAL;
    if (!aligned16(w) || !aligned16(bits) || !aligned16(scales)) return BIT1_EINVAL;
    if (d_flags && ((uintptr_t)d_flags & 3u)) return BIT1_EINVAL;
    return from_cuda(launch_pack(w, w_dtype, N, K, bits, scales, d_flags, (cudaStream_t)stream));
}

bit1_status bit1_pack_flags_status(uint32_t flags) {
    if (flags & 1u) return BIT1_ENAN;
    if (flags & 14u) return BIT1_ERANGE;
    return BIT1_OK;
}

}  // extern "C"

namespace {

// Everything bit1_gemv_ex checks before launching: the status it would
// return, with `variant` resolved (AUTO -> the pick for this shape).
bit1_status gemv_check(const uint8_t* bits, const uint16_t* scales, const uint16_t* x, int64_t B,
                       int64_t N, int64_t K, const void* y, int y_dtype, const void* workspace,
                       size_t ws_bytes, int* variant, unsigned flags) {
    if (!shape_ok(B, N, K)) return BIT1_ESHAPE;
    if (!bits || !scales || !x || !y) return BIT1_EINVAL;
    if (!aligned16(bits) || !aligned16(scales) || !aligned16(x) || !aligned16(y)) return BIT1_EINVAL;
    if (y_dtype != BIT1_F32 && y_dtype != BIT1_BF16) return BIT1_EINVAL;
    if (ws_bytes > 0 && (!workspace || !aligned16(workspace))) return BIT1_EINVAL;
    if (flags & ~(BIT1_FLAG_PDL | BIT1_FLAG_SWIGLU)) return BIT1_EINVAL;
    if (flags & BIT1_FLAG_SWIGLU) {
        // Gate/up pairs: every kernel but the warp-per-row one pairs rows in
        // its epilogue -- at batch 1 the two table kernels, at 2-8 rows the
        // 6-bit cluster kernel, from 16 rows the tensor cores.
        if (N % 2 != 0) return BIT1_ESHAPE;
        if (*variant == BIT1_GEMV_AUTO) {
            if (B == 1) *variant = lut_supported(B, N, K) ? BIT1_GEMV_LUT : BIT1_GEMV_STREAM;
            else *variant = pick_variant(B, N, K, ws_bytes);
        }
        if (*variant == BIT1_GEMV_SIMPLE) return BIT1_ESHAPE;
    }
    if (*variant == BIT1_GEMV_AUTO) *variant = pick_variant(B, N, K, ws_bytes);
    switch (*variant) {
        case BIT1_GEMV_SIMPLE: return BIT1_OK;
        case BIT1_GEMV_LUT: return lut_supported(B, N, K) ? BIT1_OK : BIT1_ESHAPE;
        case BIT1_GEMV_STREAM: return group1_supported(B, N, K) ? BIT1_OK : BIT1_ESHAPE;
        case BIT1_GEMV_MMA: return mma1_supported(B, N, K) ? BIT1_OK : BIT1_ESHAPE;
        case BIT1_GEMV_TC:
            if (!tc_supported(B, N, K)) return BIT1_ESHAPE;
            return ws_bytes < tc_min_workspace_bytes(B, N, K) ? BIT1_EINVAL : BIT1_OK;
        case BIT1_GEMV_SPLITK:  // the cluster split-K table kernel, named explicitly
        case BIT1_GEMV_LUT6: return t6_supported(B, N, K) ? BIT1_OK : BIT1_ESHAPE;
        default: return BIT1_EINVAL;
    }
}

// Launch a checked call (variant already resolved).
bit1_status gemv_run(const uint8_t* bits, const uint16_t* scales, const uint16_t* x, int64_t B,
                     int64_t N, int64_t K, void* y, int y_dtype, void* workspace, size_t ws_bytes,
                     int variant, unsigned flags, cudaStream_t stream) {
    GemvArgs a;
    a.bits = bits; a.scales = scales; a.x = x;
    a.B = B; a.N = N; a.K = K;
    a.y = y; a.y_bf16 = (y_dtype == BIT1_BF16);
    a.workspace = workspace; a.ws_bytes = ws_bytes;
    a.pdl = (flags & BIT1_FLAG_PDL) != 0;
    a.swiglu = (flags & BIT1_FLAG_SWIGLU) != 0;
    a.stream = stream;
    switch (variant) {
        case BIT1_GEMV_SIMPLE: return from_cuda(launch_gemv_simple(a));
        case BIT1_GEMV_LUT: return from_cuda(launch_gemv_lut(a));
        case BIT1_GEMV_SPLITK:
        case BIT1_GEMV_LUT6: return from_cuda(launch_gemv_t6(a));
        case BIT1_GEMV_STREAM: return from_cuda(launch_gemv_group1(a));
        case BIT1_GEMV_MMA: return from_cuda(launch_gemv_mma1(a));
        case BIT1_GEMV_TC: return from_cuda(launch_gemv_tc(a));
        default: return BIT1_EINVAL;
    }
}

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

// fp32 scratch of one half of a ternary product.
size_t ternary_half_bytes(int64_t B, int64_t N) { return align256((size_t)B * (size_t)N * sizeof(float)); }

}  // namespace

extern "C" {

bit1_status bit1_gemv_ex(const uint8_t* bits, const uint16_t* scales, const uint16_t* x,
                         int64_t B, int64_t N, int64_t K, void* y, int y_dtype, void* workspace,
                         size_t ws_bytes, int variant, unsigned flags, bit1_stream_t stream) {
    bit1_status st = gemv_check(bits, scales, x, B, N, K, y, y_dtype, workspace, ws_bytes, &variant, flags);
    if (st != BIT1_OK) return st;
    return gemv_run(bits, scales, x, B, N, K, y, y_dtype, workspace, ws_bytes, variant, flags,
                    (cudaStream_t)stream);
}

bit1_status bit1_gemv(const uint8_t* bits, const uint16_t* scales, const uint16_t* x, int64_t B,
                      int64_t N, int64_t K, void* y, int y_dtype, void* workspace, size_t ws_bytes,
                      bit1_stream_t stream) {
    return bit1_gemv_ex(bits, scales, x, B, N, K, y, y_dtype, workspace, ws_bytes, BIT1_GEMV_AUTO,
                        0u, stream);
}

size_t bit1_gemv_workspace_bytes(int64_t B, int64_t N, int64_t K) {
    if (!shape_ok(B, N, K)) return 0;
    if (tc_supported(B, N, K) && tc_beats_tables(B, N, K, t6_supported(B, N, K))) return tc_workspace_bytes(B, N, K);
    return 0;
}

int bit1_gemv_pick(int64_t B, int64_t N, int64_t K, size_t ws_bytes) {
    if (!shape_ok(B, N, K)) return 0;
    return pick_variant(B, N, K, ws_bytes);
}

int bit1_gemv_launches(int64_t B, int64_t N, int64_t K, int variant) {
    if (!shape_ok(B, N, K)) return 0;
    if (variant == BIT1_GEMV_AUTO) variant = pick_variant(B, N, K, bit1_gemv_workspace_bytes(B, N, K));
    switch (variant) {
        case BIT1_GEMV_SIMPLE: return 1;
        case BIT1_GEMV_LUT: return lut_supported(B, N, K) ? 1 : 0;
        case BIT1_GEMV_SPLITK:
        case BIT1_GEMV_LUT6: return t6_launch_count(B, N, K);
        case BIT1_GEMV_STREAM: return group1_supported(B, N, K) ? group1_launch_count(B) : 0;
        case BIT1_GEMV_MMA: return mma1_supported(B, N, K) ? mma1_launch_count(B) : 0;
        case BIT1_GEMV_TC: return tc_launch_count(B, N, K);
        default: return 0;
    }
}

bit1_status bit1_xor_patch(uint8_t* bits, int64_t N, int64_t K, const int32_t* rows,
                           int64_t n_rows, bit1_stream_t stream) {
    if (!shape_ok(1, N, K)) return BIT1_ESHAPE;
    if (n_rows < 0) return BIT1_EINVAL;
    if (n_rows == 0) return BIT1_OK;
    if (!bits || !rows || !aligned16(bits)) return BIT1_EINVAL;
    for (int64_t i = 0; i < n_rows; ++i)
        if (rows[i] < 0 || (int64_t)rows[i] >= N) return BIT1_ERANGE;
    return from_cuda(launch_xor_patch(bits, N, K, rows, n_rows, (cudaStream_t)stream));
}

const char* bit1_status_str(bit1_status s) {
    switch (s) {
        case BIT1_OK: return "ok";
        case BIT1_EINVAL: return "invalid argument (null or misaligned pointer, unknown dtype, variant or flag)";
        case BIT1_ESHAPE: return "unsupported shape (B, N >= 1; K a positive multiple of 128; variant limits)";
        case BIT1_ERANGE: return "value out of range (patch row outside [0, N) or packed scale not finite)";
        case BIT1_ECUDA: return "CUDA runtime or launch error";
        case BIT1_ENAN: return "NaN in the weights given to bit1_pack";
        default: return "unknown status";
    }
}

const char* bit1_version(void) { return "bit1 0.2 (sm_103a)"; }

unsigned int bit1_device_wait_timeouts(void) {
    const unsigned int a = t6_take_timeouts(), b = group_take_timeouts(), c = tc_take_timeouts();
    const unsigned int d = tcg_take_timeouts();
    if (a == 0xffffffffu || b == 0xffffffffu || c == 0xffffffffu || d == 0xffffffffu) return 0xffffffffu;
    return a + b + c + d;
}

size_t bit1_group_plan_bytes(int count) { return group_plan_bytes(count); }

bit1_status bit1_group_plan(const bit1_gemv_problem* problems, int count, void* host_plan,
                            size_t plan_bytes) {
    return group_plan(problems, count, 1, BIT1_LAYOUT_CANONICAL, 0, host_plan, plan_bytes);
}

bit1_status bit1_group_plan_batched(const bit1_gemv_problem* problems, int count, int B, void* host_plan,
                                    size_t plan_bytes) {
    return group_plan(problems, count, B, BIT1_LAYOUT_CANONICAL, 0, host_plan, plan_bytes);
}

bit1_status bit1_group_plan_mma(const bit1_gemv_problem* problems, int count, int B, void* host_plan,
                                size_t plan_bytes) {
    return group_plan(problems, count, B, BIT1_LAYOUT_CANONICAL, 1, host_plan, plan_bytes);
}

bit1_status bit1_group_plan_ex(const bit1_gemv_problem* problems, int count, int B, int layout, void* host_plan,
                               size_t plan_bytes) {
    if (layout != BIT1_LAYOUT_CANONICAL && layout != BIT1_LAYOUT_G128X) return BIT1_EINVAL;
    return group_plan(problems, count, B, layout, 0, host_plan, plan_bytes);
}

bit1_status bit1_repack_g128x(const uint8_t* bits, int64_t N, int64_t K, uint8_t* out, bit1_stream_t stream) {
    if (!shape_ok(1, N, K)) return BIT1_ESHAPE;
    if (!bits || !out || !aligned16(bits) || !aligned16(out)) return BIT1_EINVAL;
    return from_cuda(launch_relayout(bits, out, N, K, true, (cudaStream_t)stream));
}

bit1_status bit1_unpack_g128x(const uint8_t* bits, int64_t N, int64_t K, uint8_t* out, bit1_stream_t stream) {
    if (!shape_ok(1, N, K)) return BIT1_ESHAPE;
    if (!bits || !out || !aligned16(bits) || !aligned16(out)) return BIT1_EINVAL;
    return from_cuda(launch_relayout(bits, out, N, K, false, (cudaStream_t)stream));
}

bit1_status bit1_ternary_planes(const int8_t* codes, int64_t N, int64_t K, uint8_t* a, uint8_t* b,
                                uint32_t* d_flags, bit1_stream_t stream) {
    if (!shape_ok(1, N, K)) return BIT1_ESHAPE;
    if (!codes || !a || !b) return BIT1_EINVAL;
    if (!aligned16(codes) || !aligned16(a) || !aligned16(b)) return BIT1_EINVAL;
    if (d_flags && ((uintptr_t)d_flags & 3u)) return BIT1_EINVAL;
    return from_cuda(launch_ternary_planes(codes, N, K, a, b, d_flags, (cudaStream_t)stream));
}

size_t bit1_gemv_ternary_workspace_bytes(int64_t B, int64_t N, int64_t K) {
    if (!shape_ok(B, N, K)) return 0;
    return 2 * ternary_half_bytes(B, N) + bit1_gemv_workspace_bytes(B, N, K);
}

bit1_status bit1_gemv_ternary(const uint8_t* a, const uint8_t* b, const uint16_t* scales,
                              const uint16_t* x, int64_t B, int64_t N, int64_t K, void* y,
                              int y_dtype, void* workspace, size_t ws_bytes, int variant,
                              unsigned flags, bit1_stream_t stream) {
    if (!shape_ok(B, N, K)) return BIT1_ESHAPE;
    if (!a || !b || !aligned16(a) || !aligned16(b)) return BIT1_EINVAL;
    if (!workspace || !aligned16(workspace)) return BIT1_EINVAL;
    // SwiGLU: the two binary halves run plain; the combine forms the pairs.
    const bool swiglu = (flags & BIT1_FLAG_SWIGLU) != 0;
    if (swiglu && N % 2 != 0) return BIT1_ESHAPE;
    flags &= ~BIT1_FLAG_SWIGLU;
    const size_t half = ternary_half_bytes(B, N);
    if (ws_bytes < 2 * half) return BIT1_EINVAL;
    float* ya = reinterpret_cast<float*>(workspace);
    float* yb = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + half);
    void* rest = static_cast<uint8_t*>(workspace) + 2 * half;
    const size_t rest_bytes = ws_bytes - 2 * half;
    if (!y || !aligned16(y) || (y_dtype != BIT1_F32 && y_dtype != BIT1_BF16)) return BIT1_EINVAL;
    // Both halves take the same checks (only the bits pointer differs).
    bit1_status st = gemv_check(a, scales, x, B, N, K, ya, BIT1_F32, rest_bytes ? rest : nullptr,
                                rest_bytes, &variant, flags);
    if (st != BIT1_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    st = gemv_run(a, scales, x, B, N, K, ya, BIT1_F32, rest, rest_bytes, variant, flags, s);
    if (st != BIT1_OK) return st;
    st = gemv_run(b, scales, x, B, N, K, yb, BIT1_F32, rest, rest_bytes, variant, flags, s);
    if (st != BIT1_OK) return st;
    return from_cuda(launch_ternary_combine(ya, yb, B * N, y, y_dtype == BIT1_BF16, s, swiglu));
}

int bit1_gemv_ternary_launches(int64_t B, int64_t N, int64_t K, int variant) {
    if (!shape_ok(B, N, K)) return 0;
    if (variant == BIT1_GEMV_AUTO)
        variant = pick_variant(B, N, K, bit1_gemv_workspace_bytes(B, N, K));
    const int one = bit1_gemv_launches(B, N, K, variant);
    return one ? 2 * one + 1 : 0;
}

bit1_status bit1_ternary_combine(const float* ya, const float* yb, int64_t n, void* y, int y_dtype,
                                 bit1_stream_t stream) {
    if (n < 1) return BIT1_ESHAPE;
    if (!ya || !yb || !y || !aligned16(ya) || !aligned16(yb) || !aligned16(y)) return BIT1_EINVAL;
    if (y_dtype != BIT1_F32 && y_dtype != BIT1_BF16) return BIT1_EINVAL;
    return from_cuda(launch_ternary_combine(ya, yb, n, y, y_dtype == BIT1_BF16, (cudaStream_t)stream));
}

bit1_status bit1_t5_pack(const int8_t* codes, int64_t N, int64_t K, uint8_t* packed, uint32_t* d_flags,
                         bit1_stream_t stream) {
    if (!shape_ok(1, N, K)) return BIT1_ESHAPE;
    if (!codes || !packed || !aligned16(codes) || !aligned16(packed)) return BIT1_EINVAL;
    if (d_flags && ((uintptr_t)d_flags & 3u)) return BIT1_EINVAL;
    return from_cuda(launch_t5_pack(codes, N, K, packed, d_flags, (cudaStream_t)stream));
}

bit1_status bit1_t5_to_planes(const uint8_t* packed, int64_t N, int64_t K, uint8_t* a, uint8_t* b,
                              uint32_t* d_flags, bit1_stream_t stream) {
    if (!shape_ok(1, N, K)) return BIT1_ESHAPE;
    if (!packed || !a || !b || !aligned16(packed) || !aligned16(a) || !aligned16(b)) return BIT1_EINVAL;
    if (d_flags && ((uintptr_t)d_flags & 3u)) return BIT1_EINVAL;
    return from_cuda(launch_t5_planes(packed, N, K, a, b, d_flags, (cudaStream_t)stream));
}

bit1_status bit1_gemv_t5(const uint8_t* packed, const uint16_t* scales, const uint16_t* x, int64_t B,
                         int64_t N, int64_t K, void* y, int y_dtype, bit1_stream_t stream) {
    if (!shape_ok(B, N, K)) return BIT1_ESHAPE;
    if (!packed || !scales || !x || !y) return BIT1_EINVAL;
    if (!aligned16(packed) || !aligned16(scales) || !aligned16(x) || !aligned16(y)) return BIT1_EINVAL;
    if (y_dtype != BIT1_F32 && y_dtype != BIT1_BF16) return BIT1_EINVAL;
    if (t5lut_supported(B, N, K))   // batch 1: table-lookup kernel
        return from_cuda(launch_gemv_t5lut(packed, scales, x, N, K, y, y_dtype == BIT1_BF16, (cudaStream_t)stream));
    return from_cuda(launch_gemv_t5(packed, scales, x, B, N, K, y, y_dtype == BIT1_BF16, (cudaStream_t)stream));
}

int bit1_gemv_t5_launches(int64_t B, int64_t N, int64_t K) {
    if (!shape_ok(B, N, K)) return 0;
    return t5lut_supported(B, N, K) ? 1 : t5_launch_count(B);
}

bit1_status bit1_selftest_wait_timeout(unsigned int* d_done, bit1_stream_t stream) {
    if (!d_done || ((uintptr_t)d_done & 3u)) return BIT1_EINVAL;
    return from_cuda(launch_wait_selftest(d_done, (cudaStream_t)stream));
}

bit1_status bit1_gemv_group(const void* device_plan, const void* host_plan, unsigned flags,
                            bit1_stream_t stream) {
    if (!device_plan || !host_plan || ((uintptr_t)device_plan & 127) || ((uintptr_t)host_plan & 127))
        return BIT1_EINVAL;
    if (flags & ~BIT1_FLAG_PDL) return BIT1_EINVAL;
    int kind;
    std::memcpy(&kind, static_cast<const uint8_t*>(host_plan) + kPlanKindOffset, sizeof(kind));
    const bool pdl = (flags & BIT1_FLAG_PDL) != 0;
    if (kind == kPlanKindTensor) return from_cuda(launch_tc_group(device_plan, host_plan, pdl, (cudaStream_t)stream));
    if (kind != kPlanKindTables) return BIT1_EINVAL;
    return from_cuda(launch_group(device_plan, host_plan, pdl, (cudaStream_t)stream));
}

size_t bit1_group_tc_plan_bytes(int count) { return tcg_plan_bytes(count); }

size_t bit1_group_tc_workspace_bytes(const bit1_gemv_problem* problems, int count, int B) {
    return tcg_workspace_bytes(problems, count, B);
}

bit1_status bit1_group_plan_tc(const bit1_gemv_problem* problems, int count, int B, void* workspace,
                               size_t ws_bytes, void* host_plan, size_t plan_bytes) {
    return tcg_plan(problems, count, B, workspace, ws_bytes, host_plan, plan_bytes);
}

}  // extern "C"
