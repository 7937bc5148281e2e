// Host-side launchers of the bit1 kernels (called by the C ABI in bit1_api.cu
// after argument validation; they only configure and launch).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "bit1.h"

namespace bit1 {

struct GemvArgs {
    const uint8_t* bits;
    const uint16_t* scales;
    const uint16_t* x;
    int64_t B, N, K;
    void* y;
    int y_bf16;          // 1: bf16 output, 0: fp32 output
    void* workspace;
    size_t ws_bytes;
    bool pdl;            // launch with programmatic stream serialization
    cudaStream_t stream;
    bool swiglu = false; // rows are (gate, up) pairs; y is h = silu(gate) * up, [B][N/2]
};

// Raise a kernel's dynamic shared-memory limit to smem_bytes (and allow
// non-portable cluster sizes when asked) on the current device.  Function
// attributes are per device, so this runs once per (device, kernel); a
// failure is returned and retried on the next call.
cudaError_t func_attrs(const void* fn, int smem_bytes, bool nonportable_clusters);

// Launch helper: grid/block/smem with optional PDL attribute.
cudaError_t launch(const void* func, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                   bool pdl, void** args);

cudaError_t launch_pack(const void* w, int dtype, int64_t N, int64_t K, uint8_t* bits,
                        uint16_t* scales, uint32_t* flags, cudaStream_t stream);

// Sign bits between the canonical and the g128x layout (layout.cu); in == out allowed.
cudaError_t launch_relayout(const uint8_t* in, uint8_t* out, int64_t N, int64_t K, bool to_g128x,
                            cudaStream_t stream);

cudaError_t launch_xor_patch(uint8_t* bits, int64_t N, int64_t K, const int32_t* rows,
                             int64_t n_rows, cudaStream_t stream);

cudaError_t launch_gemv_simple(const GemvArgs& a);

// Table-lookup batch-1..8 kernel. Returns cudaErrorNotSupported if the shape
// is outside its limits (checked by lut_supported first).
bool lut_supported(int64_t B, int64_t N, int64_t K);
cudaError_t launch_gemv_lut(const GemvArgs& a);

// Row-per-lane 6-bit-table kernel with TMA staging and cluster split-K
// (needs K a multiple of 1024 with a usable cluster split); up to 8 batch
// rows per launch, larger batches in several launches (t6_launch_count).
bool t6_supported(int64_t B, int64_t N, int64_t K);
int t6_launch_count(int64_t B, int64_t N, int64_t K);
cudaError_t launch_gemv_t6(const GemvArgs& a);
// Number of bounded device waits that gave up since the last call (and reset).
unsigned int t6_take_timeouts();
// One kernel whose bounded wait runs out on purpose (sets *d_done = 1 on exit).
cudaError_t launch_wait_selftest(unsigned int* d_done, cudaStream_t stream);

// Grouped plans: the int at byte kPlanKindOffset of a plan's 128-byte
// header says which grouped kernel it is for.
constexpr int kPlanKindOffset = 68;
constexpr int kPlanKindTables = 0;        // gemv_group.cu (CUDA cores, B <= 6)
constexpr int kPlanKindTensor = 1;        // gemv_tc_group.cu (tensor cores, B <= 64)

// Grouped persistent kernel (gemv_group.cu).
size_t group_plan_bytes(int count);
// engine: 0 = 6-bit tables (1 <= nb <= 6, either layout), 1 = register-sourced
// MMAs (1 <= nb <= 16, canonical layout).
bit1_status group_plan(const bit1_gemv_problem* problems, int count, int nb, int layout, int engine,
                       void* host_plan, size_t bytes);
cudaError_t launch_group(const void* device_plan, const void* host_plan, bool pdl, cudaStream_t stream);
bool group1_supported(int64_t B, int64_t N, int64_t K);
int group1_launch_count(int64_t B);          // ceil(B / 6): up to 6 rows per launch
cudaError_t launch_gemv_group1(const GemvArgs& a);
// One problem on the grouped kernel's register-sourced MMA engine (up to 16
// rows per launch, ceil(B / 16) launches).
bool mma1_supported(int64_t B, int64_t N, int64_t K);
int mma1_launch_count(int64_t B);
cudaError_t launch_gemv_mma1(const GemvArgs& a);
unsigned int group_take_timeouts();

// tcgen05 tensor-core batched kernel (gemv_tc.cu): K a multiple of 1024;
// needs tc_workspace_bytes() of scratch; tc_launch_count() launches per call.
bool tc_supported(int64_t B, int64_t N, int64_t K);
size_t tc_workspace_bytes(int64_t B, int64_t N, int64_t K);      // all batch chunks at once (fastest)
size_t tc_min_workspace_bytes(int64_t B, int64_t N, int64_t K);  // one 64-row chunk at a time
int tc_launch_count(int64_t B, int64_t N, int64_t K);
cudaError_t launch_gemv_tc(const GemvArgs& a);
unsigned int tc_take_timeouts();

// Grouped persistent tensor-core kernel (gemv_tc_group.cu): B <= 64 rows per
// problem, a caller-owned workspace for the activations' fp16 copies.
size_t tcg_plan_bytes(int count);
size_t tcg_workspace_bytes(const bit1_gemv_problem* problems, int count, int B);
bit1_status tcg_plan(const bit1_gemv_problem* problems, int count, int B, void* workspace, size_t ws_bytes,
                     void* host_plan, size_t bytes);
cudaError_t launch_tc_group(const void* device_plan, const void* host_plan, bool pdl, cudaStream_t stream);
unsigned int tcg_take_timeouts();

// Ternary weights in 2-bit slots (ternary.cu).
cudaError_t launch_ternary_planes(const int8_t* codes, int64_t N, int64_t K, uint8_t* a, uint8_t* b,
                                  uint32_t* flags, cudaStream_t stream);
cudaError_t launch_ternary_combine(const float* ya, const float* yb, int64_t n, void* y, bool y_bf16,
                                   cudaStream_t stream,
                                   bool swiglu = false);

// Ternary codes packed five per byte (t5.cu).
cudaError_t launch_t5_pack(const int8_t* codes, int64_t N, int64_t K, uint8_t* out, uint32_t* flags,
                           cudaStream_t stream);
cudaError_t launch_t5_planes(const uint8_t* packed, int64_t N, int64_t K, uint8_t* a, uint8_t* b,
                             uint32_t* flags, cudaStream_t stream);
cudaError_t launch_gemv_t5(const uint8_t* packed, const uint16_t* scales, const uint16_t* x, int64_t B,
                           int64_t N, int64_t K, void* y, bool y_bf16, cudaStream_t stream);
int t5_launch_count(int64_t B);
// Batch-1 table-lookup product on the five-per-byte packing (t5lut.cu).
bool t5lut_supported(int64_t B, int64_t N, int64_t K);
cudaError_t launch_gemv_t5lut(const uint8_t* packed, const uint16_t* scales, const uint16_t* x, int64_t N,
                              int64_t K, void* y, bool y_bf16, cudaStream_t stream);

int sm_count();

}  // namespace bit1
