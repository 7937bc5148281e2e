// Allocation-free entry point of the tensor-core batched product: the same
// launcher as bit1_gemv_ex(..., BIT1_GEMV_TC, ...), with its workspace taken
// from a file-scope device array instead of the caller.  Contract (sizes,
// races, setup before stream capture): bit1.h.
#include <mutex>

#include "internal.h"

namespace bit1 {
namespace {

constexpr size_t kNoAllocScratchBytes = BIT1_NOALLOC_SCRATCH_BYTES;
constexpr int kNoAllocMaxDevices = 64;

// Activation staging of one tensor-core launch (at most 64 batch rows x K
// fp16 inputs plus 256 bytes of prescale factors), shared by all calls on a
// device.
__device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// The scratch's device address, per device: set once obtained; a failed
// lookup is not remembered, so a later call on that device tries again.
std::mutex g_scratch_mu;
void* g_scratch_ptr[kNoAllocMaxDevices] = {};

}  // namespace
}  // namespace bit1

using namespace bit1;

extern "C" bit1_status bit1_gemv_tc_noalloc(const uint8_t* bits, const uint16_t* scales, const uint16_t* x,
                                            int64_t B, int64_t N, int64_t K, void* y, int y_dtype, unsigned flags,
                                            bit1_stream_t stream) {
    if (B < 1 || N < 1 || K < 128 || K % 128 != 0 || B > 0x7fffffffLL || N > 0x7fffffffLL || K > (1LL << 24))
        return BIT1_ESHAPE;
    if (!tc_supported(B, N, K)) return BIT1_ESHAPE;
    const size_t need = tc_min_workspace_bytes(B, N, K);
    if (need == 0 || need > kNoAllocScratchBytes) return BIT1_ESHAPE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return BIT1_ECUDA;
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_scratch_mu);
        if (!g_scratch_ptr[dev]) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
                (void)cudaGetLastError();     // leave no pending error behind
                return BIT1_ECUDA;
            }
            g_scratch_ptr[dev] = p;
        }
        scratch = g_scratch_ptr[dev];
    }
    return bit1_gemv_ex(bits, scales, x, B, N, K, y, y_dtype, scratch, kNoAllocScratchBytes, BIT1_GEMV_TC, flags,
                        stream);
}
