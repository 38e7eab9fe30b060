// noalloc.cu -- gemm_bf16_tn_noalloc: BF16 TN GEMM with split-K whose scratch
// lives in a fixed array inside the library, so the call allocates nothing.
//
// Who needs this: programs that may not call cudaMalloc themselves -- code
// whose device memory is owned by a caching or pooled allocator it must not
// bypass, plugins whose host application forbids device allocation, and
// latency-critical loops where cudaMalloc/cudaFree would synchronise the
// device or fail unpredictably under memory pressure.  They can still use
// split-K for shapes whose output tiles cannot fill the GPU, without
// registering a workspace (gemm_set_workspace).
//
// The scratch is g_noalloc_scratch, kNoAllocScratchBytes long, in the device
// memory of every GPU that loads the library, for as long as the library is
// loaded.  Host code cannot use the array's name as a device address: the
// address is looked up with cudaGetSymbolAddress once per device, on the first
// call made with that device current, and cached.  All calls share the array
// and it keeps the last call's contents.  Its first kSplitCounterBytes hold the
// two split-counter sets (zero when the library loads; each split launch
// zeroes the set the next one uses, and resets the counters it counted in),
// the rest the partial sums, which every split launch overwrites.  Calls
// whose execution overlaps on the GPU (different streams, or different host
// threads on one device) race on the array.
#include <mutex>

#include "launch.h"
#include "gemm.h"

namespace {

constexpr int64_t kNoAllocScratchBytes = 24LL << 20;  // 24 MiB
static_assert(kNoAllocScratchBytes == GEMM_NOALLOC_SCRATCH_BYTES, "header constant");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};
std::atomic<unsigned int> g_parity[kMaxDevices];  // the next split launch's counter set

// Device address of this device's copy of the array, looked up on first use,
// and the device's index.
int scratch_address(void** out, int* dev_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return gb300::tn_record_cuda_error(e);
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return gb300::tn_record_cuda_error(e);
        if (!p) return gb300::tn_record_cuda_error(cudaErrorInvalidSymbol);
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    *dev_out = dev;
    return GEMM_OK;
}

}  // namespace

extern "C" int gemm_bf16_tn_noalloc(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                                    const void* B, int64_t ldb, void* C, int64_t ldc,
                                    int64_t splits, void* stream) {
    if (splits < 0 || splits > 64) return GEMM_ERR_INVALID_OPTION;
    // every argument check before the first CUDA call, as for the other entry points
    int st = gb300::tn_validate(gb300::InKind::BF16, M, N, K, A, lda, B, ldb, C, ldc);
    if (st != GEMM_OK) return st;
    void* scratch = nullptr;
    int dev = 0;
    st = scratch_address(&scratch, &dev);
    if (st != GEMM_OK) return st;
    gb300::ScratchOverride ov{static_cast<char*>(scratch) + gb300::kSplitCounterBytes,
                              kNoAllocScratchBytes - gb300::kSplitCounterBytes,
                              static_cast<int>(splits)};
    ov.counters = scratch;
    ov.parity = &g_parity[dev];
    return gb300::gemm_tn_with_scratch(gb300::InKind::BF16, M, N, K, A, lda, B, ldb, C, ldc,
                                       stream, ov);
}
