// launch.h -- host-side launchers of the library's other kernels and the
// internal TN entry with caller-supplied scratch.
#pragma once

#include <atomic>

#include "common.h"

namespace gb300 {

// CUDA-core fallback for TN operands that TMA cannot address.
cudaError_t tn_fallback_launch(InKind in, bool out_f32, int64_t M, int64_t N, int64_t K,
                               const void* A, int64_t lda, const void* B, int64_t ldb, float scale,
                               void* C, int64_t ldc, cudaStream_t stream);

// Split-K counters live in two fixed sets of kCounterSetWords words at the
// start of each scratch area (the registered workspace, the no-allocation
// array), kSplitCounterBytes in all, zeroed when the area is set up.  Split
// launches alternate between the sets: each counts in one and zeroes the other
// for the next, and the last piece of every slice resets its own counter, so
// no launch needs a host-side memset in front of it.
constexpr int64_t kCounterSetWords = 16384;
constexpr int64_t kSplitCounterBytes = 2 * kCounterSetWords * 4;

// Scratch supplied by the caller of the internal TN path instead of the
// registered workspace (see gemm_tn_with_scratch).
struct ScratchOverride {
    void* ptr;       // device address, 256-byte aligned
    int64_t bytes;   // usable bytes at ptr
    int splits;      // 0 automatic, 1 never split, >= 2 that many K pieces
    int strict = 1;  // 1: a chosen split that does not fit fails with GEMM_ERR_SCRATCH;
                     // 0: the call runs unsplit instead
    void* counters = nullptr;                  // the two counter sets, or nullptr
    std::atomic<unsigned int>* parity = nullptr;  // which set the next split launch uses
};

// The argument checks of a TN call with 16-bit output (dimensions, leading
// dimensions, null pointers, alignment), without touching the device: a
// gemm.h status.
int tn_validate(InKind in, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                const void* B, int64_t ldb, const void* C, int64_t ldc);

// Records a CUDA error for gemm_status_string and returns GEMM_ERR_LAUNCH.
int tn_record_cuda_error(cudaError_t e);

// The TN path with explicit split-K scratch (16-bit inputs and output).
int gemm_tn_with_scratch(InKind in, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                         const void* B, int64_t ldb, void* C, int64_t ldc, void* stream,
                         const ScratchOverride& ov);

// Operand preparation of the tensor-core FP32 path (split_f32.cu): three-way
// BF16 splits of FP32 values in six K-segments of Kp columns (Kp a multiple of
// 64), rows of 6 Kp BF16 values at `out` (256-byte aligned).  Rows: X is
// rows x K row-major; cols: X is K x N row-major and comes out transposed.
cudaError_t f32_split_rows_launch(const float* X, int64_t ldx, int64_t rows, int64_t K,
                                  int64_t Kp, void* out, int sms, cudaStream_t stream);
cudaError_t f32_split_cols_launch(const float* X, int64_t ldx, int64_t K, int64_t N, int64_t Kp,
                                  void* out, int sms, cudaStream_t stream);

// tail_mode 0: a last wave of whole tiles that is at most half full runs as
// half-width tiles in a second grid launched with programmatic dependent launch;
// 1: whole tiles only; 2: as 0 but two plain launches; 3: halves for any last
// partial wave.
// ktail > 0: the last ktail terms of K (when K > ktail) run in the chain-
// continuing kernel that takes the terms past 2^31 - 16 (tests of that path).
cudaError_t f32_launch(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                       const float* B, int64_t ldb, float* C, int64_t ldc, cudaStream_t stream,
                       int tail_mode, int ktail = 0);

// Copies rows of row_bytes bytes from any alignment into 16-byte-aligned rows
// of pitch dp (a multiple of 16) so that TMA can address them.
cudaError_t repack_rows_launch(const void* src, int64_t sp, void* dst, int64_t dp, int64_t rows,
                               int64_t row_bytes, cudaStream_t stream);

// Writes zeros into a rows x cols block with leading dimension ld (elements of
// elem_bytes bytes); used for K == 0.
cudaError_t zero_fill_launch(void* C, int64_t rows, int64_t cols, int64_t ld, int elem_bytes,
                             cudaStream_t stream);

cudaError_t watchdog_selftest_launch(uint64_t limit_ns, unsigned int* watchdog,
                                     cudaStream_t stream);

}  // namespace gb300
