// misc_kernels.cu -- a CUDA-core TN kernel, the row repack used for operands
// whose rows are not 16-byte aligned, the K == 0 zero fill and the watchdog
// self-test.
//
// The CUDA-core TN kernel is a second, independent GPU implementation of the
// TN entry points, selected only by gemm_set_option("path", 1) (tests compare
// it with the tensor-core kernel and the oracle).  It reads elements one by
// one, so any alignment works, decodes them to FP32 in shared memory,
// accumulates in FP32 and rounds the result once to the output type, as the
// tensor-core kernel does; only the summation order differs.  Like the pages'
// buffer-descriptor loads ("FP16 GEMM Optimization on AMD RDNA 3 and RDNA 4",
// "Step 4: Buffer Resource Descriptors for Global Loads"), out-of-range
// elements read as zero.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "launch.h"
#include "ptx.cuh"
#include "tc_gemm.cuh"

namespace gb300 {
namespace {

constexpr int kFbBM = 64, kFbBN = 64, kFbBK = 32, kFbThreads = 256;

template <InKind IN>
__device__ __forceinline__ float decode_in(const uint8_t* base, int64_t idx) {
    if constexpr (IN == InKind::F16) {
        return __half2float(reinterpret_cast<const __half*>(base)[idx]);
    } else if constexpr (IN == InKind::BF16) {
        return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx]);
    } else {
        __nv_fp8_e4m3 q;
        q.__x = base[idx];
        return static_cast<float>(q);
    }
}

template <InKind IN, typename OutT>
__global__ void __launch_bounds__(kFbThreads)
    tn_fallback_kernel(int M, int N, int K, const uint8_t* __restrict__ A, int64_t lda,
                       const uint8_t* __restrict__ B, int64_t ldb, float scale,
                       OutT* __restrict__ C, int64_t ldc, int64_t tiles_m, int64_t tiles_n) {
    __shared__ float As[kFbBK][kFbBM + 1];
    __shared__ float Bs[kFbBK][kFbBN + 1];
    int64_t tm, tn;
    raster_tile(blockIdx.x, tiles_m, tiles_n, 8, &tm, &tn);
    const int64_t m0 = tm * kFbBM, n0 = tn * kFbBN;
    const int tid = threadIdx.x;
    const int tmi = tid & 15, tni = tid >> 4;
    float acc[4][4] = {};
    for (int64_t k0 = 0; k0 < K; k0 += kFbBK) {  // 64-bit: K may be 2^31 - 1
#pragma unroll
        for (int r = 0; r < (kFbBM * kFbBK) / kFbThreads; ++r) {
            const int e = tid + r * kFbThreads;
            const int row = e / kFbBK, kk = e % kFbBK;
            const int64_t m = m0 + row, n = n0 + row;
            const int64_t k = k0 + kk;
            As[kk][row] = (m < M && k < K) ? decode_in<IN>(A, m * lda + k) : 0.f;
            Bs[kk][row] = (n < N && k < K) ? decode_in<IN>(B, n * ldb + k) : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < kFbBK; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[kk][tmi + 16 * i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tni + 16 * j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int64_t n = n0 + tni + 16 * j;
        if (n >= N) continue;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t m = m0 + tmi + 16 * i;
            if (m >= M) continue;
            float v = acc[i][j];
            if constexpr (IN == InKind::E4M3) v *= scale;
            if constexpr (sizeof(OutT) == 4)
                C[n * ldc + m] = v;
            else if constexpr (IN == InKind::F16)
                C[n * ldc + m] = __float2half_rn(v);
            else
                C[n * ldc + m] = __float2bfloat16_rn(v);
        }
    }
}

// Copies `rows` rows of `row_bytes` bytes from src (row pitch sp, any
// alignment) to dst (row pitch dp; dst and dp 16-byte aligned, dp >= row_bytes
// rounded up to 16).  One warp per 512-byte segment of a row: lane l writes the
// 16-byte chunk at offset 16 l of the segment from the one or two aligned
// source chunks that cover it (all lanes of a row share the misalignment).
// Only aligned source chunks holding a byte of the row are read; bytes past the
// row's end in the last chunk are zeroed.
__global__ void repack_rows_kernel(const uint8_t* __restrict__ src, int64_t sp,
                                   uint8_t* __restrict__ dst, int64_t dp, int64_t rows,
                                   int64_t row_bytes) {
    const int64_t segs = (row_bytes + 511) / 512;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
    const int lane = threadIdx.x & 31;
    for (int64_t w = blockIdx.x * static_cast<int64_t>(blockDim.x / 32) + threadIdx.x / 32;
         w < rows * segs; w += warps) {
        const int64_t row = w / segs, seg = w % segs;
        const int64_t o = seg * 512 + 16 * lane;
        if (o >= row_bytes) continue;
        const uintptr_t a = reinterpret_cast<uintptr_t>(src + row * sp + o);
        const uint32_t delta = static_cast<uint32_t>(a & 15u);
        const uintptr_t al = a - delta;
        const int64_t valid = row_bytes - o;  // >= 1
        const uint4 lo = ldg_nc_v4(reinterpret_cast<const void*>(al));
        uint4 hi = make_uint4(0u, 0u, 0u, 0u);
        if (delta != 0 && 16 - static_cast<int64_t>(delta) < valid)
            hi = ldg_nc_v4(reinterpret_cast<const void*>(al + 16u));
        uint4 out = shift_chunk(lo, hi, delta);
        if (valid < 16) out = mask_chunk(out, static_cast<int32_t>(valid));
        *reinterpret_cast<uint4*>(dst + row * dp + o) = out;
    }
}

__global__ void zero_fill_kernel(uint8_t* C, int64_t rows, int64_t cols, int64_t ld,
                                 int elem_bytes) {
    const int64_t total = rows * cols;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / cols, c = i % cols;
        uint8_t* p = C + (r * ld + c) * elem_bytes;
        if (elem_bytes == 4)
            *reinterpret_cast<uint32_t*>(p) = 0u;
        else
            *reinterpret_cast<uint16_t*>(p) = 0u;
    }
}

// One warp waits on a barrier that nothing will complete, with the library's
// bounded wait; when the limit runs out the watchdog word records it and the
// kernel returns normally.
__global__ void watchdog_selftest_kernel(uint64_t limit_ns, unsigned int* watchdog) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const Watch w{&abort_flag, watchdog, limit_ns};
    warp_wait(smem_u32(&bar), 0, w);
}

}  // namespace

cudaError_t tn_fallback_launch(InKind in, bool out_f32, int64_t M, int64_t N, int64_t K,
                               const void* A, int64_t lda, const void* B, int64_t ldb, float scale,
                               void* C, int64_t ldc, cudaStream_t stream) {
    const int64_t tiles_m = (M + kFbBM - 1) / kFbBM, tiles_n = (N + kFbBN - 1) / kFbBN;
    if (tiles_m * tiles_n > 0x7fffffff) return cudaErrorInvalidValue;
    const dim3 grid(static_cast<unsigned>(tiles_m * tiles_n));
    const auto* a = static_cast<const uint8_t*>(A);
    const auto* b = static_cast<const uint8_t*>(B);
    switch (in) {
        case InKind::F16:
            tn_fallback_kernel<InKind::F16, __half><<<grid, kFbThreads, 0, stream>>>(
                int(M), int(N), int(K), a, lda, b, ldb, scale, static_cast<__half*>(C), ldc,
                tiles_m, tiles_n);
            break;
        case InKind::BF16:
            if (out_f32)
                tn_fallback_kernel<InKind::BF16, float><<<grid, kFbThreads, 0, stream>>>(
                    int(M), int(N), int(K), a, lda, b, ldb, scale, static_cast<float*>(C), ldc,
                    tiles_m, tiles_n);
            else
                tn_fallback_kernel<InKind::BF16, __nv_bfloat16><<<grid, kFbThreads, 0, stream>>>(
                    int(M), int(N), int(K), a, lda, b, ldb, scale,
                    static_cast<__nv_bfloat16*>(C), ldc, tiles_m, tiles_n);
            break;
        case InKind::E4M3:
            if (out_f32)
                tn_fallback_kernel<InKind::E4M3, float><<<grid, kFbThreads, 0, stream>>>(
                    int(M), int(N), int(K), a, lda, b, ldb, scale, static_cast<float*>(C), ldc,
                    tiles_m, tiles_n);
            else
                tn_fallback_kernel<InKind::E4M3, __nv_bfloat16><<<grid, kFbThreads, 0, stream>>>(
                    int(M), int(N), int(K), a, lda, b, ldb, scale, static_cast<__nv_bfloat16*>(C),
                    ldc, tiles_m, tiles_n);
            break;
    }
    return cudaGetLastError();
}

cudaError_t repack_rows_launch(const void* src, int64_t sp, void* dst, int64_t dp, int64_t rows,
                               int64_t row_bytes, cudaStream_t stream) {
    if (rows <= 0 || row_bytes <= 0) return cudaSuccess;
    const int64_t work = rows * ((row_bytes + 511) / 512);
    int64_t blocks = (work + 7) / 8;  // 8 warps a block
    if (blocks > 152 * 16) blocks = 152 * 16;
    repack_rows_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<const uint8_t*>(src), sp, static_cast<uint8_t*>(dst), dp, rows, row_bytes);
    return cudaGetLastError();
}

cudaError_t zero_fill_launch(void* C, int64_t rows, int64_t cols, int64_t ld, int elem_bytes,
                             cudaStream_t stream) {
    const int64_t total = rows * cols;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    if (blocks < 1) blocks = 1;
    zero_fill_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<uint8_t*>(C), rows, cols, ld, elem_bytes);
    return cudaGetLastError();
}

cudaError_t watchdog_selftest_launch(uint64_t limit_ns, unsigned int* watchdog,
                                     cudaStream_t stream) {
    watchdog_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns, watchdog);
    return cudaGetLastError();
}

}  // namespace gb300
