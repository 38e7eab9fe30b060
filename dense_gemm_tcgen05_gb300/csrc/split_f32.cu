// split_f32.cu -- operand preparation for the tensor-core FP32 GEMM
// (gemm_f32_bf16x6).
//
// Every FP32 value x is cut into three BF16 pieces whose sum is x exactly:
//   x0 = bf16_rn(x),  x1 = bf16_rn(x - x0),  x2 = bf16_rn(x - x0 - x1).
// Each subtraction is exact (it is the rounding error of a rounding to fewer
// bits with the same exponent range), x0 and x1 carry 8 significant bits each
// and what is left after them has at most 8, so x2 takes it whole.  The
// exactness holds for finite x whose pieces stay normal in BF16 (|x| between
// about 2^-100 and 2^127); non-finite x gives NaN pieces.
//
// A BF16 x BF16 product has at most 16 significant bits, so the tensor cores
// form a_i b_j exactly and add it into their FP32 accumulator.  Of the nine
// piece products the six largest are kept; the three left out (a1 b2, a2 b1,
// a2 b2) sum to at most about 2^-25 |a b|, below FP32's own rounding of a
// product.  Each operand is written as six K-segments of Kp columns (K
// rounded up to a multiple of 64, zero-filled), ordered so that one BF16 GEMM
// over 6 Kp columns adds the products from the smallest to the largest:
//   segment   0     1     2     3     4     5
//   A piece   a2    a1    a0    a1    a0    a0
//   B piece   b0    b1    b2    b0    b1    b0
// A (row-major M x K) keeps its row layout; B (row-major K x N) is transposed
// on the way, so that both come out K-contiguous with rows of 6 Kp BF16
// values, as the TN tensor-core kernel reads them.
#include <cuda_bf16.h>

#include <cstdint>

#include "launch.h"

namespace gb300 {
namespace {

constexpr int kSegs = 6;
// Which piece of A and of B segment s holds (the table above).
__device__ __forceinline__ constexpr int piece_a(int s) {
    return s == 0 ? 2 : (s == 1 || s == 3) ? 1 : 0;
}
__device__ __forceinline__ constexpr int piece_b(int s) {
    return s == 2 ? 2 : (s == 1 || s == 4) ? 1 : 0;
}

// The three pieces of eight values, packed as three rows of eight BF16.
struct Pieces8 {
    uint4 p[3];
};

__device__ __forceinline__ Pieces8 split8(const float (&v)[8]) {
    uint32_t w[3][4];
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
        uint16_t lo[3], hi[3];
        float x = v[j], y = v[j + 1];
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            const __nv_bfloat16 qx = __float2bfloat16_rn(x);
            const __nv_bfloat16 qy = __float2bfloat16_rn(y);
            lo[i] = __bfloat16_as_ushort(qx);
            hi[i] = __bfloat16_as_ushort(qy);
            x -= __bfloat162float(qx);  // exact: the error of the rounding above
            y -= __bfloat162float(qy);
        }
#pragma unroll
        for (int i = 0; i < 3; ++i)
            w[i][j / 2] = static_cast<uint32_t>(lo[i]) | (static_cast<uint32_t>(hi[i]) << 16);
    }
    Pieces8 r;
#pragma unroll
    for (int i = 0; i < 3; ++i) r.p[i] = make_uint4(w[i][0], w[i][1], w[i][2], w[i][3]);
    return r;
}

// out[r * 6 Kp + s * Kp + k] = piece piece_a(s) of X[r * ldx + k] (0 for
// k >= K); one thread per eight consecutive k of a row.
__global__ void __launch_bounds__(256)
    split_rows_kernel(const float* __restrict__ X, int64_t ldx, int64_t rows, int64_t K,
                      int64_t Kp, __nv_bfloat16* __restrict__ out, int vec) {
    const int64_t per_row = Kp / 8;
    const int64_t total = rows * per_row;
    const int64_t ldo = kSegs * Kp;
    for (int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; c < total;
         c += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = c / per_row;
        const int64_t k0 = (c - r * per_row) * 8;
        float v[8];
        if (vec && k0 + 8 <= K) {
            const float4* src = reinterpret_cast<const float4*>(X + r * ldx + k0);
            const float4 lo = __ldg(src), hi = __ldg(src + 1);
            v[0] = lo.x; v[1] = lo.y; v[2] = lo.z; v[3] = lo.w;
            v[4] = hi.x; v[5] = hi.y; v[6] = hi.z; v[7] = hi.w;
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = k0 + j < K ? __ldg(X + r * ldx + k0 + j) : 0.f;
        }
        const Pieces8 q = split8(v);
        __nv_bfloat16* dst = out + r * ldo + k0;
#pragma unroll
        for (int s = 0; s < kSegs; ++s)
            *reinterpret_cast<uint4*>(dst + s * Kp) = q.p[piece_a(s)];
    }
}

// out[n * 6 Kp + s * Kp + k] = piece piece_b(s) of X[k * ldx + n] (0 for
// k >= K): a 64 (k) x 32 (n) tile is read along n, transposed through shared
// memory and written along k, eight k per thread.
constexpr int kTK = 64, kTN = 32;

__global__ void __launch_bounds__(256)
    split_cols_kernel(const float* __restrict__ X, int64_t ldx, int64_t K, int64_t N, int64_t Kp,
                      __nv_bfloat16* __restrict__ out) {
    __shared__ float tile[kTK][kTN + 1];
    const int64_t tiles_k = Kp / kTK;
    const int64_t tiles = tiles_k * ((N + kTN - 1) / kTN);
    const int64_t ldo = kSegs * Kp;
    const int lx = threadIdx.x & 31, ly = threadIdx.x >> 5;
    const int nn = threadIdx.x >> 3, kc = (threadIdx.x & 7) * 8;
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int64_t tn = t / tiles_k;
        const int64_t k0 = (t - tn * tiles_k) * kTK, n0 = tn * kTN;
        const int64_t n = n0 + lx;
#pragma unroll
        for (int j = 0; j < kTK / 8; ++j) {
            const int64_t k = k0 + ly + 8 * j;
            tile[ly + 8 * j][lx] = (k < K && n < N) ? __ldg(X + k * ldx + n) : 0.f;
        }
        __syncthreads();
        const int64_t on = n0 + nn;
        if (on < N) {
            float v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = tile[kc + j][nn];
            const Pieces8 q = split8(v);
            __nv_bfloat16* dst = out + on * ldo + k0 + kc;
#pragma unroll
            for (int s = 0; s < kSegs; ++s)
                *reinterpret_cast<uint4*>(dst + s * Kp) = q.p[piece_b(s)];
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t f32_split_rows_launch(const float* X, int64_t ldx, int64_t rows, int64_t K,
                                  int64_t Kp, void* out, int sms, cudaStream_t stream) {
    if (rows <= 0 || Kp <= 0) return cudaSuccess;
    const int64_t work = rows * (Kp / 8);
    int64_t blocks = (work + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 1) * 16;
    if (blocks > cap) blocks = cap;
    const int vec = (reinterpret_cast<uintptr_t>(X) % 16 == 0 && ldx % 4 == 0) ? 1 : 0;
    split_rows_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        X, ldx, rows, K, Kp, static_cast<__nv_bfloat16*>(out), vec);
    return cudaGetLastError();
}

cudaError_t f32_split_cols_launch(const float* X, int64_t ldx, int64_t K, int64_t N, int64_t Kp,
                                  void* out, int sms, cudaStream_t stream) {
    if (N <= 0 || Kp <= 0) return cudaSuccess;
    const int64_t tiles = (Kp / kTK) * ((N + kTN - 1) / kTN);
    int64_t blocks = tiles;
    const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 1) * 8;
    if (blocks > cap) blocks = cap;
    split_cols_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        X, ldx, K, N, Kp, static_cast<__nv_bfloat16*>(out));
    return cudaGetLastError();
}

}  // namespace gb300
