// simt_f32.cu -- FP32 GEMM on the CUDA cores (FFMA), all matrices row-major.
//
// C[m*ldc + n] = sum_k A[m*lda + k] * B[k*ldb + n], one FP32 fused
// multiply-add per (m, n, k) in increasing k.
//
// Design, following "Optimizing GEMM in HIP" Steps 2-6 (shared-memory tiling,
// register tiling, double buffering, vectorised loads, register budget), made
// for a Blackwell SM:
//   - a 128 x 128 block tile, K slices of 16, 256 threads, 8 x 8 outputs per
//     thread held in registers (outer-product FFMAs, 64 per k per thread);
//   - each thread's 8 x 8 outputs are two 4-row by two 4-column groups 64 apart,
//     so its shared-memory operand reads are float4 and conflict-free;
//   - A is stored k-major in shared memory (transposed on the way in, rows
//     padded by 4 floats so the transposing stores do not collide on banks),
//     B row-major; both are fetched with float4 global loads when the pointers
//     and leading dimensions allow, with predicated scalar loads otherwise and
//     on ragged edges (zero-filled);
//   - two shared-memory buffers: the next slice is fetched into registers while
//     the current one is multiplied, then stored to the other buffer, so there
//     is one barrier per slice ("Step 4: Double buffering");
//   - tiles are visited in grouped order (raster.h) for L2 reuse.
#include <cuda_runtime.h>

#include "common.h"
#include "raster.h"

namespace gb300 {
namespace {

constexpr int kBM = 128, kBN = 128, kBK = 16, kThreads = 256, kPadA = 4;
constexpr int kLoads = kBK / 8;  // float4 loads of A and of B per thread per slice

template <bool VEC>
__global__ void __launch_bounds__(kThreads, 2)
    sgemm_kernel(int M, int N, int K, const float* __restrict__ A, int64_t lda,
                 const float* __restrict__ B, int64_t ldb, float* __restrict__ C, int64_t ldc,
                 int64_t tiles_m, int64_t tiles_n) {
    __shared__ __align__(16) float As[2][kBK][kBM + kPadA];
    __shared__ __align__(16) float Bs[2][kBK][kBN];

    int64_t tm, tn;
    raster_tile(blockIdx.x, tiles_m, tiles_n, 8, &tm, &tn);
    const int64_t m0 = tm * kBM, n0 = tn * kBN;
    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;

    // Global -> register mapping: A tile 128 x kBK (float4s along k at k offsets
    // a_k + 8l), B tile kBK x 128 (float4s along n at rows b_k + 8l).
    const int a_row = tid >> 1, a_k = (tid & 1) * 4;
    const int b_k = tid >> 5, b_col = (tid & 31) * 4;
    const int64_t gm = m0 + a_row;
    const int64_t gn = n0 + b_col;

    auto load_a = [&](int k0) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        const int k = k0 + a_k;
        if (gm < M) {
            const float* p = A + gm * lda + k;
            if (VEC && k + 3 < K) {
                v = *reinterpret_cast<const float4*>(p);
            } else {
                if (k + 0 < K) v.x = p[0];
                if (k + 1 < K) v.y = p[1];
                if (k + 2 < K) v.z = p[2];
                if (k + 3 < K) v.w = p[3];
            }
        }
        return v;
    };
    auto load_b = [&](int k0) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        const int k = k0 + b_k;
        if (k < K) {
            const float* p = B + static_cast<int64_t>(k) * ldb + gn;
            if (VEC && gn + 3 < N) {
                v = *reinterpret_cast<const float4*>(p);
            } else {
                if (gn + 0 < N) v.x = p[0];
                if (gn + 1 < N) v.y = p[1];
                if (gn + 2 < N) v.z = p[2];
                if (gn + 3 < N) v.w = p[3];
            }
        }
        return v;
    };
    auto store_a = [&](int buf, int l, float4 v) {
        As[buf][a_k + 8 * l + 0][a_row] = v.x;
        As[buf][a_k + 8 * l + 1][a_row] = v.y;
        As[buf][a_k + 8 * l + 2][a_row] = v.z;
        As[buf][a_k + 8 * l + 3][a_row] = v.w;
    };
    auto store_b = [&](int buf, int l, float4 v) {
        *reinterpret_cast<float4*>(&Bs[buf][b_k + 8 * l][b_col]) = v;
    };

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    const int ktiles = (K + kBK - 1) / kBK;
    float4 ra[kLoads], rb[kLoads];
#pragma unroll
    for (int l = 0; l < kLoads; ++l) {
        ra[l] = load_a(8 * l);
        rb[l] = load_b(8 * l);
        store_a(0, l, ra[l]);
        store_b(0, l, rb[l]);
    }
    __syncthreads();

    for (int kt = 0; kt < ktiles; ++kt) {
        const int cur = kt & 1;
        const bool more = kt + 1 < ktiles;
        if (more) {
#pragma unroll
            for (int l = 0; l < kLoads; ++l) {
                ra[l] = load_a((kt + 1) * kBK + 8 * l);
                rb[l] = load_b((kt + 1) * kBK + 8 * l);
            }
        }
#pragma unroll
        for (int k = 0; k < kBK; ++k) {
            const float4 a0 = *reinterpret_cast<const float4*>(&As[cur][k][ty * 4]);
            const float4 a1 = *reinterpret_cast<const float4*>(&As[cur][k][64 + ty * 4]);
            const float4 b0 = *reinterpret_cast<const float4*>(&Bs[cur][k][tx * 4]);
            const float4 b1 = *reinterpret_cast<const float4*>(&Bs[cur][k][64 + tx * 4]);
            const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        if (more) {
#pragma unroll
            for (int l = 0; l < kLoads; ++l) {
                store_a(cur ^ 1, l, ra[l]);
                store_b(cur ^ 1, l, rb[l]);
            }
        }
        __syncthreads();
    }

#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t m = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
        if (m >= M) continue;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t n = n0 + h * 64 + tx * 4;
            float* p = C + m * ldc + n;
            const float* v = &acc[i][h * 4];
            if (VEC && n + 3 < N) {
                *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (n + j < N) p[j] = v[j];
            }
        }
    }
}

}  // namespace

cudaError_t f32_launch(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                       const float* B, int64_t ldb, float* C, int64_t ldc, cudaStream_t stream) {
    const int64_t tiles_m = (M + kBM - 1) / kBM, tiles_n = (N + kBN - 1) / kBN;
    const int64_t tiles = tiles_m * tiles_n;
    if (tiles > 0x7fffffff) return cudaErrorInvalidValue;
    const bool vec = (reinterpret_cast<uintptr_t>(A) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(B) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(C) % 16 == 0) && lda % 4 == 0 &&
                     ldb % 4 == 0 && ldc % 4 == 0;
    const dim3 grid(static_cast<unsigned>(tiles));
    if (vec)
        sgemm_kernel<true><<<grid, kThreads, 0, stream>>>(int(M), int(N), int(K), A, lda, B, ldb,
                                                          C, ldc, tiles_m, tiles_n);
    else
        sgemm_kernel<false><<<grid, kThreads, 0, stream>>>(int(M), int(N), int(K), A, lda, B,
                                                           ldb, C, ldc, tiles_m, tiles_n);
    return cudaGetLastError();
}

}  // namespace gb300
