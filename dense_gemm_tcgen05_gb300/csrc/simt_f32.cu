// simt_f32.cu -- FP32 GEMM on the CUDA cores (FFMA), all matrices row-major.
//
// C[m*ldc + n] = sum_k A[m*lda + k] * B[k*ldb + n], one FP32 fused
// multiply-add per (m, n, k) in increasing k.
//
// Design, following "Optimizing GEMM in HIP" Steps 2-6 (shared-memory tiling,
// register tiling, double buffering, vectorised loads, register budget), made
// for a Blackwell SM:
//   - a 128 x 128 block tile, K slices of 8, 256 threads, 8 x 8 outputs per
//     thread held in registers (outer products, 64 FMAs per k per thread);
//   - the FMAs are issued as Blackwell's packed FP32 FMA (__ffma2_rn, two
//     fused multiply-adds per instruction on adjacent columns, each rounded
//     once like fmaf): the same results with half the FMA instructions, which
//     leaves issue slots for the shared-memory loads (measured on GB300 at
//     8192 x 8192 x 2048: 53 -> 60 TFLOP/s);
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
//   - tiles are visited in grouped order (raster.h) for L2 reuse;
//   - when it shortens the last partial wave (rule at full_tiles), that wave's
//     tiles are cut into two 128 x 64 halves (8 x 4 outputs per thread), run by
//     a second grid that programmatic dependent launch lets start while the
//     whole-tile grid's last blocks still run.
#include <cuda_runtime.h>

#include <atomic>

#include "launch.h"
#include "raster.h"

namespace gb300 {
namespace {

constexpr int kBM = 128, kBN = 128, kBK = 8, kThreads = 256, kPadA = 4;
constexpr int kLoadsA = kBM * kBK / 4 / kThreads;  // float4 loads of A per thread per slice
static_assert(kLoadsA == 1, "one float4 of A per thread per slice");

// One output tile of kBM x BN at (m0, n0); BN = 128 (full tile) or 64 (half).
// EXACT: M and N are multiples of the tile and K of the slice, and the float4
// path applies (VEC), so no load or store needs a bounds check.
// The FMAs are issued as packed pairs (__ffma2_rn: two FP32 FMAs per
// instruction, each rounded once exactly as fmaf), on pairs of adjacent
// columns: acc[i][p] holds columns 2p and 2p + 1 of row i.
template <bool VEC, int BN, bool EXACT>
__device__ __forceinline__ void sgemm_tile(int M, int N, int K, const float* __restrict__ A,
                                           int64_t lda, const float* __restrict__ B, int64_t ldb,
                                           float* __restrict__ C, int64_t ldc, int64_t m0,
                                           int64_t n0, float (*As)[kBK][kBM + kPadA],
                                           float (*Bs)[kBK][kBN]) {
    constexpr int kGroups = BN / 64;                // 4-column groups per thread
    constexpr int kBVec = kBK * BN / 4;             // float4s of B per slice
    static_assert(kBVec <= kThreads, "at most one float4 of B per thread per slice");
    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;

    // Global -> register mapping: A tile 128 x kBK (two threads per row, a
    // float4 each along k), B tile kBK x BN (one float4 along n for each of the
    // first kBVec threads).
    const int a_row = tid >> 1, a_k = (tid & 1) * 4;
    const int b_k = tid / (BN / 4), b_col = (tid % (BN / 4)) * 4;
    const bool b_loader = tid < kBVec;
    const int64_t gm = m0 + a_row;
    const int64_t gn = n0 + b_col;

    auto load_a = [&](int k0) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        const int k = k0 + a_k;
        if (EXACT) return *reinterpret_cast<const float4*>(A + gm * lda + k);
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
        if (EXACT && kBVec == kThreads)
            return *reinterpret_cast<const float4*>(B + static_cast<int64_t>(k) * ldb + gn);
        if (b_loader && (EXACT || k < K)) {
            const float* p = B + static_cast<int64_t>(k) * ldb + gn;
            if (EXACT || (VEC && gn + 3 < N)) {
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
    auto store_a = [&](int buf, float4 v) {
        As[buf][a_k + 0][a_row] = v.x;
        As[buf][a_k + 1][a_row] = v.y;
        As[buf][a_k + 2][a_row] = v.z;
        As[buf][a_k + 3][a_row] = v.w;
    };
    auto store_b = [&](int buf, float4 v) {
        if (b_loader) *reinterpret_cast<float4*>(&Bs[buf][b_k][b_col]) = v;
    };

    float2 acc[8][2 * kGroups];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 2 * kGroups; ++j) acc[i][j] = make_float2(0.f, 0.f);

    const int ktiles = (K + kBK - 1) / kBK;
    store_a(0, load_a(0));
    store_b(0, load_b(0));
    __syncthreads();

    for (int kt = 0; kt < ktiles; ++kt) {
        const int cur = kt & 1;
        const bool more = kt + 1 < ktiles;
        float4 ra, rb;
        if (more) {
            ra = load_a((kt + 1) * kBK);
            rb = load_b((kt + 1) * kBK);
        }
#pragma unroll
        for (int k = 0; k < kBK; ++k) {
            const float4 a0 = *reinterpret_cast<const float4*>(&As[cur][k][ty * 4]);
            const float4 a1 = *reinterpret_cast<const float4*>(&As[cur][k][64 + ty * 4]);
            const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            float2 b[2 * kGroups];
#pragma unroll
            for (int g = 0; g < kGroups; ++g) {
                const float4 bv = *reinterpret_cast<const float4*>(&Bs[cur][k][g * 64 + tx * 4]);
                b[2 * g] = make_float2(bv.x, bv.y);
                b[2 * g + 1] = make_float2(bv.z, bv.w);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float2 ai = make_float2(a[i], a[i]);
#pragma unroll
                for (int j = 0; j < 2 * kGroups; ++j) acc[i][j] = __ffma2_rn(ai, b[j], acc[i][j]);
            }
        }
        if (more) {
            store_a(cur ^ 1, ra);
            store_b(cur ^ 1, rb);
        }
        __syncthreads();
    }

#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t m = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
        if (!EXACT && m >= M) continue;
#pragma unroll
        for (int h = 0; h < kGroups; ++h) {
            const int64_t n = n0 + h * 64 + tx * 4;
            float* p = C + m * ldc + n;
            const float v[4] = {acc[i][2 * h].x, acc[i][2 * h].y, acc[i][2 * h + 1].x,
                                acc[i][2 * h + 1].y};
            if (EXACT || (VEC && n + 3 < N)) {
                *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (n + j < N) p[j] = v[j];
            }
        }
    }
}

// Block b takes tile tile_base + b (BN = 128) or one half of tile
// tile_base + b / 2 (BN = 64), tiles in grouped order.  With `dependent` set
// (half tiles launched behind the whole-tile grid with programmatic dependent
// launch), a block first lets the next grid start early and, at the end, waits
// for the grid before it to finish, so that whatever follows this grid in the
// stream sees both grids' results.
template <bool VEC, int BN, bool EXACT>
__global__ void __launch_bounds__(kThreads, 2)
    sgemm_kernel(int M, int N, int K, const float* __restrict__ A, int64_t lda,
                 const float* __restrict__ B, int64_t ldb, float* __restrict__ C, int64_t ldc,
                 int64_t tiles_m, int64_t tiles_n, int64_t tile_base, int dependent) {
    __shared__ __align__(16) float As[2][kBK][kBM + kPadA];
    __shared__ __align__(16) float Bs[2][kBK][kBN];

    if (dependent) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t b = blockIdx.x;
    int64_t tm, tn;
    raster_tile(tile_base + (BN == kBN ? b : b / 2), tiles_m, tiles_n, 8, &tm, &tn);
    const int64_t n0 = tn * kBN + (BN == kBN ? 0 : (b & 1) * BN);
    sgemm_tile<VEC, BN, EXACT>(M, N, K, A, lda, B, ldb, C, ldc, tm * kBM, n0, As, Bs);
    if (dependent && BN != kBN) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// The last k1 - k0 terms of every output's FMA chain: C[m][n] continues from
// the value the tile kernel stored for terms [0, k0), one fused multiply-add
// per term in increasing k, so the result is the chain over [0, k1) exactly.
// Used when K does not fit the tile kernel's 32-bit slice count (K > 2^31 - 8;
// then k1 - k0 <= 7).
__global__ void f32_ktail_kernel(int64_t M, int64_t N, int64_t k0, int64_t k1,
                                 const float* __restrict__ A, int64_t lda,
                                 const float* __restrict__ B, int64_t ldb, float* __restrict__ C,
                                 int64_t ldc) {
    const int64_t total = M * N;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t m = i / N, n = i - m * N;
        float acc = C[m * ldc + n];
        for (int64_t k = k0; k < k1; ++k) acc = fmaf(A[m * lda + k], B[k * ldb + n], acc);
        C[m * ldc + n] = acc;
    }
}

// How many tiles run whole (the rest run as halves), given the SM count and
// the resident blocks per SM.  Measured on GB300 (two blocks per SM): the time
// is set by the most tiles any SM runs -- it grows by one step per 152 tiles --
// and a block left alone on its SM runs about twice as fast as one of a pair,
// while a half tile alone takes nearly as long as a whole one.  Halving the
// rem = tiles mod (2 x SMs) tiles of the last partial wave therefore only pays
// when the halves still leave at most one block per SM (rem <= SMs / 2:
// 0.5-1 % faster); with larger remainders it loses up to 7 %.
int64_t full_tiles(int64_t tiles, int sms, int per_sm) {
    const int64_t slots = static_cast<int64_t>(sms) * per_sm;
    if (slots <= 0) return tiles;
    const int64_t rem = tiles % slots;
    return (rem > 0 && 2 * rem <= sms) ? tiles - rem : tiles;
}

// SM count and resident blocks per SM for each device and variant, queried
// once; 0 = not yet known.
constexpr int kMaxDevices = 64;
std::atomic<int> g_sms[kMaxDevices][2], g_per_sm[kMaxDevices][2];

cudaError_t residency(bool vec, int* sms_out, int* per_sm_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices && (*per_sm_out = g_per_sm[dev][vec].load()) > 0) {
        *sms_out = g_sms[dev][vec].load();
        return cudaSuccess;
    }
    int sms = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = vec ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                      &per_sm, sgemm_kernel<true, kBN, false>, kThreads, 0)
                : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                      &per_sm, sgemm_kernel<false, kBN, false>, kThreads, 0);
    if (e != cudaSuccess) return e;
    *sms_out = sms;
    *per_sm_out = per_sm;
    if (dev >= 0 && dev < kMaxDevices) {
        g_sms[dev][vec].store(sms);
        g_per_sm[dev][vec].store(per_sm);
    }
    return cudaSuccess;
}

template <bool VEC, bool EXACT>
cudaError_t launch_f32(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                       const float* B, int64_t ldb, float* C, int64_t ldc, cudaStream_t stream,
                       int64_t tiles_m, int64_t tiles_n, int64_t full, int64_t tiles, int mode) {
    // mode 0: half tiles behind the whole ones with programmatic dependent
    // launch; 2: the same as two plain launches.
    const int dependent = (mode == 0 && full > 0) ? 1 : 0;
    if (full > 0) {
        sgemm_kernel<VEC, kBN, EXACT><<<dim3(static_cast<unsigned>(full)), kThreads, 0, stream>>>(
            int(M), int(N), int(K), A, lda, B, ldb, C, ldc, tiles_m, tiles_n, 0, dependent);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (tiles == full) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * (tiles - full)));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = dependent ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, sgemm_kernel<VEC, kBN / 2, EXACT>, int(M), int(N), int(K), A, lda,
                              B, ldb, C, ldc, tiles_m, tiles_n, full, dependent);
}

}  // namespace

cudaError_t f32_tiles_launch(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                             const float* B, int64_t ldb, float* C, int64_t ldc,
                             cudaStream_t stream, int tail_mode);

cudaError_t f32_launch(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                       const float* B, int64_t ldb, float* C, int64_t ldc, cudaStream_t stream,
                       int tail_mode, int ktail) {
    // The tile kernel counts K slices of 8 as (K + 7) / 8 in 32 bits, so it
    // takes at most 2^31 - 8 terms; the rest (at most 7) continue each chain
    // in f32_ktail_kernel.  `ktail` > 0 moves that many terms there for any K
    // larger than it (to test that path at small sizes).
    constexpr int64_t kMaxTileK = 0x7fffffffLL - (kBK - 1);
    int64_t k_main = K > kMaxTileK ? kMaxTileK : K;
    if (ktail > 0 && K > ktail && K - ktail < k_main) k_main = K - ktail;
    cudaError_t e = f32_tiles_launch(M, N, k_main, A, lda, B, ldb, C, ldc, stream, tail_mode);
    if (e != cudaSuccess || k_main == K) return e;
    int sms = 0, per_sm = 0;
    e = residency(true, &sms, &per_sm);
    if (e != cudaSuccess) return e;
    const int64_t total = M * N;
    int64_t blocks = (total + 255) / 256;
    if (blocks > static_cast<int64_t>(sms) * 8) blocks = static_cast<int64_t>(sms) * 8;
    f32_ktail_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(M, N, k_main, K, A, lda,
                                                                        B, ldb, C, ldc);
    return cudaGetLastError();
}

cudaError_t f32_tiles_launch(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                             const float* B, int64_t ldb, float* C, int64_t ldc,
                             cudaStream_t stream, int tail_mode) {
    const int64_t tiles_m = (M + kBM - 1) / kBM, tiles_n = (N + kBN - 1) / kBN;
    const int64_t tiles = tiles_m * tiles_n;
    if (tiles > 0x3fffffff) return cudaErrorInvalidValue;
    const bool vec = (reinterpret_cast<uintptr_t>(A) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(B) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(C) % 16 == 0) && lda % 4 == 0 &&
                     ldb % 4 == 0 && ldc % 4 == 0;
    int sms = 0, per_sm = 0;
    const cudaError_t e = residency(vec, &sms, &per_sm);
    if (e != cudaSuccess) return e;
    const int64_t full = tail_mode == 1 ? tiles : full_tiles(tiles, sms, per_sm);
    const bool exact = vec && M % kBM == 0 && N % kBN == 0 && K % kBK == 0;
    if (exact)
        return launch_f32<true, true>(M, N, K, A, lda, B, ldb, C, ldc, stream, tiles_m, tiles_n,
                                      full, tiles, tail_mode);
    return vec ? launch_f32<true, false>(M, N, K, A, lda, B, ldb, C, ldc, stream, tiles_m, tiles_n,
                                         full, tiles, tail_mode)
               : launch_f32<false, false>(M, N, K, A, lda, B, ldb, C, ldc, stream, tiles_m,
                                          tiles_n, full, tiles, tail_mode);
}

}  // namespace gb300
