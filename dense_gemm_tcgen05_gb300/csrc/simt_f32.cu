// simt_f32.cu -- FP32 GEMM on the CUDA cores (FFMA), all matrices row-major.
//
// C[m*ldc + n] = sum_k A[m*lda + k] * B[k*ldb + n], one FP32 fused
// multiply-add per (m, n, k) in increasing k.
//
// Design, following "Optimizing GEMM in HIP" Steps 2-6 (shared-memory tiling,
// register tiling, double buffering, vectorised loads, register budget), made
// for a Blackwell SM:
//   - a 128 x 128 block tile, K slices of 16, 128 threads, 16 x 8 outputs per
//     thread held in registers (outer products, 128 FMAs per k per thread),
//     two blocks per SM;
//   - the FMAs are issued as Blackwell's packed FP32 FMA (__ffma2_rn, two
//     fused multiply-adds per instruction on adjacent columns, each rounded
//     once like fmaf), the A value of a row broadcast to both lanes: half the
//     FMA instructions, which leaves issue slots for the shared-memory loads;
//   - slices move from global to shared memory with cp.async (no registers
//     staged) into a ring of three buffers, one barrier per slice; A is
//     written k-major (transposed on the way in by 4-byte copies, rows padded
//     by 4 floats), B row-major by 16-byte copies when its rows allow, 4-byte
//     copies otherwise; ragged edges are zero-filled by the copies;
//   - a thread's 8 columns are two groups of 4, 64 apart, and its 16 rows four
//     groups of 4, 32 apart; a warp's threads are 16 along n by 2 along m, so
//     every fragment load is one conflict-free float4 per thread, and a B load
//     of a warp reads 256 distinct bytes (shared-memory wavefronts per k: 15.5
//     per warp against 19 with 8 x 16 outputs per thread, whose B loads read
//     128 distinct bytes four times over);
//   - inside a slice the A fragments of the next k are loaded while the
//     current ones are multiplied;
//   - tiles are visited in grouped order (raster.h) for L2 reuse;
//   - when it shortens the last partial wave (rule at full_tiles), that wave's
//     tiles are cut into two 128 x 64 halves (8 x 8 outputs per thread), run by
//     a second grid that programmatic dependent launch lets start while the
//     whole-tile grid's last blocks still run.
// Measured on GB300: 65.2 TFLOP/s at 4096^3 and 68.0 at 8192 x 8192 x 2048
// (0.81 and 0.84 of 152 SMs x 128 lanes x 2 x 2.07 GHz), against 56 and 59 for
// the previous design (128 x 128 x 8 tiles, 256 threads of 8 x 8 outputs,
// register-staged double buffering).
#include <cuda_runtime.h>

#include <atomic>

#include "launch.h"
#include "raster.h"

namespace gb300 {
namespace {

constexpr int kBM = 128, kBN = 128, kBK = 16, kStages = 3, kThreads = 128, kPadA = 4;
constexpr int kAS = kBM + kPadA;             // k-major A row stride in shared memory (floats)
constexpr int kAStage = kBK * kAS;           // floats of A per ring slot

constexpr int kTM = 16;                      // rows per thread: four groups of 4, 32 apart
constexpr int kRowGroups = kTM / 4, kRowStride = kBM / kRowGroups;
constexpr int kThreadsN = 16;                 // threads along n
static_assert(kThreads / kThreadsN * 4 == kRowStride, "row groups tile the block rows");

template <int BN>
struct SimtShape {
    static constexpr int kTN = BN / kThreadsN;  // columns per thread
    static constexpr int kGroups = kTN / 4;     // 4-column groups per thread
    static constexpr int kGroupStride = BN / kGroups;
    static constexpr int kStage = kAStage + kBK * BN;           // floats per ring slot
    static constexpr int kSmemBytes = kStages * kStage * 4;
    static constexpr int kBChunksPerRow = BN / 4;               // 16-byte chunks of a B row
    static constexpr int kBRowsPerPass = kThreads / kBChunksPerRow;
    static constexpr int kBPerThread = kBK / kBRowsPerPass;     // chunks per thread per slice
    static_assert(kBK % kBRowsPerPass == 0, "B slice rows divide among the threads");
};

constexpr int kAPerThread = kBM * kBK / kThreads;  // 4-byte A copies per thread per slice
static_assert(kAPerThread == 16, "a thread's A copies cover 16 rows 4 apart");

// FILL: the form with a source size, whose missing bytes are zero-filled (ragged
// edges); without it every copy moves all of its bytes.
template <bool FILL>
__device__ __forceinline__ void cp_async4(uint32_t dst, const float* src, uint32_t bytes) {
    if (FILL)
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src),
                     "r"(bytes)
                     : "memory");
    else
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
template <bool FILL>
__device__ __forceinline__ void cp_async16(uint32_t dst, const float* src, uint32_t bytes) {
    if (FILL)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                     "r"(bytes)
                     : "memory");
    else
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// p += step in an opaque add: keeps one running pointer live instead of one
// precomputed address per copy.
__device__ __forceinline__ const float* step_ptr(const float* p, int64_t step_bytes) {
    asm volatile("add.s64 %0, %0, %1;" : "+l"(p) : "l"(step_bytes));
    return p;
}

// One output tile of kBM x BN at (m0, n0); BN = 128 (full tile) or 64 (half).
// VEC: B's rows and C's rows are 16-byte aligned (16-byte B copies, float4
// stores).  EXACT: M and N are multiples of the tile, K of the slice, and VEC
// holds, so no copy or store needs a bounds check.
template <bool VEC, int BN, bool EXACT>
__device__ __forceinline__ void sgemm_tile(int M, int N, int K, const float* __restrict__ A,
                                           int64_t lda, const float* __restrict__ B, int64_t ldb,
                                           float* __restrict__ C, int64_t ldc, int64_t m0,
                                           int64_t n0, float* smem) {
    using S = SimtShape<BN>;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int tx = tid % kThreadsN;           // columns g*kGroupStride + tx*4 + 0..3
    const int ty = tid / kThreadsN;           // rows q*kRowStride + ty*4 + 0..3

    // A copies: instruction j of warp w covers rows r0 + 4 j (r0 = 64 (w & 1)
    // + lane & 3), k = 8 (w >> 1) + lane >> 2 of the slice: a warp reads 4 rows
    // x 8 consecutive k (32 bytes each) and writes 32 distinct banks.
    const int a_row = 64 * (warp & 1) + (lane & 3);
    const int a_k = 8 * (warp >> 1) + (lane >> 2);
    const int64_t a_step = 4 * lda * static_cast<int64_t>(sizeof(float));
    const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    const uint32_t a_dst = sbase + 4u * (a_k * kAS + a_row);
    uint32_t a_rows_ok = 0xffffu;             // bit j: row a_row + 4 j exists
    if (!EXACT) {
        a_rows_ok = 0;
#pragma unroll
        for (int j = 0; j < kAPerThread; ++j)
            if (m0 + a_row + 4 * j < M) a_rows_ok |= 1u << j;
    }
    const float* a_src = A + (m0 + a_row) * lda + a_k;
    // B copies: chunk j = row tid / kBChunksPerRow + kBRowsPerPass j, columns
    // (tid % kBChunksPerRow) * 4 .. + 3.
    const int b_k = tid / S::kBChunksPerRow;
    const int b_n = (tid % S::kBChunksPerRow) * 4;
    const int64_t b_step = S::kBRowsPerPass * ldb * static_cast<int64_t>(sizeof(float));
    const uint32_t b_dst = sbase + 4u * (kAStage + b_k * BN + b_n);
    const int64_t gn = n0 + b_n;
    uint32_t b_bytes = 16;                    // valid bytes of the chunk (VEC)
    if (!EXACT) {
        const int64_t left = gn < N ? N - gn : 0;
        b_bytes = left >= 4 ? 16u : static_cast<uint32_t>(left * 4);
    }
    const float* b_src = B + static_cast<int64_t>(b_k) * ldb + gn;

    int k0 = 0;
    auto issue = [&](int slot) {
        const uint32_t off = 4u * slot * S::kStage;
        const bool k_ok = EXACT || k0 + a_k < K;
        const float* p = a_src;
#pragma unroll
        for (int j = 0; j < kAPerThread; ++j) {
            const bool ok = EXACT || (k_ok && ((a_rows_ok >> j) & 1u));
            cp_async4<!EXACT>(a_dst + off + 16u * j, ok ? p : A, ok ? 4u : 0u);
            if (j + 1 < kAPerThread) p = step_ptr(p, a_step);
        }
        const float* q = b_src;
#pragma unroll
        for (int j = 0; j < S::kBPerThread; ++j) {
            const uint32_t d = b_dst + off + 4u * S::kBRowsPerPass * BN * j;
            const bool row_ok = EXACT || k0 + b_k + S::kBRowsPerPass * j < K;
            if (VEC) {
                const uint32_t bytes = row_ok ? b_bytes : 0u;
                cp_async16<!EXACT>(d, bytes ? q : B, bytes);
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const bool ok = row_ok && gn + e < N;
                    cp_async4<true>(d + 4u * e, ok ? q + e : B, ok ? 4u : 0u);
                }
            }
            if (j + 1 < S::kBPerThread) q = step_ptr(q, b_step);
        }
        a_src += kBK;
        b_src += static_cast<int64_t>(kBK) * ldb;
        k0 += kBK;
    };

    float2 acc[kTM][S::kTN / 2];
#pragma unroll
    for (int i = 0; i < kTM; ++i)
#pragma unroll
        for (int j = 0; j < S::kTN / 2; ++j) acc[i][j] = make_float2(0.f, 0.f);

    const int ktiles = (K + kBK - 1) / kBK;
#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
        if (s < ktiles) issue(s);
        cp_async_commit();
    }
    int rd = 0, wr = kStages - 1;
    for (int kt = 0; kt < ktiles; ++kt) {
        cp_async_wait<kStages - 2>();         // this thread's copies of slice kt landed
        __syncthreads();                      // everyone's; and slot wr is no longer read
        if (kt + kStages - 1 < ktiles) issue(wr);
        cp_async_commit();
        const float* As = smem + rd * S::kStage;
        const float* Bs = As + kAStage;
        float4 an[kRowGroups], ac[kRowGroups];
#pragma unroll
        for (int q = 0; q < kRowGroups; ++q)
            an[q] = *reinterpret_cast<const float4*>(As + q * kRowStride + 4 * ty);
#pragma unroll
        for (int k = 0; k < kBK; ++k) {
#pragma unroll
            for (int q = 0; q < kRowGroups; ++q) ac[q] = an[q];
            if (k + 1 < kBK) {
#pragma unroll
                for (int q = 0; q < kRowGroups; ++q)
                    an[q] = *reinterpret_cast<const float4*>(As + (k + 1) * kAS + q * kRowStride +
                                                             4 * ty);
            }
            float4 bq[S::kGroups];
#pragma unroll
            for (int g = 0; g < S::kGroups; ++g)
                bq[g] = *reinterpret_cast<const float4*>(Bs + k * BN + g * S::kGroupStride + 4 * tx);
            // Column pair outer, rows inner: one B pair feeds 16 FMA pairs in a row.
#pragma unroll
            for (int g = 0; g < S::kGroups; ++g) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float2 b = h ? make_float2(bq[g].z, bq[g].w) : make_float2(bq[g].x, bq[g].y);
#pragma unroll
                    for (int q = 0; q < kRowGroups; ++q) {
                        const float a4[4] = {ac[q].x, ac[q].y, ac[q].z, ac[q].w};
#pragma unroll
                        for (int r = 0; r < 4; ++r)
                            acc[4 * q + r][2 * g + h] =
                                __ffma2_rn(make_float2(a4[r], a4[r]), b, acc[4 * q + r][2 * g + h]);
                    }
                }
            }
        }
        rd = rd + 1 == kStages ? 0 : rd + 1;
        wr = wr + 1 == kStages ? 0 : wr + 1;
    }
    cp_async_wait<0>();

#pragma unroll
    for (int i = 0; i < kTM; ++i) {
        const int64_t m = m0 + (i / 4) * kRowStride + ty * 4 + (i % 4);
        if (!EXACT && m >= M) continue;
#pragma unroll
        for (int g = 0; g < S::kGroups; ++g) {
            const int64_t n = n0 + g * S::kGroupStride + tx * 4;
            float* p = C + m * ldc + n;
            const float v[4] = {acc[i][2 * g].x, acc[i][2 * g].y, acc[i][2 * g + 1].x,
                                acc[i][2 * g + 1].y};
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

// Block b takes tile tile_base + b (BN = 128) or half b % 2 of tile
// tile_base + b / 2 (BN = 64), tiles in grouped order.  With `dependent` set
// (halves launched behind the whole-tile grid with programmatic dependent
// launch), a block first lets the next grid start early and, at the end,
// waits for the grid before it to finish, so that whatever follows this grid
// in the stream sees both grids' results.
template <bool VEC, int BN, bool EXACT>
__global__ void __launch_bounds__(kThreads, 2)
    sgemm_kernel(int M, int N, int K, const float* __restrict__ A, int64_t lda,
                 const float* __restrict__ B, int64_t ldb, float* __restrict__ C, int64_t ldc,
                 int64_t tiles_m, int64_t tiles_n, int64_t tile_base, int dependent) {
    extern __shared__ __align__(16) float smem[];

    if (dependent) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t b = blockIdx.x;
    int64_t tm, tn;
    constexpr int kPieces = kBN / BN;
    raster_tile(tile_base + b / kPieces, tiles_m, tiles_n, 8, &tm, &tn);
    const int64_t n0 = tn * kBN + (b % kPieces) * BN;
    sgemm_tile<VEC, BN, EXACT>(M, N, K, A, lda, B, ldb, C, ldc, tm * kBM, n0, smem);
    if (dependent && BN != kBN) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// The last k1 - k0 terms of every output's FMA chain: C[m][n] continues from
// the value the tile kernel stored for terms [0, k0), one fused multiply-add
// per term in increasing k, so the result is the chain over [0, k1) exactly.
// Used when K does not fit the tile kernel's 32-bit slice count (K > 2^31 - 16;
// then k1 - k0 <= 15).
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
// the resident blocks per SM.  Measured on GB300 (two blocks per SM, 4096-term
// tiles): a block left alone on its SM takes about half the time of one of a
// pair (one block's four warps nearly fill the FMA pipes), and two halves
// sharing an SM take about as long as a lone whole tile.  With rem = tiles mod
// (2 x SMs) whole tiles left for the last partial wave:
//   rem <= SMs / 2: every half runs alone on its SM -- halves (64 tiles on 152
//     SMs: 41.0 against 25.1 TFLOP/s; 20: 51.7 against 44.4);
//   SMs / 2 < rem <= SMs: whole tiles run alone, halves in pairs -- whole
//     (112: 64.1 against 63.3; 144: 61.1 against 50.8);
//   SMs < rem <= 3 SMs / 2: whole tiles end with some SMs running a pair,
//     halves with one wave of pairs and a few lone halves -- halves (176: 53.3
//     against 49.2 and 65.1 against 63.8);
//   larger: two waves of half pairs against one of whole pairs -- whole (256:
//     53.9 against 48.9; 272: 62.3 against 59.4).
int64_t full_tiles(int64_t tiles, int sms, int per_sm) {
    const int64_t slots = static_cast<int64_t>(sms) * per_sm;
    if (slots <= 0) return tiles;
    const int64_t rem = tiles % slots;
    if (rem == 0) return tiles;
    const bool halve = 2 * rem <= sms || (per_sm == 2 && rem > sms && 2 * rem <= 3 * sms);
    return halve ? tiles - rem : tiles;
}

// SM count and resident blocks per SM for each device and variant, queried
// once; 0 = not yet known.
constexpr int kMaxDevices = 64;
std::atomic<int> g_sms[kMaxDevices][2], g_per_sm[kMaxDevices][2];

// The whole-tile ring (3 x 16.3 KiB) is above the 48 KiB that a launch may
// take without opting in; every instantiation opts in to its own size.
template <bool VEC, int BN, bool EXACT>
cudaError_t allow_smem() {
    return cudaFuncSetAttribute(sgemm_kernel<VEC, BN, EXACT>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                SimtShape<BN>::kSmemBytes);
}

cudaError_t allow_smem_all() {
    cudaError_t e = allow_smem<true, kBN, true>();
    if (e == cudaSuccess) e = allow_smem<true, kBN, false>();
    if (e == cudaSuccess) e = allow_smem<false, kBN, false>();
    if (e == cudaSuccess) e = allow_smem<true, kBN / 2, true>();
    if (e == cudaSuccess) e = allow_smem<true, kBN / 2, false>();
    if (e == cudaSuccess) e = allow_smem<false, kBN / 2, false>();
    return e;
}

cudaError_t residency(bool vec, int* sms_out, int* per_sm_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices && (*per_sm_out = g_per_sm[dev][vec].load()) > 0) {
        *sms_out = g_sms[dev][vec].load();
        return cudaSuccess;
    }
    // First use on this device: the opt-in comes before any launch (the
    // cached residency below is only stored after it succeeded).
    e = allow_smem_all();
    if (e != cudaSuccess) return e;
    int sms = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = vec ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                      &per_sm, sgemm_kernel<true, kBN, false>, kThreads, SimtShape<kBN>::kSmemBytes)
                : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                      &per_sm, sgemm_kernel<false, kBN, false>, kThreads,
                      SimtShape<kBN>::kSmemBytes);
    if (e != cudaSuccess) return e;
    *sms_out = sms;
    *per_sm_out = per_sm;
    if (dev >= 0 && dev < kMaxDevices) {
        g_sms[dev][vec].store(sms);
        g_per_sm[dev][vec].store(per_sm);
    }
    return cudaSuccess;
}

// Whole tiles [0, full) in one grid, the rest cut into halves in a second.
// mode 2 launches the second grid plainly; every other mode behind the first
// with programmatic dependent launch.
template <bool VEC, bool EXACT>
cudaError_t launch_f32(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                       const float* B, int64_t ldb, float* C, int64_t ldc, cudaStream_t stream,
                       int64_t tiles_m, int64_t tiles_n, int64_t full, int64_t tiles, int mode) {
    constexpr int BN = kBN / 2;
    const int dependent = (mode != 2 && full > 0) ? 1 : 0;
    if (full > 0) {
        sgemm_kernel<VEC, kBN, EXACT>
            <<<dim3(static_cast<unsigned>(full)), kThreads, SimtShape<kBN>::kSmemBytes, stream>>>(
                int(M), int(N), int(K), A, lda, B, ldb, C, ldc, tiles_m, tiles_n, 0, dependent);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (tiles == full) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((kBN / BN) * (tiles - full)));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = SimtShape<BN>::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = dependent ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, sgemm_kernel<VEC, BN, EXACT>, int(M), int(N), int(K), A, lda, B,
                              ldb, C, ldc, tiles_m, tiles_n, full, dependent);
}

}  // namespace

cudaError_t f32_tiles_launch(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                             const float* B, int64_t ldb, float* C, int64_t ldc,
                             cudaStream_t stream, int tail_mode);

cudaError_t f32_launch(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                       const float* B, int64_t ldb, float* C, int64_t ldc, cudaStream_t stream,
                       int tail_mode, int ktail) {
    // The tile kernel counts K slices of 16 as (K + 15) / 16 in 32 bits, so it
    // takes at most 2^31 - 16 terms; the rest (at most 15) continue each chain
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
    // A moves in 4-byte copies whatever its alignment; B's 16-byte copies and
    // C's float4 stores need 16-byte rows.
    const bool vec = (reinterpret_cast<uintptr_t>(B) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(C) % 16 == 0) && ldb % 4 == 0 && ldc % 4 == 0;
    int sms = 0, per_sm = 0;
    const cudaError_t e = residency(vec, &sms, &per_sm);
    if (e != cudaSuccess) return e;
    // tail_mode 3 halves the last partial wave whatever its size (tests, tuning).
    const int64_t slots = static_cast<int64_t>(sms) * per_sm;
    const int64_t full = tail_mode == 1   ? tiles
                         : tail_mode == 3 ? (slots > 0 ? tiles - tiles % slots : tiles)
                                          : full_tiles(tiles, sms, per_sm);
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
