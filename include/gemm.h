/*
 * gemm.h -- C ABI of libgemm.so, a dense GEMM library for one NVIDIA GB300
 * GPU (sm_103a).
 *
 * Every entry point computes the plain product C := A x B,
 *
 *     C[m][n] = sum_{k < K} a(m, k) * b(k, n),
 *
 * with no alpha/beta ("Optimizing GEMM in HIP", section "GEMM fundamentals":
 * an M x K matrix times a K x N matrix gives the M x N product).
 *
 * Conventions shared by all compute entry points
 * ------------------------------------------------
 *  - Dimensions and leading dimensions are element counts (int64_t).  M, N and
 *    K must lie in [0, 2^31 - 1]; a leading dimension must be at least its
 *    documented minimum and at most 2^48 (GEMM_ERR_INVALID_LD otherwise).
 *  - All matrix pointers are DEVICE pointers on the current CUDA device.  The
 *    caller owns every buffer; the library allocates no device memory per call.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Work is enqueued on it and the call returns without
 *    synchronising; results are valid once the stream has been synchronised.
 *  - All arguments are validated before anything is launched.  On any error
 *    status nothing is launched and C is not written.
 *  - M == 0 or N == 0 is a successful no-op.  K == 0 writes C = 0 (the empty
 *    sum).  C overlapping A or B gives undefined results.
 *  - Calls may be made from several host threads; the library keeps only
 *    per-device cached attributes and the options set by gemm_set_option.
 *
 * Status codes (return values)
 * ----------------------------
 */
#ifndef DENSE_GEMM_TCGEN05_GB300_GEMM_H
#define DENSE_GEMM_TCGEN05_GB300_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GEMM_OK 0                     /* success */
#define GEMM_ERR_INVALID_DIM 1        /* M, N or K negative or above 2^31 - 1 */
#define GEMM_ERR_INVALID_LD 2         /* a leading dimension below its minimum or above 2^48 */
#define GEMM_ERR_NULL_PTR 3           /* NULL matrix pointer with a nonzero extent */
#define GEMM_ERR_MISALIGNED 4         /* pointer not aligned to its element size */
#define GEMM_ERR_UNSUPPORTED_DEVICE 5 /* current device is not compute capability 10.3 */
#define GEMM_ERR_LAUNCH 6             /* a CUDA runtime error; see gemm_status_string */
#define GEMM_ERR_TIMEOUT 7            /* a device-side wait ran out (gemm_read_watchdog) */
#define GEMM_ERR_INVALID_OPTION 8     /* unknown option name or value (gemm_set_option) */
#define GEMM_ERR_SCRATCH 9            /* split needs more than gemm_bf16_tn_noalloc's scratch */
#define GEMM_ERR_WORKSPACE 10         /* gemm_f32_bf16x6 without a large enough workspace */

/*
 * gemm_f32 -- FP32 GEMM, every matrix row-major ("Optimizing GEMM in HIP":
 * FP32 matrices in row-major layout, Steps 3-6 register tiling, double
 * buffering, vectorised loads).
 *
 *   a(m, k) = A[m*lda + k]   lda >= max(1, K)
 *   b(k, n) = B[k*ldb + n]   ldb >= max(1, N)
 *   C[m*ldc + n]             ldc >= max(1, N)
 *
 * Products and sums in FP32 (fused multiply-add), one rounding per step.
 * A, B and C must be 4-byte aligned.  K may be up to 2^31 - 1: the tile
 * kernel counts K slices of 16 in 32 bits and takes the first 2^31 - 16
 * terms, and a second kernel continues each output's FMA chain over the rest
 * (at most 15), so the result is the same chain.
 */
int gemm_f32(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda, const float* B,
             int64_t ldb, float* C, int64_t ldc, void* stream);

/*
 * gemm_f32_bf16x6 -- the FP32 GEMM of gemm_f32 (same arguments, layouts and
 * checks), computed on the tensor cores instead of the CUDA cores.  The pages
 * compute FP32 GEMMs with FP32 FMAs only ("Optimizing GEMM in HIP"); this is a
 * library extension for the same product:
 *
 *   each FP32 value x is split exactly into three bfloat16 pieces,
 *   x = x0 + x1 + x2 (x0 = bf16_rne(x), x1 = bf16_rne(x - x0), x2 = x - x0 - x1);
 *   C = sum of the six piece products a2 b0, a1 b1, a0 b2, a1 b0, a0 b1, a0 b0,
 *   each formed exactly and summed in the tensor cores' FP32 accumulator, the
 *   smallest first.
 *
 * The three products left out are below 2^-25 |a b|, so the error is that of
 * an FP32 GEMM: FP32 accumulation over 6 K terms.  Results are not bit-equal
 * to gemm_f32 (another summation order), but inputs whose products and partial
 * sums are exact in FP32 (small integers, +-1, an identity operand) give exact
 * results on both.  Exact splitting needs finite inputs with |x| in about
 * [2^-100, 2^127); outside that range pieces lose bits, and Inf or NaN inputs
 * give NaN.
 *
 * Workspace: the splits are written to the workspace registered with
 * gemm_set_workspace for the current device.  The call needs at least
 * gemm_f32_bf16x6_workspace_bytes(M, N, K) bytes there and returns
 * GEMM_ERR_WORKSPACE, launching nothing, without them.  Bytes beyond that let
 * shapes with few output tiles split K, and long tiles cut their last wave
 * into K pieces, as the TN calls do (up to
 * gemm_workspace_bytes(N, M, 6 * Kp) more, Kp = K rounded up to a multiple of
 * 64).  The workspace is in use until the call's work on `stream` has ended.
 * Launches: two split kernels, then the tensor-core GEMM (the split counters
 * in the workspace need no memset; see gemm_set_workspace).
 */
int gemm_f32_bf16x6(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda, const float* B,
                    int64_t ldb, float* C, int64_t ldc, void* stream);

/*
 * Workspace bytes gemm_f32_bf16x6 needs for an M x N x K product: two split
 * operands of (M + N) rows of 6 Kp bfloat16 values, each rounded up to 256
 * bytes, plus the 128 KiB of split counters.  0 when M, N or K is 0 or out of
 * range; sizes that no device could hold are not exact but at least INT64_MAX / 4.
 */
int64_t gemm_f32_bf16x6_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * gemm_f16_tn -- FP16 inputs, FP32 accumulation, FP16 output, "TN" layout
 * ("FP16 GEMM Optimization on AMD RDNA 3 and RDNA 4", section "What We Are
 * Computing": A row-major, B column-major so both are contiguous along K, and
 * C column-major with leading dimension M):
 *
 *   a(m, k) = A[m*lda + k]   lda >= max(1, K)   (IEEE binary16 codes)
 *   b(k, n) = B[n*ldb + k]   ldb >= max(1, K)
 *   C[n*ldc + m]             ldc >= max(1, M)   (binary16, round to nearest even)
 *
 * Pointers must be 2-byte aligned.  The tensor-core (tcgen05) kernel runs for
 * every alignment: operands whose rows are 16-byte aligned (base and lda*2,
 * ldb*2) are loaded by TMA, others by producer warps with aligned 16-byte
 * loads; a C whose rows are 16-byte aligned is written by TMA, otherwise by
 * row-wise stores.  Accumulation is FP32; the output is rounded once, to
 * nearest even.
 */
int gemm_f16_tn(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                int64_t ldb, void* C, int64_t ldc, void* stream);

/*
 * gemm_f16_tn_acc16 -- as gemm_f16_tn, but the tensor core accumulates in FP16,
 * the mode the FP16 page measures ("FP16 GEMM Optimization on AMD RDNA 3 and
 * RDNA 4", "The Target": both the kernels and hipBLASLt accumulate in FP16,
 * HIPBLAS_COMPUTE_16F).  On GB300 it runs at the same tensor rate as FP32
 * accumulation and is less accurate over long K; it is exact while every
 * partial sum is an integer FP16 holds (|sum| <= 2048), e.g. for +-1 inputs
 * with K <= 2048.  Never splits K; option "path" = 1 does not apply.
 */
int gemm_f16_tn_acc16(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                      int64_t ldb, void* C, int64_t ldc, void* stream);

/*
 * gemm_bf16_tn -- as gemm_f16_tn with bfloat16 inputs and a bfloat16 output
 * ("An Educational GEMM Ladder for Helios GPUs": BF16 inputs and output with
 * FP32 accumulation).
 */
int gemm_bf16_tn(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                 int64_t ldb, void* C, int64_t ldc, void* stream);

/*
 * gemm_fp8_tn -- FP8 E4M3 inputs with per-tensor FP32 scales, FP32
 * accumulation, bfloat16 output, TN layout ("FP8 GEMM Optimization on AMD
 * RDNA 4", section "What Changes at FP8": E4M3 x E4M3 accumulated in FP32;
 * that page applies no scales, the per-tensor scales here are applied once, in
 * the epilogue):
 *
 *   C[n*ldc + m] = bf16_rne( fp32(scale_a * scale_b) * sum_k qa(m,k) * qb(k,n) )
 *
 *   qa(m, k) = A[m*lda + k] (OCP E4M3 codes, one byte)   lda >= max(1, K)
 *   qb(k, n) = B[n*ldb + k]                              ldb >= max(1, K)
 *   C: bfloat16, column-major                            ldc >= max(1, M)
 *
 * C must be 2-byte aligned.  A and B may have any alignment; TMA loads them
 * when their bases are 16-byte aligned and lda, ldb are multiples of 16.
 */
int gemm_fp8_tn(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                int64_t ldb, float scale_a, float scale_b, void* C, int64_t ldc, void* stream);

/*
 * gemm_fp8_tn_f32 -- as gemm_fp8_tn with an FP32 output, the layout the FP8
 * page writes ("FP8 GEMM Optimization on AMD RDNA 4", "What Changes at FP8",
 * "Accumulator type": FP32 C, column-major, leading dimension M):
 *
 *   C[n*ldc + m] = fp32(scale_a * scale_b) * sum_k qa(m,k) * qb(k,n)
 *
 * (one FP32 multiply of the FP32 accumulator, no further rounding).  C must be
 * 4-byte aligned; TMA writes it when C is 16-byte aligned and ldc is a multiple
 * of 4.
 */
int gemm_fp8_tn_f32(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                    int64_t ldb, float scale_a, float scale_b, float* C, int64_t ldc,
                    void* stream);

/*
 * gemm_tn_plan -- what a TN call would run, decided on the host without a GPU
 * (for tests and tuning; nothing is launched and no device is touched).  The
 * calls plan with exactly this function, reading the same options
 * (gemm_set_option).
 *
 *   kind             GEMM_PLAN_F16 (gemm_f16_tn), GEMM_PLAN_BF16, GEMM_PLAN_FP8,
 *                    GEMM_PLAN_F16_ACC16 (gemm_f16_tn_acc16), GEMM_PLAN_FP8_F32OUT
 *   M, N, K          as for the call (all > 0)
 *   flags            GEMM_PLAN_A_TMA / _B_TMA / _C_TMA: that matrix's base and row
 *                    pitch are 16-byte aligned (TMA can address its rows);
 *                    GEMM_PLAN_A_128 / _B_128: A's or B's rows start on 128-byte
 *                    boundaries (base and pitch); GEMM_PLAN_NOALLOC: plan as
 *                    gemm_bf16_tn_noalloc does, with workspace_bytes standing for
 *                    its fixed array (pass GEMM_NOALLOC_SCRATCH_BYTES) and the
 *                    value of option "splits" for its `splits` argument
 *   workspace_bytes  the registered workspace (0: none)
 *   sms              the device's SM count (152 on GB300)
 *   out[nout]        nout >= GEMM_PLAN_FIELDS; receives, in this order: status
 *                    (GEMM_OK), CTA pairs (0/1), producer (0 TMA, 1 load-based),
 *                    tile width along M, 64-row tiles (0/1), K pieces per tile,
 *                    last-wave units per tile (1: untouched), last wave cut along K
 *                    (0/1; else along M), ring stages, grid (CTAs), A repacked,
 *                    B repacked, tiles along N, tiles along M, K stages per
 *                    piece, K stages per last-wave piece, ring stage bytes,
 *                    MMA-issuing warps (1 or 2), K atoms per ring stage (1 or 2),
 *                    ring over the epilogue's staging area (0/1: only where every
 *                    CTA or CTA pair runs one unit).
 *
 * Returns GEMM_OK, GEMM_ERR_INVALID_DIM or GEMM_ERR_INVALID_OPTION (kind, out
 * or nout).  A call that would be refused reports its status in out[0]
 * (GEMM_ERR_SCRATCH for a forced no-allocation split that cannot fit).
 */
#define GEMM_PLAN_F16 0
#define GEMM_PLAN_BF16 1
#define GEMM_PLAN_FP8 2
#define GEMM_PLAN_F16_ACC16 3
#define GEMM_PLAN_FP8_F32OUT 4
#define GEMM_PLAN_A_TMA 1
#define GEMM_PLAN_B_TMA 2
#define GEMM_PLAN_C_TMA 4
#define GEMM_PLAN_A_128 8
#define GEMM_PLAN_B_128 16
#define GEMM_PLAN_NOALLOC 32
#define GEMM_PLAN_FIELDS 20
int gemm_tn_plan(int kind, int64_t M, int64_t N, int64_t K, int flags, int64_t workspace_bytes,
                 int sms, int64_t* out, int nout);

/* Human-readable text for a status code.  For GEMM_ERR_LAUNCH it names the
 * last CUDA error this thread saw.  The returned string is static. */
const char* gemm_status_string(int status);

/*
 * gemm_read_watchdog -- every wait inside the library's kernels gives up after
 * a time limit (gemm_set_option "timeout_ns"), records GEMM_ERR_TIMEOUT in a
 * per-device status word and lets its kernel exit cleanly instead of hanging.
 * This call synchronises the current device, returns GEMM_OK when no wait has
 * run out since the last reset, GEMM_ERR_TIMEOUT when one has (or when a
 * kernel refused launch parameters that break one of its invariants, which
 * the library's planner does not produce), and GEMM_ERR_LAUNCH on a CUDA
 * error.  reset != 0 clears the word.
 */
int gemm_read_watchdog(int reset);

/*
 * gemm_set_option -- process-wide tuning and test switches.  Not meant to be
 * changed while calls are in flight on other host threads.
 *   "pair"        -1 auto (default: CTA pairs, except when the pair tiles fill less
 *                 than one wave and single-CTA tiles 64 (M <= 128) or 128 wide along
 *                 M fit in one: then those), 0 one CTA per tile, 1 a cta_group::2 pair
 *   "group"       tile-rasteriser group size in tile rows, 1..64, or 0 (default):
 *                 16, chosen for the GB300 L2 (two per-die partitions)
 *   "band_snake"  1 (default): odd rasteriser groups walk the tile columns backwards
 *                 (gemm_tile_coord), so a group starts on the column panels the
 *                 previous one ended on; 0: every group walks forwards
 *   "k_snake"     1 (default): every second tile a CTA runs reads its K range
 *                 backwards, so the K slices one wave of tiles ends on are still in
 *                 L2 when the next wave starts on them; 0: always ascending.  The
 *                 summation order of those tiles changes, not the result's
 *                 accuracy; results stay deterministic for a given shape
 *   "k_rotate"    2: the TMA producer starts each unit at the K stage
 *                 tp * stages / tiles_p of its range (tp: the unit's tile row)
 *                 and wraps around; 1: every unit reads its K range in order (or
 *                 backwards, "k_snake"); 0 (default): 2 for unsplit plans with
 *                 two MMA issuers (the skinny shapes), else 1.  The summation
 *                 order changes, not the accuracy; results stay deterministic
 *                 for a given shape
 *   "path"        0 auto (default), 1 force the CUDA-core kernel, 2 force the
 *                 tensor-core kernel's load-based producer (as for unaligned rows)
 *   "timeout_ns"  device wait limit in ns, 1e6..6e10 (default 2e9).  The longest
 *                 wait lasts one tile's whole K loop (one K piece when K is split),
 *                 so calls with K in the hundreds of millions and no split-K need
 *                 a larger limit
 *   "max_ctas"    cap on persistent CTAs, 0 = one per SM (default)
 *   "tile_q"      output tile width along M (= MMA N): 0 auto (default, by
 *                 padding cost; 16 or 32 when all of M fits in one such tile and
 *                 single-CTA tiles run), or 16, 32, 64, 128, 192, 256 (16 and 32
 *                 only apply when M fits in one tile and CTAs do not pair; else 64)
 *   "half"        64-row tiles: 0 or 2 never (default); 1 one CTA per 64 rows of N
 *                 (MMA M = 64) wherever single-CTA TMA tiles with FP32 accumulation
 *                 run; 3 CTA pairs of 64-row halves (128 rows of N per pair, MMA
 *                 M = 128 over the pair, tile width along M: "tile_q" when that is
 *                 128, 192 or 256, else M rounded up to a multiple of 32, from 160
 *                 to 256, and 128 for M <= 128) wherever TMA tiles with FP32
 *                 accumulation run.  They never split K
 *   "issuers"     MMA-issuing warps per CTA, taking alternate K stages into
 *                 accumulators of their own that the epilogue adds: 0 auto (default: two
 *                 for one-CTA TMA tiles of at most 64 columns that run unsplit in one
 *                 wave, and for pairs of 64-row halves), 1 always one, 2 two wherever
 *                 one-CTA TMA tiles of at most 128 columns run unsplit
 *   "atoms"       K depth of a ring stage in 128-byte swizzle spans: 0 auto
 *                 (default), 1, or 2 (twice the K per stage and per MMA commit, half
 *                 as many stages; TMA tiles only, and not pairs of 64-row halves
 *                 wider than 128 columns, which keep 1)
 *   "tail"        the last, partial wave of tiles: 0 auto (default) cuts its tiles
 *                 into 2 or 4 narrower ones when that ends it sooner, 1 never, 2 or
 *                 4 always
 *   "l2_hints"    L2 eviction hints on the TMA loads: 0 none (default), 1 keep the
 *                 band-reused A panels and drop the B panels first, 2 keep A only
 *                 (measured on GB300: 1 raises DRAM reads by half and loses 3-5 %,
 *                 2 changes nothing measurable)
 *   "repack"      0 (default): with a workspace, operands whose rows are not 16-byte
 *                 aligned (or, for compute-heavy shapes, not 128-byte aligned) are
 *                 first copied into it with 128-byte-aligned rows; 1 never
 *   "tail_k"      0 (default), or 2..8: with a workspace, cut the last partial wave's
 *                 tiles into that many K pieces instead of narrower tiles.  With 0
 *                 and "tail" 0 the library takes two pieces by itself when the
 *                 tiles have at least 192 K stages (K >= 12288 for 16-bit inputs,
 *                 24576 for e4m3) and the doubled tail still fits in one wave
 *   "f32_ktail"   gemm_f32 only, for tests: 0 (default), or 1..15: the last that
 *                 many terms of K (when K is larger) run in the chain-continuing
 *                 kernel that otherwise takes only the terms past 2^31 - 16
 *   "f32_tail"    gemm_f32 only: 0 (default) runs the last partial wave of 128 x 128 tiles
 *                 as 128 x 64 halves where that shortens it, in a second grid started
 *                 early by programmatic dependent launch; 1 keeps whole tiles; 2 is 0
 *                 with a plain second launch; 3 halves the last partial wave whatever
 *                 its size.  Results are bit-identical in every mode.
 *   "splits"      K pieces per tile: 0 auto (default, needs a workspace), 1 never
 *                 split, 2..64 split that many ways when the workspace suffices
 * Returns GEMM_OK or GEMM_ERR_INVALID_OPTION.
 */
int gemm_set_option(const char* name, int64_t value);

/*
 * gemm_set_workspace -- registers caller-owned device scratch for the current
 * device (ptr 256-byte aligned, `bytes` long; NULL, 0 unregisters).  With a
 * workspace registered, a TN call whose A or B rows are not 16-byte aligned
 * first copies that operand into the workspace with 128-byte-aligned rows
 * (when it fits: rows * K * element size, rounded up), so that the TMA path
 * can run; rows that are 16-byte but not 128-byte aligned are copied too when
 * MN / (M + N) >= 1100 x element size, where the copy costs less than the
 * slower loads would;
 * and TN calls whose output tiles cannot fill the GPU in one wave split K: each K piece writes its FP32 partial tile to the workspace and
 * the last piece to finish a 32-row slice sums the pieces in piece order (so
 * the result does not depend on timing) and stores C.  gemm_f32_bf16x6 writes
 * its split operands there (and needs them to fit).  The first 128 KiB of a
 * workspace of at least that size hold the split counters: registration
 * zeroes them (a synchronous cudaMemset followed by cudaDeviceSynchronize),
 * and every split launch zeroes the set the next one uses, so no split call
 * needs a memset of its own; after a call that ran into GEMM_ERR_TIMEOUT,
 * register the workspace again before replaying a captured CUDA graph that
 * splits K.  Calls that use the workspace on the same device share it, so they must not overlap in time
 * (issue them on one stream, or register a workspace per device and stream
 * order them).  The library never frees or reallocates the buffer.  Option
 * "splits" (gemm_set_option) forces or disables splitting.  Returns GEMM_OK,
 * GEMM_ERR_MISALIGNED, GEMM_ERR_INVALID_DIM, or GEMM_ERR_LAUNCH if zeroing the
 * counters fails.
 */
int gemm_set_workspace(void* ptr, int64_t bytes);

/* Workspace bytes that suffice for any M x N x K TN call under the automatic
 * rules: the split counters, aligned copies of A and B, and the largest split
 * those rules choose (16 K pieces of the narrowest tiles).  A split forced with
 * option "splits" that does not fit in the registered workspace runs unsplit.
 * 0 when M, N or K is not in [1, 2^31 - 1]; sizes that no device could hold
 * saturate at INT64_MAX / 4. */
int64_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * gemm_bf16_tn_noalloc -- gemm_bf16_tn with split-K scratch taken from a fixed
 * array inside the library instead of caller memory, so the call allocates
 * nothing and needs no registered workspace.  (The pages have no counterpart:
 * this entry point exists for callers that may not call cudaMalloc -- code
 * whose device memory belongs to a pooled allocator it must not bypass,
 * plugins whose host forbids device allocation, latency-critical loops where
 * an allocation would synchronise the device.)
 *
 * Arguments and layouts are those of gemm_bf16_tn, plus `splits`: 0 splits K
 * by the automatic rule (only when the output tiles cannot fill the GPU), 1
 * never splits, 2..64 forces that many K pieces.  The array holds
 * GEMM_NOALLOC_SCRATCH_BYTES (24 MiB) on every GPU that loads the library,
 * until the library is unloaded.  It serves, in this order, the copies of an
 * operand whose rows TMA cannot address (or, for compute-heavy shapes, whose
 * rows are not 128-byte aligned), as gemm_set_workspace describes, and the
 * split's partial sums.  With splits = 0 the split takes as many K pieces as
 * fit in what the copies leave (none: the call runs unsplit), so it never
 * fails for lack of room.  A forced split that does not fit beside the copies
 * runs without them (the operand is then read in place, more slowly); one
 * that does not fit the array on its own returns GEMM_ERR_SCRATCH without
 * launching anything.  The first call on a device looks up the
 * array's device address (cudaGetSymbolAddress) with that device current; make
 * that first call before any stream capture.  All calls share the array and it
 * keeps the last call's contents; its first 128 KiB hold the split counters
 * (zero at load, and each split launch zeroes the set the next one uses), the
 * rest the partial sums.  Calls that overlap in time on the GPU race.
 */
#define GEMM_NOALLOC_SCRATCH_BYTES (24LL << 20)
int gemm_bf16_tn_noalloc(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                         const void* B, int64_t ldb, void* C, int64_t ldc, int64_t splits,
                         void* stream);

/*
 * gemm_tile_coord -- the persistent kernels' tile rasteriser, exported for
 * tests (host only, no GPU needed).  Maps work index t in [0, tiles_m*tiles_n)
 * to an output tile (tm, tn): tiles are handed out in groups of `group` tile
 * rows, walking down the rows of a group before moving to the next tile column;
 * the last group is short when group does not divide tiles_m ("FP16 GEMM
 * Optimization on AMD RDNA 3 and RDNA 4", "Step 6: Block Scheduling for Cache
 * Reuse").  With snake != 0 the odd groups walk the tile columns from the last
 * to the first (the tensor-core kernel's order under option "band_snake" = 1,
 * the default), so each group starts on the columns the previous one ended on.
 * Returns GEMM_OK, or GEMM_ERR_INVALID_DIM for an index out of range.
 */
int gemm_tile_coord(int64_t t, int64_t tiles_m, int64_t tiles_n, int64_t group, int snake,
                    int64_t* tm, int64_t* tn);

/*
 * gemm_watchdog_selftest -- launches one block that waits on a shared-memory
 * barrier nothing will ever complete, with the given limit (ns, 1e5..1e10),
 * so that the wait runs out.  The kernel then records GEMM_ERR_TIMEOUT in the
 * watchdog word and exits; read it with gemm_read_watchdog.  For tests of the
 * timeout machinery only.
 */
int gemm_watchdog_selftest(int64_t limit_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DENSE_GEMM_TCGEN05_GB300_GEMM_H */
