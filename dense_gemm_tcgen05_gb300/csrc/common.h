// common.h -- the tensor-core kernel's parameter block and launch interface,
// shared by the kernel and the host code that launches it.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace gb300 {

enum class InKind : int { F16 = 0, BF16 = 1, E4M3 = 2 };

// Watchdog status bits recorded by kernels whose bounded waits ran out, or
// that refused launch parameters breaking one of their invariants.
constexpr unsigned int kWatchTimeout = 1u;
constexpr unsigned int kWatchBadParams = 2u;

// Parameters of the persistent tensor-core kernel.  "P" is the operand whose
// rows become TMEM lanes (the API's B, rows n), "Q" the operand whose rows
// become accumulator columns (the API's A, rows m).  The kernel computes
// D[i][j] = sum_k P[i][k] * Q[j][k] and stores D row-major, which is exactly
// the column-major C of the TN layout.
struct TcParams {
    int32_t rows_p;      // N
    int32_t rows_q;      // M
    int32_t num_kb;      // K stages per tile: ceil(K / stage depth)
    int32_t tiles_p;     // tiles along P
    int32_t tiles_q;     // tiles along Q (the grouped dimension)
    int32_t group;       // rasteriser group size, in tiles along Q
    float scale;         // epilogue scale (FP8 per-tensor scales; 1 otherwise)
    uint64_t timeout_ns; // limit for every wait
    unsigned int* watchdog;
    void* out;           // D (= C) base pointer, for the ragged-edge stores
    int64_t ld_out;      // D row pitch in elements (= ldc)
    int32_t direct_store;  // 1: no TMA map for D; the epilogue stores rows itself
    int64_t k_bytes;       // K * element size (row length of P and Q in bytes)
    const void* p_ptr;     // P (= B) base, for the non-TMA producer
    const void* q_ptr;     // Q (= A) base, for the non-TMA producer
    int64_t ld_p_bytes;    // row pitch of P in bytes (= ldb * element size)
    int64_t ld_q_bytes;    // row pitch of Q in bytes (= lda * element size)
    // Split-K: each tile's K range is cut into `splits` pieces of kb_per_split
    // stages; work unit u is tile u / splits, piece u % splits.  With splits > 1
    // every piece writes its FP32 partial to ws_partials and the last piece to
    // finish a 32-row slice (counted in ws_counters) sums them and stores C.
    int32_t splits;
    int32_t kb_per_split;
    float* ws_partials;
    unsigned int* ws_counters;
    // The other of the two fixed counter sets, which this launch zeroes for
    // the next split launch (nullptr when the counters were zeroed on the
    // host instead), and its length in words (a multiple of 4).
    unsigned int* ws_clear;
    int32_t clear_words;
    // Q rows per tile = N of the MMA instruction (64, 128, 192 or 256), chosen
    // per shape; the instruction descriptor and the per-stage TMA byte count
    // follow from it.
    int32_t tile_q;
    uint32_t idesc;
    uint32_t stage_tx_bytes;
    // Tail splitting: the first full_units units are whole tiles (times K
    // pieces); the remaining tiles of the last, partial wave are cut into
    // tail_f narrower units of tile_q / tail_f rows of Q each, loaded through
    // the tail tensor map with their own instruction descriptor and stage bytes.
    int64_t full_units;
    int32_t tail_f;
    uint32_t idesc_tail;
    uint32_t stage_tx_tail;
    // 1: the tail tiles keep their width and are cut into tail_f K pieces of
    // tail_kb_per stages instead, combined through the split-K workspace.
    int32_t tail_ksplit;
    int32_t tail_kb_per;
    // 1: the tensor core accumulates in FP16 (fp16 inputs and output); each
    // accumulator column then holds the final FP16 code in its low half.
    int32_t acc16;
    // TMA L2 hints: 0 none, 1 Q panels (reused by every tile of a rasteriser
    // band) evict last and P panels evict first, 2 Q panels evict last only.
    int32_t l2_hints;
    // Shared-memory ring: `stages` stages of `stage_bytes` (P tile then Q
    // tile, a multiple of 1024) in the kernel's fixed stage region.
    int32_t stages;
    uint32_t stage_bytes;
    // 1: the TMA producer walks the K range of every second unit a CTA runs
    // backwards, so that the K slices a wave of tiles ends on are the ones the
    // next wave starts with, while they are still in L2.
    int32_t k_snake;
    // 1: odd rasteriser bands walk the tile columns backwards (raster.h).
    int32_t band_snake;
    // 1: the TMA producer starts each unit's K range at a stage of its own,
    // spaced over the range by the unit's tile row (tp * stages / tiles_p),
    // and wraps around, so that concurrent units do not read the same K
    // offset at the same time (the MMA warp sums stages in any order).
    int32_t k_rotate;
    // K atoms (128-byte swizzle spans of K) per ring stage, 1 or 2, which
    // selects the kernel instantiation: a stage of two holds P atom 0, P atom
    // 1, Q atom 0, Q atom 1 (each atom of Q q_atom_bytes long, the full tile
    // width), and the MMA warp issues all of a stage's MMAs before one
    // commit.  The load-based producer takes 1.
    int32_t atoms;
    uint32_t q_atom_bytes;
    // 1: the ring extends over the epilogue's staging area.  Only for launches
    // in which every CTA (or pair) runs at most one unit: its epilogue then
    // starts after the ring has drained (the accumulator-full barrier waits
    // for every MMA, and every load was consumed by one).  The kernel checks
    // the unit count and refuses the launch otherwise.
    int32_t ring_epi;
};

struct TcLaunch {
    CUtensorMap map_p, map_q, map_out, map_q_tail;
    TcParams prm;
    int grid;
    cudaStream_t stream;
    bool half;  // 64-row tiles (one CTA, MMA M = 64; or pair halves, MMA M = 128)
    int issuers;  // MMA-issuing warps: 1, 2 or 4 (several: TMA, unsplit)
};

// Tile geometry of one persistent CTA (or CTA pair), for the host's grid sizing.
struct TcGeometry {
    int tile_p;            // P rows of the output tile of one CTA (or CTA pair)
    int max_tile_q;        // largest Q tile (MMA N)
    int load_p;            // P rows each CTA loads per stage
    int stage_k;           // K elements per stage
    int cluster;           // CTAs per tile
    int mma_m;             // M of the MMA instruction
    uint32_t format;       // A/B format code of the instruction descriptor
    int stage_region;      // shared-memory bytes for the stage ring
    int max_stages;        // barrier slots
    int epi_region;        // the epilogue's staging bytes, right after the ring
};

// Operand producer of the tensor-core kernel: TMA tensor copies, or (for rows
// TMA cannot address) producer warps using 16-byte-aligned loads.
enum class Producer : int { Tma = 0, Loads = 1 };

// half: one CTA per 64-row tile (MMA M = 64).
TcGeometry tc_geometry(InKind in, bool pair, bool half = false);
// out_f32: FP32 output (E4M3 or BF16 inputs); otherwise the input's 16-bit
// type (bf16 for E4M3).
cudaError_t tc_launch(InKind in, bool pair, Producer prod, bool out_f32, const TcLaunch& L);

}  // namespace gb300
