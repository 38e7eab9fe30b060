// tc_gemm.cuh -- persistent, warp-specialised tcgen05 GEMM for sm_103a.
//
// Computes D[i][j] = sum_k P[i][k] * Q[j][k] (both operands K-major) with FP32
// accumulators in tensor memory and stores D row-major.  With P = B (rows n)
// and Q = A (rows m) this is the TN product C = A x B with C column-major
// ("FP16 GEMM Optimization on AMD RDNA 3 and RDNA 4", "What We Are
// Computing"), so the epilogue's contiguous dimension is C's leading one.
//
// Structure (one CTA per SM, or one CTA pair per two SMs with cta_group::2):
//   producer    fills a ring of kStages shared-memory stages with 128-byte-
//               swizzled tiles of P and Q; each stage is one 128-byte swizzle
//               atom deep in K (64 fp16/bf16 or 128 e4m3 values).
//                 Tma:   warp 0, one lane issues 2D TMA copies; rows and K
//                        columns outside the matrix are zero-filled by TMA,
//                        which is what makes ragged M, N and K work.
//                 Loads: warps 6-17 (for rows TMA cannot address, i.e. rows
//                        not 16-byte aligned): each thread loads a row's
//                        window as nine aligned 16-byte chunks, funnel-shifts
//                        it into place, zeroes what lies outside the matrix and
//                        writes it to the swizzled stage.
//   warp 1      allocates tensor memory; one lane issues tcgen05.mma (4 per
//               stage) and releases each stage with tcgen05.commit as soon as
//               its MMAs are issued.
//   warps 2-5   epilogue: tcgen05.ld of the accumulator, conversion (and FP8
//               scaling) in registers, swizzled shared-memory staging, then a
//               TMA store (or, when D's rows are not 16-byte aligned, row-wise
//               coalesced stores).  Two accumulators (2 x 256 TMEM columns) let
//               the epilogue of one tile overlap the main loop of the next.
// Tiles are visited in the grouped order of raster.h.
//
// Correspondence with the pages' ladders: the staged shared-memory pipeline
// stands in for "Step 2: Tiling for Reuse and a Software Pipeline"; TMA's
// swizzle replaces LDS padding ("Step 3: Avoiding LDS Bank Conflicts"); TMA's
// zero fill replaces buffer resource descriptors ("Step 4"); one swizzle atom
// of K per stage, and twice as many FP8 values per stage, follow "Step 5:
// Trading Tile Area for K Depth" and the FP8 page's deeper-K configurations;
// the mbarrier handshakes follow the Helios ladder's asynchronous loads and
// split barriers (Levels 2 and 8), and the staged epilogue its Level 10.
//
// Every wait is bounded (see warp_wait): when a limit runs out the kernel
// records a timeout in the watchdog word, all roles leave their loops, and the
// CTA waits for its own copies and MMAs before freeing tensor memory.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.h"
#include "ptx.cuh"
#include "raster.h"

namespace gb300 {

// HALF: 64 P rows per CTA; used for unsplit TMA launches only.
//   one CTA (MMA M = 64): accumulator row 16 q + i sits in TMEM lane 32 q + i
//     (i < 16), so each epilogue warp owns 16 rows;
//   a CTA pair (MMA M = 128, cta_group::2): each CTA holds its 64 rows for all
//     N columns of the MMA, row r and column n in lane r + 64 (n / (N / 2)),
//     column n % (N / 2) (measured on GB300 with an in-bounds probe), so each
//     epilogue warp owns 32 rows of one half of the columns.
// NI: MMA-issuing warps (1 or 2: warp 1, then warp 6).  Issuer j takes
// the K stages s of each unit with s % NI == j into an accumulator of its own
// (j * tile_q columns after the first, tile_q / 2 for a pair of halves), and
// the epilogue adds them.  tcgen05.mma instructions from one issuing thread
// that commits after every stage complete one at a time, so small MMAs (narrow
// tiles) are limited by the issue rate; measured on GB300 (one CTA, MMA N = 64,
// a commit every 4 MMAs) one issuer completes an MMA every ~250 cycles, two
// issuers one every ~126.  Needs NI accumulators in one 256-column buffer;
// one CTA, TMA, unsplit (or a pair of halves).
template <InKind IN, bool PAIR, bool LOADS, bool HALF = false, int NI = 1>
struct TcCfg {
    static_assert(!(PAIR && LOADS), "the load-based producer runs one CTA per tile");
    static_assert(!(HALF && LOADS), "64-row tiles: TMA producer");
    static_assert(NI == 1 || NI == 2, "one or two MMA issuers");
    static_assert(NI == 1 || (!LOADS && PAIR == HALF),
                  "several issuers: TMA; one CTA with 128-row tiles, or a pair of 64-row halves");
    static constexpr int kCG = PAIR ? 2 : 1;
    static constexpr int kElemBytes = IN == InKind::E4M3 ? 1 : 2;
    static constexpr int kBlockP = HALF ? 64 : 128;  // accumulator rows per CTA
    static constexpr int kMmaM = kBlockP * kCG;      // M of one MMA instruction
    static constexpr int kMmaN = 256;                // N of one MMA instruction
    static constexpr int kTileP = kMmaM;             // P rows per tile (per pair)
    static constexpr int kMaxLoadQ = kMmaN / (PAIR ? 2 : 1);  // Q rows a CTA loads, at most
    static constexpr int kAtomBytes = 128;           // K bytes per stage row
    static constexpr int kStageK = kAtomBytes / kElemBytes;
    static constexpr int kMmaKBytes = 32;            // K bytes per MMA (16 x 16-bit, 32 x 8-bit)
    static constexpr int kMmasPerStage = kAtomBytes / kMmaKBytes;
    static constexpr int kBytesP = kBlockP * kAtomBytes;
    static constexpr int kBytesQ = kMaxLoadQ * kAtomBytes;
    static constexpr int kStageBytes = kBytesP + kBytesQ;    // widest stage
    static constexpr int kStages = PAIR ? 6 : 4;              // widest stages that fit
    static constexpr int kStageRegion = 192 * 1024;
    static_assert(kStages * kStageBytes <= kStageRegion, "widest stages fit the ring");
    static constexpr int kMaxStages = 20;  // narrow tiles: more, smaller stages in the region
    static constexpr int kEpiWarps = 4;
    // accumulator rows per epilogue warp (a pair of 64-row halves: 32 rows of
    // one half of the columns)
    static constexpr int kRowsPerWarp = (PAIR && HALF) ? 32 : kBlockP / kEpiWarps;
    static constexpr bool kColHalves = PAIR && HALF;
    static constexpr int kEpiBufBytes = 32 * 128;            // 32 rows x one 128-byte row
    static constexpr int kEpiBytes = kEpiWarps * 2 * kEpiBufBytes;
    static constexpr int kFirstLoadWarp = 6;
    static constexpr int kLoadWarps = 12;
    static constexpr int kExtraIssuerWarp = 6;  // issuer 1: warp 6
    static constexpr int kThreads = LOADS ? (kFirstLoadWarp + kLoadWarps) * 32 : 192 + (NI - 1) * 32;
    static constexpr int kFullArrivals = LOADS ? kLoadWarps : 1;
    static constexpr int kAccCols = kMmaN;
    static constexpr int kTmemCols = 512;
    static constexpr int kNumBars = 2 * kMaxStages + 4 + 1;
    static constexpr int kOffEpi = kStageRegion;  // a ring with ring_epi runs on into it
    static constexpr int kOffBars = kOffEpi + kEpiBytes;
    static constexpr int kOffTmemSlot = kOffBars + kNumBars * 8;
    static constexpr int kOffAbort = kOffTmemSlot + 4;
    static constexpr int kSmemBytes = kOffAbort + 4 + 1024;  // + alignment slack
    static constexpr uint32_t kFormat = IN == InKind::BF16 ? 1u : 0u;
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(kStageBytes % 1024 == 0 && kBytesP % 1024 == 0, "1024-byte stage alignment");
    static_assert(PAIR || HALF || kLoadWarps * 32 == kBlockP + kMaxLoadQ,
                  "load-producer row split");
};

// Bounded-wait bookkeeping shared by a CTA's warps.
struct Watch {
    volatile int* abort_flag;   // shared memory: set when any warp gives up
    unsigned int* word;         // global watchdog word read by the host
    uint64_t limit_ns;
};

// Warp-collective wait for barrier phase `parity`.  Returns false (on every
// lane) when the CTA is aborting or this wait exceeded the limit; in the latter
// case the abort flag and the watchdog word are set.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const Watch& w) {
    uint64_t t0 = 0;
    for (uint32_t spin = 1;; ++spin) {
        const bool ok = mbar_try_wait(bar, parity);
        if (__all_sync(0xffffffffu, ok)) return true;
        if ((spin & 63u) == 0) {
            int give_up = 0;
            if (lane_idx() == 0) {
                if (*w.abort_flag) {
                    give_up = 1;
                } else {
                    const uint64_t now = global_timer_ns();
                    if (t0 == 0) {
                        t0 = now;
                    } else if (now - t0 > w.limit_ns) {
                        *w.abort_flag = 1;
                        atomicOr(w.word, kWatchTimeout);
                        give_up = 1;
                    }
                }
            }
            if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
        }
    }
}

// Bounded pause used on the abort path only.
__device__ __forceinline__ void pause_ns(uint64_t ns) {
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < ns) {
    }
}

template <int CG>
__device__ __forceinline__ void commit_to(uint32_t bar, uint16_t mask) {
    if constexpr (CG == 1)
        tc_commit(bar);
    else
        tc_commit_pair(bar, mask);
}

template <typename OutT>
__device__ __forceinline__ uint32_t pack2(float lo, float hi);

template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

template <>
__device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// ------------------------------------------------- load-based producer
//
// For rows that are not 16-byte aligned.  Work unit: a "quad" of four stage
// rows whose addresses agree modulo 16 (rows kPeriod = 16 / element-size apart:
// the row pitch times kPeriod is a multiple of 16 bytes), so the whole warp
// shares one misalignment delta.  Lanes 8s..8s+7 own row s of the quad and
// 16-byte chunk c = lane % 8 of its 128-byte K window: each lane loads the two
// aligned 16-byte chunks that cover its chunk (consecutive lanes read
// consecutive addresses), funnel-shifts them by delta, zeroes bytes outside
// the matrix and stores the chunk at its 128-byte-swizzle position.  Only
// aligned chunks holding at least one byte of the row inside the matrix are
// loaded, so no load leaves the 16-byte blocks the matrix occupies.

__device__ __forceinline__ uint4 shift_chunk(uint4 lo, uint4 hi, uint32_t delta) {
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    const uint32_t sh = (delta & 3u) * 8u;
    uint4 o;
    switch (delta >> 2) {  // uniform across the warp: all rows of a quad share delta
        case 0:
            o = make_uint4(__funnelshift_r(w[0], w[1], sh), __funnelshift_r(w[1], w[2], sh),
                           __funnelshift_r(w[2], w[3], sh), __funnelshift_r(w[3], w[4], sh));
            break;
        case 1:
            o = make_uint4(__funnelshift_r(w[1], w[2], sh), __funnelshift_r(w[2], w[3], sh),
                           __funnelshift_r(w[3], w[4], sh), __funnelshift_r(w[4], w[5], sh));
            break;
        case 2:
            o = make_uint4(__funnelshift_r(w[2], w[3], sh), __funnelshift_r(w[3], w[4], sh),
                           __funnelshift_r(w[4], w[5], sh), __funnelshift_r(w[5], w[6], sh));
            break;
        default:
            o = make_uint4(__funnelshift_r(w[3], w[4], sh), __funnelshift_r(w[4], w[5], sh),
                           __funnelshift_r(w[5], w[6], sh), __funnelshift_r(w[6], w[7], sh));
            break;
    }
    return o;
}

// Keeps bytes [0, lim) of a 16-byte chunk and zeroes the rest.
__device__ __forceinline__ uint4 mask_chunk(uint4 v, int32_t lim) {
    auto m = [](int32_t l) -> uint32_t {
        return l >= 4 ? 0xFFFFFFFFu : (l <= 0 ? 0u : ((1u << (8 * l)) - 1u));
    };
    v.x &= m(lim);
    v.y &= m(lim - 4);
    v.z &= m(lim - 8);
    v.w &= m(lim - 12);
    return v;
}

// ------------------------------------------------------------------ kernel

// SPLIT: the launch cuts tiles into K pieces (split-K or a K-split tail) and
// combines them through the workspace.  Launches without K pieces run the
// instantiation without that code.
template <InKind IN, typename OutT, bool PAIR, bool LOADS, bool SPLIT, bool HALF, int NI = 1,
          int AT = 1>
__global__ void __launch_bounds__(TcCfg<IN, PAIR, LOADS, HALF, NI>::kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap map_p,
                   const __grid_constant__ CUtensorMap map_q,
                   const __grid_constant__ CUtensorMap map_out,
                   const __grid_constant__ CUtensorMap map_q_tail, const TcParams prm) {
    using Cfg = TcCfg<IN, PAIR, LOADS, HALF, NI>;
    static_assert(!(SPLIT && HALF), "64-row tiles never split K");
    static_assert(!(SPLIT && NI > 1), "several issuers: unsplit launches only");
    constexpr int SM = Cfg::kMaxStages;                 // barrier slots
    const uint32_t S = static_cast<uint32_t>(prm.stages);  // ring depth for this call
    const uint32_t stage_bytes = prm.stage_bytes;
    static_assert(AT == 1 || (AT == 2 && !LOADS), "two K atoms per stage: TMA producer only");
    constexpr int32_t atoms = AT;                          // K atoms per stage

    // A ring over the epilogue's staging area (ring_epi) needs every CTA (or
    // pair) to run at most one unit; the planner only asks for it then.  The
    // check is uniform over the grid, so all CTAs leave together, before any
    // barrier, tensor-memory or cluster operation.
    if (prm.ring_epi) {
        const int64_t tiles = static_cast<int64_t>(prm.tiles_p) * prm.tiles_q;
        const int64_t units = prm.full_units + (tiles - prm.full_units / prm.splits) * prm.tail_f;
        const int64_t slots = PAIR ? gridDim.x / 2 : gridDim.x;
        if (LOADS || units > slots ||
            static_cast<int64_t>(prm.stages) * prm.stage_bytes >
                static_cast<int64_t>(TcCfg<IN, PAIR, LOADS, HALF, NI>::kOffBars)) {
            if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(prm.watchdog, kWatchBadParams);
            return;
        }
    }
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);

    const uint32_t warp = warp_idx();
    const uint32_t lane = lane_idx();
    const uint32_t bars = base + Cfg::kOffBars;
    auto full_bar = [&](uint32_t s) { return bars + 8u * s; };
    auto empty_bar = [&](uint32_t s) { return bars + 8u * (SM + s); };
    auto accf_bar = [&](uint32_t b) { return bars + 8u * (2 * SM + b); };
    auto acce_bar = [&](uint32_t b) { return bars + 8u * (2 * SM + 2 + b); };
    const uint32_t done_bar = bars + 8u * (2 * SM + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + Cfg::kOffTmemSlot);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + Cfg::kOffAbort);

    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;
    // TMEM columns between the accumulators of consecutive issuers (NI > 1):
    // tile_q (tile_q / 2 for a pair of halves).
    const uint32_t kAcc2Off = static_cast<uint32_t>(PAIR ? prm.tile_q / 2 : prm.tile_q);

    if (threadIdx.x == 0) {
        for (int s = 0; s < SM; ++s) {
            mbar_init(full_bar(s), Cfg::kFullArrivals);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), NI);   // one commit per issuer
            mbar_init(acce_bar(b), (PAIR ? 2 : 1) * Cfg::kEpiWarps);
        }
        mbar_init(done_bar, NI);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        if (!LOADS) {
            prefetch_tensormap(&map_p);
            prefetch_tensormap(&map_q);
            if (prm.tail_f > 1) prefetch_tensormap(&map_q_tail);
        }
        if (!prm.direct_store) prefetch_tensormap(&map_out);
    }
    if (warp == 1) {
        tmem_alloc<Cfg::kCG>(smem_u32(tmem_slot), Cfg::kTmemCols);
        tmem_relinquish<Cfg::kCG>();
    }
    tc_fence_before_sync();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();
    tc_fence_after_sync();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

    const Watch wd{abort_flag, prm.watchdog, prm.timeout_ns};
    const int64_t num_tiles = static_cast<int64_t>(prm.tiles_p) * prm.tiles_q;
    // Work units: whole tiles times K pieces, then the tail tiles cut into
    // tail_f units each -- narrower along Q, or (tail_ksplit) K pieces.
    const int64_t full_tiles = prm.full_units / prm.splits;
    const int64_t num_units = prm.full_units + (num_tiles - full_tiles) * prm.tail_f;
    struct Unit {
        int64_t tile, tq, tp;
        int64_t ws_tile;  // the tile's slot in the split-K workspace
        int32_t q_off;    // first Q row (C column) of the unit
        int32_t width;    // Q rows of the unit = MMA N
        int32_t piece;    // K piece of the tile (0 unless split)
        int32_t pieces;   // K pieces of the tile
        int32_t kb_lo, kb_hi;
        bool narrow;      // narrow tail unit
    };
    auto unit_of = [&](int64_t u) {
        Unit w;
        int32_t part = 0, kb_per = prm.kb_per_split;
        if (u < prm.full_units) {
            w.tile = u / prm.splits;
            w.piece = static_cast<int32_t>(u % prm.splits);
            w.pieces = prm.splits;
            w.ws_tile = w.tile;
            w.width = prm.tile_q;
            w.narrow = false;
        } else {
            const int64_t v = u - prm.full_units;
            w.tile = full_tiles + v / prm.tail_f;
            if (prm.tail_ksplit) {
                w.piece = static_cast<int32_t>(v % prm.tail_f);
                w.pieces = prm.tail_f;
                w.ws_tile = w.tile - full_tiles;
                w.width = prm.tile_q;
                w.narrow = false;
                kb_per = prm.tail_kb_per;
            } else {
                part = static_cast<int32_t>(v % prm.tail_f);
                w.piece = 0;
                w.pieces = 1;
                w.ws_tile = 0;
                w.width = prm.tile_q / prm.tail_f;
                w.narrow = true;
            }
        }
        raster_tile(w.tile, prm.tiles_q, prm.tiles_p, prm.group, &w.tq, &w.tp,
                    prm.band_snake != 0);
        w.q_off = static_cast<int32_t>(w.tq * prm.tile_q) + part * w.width;
        w.kb_lo = w.piece * kb_per;
        w.kb_hi = w.kb_lo + kb_per < prm.num_kb ? w.kb_lo + kb_per : prm.num_kb;
        return w;
    };
    const int64_t first = PAIR ? blockIdx.x / 2 : blockIdx.x;
    const int64_t stride = PAIR ? gridDim.x / 2 : gridDim.x;
    // The TMA producer's first unit (64-bit divisions, about half a microsecond
    // on a skinny launch's critical path), worked out from the parameters
    // alone before the wait below.
    Unit u_first{};
    if (warp == 0 && !LOADS && first < num_units) u_first = unit_of(first);

    // Launched with programmatic stream serialisation: everything above ran
    // while the previous grid in the stream may still be finishing; nothing
    // below may touch global memory before that grid is complete.  Only then
    // may the next grid be scheduled, so that grids waiting here never hold
    // SMs an earlier grid still needs.
    pdl_wait();
    pdl_trigger();

    if (warp == 0 && !LOADS) {
        // ------------------------------------------------ TMA producer
        uint32_t it = 0, rs = 0, rph = 0;   // stages issued; ring slot and phase
        bool ok = true;
        const uint64_t pol_p = l2_evict_first_policy();
        const uint64_t pol_q = l2_evict_last_policy();
        const bool hints = prm.l2_hints != 0;
        uint32_t lu = 0;                     // units this CTA has run
        // stage layout: P atoms, then Q atoms (q_atom bytes each)
        const uint32_t q_region = atoms > 1 ? 2u * Cfg::kBytesP : Cfg::kBytesP;
        const uint32_t q_atom = prm.q_atom_bytes;
        const int32_t stage_k = atoms > 1 ? 2 * Cfg::kStageK : Cfg::kStageK;
        for (int64_t u = first; ok && u < num_units; u += stride, ++lu) {
            const Unit w = u == first ? u_first : unit_of(u);
            // Every second unit reads its K range backwards (the MMA warp sums
            // the stages in whatever order they arrive).
            const bool k_rev = prm.k_snake && (lu & 1u);
            const int32_t nkb = w.kb_hi - w.kb_lo;
            const int32_t k_rot =
                prm.k_rotate && nkb > 1
                    ? static_cast<int32_t>(w.tp * static_cast<int64_t>(nkb) / prm.tiles_p % nkb)
                    : 0;
            const int32_t p0 = static_cast<int32_t>(w.tp * Cfg::kTileP + rank * Cfg::kBlockP);
            const int32_t q0 = w.q_off + static_cast<int32_t>(rank) * (w.width / Cfg::kCG);
            const CUtensorMap* mq = w.narrow ? &map_q_tail : &map_q;
            const uint32_t tx = w.narrow ? prm.stage_tx_tail : prm.stage_tx_bytes;
            for (int32_t kb = w.kb_lo; kb < w.kb_hi; ++kb, ++it) {
                const uint32_t s = rs, ph = rph;
                if (++rs == S) {
                    rs = 0;
                    rph ^= 1u;
                }
                if (!warp_wait(empty_bar(s), ph ^ 1u, wd)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const uint32_t sp = base + s * stage_bytes;
                    const uint32_t sq = sp + q_region;
                    int32_t ki = kb - w.kb_lo + k_rot;   // the unit's ki-th K stage
                    if (ki >= nkb) ki -= nkb;
                    const int32_t kx = (k_rev ? w.kb_hi - 1 - ki : w.kb_lo + ki) * stage_k;
                    if constexpr (PAIR) {
                        const uint32_t fb = mapa_shared(full_bar(s), 0);
                        if (leader) mbar_arrive_expect_tx(full_bar(s), 2 * tx);
                        if (hints) {
                            if (prm.l2_hints == 1)
                                tma_load_2d_pair_hint(sp, &map_p, fb, kx, p0, pol_p);
                            else
                                tma_load_2d_pair(sp, &map_p, fb, kx, p0);
                            tma_load_2d_pair_hint(sq, mq, fb, kx, q0, pol_q);
                        } else {
                            tma_load_2d_pair(sp, &map_p, fb, kx, p0);
                            tma_load_2d_pair(sq, mq, fb, kx, q0);
                        }
                        if (atoms > 1) {   // the stage's second K atom, behind the first
                            tma_load_2d_pair(sp + Cfg::kBytesP, &map_p, fb, kx + Cfg::kStageK, p0);
                            tma_load_2d_pair(sq + q_atom, mq, fb, kx + Cfg::kStageK, q0);
                        }
                    } else {
                        mbar_arrive_expect_tx(full_bar(s), tx);
                        if (hints) {
                            if (prm.l2_hints == 1)
                                tma_load_2d_hint(sp, &map_p, full_bar(s), kx, p0, pol_p);
                            else
                                tma_load_2d(sp, &map_p, full_bar(s), kx, p0);
                            tma_load_2d_hint(sq, mq, full_bar(s), kx, q0, pol_q);
                        } else {
                            tma_load_2d(sp, &map_p, full_bar(s), kx, p0);
                            tma_load_2d(sq, mq, full_bar(s), kx, q0);
                        }
                        if (atoms > 1) {
                            tma_load_2d(sp + Cfg::kBytesP, &map_p, full_bar(s), kx + Cfg::kStageK,
                                        p0);
                            tma_load_2d(sq + q_atom, mq, full_bar(s), kx + Cfg::kStageK, q0);
                        }
                    }
                }
                __syncwarp();
            }
        }
        if (!ok) {
            // Aborting: let this CTA's own copies still in flight land before
            // the CTA can exit.
            if constexpr (PAIR) {
                if (lane == 0) pause_ns(200000);
            } else {
                const uint32_t outstanding = it < static_cast<uint32_t>(S) ? it : S;
                for (uint32_t i = it - outstanding; i < it; ++i) {
                    const uint64_t t0 = global_timer_ns();
                    while (!__all_sync(0xffffffffu, mbar_try_wait(full_bar(i % S), (i / S) & 1u))) {
                        if (global_timer_ns() - t0 > prm.timeout_ns) break;
                    }
                }
            }
            __syncwarp();
        }
    } else if (LOADS && warp >= Cfg::kFirstLoadWarp) {
        // ------------------------------------------------ load-based producer
        // Producer warp pw owns quads 8pw .. 8pw+7 of the stage.  Quad i of the
        // warp is stage rows r0 + i + kPeriod * s (s = lane / 8), so the warp
        // stays within P (pw < 4) or within Q, row pointers advance by one
        // pitch per quad, and the swizzle row (r % 8) is i.
        constexpr int kPeriod = 16 / Cfg::kElemBytes;        // rows sharing one delta
        constexpr int kQuadsPerWarp = 8;
        static_assert(!LOADS || (Cfg::kBlockP + Cfg::kMaxLoadQ) / 4 == kQuadsPerWarp * Cfg::kLoadWarps,
                      "quad split");
        const uint32_t pw = warp - Cfg::kFirstLoadWarp;
        const uint32_t sub = lane >> 3, c = lane & 7u;
        const uint32_t qd0 = pw * kQuadsPerWarp;
        const uint32_t r0 = (qd0 / kPeriod) * (4 * kPeriod) + (qd0 % kPeriod) + kPeriod * sub;
        const bool is_p = r0 < static_cast<uint32_t>(Cfg::kBlockP);  // warp-uniform
        const uint8_t* mat = static_cast<const uint8_t*>(is_p ? prm.p_ptr : prm.q_ptr);
        const int64_t pitch = is_p ? prm.ld_p_bytes : prm.ld_q_bytes;
        const int64_t rows_lim = is_p ? prm.rows_p : prm.rows_q;
        const uint32_t srow0 = r0 * Cfg::kAtomBytes;  // P then Q are contiguous, 128 B a row
        uint32_t rs = 0, rph = 0;   // ring slot and phase
        bool ok = true;
        for (int64_t u = first; ok && u < num_units; u += stride) {
            const Unit w = unit_of(u);
            const int64_t g0 =
                is_p ? w.tp * Cfg::kTileP + r0 : static_cast<int64_t>(w.q_off) + (r0 - Cfg::kBlockP);
            const uint8_t* row0 = mat + g0 * pitch;   // address arithmetic only
            // quad i exists iff i < rows_left: inside the matrix and, for Q,
            // inside this unit's rows (the rest of the stage is unused)
            int64_t rows_left = rows_lim - g0;
            if (!is_p && w.width - static_cast<int64_t>(r0 - Cfg::kBlockP) < rows_left)
                rows_left = w.width - static_cast<int64_t>(r0 - Cfg::kBlockP);
            for (int32_t kb = w.kb_lo; kb < w.kb_hi; ++kb) {
                const uint32_t s = rs, ph = rph;
                if (++rs == S) {
                    rs = 0;
                    rph ^= 1u;
                }
                const int64_t kb_byte = static_cast<int64_t>(kb) * Cfg::kAtomBytes;
                const int64_t left = prm.k_bytes - kb_byte;
                const int32_t win = left > 128 ? 128 : static_cast<int32_t>(left);  // >= 1
                // Global loads first: they do not touch the stage being refilled.
                uint4 lo[kQuadsPerWarp], hi[kQuadsPerWarp];
#pragma unroll
                for (int i = 0; i < kQuadsPerWarp; ++i) {
                    const uintptr_t a = reinterpret_cast<uintptr_t>(row0) +
                                        static_cast<uintptr_t>(i * pitch + kb_byte);
                    const uint32_t delta = static_cast<uint32_t>(a & 15u);
                    const uintptr_t al = a - delta + 16u * c;
                    // Row bytes [0, v) are valid (v = 0 for a row outside the
                    // matrix or the unit).  A 16-byte chunk is read only when it
                    // starts inside them or, for lane 0 of a misaligned row,
                    // covers their first byte; a chunk that starts inside valid
                    // bytes never leaves their 16-byte granule, hence their page.
                    const int32_t v = i < rows_left ? win : 0;
                    const int32_t first16 = 16 * static_cast<int32_t>(c) - static_cast<int32_t>(delta);
                    lo[i] = make_uint4(0u, 0u, 0u, 0u);
                    hi[i] = make_uint4(0u, 0u, 0u, 0u);
                    if (v > 0 && first16 < v) lo[i] = ldg_nc_v4(reinterpret_cast<const void*>(al));
                    if (delta != 0 && first16 + 16 < v)
                        hi[i] = ldg_nc_v4(reinterpret_cast<const void*>(al + 16u));
                }
                if (!warp_wait(empty_bar(s), ph ^ 1u, wd)) {
                    ok = false;
                    break;
                }
                const uint32_t sp = base + s * stage_bytes + srow0;
#pragma unroll
                for (int i = 0; i < kQuadsPerWarp; ++i) {
                    const uintptr_t a = reinterpret_cast<uintptr_t>(row0) +
                                        static_cast<uintptr_t>(i * pitch + kb_byte);
                    uint4 o = shift_chunk(lo[i], hi[i], static_cast<uint32_t>(a & 15u));
                    const int32_t v = i < rows_left ? win : 0;
                    if (v < 128) o = mask_chunk(o, v - 16 * static_cast<int32_t>(c));
                    st_shared_v4(sp + i * Cfg::kAtomBytes + ((c ^ static_cast<uint32_t>(i)) << 4),
                                 o.x, o.y, o.z, o.w);
                }
                // generic-proxy writes -> visible to the tensor core's reads
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(full_bar(s));
            }
        }
    } else if (warp == 1 || (NI > 1 && warp >= Cfg::kExtraIssuerWarp &&
                             warp < Cfg::kExtraIssuerWarp + NI - 1)) {
        // ------------------------------------------------ MMA issuer
        // issuer j (NI > 1) takes the K stages s of each unit with s % NI == j
        // into the accumulator j * kAcc2Off columns after issuer 0's
        const uint32_t issuer = warp == 1 ? 0u : warp - (Cfg::kExtraIssuerWarp - 1);
        if (!PAIR || leader) {
            uint32_t lt = 0, rs = 0, rph = 0;   // tiles; ring slot and phase
            const uint64_t adesc0 = sdesc_kmajor_sw128(base);
            const uint64_t bdesc0 =
                sdesc_kmajor_sw128(base + (atoms > 1 ? 2u * Cfg::kBytesP : Cfg::kBytesP));
            // descriptor steps to a stage's second K atom (start address in
            // 16-byte units)
            const uint64_t a_atom = static_cast<uint64_t>(Cfg::kBytesP >> 4);
            const uint64_t b_atom = static_cast<uint64_t>(prm.q_atom_bytes >> 4);
            bool ok = true;
            for (int64_t u = first; ok && u < num_units; u += stride, ++lt) {
                const uint32_t b = lt & 1u, aph = (lt >> 1) & 1u;
                if (!warp_wait(acce_bar(b), aph ^ 1u, wd)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem =
                    tmem_base + b * Cfg::kAccCols + issuer * kAcc2Off;
                const Unit w = unit_of(u);
                const uint32_t idesc = w.narrow ? prm.idesc_tail : prm.idesc;
                const int32_t kb_lo = w.kb_lo;
                for (int32_t kb = w.kb_lo; kb < w.kb_hi; ++kb) {
                    const uint32_t s = rs, ph = rph;
                    if (++rs == S) {
                        rs = 0;
                        rph ^= 1u;
                    }
                    if constexpr (NI > 1) {
                        if (static_cast<uint32_t>((kb - kb_lo) % NI) != issuer) continue;
                    }
                    if (!warp_wait(full_bar(s), ph, wd)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    if (lane == 0) {
                        // descriptors of stage s: the ring's first ones advanced by
                        // s stages (start-address field counts 16-byte units)
                        const uint64_t soff = static_cast<uint64_t>(s * (stage_bytes >> 4));
                        const uint64_t adesc = adesc0 + soff;
                        const uint64_t bdesc = bdesc0 + soff;
#pragma unroll
                        for (int kk = 0; kk < Cfg::kMmasPerStage; ++kk) {
                            // advance the start address by 32 bytes of K per MMA
                            const uint64_t off = static_cast<uint64_t>(kk * (Cfg::kMmaKBytes >> 4));
                            uint32_t acc;
                            if constexpr (NI > 1)
                                acc = (kb - kb_lo > static_cast<int32_t>(issuer) || kk != 0) ? 1u : 0u;
                            else
                                acc = (kb != kb_lo || kk != 0) ? 1u : 0u;
                            if constexpr (IN == InKind::E4M3)
                                mma_f8<Cfg::kCG>(d_tmem, adesc + off, bdesc + off, idesc, acc);
                            else
                                mma_f16<Cfg::kCG>(d_tmem, adesc + off, bdesc + off, idesc, acc);
                        }
                        if (atoms > 1) {   // the second K atom: always accumulates
#pragma unroll
                            for (int kk = 0; kk < Cfg::kMmasPerStage; ++kk) {
                                const uint64_t off =
                                    static_cast<uint64_t>(kk * (Cfg::kMmaKBytes >> 4));
                                if constexpr (IN == InKind::E4M3)
                                    mma_f8<Cfg::kCG>(d_tmem, adesc + a_atom + off,
                                                     bdesc + b_atom + off, idesc, 1u);
                                else
                                    mma_f16<Cfg::kCG>(d_tmem, adesc + a_atom + off,
                                                      bdesc + b_atom + off, idesc, 1u);
                            }
                        }
                        commit_to<Cfg::kCG>(empty_bar(s), 0x3);
                    }
                    __syncwarp();
                }
                if (!ok) break;
                if (lane == 0) commit_to<Cfg::kCG>(accf_bar(b), 0x3);
                __syncwarp();
            }
            // Every MMA issued here must finish before tensor memory is freed.
            if (lane == 0) commit_to<Cfg::kCG>(done_bar, 0x1);
            __syncwarp();
            const uint64_t t0 = global_timer_ns();
            while (!__all_sync(0xffffffffu, mbar_try_wait(done_bar, 0))) {
                if (global_timer_ns() - t0 > prm.timeout_ns) {
                    if (lane == 0) atomicOr(prm.watchdog, kWatchTimeout);
                    break;
                }
            }
        }
    } else if (warp >= 2 && warp < 2 + Cfg::kEpiWarps) {
        // ------------------------------------------------ epilogue
        // A staged chunk is one 128-byte row per accumulator row: 64 fp16/bf16
        // or 32 fp32 output values.
        constexpr int kOB = static_cast<int>(sizeof(OutT));   // output bytes: 2 or 4
        constexpr int kCols = 128 / kOB;                        // columns per chunk
        constexpr int kGran = 16 / kOB;                         // elements per 16-byte granule
        constexpr int kSlices = (PAIR ? 2 : 1) * Cfg::kEpiWarps;  // 32-row slices per tile
        constexpr int kSliceFloats = 32 * Cfg::kAccCols;
        const uint32_t quarter = warp & 3u;     // TMEM lanes this warp may access
        const uint32_t ew = warp - 2u;          // staging buffers owned by this warp
        const uint32_t stage0 = base + Cfg::kOffEpi + ew * 2u * Cfg::kEpiBufBytes;
        const uint32_t slice = rank * Cfg::kEpiWarps + quarter;
        const float scale = prm.scale;
        uint8_t* const out8 = static_cast<uint8_t*>(prm.out);
        uint32_t lt = 0, chunk = 0;
        if constexpr (SPLIT) {
            // Zero the counter set the next split launch will use.  The last
            // launch that used it is complete (pdl_wait above); this launch
            // counts in the other set.
            if (blockIdx.x == 0 && prm.ws_clear) {
                uint4* clr = reinterpret_cast<uint4*>(prm.ws_clear);
                for (int32_t i = static_cast<int32_t>(threadIdx.x) - 64; i < prm.clear_words / 4;
                     i += 32 * Cfg::kEpiWarps)
                    clr[i] = make_uint4(0u, 0u, 0u, 0u);
            }
        }

        // Converts 32 words' worth of FP32 values (kCols of them) into this
        // lane's 128 output bytes.
        auto pack = [&](const float* f, uint32_t (&pk)[32]) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                if constexpr (kOB == 2) {
                    float lo = f[2 * j], hi = f[2 * j + 1];
                    if constexpr (IN == InKind::E4M3) {
                        lo *= scale;
                        hi *= scale;
                    }
                    pk[j] = pack2<OutT>(lo, hi);
                } else {
                    float v = f[j];
                    if constexpr (IN == InKind::E4M3) v *= scale;
                    pk[j] = __float_as_uint(v);
                }
            }
        };

        // Writes this warp's packed chunk: rows row0 + lane, columns [x, x + kCols)
        // that lie below xlim (min(M, end of the warp's columns): a pair of
        // halves 192 wide gives each warp 96 columns, so its second chunk ends
        // halfway, where the other half's columns begin).
        auto emit = [&](const uint32_t (&pk)[32], int32_t x, int32_t row0, int32_t xlim) {
            const bool in_range = x < xlim && row0 < prm.rows_p;
            const uint32_t buf = stage0 + (chunk & 1u) * Cfg::kEpiBufBytes;
            ++chunk;
            if (!prm.direct_store && in_range && x + kCols > xlim &&
                (xlim < prm.rows_q || (prm.rows_q % kGran) != 0)) {
                // A TMA store writes the whole box up to M, and whole 16-byte
                // granules of the contiguous dimension, so a chunk cut short
                // by xlim, or one that ends inside a granule (it would spill into
                // the caller's padding between M and ld_out), is stored by the
                // lanes: whole granules where they are aligned, the rest element
                // by element.
                const int32_t r = row0 + static_cast<int32_t>(lane);
                if (static_cast<int>(lane) < Cfg::kRowsPerWarp && r < prm.rows_p) {
                    uint8_t* dst = out8 + (static_cast<int64_t>(r) * prm.ld_out + x) * kOB;
                    const int32_t ncols = xlim - x;
                    const bool al16 = (reinterpret_cast<uintptr_t>(dst) & 15u) == 0;
#pragma unroll
                    for (int gi = 0; gi < 8; ++gi) {
                        if (al16 && (gi + 1) * kGran <= ncols) {
                            *reinterpret_cast<uint4*>(dst + 16 * gi) =
                                make_uint4(pk[4 * gi], pk[4 * gi + 1], pk[4 * gi + 2], pk[4 * gi + 3]);
                            continue;
                        }
#pragma unroll
                        for (int j = 4 * gi; j < 4 * gi + 4; ++j) {
                            if constexpr (kOB == 2) {
                                uint16_t* d16 = reinterpret_cast<uint16_t*>(dst);
                                if (2 * j < ncols) d16[2 * j] = static_cast<uint16_t>(pk[j] & 0xFFFFu);
                                if (2 * j + 1 < ncols)
                                    d16[2 * j + 1] = static_cast<uint16_t>(pk[j] >> 16);
                            } else {
                                if (j < ncols) reinterpret_cast<uint32_t*>(dst)[j] = pk[j];
                            }
                        }
                    }
                }
                // Keep one bulk group per chunk: the staging buffers alternate
                // with the chunk count, and the wait before a buffer is reused
                // counts groups, so a skipped group would let the next chunk
                // overwrite a buffer an earlier TMA store is still reading.
                if (lane == 0) bulk_commit_group();
                __syncwarp();
                return;
            }
            if (!prm.direct_store) {
                if (lane == 0) bulk_wait_group_read<1>();
                __syncwarp();
            }
            // Row `lane` of the 32 x 128-byte box; 16-byte chunk j is stored at
            // chunk j ^ (row % 8), the TMA 128-byte swizzle pattern.
            const uint32_t row_addr = buf + lane * 128u;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                st_shared_v4(row_addr + ((static_cast<uint32_t>(j) ^ (lane & 7u)) << 4), pk[4 * j],
                             pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
            if (!prm.direct_store) {
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (in_range) tma_store_2d(&map_out, buf, x, row0);
                    bulk_commit_group();
                }
            } else if (in_range) {
                // D rows are not 16-byte aligned: the warp writes the box one row
                // at a time, lane l storing bytes [4l, 4l + 4) of the row
                // (elements 2l, 2l + 1 of a 16-bit output, element l of fp32).
                __syncwarp();
                constexpr int kPerLane = 4 / kOB;
                const int32_t m = x + kPerLane * static_cast<int32_t>(lane);
                const uint32_t lane_off = ((lane >> 2) << 4) + ((lane & 3u) << 2);
                for (int r = 0; r < Cfg::kRowsPerWarp; ++r) {
                    const int32_t grow = row0 + r;
                    if (grow >= prm.rows_p) break;
                    const uint32_t v = ld_shared_u32(
                        buf + r * 128u + (lane_off ^ ((static_cast<uint32_t>(r) & 7u) << 4)));
                    uint8_t* dst = out8 + (static_cast<int64_t>(grow) * prm.ld_out + m) * kOB;
                    if (m + kPerLane - 1 < xlim) {
                        if ((reinterpret_cast<uintptr_t>(dst) & 3u) == 0) {
                            *reinterpret_cast<uint32_t*>(dst) = v;
                        } else {
                            reinterpret_cast<uint16_t*>(dst)[0] = static_cast<uint16_t>(v & 0xFFFFu);
                            reinterpret_cast<uint16_t*>(dst)[1] = static_cast<uint16_t>(v >> 16);
                        }
                    } else if (m < xlim) {  // 16-bit output only
                        reinterpret_cast<uint16_t*>(dst)[0] = static_cast<uint16_t>(v & 0xFFFFu);
                    }
                }
                __syncwarp();
            } else {
                __syncwarp();
            }
        };

        auto release_acc = [&](uint32_t b) {
            // The accumulator has been read: hand it back to the MMA warp.
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                if constexpr (PAIR)
                    mbar_arrive_cluster(mapa_shared(acce_bar(b), 0));
                else
                    mbar_arrive(acce_bar(b));
            }
        };

        for (int64_t u = first; u < num_units; u += stride, ++lt) {
            const Unit w = unit_of(u);
            const int64_t tp = w.tp;
            // A tile narrower than one chunk (16 or 32 columns) spans all of M, so
            // the chunk's columns past the tile lie past M and are not stored.
            // A pair of 64-row halves: this warp's rows carry half the columns.
            const int wcols = Cfg::kColHalves ? w.width / 2 : w.width;
            const int chunks = (wcols + kCols - 1) / kCols;
            const uint32_t b = lt & 1u, aph = (lt >> 1) & 1u;
            if (!warp_wait(accf_bar(b), aph, wd)) break;
            tc_fence_after_sync();
            const uint32_t wrow = Cfg::kColHalves ? (quarter & 1u) : quarter;
            const int32_t row0 =
                static_cast<int32_t>(tp * Cfg::kTileP + rank * Cfg::kBlockP +
                                     wrow * Cfg::kRowsPerWarp);
            const int32_t col0 =
                w.q_off + (Cfg::kColHalves ? static_cast<int32_t>(quarter >> 1) * wcols : 0);
            const int32_t xlim = Cfg::kColHalves && col0 + wcols < prm.rows_q ? col0 + wcols
                                                                              : prm.rows_q;
            const uint32_t t_row = tmem_base + ((quarter * 32u) << 16) + b * Cfg::kAccCols;
            if (!SPLIT || w.pieces == 1) {
#pragma unroll 1
                for (int c = 0; c < chunks; ++c) {
                    uint32_t v0[32], v1[32];
                    tmem_ld_32x32b_x32(t_row + c * kCols, v0);
                    if constexpr (kCols == 64) tmem_ld_32x32b_x32(t_row + c * kCols + 32, v1);
                    tmem_wait_ld();
                    if constexpr (NI > 1) {
                        // the other issuers' sums, in issuer order, for those that
                        // had any of the unit's K stages
#pragma unroll 1
                        for (int ij = 1; ij < NI; ++ij) {
                            if (w.kb_hi - w.kb_lo <= ij) break;
                            uint32_t u0[32], u1[32];
                            const uint32_t t2 = t_row + ij * kAcc2Off + c * kCols;
                            tmem_ld_32x32b_x32(t2, u0);
                            if constexpr (kCols == 64) tmem_ld_32x32b_x32(t2 + 32, u1);
                            tmem_wait_ld();
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                v0[j] = __float_as_uint(__uint_as_float(v0[j]) + __uint_as_float(u0[j]));
                                if constexpr (kCols == 64)
                                    v1[j] = __float_as_uint(__uint_as_float(v1[j]) + __uint_as_float(u1[j]));
                            }
                        }
                    }
                    if (c == chunks - 1) release_acc(b);
                    uint32_t pk[32];
                    if (kOB == 2 && prm.acc16) {
                        // FP16 accumulators: the low halves are the output codes.
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const uint32_t lo = j < 16 ? v0[2 * j] : v1[2 * j - 32];
                            const uint32_t hi = j < 16 ? v0[2 * j + 1] : v1[2 * j - 31];
                            pk[j] = (lo & 0xFFFFu) | (hi << 16);
                        }
                    } else {
                        float f[kCols];
#pragma unroll
                        for (int j = 0; j < kCols; ++j)
                            f[j] = __uint_as_float(j < 32 ? v0[j] : v1[j - 32]);
                        pack(f, pk);
                    }
                    emit(pk, col0 + c * kCols, row0, xlim);
                }
            } else if constexpr (SPLIT) {
                // This K piece's partial sums -> workspace, column-major within
                // the slice so that a warp's stores (and loads) are coalesced.
                // The accumulator stays in TMEM until this warp knows whether
                // it combines the pieces: the last piece to arrive reads its
                // own sums from there instead of back from memory.
                const int32_t piece = w.piece;
                float* part = prm.ws_partials +
                              ((w.ws_tile * w.pieces + piece) * kSlices + slice) * kSliceFloats;
#pragma unroll 1
                for (int c = 0; c < (w.width + 31) / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(t_row + c * 32, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        __stcg(part + (c * 32 + j) * 32 + lane, __uint_as_float(v[j]));
                }
                __threadfence();
                __syncwarp();
                unsigned int prev = 0;
                unsigned int* counter = prm.ws_counters + w.ws_tile * kSlices + slice;
                if (lane == 0) prev = atomicAdd(counter, 1u);
                prev = __shfl_sync(0xffffffffu, prev, 0);
                if (prev + 1 != static_cast<unsigned int>(w.pieces)) {
                    release_acc(b);
                    continue;
                }
                // Last piece of this slice: sum all pieces in piece order (the
                // result does not depend on which piece finished last).
                __threadfence();
                if (lane == 0) *counter = 0u;  // ready for the next call
                const float* base_part =
                    prm.ws_partials + (w.ws_tile * w.pieces * kSlices + slice) * kSliceFloats;
#pragma unroll 1
                for (int c = 0; c < chunks; ++c) {
                    float f[kCols];
#pragma unroll
                    for (int j = 0; j < kCols; ++j) f[j] = 0.f;
                    for (int32_t pc = 0; pc < w.pieces; ++pc) {
                        if (pc == piece) {
                            uint32_t v0[32], v1[32];
                            tmem_ld_32x32b_x32(t_row + c * kCols, v0);
                            if constexpr (kCols == 64)
                                tmem_ld_32x32b_x32(t_row + c * kCols + 32, v1);
                            tmem_wait_ld();
#pragma unroll
                            for (int j = 0; j < kCols; ++j)
                                f[j] += __uint_as_float(j < 32 ? v0[j] : v1[j - 32]);
                        } else {
                            const float* src =
                                base_part + static_cast<int64_t>(pc) * kSlices * kSliceFloats;
#pragma unroll
                            for (int j = 0; j < kCols; ++j)
                                f[j] += __ldcg(src + (c * kCols + j) * 32 + lane);
                        }
                    }
                    uint32_t pk[32];
                    pack(f, pk);
                    emit(pk, col0 + c * kCols, row0, xlim);
                }
                release_acc(b);
            }
        }
        // The staging buffers must have been read before the CTA exits; the
        // stores' global writes complete with the grid, which the next grid
        // in the stream waits for (griddepcontrol.wait) before it reads C.
        if (!prm.direct_store && lane == 0) bulk_wait_group_read<0>();
        __syncwarp();
    }

    // ---------------------------------------------------- teardown
    tc_fence_before_sync();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc<Cfg::kCG>(tmem_base, Cfg::kTmemCols);
    }
}

template <InKind IN, typename OutT, bool PAIR, bool LOADS, bool SPLIT, bool HALF = false,
          int NI = 1, int AT = 1>
cudaError_t tc_launch_one_at(const TcLaunch& L) {
    using Cfg = TcCfg<IN, PAIR, LOADS, HALF, NI>;
    auto kernel = tc_gemm_kernel<IN, OutT, PAIR, LOADS, SPLIT, HALF, NI, AT>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !attr_set[dev]) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Cfg::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(L.grid), 1, 1);
    cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cfg.stream = L.stream;
    // The kernel starts its prologue while the previous grid in the stream
    // finishes, and waits for it (pdl_wait) before touching global memory.
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (PAIR) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = 2;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, kernel, L.map_p, L.map_q, L.map_out, L.map_q_tail, L.prm);
}

// One or two K atoms per stage (TMA producer only), as the plan says.
template <InKind IN, typename OutT, bool PAIR, bool LOADS, bool SPLIT, bool HALF = false,
          int NI = 1>
cudaError_t tc_launch_one(const TcLaunch& L) {
    if constexpr (LOADS) {
        if (L.prm.atoms != 1) return cudaErrorInvalidConfiguration;
        return tc_launch_one_at<IN, OutT, PAIR, LOADS, SPLIT, HALF, NI, 1>(L);
    } else {
        if (L.prm.atoms == 2) return tc_launch_one_at<IN, OutT, PAIR, LOADS, SPLIT, HALF, NI, 2>(L);
        if (L.prm.atoms != 1) return cudaErrorInvalidConfiguration;
        return tc_launch_one_at<IN, OutT, PAIR, LOADS, SPLIT, HALF, NI, 1>(L);
    }
}

template <InKind IN, typename OutT, bool SPLIT>
cudaError_t tc_launch_split(bool pair, Producer prod, const TcLaunch& L) {
    if (prod == Producer::Loads) {
        if (pair || L.half) return cudaErrorInvalidConfiguration;
        return tc_launch_one<IN, OutT, false, true, SPLIT>(L);
    }
    if (L.issuers > 1) {
        if constexpr (SPLIT) {
            return cudaErrorInvalidConfiguration;
        } else {
            if (pair != L.half || L.issuers != 2) return cudaErrorInvalidConfiguration;
            return pair ? tc_launch_one<IN, OutT, true, false, false, true, 2>(L)
                        : tc_launch_one<IN, OutT, false, false, false, false, 2>(L);
        }
    }
    if (L.half) {
        if constexpr (SPLIT) {
            return cudaErrorInvalidConfiguration;
        } else {
            return pair ? tc_launch_one<IN, OutT, true, false, false, true>(L)
                        : tc_launch_one<IN, OutT, false, false, false, true>(L);
        }
    }
    return pair ? tc_launch_one<IN, OutT, true, false, SPLIT>(L)
                : tc_launch_one<IN, OutT, false, false, SPLIT>(L);
}

template <InKind IN, typename OutT>
cudaError_t tc_launch_impl(bool pair, Producer prod, const TcLaunch& L) {
    const bool split = L.prm.splits > 1 || L.prm.tail_ksplit != 0;
    return split ? tc_launch_split<IN, OutT, true>(pair, prod, L)
                 : tc_launch_split<IN, OutT, false>(pair, prod, L);
}

template <InKind IN>
TcGeometry tc_geometry_impl(bool pair, bool half) {
    if (half && pair) {
        using Cfg = TcCfg<IN, true, false, true>;
        return TcGeometry{Cfg::kTileP,  Cfg::kMmaN,    Cfg::kBlockP,      Cfg::kStageK,
                          2,            Cfg::kMmaM,    Cfg::kFormat,      Cfg::kStageRegion,
                          Cfg::kMaxStages, Cfg::kEpiBytes};
    }
    if (half) {
        using Cfg = TcCfg<IN, false, false, true>;
        return TcGeometry{Cfg::kTileP,  Cfg::kMmaN,    Cfg::kBlockP,      Cfg::kStageK,
                          1,            Cfg::kMmaM,    Cfg::kFormat,      Cfg::kStageRegion,
                          Cfg::kMaxStages, Cfg::kEpiBytes};
    }
    if (pair) {
        using Cfg = TcCfg<IN, true, false>;
        return TcGeometry{Cfg::kTileP,  Cfg::kMmaN,    Cfg::kBlockP,      Cfg::kStageK,
                          2,            Cfg::kMmaM,    Cfg::kFormat,      Cfg::kStageRegion,
                          Cfg::kMaxStages, Cfg::kEpiBytes};
    }
    using Cfg = TcCfg<IN, false, false>;
    return TcGeometry{Cfg::kTileP,  Cfg::kMmaN,    Cfg::kBlockP,      Cfg::kStageK,
                      1,            Cfg::kMmaM,    Cfg::kFormat,      Cfg::kStageRegion,
                      Cfg::kMaxStages, Cfg::kEpiBytes};
}

}  // namespace gb300
