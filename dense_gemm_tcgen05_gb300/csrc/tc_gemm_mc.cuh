// tc_gemm_mc.cuh -- the tensor-core GEMM with clusters of two CTA pairs that
// share their P tiles through TMA multicast.
//
// Computes the same D = P Q^T as tc_gemm_kernel (P = B, rows n; Q = A, rows m;
// D row-major = C column-major), with the same cta_group::2 pairs, 256 rows of
// P per pair tile, one swizzle atom of K per stage, double-buffered TMEM
// accumulators and the same epilogue arithmetic.  What differs is that a
// cluster holds four CTAs, two pairs, and the two pairs compute horizontally
// adjacent tiles (tq, tp) and (tq + 1, tp): they need the same 256 rows of P.
// CTA rp of each pair holds the same 128 of them, so each of those two CTAs
// loads one 64-row half of its block and multicasts it into both CTAs' stage:
// every P stage costs each CTA half the L2 reads (measured: 26 % fewer L2 bytes
// at 4096^3).  The aim was to let narrower tiles (tile_q = 192: 4.63 waves at
// 4096^3 instead of 3.37) run without being bound by operand loads.  Measured
// on GB300 it matches the pair kernel at 4096^3 (1692 TFLOP/s at tile_q = 192
// with the 7-stage ring below) and is 2-4 % slower at 8192^3: a stage slot is
// free only once both pairs are done with it, and the follower's forwarding
// adds a hop to every stage.  It is therefore an option ("cluster" = 4), not
// the default.
//
// Synchronisation per ring slot s:
//   full[s]  in every CTA counts the bytes that land in that CTA (its own Q
//            half, its own P half-block and the partner pair's multicast P
//            half-block; a multicast may complete before the local
//            expect_tx, which mbarrier transaction counts allow).  The
//            follower CTA of a pair forwards "slot full" to the pair leader,
//            whose full[s] therefore expects two arrivals: its own producer's
//            and the follower's.
//   empty[s] in every CTA expects two arrivals: one tcgen05.commit from each
//            pair leader's MMA warp, multicast to all four CTAs, because a
//            producer's multicast writes into its partner's slot as well as
//            its own.
// The accumulator barriers stay within each pair.  Work: cluster unit u is the
// tile pair (tq2, tp) of the grouped raster over (ceil(tiles_q / 2), tiles_p);
// pair pp computes tq = 2 tq2 + pp.  When tiles_q is odd the second pair of the
// last column computes a tile outside the matrix: its Q loads are zero-filled,
// its stores are skipped, and it still multicasts its P half-block.
//
// No split-K, tail splitting, FP16 accumulation or row-wise stores here; the
// host uses this kernel only where none of them is needed.  Every wait is
// bounded as in tc_gemm_kernel.
#pragma once

#include "tc_gemm.cuh"

namespace gb300 {

// 2D tiled load with cluster multicast: the box lands at `dst` in every CTA of
// `mask`, and each of those CTAs' barrier at offset `bar` receives the
// transaction bytes that landed in it.
__device__ __forceinline__ void tma_load_2d_mc(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                               int32_t x, int32_t y, uint16_t mask) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".multicast::cluster [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "h"(mask)
        : "memory");
}

// Arrive on a barrier in another CTA of the cluster with the default
// (release, CTA scope) semantics: the forwarded "slot full" carries no data of
// its own (the slot was filled by TMA and observed complete by this CTA), so
// the cluster-scope release of mbar_arrive_cluster is not needed -- and its
// fence on every stage made this kernel three times slower.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Shared-memory layout: a 200 KB ring (7 stages at tile_q = 192, 6 at 256, 8
// at 128) and one epilogue staging buffer per warp.
template <InKind IN>
struct McCfg : TcCfg<IN, true, false> {
    using Base = TcCfg<IN, true, false>;
    static constexpr int kStageRegion = 200 * 1024;
    static constexpr int kEpiBytes = Base::kEpiWarps * Base::kEpiBufBytes;
    static constexpr int kOffEpi = kStageRegion;
    static constexpr int kOffBars = kOffEpi + kEpiBytes;
    static constexpr int kOffTmemSlot = kOffBars + Base::kNumBars * 8;
    static constexpr int kOffAbort = kOffTmemSlot + 4;
    static constexpr int kSmemBytes = kOffAbort + 4 + 1024;  // + alignment slack
    static_assert(kSmemBytes <= 232448, "shared memory budget");
};

template <InKind IN, typename OutT>
__global__ void __launch_bounds__(192, 1)
    tc_mc_kernel(const __grid_constant__ CUtensorMap map_p,
                 const __grid_constant__ CUtensorMap map_q,
                 const __grid_constant__ CUtensorMap map_out, const TcParams prm) {
    using Cfg = McCfg<IN>;
    constexpr int SM = Cfg::kMaxStages;
    constexpr int kHalfP = Cfg::kBlockP / 2;          // P rows each CTA loads per stage
    const uint32_t S = static_cast<uint32_t>(prm.stages);
    const uint32_t stage_bytes = prm.stage_bytes;

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

    const uint32_t rank = cluster_ctarank();   // 0..3
    const uint32_t pp = rank >> 1;             // pair within the cluster
    const uint32_t rp = rank & 1u;             // CTA within the pair
    const bool leader = rp == 0;
    const uint32_t lead_rank = rank & ~1u;
    const uint32_t partner = rank ^ 2u;        // same position in the other pair
    const uint16_t pair_mask = static_cast<uint16_t>(0x3u << lead_rank);
    const uint16_t mc_mask = static_cast<uint16_t>((1u << rank) | (1u << partner));

    if (threadIdx.x == 0) {
        for (int s = 0; s < SM; ++s) {
            mbar_init(full_bar(s), leader ? 2u : 1u);
            mbar_init(empty_bar(s), 2u);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), 2 * Cfg::kEpiWarps);
        }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&map_p);
        prefetch_tensormap(&map_q);
        prefetch_tensormap(&map_out);
    }
    if (warp == 1) {
        tmem_alloc<2>(smem_u32(tmem_slot), Cfg::kTmemCols);
        tmem_relinquish<2>();
    }
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();
    tc_fence_after_sync();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

    const Watch wd{abort_flag, prm.watchdog, prm.timeout_ns};
    const int64_t tiles_q2 = (static_cast<int64_t>(prm.tiles_q) + 1) / 2;
    const int64_t num_units = tiles_q2 * prm.tiles_p;
    const int64_t first = blockIdx.x / 4;
    const int64_t stride = gridDim.x / 4;
    // This pair's tile of cluster unit u: its first P row and Q column.
    auto tile_of = [&](int64_t u, int32_t* p_tile0, int32_t* q_off) {
        int64_t tq2, tp;
        raster_tile(u, tiles_q2, prm.tiles_p, prm.group, &tq2, &tp);
        *p_tile0 = static_cast<int32_t>(tp * Cfg::kTileP);
        *q_off = static_cast<int32_t>((2 * tq2 + pp) * prm.tile_q);
    };

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        uint32_t it = 0, rs = 0, rph = 0;
        bool ok = true;
        const int32_t half_q = prm.tile_q / 2;
        for (int64_t u = first; ok && u < num_units; u += stride) {
            int32_t p_tile0, q_off;
            tile_of(u, &p_tile0, &q_off);
            const int32_t p_rows = p_tile0 + static_cast<int32_t>(rp) * Cfg::kBlockP;
            const int32_t q0 = q_off + static_cast<int32_t>(rp) * half_q;
            for (int32_t kb = 0; kb < prm.num_kb; ++kb, ++it) {
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
                    const uint32_t sq = sp + Cfg::kBytesP;
                    const int32_t kx = kb * Cfg::kStageK;
                    mbar_arrive_expect_tx(full_bar(s), prm.stage_tx_bytes);
                    tma_load_2d(sq, &map_q, full_bar(s), kx, q0);
                    tma_load_2d_mc(sp + pp * (kHalfP * Cfg::kAtomBytes), &map_p, full_bar(s), kx,
                                   p_rows + static_cast<int32_t>(pp) * kHalfP, mc_mask);
                }
                __syncwarp();
            }
        }
        if (!ok) {
            // Aborting: copies of this CTA and its partner may still be in
            // flight into this CTA's stages; give them time to land.
            if (lane == 0) pause_ns(200000);
            __syncwarp();
        }
    } else if (warp == 1 && !leader) {
        // ------------------------------------------------ follower: forward "slot full"
        uint32_t rs = 0, rph = 0;
        bool ok = true;
        for (int64_t u = first; ok && u < num_units; u += stride) {
            for (int32_t kb = 0; kb < prm.num_kb; ++kb) {
                const uint32_t s = rs, ph = rph;
                if (++rs == S) {
                    rs = 0;
                    rph ^= 1u;
                }
                if (!warp_wait(full_bar(s), ph, wd)) {
                    ok = false;
                    break;
                }
                if (lane == 0) mbar_arrive_remote(mapa_shared(full_bar(s), lead_rank));
                __syncwarp();
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (pair leader)
        uint32_t lt = 0, rs = 0, rph = 0;
        const uint64_t adesc0 = sdesc_kmajor_sw128(base);
        const uint64_t bdesc0 = sdesc_kmajor_sw128(base + Cfg::kBytesP);
        bool ok = true;
        for (int64_t u = first; ok && u < num_units; u += stride, ++lt) {
            const uint32_t b = lt & 1u, aph = (lt >> 1) & 1u;
            if (!warp_wait(acce_bar(b), aph ^ 1u, wd)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            const uint32_t d_tmem = tmem_base + b * Cfg::kAccCols;
            for (int32_t kb = 0; kb < prm.num_kb; ++kb) {
                const uint32_t s = rs, ph = rph;
                if (++rs == S) {
                    rs = 0;
                    rph ^= 1u;
                }
                if (!warp_wait(full_bar(s), ph, wd)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                if (lane == 0) {
                    const uint64_t soff = static_cast<uint64_t>(s * (stage_bytes >> 4));
                    const uint64_t adesc = adesc0 + soff;
                    const uint64_t bdesc = bdesc0 + soff;
#pragma unroll
                    for (int kk = 0; kk < Cfg::kMmasPerStage; ++kk) {
                        const uint64_t off = static_cast<uint64_t>(kk * (Cfg::kMmaKBytes >> 4));
                        const uint32_t acc = (kb != 0 || kk != 0) ? 1u : 0u;
                        if constexpr (IN == InKind::E4M3)
                            mma_f8<2>(d_tmem, adesc + off, bdesc + off, prm.idesc, acc);
                        else
                            mma_f16<2>(d_tmem, adesc + off, bdesc + off, prm.idesc, acc);
                    }
                    // the slot is free in all four CTAs once both pairs are done
                    commit_to<2>(empty_bar(s), 0xF);
                }
                __syncwarp();
            }
            if (!ok) break;
            if (lane == 0) commit_to<2>(accf_bar(b), pair_mask);
            __syncwarp();
        }
        if (lane == 0) commit_to<2>(done_bar, static_cast<uint16_t>(1u << rank));
        __syncwarp();
        const uint64_t t0 = global_timer_ns();
        while (!__all_sync(0xffffffffu, mbar_try_wait(done_bar, 0))) {
            if (global_timer_ns() - t0 > prm.timeout_ns) {
                if (lane == 0) atomicOr(prm.watchdog, kWatchTimeout);
                break;
            }
        }
    } else if (warp >= 2 && warp < 2 + Cfg::kEpiWarps) {
        // ------------------------------------------------ epilogue
        constexpr int kOB = static_cast<int>(sizeof(OutT));
        constexpr int kCols = 128 / kOB;
        constexpr int kGran = 16 / kOB;
        const uint32_t quarter = warp & 3u;
        const uint32_t ew = warp - 2u;
        const uint32_t buf = base + Cfg::kOffEpi + ew * Cfg::kEpiBufBytes;  // one per warp
        const float scale = prm.scale;
        uint8_t* const out8 = static_cast<uint8_t*>(prm.out);
        uint32_t lt = 0;

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
        // Stages this warp's chunk (rows row0 + lane, columns [x, x + kCols))
        // and stores it with TMA; a chunk that ends inside a 16-byte granule
        // past rows_q is stored element by element instead (TMA stores whole
        // granules).  The staging buffer is reused once the previous chunk's
        // TMA store has read it.
        auto emit = [&](const uint32_t (&pk)[32], int32_t x, int32_t row0) {
            const bool in_range = x < prm.rows_q && row0 < prm.rows_p;
            if (in_range && x + kCols > prm.rows_q && (prm.rows_q % kGran) != 0) {
                const int32_t r = row0 + static_cast<int32_t>(lane);
                if (r < prm.rows_p) {
                    uint8_t* dst = out8 + (static_cast<int64_t>(r) * prm.ld_out + x) * kOB;
                    const int32_t ncols = prm.rows_q - x;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if constexpr (kOB == 2) {
                            uint16_t* d16 = reinterpret_cast<uint16_t*>(dst);
                            if (2 * j < ncols) d16[2 * j] = static_cast<uint16_t>(pk[j] & 0xFFFFu);
                            if (2 * j + 1 < ncols) d16[2 * j + 1] = static_cast<uint16_t>(pk[j] >> 16);
                        } else {
                            if (j < ncols) reinterpret_cast<uint32_t*>(dst)[j] = pk[j];
                        }
                    }
                }
                __syncwarp();
                return;
            }
            if (lane == 0) bulk_wait_group_read<0>();
            __syncwarp();
            const uint32_t row_addr = buf + lane * 128u;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                st_shared_v4(row_addr + ((static_cast<uint32_t>(j) ^ (lane & 7u)) << 4), pk[4 * j],
                             pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                if (in_range) tma_store_2d(&map_out, buf, x, row0);
                bulk_commit_group();
            }
        };

        for (int64_t u = first; u < num_units; u += stride, ++lt) {
            int32_t p_tile0, q_off;
            tile_of(u, &p_tile0, &q_off);
            const int chunks = prm.tile_q / kCols;
            const uint32_t b = lt & 1u, aph = (lt >> 1) & 1u;
            if (!warp_wait(accf_bar(b), aph, wd)) break;
            tc_fence_after_sync();
            const int32_t row0 =
                p_tile0 + static_cast<int32_t>(rp * Cfg::kBlockP + quarter * 32);
            const uint32_t t_row = tmem_base + ((quarter * 32u) << 16) + b * Cfg::kAccCols;
#pragma unroll 1
            for (int c = 0; c < chunks; ++c) {
                uint32_t v0[32], v1[32];
                tmem_ld_32x32b_x32(t_row + c * kCols, v0);
                if constexpr (kCols == 64) tmem_ld_32x32b_x32(t_row + c * kCols + 32, v1);
                tmem_wait_ld();
                if (c == chunks - 1) {
                    // the accumulator has been read: hand it back to the pair's MMA warp
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(mapa_shared(acce_bar(b), lead_rank));
                }
                float f[kCols];
#pragma unroll
                for (int j = 0; j < kCols; ++j) f[j] = __uint_as_float(j < 32 ? v0[j] : v1[j - 32]);
                uint32_t pk[32];
                pack(f, pk);
                emit(pk, q_off + c * kCols, row0);
            }
        }
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
    }

    // ---------------------------------------------------- teardown
    // No CTA of the cluster leaves while a partner may still multicast into it
    // or arrive on its barriers.
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc<2>(tmem_base, Cfg::kTmemCols);
    }
}

// Clusters of four CTAs (two pairs); L.grid is a multiple of 4.
template <InKind IN, typename OutT>
cudaError_t tc_mc_launch_impl(const TcLaunch& L) {
    using Cfg = McCfg<IN>;
    auto kernel = tc_mc_kernel<IN, OutT>;
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
    cfg.blockDim = dim3(192, 1, 1);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 4;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, L.map_p, L.map_q, L.map_out, L.prm);
}

// Most clusters of four that can be resident at once.
template <InKind IN, typename OutT>
cudaError_t tc_mc_max_clusters_impl(int* n) {
    using Cfg = McCfg<IN>;
    auto kernel = tc_mc_kernel<IN, OutT>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(4, 1, 1);
    cfg.blockDim = dim3(192, 1, 1);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 4;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(n, kernel, &cfg);
}

}  // namespace gb300
