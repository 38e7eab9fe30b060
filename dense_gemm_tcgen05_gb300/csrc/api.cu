// api.cu -- the C ABI of libgemm.so (declared in include/gemm.h): argument
// validation, device checks, path choice, TMA tensor-map encoding and launch.
//
// Nothing here allocates device memory.  Tensor maps are encoded on the host
// per call (a few hundred nanoseconds) and passed by value as
// __grid_constant__ kernel parameters.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "launch.h"
#include "gemm.h"
#include "ptx.cuh"
#include "raster.h"

namespace gb300 {
cudaError_t tc_launch_f16(bool pair, Producer prod, const TcLaunch& L);
cudaError_t tc_launch_bf16(bool pair, Producer prod, const TcLaunch& L);
cudaError_t tc_launch_bf16_f32(bool pair, Producer prod, const TcLaunch& L);
cudaError_t tc_launch_fp8(bool pair, Producer prod, bool out_f32, const TcLaunch& L);
TcGeometry tc_geometry_f16(bool pair, bool half);
TcGeometry tc_geometry_bf16(bool pair, bool half);
TcGeometry tc_geometry_fp8(bool pair, bool half);

TcGeometry tc_geometry(InKind in, bool pair, bool half) {
    switch (in) {
        case InKind::F16: return tc_geometry_f16(pair, half);
        case InKind::BF16: return tc_geometry_bf16(pair, half);
        default: return tc_geometry_fp8(pair, half);
    }
}

cudaError_t tc_launch(InKind in, bool pair, Producer prod, bool out_f32, const TcLaunch& L) {
    switch (in) {
        case InKind::F16: return tc_launch_f16(pair, prod, L);
        case InKind::BF16:
            return out_f32 ? tc_launch_bf16_f32(pair, prod, L) : tc_launch_bf16(pair, prod, L);
        default: return tc_launch_fp8(pair, prod, out_f32, L);
    }
}
}  // namespace gb300

using namespace gb300;

// Per-device watchdog word: kernels OR kWatchTimeout into it when a bounded
// wait runs out.  Its device address is looked up once per device.
__device__ unsigned int g_gemm_watchdog_word;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool ready = false;
    int cc_major = 0, cc_minor = 0, sms = 0;
    unsigned int* watchdog = nullptr;
    void* workspace = nullptr;      // caller-registered split-K scratch (gemm_set_workspace)
    int64_t workspace_bytes = 0;
};

std::mutex g_mutex;
DeviceInfo g_devices[kMaxDevices];
// Which fixed counter set of the registered workspace the next split launch
// on each device counts in.
std::atomic<unsigned int> g_cnt_parity[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

std::atomic<int> g_opt_pair{-1};
std::atomic<int> g_opt_group{0};
std::atomic<int> g_opt_k_snake{1};
std::atomic<int> g_opt_k_rotate{0};
std::atomic<int> g_opt_band_snake{1};
std::atomic<int> g_opt_path{0};
std::atomic<int> g_opt_max_ctas{0};
std::atomic<int> g_opt_splits{0};
std::atomic<int> g_opt_tile_q{0};
std::atomic<int> g_opt_tail{0};
std::atomic<int> g_opt_tail_k{0};
std::atomic<int> g_opt_repack{0};
std::atomic<int> g_opt_f32_tail{0};
std::atomic<int> g_opt_f32_ktail{0};
std::atomic<int> g_opt_atoms{0};
std::atomic<int> g_opt_l2hints{0};
std::atomic<int> g_opt_half{0};
std::atomic<int> g_opt_issuers{0};
std::atomic<int64_t> g_opt_timeout_ns{2000000000LL};

thread_local cudaError_t t_last_cuda_error = cudaSuccess;
thread_local char t_status_buf[256];

int fail_cuda(cudaError_t e) {
    t_last_cuda_error = e;
    return GEMM_ERR_LAUNCH;
}

// Looks up (once) the attributes of the current device.  Returns a status.
int current_device(const DeviceInfo** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e);
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo& d = g_devices[dev];
    if (!d.ready) {
        if ((e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) !=
                cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) !=
                cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) !=
                cudaSuccess)
            return fail_cuda(e);
        if (d.cc_major == 10 && d.cc_minor == 3) {
            void* p = nullptr;
            if ((e = cudaGetSymbolAddress(&p, g_gemm_watchdog_word)) != cudaSuccess)
                return fail_cuda(e);
            d.watchdog = static_cast<unsigned int*>(p);
        }
        if (!g_encode) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q);
            if (e != cudaSuccess) return fail_cuda(e);
            if (q != cudaDriverEntryPointSuccess || !fn) return fail_cuda(cudaErrorNotSupported);
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        d.ready = true;
    }
    if (!(d.cc_major == 10 && d.cc_minor == 3)) return GEMM_ERR_UNSUPPORTED_DEVICE;
    *out = &d;
    return GEMM_OK;
}

bool aligned(const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

// Q rows per tile (= MMA N) for a problem with M rows of Q.  Cost = padded
// MMA columns, ceil(M / t) * t, with narrow tiles charged as 96 columns (below
// that the per-stage P traffic, not the MMA, sets the pace); ties go to the
// wider tile, which re-reads P fewer times.
int choose_tile_q(int64_t M, int max_tile_q) {
    static const int kChoices[] = {256, 192, 128, 64};
    int best = max_tile_q;
    int64_t best_cost = INT64_MAX;
    for (int t : kChoices) {
        if (t > max_tile_q) continue;
        const int64_t cost = ((M + t - 1) / t) * (t > 96 ? t : 96);
        if (cost < best_cost) {
            best_cost = cost;
            best = t;
        }
    }
    return best;
}

// Rasteriser group (tile rows of Q per band) when option "group" is 0.  The
// GB300 L2 is two partitions, one per die, and a line an SM reads from the
// other die's memory is also kept in the reading die's partition, so data that
// both dies read takes twice its size.  An LRU model of that, run over the
// persistent schedule, reproduces the DRAM reads measured per 8192^3 FP16
// launch at groups 2, 4, 8, 16 and 32 (2.17, 1.53, 1.07, 1.22, 2.11 GB; model
// 2.06, 1.42, 1.10, 1.29, 2.06).  With every second unit's K range read
// backwards (TcParams::k_snake) it predicts 0.62-0.80 GB at group 16, against
// 0.71-0.78 at 12 and 0.85-0.89 at 8, depending on how CTA pairs fall on the
// dies, and group 16 is as good or better on the other large shapes tried
// (FP8 8192^3, BF16 4096 x 14336 x 4096, FP16 8192 x 28672 x 8192).
constexpr int kDefaultGroup = 16;

constexpr int64_t kMaxDim = 0x7fffffffLL;
// Leading dimensions above this many elements cannot address device memory;
// the bound keeps every pitch and size product below 2^63.
constexpr int64_t kMaxLd = 1LL << 48;
// Byte counts for sizes no device can hold saturate here, a quarter of the
// int64 range, so that a few of them can still be added without overflow.
constexpr int64_t kSatBytes = INT64_MAX / 4;

// a * b for a, b >= 0, saturating at kSatBytes.
int64_t sat_mul(int64_t a, int64_t b) {
    if (a == 0 || b == 0) return 0;
    return a > kSatBytes / b ? kSatBytes : a * b;
}

// x rounded up to a multiple of 256, for x in [0, kSatBytes].
int64_t round256(int64_t x) { return (x + 255) / 256 * 256; }

// Whether `need` bytes (possibly a saturated sum) fit in `room`: a saturated
// size never does, however large the room.
bool fits(int64_t need, int64_t room) { return need < kSatBytes && need <= room; }

// What a TN call is given, for planning: shapes, what TMA can address, the
// scratch available, and the device.
struct TnPlanIn {
    InKind in;
    bool out_f32, acc16;
    int64_t M, N, K;
    bool a_tma, b_tma, c_tma;   // rows TMA can address (16-byte bases and pitches)
    bool a_al128, b_al128;      // rows starting on 128-byte boundaries
    bool has_scratch;           // a registered workspace or an override
    int64_t ws_total;           // its bytes for repacks and partial sums
    int ov_splits;              // -1: option "splits" applies; else the override's value
    bool strict;                // the no-allocation call's rules (see plan_tn)
    bool no_copy = false;       // never repack operands into the scratch
    int sms;                    // SMs of the device
};

// Everything gemm_tn decides before it encodes tensor maps and launches.
struct TnPlan {
    int status = GEMM_OK;       // GEMM_ERR_SCRATCH when a strict split does not fit
    bool copy_a = false, copy_b = false;  // repacked into the scratch
    int64_t dp = 0;             // repacked row pitch in bytes
    int64_t ws_used = 0;        // scratch bytes taken by the repacks
    Producer prod = Producer::Tma;
    bool pair = false, half = false;
    int issuers = 1;            // MMA-issuing warps (TcCfg NI)
    int tile_q = 0, load_q = 0;
    TcGeometry g{};
    int64_t tiles_p = 0, tiles_q = 0, tiles = 0, slots = 0;
    int num_kb = 0, stages = 0, stage_bytes = 0;
    int atoms = 1;              // K atoms (128-byte swizzle spans) per ring stage
    bool ring_epi = false;      // the ring extends over the epilogue's staging area
    int splits = 1, kb_per_split = 0;
    int64_t split_cnt_bytes = 0;  // counter bytes ahead of the split partials
    int tail_f = 1, tail_kb_per = 0;
    bool tail_ksplit = false;
    int64_t full_units = 0;
    int64_t tail_cnt_bytes = 0;   // counter bytes ahead of the K-split tail's partials
    int grid = 0;
};

// The planning half of gemm_tn: a pure function of its input and the
// process-wide options, so that the rules can be checked without a GPU
// (gemm_tn_plan).  Each rule is measured on GB300; the numbers are with the
// rules below.
TnPlan plan_tn_once(const TnPlanIn& a) {
    TnPlan p;
    const int es = a.in == InKind::E4M3 ? 1 : 2;
    const int os = a.out_f32 ? 4 : 2;
    const int64_t M = a.M, N = a.N, K = a.K;
    bool a_tma = a.a_tma, b_tma = a.b_tma;

    // Operands whose rows TMA cannot address are copied once into the scratch
    // with 128-byte-aligned rows (one pass at memory speed), after which the
    // TMA path runs at full rate; without room for that, the load-based
    // producer reads them in place.  Rows TMA can address but that do not start
    // on 128-byte boundaries make every 128-byte row segment of a box straddle
    // two cache lines, which measured on GB300 costs 20-45 % (BF16 4096^3 with
    // ld = 4104: 107 against 80 us; FP16 8192^3 with ld = 8200: 786 against
    // 575-646 us).  They are copied too when the product is compute-heavy
    // enough for the copy (2 (M + N) K element bytes at ~5.8 TB/s) to cost
    // clearly less: MN / (M + N) >= 1100 x element size.  Measured with the
    // copy: 6144^3 383 -> 319-358 us, 8192^3 786 -> 662-703 us, 16384^3 6652 ->
    // 5763-5804 us; at 4096^3 the copy (22 us) and the penalty (27 us) cancel.
    const bool heavy = static_cast<double>(M) * static_cast<double>(N) /
                           static_cast<double>(M + N) >= 1100.0 * es;
    const bool copy_a = !a_tma || (heavy && !a.a_al128);
    const bool copy_b = !b_tma || (heavy && !a.b_al128);
    if ((copy_a || copy_b) && g_opt_path.load() == 0 && g_opt_repack.load() == 0 &&
        a.has_scratch && !a.no_copy) {
        const int64_t rb = K * es;                       // row bytes
        const int64_t dp = (rb + 127) / 128 * 128;       // aligned pitch
        const int64_t need_a = copy_a ? round256(sat_mul(M, dp)) : 0;
        const int64_t need_b = copy_b ? round256(sat_mul(N, dp)) : 0;
        if (fits(need_a + need_b, a.ws_total)) {
            p.copy_a = copy_a;
            p.copy_b = copy_b;
            p.dp = dp;
            if (copy_a) a_tma = true;
            if (copy_b) b_tma = true;
            p.ws_used = need_a + need_b;
        }
    }
    const bool ab_tma = a_tma && b_tma;
    p.prod = (ab_tma && g_opt_path.load() != 2) ? Producer::Tma : Producer::Loads;
    const int opt_pair = g_opt_pair.load();
    // cta_group::2 pairs measured faster on every shape with at least a wave
    // of tiles; they need TMA.  When the pair tiles (256 rows of N each) fill
    // less than one wave but single-CTA tiles of 128 rows of N by `small_q`
    // columns of M (16 or 32 when M fits, 64 for M <= 128, else 128) still fit
    // in one, the smaller tiles run instead: up to four times the tiles in
    // flight.  Measured on GB300 against pairs: BF16 M x N x K = 16..128 x 8192
    // x 8192 5-7 % faster, 128 x 8192 x 2048 31 %, 256 x 8192 x 8192 17 %,
    // 1024 x 1024 x 8192 21 % (FP8 45 %), 1024 x 2048 x 4096 30 %; where the
    // small tiles would need a second wave (512 x 8192 x 8192, 2048^3) pairs
    // stay 10-26 % faster.
    p.pair = p.prod == Producer::Tma && opt_pair != 0;
    int small_q = 0;
    bool pair_q128 = false;
    if (p.pair && opt_pair < 0) {
        const int64_t pair_tiles = ((N + 255) / 256) * ((M + choose_tile_q(M, 256) - 1) /
                                                        choose_tile_q(M, 256));
        const int q = M <= 16 ? 16 : M <= 32 ? 32 : M <= 128 ? 64 : 128;
        const int64_t small_tiles = ((N + 127) / 128) * ((M + q - 1) / q);
        if (pair_tiles < a.sms / 2 && small_tiles <= a.sms) {
            // ... except with long K (16-bit inputs, K >= 8192) and M > 256,
            // where pair tiles 128 columns wide still fit in one wave: a CTA
            // of a pair takes in 24 KB per K atom for its 128 x 128 outputs,
            // one CTA alone 32 KB, and these launches stream operands for
            // most of their time.  Measured on GB300 (graph-replayed, BF16,
            // one-CTA -> pair 128 wide): 1024 x 1536 x 8192 30.2 -> 26.8 us,
            // 1024 x 1024 x 8192 20.9 -> 20.0, 512 x 512 x 16384 21.4 -> 20.9,
            // 768 x 1024 x 8192 18.0 -> 17.8; with K <= 4096 the one-CTA tiles
            // stay ahead (2048 x 1024 x 2048 9.2 against 10.5, 512 x 2048 x
            // 4096 14.1 against 14.4).
            const int64_t pair128_tiles = ((N + 255) / 256) * ((M + 127) / 128);
            if (q == 128 && M > 256 && a.in != InKind::E4M3 && K >= 8192 &&
                pair128_tiles <= a.sms / 2 && g_opt_tile_q.load() == 0) {
                pair_q128 = true;
            } else {
                p.pair = false;
                small_q = q;
            }
        }
    }
    p.g = tc_geometry(a.in, p.pair);
    // Tiles narrower than the epilogue's 64-column chunk (16 or 32 columns, MMA
    // N = 16 / 32) leave room in each ring stage for more of P; they are used
    // only when M fits in one of them, so that the rest of a chunk lies past M
    // (the TMA store clips it), and never for CTA pairs.
    const int opt_tq = g_opt_tile_q.load();
    {
        const int t = opt_tq      ? opt_tq
                      : small_q   ? small_q
                      : pair_q128 ? 128
                                  : choose_tile_q(M, p.g.max_tile_q);
        p.tile_q = t < 64 && (p.pair || M > t) ? 64 : t;
    }
    // 64-row tiles (one CTA each, MMA M = 64), option "half" = 1: they cover
    // N with twice as many CTAs without cutting K.  Measured on GB300 they have
    // not beaten 128-row tiles with K split in two on any skinny shape (BF16
    // 16 x 8192 x 8192: 31.1 against 27.5 us; 16 x 4096 x 8192: 29.7 against
    // 17.4 us), so they run only when forced, and only for one-CTA TMA tiles
    // with FP32 accumulation.
    const int opt_half = g_opt_half.load();
    p.half = opt_half == 1 && !p.pair && p.prod == Producer::Tma && !a.acc16;
    if (p.half) p.g = tc_geometry(a.in, false, true);
    // Pairs of 64-row halves (option "half" = 3): a CTA pair computes 128 rows
    // of N (64 per CTA, MMA M = 128 over the pair) by 128 or 256 columns of M,
    // each CTA loading its own 64 rows of B and half of the tile's A rows, so
    // every B row has one reader and a stage is 16 KB (tile width 128).  The
    // width is 32 or 64 for M up to that, 128 for M <= 128 (width 96 measured
    // level with 128 at M = 80 and 96), else M rounded up to a multiple of 32,
    // or 128, 192 or 256 when option "tile_q" says so: a pair streams in
    // lockstep, so every A row a CTA loads past M would cost time (BF16 192 x
    // 8192 x 8192, graph-replayed on GB300: 30.2 us at width 256, 28.7 at 192).
    // Each epilogue warp stores half the tile's columns; a half that ends
    // inside a 64-column chunk has that chunk stored by the lanes.
    // Automatically (option "half" = 0) for 16-bit inputs with 64 < M <= 256
    // (M <= 64: below) where one-CTA small tiles were chosen above (the pair tiles of 256 rows
    // fill less than a wave) and the pairs of halves fit in one wave; they then
    // run with two MMA issuers (below).  Measured on GB300 against the one-CTA
    // 64- or 128-column tiles with two issuers (paired A/B): BF16 M x 8192 x 8192
    // M = 128 30.7 -> 29.6 us, 192 35.0 -> 33.8, 256 35.1 -> 33.6; K = 16384,
    // M = 128 55.9 -> 54.0, 256 63.2 -> 60.9; FP16 128 x 8192 x 8192 30.0 -> 29.2.
    // FP8 (1-2 % slower), M <= 64 (level) and two waves (6 % slower) keep the
    // one-CTA tiles.
    // They must also fill at least three quarters of the pair slots (64 pairs
    // on 152 SMs were measured); fewer leave SMs idle where split-K fills them.
    const int tq_half = (opt_tq == 128 || opt_tq == 192 || opt_tq == 256) ? opt_tq
                        : M <= 32                                         ? 32
                        : M <= 64                                         ? 64
                        : M <= 128                                        ? 128
                        : M >= 256                                        ? 256
                                    : static_cast<int>((M + 31) / 32 * 32);
    const int64_t pairs_half = ((N + 127) / 128) * ((M + tq_half - 1) / tq_half);
    // For M <= 64 (halves 32 or 64 wide) only without a workspace: then K
    // cannot be split and the one-CTA tiles fill half the SMs (BF16 16 x 8192 x
    // 8192 27.3 -> 25.0 us, 64 x 8192 x 8192 28.4 -> 25.6); with one, the
    // split one-CTA tiles are level at K = 8192 and 6 % faster at K = 16384.
    // (A forced tile width they cannot take, 16 to 64, keeps one-CTA tiles.)
    const bool auto_halves = opt_half == 0 && small_q != 0 && a.in != InKind::E4M3 &&
                             (opt_tq == 0 || opt_tq >= 128) &&
                             (M > 64 || !a.has_scratch) && M <= 256 &&
                             g_opt_issuers.load() != 1 && pairs_half <= a.sms / 2 &&
                             4 * pairs_half >= 3 * (a.sms / 2);
    if ((opt_half == 3 || auto_halves) && p.prod == Producer::Tma && !a.acc16) {
        p.pair = true;
        p.half = true;
        p.tile_q = tq_half;
        p.g = tc_geometry(a.in, true, true);
    }
    const TcGeometry& g = p.g;
    p.load_q = p.tile_q / g.cluster;
    p.tiles_p = (N + g.tile_p - 1) / g.tile_p;
    p.tiles_q = (M + p.tile_q - 1) / p.tile_q;
    p.tiles = p.tiles_p * p.tiles_q;
    p.slots = a.sms / g.cluster;
    const int cap = g_opt_max_ctas.load();
    if (cap > 0 && cap / g.cluster < p.slots) p.slots = cap / g.cluster > 0 ? cap / g.cluster : 1;
    const int64_t tiles = p.tiles, slots = p.slots;
    p.grid = static_cast<int>((tiles < slots ? tiles : slots) * g.cluster);
    // K atoms per stage (option "atoms"; the load-based producer takes one):
    // a stage of two atoms carries twice the K of each row and its MMAs end in
    // one commit instead of two.  The MMA warp's loop costs ~580 cycles per
    // stage, more than a stage's tensor work in tiles up to 128 columns wide
    // (at most 256 cycles per SM), so automatically (option 0) those run two
    // atoms when the ring still holds three stages; wider tiles keep one.
    // Measured on GB300 against the build without the second atom (same box,
    // processes alternating; time ratio old / new): one-CTA 128 x 128 tiles
    // 1024 x 2048 x 4096 1.04, 1024 x 1024 x 8192 1.03; 16-column tiles, K
    // split in two, 16 x 8192 x 8192 1.03; pairs of 64-row halves 128 wide,
    // 128 x 8192 x 8192 1.014.  Halves 256 wide lost (192 / 256 x 8192 x 8192
    // 0.974 / 0.982), and so did 256 x 256 pair tiles on whole waves (2048^3
    // 0.986, 3072^3 0.986, 2048 x 2048 x 8192 0.984).
    {
        const int opt_atoms = g_opt_atoms.load();
        // Pairs of halves other than 128 wide keep one atom even when forced:
        // one such configuration (width 160, two atoms, two issuers, a
        // five-stage ring) faulted on GB300 with no cause found by reading.
        const bool one_atom_halves = p.half && p.pair && p.tile_q != 128;
        if (p.prod == Producer::Tma && !one_atom_halves) {
            if (opt_atoms == 2) {
                p.atoms = 2;
            } else if (opt_atoms == 0 && p.tile_q <= 128) {
                const int rows = g.load_p + p.load_q;
                const int sb2 = (rows * 128 * 2 + 1023) / 1024 * 1024;
                if (g.stage_region / sb2 >= 3) p.atoms = 2;
            }
        }
    }
    p.num_kb = static_cast<int>((K + g.stage_k * p.atoms - 1) / (g.stage_k * p.atoms));
    // Ring: as many stages of this width as the stage region holds (narrow
    // tiles get a deeper ring, i.e. more loads in flight).  The load-based
    // producer's row split assumes the full-width stage.
    {
        const int max_q = g.max_tile_q / g.cluster;
        const int rows = g.load_p + (p.prod == Producer::Loads ? max_q : p.load_q);
        const int sb = (rows * 128 * p.atoms + 1023) / 1024 * 1024;
        int st_count = g.stage_region / sb;
        if (st_count > g.max_stages) st_count = g.max_stages;
        p.stages = st_count;
        p.stage_bytes = sb;
    }

    // Split-K (shape-aware): when one wave of tiles cannot occupy the GPU and
    // there is scratch, cut each tile's K range into pieces so that tiles x
    // pieces fills the SMs; each piece still runs >= 4 K stages.  FP16
    // accumulation (combining pieces would add FP32 sums) and 64-row tiles
    // never split K.
    p.kb_per_split = p.num_kb;
    {
        const int opt = (a.acc16 || p.half) ? 1 : (a.ov_splits >= 0 ? a.ov_splits
                                                                     : g_opt_splits.load());
        int64_t want = 1;
        if (opt >= 2) {
            want = opt;
        } else if (opt == 0 && tiles < slots) {
            want = slots / tiles;
            const int64_t by_k = p.num_kb / 4;
            if (want > by_k) want = by_k;
            if (want > 16) want = 16;
        }
        if (want > p.num_kb) want = p.num_kb;
        // Scratch bytes of a split into `pieces`: counters, then the FP32
        // partial tiles (32-row slices of 256 columns).
        const int64_t slices = 4 * g.cluster;                    // 32-row slices per tile
        const int64_t cnt_bytes = round256(sat_mul(tiles, slices * 4));
        const int64_t room = a.ws_total - p.ws_used;
        auto split_bytes = [&](int64_t pieces) {
            return cnt_bytes + sat_mul(sat_mul(tiles, pieces), slices * 32 * 256 * 4);
        };
        // The no-allocation call's automatic split shrinks to what its fixed
        // array has left after any operand copies (none at all: unsplit).
        if (a.strict && opt == 0) {
            while (want >= 2) {
                const int64_t kb_per = (p.num_kb + want - 1) / want;
                if (fits(split_bytes((p.num_kb + kb_per - 1) / kb_per), room)) break;
                --want;
            }
        }
        if (want >= 2) {
            const int64_t kb_per = (p.num_kb + want - 1) / want;
            const int64_t pieces = (p.num_kb + kb_per - 1) / kb_per;
            const bool fit = fits(split_bytes(pieces), room);
            if (a.strict && pieces >= 2 && !fit) {
                p.status = GEMM_ERR_SCRATCH;
                return p;
            }
            if (pieces >= 2 && a.has_scratch && fit) {
                p.splits = static_cast<int>(pieces);
                p.kb_per_split = static_cast<int>(kb_per);
                p.split_cnt_bytes = cnt_bytes;
                const int64_t units = tiles * pieces;
                p.grid = static_cast<int>((units < slots ? units : slots) * g.cluster);
            }
        }
    }
    // Tail splitting: when the last wave of tiles is partial, cut its tiles
    // into f narrower units along M (f = 2 or 4, tile_q / f still a whole
    // number of epilogue chunks) so that it ends sooner.  Narrow units are
    // L2-bound; measured on GB300, a half-width unit takes ~0.8 of a full
    // tile's time (0.9 for FP8), a quarter-width one ~0.65 (0.8 for FP8).
    // Cutting the tail tiles into K pieces of full width instead, combined
    // through the workspace like split-K, pays a fix-up per tile that long
    // tiles amortise: measured at the power cap against narrowing, two pieces
    // are 2.7 % faster at BF16 4096 x 4096 x 14336 (224 K stages), level at
    // FP16 8192^3 (128: +0.35 % back to back, but 4 % more cycles in a single
    // profiled launch), 1.2 % slower at BF16 4096^3 (64).  So with the tail
    // left to the automatic rule they are taken when the tiles have at least
    // 192 K stages and the doubled tail still fits in one wave; option
    // "tail_k" = f forces f pieces.
    p.full_units = tiles * p.splits;
    p.tail_kb_per = p.num_kb;
    {
        const int opt_tail = g_opt_tail.load();
        const int64_t waves = tiles / slots, rem = tiles % slots;
        const int min_w = 128 / os;  // one epilogue chunk
        const int64_t slices = 4 * g.cluster;
        const int64_t cnt_bytes = ((rem * slices * 4 + 255) / 256) * 256;
        const int64_t room = a.ws_total - p.ws_used;
        int f = 1;
        bool ksplit = false;
        int64_t kb_per_t = p.num_kb;
        auto narrow_ok = [&](int c) {
            return p.tile_q % c == 0 && (p.tile_q / c) % min_w == 0 && p.tile_q / c >= 64;
        };
        if (p.splits == 1 && rem > 0 && opt_tail != 1 && !(p.half && p.pair)) {
            if (opt_tail == 2 || opt_tail == 4) {
                f = narrow_ok(opt_tail) ? opt_tail : 1;
            } else {
                const bool fp8 = a.in == InKind::E4M3;
                double best = 1.0;
                for (int cand : {2, 4}) {
                    if (!narrow_ok(cand)) continue;
                    const double unit_cost = cand == 2 ? (fp8 ? 0.9 : 0.8) : (fp8 ? 0.8 : 0.65);
                    const double t =
                        static_cast<double>((cand * rem + slots - 1) / slots) * unit_cost;
                    if (t < best - 0.02) {
                        best = t;
                        f = cand;
                    }
                }
            }
            int want_k = g_opt_tail_k.load();
            // (192 one-atom stages: K >= 12288 for 16-bit inputs, 24576 for e4m3)
            if (want_k == 0 && opt_tail == 0 && p.num_kb * p.atoms >= 192 && 2 * rem <= slots)
                want_k = 2;
            if (want_k >= 2 && !a.acc16 && !p.half && a.has_scratch) {
                const int64_t kb_per = (p.num_kb + want_k - 1) / want_k;
                const int64_t pieces = (p.num_kb + kb_per - 1) / kb_per;
                const int64_t need = cnt_bytes + rem * pieces * slices * 32 * 256 * 4;
                if (pieces >= 2 && fits(need, room)) {
                    f = static_cast<int>(pieces);
                    ksplit = true;
                    kb_per_t = kb_per;
                }
            }
        }
        if (f > 1) {
            p.tail_f = f;
            p.tail_ksplit = ksplit;
            p.full_units = waves * slots;
            if (ksplit) {
                p.tail_kb_per = static_cast<int>(kb_per_t);
                p.tail_cnt_bytes = cnt_bytes;
            }
            const int64_t units = p.full_units + (tiles - p.full_units) * f;
            p.grid = static_cast<int>((units < slots ? units : slots) * g.cluster);
        }
    }
    // Several MMA-issuing warps (TcCfg NI): one-CTA TMA tiles without K pieces
    // whose NI accumulators (and the epilogue's 64-column chunk reads past the
    // last one) fit in one 256-column TMEM buffer.  Narrow skinny tiles are
    // bound by the MMA issue rate, so automatically (option "issuers" = 0) two
    // run where the tiles are at most 64 columns wide and fit in one wave.
    // Measured on GB300 (paired A/B, 10-launch blocks alternating over 12
    // rounds): BF16 128 x 8192 x 8192 32.8 -> 30.5 us, FP16 the same shape 32.8
    // -> 30.3, FP8 18.9 -> 17.4, BF16 128 x 8192 x 16384 59.5 -> 56.0, 64 x 14336
    // x 4096 23.9 -> 23.0; with 128-column tiles (M = 192, 256) 1.2-1.4 %
    // slower, so not there.
    const int opt_iss = g_opt_issuers.load();
    auto issuers_fit = [&](int ni) {
        return (ni - 1) * p.tile_q + (p.tile_q > 64 ? p.tile_q : 64) <= 256;
    };
    if (!p.pair && !p.half && p.prod == Producer::Tma && !a.acc16 && p.splits == 1 &&
        !p.tail_ksplit) {
        if (opt_iss == 2) {
            if (issuers_fit(2)) p.issuers = 2;
        } else if (opt_iss == 0 && p.tile_q <= 64 && p.tiles <= p.slots) {
            p.issuers = 2;
        }
    }
    // ... and for pairs of 64-row halves (two accumulators of tile_q / 2
    // columns per CTA): automatically whenever they run, since without two
    // issuers they measured slower than one-CTA tiles on every skinny shape
    // tried (BF16 128 x 8192 x 8192: 35.0 against 30.7 us)
    if (opt_iss != 1 && p.pair && p.half && p.prod == Producer::Tma && !a.acc16) p.issuers = 2;
    // Two issuers get an even ring depth, so that every ring slot is always
    // consumed (and released) by the same issuer.  The three unspecified launch
    // failures seen on GB300 with several issuers (no cause found by reading)
    // all ran odd rings, where consecutive uses of a slot alternate between the
    // issuers and both commit to its barrier: five stages with two K atoms
    // (twice), nine with one atom and split K.  The stage given up costs up to
    // 3 % (pairs of halves 192 wide, 9 -> 8 stages: 28.9 -> 29.9 us), which the
    // ring wins back below where it can.
    if (p.issuers > 1 && (p.stages & 1) && p.stages > 2) --p.stages;
    // Where every CTA (or pair) runs one unit, its epilogue starts only after
    // the ring has drained, so the ring may run on over the epilogue's staging
    // area (224 KB instead of 192).  Pairs of 64-row halves gain from the
    // loads in flight (graph-replayed BF16 on GB300, 192 KB -> 224 KB: width
    // 192 29.9 -> 28.5 us, 160 28.0 -> 27.6, 224 30.5 -> 29.0, 192 x 8192 x
    // 16384 54.2 -> 51.6); the split one-CTA 16-wide tiles (25.6 -> 26.0) and
    // 2048^3 pairs (15.3 -> 15.6) lost, so only pairs of halves take it.
    if (p.prod == Producer::Tma && p.pair && p.half && p.tail_f == 1 && !p.tail_ksplit &&
        p.tiles * p.splits <= p.slots) {
        int st = (g.stage_region + g.epi_region) / p.stage_bytes;
        if (st > g.max_stages) st = g.max_stages;
        if (p.issuers > 1 && (st & 1) && st > 2) --st;
        if (st > p.stages) {
            p.stages = st;
            p.ring_epi = true;
        }
    }
    return p;
}

// The planning half of gemm_tn.  Under the no-allocation call's rules
// (a.strict) operand copies share the fixed array with the split: a forced
// split that does not fit beside the copies runs without them (the load-based
// producer reads the unaligned operand in place) and fails with
// GEMM_ERR_SCRATCH only when it does not fit the array on its own.
TnPlan plan_tn(const TnPlanIn& a) {
    TnPlan p = plan_tn_once(a);
    if (a.strict && p.status == GEMM_ERR_SCRATCH && (p.copy_a || p.copy_b)) {
        TnPlanIn b = a;
        b.no_copy = true;
        p = plan_tn_once(b);
    }
    return p;
}

// 2D tensor map over a matrix with `outer` rows of `inner` contiguous elements
// and a row pitch of `pitch_bytes`, copied in boxes of box_inner x box_outer
// with 128-byte swizzling and zero fill outside the matrix.
CUresult encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* ptr, int64_t inner,
                   int64_t outer, int64_t pitch_bytes, uint32_t box_inner, uint32_t box_outer) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch_bytes)};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return g_encode(map, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// `ov`, when given, replaces the registered workspace and the "splits" option:
// the call splits K with that scratch (ov->splits: 0 by the automatic rule,
// >= 2 forced, 1 never) and fails with GEMM_ERR_SCRATCH when the split it
// chooses needs more than ov->bytes.  Every public entry point but the
// no-allocation one passes nullptr.
// Argument checks of a TN call, in the order the header documents; nothing
// here touches the device.
int validate_tn(InKind in, bool out_f32, int64_t M, int64_t N, int64_t K, const void* A,
                int64_t lda, const void* B, int64_t ldb, const void* C, int64_t ldc) {
    const int es = in == InKind::E4M3 ? 1 : 2;
    const int os = out_f32 ? 4 : 2;  // output element size
    if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return GEMM_ERR_INVALID_DIM;
    const int64_t kmin = K > 1 ? K : 1;
    if (lda < kmin || ldb < kmin || ldc < (M > 1 ? M : 1) || lda > kMaxLd || ldb > kMaxLd ||
        ldc > kMaxLd)
        return GEMM_ERR_INVALID_LD;
    if ((M > 0 && K > 0 && !A) || (N > 0 && K > 0 && !B) || (M > 0 && N > 0 && !C))
        return GEMM_ERR_NULL_PTR;
    if (!aligned(A, es) || !aligned(B, es) || !aligned(C, os)) return GEMM_ERR_MISALIGNED;
    return GEMM_OK;
}

int gemm_tn(InKind in, bool out_f32, int64_t M, int64_t N, int64_t K, const void* A,
            int64_t lda, const void* B, int64_t ldb, float scale, void* C, int64_t ldc,
            void* stream_v, const ScratchOverride* ov = nullptr, bool acc16 = false) {
    const int es = in == InKind::E4M3 ? 1 : 2;
    const int os = out_f32 ? 4 : 2;  // output element size
    int st = validate_tn(in, out_f32, M, N, K, A, lda, B, ldb, C, ldc);
    if (st != GEMM_OK) return st;
    const DeviceInfo* dev = nullptr;
    st = current_device(&dev);
    if (st != GEMM_OK) return st;
    if (M == 0 || N == 0) return GEMM_OK;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    cudaError_t e;
    if (K == 0) {
        e = zero_fill_launch(C, N, M, ldc, os, stream);
        return e == cudaSuccess ? GEMM_OK : fail_cuda(e);
    }

    // Path choice.  TMA needs 16-byte-aligned bases and row pitches; operands
    // that miss it are repacked into the workspace when there is one (below)
    // or read by the load-based producer, and a C that misses it is written by
    // the epilogue's row-wise stores.  Option "path" = 1 forces the CUDA-core
    // kernel (a second, independent implementation).
    if (g_opt_path.load() == 1 && !acc16) {
        e = tn_fallback_launch(in, out_f32, M, N, K, A, lda, B, ldb, scale, C, ldc, stream);
        return e == cudaSuccess ? GEMM_OK : fail_cuda(e);
    }
    const int64_t lim = 1LL << 40;
    bool a_tma = aligned(A, 16) && (lda * es) % 16 == 0 && lda * es < lim;
    bool b_tma = aligned(B, 16) && (ldb * es) % 16 == 0 && ldb * es < lim;
    const bool c_tma = aligned(C, 16) && (ldc * os) % 16 == 0 && ldc * os < lim;

    // Scratch: the caller's workspace (registered, or the override).
    char* ws_base = nullptr;
    int64_t ws_total = 0;
    char* cnt_base = nullptr;  // the two fixed split-counter sets, if this scratch has them
    std::atomic<unsigned int>* cnt_parity = nullptr;
    if (ov) {
        ws_base = static_cast<char*>(ov->ptr);
        ws_total = ov->bytes;
        cnt_base = static_cast<char*>(ov->counters);
        cnt_parity = ov->parity;
    } else {
        std::lock_guard<std::mutex> lock(g_mutex);
        ws_base = static_cast<char*>(dev->workspace);
        ws_total = dev->workspace_bytes;
        if (ws_base && ws_total >= kSplitCounterBytes) {
            cnt_base = ws_base;
            cnt_parity = &g_cnt_parity[dev - g_devices];
            ws_base += kSplitCounterBytes;
            ws_total -= kSplitCounterBytes;
        }
    }
    // Counters for a split launch: a fixed set when there is one large enough
    // (the launch zeroes the other set for the next split launch), otherwise
    // `fallback` in the scratch, zeroed on the stream first.
    auto take_counters = [&](TcParams& prm, int64_t words, char* fallback,
                             int64_t fallback_bytes) {
        if (cnt_base && cnt_parity && words <= kCounterSetWords) {
            const unsigned int p = cnt_parity->fetch_xor(1u) & 1u;
            prm.ws_counters = reinterpret_cast<unsigned int*>(cnt_base + p * kCounterSetWords * 4);
            prm.ws_clear =
                reinterpret_cast<unsigned int*>(cnt_base + (p ^ 1u) * kCounterSetWords * 4);
            prm.clear_words = static_cast<int32_t>(kCounterSetWords);
            return cudaSuccess;
        }
        prm.ws_counters = reinterpret_cast<unsigned int*>(fallback);
        prm.ws_clear = nullptr;
        prm.clear_words = 0;
        return cudaMemsetAsync(fallback, 0, static_cast<size_t>(fallback_bytes), stream);
    };
    // Plan the call (pure: shapes, alignment, scratch, options, device), then
    // carry it out.
    TnPlanIn pin;
    pin.in = in;
    pin.out_f32 = out_f32;
    pin.acc16 = acc16;
    pin.M = M;
    pin.N = N;
    pin.K = K;
    pin.a_tma = a_tma;
    pin.b_tma = b_tma;
    pin.c_tma = c_tma;
    pin.a_al128 = aligned(A, 128) && (lda * es) % 128 == 0;
    pin.b_al128 = aligned(B, 128) && (ldb * es) % 128 == 0;
    pin.has_scratch = ws_base != nullptr;
    pin.ws_total = ws_base ? ws_total : 0;
    pin.ov_splits = ov ? ov->splits : -1;
    pin.strict = ov && ov->strict;
    pin.sms = dev->sms;
    const TnPlan pl = plan_tn(pin);
    if (pl.status != GEMM_OK) return pl.status;

    // Repacks into the scratch: 128-byte-aligned rows of pitch pl.dp.
    if (pl.copy_a || pl.copy_b) {
        const int64_t rb = K * es;  // row bytes
        const int64_t need_a = pl.copy_a ? (M * pl.dp + 255) / 256 * 256 : 0;
        if (pl.copy_a) {
            e = repack_rows_launch(A, lda * es, ws_base, pl.dp, M, rb, stream);
            if (e != cudaSuccess) return fail_cuda(e);
            A = ws_base;
            lda = pl.dp / es;
        }
        if (pl.copy_b) {
            e = repack_rows_launch(B, ldb * es, ws_base + need_a, pl.dp, N, rb, stream);
            if (e != cudaSuccess) return fail_cuda(e);
            B = ws_base + need_a;
            ldb = pl.dp / es;
        }
    }
    const Producer prod = pl.prod;
    const bool pair = pl.pair;
    const TcGeometry& g = pl.g;
    TcLaunch L;
    std::memset(&L, 0, sizeof(L));
    L.half = pl.half;
    L.issuers = pl.issuers;
    const CUtensorMapDataType in_dt = in == InKind::F16    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                      : in == InKind::BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                           : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const CUtensorMapDataType out_dt = out_f32            ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                       : in == InKind::F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                           : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    // P = B: N rows of K contiguous elements.  Q = A: M rows of K.  Out = C: N rows of M.
    const int tile_q = pl.tile_q, load_q = pl.load_q;
    CUresult r = CUDA_SUCCESS;
    if (prod == Producer::Tma) {
        r = encode_2d(&L.map_p, in_dt, B, K, N, ldb * es, g.stage_k, g.load_p);
        if (r == CUDA_SUCCESS)
            r = encode_2d(&L.map_q, in_dt, A, K, M, lda * es, g.stage_k, load_q);
    }
    // One staged chunk is one 128-byte row per accumulator row of an
    // epilogue warp: a box of 128 / os columns x 32 rows (16 for 64-row tiles).
    if (r == CUDA_SUCCESS && c_tma)
        r = encode_2d(&L.map_out, out_dt, C, M, N, ldc * os, 128 / os,
                      (L.half && !pair) ? 16 : 32);
    if (r != CUDA_SUCCESS) return fail_cuda(cudaErrorInvalidValue);

    const int64_t tiles_p = pl.tiles_p, tiles_q = pl.tiles_q, tiles = pl.tiles;
    L.prm.rows_p = static_cast<int32_t>(N);
    L.prm.rows_q = static_cast<int32_t>(M);
    L.prm.num_kb = pl.num_kb;
    L.prm.tiles_p = static_cast<int32_t>(tiles_p);
    L.prm.tiles_q = static_cast<int32_t>(tiles_q);
    L.prm.group = g_opt_group.load() > 0 ? g_opt_group.load() : kDefaultGroup;
    L.prm.k_snake = g_opt_k_snake.load();
    // K rotation (option "k_rotate"): automatically for the unsplit skinny
    // plans that run two MMA issuers (one-CTA tiles up to 64 wide in one wave,
    // pairs of 64-row halves), whose units all stream their own rows of B at
    // once.  Measured on GB300 (graph-replayed BF16, paired A/B, in order ->
    // rotated): 128 x 8192 x 8192 26.65 -> 26.18 us, 192x 29.36 -> 28.78, 256x
    // 31.42 -> 31.00, 64 x 14336 x 4096 21.91 -> 21.36, 256 x 8192 x 16384
    // 56.89 -> 56.14; split plans level (16 x 8192 x 8192) or slower (1024 x
    // 1024 x 8192 pairs, 19.64 -> 20.21).
    {
        const int opt_rot = g_opt_k_rotate.load();
        L.prm.k_rotate =
            opt_rot == 2 || (opt_rot == 0 && pl.issuers > 1 && pl.splits == 1 && !pl.tail_ksplit)
                ? 1
                : 0;
    }
    L.prm.band_snake = g_opt_band_snake.load();
    L.prm.scale = scale;
    L.prm.timeout_ns = static_cast<uint64_t>(g_opt_timeout_ns.load());
    L.prm.watchdog = dev->watchdog;
    L.prm.out = C;
    L.prm.ld_out = ldc;
    L.prm.direct_store = c_tma ? 0 : 1;
    L.prm.k_bytes = K * es;
    L.prm.l2_hints = g_opt_l2hints.load();
    L.prm.tile_q = tile_q;
    const uint32_t d_format = acc16 ? 0u : 1u;
    L.prm.acc16 = acc16 ? 1 : 0;
    L.prm.idesc = make_idesc(g.format, static_cast<uint32_t>(g.mma_m), static_cast<uint32_t>(tile_q),
                             d_format);
    L.prm.stage_tx_bytes = static_cast<uint32_t>((g.load_p + load_q) * 128 * pl.atoms);
    L.prm.atoms = pl.atoms;
    L.prm.ring_epi = pl.ring_epi ? 1 : 0;
    L.prm.q_atom_bytes = static_cast<uint32_t>(load_q * 128);
    L.prm.stages = pl.stages;
    L.prm.stage_bytes = static_cast<uint32_t>(pl.stage_bytes);
    L.prm.p_ptr = B;
    L.prm.q_ptr = A;
    L.prm.ld_p_bytes = ldb * es;
    L.prm.ld_q_bytes = lda * es;
    L.grid = pl.grid;
    L.stream = stream;

    // Split-K: partial sums after the counters in the scratch.
    char* ws = ws_base ? ws_base + pl.ws_used : nullptr;
    const int64_t slices = 4 * g.cluster;  // 32-row slices per tile
    L.prm.splits = pl.splits;
    L.prm.kb_per_split = pl.kb_per_split;
    if (pl.splits > 1) {
        L.prm.ws_partials = reinterpret_cast<float*>(ws + pl.split_cnt_bytes);
        e = take_counters(L.prm, tiles * slices, ws, pl.split_cnt_bytes);
        if (e != cudaSuccess) return fail_cuda(e);
    }
    // The last wave: narrower units (a tail tensor map, instruction descriptor
    // and stage byte count of their own) or K pieces through the scratch.
    L.prm.full_units = pl.full_units;
    L.prm.tail_f = pl.tail_f;
    L.prm.idesc_tail = L.prm.idesc;
    L.prm.stage_tx_tail = L.prm.stage_tx_bytes;
    L.prm.tail_ksplit = pl.tail_ksplit ? 1 : 0;
    L.prm.tail_kb_per = pl.tail_kb_per;
    if (pl.tail_f > 1 && pl.tail_ksplit) {
        const int64_t rem = tiles % pl.slots;
        L.prm.ws_partials = reinterpret_cast<float*>(ws + pl.tail_cnt_bytes);
        e = take_counters(L.prm, rem * slices, ws, pl.tail_cnt_bytes);
        if (e != cudaSuccess) return fail_cuda(e);
    } else if (pl.tail_f > 1) {
        const int width = tile_q / pl.tail_f;
        const int load_qt = width / g.cluster;
        if (prod == Producer::Tma) {
            r = encode_2d(&L.map_q_tail, in_dt, A, K, M, lda * es, g.stage_k, load_qt);
            if (r != CUDA_SUCCESS) return fail_cuda(cudaErrorInvalidValue);
        }
        L.prm.idesc_tail = make_idesc(g.format, static_cast<uint32_t>(g.mma_m),
                                      static_cast<uint32_t>(width), d_format);
        L.prm.stage_tx_tail = static_cast<uint32_t>((g.load_p + load_qt) * 128 * pl.atoms);
    }
    if (std::getenv("GEMM_DEBUG"))
        std::fprintf(stderr,
                     "[gemm] tn in=%d M=%lld N=%lld K=%lld pair=%d producer=%d direct_store=%d "
                     "splits=%d tile_q=%d tail=%d ktail=%d stages=%d tiles=%lldx%lld grid=%d "
                     "half=%d issuers=%d atoms=%d k_rotate=%d ring_epi=%d\n",
                     int(in), (long long)M, (long long)N, (long long)K, int(pair), int(prod),
                     L.prm.direct_store, L.prm.splits, L.prm.tile_q, L.prm.tail_f,
                     L.prm.tail_ksplit, L.prm.stages,
                     (long long)tiles_q, (long long)tiles_p, L.grid, int(L.half), L.issuers,
                     L.prm.atoms, L.prm.k_rotate, L.prm.ring_epi);
    e = tc_launch(in, pair, prod, out_f32, L);
    return e == cudaSuccess ? GEMM_OK : fail_cuda(e);
}

}  // namespace

namespace gb300 {
int tn_validate(InKind in, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                const void* B, int64_t ldb, const void* C, int64_t ldc) {
    return validate_tn(in, false, M, N, K, A, lda, B, ldb, C, ldc);
}

int tn_record_cuda_error(cudaError_t e) { return fail_cuda(e); }

int gemm_tn_with_scratch(InKind in, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                         const void* B, int64_t ldb, void* C, int64_t ldc, void* stream,
                         const ScratchOverride& ov) {
    return gemm_tn(in, false, M, N, K, A, lda, B, ldb, 1.0f, C, ldc, stream, &ov);
}
}  // namespace gb300

extern "C" {

int gemm_f32(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda, const float* B,
             int64_t ldb, float* C, int64_t ldc, void* stream_v) {
    if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return GEMM_ERR_INVALID_DIM;
    const int64_t nmin = N > 1 ? N : 1;
    if (lda < (K > 1 ? K : 1) || ldb < nmin || ldc < nmin || lda > kMaxLd || ldb > kMaxLd ||
        ldc > kMaxLd)
        return GEMM_ERR_INVALID_LD;
    if ((M > 0 && K > 0 && !A) || (N > 0 && K > 0 && !B) || (M > 0 && N > 0 && !C))
        return GEMM_ERR_NULL_PTR;
    if (!aligned(A, 4) || !aligned(B, 4) || !aligned(C, 4)) return GEMM_ERR_MISALIGNED;
    const DeviceInfo* dev = nullptr;
    int st = current_device(&dev);
    if (st != GEMM_OK) return st;
    if (M == 0 || N == 0) return GEMM_OK;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    cudaError_t e = K == 0 ? zero_fill_launch(C, M, N, ldc, 4, stream)
                           : f32_launch(M, N, K, A, lda, B, ldb, C, ldc, stream,
                                        g_opt_f32_tail.load(), g_opt_f32_ktail.load());
    return e == cudaSuccess ? GEMM_OK : fail_cuda(e);
}

int gemm_f16_tn(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                int64_t ldb, void* C, int64_t ldc, void* stream) {
    return gemm_tn(InKind::F16, false, M, N, K, A, lda, B, ldb, 1.0f, C, ldc, stream);
}

int gemm_f16_tn_acc16(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                      int64_t ldb, void* C, int64_t ldc, void* stream) {
    return gemm_tn(InKind::F16, false, M, N, K, A, lda, B, ldb, 1.0f, C, ldc, stream, nullptr,
                   true);
}

int gemm_bf16_tn(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                 int64_t ldb, void* C, int64_t ldc, void* stream) {
    return gemm_tn(InKind::BF16, false, M, N, K, A, lda, B, ldb, 1.0f, C, ldc, stream);
}

int gemm_fp8_tn(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                int64_t ldb, float scale_a, float scale_b, void* C, int64_t ldc, void* stream) {
    const float scale = scale_a * scale_b;  // one FP32 product, applied in the epilogue
    return gemm_tn(InKind::E4M3, false, M, N, K, A, lda, B, ldb, scale, C, ldc, stream);
}

int gemm_fp8_tn_f32(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                    int64_t ldb, float scale_a, float scale_b, float* C, int64_t ldc,
                    void* stream) {
    const float scale = scale_a * scale_b;
    return gemm_tn(InKind::E4M3, true, M, N, K, A, lda, B, ldb, scale, C, ldc, stream);
}

// The tensor-core FP32 path: three-way BF16 splits of A and B (split_f32.cu)
// in the caller's workspace, then one BF16 TN GEMM with FP32 output over the
// six K-segments.  Row-major C = A B is the TN product with the roles of the
// operands swapped: TN "M" = N with P rows from the split of B, TN "N" = M
// with Q rows from the split of A, and C[m * ldc + n] its column-major output.
int64_t gemm_f32_bf16x6_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return 0;
    const int64_t row = 6 * ((K + 63) / 64 * 64) * 2;  // bytes of one split row
    return kSplitCounterBytes + round256(sat_mul(M, row)) + round256(sat_mul(N, row));
}

int gemm_f32_bf16x6(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda, const float* B,
                    int64_t ldb, float* C, int64_t ldc, void* stream_v) {
    if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return GEMM_ERR_INVALID_DIM;
    const int64_t kp = (K + 63) / 64 * 64;
    if (6 * kp > kMaxDim) return GEMM_ERR_INVALID_DIM;
    const int64_t nmin = N > 1 ? N : 1;
    if (lda < (K > 1 ? K : 1) || ldb < nmin || ldc < nmin || lda > kMaxLd || ldb > kMaxLd ||
        ldc > kMaxLd)
        return GEMM_ERR_INVALID_LD;
    if ((M > 0 && K > 0 && !A) || (N > 0 && K > 0 && !B) || (M > 0 && N > 0 && !C))
        return GEMM_ERR_NULL_PTR;
    if (!aligned(A, 4) || !aligned(B, 4) || !aligned(C, 4)) return GEMM_ERR_MISALIGNED;
    const DeviceInfo* dev = nullptr;
    int st = current_device(&dev);
    if (st != GEMM_OK) return st;
    if (M == 0 || N == 0) return GEMM_OK;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    cudaError_t e;
    if (K == 0) {
        e = zero_fill_launch(C, M, N, ldc, 4, stream);
        return e == cudaSuccess ? GEMM_OK : fail_cuda(e);
    }
    char* ws = nullptr;
    int64_t ws_bytes = 0;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        ws = static_cast<char*>(dev->workspace);
        ws_bytes = dev->workspace_bytes;
    }
    const int64_t need = gemm_f32_bf16x6_workspace_bytes(M, N, K);
    if (!ws || !fits(need, ws_bytes)) return GEMM_ERR_WORKSPACE;
    const int64_t a_bytes = round256(sat_mul(M, 6 * kp * 2));
    char* sa = ws + kSplitCounterBytes;  // M rows of 6 kp BF16: the split of A
    char* sb = sa + a_bytes;             // N rows of 6 kp BF16: the split of B, transposed
    e = f32_split_rows_launch(A, lda, M, K, kp, sa, dev->sms, stream);
    if (e == cudaSuccess) e = f32_split_cols_launch(B, ldb, K, N, kp, sb, dev->sms, stream);
    if (e != cudaSuccess) return fail_cuda(e);
    // What is left of the workspace serves split-K where it fits; otherwise
    // the GEMM runs unsplit.
    ScratchOverride ov{ws + need, ws_bytes - need, 0, 0};
    ov.counters = ws;  // the workspace's own counter sets
    ov.parity = &g_cnt_parity[dev - g_devices];
    return gemm_tn(InKind::BF16, true, N, M, 6 * kp, sb, 6 * kp, sa, 6 * kp, 1.0f, C, ldc,
                   stream, &ov);
}

int gemm_tn_plan(int kind, int64_t M, int64_t N, int64_t K, int flags, int64_t workspace_bytes,
                 int sms, int64_t* out, int nout) {
    if (kind < GEMM_PLAN_F16 || kind > GEMM_PLAN_FP8_F32OUT || !out || nout < GEMM_PLAN_FIELDS)
        return GEMM_ERR_INVALID_OPTION;
    if (M <= 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim || sms <= 0 ||
        workspace_bytes < 0)
        return GEMM_ERR_INVALID_DIM;
    TnPlanIn pin;
    pin.in = kind == GEMM_PLAN_BF16 ? InKind::BF16
             : (kind == GEMM_PLAN_FP8 || kind == GEMM_PLAN_FP8_F32OUT) ? InKind::E4M3
                                                                       : InKind::F16;
    pin.out_f32 = kind == GEMM_PLAN_FP8_F32OUT;
    pin.acc16 = kind == GEMM_PLAN_F16_ACC16;
    pin.M = M;
    pin.N = N;
    pin.K = K;
    pin.a_tma = (flags & GEMM_PLAN_A_TMA) != 0;
    pin.b_tma = (flags & GEMM_PLAN_B_TMA) != 0;
    pin.c_tma = (flags & GEMM_PLAN_C_TMA) != 0;
    pin.a_al128 = (flags & GEMM_PLAN_A_128) != 0;
    pin.b_al128 = (flags & GEMM_PLAN_B_128) != 0;
    // as gemm_tn sees a registered workspace (or the no-allocation array): the
    // counter sets come off the top
    pin.has_scratch = workspace_bytes > 0;
    pin.ws_total = workspace_bytes >= kSplitCounterBytes ? workspace_bytes - kSplitCounterBytes
                                                         : workspace_bytes;
    const bool noalloc = (flags & GEMM_PLAN_NOALLOC) != 0;
    pin.ov_splits = noalloc ? g_opt_splits.load() : -1;
    pin.strict = noalloc;
    pin.sms = sms;
    const TnPlan pl = plan_tn(pin);
    const int64_t v[GEMM_PLAN_FIELDS] = {pl.status,
                                         pl.pair,
                                         static_cast<int64_t>(pl.prod),
                                         pl.tile_q,
                                         pl.half,
                                         pl.splits,
                                         pl.tail_f,
                                         pl.tail_ksplit,
                                         pl.stages,
                                         pl.grid,
                                         pl.copy_a,
                                         pl.copy_b,
                                         pl.tiles_p,
                                         pl.tiles_q,
                                         pl.kb_per_split,
                                         pl.tail_kb_per,
                                         pl.stage_bytes,
                                         pl.issuers,
                                         pl.atoms,
                                         pl.ring_epi ? 1 : 0};
    for (int i = 0; i < GEMM_PLAN_FIELDS; ++i) out[i] = v[i];
    return GEMM_OK;
}

const char* gemm_status_string(int status) {
    switch (status) {
        case GEMM_OK: return "ok";
        case GEMM_ERR_INVALID_DIM: return "invalid dimension (negative or above 2^31-1)";
        case GEMM_ERR_INVALID_LD: return "leading dimension below its minimum or above 2^48";
        case GEMM_ERR_NULL_PTR: return "null matrix pointer with a nonzero extent";
        case GEMM_ERR_MISALIGNED: return "pointer not aligned to its element size";
        case GEMM_ERR_UNSUPPORTED_DEVICE: return "current device is not compute capability 10.3";
        case GEMM_ERR_LAUNCH:
            std::snprintf(t_status_buf, sizeof(t_status_buf), "CUDA error: %s",
                          cudaGetErrorString(t_last_cuda_error));
            return t_status_buf;
        case GEMM_ERR_TIMEOUT: return "a device-side wait ran out of time";
        case GEMM_ERR_INVALID_OPTION: return "unknown option or value out of range";
        case GEMM_ERR_SCRATCH:
            return "the call needs more split-K scratch than the library's static array holds";
        case GEMM_ERR_WORKSPACE:
            return "the call needs a registered workspace of at least its "
                   "gemm_f32_bf16x6_workspace_bytes";
        default: return "unknown status";
    }
}

int gemm_read_watchdog(int reset) {
    const DeviceInfo* dev = nullptr;
    int st = current_device(&dev);
    if (st != GEMM_OK) return st;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail_cuda(e);
    unsigned int word = 0;
    e = cudaMemcpy(&word, dev->watchdog, sizeof(word), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail_cuda(e);
    if (reset) {
        e = cudaMemset(dev->watchdog, 0, sizeof(word));
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return fail_cuda(e);
    }
    return word ? GEMM_ERR_TIMEOUT : GEMM_OK;
}

int gemm_set_option(const char* name, int64_t value) {
    if (!name) return GEMM_ERR_INVALID_OPTION;
    if (!std::strcmp(name, "pair")) {
        if (value < -1 || value > 1) return GEMM_ERR_INVALID_OPTION;
        g_opt_pair.store(static_cast<int>(value));
    } else if (!std::strcmp(name, "group")) {
        if (value < 0 || value > 64) return GEMM_ERR_INVALID_OPTION;
        g_opt_group.store(static_cast<int>(value));
    } else if (!std::strcmp(name, "k_snake")) {
        if (value < 0 || value > 1) return GEMM_ERR_INVALID_OPTION;
        g_opt_k_snake.store(static_cast<int>(value));
    } else if (!std::strcmp(name, "k_rotate")) {
        if (value < 0 || value > 2) return GEMM_ERR_INVALID_OPTION;
        g_opt_k_rotate.store(static_cast<int>(value));
    } else if (!std::strcmp(name, "band_snake")) {
        if (value < 0 || value > 1) return GEMM_ERR_INVALID_OPTION;
        g_opt_band_snake.store(static_cast<int>(value));
    } else if (!std::strcmp(name, "path")) {
        if (value < 0 || value > 2) return GEMM_ERR_INVALID_OPTION;
        g_opt_path.store(static_cast<int>(value));
    } else if (!std::strcmp(name, "timeout_ns")) {
        if (value < 1000000LL || value > 60000000000LL) return GEMM_ERR_INVALID_OPTION;
        g_opt_timeout_ns.store(value);
    } else if (!std::strcmp(name, "splits")) {
        if (value < 0 || value > 64) return GEMM_ERR_INVALID_OPTION;
        g_opt_splits.store(static_cast<int>(value));
    } else if (!std::strcmp(name, "tile_q")) {
        if (!(value == 0 || value == 16 || value == 32 || value == 64 || value == 128 ||
              value == 192 || value == 256))
            return GEMM_ERR_INVALID_OPTION;
        g_opt_tile_q.store(static_cast<int>(value));
    } else if (!std::strcmp(name, "tail_k")) {
        if (value < 0 || value > 8 || value == 1) return GEMM_ERR_INVALID_OPTION;
        g_opt_tail_k.store(static_cast<int>(value));
    } else if (!std::strcmp(name, "tail")) {
        if (!(value == 0 || value == 1 || value == 2 || value == 4)) return GEMM_ERR_INVALID_OPTION;
        g_opt_tail.store(static_cast<int>(value));
    } else if (!std::strcmp(name, "l2_hints")) {
        if (value < 0 || value > 2) return GEMM_ERR_INVALID_OPTION;
        g_opt_l2hints.store(static_cast<int>(value));
    } else if (!std::strcmp(name, "f32_ktail")) {
        if (value < 0 || value > 15) return GEMM_ERR_INVALID_OPTION;
        g_opt_f32_ktail.store(static_cast<int>(value));
    } else if (!std::strcmp(name, "f32_tail")) {
        if (value < 0 || value > 3) return GEMM_ERR_INVALID_OPTION;
        g_opt_f32_tail.store(static_cast<int>(value));
    } else if (!std::strcmp(name, "repack")) {
        if (value < 0 || value > 1) return GEMM_ERR_INVALID_OPTION;
        g_opt_repack.store(static_cast<int>(value));
    } else if (!std::strcmp(name, "issuers")) {
        if (value < 0 || value > 2) return GEMM_ERR_INVALID_OPTION;
        g_opt_issuers.store(static_cast<int>(value));
    } else if (!std::strcmp(name, "half")) {
        if (value < 0 || value > 3) return GEMM_ERR_INVALID_OPTION;
        g_opt_half.store(static_cast<int>(value));
    } else if (!std::strcmp(name, "atoms")) {
        if (value < 0 || value > 2) return GEMM_ERR_INVALID_OPTION;
        g_opt_atoms.store(static_cast<int>(value));
    } else if (!std::strcmp(name, "max_ctas")) {
        if (value < 0 || value > 1 << 20) return GEMM_ERR_INVALID_OPTION;
        g_opt_max_ctas.store(static_cast<int>(value));
    } else {
        return GEMM_ERR_INVALID_OPTION;
    }
    return GEMM_OK;
}

int gemm_set_workspace(void* ptr, int64_t bytes) {
    if (bytes < 0 || (ptr == nullptr && bytes != 0)) return GEMM_ERR_INVALID_DIM;
    if (ptr && !aligned(ptr, 256)) return GEMM_ERR_MISALIGNED;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e);
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (ptr && bytes >= kSplitCounterBytes) {
        // The split counters at the start of the workspace start at zero; the
        // device must hold them before any stream uses the workspace.
        e = cudaMemset(ptr, 0, static_cast<size_t>(kSplitCounterBytes));
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return fail_cuda(e);
    }
    g_devices[dev].workspace = ptr;
    g_devices[dev].workspace_bytes = ptr ? bytes : 0;
    g_cnt_parity[dev].store(0u);
    return GEMM_OK;
}

int64_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    // Upper bound over the automatic configurations: aligned copies of A and B
    // (16-bit elements), then 16 K pieces of every tile of the narrowest
    // layout (128 rows of N by 64 of M per tile), plus the counters.
    if (M <= 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return 0;
    const int64_t dp = (K * 2 + 127) / 128 * 128;
    const int64_t repack = round256(sat_mul(M, dp)) + round256(sat_mul(N, dp));
    const int64_t tiles = ((N + 127) / 128) * ((M + 63) / 64);
    const int64_t total = kSplitCounterBytes + repack + round256(sat_mul(tiles, 4 * 4)) +
                          sat_mul(tiles, 16 * 4 * 32 * 256 * 4);
    return total < kSatBytes ? total : kSatBytes;
}

int gemm_tile_coord(int64_t t, int64_t tiles_m, int64_t tiles_n, int64_t group, int snake,
                    int64_t* tm, int64_t* tn) {
    if (tiles_m <= 0 || tiles_n <= 0 || group <= 0 || t < 0 || t >= tiles_m * tiles_n || !tm ||
        !tn)
        return GEMM_ERR_INVALID_DIM;
    raster_tile(t, tiles_m, tiles_n, group, tm, tn, snake != 0);
    return GEMM_OK;
}

int gemm_watchdog_selftest(int64_t limit_ns, void* stream) {
    if (limit_ns < 100000LL || limit_ns > 10000000000LL) return GEMM_ERR_INVALID_OPTION;
    const DeviceInfo* dev = nullptr;
    int st = current_device(&dev);
    if (st != GEMM_OK) return st;
    cudaError_t e = watchdog_selftest_launch(static_cast<uint64_t>(limit_ns), dev->watchdog,
                                             static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GEMM_OK : fail_cuda(e);
}

}  // extern "C"
