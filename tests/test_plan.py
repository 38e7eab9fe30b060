"""The TN calls' planning rules, checked on the CPU through gemm_tn_plan (the
same host function every TN call plans with; no GPU needed).  Each case pins
one rule measured on GB300: tile shape, producer and repacks, narrow Q tiles,
split-K, the last wave's treatment, and the opt-in kernels."""
import pytest

from dense_gemm_tcgen05_gb300 import build, capi

WS = 1 << 30
ALIGNED = capi.PLAN_ALIGNED


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    yield


@pytest.fixture
def options():
    """Sets library options for one test and restores the defaults after it."""
    touched = []

    def set_(name, value):
        assert capi.gemm_set_option(name, value) == 0
        touched.append(name)
    yield set_
    defaults = {"pair": -1, "group": 0, "k_snake": 1, "band_snake": 1}
    for name in touched:
        capi.gemm_set_option(name, defaults.get(name, 0))


def plan(kind, M, N, K, **kw):
    st, p = capi.gemm_tn_plan(kind, M, N, K, **kw)
    assert st == capi.GEMM_OK and p["status"] == capi.GEMM_OK
    return p


def test_square_8192_pairs_and_narrowed_tail():
    """FP16 8192^3: 32 x 32 pair tiles of 256 x 256 on 76 pairs; the last
    wave's 36 tiles become 72 half-width units (0.8 of a tile each)."""
    p = plan("f16", 8192, 8192, 8192, workspace_bytes=WS)
    assert (p["pair"], p["tile_q"], p["tiles_p"], p["tiles_q"]) == (1, 256, 32, 32)
    assert (p["splits"], p["tail_f"], p["tail_ksplit"]) == (1, 2, 0)
    assert (p["stages"], p["stage_bytes"], p["grid"]) == (6, 32 * 1024, 152)


def test_long_k_tail_in_k_pieces_only_with_room():
    """192+ K stages and a tail that fits twice in a wave: K pieces, but only
    with a workspace; 4096^3 (64 stages) keeps the narrowed tail."""
    p = plan("bf16", 4096, 4096, 14336, workspace_bytes=WS)
    assert (p["tail_f"], p["tail_ksplit"], p["tail_kb_per"]) == (2, 1, 112)
    p = plan("bf16", 4096, 4096, 14336)
    assert (p["tail_f"], p["tail_ksplit"]) == (2, 0)
    p = plan("bf16", 4096, 4096, 4096, workspace_bytes=WS)
    assert (p["tail_f"], p["tail_ksplit"]) == (2, 0)


def test_tail_options(options):
    options("tail", 1)
    assert plan("f16", 8192, 8192, 8192)["tail_f"] == 1
    options("tail", 4)
    assert plan("f16", 8192, 8192, 8192)["tail_f"] == 4
    options("tail", 0)
    options("tail_k", 3)
    p = plan("f16", 8192, 8192, 8192, workspace_bytes=WS)
    assert (p["tail_f"], p["tail_ksplit"]) == (3, 1)


@pytest.mark.parametrize("kind", ["bf16", "e4m3"])
@pytest.mark.parametrize("M,q", [(1, 16), (16, 16), (17, 32), (32, 32), (33, 64), (128, 64),
                                 (129, 128)])
def test_skinny_single_cta_tiles_and_width(M, q, kind, options):
    """Decode-like shapes: single-CTA 128-row tiles, 16/32 columns when M fits
    in one such tile, else 64 (M <= 128) or 128.  (16-bit inputs with M > 64,
    or M <= 64 without a workspace, run pairs of 64-row halves instead unless
    option "half" = 2.)"""
    if kind == "bf16":
        options("half", 2)
    p = plan(kind, M, 8192, 8192)
    assert p["pair"] == 0 and p["tile_q"] == q and p["tiles_p"] == 64


def test_skinny_split_k_needs_a_workspace(options):
    """64 tiles on 152 SMs: two K pieces each with a workspace (128 CTAs; 32
    stages of two K atoms each); without one, 64 pairs of 64-row halves 32
    wide (128 CTAs, K whole), or 64 one-CTA tiles when halves are off."""
    p = plan("bf16", 16, 8192, 8192, workspace_bytes=WS)
    assert (p["splits"], p["kb_per_split"], p["grid"], p["atoms"]) == (2, 32, 128, 2)
    p = plan("bf16", 16, 8192, 8192)
    assert (p["splits"], p["pair"], p["half"], p["tile_q"], p["grid"]) == (1, 1, 1, 32, 128)
    options("half", 2)
    p = plan("bf16", 16, 8192, 8192)
    assert (p["splits"], p["pair"], p["grid"]) == (1, 0, 64)


def test_narrow_ring_is_deeper(options):
    """A 16-column one-CTA tile's one-atom stage holds 16 KB of B and 2 KB of
    A: 10 stages of 18 KB in the 192 KB ring, against 8 of 24 KB at 64
    columns; with two atoms per stage (the automatic choice there), 5 of 36 KB
    and 4 of 48 KB (K split, one issuer)."""
    def ring(M, **kw):
        p = plan("bf16", M, 8192, 8192, workspace_bytes=WS, **kw)
        assert p["pair"] == 0 and p["issuers"] == 1 and p["ring_epi"] == 0, p
        return p["stages"], p["stage_bytes"]
    assert ring(16) == (5, 36 * 1024)
    assert ring(64) == (4, 48 * 1024)
    options("max_ctas", 32)                     # 64 tiles on 32 CTAs: 192 KB
    p = plan("bf16", 16, 8192, 8192, workspace_bytes=WS)
    assert (p["ring_epi"], p["issuers"], p["stages"], p["stage_bytes"]) == (0, 1, 5, 36 * 1024)
    options("max_ctas", 0)
    options("half", 2)
    options("atoms", 1)
    assert (plan("bf16", 16, 8192, 8192)["stages"], plan("bf16", 16, 8192, 8192)["stage_bytes"]) \
        == (10, 18 * 1024)
    assert (plan("bf16", 64, 8192, 8192)["stages"], plan("bf16", 64, 8192, 8192)["stage_bytes"]) \
        == (8, 24 * 1024)


def test_atoms_rule(options):
    """Two K atoms per stage for tiles at most 128 columns wide whose ring keeps
    three stages; one for tiles 256 wide (pairs, pairs of halves, one CTA) and
    for the load-based producer; option 1 / 2 forces it (2 only with TMA)."""
    assert plan("f16", 8192, 8192, 8192)["atoms"] == 1                       # pairs, 256 wide
    assert plan("bf16", 1024, 2048, 4096)["atoms"] == 2                      # one CTA, 128 wide
    p = plan("bf16", 128, 8192, 8192)
    assert (p["half"], p["atoms"], p["stages"]) == (1, 2, 6)                # pairs of halves
    assert plan("bf16", 256, 8192, 8192)["atoms"] == 1                       # halves, 256 wide
    assert plan("e4m3", 128, 8192, 8192)["atoms"] == 2
    no_tma_a = ALIGNED & ~(capi.PLAN_A_TMA | capi.PLAN_A_128)
    assert plan("bf16", 1024, 2048, 4096, flags=no_tma_a)["atoms"] == 1     # load producer
    options("atoms", 2)
    p = plan("f16", 8192, 8192, 8192)
    assert (p["atoms"], p["stages"], p["stage_bytes"], p["kb_per_split"]) == (2, 3, 65536, 64)
    assert plan("bf16", 1024, 2048, 4096, flags=no_tma_a)["atoms"] == 1
    options("atoms", 1)
    assert plan("bf16", 1024, 2048, 4096)["atoms"] == 1


def test_forced_narrow_width_needs_m_to_fit(options):
    options("tile_q", 16)
    assert plan("bf16", 16, 8192, 8192)["tile_q"] == 16
    assert plan("bf16", 40, 8192, 8192)["tile_q"] == 64       # three tiles would overlap
    options("pair", 1)
    assert plan("bf16", 16, 8192, 8192)["tile_q"] == 64       # never with CTA pairs


def test_sub_wave_rule():
    """Pair tiles filling less than a wave give way to single-CTA tiles that
    fit in one (1024 x 1024 x 4096: 64 tiles of 128 x 128, two K pieces with a
    workspace); where those would need a second wave (2048^2) pairs stay.  With
    K >= 8192, 16-bit inputs and M > 256, pair tiles 128 wide run instead when
    they fit in one wave (1024 x 1024 x 8192: 32 pair tiles, two K pieces);
    FP8 and M <= 256 keep their rules."""
    p = plan("bf16", 1024, 1024, 4096, workspace_bytes=WS)
    assert (p["pair"], p["tile_q"], p["splits"], p["grid"]) == (0, 128, 2, 128)
    assert plan("bf16", 2048, 2048, 8192)["pair"] == 1
    p = plan("bf16", 1024, 1024, 8192, workspace_bytes=WS)
    assert (p["pair"], p["tile_q"], p["splits"], p["grid"]) == (1, 128, 2, 128)
    assert (plan("e4m3", 1024, 1024, 8192)["pair"], plan("bf16", 1024, 1024, 8192)["pair"]) \
        == (0, 1)
    assert plan("bf16", 256, 8192, 8192)["half"] == 1


def test_unaligned_operands_repacked_or_load_producer():
    """A's rows not 16-byte aligned: copied into the workspace when it has room
    (TMA path), read by the load-based producer (single CTA) otherwise."""
    flags = ALIGNED & ~(capi.PLAN_A_TMA | capi.PLAN_A_128)
    p = plan("bf16", 2047, 3001, 1023, flags=flags)
    assert (p["producer"], p["pair"], p["copy_a"]) == (1, 0, 0)
    p = plan("bf16", 2047, 3001, 1023, flags=flags, workspace_bytes=WS)
    assert (p["producer"], p["copy_a"], p["copy_b"]) == (0, 1, 0)
    p = plan("bf16", 2047, 3001, 1023, flags=flags, workspace_bytes=1 << 20)   # too small
    assert (p["producer"], p["copy_a"]) == (1, 0)


def test_not_128_byte_aligned_copied_only_when_heavy():
    """Rows 16- but not 128-byte aligned are copied when MN / (M + N) >= 1100 x
    element size (8192^3: 4096 >= 2200), not at 4096^3 (2048)."""
    flags = ALIGNED & ~capi.PLAN_A_128
    assert plan("f16", 8192, 8192, 8192, flags=flags, workspace_bytes=WS)["copy_a"] == 1
    assert plan("f16", 4096, 4096, 4096, flags=flags, workspace_bytes=WS)["copy_a"] == 0


def test_fp16_accumulation_never_splits():
    p = plan("f16_acc16", 16, 8192, 8192, workspace_bytes=WS)
    assert p["splits"] == 1
    assert plan("f16", 16, 8192, 8192, workspace_bytes=WS)["splits"] == 2


def test_fp8_stages_and_tail():
    """E4M3 stages hold 128 K values: 8192^3 has 64 K stages per tile (no
    K-split tail); its narrowed tail units cost 0.9 of a tile, still worth it."""
    p = plan("e4m3", 8192, 8192, 8192, workspace_bytes=WS)
    assert (p["pair"], p["kb_per_split"], p["tail_f"], p["tail_ksplit"]) == (1, 64, 2, 0)


def test_64_row_tiles_only_when_forced(options):
    """One CTA per 64 rows of N (MMA M = 64) only with option "half" = 1;
    pairs of 64-row halves (pair = 1) are another plan."""
    assert plan("bf16", 16, 8192, 8192, workspace_bytes=WS)["half"] == 0
    p = plan("bf16", 16, 8192, 8192)
    assert p["half"] == 0 or p["pair"] == 1
    options("half", 1)
    p = plan("bf16", 16, 8192, 8192, workspace_bytes=WS)
    assert (p["half"], p["tiles_p"], p["splits"], p["grid"]) == (1, 128, 1, 128)
    assert plan("f16_acc16", 16, 8192, 8192)["half"] == 0
    assert plan("bf16", 4096, 4096, 4096)["half"] == 0          # CTA pairs


def test_noalloc_split_rules(options):
    """The no-allocation call's fixed 24 MiB array serves operand copies first
    and the split second: an automatic split shrinks to what the copies leave
    (never failing), a forced split that does not fit beside them runs without
    them, and one that does not fit the array at all is refused."""
    na = dict(flags=ALIGNED | capi.PLAN_NOALLOC, workspace_bytes=capi.GEMM_NOALLOC_SCRATCH_BYTES)
    mis_b = (ALIGNED | capi.PLAN_NOALLOC) & ~(capi.PLAN_B_TMA | capi.PLAN_B_128)
    nb = dict(na, flags=mis_b)
    p = plan("bf16", 64, 2048, 4096, **na)                      # aligned: the full automatic split
    assert (p["splits"], p["copy_b"], p["producer"]) == (8, 0, 0)
    p = plan("bf16", 64, 2048, 4096, **nb)                      # B copied (16 MiB), split shrinks
    assert (p["splits"], p["copy_b"], p["producer"]) == (3, 1, 0)
    # the same inputs with a registered workspace of that size: no shrinking, no split
    p = plan("bf16", 64, 2048, 4096, flags=mis_b & ~capi.PLAN_NOALLOC,
             workspace_bytes=capi.GEMM_NOALLOC_SCRATCH_BYTES)
    assert (p["splits"], p["copy_b"]) == (1, 1)
    options("splits", 8)                                        # forced: the copy gives way
    p = plan("bf16", 64, 2048, 4096, **nb)
    assert (p["splits"], p["copy_b"], p["producer"]) == (8, 0, 1)
    options("splits", 16)                                       # does not fit at all
    st, p = capi.gemm_tn_plan("bf16", 4096, 4096, 4096, **na)
    assert st == capi.GEMM_OK and p["status"] == capi.GEMM_ERR_SCRATCH
    options("splits", 0)
    assert plan("bf16", 4096, 4096, 4096, **na)["splits"] == 1  # a full wave: no split


def test_issuers_and_pair_halves_rules(options):
    """Skinny shapes: 16-bit inputs with 64 < M <= 256 run pairs of 64-row
    halves (128 rows of N per pair, tile width M rounded up to a multiple of
    32) with two MMA issuers when they fit in one wave; an explicit tile_q of
    128, 192 or 256 sets the width.  FP8 and other one-wave skinny shapes run
    one-CTA tiles, with two
    issuers when the tiles are at most 64 columns wide and unsplit.  Option
    "issuers" = 1 turns both off; 2 forces two on one-CTA tiles of at most 128
    columns; "half" = 2 keeps one-CTA tiles."""
    for M, tq in ((65, 128), (100, 128), (128, 128), (129, 160), (192, 192),
                  (200, 224), (225, 256), (256, 256)):
        p = plan("bf16", M, 8192, 8192, workspace_bytes=WS)
        assert (p["pair"], p["half"], p["issuers"], p["tile_q"], p["grid"]) == (1, 1, 2, tq, 128), M
    for forced in (128, 192, 256):
        options("tile_q", forced)
        assert plan("bf16", 150, 8192, 8192, workspace_bytes=WS)["tile_q"] == forced
    options("tile_q", 0)
    # two K atoms per stage: halves up to 128 wide take them by themselves;
    # wider halves keep one atom even when forced
    assert plan("bf16", 128, 8192, 8192, workspace_bytes=WS)["atoms"] == 2
    assert plan("bf16", 160, 8192, 8192, workspace_bytes=WS)["atoms"] == 1
    options("atoms", 2)
    for M, atoms in ((100, 2), (160, 1), (192, 1), (256, 1)):
        assert plan("bf16", M, 8192, 8192, workspace_bytes=WS)["atoms"] == atoms, M
    options("half", 2)
    assert plan("bf16", 256, 8192, 8192, workspace_bytes=WS)["atoms"] == 2  # one-CTA tiles
    options("half", 0)
    options("atoms", 0)
    p = plan("e4m3", 128, 8192, 8192, workspace_bytes=WS)   # FP8: 128 tiles of 128 x 64
    assert (p["pair"], p["half"], p["issuers"], p["tile_q"], p["splits"]) == (0, 0, 2, 64, 1)
    assert plan("bf16", 64, 8192, 8192, workspace_bytes=WS)["half"] == 0     # M <= 64: split
    for M, tq in ((1, 32), (16, 32), (32, 32), (48, 64), (64, 64)):           # no workspace
        p = plan("bf16", M, 8192, 8192)
        assert (p["pair"], p["half"], p["tile_q"], p["issuers"], p["atoms"]) == (1, 1, tq, 2, 1), M
    assert plan("e4m3", 16, 8192, 8192)["half"] == 0                         # FP8
    assert plan("bf16", 16, 4096, 8192)["half"] == 0                         # half a wave
    assert plan("bf16", 16, 8192, 8192, workspace_bytes=WS)["issuers"] == 1  # split K
    assert plan("bf16", 8192, 8192, 8192)["issuers"] == 1                    # CTA pairs
    p = plan("f16_acc16", 128, 8192, 8192)                                   # FP16 accumulation
    assert (p["issuers"], p["half"]) == (1, 0)
    assert plan("bf16", 128, 16384, 8192)["half"] == 0                       # two waves
    assert plan("bf16", 256, 512, 4096, workspace_bytes=WS)["half"] == 0     # 4 pairs: split-K
    assert plan("bf16", 128, 6144, 8192)["half"] == 0                        # 48 of 76 pairs
    assert plan("bf16", 64, 131072, 8192)["issuers"] == 1                    # several waves
    options("half", 2)
    p = plan("bf16", 128, 8192, 8192, workspace_bytes=WS)                    # one-CTA tiles
    assert (p["pair"], p["half"], p["issuers"], p["tile_q"]) == (0, 0, 2, 64)
    assert plan("bf16", 256, 8192, 8192, workspace_bytes=WS)["issuers"] == 1  # 128 columns
    options("issuers", 1)
    p = plan("bf16", 128, 8192, 8192, workspace_bytes=WS)
    assert (p["issuers"], p["half"]) == (1, 0)
    options("half", 0)
    assert plan("bf16", 128, 8192, 8192, workspace_bytes=WS)["half"] == 0    # issuers 1: no halves
    options("half", 2)
    options("issuers", 2)
    assert plan("bf16", 256, 8192, 8192, workspace_bytes=WS)["issuers"] == 2
    assert plan("bf16", 16, 8192, 8192)["issuers"] == 2                      # unsplit here
    assert capi.gemm_set_option("issuers", 4) == capi.GEMM_ERR_INVALID_OPTION


def test_persistent_grid_follows_sms_and_cap(options):
    assert plan("f16", 8192, 8192, 8192, sms=148)["grid"] == 148
    options("max_ctas", 64)
    assert plan("f16", 8192, 8192, 8192)["grid"] == 64


def test_argument_errors():
    assert capi.gemm_tn_plan("f16", 0, 8, 8)[0] == capi.GEMM_ERR_INVALID_DIM
    assert capi.gemm_tn_plan("f16", 8, 8, 8, sms=0)[0] == capi.GEMM_ERR_INVALID_DIM
    lib = capi.lib()
    assert lib.gemm_tn_plan(9, 8, 8, 8, 0, 0, 152, None, 17) == capi.GEMM_ERR_INVALID_OPTION
    assert lib.gemm_tn_plan(0, 8, 8, 8, 0, 0, 152, None, 17) == capi.GEMM_ERR_INVALID_OPTION


def test_sizes_beyond_any_device_plan_without_overflow(options):
    """The largest dimensions with a forced 64-piece split: the partial sums
    cannot fit in any workspace, so the call stays unsplit (the byte counts
    saturate instead of wrapping around into a small number)."""
    top = (1 << 31) - 1
    options("splits", 64)
    p = plan("bf16", top, top, top, workspace_bytes=(1 << 62))
    assert p["splits"] == 1 and p["copy_a"] == 0
    flags = ALIGNED & ~(capi.PLAN_A_TMA | capi.PLAN_A_128)
    p = plan("bf16", top, top, top, flags=flags, workspace_bytes=(1 << 62))
    assert (p["copy_a"], p["producer"]) == (0, 1)   # A's copy cannot fit either


@pytest.mark.parametrize("M,q", [(192, 192), (200, 256), (384, 192), (640, 128)])
def test_tile_width_by_padding_cost(M, q):
    """Pair tiles (N = 32768 fills many waves): the width t minimising
    ceil(M / t) * max(t, 96), ties to the wider tile.  M = 200: 256 and 128
    both cost 256, so 256; M = 640: 128 costs 640 against 768 for 256 and 192."""
    p = plan("bf16", M, 32768, 4096)
    assert p["pair"] == 1 and p["tile_q"] == q


def test_repack_threshold_boundary():
    """Rows 16- but not 128-byte aligned are copied when MN / (M + N) >= 1100 x
    element size: BF16 M = N = 4400 gives exactly 2200 (copied), 4398 gives
    2199 (not)."""
    flags = ALIGNED & ~capi.PLAN_A_128
    assert plan("bf16", 4400, 4400, 4096, flags=flags, workspace_bytes=WS)["copy_a"] == 1
    assert plan("bf16", 4398, 4398, 4096, flags=flags, workspace_bytes=WS)["copy_a"] == 0


@pytest.mark.parametrize("kind", ["f16", "e4m3"])
def test_last_wave_cost_model(kind):
    """86 pair tiles on 76 pair slots leave 10: quarter-width units (one wave
    at 0.65, or 0.8 for FP8, of a tile's time) beat half-width ones (0.8 / 0.9)
    and the whole tiles (1.0).  146 tiles leave 70: cut in two they would need
    two waves (1.6), so the last wave stays whole."""
    p = plan(kind, 256, 256 * 86, 4096)
    assert (p["tiles_p"], p["tiles_q"], p["tail_f"], p["tail_ksplit"]) == (86, 1, 4, 0)
    p = plan(kind, 256, 256 * 146, 4096)
    assert (p["tiles_p"], p["tail_f"]) == (146, 1)


def test_two_issuers_get_an_even_ring(options):
    """Two MMA issuers: the ring depth is rounded down to an even count, so
    each slot always belongs to one issuer (with one or two K atoms)."""
    shapes = [("bf16", 16, 16384, 8192), ("bf16", 16, 8192, 8192), ("bf16", 64, 14336, 4096),
              ("e4m3", 16, 16384, 8192), ("f16", 128, 8192, 8192), ("bf16", 32, 16384, 8192),
              ("bf16", 192, 8192, 8192), ("bf16", 160, 8192, 8192), ("bf16", 250, 8192, 8192),
              ("f16", 48, 8192, 8192)]
    seen = {1: 0, 2: 0}
    for kind, M, N, K in shapes:
        for ws in (0, WS):
            p = plan(kind, M, N, K, workspace_bytes=ws)
            if p["issuers"] == 2:
                assert p["stages"] % 2 == 0, (kind, M, N, K, p)
                seen[p["atoms"]] += 1
    assert seen[1] >= 4 and seen[2] >= 6, seen
    options("max_ctas", 64)      # 64 pairs on 32 pair slots: the 192 KB ring
    p = plan("bf16", 192, 8192, 8192, workspace_bytes=WS)   # 20 KB stages: nine fit, eight run
    assert (p["half"], p["tile_q"], p["atoms"], p["stages"], p["ring_epi"]) == (1, 192, 1, 8, 0)
    options("max_ctas", 0)       # one pair tile each: 224 KB, eleven fit, ten run
    p = plan("bf16", 192, 8192, 8192, workspace_bytes=WS)
    assert (p["half"], p["tile_q"], p["atoms"], p["stages"], p["ring_epi"]) == (1, 192, 1, 10, 1)
    p = plan("bf16", 16, 8192, 8192)                         # halves 32 wide: 20 barrier slots
    assert (p["half"], p["tile_q"], p["atoms"], p["stages"]) == (1, 32, 1, 20)
    # one-CTA 16-wide tiles: 36 KB stages, five fit; two issuers keep four
    p = plan("bf16", 16, 16384, 8192, workspace_bytes=WS)
    assert (p["pair"], p["tile_q"], p["issuers"], p["atoms"], p["stages"]) == (0, 16, 2, 2, 4)
    # one issuer (the split plan) keeps all five
    p = plan("bf16", 16, 8192, 8192, workspace_bytes=WS)
    assert (p["splits"], p["issuers"], p["atoms"], p["stages"]) == (2, 1, 2, 5)
    # two tiles per CTA: one issuer takes all five, two (forced) keep four
    options("max_ctas", 64)
    p = plan("bf16", 16, 16384, 8192, workspace_bytes=WS)
    assert (p["tile_q"], p["atoms"], p["ring_epi"], p["issuers"], p["stages"]) == (16, 2, 0, 1, 5)
    options("issuers", 2)
    p = plan("bf16", 16, 16384, 8192, workspace_bytes=WS)
    assert (p["tile_q"], p["atoms"], p["ring_epi"], p["issuers"], p["stages"]) == (16, 2, 0, 2, 4)
    options("issuers", 0)
    options("max_ctas", 0)
    options("issuers", 2)
    options("pair", 0)
    p = plan("bf16", 100, 1100, 1000)                   # 64 KB stages: three fit, two run
    assert (p["tile_q"], p["issuers"], p["atoms"], p["stages"]) == (128, 2, 2, 2)


def test_ring_over_the_epilogue_area(options):
    """Pairs of 64-row halves whose pairs run one unit each also take the
    epilogue's 32 KB staging area for the ring (224 KB instead of 192), still
    rounded to an even depth with two issuers; other plans (measured slower
    with it), several units per pair, a cut last wave or the load-based
    producer keep 192 KB."""
    def ring(kind, M, N, K, **kw):
        p = plan(kind, M, N, K, workspace_bytes=WS, **kw)
        return p["ring_epi"], p["stages"], p["stage_bytes"]
    assert ring("bf16", 192, 8192, 8192) == (1, 10, 20 * 1024)     # halves 192 wide: 8 -> 10
    assert ring("bf16", 160, 8192, 8192) == (1, 12, 18 * 1024)     # 10 -> 12
    assert ring("bf16", 224, 8192, 8192) == (1, 10, 22 * 1024)     # 8 -> 10
    assert ring("bf16", 16, 8192, 8192) == (0, 5, 36 * 1024)       # split one-CTA tiles
    assert ring("bf16", 2048, 2048, 2048) == (0, 6, 32 * 1024)     # CTA pairs 256 wide
    assert ring("bf16", 128, 8192, 8192)[0] == 0                   # 7 rounds down to 6
    assert ring("bf16", 256, 8192, 8192)[0] == 0                   # 9 rounds down to 8
    assert ring("f16", 8192, 8192, 8192)[0] == 0                   # several tiles per pair
    assert ring("bf16", 4096, 4096, 4096)[0] == 0
    options("max_ctas", 64)
    assert ring("bf16", 192, 8192, 8192)[0] == 0                   # 64 tiles on 32 pairs
    options("max_ctas", 0)
    options("tail", 2)
    assert ring("bf16", 512, 8192, 4096)[0] == 0                   # narrowed last wave
    options("tail", 0)
    flags = ALIGNED & ~(capi.PLAN_A_TMA | capi.PLAN_A_128)
    p = plan("bf16", 130, 300, 257, flags=flags)                   # load-based producer
    assert p["producer"] == 1 and p["ring_epi"] == 0


def _sweep_shapes():
    Ms = (1, 7, 16, 17, 32, 33, 48, 64, 65, 96, 100, 128, 129, 150, 160, 176, 192, 200, 224,
          225, 255, 256, 257, 384, 1000, 2048, 8192)
    Ns = (64, 1000, 4096, 8192, 9728, 16384)
    Ks = (64, 200, 2048, 8192)
    for M in Ms:
        for N in Ns:
            for K in Ks:
                yield M, N, K


@pytest.mark.parametrize("kind", ["f16", "bf16", "e4m3", "e4m3_f32out"])
def test_ring_layout_invariants(kind, options):
    """Over a grid of shapes, with and without a workspace, automatic and with
    pairs of halves forced: the ring fits its region (192 KB, or 224 KB when it
    runs on over the epilogue's staging area), stays within the 20 barrier
    slots, keeps 1024-byte stages, is even with two issuers, and runs over the
    staging area only for pairs of halves whose pairs run one unit each."""
    for forced in (0, 3):
        options("half", forced)
        for M, N, K in _sweep_shapes():
            for ws in (0, WS):
                p = plan(kind, M, N, K, workspace_bytes=ws)
                if p["status"] != 0:
                    continue
                region = (224 if p["ring_epi"] else 192) * 1024
                assert p["stages"] * p["stage_bytes"] <= region, (M, N, K, ws, p)
                assert 2 <= p["stages"] <= 20 and p["stage_bytes"] % 1024 == 0, p
                if p["issuers"] == 2:
                    assert p["stages"] % 2 == 0, (M, N, K, ws, p)
                if p["ring_epi"]:
                    units = p["tiles_p"] * p["tiles_q"] * p["splits"]
                    slots = p["grid"] // 2
                    assert (p["pair"], p["half"], p["producer"], p["tail_f"]) == (1, 1, 0, 1), p
                    assert units <= slots, (M, N, K, ws, p)
                if p["atoms"] == 2 and p["pair"] and p["half"]:
                    assert p["tile_q"] == 128, p
    options("half", 0)


@pytest.mark.parametrize("kind,out_bytes", [("bf16", 2), ("f16", 2), ("e4m3", 2), ("e4m3_f32out", 4)])
def test_halves_widths_keep_stores_aligned(kind, out_bytes, options):
    """Pairs of 64-row halves: the width is a multiple of 32 from 32 to 256, so
    each half starts 16 * k bytes into the tile (its TMA stores need a 16-byte
    aligned innermost coordinate), and a CTA's A box is at most 128 rows."""
    options("half", 3)
    for M in range(1, 300):
        p = plan(kind, M, 8192, 2048)
        if not (p["pair"] and p["half"]):
            continue
        w = p["tile_q"]
        assert w % 32 == 0 and 32 <= w <= 256, (M, p)
        assert (w // 2 * out_bytes) % 16 == 0 and (w * out_bytes) % 16 == 0, (M, p)
        assert M > 256 or w >= M, (M, p)                      # one column of tiles
