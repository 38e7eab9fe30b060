"""Host-side checks of the C ABI (CPU only, no GPU needed): the library
builds for sm_103a, loads, exports every function include/gemm.h declares,
rejects bad arguments before touching the GPU, and its tile rasteriser is a
bijection with the grouped order the pages describe."""
import ctypes
import os

import pytest

from dense_gemm_tcgen05_gb300 import build, capi


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    yield


def test_exports_every_declared_symbol():
    names = capi.declared_symbols()
    assert {"gemm_f32", "gemm_f16_tn", "gemm_bf16_tn", "gemm_fp8_tn",
            "gemm_status_string"} <= set(names)
    handle = ctypes.CDLL(capi.LIB_PATH)
    for name in names:
        assert hasattr(handle, name), name
    assert set(names) == set(capi._SIGNATURES)


def test_binding_constants_match_the_header():
    """Every status code and planner constant the binding hard-codes has the
    value include/gemm.h defines."""
    import re
    defs = {}
    for line in open(capi.HEADER):
        m = re.match(r"#define (GEMM_\w+) \(?(\d+)", line)
        if m:
            defs[m.group(1)] = int(m.group(2))
    status = {k: v for k, v in defs.items() if k == "GEMM_OK" or k.startswith("GEMM_ERR_")}
    assert len(status) == 11
    for name, value in status.items():
        assert getattr(capi, name) == value, name
    kinds = {"GEMM_PLAN_F16": "f16", "GEMM_PLAN_BF16": "bf16", "GEMM_PLAN_FP8": "e4m3",
             "GEMM_PLAN_F16_ACC16": "f16_acc16", "GEMM_PLAN_FP8_F32OUT": "e4m3_f32out"}
    for name, key in kinds.items():
        assert capi.PLAN_KINDS[key] == defs[name], name
    for flag in ("A_TMA", "B_TMA", "C_TMA", "A_128", "B_128", "NOALLOC"):
        assert getattr(capi, "PLAN_" + flag) == defs["GEMM_PLAN_" + flag], flag
    assert len(capi.PLAN_FIELDS) == defs["GEMM_PLAN_FIELDS"]
    assert "#define GEMM_NOALLOC_SCRATCH_BYTES (24LL << 20)" in open(capi.HEADER).read()
    assert capi.GEMM_NOALLOC_SCRATCH_BYTES == 24 << 20


def test_status_strings():
    for st in range(11):
        assert capi.status_text(st) and capi.status_text(st) != "unknown status"
    assert capi.status_text(99) == "unknown status"


FNS = ["gemm_f16_tn", "gemm_bf16_tn"]


@pytest.mark.parametrize("fn", FNS)
def test_argument_errors_without_gpu(fn):
    f = getattr(capi, fn)
    p = 0x10000  # never dereferenced: validation fails first
    assert f(-1, 4, 4, p, 4, p, 4, p, 4) == capi.GEMM_ERR_INVALID_DIM
    assert f(4, 4, 1 << 31, p, 1 << 31, p, 1 << 31, p, 4) == capi.GEMM_ERR_INVALID_DIM
    assert f(4, 4, 8, p, 7, p, 8, p, 4) == capi.GEMM_ERR_INVALID_LD
    assert f(4, 4, 8, p, 8, p, 7, p, 4) == capi.GEMM_ERR_INVALID_LD
    assert f(4, 4, 8, p, 8, p, 8, p, 3) == capi.GEMM_ERR_INVALID_LD
    assert f(4, 4, 8, None, 8, p, 8, p, 4) == capi.GEMM_ERR_NULL_PTR
    assert f(4, 4, 8, p, 8, None, 8, p, 4) == capi.GEMM_ERR_NULL_PTR
    assert f(4, 4, 8, p, 8, p, 8, None, 4) == capi.GEMM_ERR_NULL_PTR
    assert f(4, 4, 8, p + 1, 8, p, 8, p, 4) == capi.GEMM_ERR_MISALIGNED
    assert f(4, 4, 8, p, 8, p, 8, p + 1, 4) == capi.GEMM_ERR_MISALIGNED
    big = (1 << 48) + 8   # above the leading-dimension bound
    assert f(4, 4, 8, p, big, p, 8, p, 4) == capi.GEMM_ERR_INVALID_LD
    assert f(4, 4, 8, p, 8, p, big, p, 4) == capi.GEMM_ERR_INVALID_LD
    assert f(4, 4, 8, p, 8, p, 8, p, big) == capi.GEMM_ERR_INVALID_LD


def test_fp8_and_f32_argument_errors_without_gpu():
    p = 0x10000
    assert capi.gemm_fp8_tn(4, 4, -2, p, 8, p, 8, 1.0, 1.0, p, 4) == capi.GEMM_ERR_INVALID_DIM
    assert capi.gemm_fp8_tn(4, 4, 8, p, 8, p, 8, 1.0, 1.0, p + 1, 4) == capi.GEMM_ERR_MISALIGNED
    # e4m3 operands need no alignment beyond one byte: validation passes them
    assert capi.gemm_fp8_tn(4, 4, 8, p + 1, 8, p, 8, 1.0, 1.0, p, 3) == capi.GEMM_ERR_INVALID_LD
    assert capi.gemm_f32(4, 5, 6, p, 5, p, 5, p, 5) == capi.GEMM_ERR_INVALID_LD
    assert capi.gemm_f32(4, 5, 6, p, 6, p, 4, p, 5) == capi.GEMM_ERR_INVALID_LD
    assert capi.gemm_f32(4, 5, 6, p + 2, 6, p, 5, p, 5) == capi.GEMM_ERR_MISALIGNED
    assert capi.gemm_f32(4, 5, 6, None, 6, p, 5, p, 5) == capi.GEMM_ERR_NULL_PTR
    f6 = capi.gemm_f32_bf16x6
    assert f6(4, 5, -6, p, 6, p, 5, p, 5) == capi.GEMM_ERR_INVALID_DIM
    # 6 x K rounded up to 64 must stay below 2^31
    assert f6(4, 5, 1 << 29, p, 1 << 29, p, 5, p, 5) == capi.GEMM_ERR_INVALID_DIM
    assert f6(4, 5, 6, p, 5, p, 5, p, 5) == capi.GEMM_ERR_INVALID_LD
    assert f6(4, 5, 6, p, 6, p, 5, p, 4) == capi.GEMM_ERR_INVALID_LD
    assert f6(4, 5, 6, p, 6, None, 5, p, 5) == capi.GEMM_ERR_NULL_PTR
    assert f6(4, 5, 6, p, 6, p, 5, p + 2, 5) == capi.GEMM_ERR_MISALIGNED
    # K up to 2^31 - 1 passes the dimension check (the terms past 2^31 - 16 run in
    # the chain-continuing kernel); 2^31 does not
    assert capi.gemm_f32(4, 5, (1 << 31) - 1, p, 1 << 31, p, 5, p, 4) == capi.GEMM_ERR_INVALID_LD
    assert capi.gemm_f32(4, 5, 1 << 31, p, 1 << 31, p, 5, p, 5) == capi.GEMM_ERR_INVALID_DIM
    big = (1 << 48) + 4
    for fn in (capi.gemm_f32, f6):
        assert fn(4, 5, 6, p, big, p, 5, p, 5) == capi.GEMM_ERR_INVALID_LD
        assert fn(4, 5, 6, p, 6, p, big, p, 5) == capi.GEMM_ERR_INVALID_LD
        assert fn(4, 5, 6, p, 6, p, 5, p, big) == capi.GEMM_ERR_INVALID_LD
    assert capi.gemm_fp8_tn(4, 4, 8, p, big, p, 8, 1.0, 1.0, p, 4) == capi.GEMM_ERR_INVALID_LD


def test_noalloc_argument_errors_without_gpu():
    """The no-allocation entry point checks every argument before its first
    CUDA call (the scratch lookup), like the other entry points."""
    f = capi.gemm_bf16_tn_noalloc
    p = 0x10000
    assert f(4, 4, 8, p, 8, p, 8, p, 4, 65, None) == capi.GEMM_ERR_INVALID_OPTION
    assert f(-1, 4, 8, p, 8, p, 8, p, 4, 0, None) == capi.GEMM_ERR_INVALID_DIM
    assert f(4, 4, 8, p, 7, p, 8, p, 4, 0, None) == capi.GEMM_ERR_INVALID_LD
    assert f(4, 4, 8, p, 8, p, 8, p, 1 << 49, 0, None) == capi.GEMM_ERR_INVALID_LD
    assert f(4, 4, 8, p, 8, None, 8, p, 4, 0, None) == capi.GEMM_ERR_NULL_PTR
    assert f(4, 4, 8, p, 8, p + 1, 8, p, 4, 0, None) == capi.GEMM_ERR_MISALIGNED


def test_options():
    assert capi.gemm_set_option("pair", 1) == 0
    assert capi.gemm_set_option("pair", -1) == 0
    assert capi.gemm_set_option("pair", 2) == capi.GEMM_ERR_INVALID_OPTION
    assert capi.gemm_set_option("group", -1) == capi.GEMM_ERR_INVALID_OPTION
    assert capi.gemm_set_option("group", 65) == capi.GEMM_ERR_INVALID_OPTION
    assert capi.gemm_set_option("group", 8) == 0
    assert capi.gemm_set_option("group", 0) == 0
    assert capi.gemm_set_option("k_snake", 2) == capi.GEMM_ERR_INVALID_OPTION
    assert capi.gemm_set_option("k_snake", 0) == 0
    assert capi.gemm_set_option("k_snake", 1) == 0
    assert capi.gemm_set_option("band_snake", 2) == capi.GEMM_ERR_INVALID_OPTION
    assert capi.gemm_set_option("band_snake", 0) == 0
    assert capi.gemm_set_option("band_snake", 1) == 0
    assert capi.gemm_set_option("k_rotate", 3) == capi.GEMM_ERR_INVALID_OPTION
    assert capi.gemm_set_option("k_rotate", -1) == capi.GEMM_ERR_INVALID_OPTION
    for v in (2, 1, 0):
        assert capi.gemm_set_option("k_rotate", v) == 0
    assert capi.gemm_set_option("timeout_ns", 10) == capi.GEMM_ERR_INVALID_OPTION
    assert capi.gemm_set_option("nonsense", 1) == capi.GEMM_ERR_INVALID_OPTION
    assert capi.gemm_set_option("splits", 65) == capi.GEMM_ERR_INVALID_OPTION
    assert capi.gemm_set_option("splits", 0) == 0
    assert capi.gemm_set_option("tile_q", 96) == capi.GEMM_ERR_INVALID_OPTION
    assert capi.gemm_set_option("tile_q", 192) == 0
    assert capi.gemm_set_option("tile_q", 0) == 0
    assert capi.gemm_set_option("tail", 3) == capi.GEMM_ERR_INVALID_OPTION
    assert capi.gemm_set_option("tail", 0) == 0
    assert capi.gemm_set_option("cluster", 0) == capi.GEMM_ERR_INVALID_OPTION  # removed
    assert capi.gemm_set_option("f32_ktail", 16) == capi.GEMM_ERR_INVALID_OPTION
    assert capi.gemm_set_option("f32_ktail", 15) == 0
    assert capi.gemm_set_option("f32_ktail", 0) == 0
    assert capi.gemm_set_option("f32_tail", 4) == capi.GEMM_ERR_INVALID_OPTION
    assert capi.gemm_set_option("f32_tail", 3) == 0
    assert capi.gemm_set_option("f32_tail", 0) == 0
    assert capi.gemm_set_option("tail_k", 1) == capi.GEMM_ERR_INVALID_OPTION
    assert capi.gemm_set_option("tail_k", 0) == 0
    assert capi.gemm_set_option("repack", 2) == capi.GEMM_ERR_INVALID_OPTION
    assert capi.gemm_set_option("repack", 0) == 0
    assert capi.gemm_set_option("half", 4) == capi.GEMM_ERR_INVALID_OPTION
    assert capi.gemm_set_option("half", 3) == 0
    assert capi.gemm_set_option("half", 0) == 0


SPLIT_COUNTER_BYTES = 2 * 16384 * 4  # two fixed split-counter sets at the workspace's start


def test_workspace_size_bound():
    # aligned copies of A and B, then 16 pieces of every 128 x 64 tile (32 KB a slice)
    tiles = (1024 // 128) * (512 // 64)
    repack = (512 + 1024) * 64 * 2
    assert capi.gemm_workspace_bytes(512, 1024, 64) >= (SPLIT_COUNTER_BYTES + repack +
                                                         tiles * 16 * 4 * 32 * 1024)
    assert capi.gemm_workspace_bytes(0, 1, 1) == 0
    assert capi.gemm_workspace_bytes(1, 1, 1 << 31) == 0          # out of range


def test_workspace_sizes_saturate():
    """Sizes no device could hold saturate instead of wrapping around."""
    top = (1 << 31) - 1
    sat = ((1 << 63) - 1) // 4
    assert capi.gemm_workspace_bytes(top, top, top) == sat
    assert capi.gemm_workspace_bytes(top, top, 1) == sat            # the split bound alone
    assert capi.gemm_f32_bf16x6_workspace_bytes(top, top, top) >= sat
    # the exact figure where it fits in a device
    assert capi.gemm_workspace_bytes(4096, 4096, 4096) < 1 << 40


def test_f32_bf16x6_workspace_size():
    # the split-counter sets, then two operands of (rows x 6 Kp) bf16 values,
    # Kp = K rounded up to 64, each rounded up to 256 bytes
    def expect(M, N, K):
        kp = (K + 63) // 64 * 64
        r = lambda n: (n + 255) // 256 * 256  # noqa: E731
        return SPLIT_COUNTER_BYTES + r(M * 6 * kp * 2) + r(N * 6 * kp * 2)
    for shape in [(1, 1, 1), (4096, 4096, 4096), (3, 5, 65), (2047, 3001, 1023)]:
        assert capi.gemm_f32_bf16x6_workspace_bytes(*shape) == expect(*shape)
    assert (capi.gemm_f32_bf16x6_workspace_bytes(4096, 4096, 4096) ==
            SPLIT_COUNTER_BYTES + 2 * 4096 * 6 * 4096 * 2)
    assert capi.gemm_f32_bf16x6_workspace_bytes(0, 4, 4) == 0
    assert capi.gemm_f32_bf16x6_workspace_bytes(4, 4, -1) == 0


@pytest.mark.parametrize("snake", [0, 1])
@pytest.mark.parametrize("tiles_m,tiles_n,group", [(1, 1, 8), (32, 64, 8), (16, 12, 8),
                                                   (17, 5, 8), (7, 9, 3), (5, 5, 64), (64, 3, 1),
                                                   (32, 32, 16)])
def test_rasteriser_bijection_and_bands(tiles_m, tiles_n, group, snake):
    """Every work index maps to a distinct tile; indices t in one band of
    `group` tile rows stay in that band and walk down its rows first, moving
    one column right (left, for odd bands with snake) after each."""
    seen = set()
    for t in range(tiles_m * tiles_n):
        st, tm, tn = capi.gemm_tile_coord(t, tiles_m, tiles_n, group, snake)
        assert st == 0
        assert 0 <= tm < tiles_m and 0 <= tn < tiles_n
        band = t // (group * tiles_n)
        assert tm // group == band
        rows = min(group, tiles_m - band * group)
        local = t - band * group * tiles_n
        col = local // rows
        assert tm == band * group + local % rows
        assert tn == (tiles_n - 1 - col if snake and band % 2 else col)
        seen.add((tm, tn))
    assert len(seen) == tiles_m * tiles_n
    assert capi.gemm_tile_coord(tiles_m * tiles_n, tiles_m, tiles_n, group, snake)[0] != 0


def test_rasteriser_hand_listed_order():
    """3 x 2 tiles in bands of 2 rows, listed by hand: the first band walks
    down its two rows, then moves one column right; the short last band (one
    row) follows."""
    expect = [(0, 0), (1, 0), (0, 1), (1, 1), (2, 0), (2, 1)]
    got = [capi.gemm_tile_coord(t, 3, 2, 2)[1:] for t in range(6)]
    assert got == expect
    # snake: the second band walks right to left
    expect = [(0, 0), (1, 0), (0, 1), (1, 1), (2, 1), (2, 0)]
    got = [capi.gemm_tile_coord(t, 3, 2, 2, 1)[1:] for t in range(6)]
    assert got == expect


def test_tuner_shape_parser():
    from dense_gemm_tcgen05_gb300 import tune

    assert tune._parse("f16:8192x28672x8192") == ("f16", 8192, 28672, 8192)
    assert all(tune._parse(s)[0] in ("f16", "bf16", "e4m3") for s in tune.DEFAULT_SHAPES)


def test_binding_signatures_match_the_prototypes():
    """Every ctypes signature in the binding has the argument and return types
    of its prototype in include/gemm.h, position by position."""
    import re
    text = re.sub(r"/\*.*?\*/", "", open(capi.HEADER).read(), flags=re.S)
    protos = {}
    for m in re.finditer(r"^\s*([A-Za-z_][\w ]*?[\w\*])\s*(\**)\s*(gemm_\w+)\s*\(([^)]*)\)\s*;",
                         text, flags=re.M):
        ret = (m.group(1) + m.group(2)).replace(" ", "")
        params = [p.strip() for p in m.group(4).split(",") if p.strip() not in ("", "void")]
        protos[m.group(3)] = (ret, params)
    assert set(protos) == set(capi._SIGNATURES)

    def ctype_of(decl):
        decl = re.sub(r"\b(const)\b", "", decl)
        decl = re.sub(r"\s+", " ", decl).strip()
        typ = re.sub(r"\s*\w+$", "", decl) if not decl.endswith("*") else decl
        typ = typ.replace(" ", "")
        if typ.endswith("*"):
            if typ == "char*":
                return ctypes.c_char_p
            if typ == "int64_t*":
                return ctypes.POINTER(ctypes.c_int64)
            return ctypes.c_void_p
        return {"int64_t": ctypes.c_int64, "int": ctypes.c_int, "float": ctypes.c_float}[typ]

    for name, (ret, params) in protos.items():
        args, res = capi._SIGNATURES[name]
        assert len(args) == len(params), name
        for a, p in zip(args, params):
            assert a == ctype_of(p), (name, p)
        want_ret = {"int": ctypes.c_int, "int64_t": ctypes.c_int64,
                    "constchar*": ctypes.c_char_p}[ret]
        assert res == want_ret, (name, ret)


def test_product_and_oracle_share_nothing():
    """The product (the package, its CUDA sources and the header) never imports,
    loads or includes the oracle, and the oracle includes only the C standard
    library and OpenMP: the two implementations share no code."""
    import re
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    product = []
    for d in ("dense_gemm_tcgen05_gb300", "include"):
        for dirpath, _, files in os.walk(os.path.join(root, d)):
            product += [os.path.join(dirpath, f) for f in files
                        if f.endswith((".py", ".cu", ".cuh", ".h"))]
    assert len(product) > 10
    for path in product:
        code = open(path).read()
        if path.endswith(".py"):
            code = re.sub(r"#[^\n]*", "", code)                      # comments
        else:
            code = re.sub(r"//[^\n]*|/\*.*?\*/", "", code, flags=re.S)
        assert not re.search(r"^\s*(import|from)\s+oracle\b", code, flags=re.M), path
        assert "liboracle" not in code and "oracle.c" not in code, path
        assert not re.search(r'#include\s*[<"][^>"]*oracle', code), path
    includes = re.findall(r'#include\s*[<"]([^>"]+)[>"]',
                          open(os.path.join(root, "oracle", "oracle.c")).read())
    assert set(includes) <= {"math.h", "stdint.h", "stdlib.h", "string.h", "omp.h"}, includes
