"""Configuration sweep for the tensor-core GEMM: times every combination of the
library's tuning options on the given shapes and reports the fastest.

The options swept are the ones gemm_set_option exposes -- CTA pairing
("pair"), the rasteriser's group size ("group"), the output tile width along M
("tile_q") and split-K ("splits", with a workspace registered) -- so a
result can be applied directly.  The pages observe that no single tile configuration
is best everywhere ("FP16 GEMM Optimization on AMD RDNA 3 and RDNA 4",
"Tuning Further"; "FP8 GEMM Optimization on AMD RDNA 4", "Results"); this
script measures how far the automatic choices are from the best one found.

  python -m dense_gemm_tcgen05_gb300.tune [--shapes f16:8192x8192x8192,...]
         [--iters 20] [--quick]

Each sweep timing: 3 warm-up calls, then `iters` calls on the same stream
between CUDA events, inputs rotating over two sets; each shape starts with a
longer warm-up run so that clocks have settled.  A single pass over many
configurations drifts with the GPU's clock and power (the same configuration
can differ by several per cent within one sweep), so the automatic choice and
the three fastest configurations of the sweep are then timed again, paired:
`rounds` rounds in alternating order, `iters` calls each, and the medians
decide.  One JSON line per shape is printed with every configuration's sweep
TFLOP/s, the paired medians, the best configuration and the automatic
choice's fraction of it.
"""
from __future__ import annotations

import argparse
import itertools
import json
import statistics

import torch

from . import capi

DEFAULT_SHAPES = ["f16:8192x8192x8192", "bf16:4096x4096x4096", "bf16:4096x14336x4096",
                  "e4m3:8192x8192x8192", "e4m3:3072x4096x8192", "bf16:128x8192x8192",
                  "bf16:256x8192x8192", "e4m3:128x8192x8192", "bf16:1024x1024x8192"]
_DT = {"f16": torch.float16, "bf16": torch.bfloat16, "e4m3": torch.float8_e4m3fn}


def _parse(spec: str):
    kind, dims = spec.split(":")
    M, N, K = (int(x) for x in dims.lower().split("x"))
    return kind, M, N, K


def _operands(kind, M, N, K, sets=2):
    out = []
    for s in range(sets):
        g = torch.Generator(device="cuda").manual_seed(s)
        a = torch.randn((M, K), device="cuda", generator=g).to(_DT[kind])
        b = torch.randn((N, K), device="cuda", generator=g).to(_DT[kind])
        c = torch.empty((N, M), device="cuda",
                        dtype=torch.float16 if kind == "f16" else torch.bfloat16)
        out.append((a, b, c))
    return out


def _call(kind, M, N, K, a, b, c, stream):
    if kind == "e4m3":
        return capi.gemm_fp8_tn(M, N, K, a.data_ptr(), K, b.data_ptr(), K, 1.0, 1.0, c.data_ptr(),
                                M, stream)
    fn = capi.gemm_f16_tn if kind == "f16" else capi.gemm_bf16_tn
    return fn(M, N, K, a.data_ptr(), K, b.data_ptr(), K, c.data_ptr(), M, stream)


def time_config(kind, M, N, K, ops, iters, stream) -> float:
    """TFLOP/s of the current option settings (mean over `iters` calls)."""
    h = stream.cuda_stream
    with torch.cuda.stream(stream):
        for i in range(3):
            st = _call(kind, M, N, K, *ops[i % len(ops)], h)
            if st != 0:
                raise RuntimeError(capi.status_text(st))
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(iters):
            _call(kind, M, N, K, *ops[i % len(ops)], h)
        t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / iters
    return 2.0 * M * N * K / (ms * 1e-3) / 1e12


def _set(pair, group, tile_q, splits):
    for name, value in (("pair", pair), ("group", group), ("tile_q", tile_q), ("splits", splits)):
        st = capi.gemm_set_option(name, value)
        if st != 0:
            raise RuntimeError("option %s=%s: %s" % (name, value, capi.status_text(st)))


def paired(kind, M, N, K, ops, configs, iters, rounds, stream) -> list:
    """Median TFLOP/s of each configuration (None: the automatic choice) over
    `rounds` rounds in alternating order."""
    res = [[] for _ in configs]
    order = list(range(len(configs)))
    for r in range(rounds):
        for i in (order if r % 2 == 0 else order[::-1]):
            c = configs[i]
            _set(*(c if c is not None else (-1, 0, 0, 0)))
            res[i].append(time_config(kind, M, N, K, ops, iters, stream))
    _set(-1, 0, 0, 0)
    return [statistics.median(v) for v in res]


def tune_shape(spec: str, iters: int, quick: bool, rounds: int = 8) -> dict:
    kind, M, N, K = _parse(spec)
    ops = _operands(kind, M, N, K)
    stream = torch.cuda.Stream()
    pairs = [0, 1]
    groups = [0] if quick else [0, 8, 12, 24]
    tile_qs = [0, 128, 256] if quick else [0, 64, 128, 192, 256]
    splits = [1, 0]
    rows = []
    try:
        _set(-1, 0, 0, 0)
        time_config(kind, M, N, K, ops, 4 * iters, stream)  # bring clocks up first
        auto = time_config(kind, M, N, K, ops, iters, stream)
        for p, g, t, s in itertools.product(pairs, groups, tile_qs, splits):
            _set(p, g, t, s)
            rows.append({"pair": p, "group": g, "tile_q": t, "splits": s,
                         "tflops": round(time_config(kind, M, N, K, ops, iters, stream), 1)})
        _set(-1, 0, 0, 0)
        top = sorted(rows, key=lambda r: -r["tflops"])[:3]
        cands = [None] + [(r["pair"], r["group"], r["tile_q"], r["splits"]) for r in top]
        med = paired(kind, M, N, K, ops, cands, iters, rounds, stream)
    finally:
        _set(-1, 0, 0, 0)
    auto = med[0]
    finals = [dict(r, paired_tflops=round(m, 1)) for r, m in zip(top, med[1:])]
    best = max(finals, key=lambda r: r["paired_tflops"])
    return {"shape": spec, "auto_tflops": round(auto, 1), "best": best,
            "auto_over_best": round(min(1.0, auto / best["paired_tflops"]), 4),
            "auto_over_best_raw": round(auto / best["paired_tflops"], 4),
            "paired": finals, "configs": rows}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--shapes", default=",".join(DEFAULT_SHAPES))
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--quick", action="store_true", help="fewer group sizes and tile widths")
    ap.add_argument("--rounds", type=int, default=8, help="paired rounds for the final candidates")
    args = ap.parse_args(argv)
    from . import build

    build.build()
    capi.lib()
    ws = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")
    capi.gemm_set_workspace(ws.data_ptr(), ws.numel())
    try:
        for spec in args.shapes.split(","):
            print(json.dumps(tune_shape(spec.strip(), args.iters, args.quick, args.rounds)),
                  flush=True)
    finally:
        capi.gemm_set_workspace(None, 0)


if __name__ == "__main__":
    main()
