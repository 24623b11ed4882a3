"""Measured tile-configuration sweep of the INT8 GEMM on the current GPU.

For each M x N x K problem the GEMM is timed with every tile configuration it supports
(CTA pairs with 256-row tiles or single CTAs with 128-row tiles, times tile widths 32,
64, ..., 256 output columns; each without and, where the last wave is partial, with the
K-split of that wave) and with the configuration the library picks by itself
(ck_gemm_tile_config).  The report gives, per shape, the picked and the best
configuration and the regret of the pick: the per-shape tile sweep of the comfy-kitchen
pages (issue #280, "Kernel used": one fixed config found best on every H3 shape; the
A6000 tile-chooser discussion it links to: a measured table per GPU), done here against
the library's own per-launch choice.

  python -m int8_weight_quantized_gb300.tune [--shapes 4096x4096x4096,...] [--reps 5]
                                             [--json out.json] [--markdown out.md]

Only the GEMM kernel is timed (CUDA events around it, via ck_profile_begin); L2 is
flushed before every timed launch (a 512 MiB write, then a 256 MiB read so no dirty
lines are left to write back).  The configurations of a shape are timed in rounds (one
launch of each per round) and the median over the rounds is kept, so clock drift under
the power cap does not favour the configurations timed first.  Forcing a configuration uses the library's A/B
overrides CK_GEMM_PAIR / CK_GEMM_BN / CK_GEMM_SPLIT, set in this process's environment.
"""
import argparse
import json
import os
import statistics
import sys

import torch

from . import ck_gemm_tile_config, ck_int8_gemm_dequant, ck_profile_begin, ck_profile_end, synthetic

DEFAULT_SHAPES = [
    (4096, 4096, 4096), (274, 2048, 2048), (1024, 4096, 4096), (8192, 16384, 4096), (25900, 16384, 4096),
    (4096, 12288, 3072), (80666, 28672, 5376), (99865, 21504, 5376),
]
WIDTHS = list(range(256, 0, -32))
FLUSH_BYTES = 512 << 20
CLEAN_BYTES = 256 << 20


def parse_shapes(text):
    out = []
    for item in text.split(","):
        m, n, k = (int(v) for v in item.lower().split("x"))
        out.append((m, n, k))
    return out


def _set_override(pair, bn, split=None):
    for key, val in (("CK_GEMM_PAIR", pair), ("CK_GEMM_BN", bn), ("CK_GEMM_SPLIT", split)):
        if val is None:
            os.environ.pop(key, None)
        else:
            os.environ[key] = str(val)


def flush_l2(flush):
    flush[0].zero_()
    torch.sum(flush[1], dim=0, out=flush[2])


def _launch_ms(args, flush, cfg):
    """One flushed, event-bracketed GEMM launch with configuration cfg = (pair, bn, split)
    forced (pair None = the library's own pick; split 1 = no K-split)."""
    pair, bn, split = cfg
    _set_override(None if pair is None else (1 if pair else 0), bn, split)
    try:
        flush_l2(flush)
        ck_profile_begin(with_events=True)
        ck_int8_gemm_dequant(*args)
        return ck_profile_end()["gemm"][0]
    finally:
        _set_override(None, None)


def sweep_shape(M, N, K, reps, flush, seed=7):
    """Every configuration of one shape, timed in rounds: each round launches every
    configuration once, so a drift of the clocks (the power cap of long launches) hits all
    of them alike; the median over the rounds is reported."""
    dev = "cuda"
    q = synthetic.int8_uniform((M, K), seed, device=dev)
    w = synthetic.int8_uniform((N, K), seed + 1, device=dev)
    xs = synthetic.scale_uniform(M, seed + 2, mul=0.02, device=dev)
    ws = synthetic.scale_uniform(N, seed + 3, mul=0.01, device=dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    args = (q, xs, w, ws, None, False, y)
    pick_bn, pick_pair, resident, pick_split = ck_gemm_tile_config(M, N, K)
    cfgs = {}
    pairs = [True, False] if (M + 127) // 128 >= 2 else [False]
    for pair in pairs:
        for bn in WIDTHS:
            name = "%s/%d" % ("pair" if pair else "single", bn)
            cfgs[name] = (pair, bn, 1)
            _set_override(1 if pair else 0, bn)
            split = ck_gemm_tile_config(M, N, K)[3]
            _set_override(None, None)
            if split > 1:
                cfgs["%s/split%d" % (name, split)] = (pair, bn, None)
    cfgs["picked"] = (None, None, None)
    for cfg in cfgs.values():  # warm-up: every instance loaded, attributes set
        for _ in range(2):
            _launch_ms(args, flush, cfg)
    samples = {name: [] for name in cfgs}
    for _ in range(reps):
        for name, cfg in cfgs.items():
            samples[name].append(_launch_ms(args, flush, cfg))
    configs = {name: statistics.median(v) for name, v in samples.items() if name != "picked"}
    picked_ms = statistics.median(samples["picked"])
    best = min(configs, key=configs.get)
    flops = 2.0 * M * N * K
    del q, w, xs, ws, y
    torch.cuda.empty_cache()
    return {
        "shape": [M, N, K],
        "picked": "%s/%d%s" % ("pair" if pick_pair else "single", pick_bn,
                               "/split%d" % pick_split if pick_split > 1 else ""),
        "picked_ms": picked_ms,
        "picked_tflops": flops / picked_ms / 1e9,
        "best": best,
        "best_ms": configs[best],
        "best_tflops": flops / configs[best] / 1e9,
        "regret": picked_ms / configs[best] - 1.0,
        "resident_units": resident,
        "configs_ms": configs,
    }


def markdown(results):
    lines = ["| M x N x K | picked | ms | TFLOP/s | best measured | ms | TFLOP/s | regret |",
             "|---|---|---|---|---|---|---|---|"]
    for r in results:
        lines.append("| %s | %s | %.4f | %.0f | %s | %.4f | %.0f | %+.1f%% |" % (
            "x".join(str(v) for v in r["shape"]), r["picked"], r["picked_ms"], r["picked_tflops"], r["best"],
            r["best_ms"], r["best_tflops"], 100.0 * r["regret"]))
    return "\n".join(lines)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--shapes", type=parse_shapes, default=DEFAULT_SHAPES)
    ap.add_argument("--reps", type=int, default=5)
    ap.add_argument("--json", default=None)
    ap.add_argument("--markdown", default=None)
    a = ap.parse_args(argv)
    if not torch.cuda.is_available():
        sys.exit("tune: needs a CUDA device")
    flush = (torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda"),
             torch.zeros(CLEAN_BYTES // 8, dtype=torch.int64, device="cuda"),
             torch.empty((), dtype=torch.int64, device="cuda"))
    results = []
    for M, N, K in a.shapes:
        r = sweep_shape(M, N, K, a.reps, flush)
        results.append(r)
        print("%dx%dx%d picked %s %.4f ms, best %s %.4f ms (%+.1f%%)" % (
            M, N, K, r["picked"], r["picked_ms"], r["best"], r["best_ms"], 100 * r["regret"]), flush=True)
    text = markdown(results)
    print(text)
    if a.json:
        with open(a.json, "w") as f:
            json.dump({"device": torch.cuda.get_device_name(), "results": results}, f, indent=1)
    if a.markdown:
        with open(a.markdown, "w") as f:
            f.write(text + "\n")


if __name__ == "__main__":
    main()
