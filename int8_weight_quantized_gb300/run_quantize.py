"""Run the stand-alone activation quantize a few times on synthetic input, for profilers.

    python -m int8_weight_quantized_gb300.run_quantize --rows 4096 --cols 3072 --mode convrot

Each launch follows a 512 MiB write, so it finds neither its input nor its code in L2
(as in the bench's per-launch timing).  x is bf16 ~N(0,1); ConvRot rows get the
outlier channels of the ConvRot workload (1% of the channels scaled by 20).
"""
import argparse

import torch

import int8_weight_quantized_gb300 as ck
from int8_weight_quantized_gb300 import synthetic


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--rows", type=int, default=4096)
    ap.add_argument("--cols", type=int, default=3072)
    ap.add_argument("--mode", choices=["per_row", "convrot", "tensorwise"], default="convrot")
    ap.add_argument("--launches", type=int, default=4)
    args = ap.parse_args(argv)
    M, K = args.rows, args.cols
    dev = "cuda"
    oc = synthetic.outlier_columns(K, 0.01, seed=5 + 404) if args.mode == "convrot" else None
    x = synthetic.normal_bf16((M, K), seed=5, outlier_channels=oc).to(dev)
    q = torch.empty((M, K), dtype=torch.int8, device=dev)
    xs = torch.empty((1 if args.mode == "tensorwise" else M,), dtype=torch.float32, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    for _ in range(args.launches):
        flush.fill_(1)
        if args.mode == "tensorwise":
            ck.ck_quantize_int8_tensorwise(x, q=q, x_scale=xs)
        else:
            ck.ck_quantize_int8_rowwise(x, rotate=args.mode == "convrot", q=q, x_scale=xs)
    torch.cuda.synchronize()
    print("%d launches of the %s quantize, %d x %d" % (args.launches, args.mode, M, K))


if __name__ == "__main__":
    main()
