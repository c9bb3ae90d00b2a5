"""Runs one libbfp8 kernel configuration a few times, for profilers.

    python profile_case.py --M 2048 --N 4096 --K 4096 --iters 2
    python profile_case.py --M 8192 --K 4096 --quant --iters 2

Inputs are seeded synthetic data of the bench's distributions (bf16 N(0,1)
activations, e4m3 weights from U[-448, 448], weight scales U[1e-4, 1e-2)).
With --quant only the quantisation kernel runs; otherwise the activations are
quantised once and the GEMM launches --iters times (profile with `-s 1` to skip
the first launch).
"""
from __future__ import annotations

import argparse

import torch

import block_scaled_fp8_02_gb300 as bf
from block_scaled_fp8_02_gb300 import workloads as wl


def main() -> None:
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--M", type=int, required=True)
    p.add_argument("--N", type=int, default=4096)
    p.add_argument("--K", type=int, default=4096)
    p.add_argument("--iters", type=int, default=3)
    p.add_argument("--quant", action="store_true", help="run only the quantisation kernel")
    p.add_argument("--schedule", type=int, default=0)
    p.add_argument("--tile_n", type=int, default=0)
    a = p.parse_args()
    dev = torch.device("cuda:0")
    x = wl.activations(a.M, a.K, seed=1).to(dev)
    if a.quant:
        for _ in range(a.iters):
            bf.bfp8_group_quant(x)
    else:
        case = wl.linear_case(1, a.N, a.K, seed=2)
        B, Bs = case["B"].to(dev), case["Bs"].to(dev)
        q, s = bf.bfp8_group_quant(x)
        opts = {"schedule": a.schedule, "tile_n": a.tile_n}
        for _ in range(a.iters):
            bf.bfp8_gemm(q, B, s, Bs, options=opts)
    torch.cuda.synchronize()
    print("ok")


if __name__ == "__main__":
    main()
