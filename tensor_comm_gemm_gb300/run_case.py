"""Run one library call on seeded synthetic inputs a few times and print its time.

A command-line tool for timing or profiling a single shape without the full
benchmark, e.g. one RS launch under a profiler:

    python -m tensor_comm_gemm_gb300.run_case --op rs --tp 8 --n 4096 --k 28672 --m 4096 --calls 3

Inputs follow the benchmark recipe (normal, sigma = K^-1/4, bf16 or e4m3 with
one amax scale per operand).  Library options can be set through the
environment (TPO_<OPTION>=value, e.g. TPO_COOPERATIVE=0).
"""

import argparse

import numpy as np
import torch

from . import synth
from . import tpoverlap as t


def _dev(a: np.ndarray) -> torch.Tensor:
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--op", choices=["ag", "rs", "ar"], required=True)
    ap.add_argument("--tp", type=int, required=True)
    ap.add_argument("--n", type=int, required=True)
    ap.add_argument("--k", type=int, required=True, help="global contraction length")
    ap.add_argument("--m", type=int, required=True)
    ap.add_argument("--dtype", choices=["bf16", "e4m3"], default="bf16")
    ap.add_argument("--chunks", type=int, default=1, help="AR row chunks")
    ap.add_argument("--calls", type=int, default=3)
    ap.add_argument("--seed", type=int, default=7)
    args = ap.parse_args(argv)
    if not torch.cuda.is_available():
        raise SystemExit("run_case needs a CUDA device")
    t.lib()
    fp8 = args.dtype == "e4m3"
    dt = t.TPO_FP8_E4M3 if fp8 else t.TPO_BF16
    sigma = 1.0 if fp8 else args.k ** -0.25
    if args.op == "ag":
        wl = synth.make_ag(args.tp, args.n, args.k, args.m, seed=args.seed, dist="normal", sigma=sigma,
                           dtype=args.dtype)
        xs, w = [_dev(x) for x in wl.x], _dev(wl.w[0])
        y = torch.empty((args.n, args.m), dtype=torch.bfloat16, device="cuda")
        sx = torch.tensor([wl.scale_inv_x], dtype=torch.float32, device="cuda") if fp8 else None
        sw = torch.tensor([wl.scale_inv_w], dtype=torch.float32, device="cuda") if fp8 else None
        ctx = t.tpo_ctx_create(args.tp, args.n, args.k, args.m, dt)
        call = lambda: t.tpo_ag_gemm(ctx, xs, w, y, sx, sw)  # noqa: E731
    else:
        wl = synth.make_ksplit(args.op, args.tp, args.n, args.k, args.m, seed=args.seed, sigma=sigma,
                               n_row_chunks=args.chunks, dtype=args.dtype)
        xs, ws = [_dev(x) for x in wl.x], [_dev(x) for x in wl.w]
        ctx = t.tpo_ctx_create(args.tp, args.n, args.k, args.m, dt)
        if fp8:
            sx = torch.tensor([wl.scale_inv_x], dtype=torch.float32, device="cuda")
            sw = torch.tensor([wl.scale_inv_w], dtype=torch.float32, device="cuda")
            t.tpo_set_fp8_scales(ctx, sx, sw)
        if args.op == "rs":
            yb = [torch.empty((args.n // args.tp, args.m), dtype=torch.bfloat16, device="cuda")
                  for _ in range(args.tp)]
            call = lambda: t.tpo_gemm_rs(ctx, xs, ws, yb)  # noqa: E731
        else:
            y = torch.empty((args.n, args.m), dtype=torch.bfloat16, device="cuda")
            call = lambda: t.tpo_gemm_ar(ctx, xs, ws, y, args.chunks)  # noqa: E731
    try:
        times = []
        for _ in range(args.calls):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            call()
            b.record()
            st = t.tpo_sync_status(ctx)
            if st:
                raise t.TpoError(st, t.tpo_last_error())
            times.append(a.elapsed_time(b))
        flops = 2.0 * args.n * args.k * args.m
        best = min(times)
        print("%s tp=%d n=%d k=%d m=%d %s: best of %d calls %.4f ms, %.1f TFLOP/s "
              "(%d producer CTAs, %d GEMM CTAs, cta_group %d)" % (
                  args.op, args.tp, args.n, args.k, args.m, args.dtype, args.calls, best,
                  flops / (best * 1e-3) / 1e12, t.tpo_get_opt(ctx, "last_producer_ctas"),
                  t.tpo_get_opt(ctx, "last_gemm_ctas"), t.tpo_get_opt(ctx, "last_cta_group")))
    finally:
        t.tpo_ctx_destroy(ctx)


if __name__ == "__main__":
    main()
