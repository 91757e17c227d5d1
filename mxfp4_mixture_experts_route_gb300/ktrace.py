"""Timeline of one step of the block from the library's trace build.

In the trace build (-DMOE_TRACE) every kernel's CTAs stamp %globaltimer at
their start (point 0), when their wait on the preceding kernel returns (1), at
their end (2) and at kernel-specific inner points (3..7); the library keeps
the earliest and the latest stamp of each point over a step's CTAs
(moe_ktrace).  On a GPU, from the repository root:

    python -m mxfp4_mixture_experts_route_gb300.ktrace [--config 1] [--latent] [--reps 30]

It builds libmoe_trace.so beside libmoe.so, runs the step as the benchmark
does (the L2 flushed before it, the step enqueued while the flush runs) and
prints, per kernel and point, the median over the repetitions of the earliest
and the latest stamp, in microseconds from the step's first CTA.
"""
from __future__ import annotations

import argparse
import ctypes
import os
import statistics
import sys

import numpy as np

from . import build as _build

POINTS = 8


def trace_library() -> str:
    return _build.build_library(["-DMOE_TRACE"], lib_path=os.path.join(_build.LIBDIR, "libmoe_trace.so"),
                                build_dir=os.path.join(_build.PKG, "_build_trace"))


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--config", type=int, default=1, help="workload index (moe_inputs.CONFIGS)")
    ap.add_argument("--latent", action="store_true", help="the latent-MoE layer (moe_inputs.LATENT_CONFIGS)")
    ap.add_argument("--reps", type=int, default=30)
    args = ap.parse_args(argv)

    import torch

    sys.path.insert(0, os.getcwd())
    import bench
    import moe_inputs as mi
    import mxfp4_mixture_experts_route_gb300 as moe

    lib = moe.load_library(trace_library())
    lib.moe_ktrace.argtypes = [ctypes.c_void_p, ctypes.c_size_t]
    lib.moe_kernel_name.restype = ctypes.c_char_p
    moe._lib = lib
    dev = torch.device("cuda")
    if args.latent:
        lc = mi.LATENT_CONFIGS[args.config]
        name = lc.name
        inp = mi.make_latent_inputs(lc)
        shape = moe.LatentShape.of(lc.S, lc.H, lc.LAT, lc.E, lc.k, lc.I, lc.SI, logit_offset=bool(lc.zipf),
                                   norm_eps=lc.norm_eps)
        blk = moe.DeviceLatentWeights(shape, inp.x, inp.w_gate, inp.bias, inp.logit_off, inp.w_ld, inp.w13,
                                      inp.w13s, inp.w2, inp.w2s, inp.ln_w, inp.w_up, inp.w_sgu, inp.w_sd,
                                      device=dev)
    else:
        cfg = mi.CONFIGS[args.config]
        name = cfg.name
        blk = bench.upload(moe, cfg, mi.make_inputs(cfg), dev)
    flush = bench.L2Flush(dev, torch.cuda.get_device_properties(dev).L2_cache_size)
    stream = torch.cuda.current_stream(dev)
    step_ms = bench.timed_steps(blk.forward, 50, flush, stream, warmup=10)

    n_kernels = 0
    while lib.moe_kernel_name(n_kernels) is not None:
        n_kernels += 1
    tables = []
    for _ in range(args.reps):
        torch.cuda.synchronize(dev)
        if lib.moe_ktrace(None, 0) != 0:
            raise RuntimeError("moe_ktrace reset failed")
        flush.zero_()      # the step is enqueued while the flush runs
        blk.forward()
        buf = np.zeros((n_kernels, 2 * POINTS), np.uint64)
        if lib.moe_ktrace(buf.ctypes.data, buf.nbytes) != 0:
            raise RuntimeError("moe_ktrace read failed")
        tables.append(buf.astype(np.int64))
    moe.check_device_status(blk.ws, "traced steps")
    t = np.stack(tables)                       # [reps, kernel, 2 * point]
    used = [k for k in range(n_kernels) if t[0, k, 5] > 0]
    t0 = np.min(t[:, used, 0], axis=1)         # the step's first CTA start, per repetition
    print(f"{name}: step {statistics.fmean(step_ms) * 1e3:.2f} us (median {statistics.median(step_ms) * 1e3:.2f}); "
          f"points in us from the step's first CTA, median of {args.reps}: earliest/latest over CTAs")
    print("  0 start, 1 wait returns, 2 end, 3..7 kernel-specific")
    for k in sorted(used, key=lambda k: float(np.median(t[:, k, 0] - t0))):
        parts = []
        for pt in range(POINTS):
            lo, hi = t[:, k, 2 * pt], t[:, k, 2 * pt + 1]
            if hi[0] == 0:
                continue
            parts.append(f"{pt}:{np.median(lo - t0) / 1e3:.2f}/{np.median(hi - t0) / 1e3:.2f}")
        print(f"  {lib.moe_kernel_name(k).decode():18s} " + "  ".join(parts))
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
