"""Run a named workload through the public API a given number of times.

    python -m mxfp8_master_weight_gb300.run_case CASE [--calls N] [--scale S]

Cases (seeded synthetic inputs of the workloads module):
  step        the 16384x6144 FP32 weight, one full fragment: partial amax -> fused MAX
              reduction + scale update -> partial cast (the benchmark's step)
  one_pass    the same weight through the one-pass kernel (no amax outputs)
  sharded     the config-5 batch in four emulated shards (dimensions divided by --scale):
              batched amax -> ranged reduction + scales -> batched cast
  nvfp4       the 16384x6144 FP32 weight through the NVFP4 amax, scale update and cast
  small       the 160x96 FP32 weight (config 1), one full fragment: amax -> scales -> cast
              (a launch of five tiles: the split kernels)

Every call runs the whole case; nothing is skipped.  The outputs are not checked here
(the tests check them against the oracle).  One untimed call comes first (it marshals the
library calls); then prints one line: case, calls, and the mean device time per call from
CUDA events around the timed calls.
"""
from __future__ import annotations

import argparse

import numpy as np
import torch

from . import api, build, driver
from . import workloads as wl


def _headline(dev):
    w = wl.cfg4_headline()
    return w.rows, w.cols, torch.from_numpy(w.data).to(dev)


def case_step(dev, scale):
    rows, cols, x = _headline(dev)
    sc = driver.ShardedCast([driver.WeightSpec(rows, cols, True)], [0, rows * cols], dev)
    return lambda: sc.step([x])


def case_one_pass(dev, scale):
    rows, cols, x = _headline(dev)
    (rr, rc), (cr, cc) = api.block_shapes(rows, cols)
    sr = torch.empty((rr, rc), dtype=torch.uint8, device=dev)
    scl = torch.empty((cr, cc), dtype=torch.uint8, device=dev)
    qr = torch.empty(rows * cols, dtype=torch.uint8, device=dev)
    qc = torch.empty(rows * cols, dtype=torch.uint8, device=dev)
    call = api.prepare_quantize_whole_blocks_batched([(x, None, None, sr, scl, qr, qc, rows, cols, 0)])
    return lambda: call.call()


def case_sharded(dev, scale):
    batch = wl.cfg5_sharded_batch(seed=0, scale=scale)
    specs = [driver.WeightSpec(w.rows, w.cols, w.colwise) for w in batch.weights]
    sc = driver.ShardedCast(specs, batch.bounds, dev)
    shards = [torch.from_numpy(np.ascontiguousarray(batch.shard(s))).to(dev) for s in range(sc.num_shards)]
    return lambda: sc.step(shards)


def case_nvfp4(dev, scale):
    rows, cols, x = _headline(dev)
    (rr, rc), (cr, cc) = api.nvfp4_block_shapes(rows, cols)
    ar = torch.empty((rr, rc), device=dev)
    ac = torch.empty((cr, cc), device=dev)
    at = torch.zeros(1, device=dev)
    sr = torch.empty((rr, rc), dtype=torch.uint8, device=dev)
    scl = torch.empty((cr, cc), dtype=torch.uint8, device=dev)
    qr = torch.empty(rows * cols // 2, dtype=torch.uint8, device=dev)
    qc = torch.empty(rows * cols // 2, dtype=torch.uint8, device=dev)
    calls = [api.prepare_nvfp4_partial_amax(x, ar, ac, at, rows, cols, 0),
             api.prepare_nvfp4_update_scales(ar, ac, at, sr, scl, rows, cols),
             api.prepare_nvfp4_partial_cast(x, sr, scl, at, qr, qc, rows, cols, 0)]

    def run():
        at.zero_()
        for c in calls:
            c.call()
    return run


def case_small(dev, scale):
    w = wl.cfg1_tiny()
    rows, cols = w.rows, w.cols
    x = torch.from_numpy(w.data).to(dev)
    (rr, rc), (cr, cc) = api.block_shapes(rows, cols)
    ar = torch.zeros((rr, rc), device=dev)
    ac = torch.zeros((cr, cc), device=dev)
    sr = torch.empty((rr, rc), dtype=torch.uint8, device=dev)
    scl = torch.empty((cr, cc), dtype=torch.uint8, device=dev)
    qr = torch.empty(rows * cols, dtype=torch.uint8, device=dev)
    qc = torch.empty(rows * cols, dtype=torch.uint8, device=dev)
    calls = [api.prepare_partial_amax(x, ar, ac, rows, cols, 0),
             api.prepare_update_scales(ar, ac, sr, scl, rows, cols),
             api.prepare_partial_cast(x, sr, scl, qr, qc, rows, cols, 0)]

    def run():
        for c in calls:
            c.call()
    return run


CASES = {"step": case_step, "one_pass": case_one_pass, "sharded": case_sharded, "nvfp4": case_nvfp4,
         "small": case_small}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("case", choices=sorted(CASES))
    ap.add_argument("--calls", type=int, default=4)
    ap.add_argument("--scale", type=int, default=1, help="config-5 dimensions divided by this")
    args = ap.parse_args(argv)
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    run = CASES[args.case](dev, args.scale)
    run()  # untimed: the first call marshals the library calls once
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    for _ in range(args.calls):
        run()
    b.record()
    torch.cuda.synchronize()
    print(f"{args.case}: {args.calls} calls, {a.elapsed_time(b) * 1e3 / max(1, args.calls):.2f} us per call")


if __name__ == "__main__":
    main()
