"""Pipelined host-staged quantisation: chunks of whole 32-row bands copied in, quantised
and copied out on three streams (the one-pass path, and the four-step partial flow with
the amax slot, MAX reduction and scale update); the host outputs equal the oracle's
whole-weight cast."""
import numpy as np
import pytest
import torch

import oracle
from mxfp8_master_weight_gb300 import api
from mxfp8_master_weight_gb300 import workloads as wl
from mxfp8_master_weight_gb300.host import HostPartialFlow, HostQuantizer

from flows import assert_bitwise

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,cols,chunk_rows,depth,colwise", [
    (1000, 512, 64, 2, True), (333, 96, 32, 3, False), (64, 4096, 1024, 3, True),
    (257, 1000, 96, 1, True)])
def test_host_pipeline_matches_oracle(rows, cols, chunk_rows, depth, colwise):
    rng = np.random.default_rng(rows + cols)
    x = wl.normal_f32(rng, rows * cols) * np.float32(10.0) ** rng.uniform(-3, 3, rows * cols).astype(np.float32)
    hq = HostQuantizer(rows, cols, colwise, chunk_rows=chunk_rows, depth=depth)
    hx = torch.from_numpy(x).pin_memory()
    (rr, rc), (cr, cc) = api.block_shapes(rows, cols)
    qr = torch.empty(rows * cols, dtype=torch.uint8).pin_memory()
    qc = torch.empty(rows * cols, dtype=torch.uint8).pin_memory() if colwise else None
    sr = torch.empty((rr, rc), dtype=torch.uint8).pin_memory()
    sc = torch.empty((cr, cc), dtype=torch.uint8).pin_memory() if colwise else None
    for _ in range(2):  # consecutive runs reuse the staging buffers
        hq.run(hx, qr, qc, sr, sc)
        torch.cuda.current_stream().synchronize()
    want = oracle.full_cast(x, rows, cols, colwise)
    got = (None, None, sr.numpy(), None if sc is None else sc.numpy(), qr.numpy(),
           None if qc is None else qc.numpy())
    assert_bitwise(got[2:], want[2:], f"host pipeline {rows}x{cols} chunk {chunk_rows}")


@pytest.mark.parametrize("direct_out", [False, True])
@pytest.mark.parametrize("rows,cols,chunk_rows,depth,colwise,dtype", [
    (1000, 512, 64, 2, True, "f32"), (333, 96, 32, 3, False, "f32"), (64, 4096, 1024, 3, True, "f32"),
    (257, 1000, 96, 1, True, "f32"), (400, 640, 128, 3, True, "bf16")])
def test_host_partial_flow_matches_oracle(rows, cols, chunk_rows, depth, colwise, dtype, direct_out):
    """Three calls in a row (the device input alternates between two buffers, the amax
    slot, staging buffers and scales are reused), each with new values; with direct_out
    the casts store into the pinned host outputs themselves (new output buffers on the
    second call, the same ones again on the third)."""
    (rr, rc), (cr, cc) = api.block_shapes(rows, cols)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    flow = HostPartialFlow(rows, cols, colwise, dtype=tdt, chunk_rows=chunk_rows, depth=depth,
                           direct_out=direct_out)
    keep = None
    for call in range(3):
        rng = np.random.default_rng(rows + cols + call)
        x = wl.normal_f32(rng, rows * cols) * np.float32(10.0) ** rng.uniform(-3, 3, rows * cols).astype(np.float32)
        if dtype == "bf16":
            x = wl.truncate_to_bf16_bits(x)
            hx = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory()
        else:
            hx = torch.from_numpy(x).pin_memory()
        if call == 2 and keep is not None:
            qr, qc = keep
            qr.fill_(0xA5)
            if qc is not None:
                qc.fill_(0xA5)
        else:
            qr = torch.full((rows * cols,), 0xA5, dtype=torch.uint8).pin_memory()
            qc = torch.full((rows * cols,), 0xA5, dtype=torch.uint8).pin_memory() if colwise else None
        keep = (qr, qc)
        sr = torch.empty((rr, rc), dtype=torch.uint8).pin_memory()
        sc = torch.empty((cr, cc), dtype=torch.uint8).pin_memory() if colwise else None
        flow.run(hx, qr, qc, sr, sc)
        torch.cuda.current_stream().synchronize()
        want = oracle.full_cast(x, rows, cols, colwise)
        got = (sr.numpy(), None if sc is None else sc.numpy(), qr.numpy(),
               None if qc is None else qc.numpy())
        assert_bitwise(got, want[2:], f"partial flow {rows}x{cols} chunk {chunk_rows} call {call}")
        assert flow.launches_per_run() == 2 * len(flow.chunks) + 1


def test_host_pipeline_rejects_pageable_memory():
    hq = HostQuantizer(64, 64, False)
    with pytest.raises(ValueError, match="pinned"):
        hq.run(torch.zeros(64 * 64), torch.zeros(64 * 64, dtype=torch.uint8))


@pytest.mark.parametrize("rows,cols,colwise", [(1000, 512, True), (333, 96, False), (16384, 6144, True)])
def test_zero_copy_matches_oracle(rows, cols, colwise):
    from mxfp8_master_weight_gb300.host import ZeroCopyQuantizer
    rng = np.random.default_rng(rows * 3 + cols)
    x = wl.normal_f32(rng, rows * cols) * np.float32(10.0) ** rng.uniform(-3, 3, rows * cols).astype(np.float32)
    (rr, rc), (cr, cc) = api.block_shapes(rows, cols)
    hx = torch.from_numpy(x).pin_memory()
    qr = torch.full((rows * cols,), 0xA5, dtype=torch.uint8).pin_memory()
    qc = torch.full((rows * cols,), 0xA5, dtype=torch.uint8).pin_memory() if colwise else None
    sr = torch.empty((rr, rc), dtype=torch.uint8).pin_memory()
    sc = torch.empty((cr, cc), dtype=torch.uint8).pin_memory() if colwise else None
    ZeroCopyQuantizer(rows, cols, colwise).run(hx, qr, qc, sr, sc)
    torch.cuda.synchronize()
    want = oracle.full_cast(x, rows, cols, colwise)
    got = (None, None, sr.numpy(), None if sc is None else sc.numpy(), qr.numpy(),
           None if qc is None else qc.numpy())
    assert_bitwise(got[2:], want[2:], f"zero-copy {rows}x{cols}")


def test_zero_copy_refuses_pageable_memory():
    from mxfp8_master_weight_gb300.host import ZeroCopyQuantizer
    assert api.device_can_access(torch.empty(16, device="cuda"))
    assert api.device_can_access(torch.empty(16).pin_memory())
    assert not api.device_can_access(torch.empty(16))
    with pytest.raises(ValueError, match="page-locked"):
        ZeroCopyQuantizer(32, 32, False).run(torch.zeros(32 * 32), torch.zeros(32 * 32, dtype=torch.uint8).pin_memory(),
                                              None, torch.zeros((32, 1), dtype=torch.uint8).pin_memory(), None)
