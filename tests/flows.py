"""Shared helpers for the GPU parity tests: run one fragment through the CUDA library
(via the C ABI binding) and through the CPU oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from mxfp8_master_weight_gb300 import api


def to_device(x: np.ndarray, shift: int = 0) -> torch.Tensor:
    """Device copy of a float32 / bf16-bits array, placed `shift` elements into a larger
    allocation (so the data pointer can be deliberately misaligned to 16 bytes)."""
    n = x.size
    if x.dtype == np.float32:
        buf = torch.empty(n + shift + 8, dtype=torch.float32, device="cuda")
        t = buf[shift:shift + n]
        t.copy_(torch.from_numpy(np.ascontiguousarray(x).reshape(-1)))
    else:
        buf = torch.empty(n + shift + 8, dtype=torch.bfloat16, device="cuda")
        t = buf[shift:shift + n]
        t.view(torch.int16).copy_(torch.from_numpy(np.ascontiguousarray(x).reshape(-1).view(np.int16)))
    return t


def to_host(t: torch.Tensor) -> np.ndarray:
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def torch_dtype(x: np.ndarray):
    return torch.float32 if x.dtype == np.float32 else torch.bfloat16


def gpu_fragment(frag: np.ndarray, rows: int, cols: int, start: int, colwise: bool, *,
                 out_offset: int | None = None, out_size: int | None = None, shift: int = 0,
                 pad: int = 0, pad_s: int | None = None, amax_fill: float = 0.0,
                 sentinel: int = 0xA5, model: str = "bf16"):
    """amax -> scales -> cast of one fragment on the GPU.  Returns host arrays
    (amax_r, amax_c, scale_r, scale_c, q_r, q_c); columnwise items None when absent.
    `pad` extra columns pad the amax grids, `pad_s` (default `pad`) the scale grids."""
    pad_s = pad if pad_s is None else pad_s
    (rr, rc), (cr, cc) = api.block_shapes(rows, cols)
    dt = torch_dtype(frag)
    x = to_device(frag, shift)
    ar = torch.full((rr, rc + pad), amax_fill, dtype=dt, device="cuda")
    ac = torch.full((cr, cc + pad), amax_fill, dtype=dt, device="cuda") if colwise else None
    api.mxfp8_partial_amax(x, ar, ac, rows, cols, start)
    sr = torch.full((rr, rc + pad_s), 0xEE, dtype=torch.uint8, device="cuda")
    sc = torch.full((cr, cc + pad_s), 0xEE, dtype=torch.uint8, device="cuda") if colwise else None
    api.mxfp8_update_scales(ar, ac, sr, sc, rows, cols)
    if out_offset is None:
        out_offset = start
    if out_size is None:
        out_size = rows * cols if out_offset == start else frag.size + out_offset
    qr = torch.full((out_size,), sentinel, dtype=torch.uint8, device="cuda")
    qc = torch.full((out_size,), sentinel, dtype=torch.uint8, device="cuda") if colwise else None
    api.mxfp8_partial_cast(x, sr, sc, qr, qc, rows, cols, start, out_offset, model_dtype=model)
    torch.cuda.synchronize()
    h = lambda t: None if t is None else to_host(t)
    return h(ar), h(ac), h(sr), h(sc), h(qr), h(qc)


def oracle_fragment(frag: np.ndarray, rows: int, cols: int, start: int, colwise: bool, *,
                    out_offset: int | None = None, out_size: int | None = None, pad: int = 0,
                    pad_s: int | None = None, amax_fill: float = 0.0, sentinel: int = 0xA5,
                    model: str = "bf16"):
    """The same step sequence on the CPU oracle."""
    pad_s = pad if pad_s is None else pad_s
    (rr, rc), (cr, cc) = api.block_shapes(rows, cols)
    npdt = frag.dtype
    fill = np.array([amax_fill], np.float32)
    if npdt == np.uint16:
        fill = (fill.view(np.uint32) >> 16).astype(np.uint16)
    ar = np.full((rr, rc + pad), fill[0], npdt)
    ac = np.full((cr, cc + pad), fill[0], npdt) if colwise else None
    oracle.partial_amax(frag, rows, cols, start, ar, ac)
    sr = np.full((rr, rc + pad_s), 0xEE, np.uint8)
    oracle.update_scales(ar, rr, rc, sr)
    sc = None
    if colwise:
        sc = np.full((cr, cc + pad_s), 0xEE, np.uint8)
        oracle.update_scales(ac, cr, cc, sc)
    if out_offset is None:
        out_offset = start
    if out_size is None:
        out_size = rows * cols if out_offset == start else frag.size + out_offset
    qr = np.full(out_size, sentinel, np.uint8)
    qc = np.full(out_size, sentinel, np.uint8) if colwise else None
    oracle.partial_cast(frag, rows, cols, start, sr, sc, qr, qc, out_offset, model=model)
    return ar, ac, sr, sc, qr, qc


NAMES = ("amax_rowwise", "amax_colwise", "scale_rowwise", "scale_colwise", "data_rowwise",
         "data_colwise")


def assert_bitwise(got, want, ctx=""):
    for name, g, w in zip(NAMES, got, want):
        if w is None:
            assert g is None, f"{ctx} {name}: expected absent"
            continue
        g = np.asarray(g)
        w = np.asarray(w)
        assert g.shape == w.shape, f"{ctx} {name}: shape {g.shape} != {w.shape}"
        gb = g.view(np.uint32) if g.dtype == np.float32 else g
        wb = w.view(np.uint32) if w.dtype == np.float32 else w
        if not np.array_equal(gb, wb):
            bad = np.flatnonzero(gb.reshape(-1) != wb.reshape(-1))
            k = bad[0]
            raise AssertionError(f"{ctx} {name}: {bad.size} mismatches, first at flat {k}: "
                                 f"gpu {gb.reshape(-1)[k]} oracle {wb.reshape(-1)[k]}")
