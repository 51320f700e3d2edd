"""Quantise a host-resident master weight through the GPU, pipelined.

For master weights that live in host memory (an optimizer that keeps them on the
CPU), one update is: copy the weight in, quantise, copy the E4M3 data and E8M0
scales out.  The weight is cut into chunks of whole 32-row bands, so every 1x32 and
32x1 block lies inside one chunk and each chunk is quantised on its own by the
one-pass kernel (``mxfp8_quantize_whole_blocks``) with results identical to
quantising the whole weight.  Chunk k+1 is copied in while chunk k is quantised and
chunk k-1 is copied out: three CUDA streams ordered by events, ``depth`` device
staging buffers allocated once, host buffers pinned.  All arithmetic runs in the
library's kernels; this module only orders copies and launches.
"""
from __future__ import annotations

import torch

from . import api


class HostQuantizer:
    """Pipelined host -> device -> host MXFP8 quantisation of one rows x cols weight."""

    def __init__(self, rows: int, cols: int, colwise: bool = True, dtype=torch.float32,
                 device="cuda", chunk_rows: int = 1024, depth: int = 3, model_dtype="bf16"):
        if rows <= 0 or cols <= 0:
            raise ValueError("rows and cols must be positive")
        self.rows, self.cols, self.colwise, self.dtype = rows, cols, colwise, dtype
        self.device = torch.device(device)
        self.model_dtype = model_dtype
        self.chunk_rows = max(32, min((chunk_rows + 31) // 32 * 32, (rows + 31) // 32 * 32))
        self.depth = max(1, depth)
        n = self.chunk_rows * cols
        with torch.cuda.device(self.device):
            self.dev_in = [torch.empty(n, dtype=dtype, device=self.device) for _ in range(self.depth)]
            self.dev_qr = [torch.empty(n, dtype=torch.uint8, device=self.device)
                           for _ in range(self.depth)]
            self.dev_qc = [torch.empty(n, dtype=torch.uint8, device=self.device)
                           for _ in range(self.depth)] if colwise else None
            (rr, rc), (cr, cc) = api.block_shapes(rows, cols)
            self.scale_r = torch.empty((rr, rc), dtype=torch.uint8, device=self.device)
            self.scale_c = torch.empty((cr, cc), dtype=torch.uint8, device=self.device) if colwise else None
            self.h2d, self.comp, self.d2h = (torch.cuda.Stream(self.device) for _ in range(3))
            self.in_ready = [torch.cuda.Event() for _ in range(self.depth)]
            self.comp_done = [torch.cuda.Event() for _ in range(self.depth)]
            self.d2h_done = [torch.cuda.Event() for _ in range(self.depth)]

    @property
    def chunks(self):
        return [(r0, min(self.rows, r0 + self.chunk_rows))
                for r0 in range(0, self.rows, self.chunk_rows)]

    def launches_per_run(self) -> int:
        return len(self.chunks)

    def run(self, host_x: torch.Tensor, host_qr: torch.Tensor, host_qc: torch.Tensor | None = None,
            host_sr: torch.Tensor | None = None, host_sc: torch.Tensor | None = None) -> None:
        """Quantise ``host_x`` (pinned, rows*cols elements) into the pinned host outputs.

        Asynchronous with respect to the host: the caller's current stream is made to
        wait for the last copy, so synchronising it (or an event recorded on it after
        this call) makes the outputs valid.
        """
        rows, cols = self.rows, self.cols
        for t, name in ((host_x, "host_x"), (host_qr, "host_qr"), (host_qc, "host_qc"),
                        (host_sr, "host_sr"), (host_sc, "host_sc")):
            if t is not None and (t.is_cuda or not t.is_pinned()):
                raise ValueError(f"{name} must be pinned host memory")
        if host_x.numel() != rows * cols or host_qr.numel() != rows * cols:
            raise ValueError("host_x and host_qr must hold rows*cols elements")
        if self.colwise != (host_qc is not None):
            raise ValueError("host_qc is required exactly when the weight is bidirectional")
        x, qr = host_x.reshape(-1), host_qr.reshape(-1)
        qc = host_qc.reshape(-1) if host_qc is not None else None
        caller = torch.cuda.current_stream(self.device)
        self.h2d.wait_stream(caller)
        self.comp.wait_stream(caller)
        self.d2h.wait_stream(caller)
        for k, (r0, r1) in enumerate(self.chunks):
            s = k % self.depth
            a, b = r0 * cols, r1 * cols
            n = b - a
            with torch.cuda.stream(self.h2d):
                self.h2d.wait_event(self.comp_done[s])  # chunk k - depth has read dev_in[s]
                self.dev_in[s][:n].copy_(x[a:b], non_blocking=True)
                self.in_ready[s].record(self.h2d)
            with torch.cuda.stream(self.comp):
                self.comp.wait_event(self.in_ready[s])
                self.comp.wait_event(self.d2h_done[s])  # chunk k - depth has left dev_q*[s]
                api.mxfp8_quantize_whole_blocks(
                    self.dev_in[s][:n], None, None, self.scale_r, self.scale_c,
                    self.dev_qr[s][:n], self.dev_qc[s][:n] if self.colwise else None,
                    rows, cols, a, 0, stream=self.comp, model_dtype=self.model_dtype)
                self.comp_done[s].record(self.comp)
            with torch.cuda.stream(self.d2h):
                self.d2h.wait_event(self.comp_done[s])
                qr[a:b].copy_(self.dev_qr[s][:n], non_blocking=True)
                if qc is not None:
                    qc[a:b].copy_(self.dev_qc[s][:n], non_blocking=True)
                self.d2h_done[s].record(self.d2h)
        with torch.cuda.stream(self.d2h):
            self.d2h.wait_stream(self.comp)
            if host_sr is not None:
                host_sr.copy_(self.scale_r, non_blocking=True)
            if host_sc is not None and self.scale_c is not None:
                host_sc.copy_(self.scale_c, non_blocking=True)
        caller.wait_stream(self.d2h)


class ZeroCopyQuantizer:
    """One launch that reads the page-locked host master weight and writes the page-locked
    host outputs directly over the coherent CPU-GPU link (no staging copies).

    Every buffer is checked to be device-accessible before the launch (pageable host
    memory is rejected with ValueError).  The one-pass kernel reads each tile twice; the
    second read is served from the GPU's L2.
    """

    def __init__(self, rows: int, cols: int, colwise: bool = True, device="cuda"):
        self.rows, self.cols, self.colwise = rows, cols, colwise
        self.device = torch.device(device)

    def launches_per_run(self) -> int:
        return 1

    def run(self, host_x: torch.Tensor, host_qr: torch.Tensor, host_qc: torch.Tensor | None,
           host_sr: torch.Tensor, host_sc: torch.Tensor | None) -> None:
        if self.colwise != (host_qc is not None):
            raise ValueError("host_qc is required exactly when the weight is bidirectional")
        with torch.cuda.device(self.device):
            api.mxfp8_quantize_whole_blocks(host_x.reshape(-1), None, None, host_sr, host_sc,
                                            host_qr.reshape(-1),
                                            None if host_qc is None else host_qc.reshape(-1),
                                            self.rows, self.cols, 0, allow_host=True)


class HostPartialFlow:
    """The four-step partial flow on a host-resident master weight, pipelined with the copies.

    Partial amax -> packed MAX reduction fused with the scale update -> partial cast, as a
    rank of the distributed writeback runs it ("Support row-only MXFP8 distributed
    master-weight casts", flow diagram), for a weight whose master copy lives in pinned
    host memory.  The weight is cut into chunks of whole 32-row bands, each a fragment of
    the weight: chunk k's block maxima are taken as soon as its copy has landed (while
    chunk k+1 is still being copied in), every chunk writing its own blocks of the one
    amax slot; after the last chunk the slot is reduced and the scales are derived; then
    every chunk is cast straight into the pinned host outputs over the CPU-GPU link
    (``direct_out``, the default), or -- ``direct_out=False`` -- chunk k is cast into a
    staging buffer while chunk k-1's E4M3 bytes are copied out by the copy engine.
    The device input is double-buffered across calls, so one call's copy-in overlaps the
    previous call's copy-out.  All arithmetic runs in the library's kernels; this class
    only orders copies and launches on three streams.
    """

    def __init__(self, rows: int, cols: int, colwise: bool = True, dtype=torch.float32,
                 device="cuda", chunk_rows: int = 4096, depth: int = 3, direct_out: bool = True):
        if rows <= 0 or cols <= 0:
            raise ValueError("rows and cols must be positive")
        self.rows, self.cols, self.colwise, self.dtype = rows, cols, colwise, dtype
        # direct_out: each chunk's cast stores its E4M3 bytes straight into the pinned host
        # outputs over the CPU-GPU link (no staging buffers, no copy engine on the way out)
        self.direct_out = direct_out
        self._direct = None
        self.device = torch.device(device)
        self.chunk_rows = max(32, min((chunk_rows + 31) // 32 * 32, (rows + 31) // 32 * 32))
        self.depth = max(1, depth)
        n = rows * cols
        cn = self.chunk_rows * cols
        (rr, rc), (cr, cc) = api.block_shapes(rows, cols)
        with torch.cuda.device(self.device):
            self.dev_x = [torch.empty(n, dtype=dtype, device=self.device) for _ in range(2)]
            entries = rr * rc + (cr * cc if colwise else 0)
            self.slot = torch.zeros((1, entries), dtype=dtype, device=self.device)
            self.reduced = torch.zeros(entries, dtype=dtype, device=self.device)
            self.amax_r = self.slot[0, :rr * rc].view(rr, rc)
            self.amax_c = self.slot[0, rr * rc:].view(cr, cc) if colwise else None
            red_r = self.reduced[:rr * rc].view(rr, rc)
            red_c = self.reduced[rr * rc:].view(cr, cc) if colwise else None
            self.scale_r = torch.empty((rr, rc), dtype=torch.uint8, device=self.device)
            self.scale_c = torch.empty((cr, cc), dtype=torch.uint8, device=self.device) if colwise else None
            self.dev_qr = [torch.empty(cn, dtype=torch.uint8, device=self.device) for _ in range(self.depth)]
            self.dev_qc = ([torch.empty(cn, dtype=torch.uint8, device=self.device) for _ in range(self.depth)]
                           if colwise else None)
            self.h2d, self.comp, self.d2h = (torch.cuda.Stream(self.device) for _ in range(3))
            self.in_ready = [torch.cuda.Event() for _ in self.chunks]
            self.x_free = [torch.cuda.Event() for _ in range(2)]
            self.comp_done = [torch.cuda.Event() for _ in range(self.depth)]
            self.d2h_done = [torch.cuda.Event() for _ in range(self.depth)]
            self.scales_out = torch.cuda.Event()
        # one marshalled library call per chunk and phase, for each device input buffer
        self._amax = [[api.prepare_partial_amax(self.dev_x[b][r0 * cols:r1 * cols], self.amax_r,
                                                self.amax_c, rows, cols, r0 * cols)
                       for r0, r1 in self.chunks] for b in range(2)]
        self._reduce = api.prepare_amax_max_reduce_update_scales(
            self.slot, self.reduced, [(red_r, red_c, self.scale_r, self.scale_c, rows, cols)])
        self._cast = [[api.prepare_partial_cast(
            self.dev_x[b][r0 * cols:r1 * cols], self.scale_r, self.scale_c,
            self.dev_qr[k % self.depth][:(r1 - r0) * cols],
            self.dev_qc[k % self.depth][:(r1 - r0) * cols] if colwise else None,
            rows, cols, r0 * cols, 0) for k, (r0, r1) in enumerate(self.chunks)] for b in range(2)]
        self._calls = 0

    @property
    def chunks(self):
        return [(r0, min(self.rows, r0 + self.chunk_rows))
                for r0 in range(0, self.rows, self.chunk_rows)]

    def launches_per_run(self) -> int:
        """Library kernel launches of one call: an amax and a cast per chunk, one reduction."""
        return 2 * len(self.chunks) + 1

    def run(self, host_x: torch.Tensor, host_qr: torch.Tensor, host_qc: torch.Tensor | None,
            host_sr: torch.Tensor, host_sc: torch.Tensor | None) -> None:
        """Quantise ``host_x`` (pinned, rows*cols elements) into the pinned host outputs.

        Asynchronous with respect to the host, like HostQuantizer.run: the caller's
        current stream waits for the last copy out.  ``host_x`` must hold its values
        when run() is called (the copy-in is not ordered after GPU work queued on the
        caller's stream); the host outputs may not be read before that stream reaches
        this call's end."""
        rows, cols = self.rows, self.cols
        for t, name in ((host_x, "host_x"), (host_qr, "host_qr"), (host_qc, "host_qc"),
                        (host_sr, "host_sr"), (host_sc, "host_sc")):
            if t is not None and (t.is_cuda or not t.is_pinned()):
                raise ValueError(f"{name} must be pinned host memory")
        if host_x.numel() != rows * cols or host_qr.numel() != rows * cols:
            raise ValueError("host_x and host_qr must hold rows*cols elements")
        if self.colwise != (host_qc is not None) or self.colwise != (host_sc is not None):
            raise ValueError("host_qc and host_sc are required exactly when the weight is bidirectional")
        if host_x.dtype != self.dtype:
            raise ValueError("host_x has the wrong dtype")
        x, qr = host_x.reshape(-1), host_qr.reshape(-1)
        qc = host_qc.reshape(-1) if host_qc is not None else None
        b = self._calls % 2
        self._calls += 1
        caller = torch.cuda.current_stream(self.device)
        if self.direct_out:
            self._run_direct(x, qr, qc, host_sr, host_sc, b, caller)
            return
        # The copy-in reads host memory only: it does not wait for the caller's stream
        # (which, after a previous call, waits for that call's copies out), so one call's
        # copy-in overlaps the previous call's copy-out.  Kernels and copies out follow
        # the caller's stream.
        self.comp.wait_stream(caller)
        self.d2h.wait_stream(caller)
        dx = self.dev_x[b]
        raw_comp = api._stream(self.comp, None)
        # copy in, chunk by chunk (the buffer is free once the casts of two calls ago ran)
        with torch.cuda.stream(self.h2d):
            self.h2d.wait_event(self.x_free[b])
            for k, (r0, r1) in enumerate(self.chunks):
                dx[r0 * cols:r1 * cols].copy_(x[r0 * cols:r1 * cols], non_blocking=True)
                self.in_ready[k].record(self.h2d)
        with torch.cuda.stream(self.comp):
            # partial amax of each chunk as soon as it has landed
            for k in range(len(self.chunks)):
                self.comp.wait_event(self.in_ready[k])
                self._amax[b][k].call(raw_comp)
            # the previous call's scales must have left before they are rewritten
            self.comp.wait_event(self.scales_out)
            self._reduce.call(raw_comp)
        # cast chunk k, then copy it out; the two streams are fed chunk by chunk so that
        # every event wait refers to the chunk before in this order
        for k, (r0, r1) in enumerate(self.chunks):
            s = k % self.depth
            with torch.cuda.stream(self.comp):
                self.comp.wait_event(self.d2h_done[s])  # staging buffer s has been copied out
                self._cast[b][k].call(raw_comp)
                self.comp_done[s].record(self.comp)
            with torch.cuda.stream(self.d2h):
                self.d2h.wait_event(self.comp_done[s])
                n = (r1 - r0) * cols
                qr[r0 * cols:r1 * cols].copy_(self.dev_qr[s][:n], non_blocking=True)
                if qc is not None:
                    qc[r0 * cols:r1 * cols].copy_(self.dev_qc[s][:n], non_blocking=True)
                self.d2h_done[s].record(self.d2h)
        with torch.cuda.stream(self.comp):
            self.x_free[b].record(self.comp)
        with torch.cuda.stream(self.d2h):
            self.d2h.wait_stream(self.comp)
            host_sr.copy_(self.scale_r, non_blocking=True)
            if host_sc is not None:
                host_sc.copy_(self.scale_c, non_blocking=True)
            self.scales_out.record(self.d2h)
        caller.wait_stream(self.d2h)

    def _direct_casts(self, qr, qc):
        """The casts of both device input buffers into these host outputs, marshalled once
        per pair of output buffers."""
        key = (qr.data_ptr(), None if qc is None else qc.data_ptr())
        if self._direct is None or self._direct[0] != key:
            rows, cols = self.rows, self.cols
            calls = [[api.prepare_partial_cast(self.dev_x[b][r0 * cols:r1 * cols], self.scale_r,
                                               self.scale_c, qr, qc, rows, cols, r0 * cols,
                                               allow_host=True)
                      for r0, r1 in self.chunks] for b in range(2)]
            self._direct = (key, calls)
        return self._direct[1]

    def _run_direct(self, x, qr, qc, host_sr, host_sc, b, caller):
        """run() with direct_out: copy-in and amax as in run(); every chunk's cast writes
        the host outputs itself; only the scale grids go out through a copy."""
        cols = self.cols
        casts = self._direct_casts(qr, qc)
        self.comp.wait_stream(caller)
        self.d2h.wait_stream(caller)
        dx = self.dev_x[b]
        raw_comp = api._stream(self.comp, None)
        with torch.cuda.stream(self.h2d):
            self.h2d.wait_event(self.x_free[b])
            for k, (r0, r1) in enumerate(self.chunks):
                dx[r0 * cols:r1 * cols].copy_(x[r0 * cols:r1 * cols], non_blocking=True)
                self.in_ready[k].record(self.h2d)
        with torch.cuda.stream(self.comp):
            for k in range(len(self.chunks)):
                self.comp.wait_event(self.in_ready[k])
                self._amax[b][k].call(raw_comp)
            self.comp.wait_event(self.scales_out)
            self._reduce.call(raw_comp)
            for c in casts[b]:
                c.call(raw_comp)
            self.x_free[b].record(self.comp)
        with torch.cuda.stream(self.d2h):
            self.d2h.wait_stream(self.comp)
            host_sr.copy_(self.scale_r, non_blocking=True)
            if host_sc is not None:
                host_sc.copy_(self.scale_c, non_blocking=True)
            self.scales_out.record(self.d2h)
        caller.wait_stream(self.d2h)
