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
