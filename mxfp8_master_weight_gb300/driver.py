"""Multi-fragment driver: a batch of weights cast from sharded master buffers.

This is the flow of "Support row-only MXFP8 distributed master-weight casts"
(flow diagram and section "Changes"): every rank computes the partial amax of
its fragments for the directions each weight has, the amaxes of the whole batch
are packed into one buffer and MAX-reduced ONCE across ranks, the scales of the
present directions are updated, and every rank casts its fragments in place.

Here the ranks are emulated on one GPU: shard s is its own device buffer (as a
rank's master shard would be) and has its own slot of the packed amax buffer;
the cross-rank MAX all-reduce is one reduction over the slots, fused with the
scale update.  A slot is read only on the entries its shard's amax writes (the
ranged reduction), so slots are never zeroed between steps.
All arithmetic runs in the CUDA library; this module only plans fragments and
packed offsets (host logic) and issues the calls.

Packed layout: weights in batch order; for each weight its rowwise block grid
[rows][ceil(cols/32)], then -- only when it has a columnwise direction -- its
columnwise grid [ceil(rows/32)][cols].  Each grid starts on a multiple of 16
elements (64 bytes for FP32) so that every view keeps 16-byte vector access;
the padding entries between grids belong to no grid and are never reduced.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import api

# NVTX range names of the step phases (the reduction range holds the fused scale update)
_PHASE_NAMES = ("mxfp8.partial_amax", "mxfp8.max_reduce", "mxfp8.update_scales", "mxfp8.partial_cast")

_ALIGN = 16

# fragments the library's batched entry points put into one launch (their job table
# travels in kernel parameter space)
_BATCH_JOBS = 64


@dataclass(frozen=True)
class WeightSpec:
    rows: int
    cols: int
    colwise: bool

    @property
    def numel(self) -> int:
        return self.rows * self.cols


@dataclass(frozen=True)
class FragmentCut:
    """Fragment of weight `weight` = weight elements [start, start+length), found at
    `shard_offset` inside shard `shard`."""
    shard: int
    weight: int
    start: int
    length: int
    shard_offset: int


def plan_fragments(specs, bounds):
    """Cut every weight of the flat batch buffer at the shard boundaries.

    ``bounds`` = [b0=0, b1, ..., bS=total] (non-decreasing; equal neighbours make an
    empty shard).  Returns, per shard, the list of non-empty FragmentCut in weight order.
    """
    if bounds[0] != 0 or any(b > c for b, c in zip(bounds[:-1], bounds[1:])):
        raise ValueError("shard bounds must start at 0 and be non-decreasing")
    total = sum(s.numel for s in specs)
    if bounds[-1] != total:
        raise ValueError(f"last shard bound {bounds[-1]} != batch size {total}")
    plan = []
    for s in range(len(bounds) - 1):
        lo, hi = bounds[s], bounds[s + 1]
        cuts, off = [], 0
        for w, spec in enumerate(specs):
            a, b = max(lo, off), min(hi, off + spec.numel)
            if a < b:
                cuts.append(FragmentCut(s, w, a - off, b - a, a - lo))
            off += spec.numel
        plan.append(cuts)
    return plan


def fragment_block_ranges(spec: WeightSpec, start: int, length: int):
    """Entries of the block grids that the fragment [start, start+length) of a weight
    touches, as ranges of linear grid indices: (rowwise ranges over r*ceil(cols/32)+b,
    columnwise ranges over c*cols+j -- empty for a row-only weight).  These are exactly
    the entries the partial amax of that fragment writes.

    Rowwise: the fragment is contiguous in row-major order, so its 1x32 blocks are one
    run of the rowwise grid.  Columnwise: every 32-row band strictly between the first
    and last band is whole; in an end band the touched columns are the union of the
    fragment's row spans inside the band (which may leave a gap when the band holds
    only two partial rows of the fragment).
    """
    if length <= 0:
        return [], []
    rows, cols = spec.rows, spec.cols
    nbr = (cols + 31) // 32
    end = start + length
    r0, cs = divmod(start, cols)
    r1, ce = divmod(end - 1, cols)
    row = [(r0 * nbr + cs // 32, r1 * nbr + ce // 32 + 1)]
    col = []
    if spec.colwise:
        c0, c1 = r0 // 32, r1 // 32
        for c in range(c0, c1 + 1):
            if c0 < c < c1:
                spans = [(0, cols - 1)]
            else:
                a, b = max(r0, 32 * c), min(r1, 32 * c + 31)
                spans = []
                for i in ((a, b) if b > a else (a,)):  # middle rows of a band are whole
                    spans.append((cs if i == r0 else 0, ce if i == r1 else cols - 1))
                if b - a >= 2:
                    spans = [(0, cols - 1)]
            for lo, hi in sorted(spans):
                lo_e, hi_e = c * cols + lo, c * cols + hi + 1
                if col and col[-1][1] >= lo_e:
                    col[-1] = (col[-1][0], max(col[-1][1], hi_e))
                else:
                    col.append((lo_e, hi_e))
    return row, col


def _merge(ranges):
    out = []
    for lo, hi in sorted(ranges):
        if out and out[-1][1] >= lo:
            out[-1] = (out[-1][0], max(out[-1][1], hi))
        else:
            out.append((lo, hi))
    return out


class PackedLayout:
    """Element offsets of every present block grid inside the packed amax buffer."""

    def __init__(self, specs):
        self.specs = list(specs)
        self.rowwise, self.colwise = [], []
        off = 0
        for spec in self.specs:
            (rr, rc), (cr, cc) = api.block_shapes(spec.rows, spec.cols)
            self.rowwise.append((off, (rr, rc)))
            off = _round_up(off + rr * rc, _ALIGN)
            if spec.colwise:
                self.colwise.append((off, (cr, cc)))
                off = _round_up(off + cr * cc, _ALIGN)
            else:
                self.colwise.append(None)
        self.total = off

    def slot_ranges(self, plan):
        """(slot, begin, end) packed-entry ranges that each slot's fragments write: the
        only entries of a slot the reduction needs to read."""
        out = []
        for s, cuts in enumerate(plan):
            rs = []
            for c in cuts:
                row, col = fragment_block_ranges(self.specs[c.weight], c.start, c.length)
                ro = self.rowwise[c.weight][0]
                rs += [(ro + a, ro + b) for a, b in row]
                if self.colwise[c.weight] is not None:
                    co = self.colwise[c.weight][0]
                    rs += [(co + a, co + b) for a, b in col]
            out += [(s, a, b) for a, b in _merge(rs)]
        return out

    def views(self, buf: torch.Tensor, w: int):
        """(rowwise view, columnwise view or None) of weight w inside a 1-D packed buffer."""
        o, shp = self.rowwise[w]
        vr = buf[o:o + shp[0] * shp[1]].view(shp)
        vc = None
        if self.colwise[w] is not None:
            o, shp = self.colwise[w]
            vc = buf[o:o + shp[0] * shp[1]].view(shp)
        return vr, vc


def _count_launches(amax_jobs, cast_jobs, n_reduce_pieces, specs, fused_reduce=False) -> int:
    """Kernel launches the library issues for one step of these jobs: the batched
    entries launch once per group of at most 64 jobs sharing the input dtype (for the
    cast also the outputs' virtual base on a V-byte boundary or not); row-only and
    bidirectional jobs, and aligned and realigning fragments, share launches."""
    def groups(keys, cap):
        counts = {}
        for k in keys:
            counts[k] = counts.get(k, 0) + 1
        return sum((n + cap - 1) // cap for n in counts.values())

    akeys = [a[0].dtype for a in amax_jobs]
    ckeys = []
    for frag, sr, sc, qr, qc, rows, cols, start in cast_jobs:
        # full-size outputs (output offset = fragment start): the byte of element f is at
        # out + f, so the outputs' virtual base is their own address
        v = 16 // frag.element_size()
        vec = all(q.data_ptr() % v == 0 for q in (qr, qc) if q is not None)
        ckeys.append((frag.dtype, vec))
    n_grids = sum(2 if s.colwise else 1 for s in specs)
    if fused_reduce:  # one launch per 64 pieces of grid entries with one set of slots
        reduce_and_scales = (n_reduce_pieces + 63) // 64
    else:             # the reduction, then one scale launch per 32 grids
        reduce_and_scales = 1 + (n_grids + 31) // 32
    return groups(akeys, _BATCH_JOBS) + reduce_and_scales + groups(ckeys, _BATCH_JOBS)


def reduce_runs(layout: PackedLayout, ranges):
    """Runs the fused reduction splits the block grids into, as (grid offset, first, end)
    in grid entries: each grid is cut at every slot range end inside it, and neighbouring
    pieces read by the same slots are joined (without ranges, one run per grid)."""
    runs = []
    grids = [g for w in range(len(layout.specs)) for g in (layout.rowwise[w], layout.colwise[w])
             if g is not None]
    for off, (nr, nc) in grids:
        span = nr * nc
        if not ranges:
            runs.append((off, 0, span))
            continue
        cuts = sorted({0, span} | {e - off for _, a, b in ranges for e in (a, b) if 0 < e - off < span})
        prev = None
        for lo, hi in zip(cuts[:-1], cuts[1:]):
            mask = frozenset(s for s, a, b in ranges if a - off <= lo and b - off >= hi)
            if mask != prev:
                runs.append((off, lo, hi))
            else:
                runs[-1] = (off, runs[-1][1], hi)
            prev = mask
    return runs


def reduce_pieces(layout: PackedLayout, ranges) -> int:
    """Work pieces the library makes of those runs (the driver's grids are dense and
    aligned): 4 entries per item from the first multiple of 4 to the last, and the ragged
    ends as pieces of single entries."""
    n = 0
    for _, lo, hi in reduce_runs(layout, ranges):
        a, z = (lo + 3) // 4 * 4, hi // 4 * 4
        n += 1 if a >= z else 1 + (lo < a) + (z < hi)
    return n


def _round_up(x: int, a: int) -> int:
    return (x + a - 1) // a * a


class ShardedCast:
    """Device state for casting one batch of weights from S emulated master shards.

    Buffers (allocated once, reused by every step, so output and scale pointers are
    stable across consecutive updates): packed amax slots [S][P], the reduced packed
    amax [P], per-weight E8M0 scales, and per-weight full-size E4M3 outputs (rowwise
    always, columnwise only for bidirectional weights).
    """

    def __init__(self, specs, bounds, device, dtype=torch.float32, fuse_reduce_scales=True,
                 ranged=True):
        self.specs = [s if isinstance(s, WeightSpec) else WeightSpec(*s) for s in specs]
        self.bounds = list(bounds)
        self.plan = plan_fragments(self.specs, self.bounds)
        self.layout = PackedLayout(self.specs)
        self.dtype = dtype
        # the emulated all-reduce and the scale update in one pass over the packed buffer
        # (mxfp8_amax_max_reduce_update_scales) or as two calls
        self.fuse_reduce_scales = fuse_reduce_scales
        S = len(self.bounds) - 1
        self.slots = torch.zeros((S, self.layout.total), dtype=dtype, device=device)
        self.reduced = torch.zeros(self.layout.total, dtype=dtype, device=device)
        # With the ranged reduction (fused path) each slot is read only on the entries its
        # fragments' amax writes every step, so no slot is ever zeroed.  The plain
        # reduction reads whole slots: a slot then needs zeroing before each step unless
        # its shard holds every weight whole (every entry of it is overwritten).
        self.ranged = bool(ranged and fuse_reduce_scales and len(self.bounds) - 1 <= 64)
        self.ranges = self.layout.slot_ranges(self.plan) if self.ranged else None
        self._zero_slot = [not self.ranged and
                           not (len(cuts) == len(self.specs) and
                                all(c.start == 0 and c.length == self.specs[c.weight].numel
                                    for c in cuts))
                           for cuts in self.plan]
        self.scales, self.outputs = [], []
        for spec in self.specs:
            (rr, rc), (cr, cc) = api.block_shapes(spec.rows, spec.cols)
            sr = torch.zeros((rr, rc), dtype=torch.uint8, device=device)
            sc = torch.zeros((cr, cc), dtype=torch.uint8, device=device) if spec.colwise else None
            self.scales.append((sr, sc))
            qr = torch.zeros(spec.numel, dtype=torch.uint8, device=device)
            qc = torch.zeros(spec.numel, dtype=torch.uint8, device=device) if spec.colwise else None
            self.outputs.append((qr, qc))

    @property
    def num_shards(self) -> int:
        return len(self.bounds) - 1

    def launches_per_step(self) -> int:
        """Library kernel launches of one step: the batched amax and cast take one launch
        per dtype group of at most 64 fragments (row-only and bidirectional, aligned and
        realigning fragments share launches), the reduction one, the batched scale
        update (when not fused with the reduction) one per 32 block grids."""
        return self._launches if hasattr(self, "_launches") else -1

    def _check_shards(self, shards) -> None:
        if len(shards) != self.num_shards:
            raise ValueError("one master shard buffer per emulated rank is required")
        for s, shard in enumerate(shards):
            if shard.numel() != self.bounds[s + 1] - self.bounds[s]:
                raise ValueError(f"shard {s} holds {shard.numel()} elements, plan expects "
                                 f"{self.bounds[s + 1] - self.bounds[s]}")

    def _prepared(self, shards):
        """The step's library calls, marshalled once per set of shard buffers."""
        key = tuple((t.data_ptr(), t.numel(), t.dtype) for t in shards)
        if getattr(self, "_cache_key", None) == key:
            return self._cache
        self._check_shards(shards)
        amax_jobs, cast_jobs = [], []
        for s, cuts in enumerate(self.plan):
            for c in cuts:
                spec = self.specs[c.weight]
                frag = shards[s][c.shard_offset:c.shard_offset + c.length]
                vr, vc = self.layout.views(self.slots[s], c.weight)
                amax_jobs.append((frag, vr, vc, spec.rows, spec.cols, c.start))
                sr, sc = self.scales[c.weight]
                qr, qc = self.outputs[c.weight]
                cast_jobs.append((frag, sr, sc, qr, qc, spec.rows, spec.cols, c.start))
        scale_jobs = []
        for w, spec in enumerate(self.specs):
            vr, vc = self.layout.views(self.reduced, w)
            sr, sc = self.scales[w]
            scale_jobs.append((vr, vc, sr, sc, spec.rows, spec.cols))
        # one batched call per phase: every fragment of every shard (each shard writes
        # its own slot, so no two jobs write the same amax entry), one reduction, every
        # weight's scales, every fragment's cast
        self._launches = _count_launches(amax_jobs, cast_jobs, reduce_pieces(self.layout, self.ranges),
                                         self.specs, self.fuse_reduce_scales)
        amax = [api.prepare_partial_amax_batched(amax_jobs)]
        if self.ranged:
            reduce = [api.prepare_amax_max_reduce_update_scales_ranged(self.slots, self.reduced,
                                                                       scale_jobs, self.ranges)]
            scales = []
        elif self.fuse_reduce_scales:
            reduce = [api.prepare_amax_max_reduce_update_scales(self.slots, self.reduced, scale_jobs)]
            scales = []
        else:
            reduce = [api.prepare_amax_max_reduce(self.slots, self.reduced)]
            scales = [api.prepare_update_scales_batched(scale_jobs)]
        casts = [api.prepare_partial_cast_batched(cast_jobs)]
        self._cache_key, self._cache = key, (amax, reduce, scales, casts)
        return self._cache

    def step(self, shards, stream=None, events=None) -> None:
        """One distributed update: partial amax -> one packed MAX reduce -> scales -> casts.

        ``events``: optional five CUDA events recorded on the stream before the amax
        phase and after the amax, reduce, scale and cast phases (for timing; with the
        fused reduction + scale update the scale phase is empty).
        """
        phases = self._prepared(shards)
        with torch.cuda.device(self.slots.device):
            torch_stream = stream if stream is not None else torch.cuda.current_stream()
            raw = api._stream(torch_stream, None)
            # amax entries a fragment does not touch must be zero before the reduction
            with torch.cuda.stream(torch_stream):
                for s in range(self.num_shards):
                    if self._zero_slot[s]:
                        self.slots[s].zero_()
            if events is not None:
                events[0].record(torch_stream)
            for k, calls in enumerate(phases):
                if calls:  # NVTX range per phase, for timeline profilers
                    torch.cuda.nvtx.range_push(_PHASE_NAMES[k])
                    for c in calls:
                        c.call(raw)
                    torch.cuda.nvtx.range_pop()
                if events is not None:
                    events[k + 1].record(torch_stream)

    def capture(self, shards) -> torch.cuda.CUDAGraph:
        """One step for these shard buffers, captured into a CUDA graph.

        ``g.replay()`` then issues the step's launches (the same library calls as
        ``step(shards)``, with their programmatic launch dependencies) from the host in one
        go: for a batch of small weights, whose kernels last a few microseconds, the host's
        per-launch cost otherwise sets the step time.  The graph holds buffer addresses: it
        is valid while ``shards`` and this object's buffers live, and a replay reads what
        the shard buffers hold at that moment.  The step runs once, uncaptured, first.
        """
        dev = self.slots.device
        with torch.cuda.device(dev):
            self._prepared(shards)  # the library calls are marshalled outside the capture
            side = torch.cuda.Stream(dev)
            side.wait_stream(torch.cuda.current_stream(dev))
            self.step(shards, stream=side)
            torch.cuda.current_stream(dev).wait_stream(side)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=side):
                self.step(shards, stream=side)
        return graph
