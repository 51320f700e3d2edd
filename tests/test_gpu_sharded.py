"""Multi-fragment driver on one GPU: a mixed row-only / bidirectional batch split into
emulated master shards (one boundary inside a 32-value block, one empty shard),
one packed on-device MAX reduction, casts in place.  Parity: the union of the
shards' casts is bit-identical to the oracle's whole-weight cast, and the reduced
packed amax equals the oracle's whole-weight amax, packed."""
import numpy as np
import pytest
import torch

import oracle
from mxfp8_master_weight_gb300 import driver
from mxfp8_master_weight_gb300 import workloads as wl

from flows import assert_bitwise, to_device, to_host

pytestmark = pytest.mark.gpu


def _run(batch, dtype=torch.float32):
    specs = [driver.WeightSpec(w.rows, w.cols, w.colwise) for w in batch.weights]
    sc = driver.ShardedCast(specs, batch.bounds, "cuda", dtype)
    shards = [to_device(np.ascontiguousarray(batch.shard(s))) for s in range(sc.num_shards)]
    return sc, shards


def _check_against_full(batch, sc):
    torch.cuda.synchronize()
    red = to_host(sc.reduced)
    for w, wt in enumerate(batch.weights):
        want = oracle.full_cast(wt.data, wt.rows, wt.cols, wt.colwise)
        vr, vc = sc.layout.views(torch.from_numpy(red), w)
        sr, scl = sc.scales[w]
        qr, qc = sc.outputs[w]
        got = (vr.numpy(), None if vc is None else vc.numpy(), to_host(sr),
               None if scl is None else to_host(scl), to_host(qr), None if qc is None else to_host(qc))
        assert_bitwise(got, want, f"weight {w} ({wt.rows}x{wt.cols} colwise={wt.colwise})")


@pytest.mark.parametrize("scale", [8, 1])
def test_cfg5_sharded_mixed_batch(scale):
    batch = wl.cfg5_sharded_batch(seed=0, scale=scale)
    assert batch.bounds[1] % 32 != 0 and batch.bounds[2] == batch.bounds[3]
    sc, shards = _run(batch)
    sc.step(shards)
    _check_against_full(batch, sc)
    amax_calls, reduce_calls, scale_calls, cast_calls = sc._prepared(shards)
    assert len(reduce_calls) == 1 and not scale_calls  # exactly one packed reduction per step
    assert len(amax_calls) == 1 and len(cast_calls) == 1  # one batched call per phase


def test_consecutive_updates_keep_pointers_and_match():
    batch = wl.cfg5_sharded_batch(seed=1, scale=16)
    sc, shards = _run(batch)
    ptrs = [(q[0].data_ptr(), None if q[1] is None else q[1].data_ptr()) for q in sc.outputs]
    sc.step(shards)
    _check_against_full(batch, sc)
    # second update of the same state: new master values, same shard layout and buffers
    rng = np.random.default_rng(99)
    flat2 = wl.normal_f32(rng, batch.total) * np.float32(3.0)
    weights2 = [wl.Weight(w.rows, w.cols, w.dtype, flat2[o:o + w.numel], w.colwise)
                for w, o in zip(batch.weights, batch.offsets)]
    batch2 = wl.ShardedBatch(weights2, batch.offsets, batch.bounds, flat2)
    for s in range(sc.num_shards):
        shards[s].copy_(torch.from_numpy(np.ascontiguousarray(batch2.shard(s))))
    sc.step(shards)
    _check_against_full(batch2, sc)
    assert ptrs == [(q[0].data_ptr(), None if q[1] is None else q[1].data_ptr()) for q in sc.outputs]


@pytest.mark.parametrize("cuts", [[0, 17, 17 + 4096 * 4096 // 4, 4096 * 4096],
                                  [0, 4096 * 4096]])
def test_cfg3_union_of_fragments(cuts):
    w = wl.cfg3_square()
    batch = wl.ShardedBatch([wl.Weight(w.rows, w.cols, wl.F32, w.data, True)], [0], cuts, w.data)
    sc, shards = _run(batch)
    sc.step(shards)
    _check_against_full(batch, sc)


def test_bf16_batch_with_empty_and_single_element_shards():
    rng = np.random.default_rng(5)
    dims = [(64, 96, True), (33, 65, False), (40, 256, True)]
    weights, offs, off = [], [], 0
    for r, c, cw in dims:
        weights.append(wl.Weight(r, c, wl.BF16, None, cw))
        offs.append(off)
        off += r * c
    flat = wl.truncate_to_bf16_bits(wl.normal_f32(rng, off))
    for wt, o in zip(weights, offs):
        wt.data = flat[o:o + wt.numel]
    bounds = [0, 1, 1, 6144 + 3, 6144 + 4, off - 100, off]
    batch = wl.ShardedBatch(weights, offs, bounds, flat)
    sc, shards = _run(batch, torch.bfloat16)
    sc.step(shards)
    _check_against_full(batch, sc)


@pytest.mark.parametrize("fuse", [False, True])
def test_cfg5_small_both_reduction_paths(fuse):
    batch = wl.cfg5_sharded_batch(seed=3, scale=8)
    specs = [driver.WeightSpec(w.rows, w.cols, w.colwise) for w in batch.weights]
    sc = driver.ShardedCast(specs, batch.bounds, "cuda", fuse_reduce_scales=fuse)
    shards = [to_device(np.ascontiguousarray(batch.shard(s))) for s in range(sc.num_shards)]
    sc.step(shards)
    _check_against_full(batch, sc)


def test_fused_reduce_scales_entry_with_padded_views():
    from mxfp8_master_weight_gb300 import _capi, api
    rng = np.random.default_rng(7)
    S, rows, cols = 3, 96, 200
    (rr, rc), (cr, cc) = api.block_shapes(rows, cols)
    # packed buffer with padded leading dimensions: rowwise [96][9], colwise [3][203]
    P = rr * 9 + 64 + cr * 203
    slots_h = np.abs(wl.normal_f32(rng, (S, P)))
    slots = torch.from_numpy(slots_h).cuda()
    reduced = torch.zeros(P, device="cuda")
    vr = reduced[:rr * 9].view(rr, 9)
    vc = reduced[rr * 9 + 64:].view(cr, 203)
    sr = torch.zeros((rr, rc), dtype=torch.uint8, device="cuda")
    sc = torch.zeros((cr, cc), dtype=torch.uint8, device="cuda")
    api.mxfp8_amax_max_reduce_update_scales(slots, reduced, [(vr, vc, sr, sc, rows, cols)])
    torch.cuda.synchronize()
    want = oracle.max_reduce(slots_h)
    got = to_host(reduced)
    wr = want[:rr * 9].reshape(rr, 9)[:, :rc]
    wc = want[rr * 9 + 64:].reshape(cr, 203)[:, :cc]
    assert np.array_equal(got[:rr * 9].reshape(rr, 9)[:, :rc], wr)
    assert np.array_equal(got[rr * 9 + 64:].reshape(cr, 203)[:, :cc], wc)
    assert np.all(got[rr * 9:rr * 9 + 64] == 0)  # entries outside every view untouched
    assert np.array_equal(to_host(sr), oracle.e8m0_from_amax(wr.astype(np.float64)))
    assert np.array_equal(to_host(sc), oracle.e8m0_from_amax(wc.astype(np.float64)))
    outside = torch.zeros((rr, rc), device="cuda")  # not a view into `reduced`
    with pytest.raises(_capi.MXFP8Error) as e:
        api.mxfp8_amax_max_reduce_update_scales(slots, reduced, [(outside, None, sr, None, rows, cols)])
    assert e.value.status == 1


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_ranged_reduction_never_reads_untouched_slot_entries(dtype):
    """The driver's slots are never zeroed: the ranged reduction reads a slot only where
    its shard's amax wrote.  Slots pre-filled with garbage (NaN, huge values) that the
    amax leaves in place must not reach the reduced amax, the scales or the data --
    over two consecutive steps."""
    batch = wl.cfg5_sharded_batch(seed=4, scale=8)
    if dtype == torch.bfloat16:
        flat = wl.truncate_to_bf16_bits(batch.flat)
        weights = [wl.Weight(w.rows, w.cols, wl.BF16, flat[o:o + w.numel], w.colwise)
                   for w, o in zip(batch.weights, batch.offsets)]
        batch = wl.ShardedBatch(weights, batch.offsets, batch.bounds, flat)
    sc, shards = _run(batch, dtype)
    assert sc.ranged and not any(sc._zero_slot)
    for fill in (float("nan"), 3.0e38 if dtype == torch.float32 else 1.0e38):
        sc.slots.fill_(fill)
        sc.reduced.fill_(-1.0)
        sc.step(shards)
        _check_against_full(batch, sc)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("padded", [True, False])
def test_ranged_entry_matches_whole_slot_reduction(dtype, padded):
    """Random slot ranges (ends anywhere, so runs of dense grids have ragged ends around
    their 4-entry vector middle) over a packed buffer with padded or dense views: the
    ranged reduction equals the whole-slot reduction of slots zeroed outside their ranges
    (entries no slot holds reduce to +0), both bit for bit against the oracle."""
    from mxfp8_master_weight_gb300 import api
    rng = np.random.default_rng(11 + padded)
    S, rows, cols = 5, 96, 200
    (rr, rc), (cr, cc) = api.block_shapes(rows, cols)
    ldr, ldc = (9, 203) if padded else (rc, cc)
    P = rr * ldr + 64 + cr * ldc
    garbage = np.abs(wl.normal_f32(rng, (S, P))) * np.float32(1e3)
    ranges = []
    for s in range(S):
        for _ in range(3):
            a = int(rng.integers(0, P))
            b = int(min(P, a + rng.integers(0, P // 3)))
            ranges.append((s, a, b))
    ranges.append((2, 0, 8))  # touching ranges of one slot
    ranges.append((2, 8, 40))
    held = np.zeros((S, P), bool)
    for s, a, b in ranges:
        held[s, a:b] = True
    zeroed = np.where(held, garbage, np.float32(0.0)).astype(np.float32)
    if dtype == torch.bfloat16:
        garbage, zeroed = wl.truncate_to_bf16_bits(garbage), wl.truncate_to_bf16_bits(zeroed)
    want = oracle.max_reduce(zeroed)
    slots = to_device(garbage).view(S, P)
    reduced = torch.full((P,), 7.0, dtype=dtype, device="cuda")
    vr = reduced[:rr * ldr].view(rr, ldr)
    vc = reduced[rr * ldr + 64:].view(cr, ldc)
    sr = torch.zeros((rr, rc), dtype=torch.uint8, device="cuda")
    scl = torch.zeros((cr, cc), dtype=torch.uint8, device="cuda")
    api.mxfp8_amax_max_reduce_update_scales_ranged(slots, reduced, [(vr, vc, sr, scl, rows, cols)], ranges)
    torch.cuda.synchronize()
    got = to_host(reduced)
    wf = want if dtype == torch.float32 else wl.bf16_bits_to_f32(want)
    for o, ld, nr, nc, st in ((0, ldr, rr, rc, sr), (rr * ldr + 64, ldc, cr, cc, scl)):
        g = got[o:o + nr * ld].reshape(nr, ld)[:, :nc]
        w_ = want[o:o + nr * ld].reshape(nr, ld)[:, :nc]
        assert np.array_equal(g.view(np.uint16 if dtype == torch.bfloat16 else np.uint32),
                              w_.view(np.uint16 if dtype == torch.bfloat16 else np.uint32))
        wf_ = wf[o:o + nr * ld].reshape(nr, ld)[:, :nc]
        assert np.array_equal(to_host(st), oracle.e8m0_from_amax(wf_.astype(np.float64)))
    with pytest.raises(Exception):
        api.mxfp8_amax_max_reduce_update_scales_ranged(slots, reduced, [(vr, vc, sr, scl, rows, cols)],
                                                       [(S, 0, 4)])  # no such slot


@pytest.mark.parametrize("ranged", [True, False])
def test_captured_step_replays_on_new_master_values(ranged):
    """A step captured into a CUDA graph, replayed after the shard buffers were refilled in
    place, gives the oracle's casts of the new values (and every replay the same bytes)."""
    batch = wl.cfg5_sharded_batch(seed=3, scale=16)
    specs = [driver.WeightSpec(w.rows, w.cols, w.colwise) for w in batch.weights]
    sc = driver.ShardedCast(specs, batch.bounds, "cuda", ranged=ranged)
    shards = [torch.from_numpy(np.ascontiguousarray(batch.shard(s))).cuda() for s in range(sc.num_shards)]
    graph = sc.capture(shards)
    torch.cuda.synchronize()
    _check_against_full(batch, sc)
    rng = np.random.default_rng(123)
    flat2 = wl.normal_f32(rng, batch.total) * np.float32(0.5)
    weights2 = [wl.Weight(w.rows, w.cols, w.dtype, flat2[o:o + w.numel], w.colwise)
                for w, o in zip(batch.weights, batch.offsets)]
    batch2 = wl.ShardedBatch(weights2, batch.offsets, batch.bounds, flat2)
    for s in range(sc.num_shards):
        shards[s].copy_(torch.from_numpy(np.ascontiguousarray(batch2.shard(s))))
    graph.replay()
    torch.cuda.synchronize()
    _check_against_full(batch2, sc)
    first = [q[0].clone() for q in sc.outputs]
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    assert all(torch.equal(a, q[0]) for a, q in zip(first, sc.outputs))
