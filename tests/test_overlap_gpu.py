"""Launch overlap of the per-bucket kernels (zero_set_launch_overlap).

The per-bucket forms stream buckets one after another: ZeRO-2 reduce-scatter + update as
each bucket's gradients appear ("CS336 2026 Lecture 8" Slides 23 and 26), ZeRO-3 gathers
just before each module with prefetch (Slides 24-26; "CS231n Lecture 11" 4.3). With
programmatic dependent launch a bucket's kernel may start while the previous one finishes.
Whatever the mode, results must equal the oracle's monolithic step bit for bit, and the
gathered parameters must equal the full parameter buffer.

Under "buckets" the caller must not enqueue, directly before a per-bucket call on the same
stream, a kernel that writes what the call reads; the tests below produce gradients the
way a data-parallel trainer does (on the compute stream, handed to the update stream by an
event) or ahead of time. Under "launch" any producer may precede the call.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
import zero_gradient_reduce_scatter_gb300 as zg
from parity_util import REL_NORM, f32, make_hyper, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    yield


def gpt_like(d, layers, vocab=1000):
    sizes = [vocab * d]
    for _ in range(layers):
        sizes += [d, d, 3 * d * d, d * d, d, d, 4 * d * d, 4 * d * d]
    return tuple(sizes + [d, d])


def _bucket_slices(opt, full, b):
    off = opt.buckets[b][0]
    return [g[off:off + opt.bucket_lanes(b)] for g in full]


# producer patterns of the bucket gradients
def _inline(opt, full, order, h, stream):
    """Each bucket's buffers are copied on the update stream right before its call (a
    foreign kernel directly precedes every call: allowed only under "launch")."""
    for b in order:
        with torch.cuda.stream(stream):
            bufs = [x.clone() for x in _bucket_slices(opt, full, b)]
        opt.step_bucket(b, bufs, h, stream=stream)


def _event_handoff(opt, full, order, h, stream):
    """Trainer pattern: buckets produced on the compute stream, each handed to the update
    stream by an event; the update stream holds only event waits and bucket launches."""
    compute = torch.cuda.current_stream()
    keep = []
    for b in order:
        with torch.cuda.stream(compute):
            bufs = [x.clone() for x in _bucket_slices(opt, full, b)]
            torch.cuda._sleep(20_000)  # a slow backward: the update stream must wait for it
            ev = torch.cuda.Event()
            ev.record(compute)
        stream.wait_event(ev)
        opt.step_bucket(b, bufs, h, stream=stream)
        keep.append(bufs)
        for x in bufs:
            x.record_stream(stream)
    return keep


def _ahead(opt, full, order, h, stream):
    """All bucket buffers exist before the first call: the calls run back to back."""
    bufs = {b: [x.clone() for x in _bucket_slices(opt, full, b)] for b in order}
    stream.wait_stream(torch.cuda.current_stream())
    for b in order:
        opt.step_bucket(b, bufs[b], h, stream=stream)
        for x in bufs[b]:
            x.record_stream(stream)
    return bufs


CASES = [
    ("launch", "inline", 2, "fused", 1),
    ("launch", "event", 3, "shards", 1),
    ("buckets", "event", 2, "fused", 1),
    ("buckets", "ahead", 2, "fused", 1),
    ("buckets", "ahead", 3, "shards", 1),
    ("buckets", "event", 1, "fused", 2),
]


@pytest.mark.parametrize("mode,producer,stage,gather,groups", CASES)
def test_overlapped_bucket_steps_match_oracle(mode, producer, stage, gather, groups):
    w = W.small_variant(W.workload("gpt2s"), gpt_like(96, 3), bucket_bytes=120_000, steps=3, stage=stage)
    dev = torch.device("cuda")
    mi = W.master_init(w, dev)
    opt = zg.ZeroOptimizer(w.numel, w.M, w.stage, mi, bucket_bytes=w.bucket_bytes, gather=gather, groups=groups)
    opt.set_launch_overlap(mode)
    nb = len(opt.buckets)
    assert nb >= 5
    p = O.plan(w.numel, w.M // groups, w.bucket_bytes)
    st = O.init_state(p, w.stage, f32(mi), groups=groups)
    h, oh = make_hyper(w)
    sig = W.sigmas(w)
    stream = torch.cuda.Stream(device=dev)
    produce = {"inline": _inline, "event": _event_handoff, "ahead": _ahead}[producer]
    for k in range(w.steps):
        full = opt.new_grad_buffers()
        for r in range(w.M):
            W.fill_grads(w, r, k, full[r], opt.tensor_offsets, sig)
        torch.cuda.synchronize()
        produce(opt, full, list(reversed(range(nb))), h, stream)
        # a kernel consumer enqueued right after the last bucket sees the finished step
        with torch.cuda.stream(stream):
            seen = opt.params().clone()
        torch.cuda.synchronize()
        assert opt.t == k + 1
        fullp, _, _, rc = O.zero_step(p, st, [u16(g) for g in full], oh)
        assert rc == 0 and opt.sync_status() == 0
        assert np.array_equal(u16(seen), fullp), k
        for name, buf in (("master", opt.master), ("mom", opt.m), ("var", opt.v)):
            assert np.array_equal(f32(buf).view(np.uint32), O.flat_state(p, st, name).view(np.uint32)), (k, name)


@pytest.mark.parametrize("order,buffers", [("forward", 2), ("backward", 2), ("forward", 3), ("backward", 4)])
def test_overlapped_prefetched_gather(order, buffers):
    """ZeRO-3 gathers on a side stream, one bucket ahead, into two transient buffers that a
    slow consumer holds: a gather overlaps the previous gather but never overwrites a buffer
    before the consumer's event says it is free. Three sweeps with a step between each."""
    w = W.small_variant(W.workload("ragged"), W.ragged_numel(60, 100, 8000, 13), bucket_bytes=25000, steps=3)
    dev = torch.device("cuda")
    opt = zg.ZeroOptimizer(w.numel, w.M, w.stage, W.master_init(w, dev), bucket_bytes=w.bucket_bytes,
                           gather="shards")
    opt.set_launch_overlap("buckets")
    h, _ = make_hyper(w)
    nb = len(opt.buckets)
    assert nb > 4
    seq = list(range(nb)) if order == "forward" else list(reversed(range(nb)))
    stream = torch.cuda.current_stream()
    side = torch.cuda.Stream(device=dev)
    for k in range(w.steps):
        grads = opt.new_grad_buffers()
        for r in range(w.M):
            W.fill_grads(w, r, k, grads[r], opt.tensor_offsets)
        opt.step(grads, h)
        check = torch.full((opt.sizes["n"],), -1, dtype=torch.int16, device=dev)
        for b, params in opt.prefetched_buckets(seq, stream=stream, side_stream=side, buffers=buffers):
            torch.cuda._sleep(100_000)  # a slow "module" keeps the buffer busy
            u0, n = opt.bucket_range(b)
            check[u0:u0 + n].copy_(params.view(torch.int16))
        torch.cuda.synchronize()
        assert torch.equal(check, opt.params().view(torch.int16)), k


def test_back_to_back_gathers_into_one_buffer():
    """Gathers into overlapping destinations keep their order: each waits for the one
    before (the library compares destinations), so the later values win."""
    w = W.small_variant(W.workload("ragged"), W.ragged_numel(40, 300, 9000, 21), bucket_bytes=20000, steps=1)
    dev = torch.device("cuda")
    opt = zg.ZeroOptimizer(w.numel, w.M, w.stage, W.master_init(w, dev), bucket_bytes=w.bucket_bytes,
                           gather="shards")
    opt.set_launch_overlap("buckets")
    full = opt.params()
    nb = len(opt.buckets)
    sizes = [opt.bucket_range(b)[1] for b in range(nb)]
    big = max(range(nb), key=lambda b: sizes[b])
    buf = torch.zeros(max(sizes) + 16, dtype=torch.bfloat16, device=dev)
    for b in range(nb):
        if b == big:
            continue
        opt.gather_bucket(big, buf)
        opt.gather_bucket(b, buf[3:])  # overlaps the first gather's destination
        torch.cuda.synchronize()
        ub, nbig = opt.bucket_range(big)
        u0, n = opt.bucket_range(b)
        assert torch.equal(buf[3:3 + n].view(torch.int16), full[u0:u0 + n].view(torch.int16)), b
        assert torch.equal(buf[:3].view(torch.int16), full[ub:ub + 3].view(torch.int16)), b
        if 3 + n < nbig:
            assert torch.equal(buf[3 + n:nbig].view(torch.int16), full[ub + 3 + n:ub + nbig].view(torch.int16)), b


def test_set_launch_overlap_refusals():
    w = W.small_variant(W.workload("gpt2s"), (3000, 3000), bucket_bytes=6000, steps=1)
    opt = zg.ZeroOptimizer(w.numel, w.M, w.stage, W.master_init(w, torch.device("cuda")),
                           bucket_bytes=w.bucket_bytes)
    for bad in (-1, 3):
        assert zg._lib().zero_set_launch_overlap(opt._ctx, bad) == -1
    opt.set_launch_overlap("none")


def _reduce_ahead(opt, full, order, stream):
    bufs = {b: [x.clone() for x in _bucket_slices(opt, full, b)] for b in order}
    stream.wait_stream(torch.cuda.current_stream())
    for b in order:
        opt.reduce_bucket(b, bufs[b], stream=stream)
        for x in bufs[b]:
            x.record_stream(stream)
    return bufs


def _reduce_event(opt, full, order, stream):
    compute = torch.cuda.current_stream()
    keep = []
    for b in order:
        bufs = [x.clone() for x in _bucket_slices(opt, full, b)]
        torch.cuda._sleep(20_000)
        ev = torch.cuda.Event()
        ev.record(compute)
        stream.wait_event(ev)
        opt.reduce_bucket(b, bufs, stream=stream)
        keep.append(bufs)
        for x in bufs:
            x.record_stream(stream)
    return keep


@pytest.mark.parametrize("mode,producer,groups", [("launch", "event", 1), ("buckets", "event", 1),
                                                   ("buckets", "ahead", 1), ("buckets", "ahead", 2)])
def test_overlapped_bucket_reductions_match_ordinary_launches(mode, producer, groups):
    """ZeRO-2 streaming with clipping (every bucket reduced, then one apply): with overlapped
    reductions the averaged gradient, the norm and the whole state equal those of ordinary
    launches bit for bit (same grid, same partial sums), and the oracle's step within the
    parity tolerances (averaged gradient bit-exact)."""
    w = W.small_variant(W.workload("gpt2s"), gpt_like(96, 3), bucket_bytes=120_000, steps=3, clip=1e-3)
    dev = torch.device("cuda")
    mi = W.master_init(w, dev)
    ref = zg.ZeroOptimizer(w.numel, w.M, w.stage, mi, bucket_bytes=w.bucket_bytes, ghat_buffer=True, groups=groups)
    opt = zg.ZeroOptimizer(w.numel, w.M, w.stage, mi, bucket_bytes=w.bucket_bytes, ghat_buffer=True, groups=groups)
    opt.set_launch_overlap(mode)
    nb = len(opt.buckets)
    assert nb >= 5
    p = O.plan(w.numel, w.M // groups, w.bucket_bytes)
    st = O.init_state(p, w.stage, f32(mi), groups=groups)
    h, oh = make_hyper(w)
    sig = W.sigmas(w)
    stream = torch.cuda.Stream(device=dev)
    order = list(reversed(range(nb)))
    for k in range(w.steps):
        full = opt.new_grad_buffers()
        for r in range(w.M):
            W.fill_grads(w, r, k, full[r], opt.tensor_offsets, sig)
        torch.cuda.synchronize()
        for b in order:
            ref.reduce_bucket(b, _bucket_slices(ref, full, b))
        ref.apply(h)
        (_reduce_event if producer == "event" else _reduce_ahead)(opt, full, order, stream)
        opt.apply(h, stream=stream)
        torch.cuda.synchronize()
        assert opt.sync_status() == 0 and ref.sync_status() == 0
        assert opt.last_norm() == ref.last_norm(), k
        for a, b_ in ((opt.ghat, ref.ghat), (opt.master, ref.master), (opt.m, ref.m), (opt.v, ref.v),
                      (opt.params(), ref.params())):
            assert torch.equal(a.view(torch.int16), b_.view(torch.int16)), k
        _, norm, _, rc = O.zero_step(p, st, [u16(g) for g in full], oh)
        assert rc == 0
        assert np.array_equal(f32(opt.ghat).view(np.uint32), O.flat_state(p, st, "ghat").view(np.uint32)), k
        assert abs(opt.last_norm()[0] - norm) <= REL_NORM * norm


def test_bucket_reduced_twice_in_one_step():
    """A bucket reduced a second time in a step (after the next bucket) replaces its first
    reduction; the repeated call waits for what came before, so the second values win."""
    w = W.small_variant(W.workload("gpt2s"), (30000, 20000, 25000), bucket_bytes=60_000, steps=1, clip=1e-3)
    dev = torch.device("cuda")
    mi = W.master_init(w, dev)
    ref = zg.ZeroOptimizer(w.numel, w.M, w.stage, mi, bucket_bytes=w.bucket_bytes, ghat_buffer=True)
    opt = zg.ZeroOptimizer(w.numel, w.M, w.stage, mi, bucket_bytes=w.bucket_bytes, ghat_buffer=True)
    opt.set_launch_overlap("buckets")
    assert len(opt.buckets) == 3
    h, _ = make_hyper(w)
    full = opt.new_grad_buffers()
    for r in range(w.M):
        W.fill_grads(w, r, 0, full[r], opt.tensor_offsets)
    junk = [torch.full_like(x, 3.0) for x in _bucket_slices(opt, full, 1)]
    good = {b: [x.clone() for x in _bucket_slices(opt, full, b)] for b in range(3)}
    torch.cuda.synchronize()
    for b, bufs in ((2, good[2]), (1, junk), (0, good[0]), (1, good[1])):
        opt.reduce_bucket(b, bufs)
    opt.apply(h)
    for b in (2, 1, 0):
        ref.reduce_bucket(b, good[b])
    ref.apply(h)
    torch.cuda.synchronize()
    assert opt.last_norm() == ref.last_norm()
    for a, b_ in ((opt.ghat, ref.ghat), (opt.master, ref.master), (opt.params(), ref.params())):
        assert torch.equal(a.view(torch.int16), b_.view(torch.int16))


@pytest.mark.parametrize("ctas", [1, 7])
def test_overlap_with_tiny_grids(ctas):
    """Grids capped at 1 or 7 CTAs keep many overlapped bucket kernels resident at once, each
    waiting at its end for the one before: fused bucket steps and clipped bucket reductions
    must still equal ordinary launches bit for bit."""
    dev = torch.device("cuda")
    for clip in (None, 1e-3):
        w = W.small_variant(W.workload("gpt2s"), W.ragged_numel(40, 100, 6000, 41), bucket_bytes=20000, steps=2,
                            clip=clip)
        mi = W.master_init(w, dev)
        ref = zg.ZeroOptimizer(w.numel, w.M, w.stage, mi, bucket_bytes=w.bucket_bytes, ghat_buffer=True)
        opt = zg.ZeroOptimizer(w.numel, w.M, w.stage, mi, bucket_bytes=w.bucket_bytes, ghat_buffer=True)
        for o in (ref, opt):
            o.set_max_ctas(ctas)
        opt.set_launch_overlap("buckets")
        nb = len(opt.buckets)
        assert nb >= 8
        h, _ = make_hyper(w)
        stream = torch.cuda.Stream(device=dev)
        for k in range(w.steps):
            full = opt.new_grad_buffers()
            for r in range(w.M):
                W.fill_grads(w, r, k, full[r], opt.tensor_offsets)
            torch.cuda.synchronize()
            order = list(reversed(range(nb)))
            if clip is None:
                for b in order:
                    ref.step_bucket(b, _bucket_slices(ref, full, b), h)
                _ahead(opt, full, order, h, stream)
            else:
                for b in order:
                    ref.reduce_bucket(b, _bucket_slices(ref, full, b))
                ref.apply(h)
                _reduce_ahead(opt, full, order, stream)
                opt.apply(h, stream=stream)
            torch.cuda.synchronize()
            assert opt.sync_status() == 0 and ref.sync_status() == 0
            for a, b_ in ((opt.master, ref.master), (opt.m, ref.m), (opt.v, ref.v), (opt.params(), ref.params())):
                assert torch.equal(a.view(torch.int16), b_.view(torch.int16)), (clip, k)


@pytest.mark.parametrize("clip", [None, 1.0])
def test_full_size_streamed_step_matches_ordinary_launches(clip):
    """The GPT-2-small shaped workload at full size (123,570,432 parameters, M=8, 25 MiB
    buckets), streamed in backward order with overlapped launches as bench.py --mode stream
    times it: two steps bit-identical to the same steps with ordinary launches (the fused
    bucket steps without clipping; bucket reductions + one apply with clipping)."""
    w = W.workload("gpt2s")
    if clip is not None:
        w = W.small_variant(w, w.numel, clip=clip, name=w.name)
    dev = torch.device("cuda")
    mi = W.master_init(w, dev)
    ref = zg.ZeroOptimizer(w.numel, w.M, w.stage, mi, bucket_bytes=w.bucket_bytes, ghat_buffer=clip is not None)
    opt = zg.ZeroOptimizer(w.numel, w.M, w.stage, mi, bucket_bytes=w.bucket_bytes, ghat_buffer=clip is not None)
    opt.set_launch_overlap("buckets")
    nb = len(opt.buckets)
    assert nb == 9
    h, _ = make_hyper(w)
    sig = W.sigmas(w)
    stream = torch.cuda.Stream(device=dev)
    order = list(reversed(range(nb)))
    for k in range(2):
        full = opt.new_grad_buffers()
        for r in range(w.M):
            W.fill_grads(w, r, k, full[r], opt.tensor_offsets, sig)
        torch.cuda.synchronize()
        if clip is None:
            for b in order:
                ref.step_bucket(b, _bucket_slices(ref, full, b), h)
            _ahead(opt, full, order, h, stream)
        else:
            for b in order:
                ref.reduce_bucket(b, _bucket_slices(ref, full, b))
            ref.apply(h)
            _reduce_ahead(opt, full, order, stream)
            opt.apply(h, stream=stream)
        torch.cuda.synchronize()
        assert opt.sync_status() == 0 and ref.sync_status() == 0
        if clip is not None:
            assert opt.last_norm() == ref.last_norm()
        for a, b_ in ((opt.master, ref.master), (opt.m, ref.m), (opt.v, ref.v), (opt.params(), ref.params())):
            assert torch.equal(a.view(torch.int16), b_.view(torch.int16)), (clip, k)
        del full


def test_full_size_prefetched_gather_sweep():
    """The 4B workload at full size (4,092,982,400 parameters, M=4, ZeRO-3 shards, 25 MiB
    buckets: 129 buckets) after one step: the overlapped prefetched sweep, as bench.py
    --mode gather times it, rebuilds every parameter bit for bit."""
    import dataclasses
    w = dataclasses.replace(W.workload("4b"), bucket_bytes=25 * 1024 * 1024)
    dev = torch.device("cuda")
    opt = zg.ZeroOptimizer(w.numel, w.M, 3, W.master_init(w, dev), bucket_bytes=w.bucket_bytes, gather="shards")
    opt.set_launch_overlap("buckets")
    nb = len(opt.buckets)
    assert nb == 129
    h, _ = make_hyper(w)
    grads = opt.new_grad_buffers()
    sig = W.sigmas(w)
    for r in range(w.M):
        W.fill_grads(w, r, 0, grads[r], opt.tensor_offsets, sig)
    opt.step(grads, h)
    del grads
    check = torch.full((opt.sizes["n"],), -1, dtype=torch.int16, device=dev)
    stream = torch.cuda.current_stream()
    side = torch.cuda.Stream(device=dev)
    for b, params in opt.prefetched_buckets(list(range(nb)), stream=stream, side_stream=side):
        u0, n = opt.bucket_range(b)
        check[u0:u0 + n].copy_(params.view(torch.int16))
    torch.cuda.synchronize()
    assert opt.sync_status() == 0
    assert torch.equal(check, opt.params().view(torch.int16))
