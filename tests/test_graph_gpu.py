"""Steps with device-resident scalars, captured once in a CUDA graph and replayed.

The scalars of AdamW change every step: lr under a schedule, and the bias corrections of
step t (Loshchilov & Hutter's decoupled weight decay with Kingma & Ba's bias correction).
A captured launch keeps its arguments. So zero_set_schedule uploads the scalars of the
coming steps, and zero_step_scheduled reads them on the device. Each replay of one
captured step must equal zero_step with that step's hyper-parameters, bit for bit (a twin
optimizer runs alongside), and the oracle within the parity tolerances. A replay past the
schedule must change no state and raise ZERO_ERR_SCHEDULE. A new schedule continues from
the last step that ran.
"""
import gc
import math

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
import zero_gradient_reduce_scatter_gb300 as zg
from parity_util import REL_NORM, bf16_ulp_diff, f32, make_hyper, state_errors, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    yield


def schedule(w, steps, first, ghat_mode="auto"):
    """Per-step hyper-parameters: linear lr warm-up and a drifting clip threshold."""
    clip = w.clip is not None
    out = []
    for i in range(steps):
        k = first + i
        lr = w.lr * min(1.0, (k + 1) / 4.0)
        mx = (w.clip * (1.0 + 0.25 * k)) if clip else 1.0
        out.append((zg.Hyper(lr=lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, weight_decay=w.weight_decay,
                             clip=clip, max_grad_norm=mx, ghat_mode=ghat_mode),
                    O.hyper(lr=lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, weight_decay=w.weight_decay, clip=clip,
                            max_grad_norm=mx)))
    return out


def state_of(opt):
    return [t.clone() for t in (opt.master, opt.m, opt.v, opt.params())]


def check_against(opt, twin, p, st, full, norm, clip, exact_twin=True):
    if exact_twin:
        for a, b, name in zip(state_of(opt), state_of(twin), ("master", "m", "v", "params")):
            assert torch.equal(a.view(torch.int32) if a.dtype == torch.float32 else a.view(torch.int16),
                               b.view(torch.int32) if b.dtype == torch.float32 else b.view(torch.int16)), name
    assert bf16_ulp_diff(u16(opt.params()), full) <= 1
    for name, buf in (("master", opt.master), ("mom", opt.m), ("var", opt.v)):
        assert state_errors(f32(buf), O.flat_state(p, st, name)) <= 1.0, name
    if clip and math.isfinite(norm):
        gn, _ = opt.last_norm()
        assert abs(gn - norm) <= REL_NORM * norm


CASES = {
    # plain fused kernel (no clip), ZeRO-2, several buckets
    "fused-noclip-M8": (lambda: W.small_variant(W.workload("gpt2s"), W.ragged_numel(30, 100, 9000, 5), bucket_bytes=40000),
                        dict(), 1),
    # clip, M = 4: norm pass + scaled fused kernel; ZeRO-3 with the separate all-gather
    "recompute-M4-shards": (lambda: W.small_variant(W.workload("4b"), W.ragged_numel(25, 200, 12000, 9), clip=0.02),
                            dict(gather="shards"), 1),
    # clip, M = 16: norm pass writing the average + AdamW from it
    "materialize-M16": (lambda: W.small_variant(W.workload("ragged"), W.ragged_numel(25, 200, 8000, 15), clip=0.02),
                        dict(ghat_buffer=True), 1),
    # hybrid sharding, 2 groups of 4
    "hybrid-2x4": (lambda: W.small_variant(W.workload("ragged"), W.ragged_numel(20, 300, 7000, 19), M=8, clip=0.02),
                   dict(), 2),
}


@pytest.mark.parametrize("case", list(CASES))
def test_captured_step_replays_match_zero_step_and_oracle(case):
    make, kw, groups = CASES[case]
    w = make()
    dev = torch.device("cuda")
    mi = W.master_init(w, dev)
    opt = zg.ZeroOptimizer(w.numel, w.M, w.stage, mi, bucket_bytes=w.bucket_bytes, groups=groups, **kw)
    twin = zg.ZeroOptimizer(w.numel, w.M, w.stage, mi, bucket_bytes=w.bucket_bytes, groups=groups, **kw)
    p = O.plan(w.numel, w.M // groups, w.bucket_bytes)
    st = O.init_state(p, w.stage, f32(mi), groups=groups)
    sig = W.sigmas(w)
    clip = w.clip is not None
    grads = opt.new_grad_buffers()

    def fill(k):
        for r in range(w.M):
            W.fill_grads(w, r, k, grads[r], opt.tensor_offsets, sig)

    first = schedule(w, 4, 0)
    opt.set_schedule([h for h, _ in first])
    graph = torch.cuda.CUDAGraph()
    gc.collect()  # collect garbage (CUDA objects) now, not inside the global-mode capture
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        opt.step_scheduled(grads)
    assert opt.t == 0  # capturing ran nothing

    def run(k, h, oh):
        fill(k)
        graph.replay()
        twin.step(grads, h)
        full, norm, _, rc = O.zero_step(p, st, [u16(g) for g in grads], oh)
        assert rc == 0 and opt.sync_status() == 0
        check_against(opt, twin, p, st, full, norm, clip)

    clipped = 0
    for k, (h, oh) in enumerate(first):
        run(k, h, oh)
        assert opt.t == k + 1
        if clip:
            clipped += opt.last_norm()[1] < 1.0
    assert clipped or not clip  # the scaled path really clipped
    # a fifth replay has no entry: nothing changes, the flag is raised and stays
    before = state_of(opt)
    fill(4)
    graph.replay()
    assert opt.sync_status() == zg.ZERO_ERR_SCHEDULE
    assert all(torch.equal(a, b) for a, b in zip(before, state_of(opt)))
    assert opt.t == 4
    with pytest.raises(zg.ZeroError) as e:  # host-scalar steps are refused in scheduled mode
        opt.step(grads, first[0][0])
    assert e.value.code == zg.ZERO_ERR_SCHEDULE
    # a new schedule continues at step 5 with the same captured graph
    second = schedule(w, 2, 4)
    opt.set_schedule([h for h, _ in second])
    for i, (h, oh) in enumerate(second):
        run(4 + i, h, oh)
    assert opt.t == 6
    # leaving scheduled mode hands the count back to the host-scalar path
    opt.set_schedule(None)
    assert opt.t == 6
    h, oh = schedule(w, 1, 6)[0]
    fill(6)
    opt.step(grads, h)
    twin.step(grads, h)
    full, norm, _, rc = O.zero_step(p, st, [u16(g) for g in grads], oh)
    check_against(opt, twin, p, st, full, norm, clip)
    assert opt.t == twin.t == 7


def test_scheduled_calls_without_schedule_are_refused():
    w = W.small_variant(W.workload("tiny"), (5000,))
    opt = zg.ZeroOptimizer(w.numel, w.M, w.stage, W.master_init(w, torch.device("cuda")))
    grads = opt.new_grad_buffers()
    with pytest.raises(zg.ZeroError) as e:
        opt.step_scheduled(grads)
    assert e.value.code == zg.ZERO_ERR_SCHEDULE
    h = zg.Hyper(lr=w.lr)
    with pytest.raises(zg.ZeroError):  # unequal clip flags across entries
        opt.set_schedule([h, zg.Hyper(lr=w.lr, clip=True, max_grad_norm=1.0)])
    with pytest.raises(zg.ZeroError):  # a bad entry
        opt.set_schedule([h, zg.Hyper(lr=-1.0)])
    with pytest.raises(zg.ZeroError) as e:  # the schedule lives in a fixed part of the scratch buffer
        opt.set_schedule([h] * (zg.ZERO_MAX_SCHEDULE + 1))
    assert e.value.code == -9
    opt.set_schedule([h] * zg.ZERO_MAX_SCHEDULE)
    with pytest.raises(zg.ZeroError) as e:
        opt.t = 3
    assert e.value.code == zg.ZERO_ERR_SCHEDULE


@pytest.mark.parametrize("overlap", ["none", "buckets"])
def test_captured_streaming_step_matches_oracle(overlap):
    """ZeRO-2: every bucket's reduce-scatter and the scheduled apply in one graph (with
    launch overlap, the bucket reductions are captured with programmatic dependencies)."""
    w = W.small_variant(W.workload("gpt2s"), W.ragged_numel(40, 100, 6000, 27), bucket_bytes=30000, clip=1e-3)
    dev = torch.device("cuda")
    mi = W.master_init(w, dev)
    opt = zg.ZeroOptimizer(w.numel, w.M, w.stage, mi, bucket_bytes=w.bucket_bytes, ghat_buffer=True)
    opt.set_launch_overlap(overlap)
    nb = len(opt.buckets)
    assert nb >= 4
    p = O.plan(w.numel, w.M, w.bucket_bytes)
    st = O.init_state(p, w.stage, f32(mi))
    sig = W.sigmas(w)
    grads = opt.new_grad_buffers()
    slices = [[g[opt.buckets[b][0]:opt.buckets[b][0] + opt.bucket_lanes(b)] for g in grads] for b in range(nb)]
    sched = schedule(w, 3, 0)
    opt.set_schedule([h for h, _ in sched])
    graph = torch.cuda.CUDAGraph()
    gc.collect()  # collect garbage (CUDA objects) now, not inside the global-mode capture
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        for b in reversed(range(nb)):
            opt.reduce_bucket(b, slices[b])
        opt.apply_scheduled()
    for k, (h, oh) in enumerate(sched):
        for r in range(w.M):
            W.fill_grads(w, r, k, grads[r], opt.tensor_offsets, sig)
        graph.replay()
        full, norm, _, rc = O.zero_step(p, st, [u16(g) for g in grads], oh)
        assert rc == 0 and opt.sync_status() == 0
        assert np.array_equal(f32(opt.ghat).view(np.uint32), O.flat_state(p, st, "ghat").view(np.uint32))
        check_against(opt, opt, p, st, full, norm, True, exact_twin=False)
    assert opt.t == 3


@pytest.mark.parametrize("gather", ["fused", "shards"])
def test_captured_fused_bucket_steps_match_oracle(gather):
    """ZeRO-2 without clipping: every bucket's fused reduce-scatter + update in one graph,
    replayed under an lr schedule; bit-identical to the oracle's monolithic step."""
    w = W.small_variant(W.workload("gpt2s"), W.ragged_numel(40, 100, 6000, 31), bucket_bytes=30000, stage=3)
    dev = torch.device("cuda")
    mi = W.master_init(w, dev)
    opt = zg.ZeroOptimizer(w.numel, w.M, w.stage, mi, bucket_bytes=w.bucket_bytes, gather=gather)
    nb = len(opt.buckets)
    assert nb >= 4
    p = O.plan(w.numel, w.M, w.bucket_bytes)
    st = O.init_state(p, w.stage, f32(mi))
    sig = W.sigmas(w)
    grads = opt.new_grad_buffers()
    slices = [[g[opt.buckets[b][0]:opt.buckets[b][0] + opt.bucket_lanes(b)] for g in grads] for b in range(nb)]
    sched = schedule(w, 3, 0)
    opt.set_schedule([h for h, _ in sched])
    graph = torch.cuda.CUDAGraph()
    gc.collect()  # collect garbage (CUDA objects) now, not inside the global-mode capture
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        for b in reversed(range(nb)):
            opt.step_bucket_scheduled(b, slices[b])
    for k, (h, oh) in enumerate(sched):
        for r in range(w.M):
            W.fill_grads(w, r, k, grads[r], opt.tensor_offsets, sig)
        graph.replay()
        full, _, _, rc = O.zero_step(p, st, [u16(g) for g in grads], oh)
        assert rc == 0 and opt.sync_status() == 0 and opt.t == k + 1
        assert np.array_equal(u16(opt.params()), full)
        for name, buf in (("master", opt.master), ("mom", opt.m), ("var", opt.v)):
            assert np.array_equal(f32(buf).view(np.uint32), O.flat_state(p, st, name).view(np.uint32)), name


@pytest.mark.parametrize("overlap", ["none", "buckets"])
def test_captured_prefetched_gather_sweep(overlap):
    """ZeRO-3: one prefetched per-bucket gather sweep (side stream, two transient buffers,
    the consumer copying each bucket out) captured in a CUDA graph; after every step a
    replay rebuilds the parameters of that step bit for bit."""
    w = W.small_variant(W.workload("ragged"), W.ragged_numel(40, 200, 9000, 43), bucket_bytes=20000, steps=3)
    dev = torch.device("cuda")
    opt = zg.ZeroOptimizer(w.numel, w.M, w.stage, W.master_init(w, dev), bucket_bytes=w.bucket_bytes,
                           gather="shards")
    opt.set_launch_overlap(overlap)
    nb = len(opt.buckets)
    assert nb > 6
    h, _ = make_hyper(w)
    check = torch.full((opt.sizes["n"],), -1, dtype=torch.int16, device=dev)
    side = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    gc.collect()  # collect garbage (CUDA objects) now, not inside the global-mode capture
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        for b, params in opt.prefetched_buckets(list(range(nb)), stream=torch.cuda.current_stream(), side_stream=side):
            u0, n = opt.bucket_range(b)
            check[u0:u0 + n].copy_(params.view(torch.int16))
    for k in range(w.steps):
        grads = opt.new_grad_buffers()
        for r in range(w.M):
            W.fill_grads(w, r, k, grads[r], opt.tensor_offsets)
        opt.step(grads, h)
        check.fill_(-1)
        graph.replay()
        torch.cuda.synchronize()
        assert opt.sync_status() == 0
        assert torch.equal(check, opt.params().view(torch.int16)), k
