"""Per-bucket forms of the step.

ZeRO-2 streaming ("CS336 2026 Lecture 8" Slide 23; "并行训练优化、MoE扩展与系统瓶颈" 2.2.4):
each bucket is reduce-scattered as soon as its gradients exist (here in backward order, from
short-lived per-bucket buffers). With clipping, one zero_apply finishes the step once every
bucket's norm is in. The result must match the oracle's monolithic step: the averaged
gradient bit for bit, the state within the tolerances (bit-identical whenever the clip scale
rounds the same). Without clipping, zero_step_bucket updates each bucket in the same pass,
and the result must match bit for bit.

ZeRO-3 per-module gather with prefetch (Lecture 8 Slides 24-26; "CS231n Lecture 11" 4.3):
buckets gathered just in time into transient buffers, the next one on a side stream.
"""
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


def gpt_like(d, layers, vocab=1000):
    sizes = [vocab * d]
    for _ in range(layers):
        sizes += [d, d, 3 * d * d, d * d, d, d, 4 * d * d, 4 * d * d]
    return tuple(sizes + [d, d])


@pytest.mark.parametrize("clip", [None, 1e-3])
def test_bucket_streaming_matches_monolithic_oracle(clip):
    w = W.small_variant(W.workload("gpt2s"), gpt_like(100, 3), bucket_bytes=150_000, steps=3, clip=clip)
    dev = torch.device("cuda")
    mi = W.master_init(w, dev)
    opt = zg.ZeroOptimizer(w.numel, w.M, w.stage, mi, bucket_bytes=w.bucket_bytes, ghat_buffer=True)
    nb = len(opt.buckets)
    assert nb >= 5
    p = O.plan(w.numel, w.M, w.bucket_bytes)
    st = O.init_state(p, w.stage, f32(mi))
    h, oh = make_hyper(w)
    sig = W.sigmas(w)
    for k in range(w.steps):
        full = opt.new_grad_buffers()
        for r in range(w.M):
            W.fill_grads(w, r, k, full[r], opt.tensor_offsets, sig)
        for b in reversed(range(nb)):  # backward order: last layers' gradients exist first
            off = opt.buckets[b][0]
            bufs = [g[off:off + opt.bucket_lanes(b)].clone() for g in full]
            opt.reduce_bucket(b, bufs)
            del bufs  # the full gradient of this bucket is no longer kept
        opt.apply(h)
        if k == 0:
            with pytest.raises(zg.ZeroError):  # the buckets must be reduced again first
                opt.apply(h)
        fullp, norm, scale, rc = O.zero_step(p, st, [u16(g) for g in full], oh)
        assert opt.sync_status() == 0 and rc == 0
        if clip:
            gn, gs = opt.last_norm()
            assert abs(gn - norm) <= REL_NORM * norm
        assert np.array_equal(f32(opt.ghat).view(np.uint32), O.flat_state(p, st, "ghat").view(np.uint32))
        assert bf16_ulp_diff(u16(opt.params()), fullp) <= 1
        for name, buf in (("master", opt.master), ("mom", opt.m), ("var", opt.v)):
            assert state_errors(f32(buf), O.flat_state(p, st, name)) <= 1.0, name


@pytest.mark.parametrize("stage,gather,groups", [(2, "fused", 1), (3, "shards", 1), (1, "fused", 1),
                                                  (2, "fused", 2)])
def test_fused_bucket_steps_match_monolithic_oracle(stage, gather, groups):
    """Without clipping each bucket is reduce-scattered and updated as soon as its gradients
    exist (backward order, short-lived buffers); the result equals the oracle's monolithic
    step bit for bit."""
    w = W.small_variant(W.workload("gpt2s"), gpt_like(100, 3), bucket_bytes=150_000, steps=3, stage=stage)
    assert w.clip is None
    dev = torch.device("cuda")
    mi = W.master_init(w, dev)
    opt = zg.ZeroOptimizer(w.numel, w.M, w.stage, mi, bucket_bytes=w.bucket_bytes, gather=gather, groups=groups)
    nb = len(opt.buckets)
    assert nb >= 5
    p = O.plan(w.numel, w.M // groups, w.bucket_bytes)
    st = O.init_state(p, w.stage, f32(mi), groups=groups)
    h, oh = make_hyper(w)
    sig = W.sigmas(w)
    for k in range(w.steps):
        full = opt.new_grad_buffers()
        for r in range(w.M):
            W.fill_grads(w, r, k, full[r], opt.tensor_offsets, sig)
        for i, b in enumerate(reversed(range(nb))):
            off = opt.buckets[b][0]
            bufs = [g[off:off + opt.bucket_lanes(b)].clone() for g in full]
            opt.step_bucket(b, bufs, h)
            del bufs  # freed as soon as the bucket is done
            assert opt.t == (k + 1 if i == nb - 1 else k)
        fullp, _, _, rc = O.zero_step(p, st, [u16(g) for g in full], oh)
        assert rc == 0 and opt.sync_status() == 0
        assert np.array_equal(u16(opt.params()), fullp)
        for name, buf in (("master", opt.master), ("mom", opt.m), ("var", opt.v)):
            assert np.array_equal(f32(buf).view(np.uint32), O.flat_state(p, st, name).view(np.uint32)), name


def test_fused_bucket_steps_refusals():
    w = W.small_variant(W.workload("gpt2s"), (3000, 3000, 3000), bucket_bytes=6000, steps=1)
    opt = zg.ZeroOptimizer(w.numel, w.M, w.stage, W.master_init(w, torch.device("cuda")),
                           bucket_bytes=w.bucket_bytes, ghat_buffer=True)
    h, _ = make_hyper(w)
    hc = zg.Hyper(lr=w.lr, clip=True, max_grad_norm=1.0)
    assert len(opt.buckets) == 3
    with pytest.raises(zg.ZeroError):  # clipping needs the norm of every bucket first
        opt.step_bucket(0, opt.new_bucket_grad_buffers(0), hc)
    opt.step_bucket(2, opt.new_bucket_grad_buffers(2), h)
    for call in (lambda: opt.step_bucket(2, opt.new_bucket_grad_buffers(2), h),  # twice in one step
                 lambda: opt.reduce_bucket(0, opt.new_bucket_grad_buffers(0)),   # the other form
                 lambda: opt.step(opt.new_grad_buffers(), h)):                   # the whole step
        with pytest.raises(zg.ZeroError) as e:
            call()
        assert e.value.code == -1
    opt.step_bucket(0, opt.new_bucket_grad_buffers(0), h)
    opt.step_bucket(1, opt.new_bucket_grad_buffers(1), h)
    assert opt.t == 1 and opt.sync_status() == 0
    opt.step(opt.new_grad_buffers(), h)  # a whole step again
    assert opt.t == 2


def test_apply_requires_every_bucket():
    w = W.small_variant(W.workload("gpt2s"), (3000, 3000, 3000), bucket_bytes=6000, steps=1)
    opt = zg.ZeroOptimizer(w.numel, w.M, w.stage, W.master_init(w, torch.device("cuda")),
                           bucket_bytes=w.bucket_bytes, ghat_buffer=True)
    h, _ = make_hyper(w)
    assert len(opt.buckets) == 3
    opt.reduce_bucket(0, opt.new_bucket_grad_buffers(0))
    opt.reduce_bucket(2, opt.new_bucket_grad_buffers(2))
    with pytest.raises(zg.ZeroError) as e:
        opt.apply(h)
    assert e.value.code == -1
    opt.reduce_bucket(1, opt.new_bucket_grad_buffers(1))
    opt.apply(h)
    assert opt.sync_status() == 0 and opt.t == 1


@pytest.mark.parametrize("order", ["forward", "backward"])
def test_prefetched_gather_per_bucket(order):
    w = W.small_variant(W.workload("ragged"), W.ragged_numel(60, 100, 8000, 13), bucket_bytes=25000, steps=2)
    dev = torch.device("cuda")
    opt = zg.ZeroOptimizer(w.numel, w.M, w.stage, W.master_init(w, dev), bucket_bytes=w.bucket_bytes,
                           gather="shards")
    h, _ = make_hyper(w)
    for k in range(w.steps):
        grads = opt.new_grad_buffers()
        for r in range(w.M):
            W.fill_grads(w, r, k, grads[r], opt.tensor_offsets)
        opt.step(grads, h)
    nb = len(opt.buckets)
    assert nb > 4
    seq = list(range(nb)) if order == "forward" else list(reversed(range(nb)))
    check = torch.full((opt.sizes["n"],), -1, dtype=torch.int16, device=dev)
    stream = torch.cuda.current_stream()
    for b, params in opt.prefetched_buckets(seq, stream=stream):
        torch.cuda._sleep(200_000)  # a slow "module" keeps the buffer busy
        u0, n = opt.bucket_range(b)
        assert params.numel() == n
        check[u0:u0 + n].copy_(params.view(torch.int16))
    torch.cuda.synchronize()
    assert torch.equal(check, opt.params().view(torch.int16))


def test_gather_bucket_into_unaligned_buffer():
    w = W.small_variant(W.workload("ragged"), W.ragged_numel(20, 300, 5000, 17), bucket_bytes=9000, steps=1)
    dev = torch.device("cuda")
    opt = zg.ZeroOptimizer(w.numel, w.M, w.stage, W.master_init(w, dev), bucket_bytes=w.bucket_bytes,
                           gather="shards")
    full = opt.params()
    for b in range(len(opt.buckets)):
        u0, n = opt.bucket_range(b)
        for shift in (0, 1, 3, 5):
            raw = torch.zeros(n + 8, dtype=torch.bfloat16, device=dev)
            dst = raw[shift:shift + n]
            opt.gather_bucket(b, dst)
            torch.cuda.synchronize()
            assert torch.equal(dst.view(torch.int16), full[u0:u0 + n].view(torch.int16)), (b, shift)
