"""The README's usage snippets, run as written (its placeholders filled in), each checked
against the plain device path: the whole step and a step captured in a CUDA graph, and ZeRO-2
streaming bucket by bucket with launch overlap."""
import pytest
import torch

import zero_gradient_reduce_scatter_gb300 as zg

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"


def _w0(n, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return torch.randn(n, device="cuda", generator=g) * 0.02


def _fill(opt, grads, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    for buf in grads:
        for i, n in enumerate(opt.numel):
            opt.tensor_view(buf, i).copy_((torch.randn(n, device="cuda", generator=g) * 1e-3).to(torch.bfloat16))


def test_readme_step_and_captured_step():
    w0 = _w0(5096, 1)
    opt = zg.ZeroOptimizer(numel=[4096, 1000], M=8, stage=2, master_init=w0)
    grads = opt.new_grad_buffers()                    # M padded bf16 buffers
    _fill(opt, grads, 2)                              # every rank's gradient of every tensor
    opt.step(grads, zg.Hyper(lr=1e-3, clip=True, max_grad_norm=1.0))
    params = opt.params()                             # bf16, unpadded, tensor order
    assert params.dtype == torch.bfloat16 and params.numel() == 5096

    opt.set_schedule([zg.Hyper(lr=1e-3 * min(1, (k + 1) / 100)) for k in range(1000)])
    g = torch.cuda.CUDAGraph()
    import gc
    gc.collect()  # no CUDA object of an earlier test released inside the capture
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        opt.step_scheduled(grads)
    g.replay()                                        # one step
    torch.cuda.synchronize()
    assert opt.sync_status() == 0

    # the same two steps through the plain device path
    ref = zg.ZeroOptimizer(numel=[4096, 1000], M=8, stage=2, master_init=w0)
    ref.step(grads, zg.Hyper(lr=1e-3, clip=True, max_grad_norm=1.0))
    ref.step(grads, zg.Hyper(lr=1e-3 * min(1, 1 / 100)))
    torch.cuda.synchronize()
    assert torch.equal(opt.params(), ref.params())
    assert torch.equal(opt.master, ref.master) and torch.equal(opt.v, ref.v)
    opt.set_schedule(None)  # leaves scheduled mode: the per-bucket calls need it left
    opt.close()
    ref.close()


def test_readme_bucket_streaming_with_launch_overlap():
    numel = [4096, 1000, 3001, 77, 6000]
    w0 = _w0(sum(numel), 3)
    opt = zg.ZeroOptimizer(numel, 4, 2, w0, bucket_bytes=8192)
    ref = zg.ZeroOptimizer(numel, 4, 2, w0, bucket_bytes=8192)
    assert len(opt.buckets) > 2
    grads = ref.new_grad_buffers()
    _fill(ref, grads, 4)
    # bucket_grads[b]: the M ranks' gradients of bucket b, M * S_b padded lanes each, made on
    # the compute stream (here: copied out of the whole buffers), grads_ready[b] after them
    bucket_grads = [[g[off:off + opt.bucket_lanes(b)].clone() for g in grads]
                    for b, (off, _n, _S, _t) in enumerate(opt.buckets)]
    grads_ready = [torch.cuda.Event() for _ in opt.buckets]
    for e in grads_ready:
        e.record()
    stream = torch.cuda.Stream()

    opt.set_launch_overlap("buckets")      # consecutive bucket calls on one stream may overlap
    for b in reversed(range(len(opt.buckets))):
        stream.wait_event(grads_ready[b])  # gradients made on the compute stream
        opt.step_bucket(b, bucket_grads[b], zg.Hyper(lr=1e-3), stream=stream)
    stream.synchronize()

    ref.step(grads, zg.Hyper(lr=1e-3))
    torch.cuda.synchronize()
    assert opt.t == ref.t == 1
    assert torch.equal(opt.params(), ref.params())
    assert torch.equal(opt.master, ref.master) and torch.equal(opt.m, ref.m) and torch.equal(opt.v, ref.v)
    opt.close()
    ref.close()
