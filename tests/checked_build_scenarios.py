"""Scenarios run against the bounds-checked library (libzero_gb300_checked.so).

Executed in a child process by tests/test_checked_build_gpu.py: the library path is switched
before the binding loads anything. Every scenario also runs its oracle comparison, and after
each the device must report no failed bounds check. Exits non-zero on the first failure.
"""
import ctypes
import gc
import math
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

from zero_gradient_reduce_scatter_gb300 import _build  # noqa: E402

_build.LIB_PATH = _build.build(checked=True)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import oracle as O  # noqa: E402
import workloads as W  # noqa: E402
import zero_gradient_reduce_scatter_gb300 as zg  # noqa: E402
from parity_util import bf16_ulp_diff, make_hyper, run_elementwise, u16  # noqa: E402


def clean(opt, what):
    assert opt.sync_status() == 0, f"{what}: status {opt.sync_status()}"
    site, idx = opt.check_report()
    assert site == 0, f"{what}: bounds check {site} failed at index {idx}"


def exact(out, what):
    assert out["bf16_ulp"] == 0 and out["state_err"] == 0.0, what
    clean(out["opt"], what)


def main():
    assert zg._lib().zero_checked_build() == 1, "not the checked library"
    dev = torch.device("cuda")

    w = W.small_variant(W.workload("gpt2s"), W.ragged_numel(60, 50, 4000, 11), bucket_bytes=9000, steps=2, clip=1.0)
    for mode in ("materialize", "recompute"):
        exact(run_elementwise(w, ghat_mode=mode, ghat_buffer=True), f"fused misaligned stores ({mode})")

    w = W.small_variant(W.workload("ragged"), W.ragged_numel(40, 100, 6000, 3), bucket_bytes=15000, steps=2)
    out = run_elementwise(w, gather="shards")
    exact(out, "shards + gather")
    opt = out["opt"]
    full = opt.params()
    for b in range(len(opt.buckets)):
        u0, n = opt.bucket_range(b)
        raw = torch.zeros(n + 8, dtype=torch.bfloat16, device=dev)
        opt.gather_bucket(b, raw[3:3 + n])
        torch.cuda.synchronize()
        assert torch.equal(raw[3:3 + n].view(torch.int16), full[u0:u0 + n].view(torch.int16))
    for _b, _p in opt.prefetched_buckets(list(range(len(opt.buckets)))):
        pass
    clean(opt, "per-bucket gathers")

    for M in (1, 3, 64):  # the one-source kernel (its own block size), the generic one
        exact(run_elementwise(W.small_variant(W.workload("ragged"), (3001, 17, 1), M=M, steps=2), gather="shards"),
              f"M={M}")
    exact(run_elementwise(W.small_variant(W.workload("ragged"), (3,), steps=2), gather="shards"), "3 lanes, 16 ranks")

    wg = W.small_variant(W.workload("ragged"), W.ragged_numel(30, 200, 5000, 23), M=8, stage=3, steps=2)
    exact(run_elementwise(wg, gather="shards", groups=2, ghat_mode="materialize", ghat_buffer=True), "hybrid")

    # a scheduled step captured in a CUDA graph, replayed past its schedule
    wq = W.small_variant(W.workload("ragged"), W.ragged_numel(20, 300, 5000, 29), M=8, steps=1, clip=0.02)
    opt = zg.ZeroOptimizer(wq.numel, wq.M, wq.stage, W.master_init(wq, dev), groups=2, gather="shards")
    gq = opt.new_grad_buffers()
    for r in range(wq.M):
        W.fill_grads(wq, r, 0, gq[r], opt.tensor_offsets)
    hq, _ = make_hyper(wq)
    opt.set_schedule([hq, hq])
    graph = torch.cuda.CUDAGraph()
    gc.collect()  # collect garbage (CUDA objects) now, not inside the global-mode capture
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        opt.step_scheduled(gq)
    for _ in range(2):
        graph.replay()
    clean(opt, "scheduled steps")
    graph.replay()
    assert opt.sync_status() == zg.ZERO_ERR_SCHEDULE and opt.check_report()[0] == 0 and opt.t == 2

    # ZeRO-2 streaming against the oracle's monolithic step
    ws = W.small_variant(W.workload("gpt2s"), (70000, 5000, 300, 70000), bucket_bytes=120000, steps=2, clip=1.0)
    opt = zg.ZeroOptimizer(ws.numel, ws.M, ws.stage, W.master_init(ws, dev), bucket_bytes=ws.bucket_bytes,
                           ghat_buffer=True)
    p = O.plan(ws.numel, ws.M, ws.bucket_bytes)
    st = O.init_state(p, ws.stage, W.master_init(ws, dev).cpu().numpy())
    h, oh = make_hyper(ws)
    for k in range(ws.steps):
        g = opt.new_grad_buffers()
        for r in range(ws.M):
            W.fill_grads(ws, r, k, g[r], opt.tensor_offsets)
        for b in reversed(range(len(opt.buckets))):
            off = opt.buckets[b][0]
            opt.reduce_bucket(b, [x[off:off + opt.bucket_lanes(b)].clone() for x in g])
        opt.apply(h)
        fullp, _, _, _ = O.zero_step(p, st, [u16(x) for x in g], oh)
        assert bf16_ulp_diff(u16(opt.params()), fullp) <= 1, "streaming"
    clean(opt, "streaming")
    # the same with overlapped bucket reductions (per-bucket partial regions)
    opt.set_launch_overlap("buckets")
    for k in range(ws.steps, ws.steps + 2):
        g = opt.new_grad_buffers()
        for r in range(ws.M):
            W.fill_grads(ws, r, k, g[r], opt.tensor_offsets)
        bufs = {b: [x[opt.buckets[b][0]:opt.buckets[b][0] + opt.bucket_lanes(b)].clone() for x in g]
                for b in range(len(opt.buckets))}
        for b in reversed(range(len(opt.buckets))):
            opt.reduce_bucket(b, bufs[b])
        opt.apply(h)
        fullp, _, _, _ = O.zero_step(p, st, [u16(x) for x in g], oh)
        assert bf16_ulp_diff(u16(opt.params()), fullp) <= 1, "overlapped streaming"
    clean(opt, "overlapped streaming")
    opt.set_launch_overlap("none")

    # ZeRO-2 fused per-bucket steps (no clipping), ZeRO-3 shards with the per-bucket gather
    wf = W.small_variant(W.workload("gpt2s"), (70000, 5000, 301, 69999), bucket_bytes=120000, steps=2, stage=3)
    optf = zg.ZeroOptimizer(wf.numel, wf.M, wf.stage, W.master_init(wf, dev), bucket_bytes=wf.bucket_bytes,
                            gather="shards")
    pf = O.plan(wf.numel, wf.M, wf.bucket_bytes)
    stf = O.init_state(pf, wf.stage, W.master_init(wf, dev).cpu().numpy())
    hf, ohf = make_hyper(wf)
    for k in range(wf.steps):
        g = optf.new_grad_buffers()
        for r in range(wf.M):
            W.fill_grads(wf, r, k, g[r], optf.tensor_offsets)
        for b in reversed(range(len(optf.buckets))):
            off = optf.buckets[b][0]
            optf.step_bucket(b, [x[off:off + optf.bucket_lanes(b)].clone() for x in g], hf)
        fullp, _, _, _ = O.zero_step(pf, stf, [u16(x) for x in g], ohf)
        assert np.array_equal(u16(optf.params()), fullp), "fused per-bucket steps"
    clean(optf, "fused per-bucket steps")

    # the same with overlapped per-bucket launches: fused bucket steps back to back, then
    # per-bucket gathers back to back into disjoint buffers
    optf.set_launch_overlap("buckets")
    side = torch.cuda.Stream(device=dev)
    for k in range(wf.steps, wf.steps + 2):
        g = optf.new_grad_buffers()
        for r in range(wf.M):
            W.fill_grads(wf, r, k, g[r], optf.tensor_offsets)
        bufs = {b: [x[optf.buckets[b][0]:optf.buckets[b][0] + optf.bucket_lanes(b)].clone() for x in g]
                for b in range(len(optf.buckets))}
        side.wait_stream(torch.cuda.current_stream())
        for b in reversed(range(len(optf.buckets))):
            optf.step_bucket(b, bufs[b], hf, stream=side)
        torch.cuda.synchronize()
        fullp, _, _, _ = O.zero_step(pf, stf, [u16(x) for x in g], ohf)
        assert np.array_equal(u16(optf.params()), fullp), "overlapped per-bucket steps"
    outs = [torch.empty(optf.bucket_range(b)[1] + 1, dtype=torch.bfloat16, device=dev)[1:]
            for b in range(len(optf.buckets))]
    for b in range(len(optf.buckets)):
        optf.gather_bucket(b, outs[b], stream=side)
    torch.cuda.synchronize()
    fullv = optf.params()
    for b in range(len(optf.buckets)):
        u0, n = optf.bucket_range(b)
        assert torch.equal(outs[b].view(torch.int16), fullv[u0:u0 + n].view(torch.int16)), "overlapped gathers"
    clean(optf, "overlapped per-bucket launches")

    # save / reshard / load
    saved = opt.save_state()
    w2 = W.small_variant(ws, ws.numel, M=5, stage=3, bucket_bytes=0)
    opt2 = zg.ZeroOptimizer(w2.numel, w2.M, w2.stage, W.master_init(w2, dev), gather="shards")
    opt2.load_state(saved)
    again = opt2.save_state()
    torch.cuda.synchronize()
    assert all(torch.equal(again[k], saved[k]) for k in ("master", "m", "v"))
    clean(opt2, "save / load")

    # the allocation-free norm
    rows = []
    for off, n, S, first in opt.buckets:
        rows += [off, n, S, first]
    table = (ctypes.c_int64 * len(rows))(*rows)
    g = opt.new_grad_buffers()
    for r in range(ws.M):
        W.fill_grads(ws, r, 9, g[r], opt.tensor_offsets)
    ptrs = (ctypes.c_void_p * ws.M)(*[x.data_ptr() for x in g])
    no = torch.empty(1, dtype=torch.float64, device=dev)
    so = torch.empty(1, dtype=torch.float32, device=dev)
    # in the checked build the call waits and returns ZERO_ERR_DEVICE if a check failed
    rc = zg._lib().zero_grad_norm_noalloc(ctypes.cast(ptrs, ctypes.c_void_p), ws.M, ctypes.cast(table, ctypes.c_void_p),
                                          len(opt.buckets), 1.0, no.data_ptr(), so.data_ptr(), None)
    assert rc == 0, f"allocation-free norm: status {rc}"
    pn = O.plan(ws.numel, ws.M, ws.bucket_bytes)
    want = math.sqrt(O.global_sumsq(pn, O.reduce_scatter(pn, [u16(x) for x in g])))
    assert abs(float(no.item()) - want) <= 1e-7 * want, "allocation-free norm vs the oracle"

    # process-per-rank mode: flat (multi-bucket, both clipped forms, unclipped) and hybrid
    import test_sharded_gpu as TS
    for kw in ({"M": 4, "stage": 3, "clip": True, "ghat_mode": "materialize"},
               {"M": 3, "stage": 1, "clip": True, "ghat_mode": "recompute"},
               {"M": 4, "stage": 2, "clip": False},
               {"M": 4, "stage": 1, "clip": True, "groups": 2},
               {"M": 8, "stage": 3, "clip": False, "groups": 2},
               {"M": 1, "stage": 2, "clip": True}):
        ranks, _, _ = TS._run(TS.RAGGED, bucket_bytes=6000, steps=2, **kw)
        for rc_ in ranks:
            site, idx = ctypes.c_int64(), ctypes.c_int64()
            assert zg._lib().zero_check_report(rc_.ctx, ctypes.byref(site), ctypes.byref(idx)) == 0
            assert site.value == 0, f"rank {rc_.rank} {kw}: bounds check {site.value} failed at {idx.value}"
            rc_.close()
    # hybrid sharding streamed bucket by bucket (per-bucket partials, bucket-restricted
    # fp32-source passes), unclipped and clipped
    for args in ((2, 4, 2, False), (2, 8, 3, True)):
        for rc_ in TS._run_hybrid_streamed(*args):
            site, idx = ctypes.c_int64(), ctypes.c_int64()
            assert zg._lib().zero_check_report(rc_.ctx, ctypes.byref(site), ctypes.byref(idx)) == 0
            assert site.value == 0, f"rank {rc_.rank} {args}: bounds check {site.value} failed at {idx.value}"
            rc_.close()
    print("checked build: all scenarios clean")


if __name__ == "__main__":
    main()
