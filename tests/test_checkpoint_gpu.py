"""Checkpoint, resume and reshard (M -> M') through zero_save_state / zero_load_state.

The saved form is unpadded fp32 master / m / v plus the step count, so it does not depend
on the rank count, bucket size or stage ("CS336 2026 Lecture 8" Slide 67: checkpointing and
elastic restart are among the needs of runs at scale). A job saved at one M continues at
another; the continuation is compared bit for bit with the oracle started from the same
unpadded state.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
import zero_gradient_reduce_scatter_gb300 as zg
from parity_util import f32, make_hyper, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    yield


NUMEL = W.ragged_numel(40, 100, 9000, 21)


def _steps(opt, w, steps, sig, first_step):
    h, _ = make_hyper(w)
    hosts = []
    for k in range(first_step, first_step + steps):
        grads = opt.new_grad_buffers()
        for r in range(w.M):
            W.fill_grads(w, r, k, grads[r], opt.tensor_offsets, sig)
        opt.step(grads, h)
        hosts.append([u16(g) for g in grads])
    assert opt.sync_status() == 0
    return hosts


def _oracle_continue(w, state, hosts):
    p = O.plan(w.numel, w.M, w.bucket_bytes)
    st = O.init_state(p, w.stage, f32(state["master"]), f32(state["m"]), f32(state["v"]), t=state["t"])
    _, oh = make_hyper(w)
    full = None
    for gs in hosts:
        full, _, _, rc = O.zero_step(p, st, gs, oh)
        assert rc == 0
    u = p.unpadded_index()
    return full, {k: O.flat_state(p, st, n)[u >= 0] for k, n in (("master", "master"), ("m", "mom"), ("v", "var"))}


def test_save_reshard_resume_matches_oracle(tmp_path):
    dev = torch.device("cuda")
    wA = W.small_variant(W.workload("ragged"), NUMEL, M=4, steps=2)                  # ZeRO-3, clip, M = 4
    sig = W.sigmas(wA)
    A = zg.ZeroOptimizer(wA.numel, wA.M, wA.stage, W.master_init(wA, dev), gather="shards")
    hostsA = _steps(A, wA, 2, sig, 0)
    saved = A.save_state()
    torch.cuda.synchronize()
    assert saved["t"] == 2
    # the saved form equals the oracle's state after the same two steps, bit for bit
    pA = O.plan(wA.numel, wA.M, 0)
    stA = O.init_state(pA, wA.stage, f32(W.master_init(wA, dev)))
    _, oh = make_hyper(wA)
    for gs in hostsA:
        O.zero_step(pA, stA, gs, oh)
    uA = pA.unpadded_index()
    for k, n in (("master", "master"), ("m", "mom"), ("v", "var")):
        assert np.array_equal(f32(saved[k]).view(np.uint32), O.flat_state(pA, stA, n)[uA >= 0].view(np.uint32)), k

    # reshard into M = 6, ZeRO-2, small buckets (generic-M kernels, several buckets)
    wB = W.small_variant(W.workload("ragged"), NUMEL, M=6, stage=2, bucket_bytes=30000, steps=2)
    B = zg.ZeroOptimizer(wB.numel, wB.M, wB.stage, W.master_init(wB, dev), bucket_bytes=wB.bucket_bytes)
    B.load_state(saved)
    assert B.t == 2
    again = B.save_state()
    torch.cuda.synchronize()
    for k in ("master", "m", "v"):
        assert torch.equal(again[k], saved[k]), k
    # parameters were rebuilt from the loaded master
    assert torch.equal(B.params(), saved["master"].to(torch.bfloat16))
    hostsB = _steps(B, wB, 2, sig, 2)
    full, want = _oracle_continue(wB, saved, hostsB)
    got = B.save_state()
    torch.cuda.synchronize()
    for k in ("master", "m", "v"):
        assert np.array_equal(f32(got[k]).view(np.uint32), want[k].view(np.uint32)), k
    assert np.array_equal(u16(B.params()), full)

    # through a checkpoint file into M = 8, ZeRO-1
    path = tmp_path / "ckpt.pt"
    torch.save(B.state_dict(), path)
    wC = W.small_variant(W.workload("ragged"), NUMEL, M=8, stage=1, steps=1)
    C = zg.ZeroOptimizer(wC.numel, wC.M, wC.stage, W.master_init(wC, dev))
    C.load_state_dict(torch.load(path))
    assert C.t == 4
    stB = B.save_state()
    hostsC = _steps(C, wC, 1, sig, 4)
    full, want = _oracle_continue(wC, stB, hostsC)
    got = C.save_state()
    torch.cuda.synchronize()
    for k in ("master", "m", "v"):
        assert np.array_equal(f32(got[k]).view(np.uint32), want[k].view(np.uint32)), k
    assert np.array_equal(u16(C.params()), full)


@pytest.mark.parametrize("stage,gather,groups", [(1, "fused", 1), (3, "shards", 1), (2, "fused", 2)])
def test_resume_is_bitwise_continuation(stage, gather, groups):
    """K steps straight == K1 steps, save, load into a fresh context of the same layout, K2 steps."""
    dev = torch.device("cuda")
    w = W.small_variant(W.workload("ragged"), NUMEL, M=8, stage=stage, steps=4, clip=0.05)
    sig = W.sigmas(w)
    mi = W.master_init(w, dev)

    def make():
        return zg.ZeroOptimizer(w.numel, w.M, w.stage, mi, gather=gather, groups=groups)

    A = make()
    _steps(A, w, 4, sig, 0)
    B = make()
    _steps(B, w, 2, sig, 0)
    saved = B.save_state()
    C = make()
    C.load_state(saved)
    assert C.t == 2
    _steps(C, w, 2, sig, 2)
    torch.cuda.synchronize()
    for name in ("master", "m", "v"):
        assert torch.equal(getattr(A, name).view(torch.int32), getattr(C, name).view(torch.int32)), name
    assert torch.equal(A.params().view(torch.int16), C.params().view(torch.int16))
    assert A.t == C.t == 4


def test_load_rejects_wrong_sizes():
    dev = torch.device("cuda")
    w = W.small_variant(W.workload("1p3b"), (1000, 24), steps=1)
    opt = zg.ZeroOptimizer(w.numel, w.M, w.stage, W.master_init(w, dev))
    with pytest.raises(ValueError):
        opt.load_state({"master": torch.zeros(10, device=dev), "t": 0})
    with pytest.raises(ValueError):
        opt.load_state_dict({"numel": [1024], "t": 0, "master": torch.zeros(1024)})
