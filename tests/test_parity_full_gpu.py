"""GPU vs oracle at the workloads' full sizes, in the launch configuration bench.py times.

At these sizes the oracle cannot hold the whole state, so it checks:
  * the global norm of every clipped step, recomputed by the oracle from all M gradient
    buffers streamed to the host (fp64, ascending flat order), within 1e-7 relative;
  * sampled lanes -- every bucket, shard and tensor boundary, padding lanes, the lanes
    around 2^31 and 2^32, and random lanes -- followed through all steps by the oracle's
    per-lane trajectories (bit-exact averaged gradient; master / m / v within 1e-6; bf16
    parameters within 1 ulp);
and, over the whole buffers, properties that hold at any size: padding lanes of the state
stay exactly 0, and the gathered bf16 parameters equal round-to-nearest-even of the fp32
master at every real lane (the all-gather indexing, bit for bit).
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
import zero_gradient_reduce_scatter_gb300 as zg
from parity_util import REL_NORM, bf16_ulp_diff, f32, make_hyper, state_errors, u16

pytestmark = pytest.mark.gpu

CHUNK = 1 << 25  # lanes per host chunk of the streamed norm


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    yield
    torch.cuda.empty_cache()


def sample_lanes(p, rng, n_random=40000):
    M = p.M
    s = set()
    for b in range(p.nb):
        off, n, S = int(p.b_off[b]), int(p.b_n[b]), int(p.b_S[b])
        end = off + M * S
        for r in range(M + 1):
            for d in (-2, -1, 0, 1):
                s.add(off + r * S + d)
        for x in (off + n - 1, off + n, off + n + 1, end - 1):
            s.add(x)
    for t in range(len(p.numel)):
        if p.numel[t]:
            s.update((int(p.t_off[t]), int(p.t_off[t]) + int(p.numel[t]) - 1))
    for x in (2 ** 31 - 1, 2 ** 31, 2 ** 32 - 1, 2 ** 32, 2 ** 32 + 7):
        s.add(x)
    s.update(int(x) for x in rng.integers(0, p.npad, n_random))
    lanes = np.array(sorted(x for x in s if 0 <= x < p.npad), dtype=np.int64)
    return lanes


def unpadded_of(p, lanes):
    """Unpadded index of each lane (-1 for padding), from the oracle's plan."""
    b = np.searchsorted(p.b_off, lanes, side="right") - 1
    uoff = np.concatenate([[0], np.cumsum(p.b_n)[:-1]])
    rel = lanes - p.b_off[b]
    real = rel < p.b_n[b]
    return np.where(real, uoff[b] + rel, -1), real


def streamed_norm(p, grads, pinned):
    acc = 0.0
    for o0 in range(0, p.npad, CHUNK):
        n = min(CHUNK, p.npad - o0)
        chunk = []
        for r, g in enumerate(grads):
            pinned[r][:n].copy_(g[o0:o0 + n].view(torch.int16))
            chunk.append(pinned[r][:n].numpy().view(np.uint16))
        acc = O.sumsq_chunk(acc, p, chunk, o0)
    return math.sqrt(acc)


@pytest.mark.parametrize("key", ["gpt2s", "1p3b", "ragged", "4b"])
def test_full_size_workload(key):
    w = W.workload(key)
    dev = torch.device("cuda")
    rng = np.random.default_rng(1000 + W.KEYS.index(key))
    mi = W.master_init(w, dev)
    # the launch configuration bench.py times: fused all-gather, automatic averaged-gradient mode
    opt = zg.ZeroOptimizer(w.numel, w.M, w.stage, mi, bucket_bytes=w.bucket_bytes, gather="fused")
    h, oh = make_hyper(w)
    p = O.plan(w.numel, w.M, w.bucket_bytes)
    assert p.npad == opt.sizes["npad"] and [int(x) for x in p.t_off] == opt.tensor_offsets

    lanes = sample_lanes(p, rng)
    u, real = unpadded_of(p, lanes)
    lanes_d = torch.from_numpy(lanes).to(dev)
    u_real_d = torch.from_numpy(u[real]).to(dev)
    p0 = np.zeros(lanes.size, np.float32)
    p0[real] = f32(mi[u_real_d])
    del mi
    K, M, L = w.steps, w.M, lanes.size
    g_samp = np.empty((K, M, L), np.uint16)
    scales, applies, ghat_gpu = [], [], []
    sig = W.sigmas(w)
    grads = opt.new_grad_buffers()
    pinned = [torch.empty(CHUNK, dtype=torch.int16).pin_memory() for _ in range(M)] if w.clip else None
    for k in range(K):
        for r in range(M):
            grads[r].zero_()
            W.fill_grads(w, r, k, grads[r], opt.tensor_offsets, sig)
            g_samp[k, r] = u16(grads[r][lanes_d])
        opt.step(grads, h)
        assert opt.sync_status() == 0
        if opt.ghat is not None and w.clip:
            ghat_gpu.append(f32(opt.ghat[lanes_d]))
        if w.clip:
            norm = streamed_norm(p, grads, pinned)
            gn, gs = opt.last_norm()
            assert abs(gn - norm) <= REL_NORM * norm, (k, gn, norm)
            scales.append(O.clip_scale(norm, w.clip))
        else:
            scales.append(1.0)
        applies.append(1)
    del grads, pinned
    torch.cuda.synchronize()

    pm, mm, vm = p0.copy(), np.zeros(L, np.float32), np.zeros(L, np.float32)
    bf, gh = O.lane_steps(M, g_samp, real, scales, applies, oh, 1, pm, mm, vm, want_ghat=True)
    assert state_errors(f32(opt.master[lanes_d]), pm) <= 1.0
    assert state_errors(f32(opt.m[lanes_d]), mm) <= 1.0
    assert state_errors(f32(opt.v[lanes_d]), vm) <= 1.0
    assert bf16_ulp_diff(u16(opt.params()[u_real_d]), bf[real]) <= 1
    if ghat_gpu and len(ghat_gpu) == K:
        assert np.array_equal(np.stack(ghat_gpu).view(np.uint32), gh.view(np.uint32)), "averaged gradient not bit-exact"

    # whole-buffer properties
    full = opt.params()
    uoff = 0
    for b in range(p.nb):
        off, n, end = int(p.b_off[b]), int(p.b_n[b]), int(p.b_off[b] + M * p.b_S[b])
        for buf in (opt.master, opt.m, opt.v):
            assert int(torch.count_nonzero(buf[off + n:end])) == 0, "padding lanes must stay 0"
        want = opt.master[off:off + n].to(torch.bfloat16)
        assert torch.equal(full[uoff:uoff + n].view(torch.int16), want.view(torch.int16)), f"bucket {b} gather"
        del want
        uoff += n
    opt.close()
