"""Process-per-rank mode at the workloads' full sizes: every rank's kernels against the oracle.

M rank contexts (zero_config.sharded = 1) in one process, through the C ABI, with device
copies in place of the collectives (tests/rank_util.py), over the full GPT-2-small, 1.3B and
4B layouts (the launch configuration of bench.py --shard --emulate-ranks). The oracle cannot
hold the whole state at these sizes, so it checks:
  * every rank's norm of every clipped step against the oracle's norm, streamed from all M
    gradient buffers (fp64, ascending flat order), within 1e-7 relative, and the same on
    every rank;
  * sampled lanes -- every bucket, shard and tensor boundary, padding lanes, the lanes around
    2^31 and 2^32, random lanes -- mapped to their owner rank and its local lane, and
    followed through all steps by the oracle's per-lane trajectories (master / m / v within
    1e-6, the materialized average bit-exact, the gathered bf16 parameters within 1 ulp);
and, over every rank's whole shard, that its bf16 shard is round-to-nearest-even of its
fp32 master at every lane and that padding lanes of the state stay exactly 0.

Sources: "CS336 2026 Lecture 8" Slides 8 and 20; "并行训练优化、MoE扩展与系统瓶颈" 1.2.2 and
2.2.1-2.2.6.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from parity_util import REL_NORM, bf16_ulp_diff, f32, make_hyper, state_errors, u16
from rank_util import RankCtx, run_step
from test_parity_full_gpu import CHUNK, sample_lanes, streamed_norm, unpadded_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    yield
    torch.cuda.empty_cache()


def owner_of(p, lanes):
    """(owner rank, local lane in its shard) of each padded lane, from the oracle's plan."""
    b = np.searchsorted(p.b_off, lanes, side="right") - 1
    S = p.b_S[b]
    rel = lanes - p.b_off[b]
    r = rel // S
    base = np.concatenate([[0], np.cumsum(p.b_S)[:-1]])
    return r, base[b] + rel - r * S


@pytest.mark.parametrize("key", ["gpt2s", "1p3b", "4b"])
def test_sharded_full_size_workload(key):
    w = W.workload(key)
    dev = torch.device("cuda")
    rng = np.random.default_rng(2000 + W.KEYS.index(key))
    mi = W.master_init(w, dev)
    M, K = w.M, w.steps
    # every rank keeps the full parameters at stages 1 and 2; at ZeRO-3 only rank 0 (the
    # all-gather's result to check), the others only their shards
    ranks = [RankCtx(w.numel, M, r, w.stage, mi, w.bucket_bytes, ghat=M > 4, full=(r == 0 or w.stage < 3))
             for r in range(M)]
    h, oh = make_hyper(w)
    p = O.plan(w.numel, M, w.bucket_bytes)
    assert p.npad == ranks[0].sizes["npad"] and [int(x) for x in p.t_off] == ranks[0].tensor_offsets

    lanes = sample_lanes(p, rng)
    u, real = unpadded_of(p, lanes)
    own, loc = owner_of(p, lanes)
    lanes_d = torch.from_numpy(lanes).to(dev)
    u_real_d = torch.from_numpy(u[real]).to(dev)
    p0 = np.zeros(lanes.size, np.float32)
    p0[real] = f32(mi[u_real_d])
    del mi
    L = lanes.size
    g_samp = np.empty((K, M, L), np.uint16)
    scales, applies, ghat_gpu = [], [], []
    sig = W.sigmas(w)
    grads = [torch.zeros(p.npad, dtype=torch.bfloat16, device=dev) for _ in range(M)]
    pinned = [torch.empty(CHUNK, dtype=torch.int16).pin_memory() for _ in range(M)] if w.clip else None
    materialized = w.clip is not None and M > 4

    def per_rank(get):
        """Values of the sampled lanes gathered from their owners' shards."""
        out = np.empty(L, np.float32)
        for r in range(M):
            sel = own == r
            if sel.any():
                out[sel] = f32(get(ranks[r])[torch.from_numpy(loc[sel]).to(dev)])
        return out

    for k in range(K):
        for r in range(M):
            grads[r].zero_()
            W.fill_grads(w, r, k, grads[r], ranks[0].tensor_offsets, sig)
            g_samp[k, r] = u16(grads[r][lanes_d])
        run_step(ranks, grads, h)
        torch.cuda.synchronize()
        assert all(rc.status() == 0 for rc in ranks)
        if materialized:
            ghat_gpu.append(per_rank(lambda rc: rc.ghat))
        if w.clip:
            norm = streamed_norm(p, grads, pinned)
            seen = {rc.last_norm() for rc in ranks}
            assert len(seen) == 1, "every rank forms the same norm and scale"
            gn, gs = seen.pop()
            assert abs(gn - norm) <= REL_NORM * norm, (k, gn, norm)
            scales.append(O.clip_scale(norm, w.clip))
        else:
            scales.append(1.0)
        applies.append(1)
    del grads, pinned
    torch.cuda.synchronize()

    pm, mm, vm = p0.copy(), np.zeros(L, np.float32), np.zeros(L, np.float32)
    bf, gh = O.lane_steps(M, g_samp, real, scales, applies, oh, 1, pm, mm, vm, want_ghat=True)
    assert state_errors(per_rank(lambda rc: rc.master), pm) <= 1.0
    assert state_errors(per_rank(lambda rc: rc.m), mm) <= 1.0
    assert state_errors(per_rank(lambda rc: rc.v), vm) <= 1.0
    assert bf16_ulp_diff(u16(ranks[0].full[lanes_d][torch.from_numpy(real).to(dev)]), bf[real]) <= 1
    if materialized:
        assert np.array_equal(np.stack(ghat_gpu).view(np.uint32), gh.view(np.uint32)), "averaged gradient not bit-exact"

    # whole-shard properties on every rank
    for rc in ranks:
        assert torch.equal(rc.shards.view(torch.int16), rc.master.to(torch.bfloat16).view(torch.int16))
        base = 0
        for b in range(p.nb):
            S, n = int(p.b_S[b]), int(p.b_n[b])
            nreal = min(max(n - rc.rank * S, 0), S)
            for buf in (rc.master, rc.m, rc.v):
                assert int(torch.count_nonzero(buf[base + nreal:base + S])) == 0, "padding lanes must stay 0"
            base += S
    for rc in ranks:
        rc.close()
