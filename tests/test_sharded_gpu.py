"""Process-per-rank mode on the GPU, every rank's kernels against the oracle.

M rank contexts (zero_config.sharded = 1) in one process on one GPU, through the C ABI, with
device copies standing in for the collectives (tests/rank_util.py). Each rank holds only its
shard of fp32 master / m / v, its bf16 shard and the padded full parameters; its kernels read
only its own buffers. After every step, every rank is compared with the oracle's M-rank step
(orc_zero_step, or the hybrid step): the averaged gradient bit-exact (materialized form),
master / m / v within 1e-6 relative (bit-identical expected), the bf16 shard and the gathered
parameters within 1 bf16 ulp, the norm within 1e-7 of the oracle's and the same on every
rank (each rank sums the same gathered values in the same order).

Sources: "CS336 2026 Lecture 8" Slides 8 and 20; "并行训练优化、MoE扩展与系统瓶颈" 1.2.2 and
2.2.1-2.2.6; "CS231n Lecture 11" 4.3-4.4.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
import zero_gradient_reduce_scatter_gb300 as zg
from parity_util import assert_state_close, bf16_ulp_diff, f32, u16
from rank_util import RankCtx, padded_to_unpadded, run_step

pytestmark = pytest.mark.gpu

RAGGED = (3001, 1000, 37, 4099, 1, 64, 777)


def _grads(p, M, k, dev, sig_seed=5):
    """M bf16 gradients of step k in the padded layout, ~N(0, sigma_T) per tensor (the
    workloads' recipe), with garbage in the padding lanes."""
    g = []
    rng = np.random.default_rng(1000 * sig_seed + k)
    real = torch.from_numpy(p.real_mask()).to(dev)
    for q in range(M):
        x = torch.from_numpy(rng.standard_normal(p.npad).astype(np.float32) * np.float32(3e-3)).to(dev)
        t = x.to(torch.bfloat16)
        t.view(torch.int16)[~real] = 0x3F80  # 1.0 in padding: must be ignored
        g.append(t)
    return g


def _run(numel, M, stage, clip, ghat_mode="auto", bucket_bytes=0, groups=1, steps=3, max_norm=0.05,
         ghat_buffer=True, full=True):
    dev = torch.device("cuda")
    K = M // groups
    p = O.plan(numel, K, bucket_bytes)
    w = W.small_variant(W.workload("tiny"), tuple(numel), steps=steps)
    mi = W.master_init(w, dev)
    ranks = [RankCtx(numel, M, r, stage, mi, bucket_bytes, groups, ghat=ghat_buffer, full=full) for r in range(M)]
    # the clipped form each rank takes: the average materialized when asked, or by default
    # with more than 4 ranks and a buffer for it
    materialized = clip and ghat_buffer and (ghat_mode == "materialize" or (ghat_mode == "auto" and M > 4))
    assert ranks[0].sizes["npad"] == p.npad and ranks[0].sizes["shard_len"] == p.shard_len
    st = O.init_state(p, stage, f32(mi), groups=groups)
    h = zg.Hyper(clip=clip, max_grad_norm=max_norm, ghat_mode=ghat_mode)
    oh = O.hyper(clip=clip, max_grad_norm=max_norm)
    # the initial state: every rank's shard and its full parameters
    for rc in ranks:
        s = rc.grp * K + rc.owner
        assert np.array_equal(f32(rc.master), st.master[s][:p.shard_len])
        if rc.full is not None:
            assert np.array_equal(padded_to_unpadded(p, u16(rc.full)), O.bf16_rne(f32(mi)))
    saw_clip = False
    for k in range(steps):
        grads = _grads(p, M, k, dev)
        run_step(ranks, grads, h)
        full, norm, scale, rc_o = O.zero_step(p, st, [u16(g) for g in grads], oh)
        assert rc_o == 0
        torch.cuda.synchronize()
        norms = set()
        for rc in ranks:
            s = rc.grp * K + rc.owner
            assert rc.status() == 0
            assert_state_close(f32(rc.master), st.master[s][:p.shard_len], f"step {k} rank {rc.rank} master")
            assert_state_close(f32(rc.m), st.mom[s][:p.shard_len], f"step {k} rank {rc.rank} m")
            assert_state_close(f32(rc.v), st.var[s][:p.shard_len], f"step {k} rank {rc.rank} v")
            if clip:
                gn, gs = rc.last_norm()
                norms.add((gn, gs))
                assert abs(gn - norm) <= 1e-7 * norm, (gn, norm)
                saw_clip |= gs < 1.0
            if stage == 3:
                assert bf16_ulp_diff(u16(rc.shards), st.param[s][:p.shard_len]) <= 1
            if rc.full is not None:
                assert bf16_ulp_diff(padded_to_unpadded(p, u16(rc.full)), full) <= 1
        if clip:
            assert len(norms) == 1, "every rank must form the same norm and scale"
        if materialized:
            for rc in ranks:  # the materialized average: bit-exact
                s = rc.grp * K + rc.owner
                assert np.array_equal(f32(rc.ghat).view(np.uint32), st.ghat[s][:p.shard_len].view(np.uint32))
    if clip:
        assert saw_clip, "the case should exercise the clip scale"
    return ranks, p, st


@pytest.mark.parametrize("M", [1, 2, 3, 4, 8, 16])
def test_sharded_flat_clipped_zero1(M):
    for rc in _run(RAGGED, M, 1, True, bucket_bytes=8192)[0]:
        rc.close()


@pytest.mark.parametrize("ghat_mode", ["materialize", "recompute"])
@pytest.mark.parametrize("stage", [1, 2, 3])
def test_sharded_stages_and_clip_forms(stage, ghat_mode):
    for rc in _run(RAGGED, 4, stage, True, ghat_mode=ghat_mode, bucket_bytes=6000)[0]:
        rc.close()


@pytest.mark.parametrize("bucket_bytes", [0, 4096])
def test_sharded_unclipped(bucket_bytes):
    for rc in _run(RAGGED, 4, 2, False, bucket_bytes=bucket_bytes)[0]:
        rc.close()


def test_sharded_no_ghat_buffer_and_lazy_full_params():
    for rc in _run((5000, 33, 129), 2, 3, True, ghat_buffer=False, full=False)[0]:
        rc.close()


@pytest.mark.parametrize("groups,M", [(2, 4), (2, 8), (4, 8)])
@pytest.mark.parametrize("clip", [True, False])
def test_sharded_hybrid(groups, M, clip):
    for rc in _run(RAGGED, M, 1 if clip else 3, clip, bucket_bytes=6000, groups=groups)[0]:
        rc.close()


def test_sharded_tiny_shards_and_padding_only_slices():
    # 3 lanes over 16 ranks: most ranks own padding only
    for rc in _run((3,), 16, 3, True, max_norm=1e-4)[0]:
        rc.close()


def test_sharded_save_load_resume():
    """Every rank saves its lanes; the assembled state equals the oracle's; fresh contexts
    loaded from it continue bit-identically to the uninterrupted oracle run."""
    dev = torch.device("cuda")
    numel, M, stage = RAGGED, 4, 3
    ranks, p, st = _run(numel, M, stage, True, bucket_bytes=6000, steps=2)
    n = p.N
    whole = {k: torch.zeros(n, dtype=torch.int32, device=dev) for k in ("master", "m", "v")}
    for rc in ranks:  # each rank's lanes into zeroed vectors; disjoint lanes: an integer sum assembles them
        outs = [torch.zeros(n, dtype=torch.float32, device=dev) for _ in range(3)]
        assert zg._lib().zero_save_state(rc.ctx, *[o.data_ptr() for o in outs], None) == 0
        for name, o in zip(("master", "m", "v"), outs):
            whole[name] += o.view(torch.int32)
    whole = {k: x.view(torch.float32) for k, x in whole.items()}
    u = p.unpadded_index()
    real = u >= 0
    for name, attr in (("master", "master"), ("m", "mom"), ("v", "var")):
        flat = O.flat_state(p, st, attr)
        want = np.empty(n, dtype=np.float32)
        want[u[real]] = flat[real]
        assert np.array_equal(f32(whole[name]).view(np.uint32), want.view(np.uint32)), name
    t = ctypes.c_int64()
    assert zg._lib().zero_get_step(ranks[0].ctx, ctypes.byref(t)) == 0 and t.value == 2
    # fresh rank contexts (another bucket size) loaded from the assembled state
    fresh = [RankCtx(numel, M, r, stage, whole["master"], 0) for r in range(M)]
    for rc in fresh:
        assert zg._lib().zero_load_state(rc.ctx, whole["master"].data_ptr(), whole["m"].data_ptr(),
                                         whole["v"].data_ptr(), 2, None) == 0
    p2 = O.plan(numel, M, 0)
    st2 = O.init_state(p2, stage, f32(whole["master"]), f32(whole["m"]), f32(whole["v"]), t=2)
    h = zg.Hyper(clip=True, max_grad_norm=0.05)
    g = _grads(p2, M, 7, dev)
    run_step(fresh, g, h)
    full, norm, scale, _ = O.zero_step(p2, st2, [u16(x) for x in g], O.hyper(clip=True, max_grad_norm=0.05))
    for rc in fresh:
        assert_state_close(f32(rc.master), st2.master[rc.rank][:p2.shard_len], "resumed master")
        assert bf16_ulp_diff(u16(rc.shards), st2.param[rc.rank][:p2.shard_len]) <= 1
    for rc in ranks + fresh:
        rc.close()


def test_sharded_argument_errors():
    dev = torch.device("cuda")
    w = W.small_variant(W.workload("tiny"), (1000, 37), steps=1)
    mi = W.master_init(w, dev)
    rc = RankCtx((1000, 37), 2, 1, 1, mi)
    emu = zg.ZeroOptimizer((1000, 37), 2, 1, mi)
    lib, s = zg._lib(), zg._stream_handle(None)
    h = zg.Hyper(clip=True)
    # clipping needs the sums pass first and the gathered sums
    assert lib.zero_rank_step(rc.ctx, rc.recv.data_ptr(), rc.sums.data_ptr(), 1, ctypes.byref(h), s) == -1
    assert lib.zero_rank_sumsq(rc.ctx, rc.recv.data_ptr(), ctypes.byref(zg.Hyper()), rc.sumsq.data_ptr(), s) == -1
    assert lib.zero_rank_step(rc.ctx, rc.recv.data_ptr(), None, 2, ctypes.byref(zg.Hyper()), s) == -4  # stage
    assert lib.zero_rank_partial(rc.ctx, rc.recv.data_ptr(), rc.master.data_ptr(), s) == -1  # not hybrid
    assert lib.zero_rank_partial_bucket(rc.ctx, 0, rc.recv.data_ptr(), rc.master.data_ptr(), s) == -1
    assert lib.zero_rank_step(rc.ctx, rc.recv.data_ptr() + 2, None, 1, ctypes.byref(zg.Hyper()), s) == -2
    # host memory where the kernels would read or write: refused before any launch
    host = torch.zeros(rc.recv.numel(), dtype=torch.bfloat16).pin_memory()
    assert lib.zero_rank_step(rc.ctx, host.data_ptr(), None, 1, ctypes.byref(zg.Hyper()), s) == -1
    assert lib.zero_rank_step_bucket(rc.ctx, 0, host.data_ptr(), 1, ctypes.byref(zg.Hyper()), s) == -1
    hsum = torch.zeros(2, dtype=torch.float64).pin_memory()
    assert lib.zero_rank_sumsq(rc.ctx, rc.recv.data_ptr(), ctypes.byref(h), hsum.data_ptr(), s) == -1
    # the emulated mode's calls refuse a rank context, and the rank calls an emulated one
    ptrs = (ctypes.c_void_p * 2)(rc.recv.data_ptr(), rc.recv.data_ptr())
    assert lib.zero_step(rc.ctx, ctypes.cast(ptrs, ctypes.c_void_p), 1, ctypes.byref(zg.Hyper()), s) == -1
    assert lib.zero_gather(rc.ctx, -1, None, s) == -1
    assert lib.zero_rank_step(emu._ctx, rc.recv.data_ptr(), None, 1, ctypes.byref(zg.Hyper()), s) == -1
    # another rank's shard
    assert lib.zero_get_state(rc.ctx, 0, 0, rc.m.data_ptr(), s) == -1
    assert lib.zero_get_state(rc.ctx, 0, 1, rc.m.data_ptr(), s) == 0
    torch.cuda.synchronize()
    assert np.array_equal(f32(rc.m), f32(rc.master))
    # a rank outside the job
    assert zg._lib().zero_plan(ctypes.byref(zg.Config(2, 1, 0, 0, 0, 1, 2)), ctypes.cast(zg._i64_array([5]), ctypes.c_void_p),
                               1, ctypes.byref(zg.Sizes())) == -1
    rc.close()
    emu.close()


def test_sharded_per_bucket_steps_in_any_order():
    """zero_rank_step_bucket: buckets updated one at a time (reverse order, each right after its
    own exchange) equal the oracle's step; the step counter advances once all are done."""
    dev = torch.device("cuda")
    numel, M, stage = RAGGED, 4, 2
    p = O.plan(numel, M, 4096)
    assert p.nb > 3
    w = W.small_variant(W.workload("tiny"), tuple(numel), steps=2)
    mi = W.master_init(w, dev)
    ranks = [RankCtx(numel, M, r, stage, mi, 4096) for r in range(M)]
    st = O.init_state(p, stage, f32(mi))
    h = zg.Hyper()
    lib, s = zg._lib(), zg._stream_handle(None)
    from rank_util import loopback_exchange, loopback_gather
    for k in range(2):
        grads = _grads(p, M, k, dev)
        loopback_exchange(ranks, grads)
        for b in reversed(range(p.nb)):
            for rc in ranks:
                assert lib.zero_rank_step_bucket(rc.ctx, b, rc.recv.data_ptr(), stage, ctypes.byref(h), s) == 0
            if b == p.nb - 1:  # a step in progress: no second call for the bucket, no whole step
                rc = ranks[0]
                assert lib.zero_rank_step_bucket(rc.ctx, b, rc.recv.data_ptr(), stage, ctypes.byref(h), s) == -1
                assert lib.zero_rank_step(rc.ctx, rc.recv.data_ptr(), None, stage, ctypes.byref(h), s) == -1
                t = ctypes.c_int64()
                assert lib.zero_get_step(rc.ctx, ctypes.byref(t)) == 0 and t.value == k
        loopback_gather(ranks)
        full, _, _, _ = O.zero_step(p, st, [u16(g) for g in grads], O.hyper())
        torch.cuda.synchronize()
        for rc in ranks:
            assert np.array_equal(f32(rc.master).view(np.uint32), st.master[rc.rank][:p.shard_len].view(np.uint32))
            assert np.array_equal(f32(rc.v).view(np.uint32), st.var[rc.rank][:p.shard_len].view(np.uint32))
            assert bf16_ulp_diff(padded_to_unpadded(p, u16(rc.full)), full) == 0
            t = ctypes.c_int64()
            assert lib.zero_get_step(rc.ctx, ctypes.byref(t)) == 0 and t.value == k + 1
    rc = ranks[0]
    assert lib.zero_rank_step_bucket(rc.ctx, 0, rc.recv.data_ptr(), stage, ctypes.byref(zg.Hyper(clip=True)), s) == -1
    assert lib.zero_rank_step_bucket(rc.ctx, p.nb, rc.recv.data_ptr(), stage, ctypes.byref(h), s) == -1
    for rc in ranks:
        rc.close()


def test_sharded_nonfinite_on_one_rank_skips_every_rank():
    """A NaN in one rank's gradient reaches every rank through the gathered sums of squares:
    every rank skips the update (state unchanged, status NONFINITE), and the next finite step
    runs on every rank as the oracle's does."""
    dev = torch.device("cuda")
    numel, M, stage = RAGGED, 4, 1
    p = O.plan(numel, M, 6000)
    w = W.small_variant(W.workload("tiny"), tuple(numel), steps=3)
    mi = W.master_init(w, dev)
    ranks = [RankCtx(numel, M, r, stage, mi, 6000) for r in range(M)]
    st = O.init_state(p, stage, f32(mi))
    h = zg.Hyper(clip=True, max_grad_norm=0.05)
    oh = O.hyper(clip=True, max_grad_norm=0.05)
    for k in range(3):
        grads = _grads(p, M, k, dev)
        if k == 1:
            grads[2][int(p.t_off[3]) + 5] = float("nan")  # one lane of rank 2
        before = [f32(rc.master).copy() for rc in ranks]
        run_step(ranks, grads, h)
        _, norm, _, rc_o = O.zero_step(p, st, [u16(g) for g in grads], oh)
        torch.cuda.synchronize()
        for i, rc in enumerate(ranks):
            if k == 1:
                assert rc_o == 1 and rc.status() == zg.ZERO_ERR_NONFINITE
                assert np.array_equal(f32(rc.master).view(np.uint32), before[i].view(np.uint32))
            else:
                assert rc_o == 0 and rc.status() == 0
            assert_state_close(f32(rc.master), st.master[rc.rank][:p.shard_len], f"step {k} rank {rc.rank}")
            assert_state_close(f32(rc.v), st.var[rc.rank][:p.shard_len], f"step {k} rank {rc.rank} v")
    for rc in ranks:
        rc.close()


def test_sharded_largest_rank_count():
    # 64 ranks: the generic (runtime M) kernels; most ranks own a few real lanes per bucket
    # (the average over 64 ranks is small: a lower threshold keeps the clip scale in play)
    for rc in _run((3001, 1000, 37, 4099), 64, 3, True, bucket_bytes=6000, steps=2, max_norm=0.01)[0]:
        rc.close()


@pytest.mark.parametrize("groups,M,stage,clip", [(2, 4, 2, False), (4, 8, 1, False), (4, 4, 2, False),
                                                  (2, 8, 3, True), (2, 4, 1, True)])
def test_sharded_hybrid_streamed_per_bucket(groups, M, stage, clip):
    for rc in _run_hybrid_streamed(groups, M, stage, clip):
        rc.close()


def _run_hybrid_streamed(groups, M, stage, clip):
    """Hybrid sharding streamed bucket by bucket, buckets in reverse order. Per bucket: the
    group partial of that bucket only (zero_rank_partial_bucket), the cross-group gather of
    that bucket's region only, then the bucket's update (unclipped, zero_rank_step_bucket) or
    its reduction into ghat (clipped, zero_rank_reduce_bucket; then the rank's sum from the
    buckets' sums, the gathered sums and one update from the average). Against the oracle's
    hybrid step: the state within 1e-6 (bit-identical expected unclipped), the average
    bit-exact, the norm within 1e-7 and equal on every rank, the parameters within 1 ulp.
    G = M (one rank per group) included."""
    dev = torch.device("cuda")
    K = M // groups
    p = O.plan(RAGGED, K, 4096)
    assert p.nb > 3
    w = W.small_variant(W.workload("tiny"), tuple(RAGGED), steps=2)
    mi = W.master_init(w, dev)
    ranks = [RankCtx(RAGGED, M, r, stage, mi, 4096, groups) for r in range(M)]
    st = O.init_state(p, stage, f32(mi), groups=groups)
    h = zg.Hyper(clip=clip, max_grad_norm=0.05)
    oh = O.hyper(clip=clip, max_grad_norm=0.05)
    lib, s = zg._lib(), zg._stream_handle(None)
    from rank_util import loopback_exchange, loopback_gather, loopback_sums
    L = p.shard_len
    bases = np.concatenate([[0], np.cumsum(p.b_S)[:-1]])
    for k in range(2):
        grads = _grads(p, M, k, dev)
        loopback_exchange(ranks, grads)
        for b in reversed(range(p.nb)):
            base, S = int(bases[b]), int(p.b_S[b])
            for rc in ranks:
                assert lib.zero_rank_partial_bucket(rc.ctx, b, rc.recv.data_ptr(), rc.part.data_ptr(), s) == 0
            for rc in ranks:  # this bucket's region of every group's partial of this rank's shard
                for g in range(groups):
                    rc.parts[g * L + base:g * L + base + S].copy_(ranks[g * K + rc.owner].part[base:base + S])
            for rc in ranks:
                if clip:
                    assert lib.zero_rank_reduce_bucket(rc.ctx, b, rc.parts.data_ptr(), s) == 0
                else:
                    assert lib.zero_rank_step_bucket(rc.ctx, b, rc.parts.data_ptr(), stage, ctypes.byref(h), s) == 0
        if clip:
            for rc in ranks:
                assert lib.zero_rank_sumsq(rc.ctx, None, ctypes.byref(h), rc.sumsq.data_ptr(), s) == 0
            loopback_sums(ranks)
            for rc in ranks:
                assert lib.zero_rank_step(rc.ctx, None, rc.sums.data_ptr(), stage, ctypes.byref(h), s) == 0
        loopback_gather(ranks)
        full, norm, scale, rc_o = O.zero_step(p, st, [u16(g) for g in grads], oh)
        assert rc_o == 0 and (scale < 1.0 or not clip)
        torch.cuda.synchronize()
        norms = set()
        for rc in ranks:
            q = rc.grp * K + rc.owner
            assert rc.status() == 0
            assert_state_close(f32(rc.master), st.master[q][:L], f"step {k} rank {rc.rank} master")
            assert_state_close(f32(rc.m), st.mom[q][:L], f"step {k} rank {rc.rank} m")
            assert_state_close(f32(rc.v), st.var[q][:L], f"step {k} rank {rc.rank} v")
            if clip:
                assert np.array_equal(f32(rc.ghat).view(np.uint32), st.ghat[q][:L].view(np.uint32))
                gn, gs = rc.last_norm()
                assert abs(gn - norm) <= 1e-7 * norm
                norms.add((gn, gs))
            assert bf16_ulp_diff(padded_to_unpadded(p, u16(rc.full)), full) <= 1
        assert len(norms) <= 1
    rc = ranks[0]
    assert lib.zero_rank_partial_bucket(rc.ctx, p.nb, rc.recv.data_ptr(), rc.part.data_ptr(), s) == -1
    assert lib.zero_rank_partial_bucket(rc.ctx, -1, rc.recv.data_ptr(), rc.part.data_ptr(), s) == -1
    return ranks


def test_sharded_clipped_streaming_reduce_then_apply():
    """zero_rank_reduce_bucket per bucket (reverse order, each right after its exchange), then
    the rank's sum from the buckets' sums, the gathered sums and the update from the average:
    the average bit-exact and the state as the oracle's clipped step."""
    dev = torch.device("cuda")
    numel, M, stage = RAGGED, 4, 2
    p = O.plan(numel, M, 4096)
    assert p.nb > 3
    w = W.small_variant(W.workload("tiny"), tuple(numel), steps=3)
    mi = W.master_init(w, dev)
    ranks = [RankCtx(numel, M, r, stage, mi, 4096) for r in range(M)]
    st = O.init_state(p, stage, f32(mi))
    h = zg.Hyper(clip=True, max_grad_norm=0.05)
    lib, s = zg._lib(), zg._stream_handle(None)
    from rank_util import loopback_exchange, loopback_gather, loopback_sums
    for k in range(3):
        grads = _grads(p, M, k, dev)
        loopback_exchange(ranks, grads)
        for b in reversed(range(p.nb)):
            for rc in ranks:
                assert lib.zero_rank_reduce_bucket(rc.ctx, b, rc.recv.data_ptr(), s) == 0
            if b == 1:  # not every bucket reduced yet: no sum, no whole-step call
                rc = ranks[0]
                assert lib.zero_rank_sumsq(rc.ctx, None, ctypes.byref(h), rc.sumsq.data_ptr(), s) == -1
                assert lib.zero_rank_sumsq(rc.ctx, rc.recv.data_ptr(), ctypes.byref(h), rc.sumsq.data_ptr(), s) == -1
                assert lib.zero_rank_step(rc.ctx, rc.recv.data_ptr(), None, stage, ctypes.byref(zg.Hyper()), s) == -1
        for rc in ranks:
            assert lib.zero_rank_sumsq(rc.ctx, None, ctypes.byref(h), rc.sumsq.data_ptr(), s) == 0
        loopback_sums(ranks)
        for rc in ranks:
            assert lib.zero_rank_step(rc.ctx, None, rc.sums.data_ptr(), stage, ctypes.byref(h), s) == 0
        loopback_gather(ranks)
        full, norm, scale, _ = O.zero_step(p, st, [u16(g) for g in grads], O.hyper(clip=True, max_grad_norm=0.05))
        assert scale < 1.0
        torch.cuda.synchronize()
        for rc in ranks:
            assert np.array_equal(f32(rc.ghat).view(np.uint32), st.ghat[rc.rank][:p.shard_len].view(np.uint32))
            gn, gs = rc.last_norm()
            assert abs(gn - norm) <= 1e-7 * norm
            assert_state_close(f32(rc.master), st.master[rc.rank][:p.shard_len], f"step {k} master")
            assert_state_close(f32(rc.m), st.mom[rc.rank][:p.shard_len], f"step {k} m")
            assert_state_close(f32(rc.v), st.var[rc.rank][:p.shard_len], f"step {k} v")
            assert bf16_ulp_diff(padded_to_unpadded(p, u16(rc.full)), full) <= 1
    rc = ranks[0]
    nog = RankCtx(numel, M, 0, stage, mi, 4096, ghat=False)
    assert lib.zero_rank_reduce_bucket(nog.ctx, 0, nog.recv.data_ptr(), s) == -3  # needs a ghat buffer
    assert lib.zero_rank_reduce_bucket(rc.ctx, p.nb, rc.recv.data_ptr(), s) == -1
    for rc in ranks + [nog]:
        rc.close()


@pytest.mark.parametrize("ghat_mode", ["materialize", "recompute"])
def test_sharded_zero_size_tensors_and_many_buckets(ghat_mode):
    # zero-size tensors between real ones, 64-byte buckets (about one tensor each: ~60 local
    # buckets walked by one launch), 3 ranks (inexact 1/M, generic source count)
    numel = tuple([0, 5, 0, 1, 33, 0] + [17 + 29 * i for i in range(50)] + [0, 1000, 3])
    for rc in _run(numel, 3, 3, True, ghat_mode=ghat_mode, bucket_bytes=64, max_norm=0.01)[0]:
        rc.close()


@pytest.mark.parametrize("seed", range(12))
def test_sharded_random_configurations(seed):
    """Seeded random configurations: tensor sizes (some zero), rank count, groups, stage,
    bucket cap and clipping form, two steps each, every rank against the oracle."""
    rng = np.random.default_rng(9000 + seed)
    T = int(rng.integers(1, 9))
    numel = tuple(int(x) if rng.random() > 0.15 else 0 for x in rng.integers(1, 6000, T))
    if sum(numel) == 0:
        numel = numel + (11,)
    groups = int(rng.choice([1, 1, 2]))
    M = groups * int(rng.choice([1, 2, 3, 4])) if groups > 1 else int(rng.integers(1, 10))
    stage = int(rng.integers(1, 4))
    clip = bool(rng.random() < 0.6)
    ghat_mode = str(rng.choice(["auto", "materialize", "recompute"]))
    bucket_bytes = int(rng.choice([0, 128, 3000]))
    for rc in _run(numel, M, stage, clip, ghat_mode=ghat_mode, bucket_bytes=bucket_bytes, groups=groups, steps=2,
                   max_norm=1e-4)[0]:
        rc.close()
