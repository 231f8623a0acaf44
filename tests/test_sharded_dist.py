"""The collectives of the process-per-rank ZeRO step on CPU (gloo), checked against the oracle.

Ranks are real processes (spawned, gloo over 127.0.0.1). Each rank runs the binding's
exchange and all-gather helpers on CPU tensors (no CUDA; the library's kernels are not
involved) and checks, against the oracle's own planner and step:

  - the exchange delivers to owner r exactly the bytes the oracle's reduce-scatter reads for
    r: the received slice of source q at the exchange position equals source q's gradient
    lane of r's shard, bit for bit (garbage in the gradients' padding travels unchanged);
    and the oracle's reduce-scatter of gradients rebuilt from the received bytes alone
    (NaN everywhere else) gives owner r's averaged shard bit for bit, so no lane outside
    the received ones is read;
  - the all-gather of the oracle's bf16 shards gives the oracle's gathered parameters at
    every real lane;
  - the per-rank sums of squares arrive in rank order, and their ordered sum equals the
    oracle's global sum of squares within the fp64 reassociation error;
  - hybrid sharding (4 ranks as 2 groups of 2): the in-group exchange and the cross-group
    gather of group partials deliver the oracle's operands in group order, and the sum of
    the gathered partials in group order times (float)(1/M) is the oracle's hybrid average.

Sources: "CS336 2026 Lecture 8" Slides 8 and 20 (reduce-scatter to owners, owner update,
all-gather); "并行训练优化、MoE扩展与系统瓶颈" 1.2.2 (reduce_scatter_sum / all_gather) and
2.2.1-2.2.6; "CS231n Lecture 11" 4.4 (hybrid sharding).
"""
import os
import socket
import sys
import traceback

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

BF16_NAN = 0x7FC0

# (numel, bucket_bytes) cases: ragged sizes not divisible by M, one bucket and several
CASES = {
    "one_bucket": ((1000, 37, 3001, 5), 0),
    "two_buckets_ragged": ((3001, 1000, 37), 6100),
    "many_buckets": ((129, 4099, 1, 64, 777, 2048, 13), 4096),
}


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _grads(p, M, seed):
    """M bf16 gradients (uint16 bit patterns) of the padded layout: small-integer dyadic
    values on real lanes (exact sums, so an averaged lane identifies its operands) and
    garbage on padding lanes."""
    import oracle as O
    rng = np.random.default_rng(seed)
    real = p.real_mask()
    out = []
    for q in range(M):
        vals = rng.integers(-64, 65, size=p.npad).astype(np.float32) * np.float32(2.0 ** -6)
        g = O.bf16_rne(vals)
        g[~real] = rng.integers(0, 0x7F00, size=int((~real).sum())).astype(np.uint16)  # garbage, finite
        out.append(g)
    return out


def _run(rank, world, port, case, q, fn):
    try:
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        import torch.distributed as dist
        dist.init_process_group("gloo", rank=rank, world_size=world)
        try:
            fn(rank, world, case)
        finally:
            dist.destroy_process_group()
        q.put((rank, "ok"))
    except BaseException:
        q.put((rank, traceback.format_exc()))


def _spawn(world, case, fn):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_run, args=(r, world, port, case, q, fn)) for r in range(world)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    bad = {r: v for r, v in got.items() if v != "ok"}
    assert not bad, "\n".join(f"rank {r}:\n{v}" for r, v in bad.items())
    assert all(p.exitcode == 0 for p in procs)


def _flat_rank(rank, M, case):
    import torch
    import torch.distributed as dist

    import oracle as O
    import zero_gradient_reduce_scatter_gb300 as zg
    from zero_gradient_reduce_scatter_gb300.sharded import exchange_gradients, gather_params

    numel, bucket_bytes = CASES[case]
    p = O.plan(numel, M, bucket_bytes)
    toff, buckets = zg.layout(numel, M, 1, bucket_bytes)  # the library's planner (host code)
    assert [int(x) for x in p.t_off] == toff
    assert [(int(a), int(b), int(c)) for a, b, c in zip(p.b_off, p.b_n, p.b_S)] == [bk[:3] for bk in buckets]
    assert p.nb >= (2 if case != "one_bucket" else 1)

    G = _grads(p, M, seed=1234)  # every rank can rebuild every rank's gradient
    mine = torch.from_numpy(G[rank].view(np.int16).copy()).view(torch.bfloat16)
    recv = torch.full((p.npad,), 0, dtype=torch.int16).view(torch.bfloat16)
    exchange_gradients(mine, recv, buckets, M)
    got = recv.view(torch.int16).numpy().view(np.uint16)

    # (1) exchange position of every (source, lane of this rank's shard), from the oracle plan
    for b in range(p.nb):
        off, S = int(p.b_off[b]), int(p.b_S[b])
        for src in range(M):
            want = G[src][off + rank * S: off + (rank + 1) * S]
            assert np.array_equal(got[off + src * S: off + (src + 1) * S], want), (b, src)

    # (1b) bucket by bucket, in backward order, asynchronously: the same bytes
    recv2 = torch.zeros(p.npad, dtype=torch.int16).view(torch.bfloat16)
    works = exchange_gradients(mine, recv2, buckets, M, which=list(reversed(range(p.nb))), async_op=True)
    for wk in works:
        wk.wait()
    assert torch.equal(recv2.view(torch.int16), recv.view(torch.int16))

    # (2) the oracle's reduce-scatter needs nothing else: rebuild the M gradients from the
    # received bytes only (NaN on every lane that did not arrive here) and average
    virt = [np.full(p.npad, BF16_NAN, dtype=np.uint16) for _ in range(M)]
    for b in range(p.nb):
        off, S = int(p.b_off[b]), int(p.b_S[b])
        for src in range(M):
            virt[src][off + rank * S: off + (rank + 1) * S] = got[off + src * S: off + (src + 1) * S]
    ghat_virtual = O.reduce_scatter(p, virt)[rank]
    ghat_true = O.reduce_scatter(p, G)[rank]
    assert np.array_equal(ghat_virtual.view(np.uint32), ghat_true.view(np.uint32))
    assert not np.isnan(ghat_virtual).any()

    # (3) the all-gather of the oracle's bf16 shards (ZeRO-3 shards after one clipped step)
    master = np.random.default_rng(7).standard_normal(p.N).astype(np.float32) * np.float32(0.02)
    st = O.init_state(p, 3, master)
    full_want, norm, scale, rc = O.zero_step(p, st, G, O.hyper(clip=True, max_grad_norm=0.05))
    assert rc == 0
    shard = torch.from_numpy(st.param[rank][:p.shard_len].view(np.int16).copy()).view(torch.bfloat16)
    full = torch.zeros(p.npad, dtype=torch.int16).view(torch.bfloat16)
    gather_params(shard, full, buckets, M)
    full_u = full.view(torch.int16).numpy().view(np.uint16)
    u = p.unpadded_index()
    real = u >= 0
    assert np.array_equal(full_u[real][np.argsort(u[real])], full_want)
    for i, n in enumerate(numel):  # tensor views of the padded buffer are the tensors
        assert np.array_equal(full_u[toff[i]:toff[i] + n], full_want[sum(numel[:i]):sum(numel[:i]) + n])

    # (4) the norm's scalars: this rank's sum of squares over the real lanes of its averaged
    # shard; gathered in rank order; their ordered sum against the oracle's global sum
    st2 = O.init_state(p, 1, master)
    O.zero_step(p, st2, G, O.hyper(clip=True, max_grad_norm=0.05))
    shard_real = np.zeros(p.shard_len, dtype=bool)
    base = 0
    for b in range(p.nb):
        S, n = int(p.b_S[b]), int(p.b_n[b])
        shard_real[base: base + S] = (rank * S + np.arange(S)) < n
        base += S
    gh = st2.ghat[rank][:p.shard_len].astype(np.float64)
    mine_sq = torch.tensor([float(np.sum(gh[shard_real] ** 2))], dtype=torch.float64)
    sums = torch.zeros(M, dtype=torch.float64)
    dist.all_gather_into_tensor(sums, mine_sq)
    assert sums[rank].item() == mine_sq.item()
    total = 0.0
    for v in sums.tolist():
        total += v
    want_sq = O.global_sumsq(p, st2.ghat)
    assert abs(total - want_sq) <= 1e-12 * want_sq
    assert abs(np.sqrt(total) - norm) <= 1e-12 * norm  # the clipped step's norm


@pytest.mark.parametrize("case", list(CASES))
def test_sharded_exchange_two_ranks(case):
    _spawn(2, case, _flat_rank)


def _hybrid_rank(rank, M, case):
    import torch
    import torch.distributed as dist

    import oracle as O
    from zero_gradient_reduce_scatter_gb300.sharded import exchange_gradients, gather_params, hybrid_groups

    G_groups = 2
    K = M // G_groups
    numel, bucket_bytes = CASES[case]
    p = O.plan(numel, K, bucket_bytes)  # hybrid: the layout is planned for the group size
    grp, k = divmod(rank, K)
    intra, cross = hybrid_groups(M, G_groups)
    assert intra[grp][k] == rank and cross[k][grp] == rank
    pg_intra = [dist.new_group(r) for r in intra][grp]
    pg_cross = [dist.new_group(r) for r in cross][k]
    buckets = [(int(p.b_off[b]), int(p.b_n[b]), int(p.b_S[b]), 0) for b in range(p.nb)]

    Gr = _grads(p, M, seed=99)
    mine = torch.from_numpy(Gr[rank].view(np.int16).copy()).view(torch.bfloat16)
    recv = torch.zeros(p.npad, dtype=torch.int16).view(torch.bfloat16)
    exchange_gradients(mine, recv, buckets, K, pg_intra)
    got = recv.view(torch.int16).numpy().view(np.uint16)
    for b in range(p.nb):
        off, S = int(p.b_off[b]), int(p.b_S[b])
        for kk in range(K):  # member kk of this group
            want = Gr[grp * K + kk][off + k * S: off + (k + 1) * S]
            assert np.array_equal(got[off + kk * S: off + (kk + 1) * S], want)

    # group partial of this shard (the library's zero_rank_partial computes it on the GPU;
    # here the oracle's own rank-ordered sum of this group's K gradients, via reduce_scatter
    # over the group with 1/K undone exactly -- K is a power of two), gathered across groups
    grp_grads = Gr[grp * K:(grp + 1) * K]
    part = O.reduce_scatter(p, grp_grads)[k] * np.float32(K)
    parts = torch.zeros(G_groups * p.shard_len, dtype=torch.float32)
    dist.all_gather_into_tensor(parts, torch.from_numpy(part.copy()), group=pg_cross)
    parts = parts.numpy().reshape(G_groups, p.shard_len)
    for g2 in range(G_groups):  # group order
        want = O.reduce_scatter(p, Gr[g2 * K:(g2 + 1) * K])[k] * np.float32(K)
        assert np.array_equal(parts[g2].view(np.uint32), want.view(np.uint32))
    # summed in group order from +0, times 1/M: the oracle's hybrid average of this shard
    acc = np.zeros(p.shard_len, dtype=np.float32)
    for g2 in range(G_groups):
        acc = acc + parts[g2]
    ghat = acc * np.float32(1.0 / M)
    master = np.zeros(p.N, dtype=np.float32)
    st = O.init_state(p, 1, master, groups=G_groups)
    O.zero_step(p, st, Gr, O.hyper())
    assert np.array_equal(ghat.view(np.uint32), st.ghat[k][:p.shard_len].view(np.uint32))

    # the all-gather inside the group
    shard = torch.from_numpy(O.bf16_rne(st.master[k][:p.shard_len]).view(np.int16).copy()).view(torch.bfloat16)
    full = torch.zeros(p.npad, dtype=torch.int16).view(torch.bfloat16)
    gather_params(shard, full, buckets, K, pg_intra)
    full_u = full.view(torch.int16).numpy().view(np.uint16)
    u = p.unpadded_index()
    real = u >= 0
    assert np.array_equal(full_u[real][np.argsort(u[real])], st.param[0][:p.N])


@pytest.mark.parametrize("case", ["two_buckets_ragged", "many_buckets"])
def test_sharded_exchange_hybrid_four_ranks(case):
    _spawn(4, case, _hybrid_rank)


def _leaving_rank(rank, world, port, q):
    """Rank 1 leaves between steps (after one exchange, with nothing in flight); rank 0's next
    exchange must end with an error, within the process group's short timeout, not hang."""
    import time

    try:
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        import datetime

        import torch
        import torch.distributed as dist

        import oracle as O
        import zero_gradient_reduce_scatter_gb300 as zg
        from zero_gradient_reduce_scatter_gb300.sharded import exchange_gradients

        dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=5))
        numel, bucket_bytes = CASES["two_buckets_ragged"]
        p = O.plan(numel, world, bucket_bytes)
        _, buckets = zg.layout(numel, world, 1, bucket_bytes)
        g = torch.from_numpy(_grads(p, world, 5)[rank].view(np.int16).copy()).view(torch.bfloat16)
        recv = torch.zeros(p.npad, dtype=torch.int16).view(torch.bfloat16)
        exchange_gradients(g, recv, buckets, world)  # step 1: both ranks
        if rank == 1:
            q.put((rank, "left"))
            q.close()
            q.join_thread()  # the message is out before the process ends
            os._exit(0)  # leaves between steps, without a word to the others
        time.sleep(1.0)
        t0 = time.time()
        try:
            exchange_gradients(g, recv, buckets, world)  # step 2: the peer is gone
            q.put((rank, "completed"))
        except Exception as e:  # detected on the host
            q.put((rank, f"error {type(e).__name__} after {time.time() - t0:.1f}s"))
    except BaseException:
        q.put((rank, traceback.format_exc()))


def test_rank_leaving_between_steps_is_detected():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_leaving_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    assert got[1] == "left"
    assert got[0].startswith("error"), got[0]
    assert float(got[0].split(" after ")[1][:-1]) < 60.0


def _random_layouts_rank(rank, M, case):
    """Five seeded random layouts (sizes 0..5000, some zero, bucket caps from one tensor to
    everything) over M = 3 ranks: the exchange delivers the oracle's operands for this owner
    and the all-gather rebuilds the oracle's parameters."""
    import torch

    import oracle as O
    import zero_gradient_reduce_scatter_gb300 as zg
    from zero_gradient_reduce_scatter_gb300.sharded import exchange_gradients, gather_params

    rng = np.random.default_rng(77)
    for trial in range(5):
        T = int(rng.integers(1, 12))
        numel = tuple(int(x) if rng.random() > 0.15 else 0 for x in rng.integers(1, 5000, T))
        if sum(numel) == 0:
            numel = numel + (7,)
        bucket_bytes = int(rng.choice([0, 64, 2048, 10000]))
        p = O.plan(numel, M, bucket_bytes)
        toff, buckets = zg.layout(numel, M, 1, bucket_bytes)
        assert [int(x) for x in p.t_off] == toff
        G = _grads(p, M, seed=500 + trial)
        mine = torch.from_numpy(G[rank].view(np.int16).copy()).view(torch.bfloat16)
        recv = torch.zeros(p.npad, dtype=torch.int16).view(torch.bfloat16)
        exchange_gradients(mine, recv, buckets, M)
        got = recv.view(torch.int16).numpy().view(np.uint16)
        virt = [np.full(p.npad, BF16_NAN, dtype=np.uint16) for _ in range(M)]
        for b in range(p.nb):
            off, S = int(p.b_off[b]), int(p.b_S[b])
            for src in range(M):
                virt[src][off + rank * S: off + (rank + 1) * S] = got[off + src * S: off + (src + 1) * S]
        want = O.reduce_scatter(p, G)[rank]
        assert np.array_equal(O.reduce_scatter(p, virt)[rank].view(np.uint32), want.view(np.uint32)), trial
        st = O.init_state(p, 3, np.zeros(p.N, np.float32))
        full_want, _, _, _ = O.zero_step(p, st, G, O.hyper())
        shard = torch.from_numpy(st.param[rank][:p.shard_len].view(np.int16).copy()).view(torch.bfloat16)
        full = torch.zeros(p.npad, dtype=torch.int16).view(torch.bfloat16)
        gather_params(shard, full, buckets, M)
        u = p.unpadded_index()
        full_u = full.view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(full_u[u >= 0][np.argsort(u[u >= 0])], full_want), trial


def test_sharded_exchange_random_layouts_three_ranks():
    _spawn(3, None, _random_layouts_rank)
