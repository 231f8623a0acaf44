"""Process-per-rank mode with real processes: two ranks on the one GPU, one process each.

NCCL does not run two ranks on one device, so the ranks exchange through gloo with their
device buffers staged through host memory (ShardedZeroOptimizer(transport="host")). Each
process runs the library's kernels on its own shard only. Three clipped steps on a ragged
multi-bucket layout, at ZeRO-1 (full parameters kept) and ZeRO-3 (per-bucket gathers into a
transient buffer), both forms of the clipped step, flat and hybrid with one rank per group;
and three ZeRO-2 steps streamed bucket by bucket in backward order (step_streamed), unclipped
and clipped, flat and hybrid. Every rank checks itself against the oracle's two-rank step: its shard of
master / m / v (1e-6 relative; bit-identical expected), the averaged gradient bit-exact when
materialized, the norm within 1e-7 and equal on both ranks, the gathered bf16 parameters within
1 ulp. Then the assembled checkpoint state equals the oracle's bit for bit, and both ranks
resume from it in another bucket layout and take one more step as the oracle does, then three
steps fed from pinned host memory (step_host_overlapped).

The ranks wait for each other only on the host (gloo), never inside a kernel.
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
sys.path.insert(0, os.path.join(ROOT, "tests"))

pytestmark = pytest.mark.gpu

NUMEL = (3001, 1000, 37, 4099, 1, 64, 777)
BUCKET_BYTES = 6000


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _grads_all(p, M, k):
    """Every rank's bf16 gradient of step k (uint16 patterns; each process can make all)."""
    import oracle as O
    rng = np.random.default_rng(4242 + k)
    out = []
    for _ in range(M):
        out.append(O.bf16_rne(rng.standard_normal(p.npad).astype(np.float32) * np.float32(3e-3)))
    real = p.real_mask()
    for g in out:
        g[~real] = 0x3F80  # padding garbage: ignored on both sides
    return out


def _rank_main(rank, world, port, stage, ghat_mode, q, streamed=False, groups=1):
    try:
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        import torch
        import torch.distributed as dist

        import oracle as O
        import workloads as W
        import zero_gradient_reduce_scatter_gb300 as zg
        from parity_util import assert_state_close, bf16_ulp_diff, f32, u16
        from rank_util import padded_to_unpadded

        dist.init_process_group("gloo", rank=rank, world_size=world)
        torch.cuda.set_device(0)
        dev = torch.device("cuda", 0)
        w = W.small_variant(W.workload("tiny"), NUMEL, steps=3)
        mi = W.master_init(w, dev)
        opt = zg.ShardedZeroOptimizer(NUMEL, stage, mi, bucket_bytes=BUCKET_BYTES, transport="host",
                                      ghat_buffer=True, groups=groups)
        assert opt.M == world and opt.rank == rank and len(opt.buckets) >= 2
        K = world // groups  # owners per group: the oracle plans for K
        assert opt.identity == (K == 1)
        if opt.identity:  # nothing to exchange, and the full parameters are the shard itself
            assert opt.recv is None and (stage == 3 or opt.params() is opt.param_shards)
        p = O.plan(NUMEL, K, BUCKET_BYTES)
        st = O.init_state(p, stage, f32(mi), groups=groups)
        clip = streamed in (False, "clipped")  # streamed=True: the unclipped streamed form
        h = zg.Hyper(clip=clip, max_grad_norm=0.05, ghat_mode=ghat_mode)
        oh = O.hyper(clip=clip, max_grad_norm=0.05)
        scratch = torch.empty(world * max(b[2] for b in opt.buckets), dtype=torch.bfloat16, device=dev)
        for k in range(3):
            G = _grads_all(p, world, k)
            mine = torch.from_numpy(G[rank].view(np.int16).copy()).to(dev).view(torch.bfloat16)
            if streamed:  # ZeRO-2 bucket streaming, buckets in backward order
                opt.step_streamed(mine, h, order=reversed(range(len(opt.buckets))))
            else:
                opt.step(mine, h)
            full, norm, scale, rc = O.zero_step(p, st, G, oh)
            assert rc == 0 and (scale < 1.0 or not clip)
            assert opt.sync_status() == 0
            if clip:
                gn, gs = opt.last_norm()
                assert abs(gn - norm) <= 1e-7 * norm
                both = torch.tensor([gn, gs], dtype=torch.float64)
                seen = [torch.zeros(2, dtype=torch.float64) for _ in range(world)]
                dist.all_gather(seen, both)
                assert all(torch.equal(x, seen[0]) for x in seen), "both ranks form the same norm and scale"
            assert_state_close(f32(opt.get_state("master")), st.master[rank][:p.shard_len], f"step {k} master")
            assert_state_close(f32(opt.get_state("m")), st.mom[rank][:p.shard_len], f"step {k} m")
            assert_state_close(f32(opt.get_state("v")), st.var[rank][:p.shard_len], f"step {k} v")
            if ghat_mode == "materialize":
                assert np.array_equal(f32(opt.get_state("ghat")).view(np.uint32),
                                      st.ghat[rank][:p.shard_len].view(np.uint32))
            if stage == 3:
                assert opt.params() is None  # ZeRO-3: no persistent full parameters
                assert bf16_ulp_diff(u16(opt.param_shards), st.param[rank][:p.shard_len]) <= 1
                uoffs = np.cumsum([0] + [b[1] for b in opt.buckets])
                for b, (_off, n_b, _S, _) in enumerate(opt.buckets):  # per-module gathers
                    got = opt.gather_bucket(b, scratch)
                    assert bf16_ulp_diff(u16(got), full[uoffs[b]:uoffs[b] + n_b]) <= 1
                seq = list(range(len(opt.buckets)))
                for order in (seq, seq[::-1]):  # forward and backward sweeps with prefetch
                    for b, got in opt.prefetched_buckets(order, buffers=2 + k):
                        assert bf16_ulp_diff(u16(got), full[uoffs[b]:uoffs[b] + opt.buckets[b][1]]) <= 1
            else:
                assert bf16_ulp_diff(padded_to_unpadded(p, u16(opt.params())), full) <= 1
        state = opt.save_state()
        u = p.unpadded_index()
        real = u >= 0
        for name, attr in (("master", "master"), ("m", "mom"), ("v", "var")):
            flat = O.flat_state(p, st, attr)
            want = np.empty(p.N, dtype=np.float32)
            want[u[real]] = flat[real]
            assert np.array_equal(f32(state[name]).view(np.uint32), want.view(np.uint32)), name
        assert state["t"] == 3
        # resume from the checkpoint in another layout (one bucket) and take one more step
        sd = opt.state_dict()
        opt.close()
        opt2 = zg.ShardedZeroOptimizer(NUMEL, stage, mi, bucket_bytes=0, transport="host", ghat_buffer=True,
                                       groups=groups)
        opt2.load_state_dict(sd)
        assert opt2.t == 3
        p2 = O.plan(NUMEL, K, 0)
        st2 = O.init_state(p2, stage, sd["master"].numpy(), sd["m"].numpy(), sd["v"].numpy(), t=3, groups=groups)
        G = _grads_all(p2, world, 9)
        mine = torch.from_numpy(G[rank].view(np.int16).copy()).to(dev).view(torch.bfloat16)
        opt2.step(mine, h)
        O.zero_step(p2, st2, G, oh)
        assert_state_close(f32(opt2.get_state("master")), st2.master[rank][:p2.shard_len], "resumed master")
        assert_state_close(f32(opt2.get_state("v")), st2.var[rank][:p2.shard_len], "resumed v")
        _host_fed_steps(opt2, p2, st2, world, rank, h, oh, dev, range(10, 13))
        opt2.close()
        dist.destroy_process_group()
        q.put((rank, "ok"))
    except BaseException:
        q.put((rank, traceback.format_exc()))


def _host_fed_steps(opt, p, st, world, rank, h, oh, dev, steps):
    """Steps from pinned host gradients (step_host_overlapped, two device buffers in turn, a
    copy stream), issued with no synchronisation in between, then checked against the oracle:
    the state, and the parameters copied back to host memory after the last step."""
    import torch

    import oracle as O
    from parity_util import assert_state_close, bf16_ulp_diff, f32, u16
    from rank_util import padded_to_unpadded

    bufs = [opt.new_grad_buffer(), opt.new_grad_buffer()]
    cs = torch.cuda.Stream(device=dev)
    keep = opt.param_full is not None
    host_p = torch.empty(p.npad, dtype=torch.bfloat16).pin_memory() if keep else None
    hgs = []
    for i, k in enumerate(steps):
        G = _grads_all(p, world, k)
        hgs.append(torch.from_numpy(G[rank].view(np.int16).copy()).view(torch.bfloat16).pin_memory())
        opt.step_host_overlapped(hgs[-1], bufs[i % 2], host_p, h, cs)
        full, _norm, _scale, rc = O.zero_step(p, st, G, oh)
        assert rc == 0
    if keep:  # the parameters reach the host on a stream of their own
        opt.params_copied.synchronize()
        assert bf16_ulp_diff(padded_to_unpadded(p, u16(host_p)), full) <= 1
    torch.cuda.synchronize()
    assert opt.sync_status() == 0
    assert_state_close(f32(opt.get_state("master")), st.master[rank][:p.shard_len], "host-fed master")
    assert_state_close(f32(opt.get_state("m")), st.mom[rank][:p.shard_len], "host-fed m")
    assert_state_close(f32(opt.get_state("v")), st.var[rank][:p.shard_len], "host-fed v")


@pytest.mark.parametrize("stage,ghat_mode,streamed,groups", [(1, "materialize", False, 1), (3, "recompute", False, 1),
                                                             (3, "materialize", False, 1), (2, "auto", True, 1),
                                                             (2, "materialize", "clipped", 1),
                                                             (1, "materialize", False, 2), (3, "recompute", False, 2),
                                                             (2, "auto", True, 2), (2, "materialize", "clipped", 2)])
def test_two_processes_on_one_gpu(stage, ghat_mode, streamed, groups):
    """groups=2: hybrid sharding with one rank per group (a replicated state whose exchange and
    all-gather are identities; the group partials still cross the process boundary)."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, stage, ghat_mode, q, streamed, groups))
             for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=600) for _ in procs)
    for p in procs:
        p.join(timeout=120)
    bad = {r: v for r, v in got.items() if v != "ok"}
    assert not bad, "\n".join(f"rank {r}:\n{v}" for r, v in bad.items())
    assert all(p.exitcode == 0 for p in procs)


def _nccl_one_rank(q, coalesce, identity):
    """A job of one rank over NCCL (the only NCCL job one GPU can hold): clipped steps,
    unclipped streamed ones and clipped streamed ones in turn, and a prefetched per-bucket
    sweep after each, against the oracle's one-rank step. identity: the exchange and the
    all-gather of one rank are skipped (the kernels read the gradient in place, the parameters
    are the shard itself); otherwise they run as NCCL collectives, grouped per step or one
    call per bucket (coalesce)."""
    try:
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(free_port()))
        import torch
        import torch.distributed as dist

        import oracle as O
        import workloads as W
        import zero_gradient_reduce_scatter_gb300 as zg
        from parity_util import assert_state_close, bf16_ulp_diff, f32, u16
        from rank_util import padded_to_unpadded

        torch.cuda.set_device(0)
        dev = torch.device("cuda", 0)
        dist.init_process_group("nccl", rank=0, world_size=1, device_id=dev)
        w = W.small_variant(W.workload("tiny"), NUMEL, steps=3)
        mi = W.master_init(w, dev)
        opt = zg.ShardedZeroOptimizer(NUMEL, 2, mi, bucket_bytes=BUCKET_BYTES, coalesce=coalesce, full_params=True,
                                      ghat_buffer=True, skip_identity=identity)
        assert opt.M == 1 and len(opt.buckets) >= 2
        assert opt.identity == identity
        assert (opt.recv is None and opt.params() is opt.param_shards) == identity
        p = O.plan(NUMEL, 1, BUCKET_BYTES)
        st = O.init_state(p, 2, f32(mi))
        for k in range(9):
            form = k % 3  # 0: clipped step, 1: unclipped streamed, 2: clipped streamed
            clip = form != 1
            G = _grads_all(p, 1, k)
            mine = torch.from_numpy(G[0].view(np.int16).copy()).to(dev).view(torch.bfloat16)
            h = zg.Hyper(clip=clip, max_grad_norm=0.05)
            if form == 0:
                opt.step(mine, h)
            else:
                opt.step_streamed(mine, h, order=reversed(range(len(opt.buckets))))
            full, norm, scale, rc = O.zero_step(p, st, G, O.hyper(clip=clip, max_grad_norm=0.05))
            assert rc == 0 and (scale < 1.0 or not clip)
            if clip:
                gn, _gs = opt.last_norm()
                assert abs(gn - norm) <= 1e-7 * norm
            assert_state_close(f32(opt.get_state("master")), st.master[0][:p.shard_len], f"step {k} master")
            assert_state_close(f32(opt.get_state("m")), st.mom[0][:p.shard_len], f"step {k} m")
            assert_state_close(f32(opt.get_state("v")), st.var[0][:p.shard_len], f"step {k} v")
            if form == 2:  # the clipped streamed step keeps the average: bit-exact
                assert np.array_equal(f32(opt.get_state("ghat")).view(np.uint32),
                                      st.ghat[0][:p.shard_len].view(np.uint32))
            assert bf16_ulp_diff(padded_to_unpadded(p, u16(opt.params())), full) <= 1
            uoffs = np.cumsum([0] + [b[1] for b in opt.buckets])
            for b, got in opt.prefetched_buckets(reversed(range(len(opt.buckets))), buffers=3):
                assert bf16_ulp_diff(u16(got), full[uoffs[b]:uoffs[b] + opt.buckets[b][1]]) <= 1
        _host_fed_steps(opt, p, st, 1, 0, zg.Hyper(clip=True, max_grad_norm=0.05),
                        O.hyper(clip=True, max_grad_norm=0.05), dev, range(20, 23))
        # argument errors of the host-fed step, each refused before anything is enqueued
        hg = torch.zeros(p.npad, dtype=torch.bfloat16).pin_memory()
        hp = torch.zeros(p.npad, dtype=torch.bfloat16).pin_memory()
        dg = opt.new_grad_buffer()
        cs = torch.cuda.Stream()
        bad = [(hg.to(dev), dg, hp, cs),                                   # gradient not on the host
               (hg[:-1], dg, hp, cs),                                      # wrong length
               (hg.float(), dg, hp, cs),                                   # wrong type
               (hg, dg, hp[:-1], cs),                                      # parameters of the wrong length
               (hg, dg.float(), hp, cs),                                   # device buffer of the wrong type
               (hg, dg, hp, torch.cuda.current_stream())]                  # copy stream = current stream
        t0 = opt.t
        for args in bad:
            try:
                opt.step_host_overlapped(args[0], args[1], args[2], zg.Hyper(), args[3])
            except ValueError:
                continue
            raise AssertionError("accepted a bad argument")
        assert opt.t == t0
        opt.close()
        dist.destroy_process_group()
        q.put("ok")
    except BaseException:
        q.put(traceback.format_exc())


@pytest.mark.parametrize("coalesce,identity", [(True, True), (True, False), (False, False)])
def test_nccl_one_rank_job(coalesce, identity):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    proc = ctx.Process(target=_nccl_one_rank, args=(q, coalesce, identity))
    proc.start()
    got = q.get(timeout=600)
    proc.join(timeout=120)
    assert got == "ok", got
    assert proc.exitcode == 0
