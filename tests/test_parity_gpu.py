"""GPU vs oracle, element by element, at sizes the oracle finishes in seconds that still
span many CTAs' tiles, several buckets and ragged tails. Every test calls the CUDA path
through the C ABI (libzero_gb300.so)."""
import math

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
import zero_gradient_reduce_scatter_gb300 as zg
from parity_util import (bf16_ulp_diff, f32, make_hyper, run_elementwise, state_errors, u16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    yield


def gpt_like(d, layers, layernorm=True, vocab=1000):
    sizes = [vocab * d]
    for _ in range(layers):
        if layernorm:
            sizes += [d, d]
        sizes += [3 * d * d, d * d]
        if layernorm:
            sizes += [d, d]
        sizes += [4 * d * d, 4 * d * d]
    if layernorm:
        sizes += [d, d]
    return tuple(sizes)


def ragged(count, lo, hi, seed):
    return W.ragged_numel(count, lo, hi, seed)


# ------------------------------------------------------------------------------------------
# The five workloads' recipes at reduced sizes (and the tiny one at full size)
# ------------------------------------------------------------------------------------------
def test_tiny_workload_full_size():
    out = run_elementwise(W.workload("tiny"))
    assert out["bf16_ulp"] == 0 and out["state_err"] == 0.0


def test_gpt2_small_recipe_multi_bucket_stage2():
    w = W.small_variant(W.workload("gpt2s"), gpt_like(100, 3), bucket_bytes=150_000, steps=4)
    p = O.plan(w.numel, w.M, w.bucket_bytes)
    assert p.nb >= 5
    out = run_elementwise(w)
    assert out["bf16_ulp"] == 0 and out["state_err"] == 0.0


def test_ragged_multi_bucket_fused_epilogue_all_alignments():
    """Odd tensor sizes and small buckets: the unpadded start of the buckets falls on every
    alignment class of the fused all-gather stores (16-, 8-, 4- and 2-byte)."""
    w = W.small_variant(W.workload("gpt2s"), ragged(60, 50, 4000, 11), bucket_bytes=9000, steps=3, clip=1.0)
    p = O.plan(w.numel, w.M, w.bucket_bytes)
    shifts = {int(p.b_off[b] - sum(p.b_n[:b])) % 8 for b in range(p.nb)}
    assert 0 in shifts and 4 in shifts and (shifts & {2, 6}) and (shifts & {1, 3, 5, 7}), shifts
    for mode in ("materialize", "recompute"):
        out = run_elementwise(w, ghat_mode=mode, ghat_buffer=True)
        assert out["bf16_ulp"] == 0 and out["state_err"] == 0.0


@pytest.mark.parametrize("ghat_mode", ["materialize", "recompute"])
def test_dense_1p3b_recipe_clip_stage1(ghat_mode):
    w = W.small_variant(W.workload("1p3b"), gpt_like(128, 2, layernorm=False, vocab=2000), steps=3)
    out = run_elementwise(w, ghat_mode=ghat_mode, ghat_buffer=True)
    assert out["bf16_ulp"] == 0 and out["state_err"] == 0.0
    if ghat_mode == "materialize":
        # the reduce-scatter result is bit-exact
        p, st, opt = out["plan"], out["oracle_state"], out["opt"]
        got = f32(opt.ghat)
        want = O.flat_state(p, st, "ghat")
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("gather", ["shards", "fused"])
def test_ragged_recipe_stage3_m16(gather):
    w = W.small_variant(W.workload("ragged"), ragged(150, 2 ** 10, 2 ** 15, 7), steps=3)
    out = run_elementwise(w, gather=gather)
    assert out["bf16_ulp"] == 0 and out["state_err"] == 0.0


def test_dense_4b_recipe_stage3_m4():
    w = W.small_variant(W.workload("4b"), gpt_like(160, 2, layernorm=False, vocab=1500), steps=3)
    out = run_elementwise(w)
    assert out["bf16_ulp"] == 0 and out["state_err"] == 0.0


# ------------------------------------------------------------------------------------------
# Edge cases
# ------------------------------------------------------------------------------------------
@pytest.mark.parametrize("M", [1, 3, 5, 7, 16, 64])
def test_rank_counts_including_generic_kernel(M):
    """M outside {1,2,4,8,16} runs the generic rank loop; non-power-of-two M makes
    (float)(1/M) inexact, which both sides apply the same way."""
    w = W.small_variant(W.workload("ragged"), (3001, 17, 8192, 1, 555), M=M, steps=2)
    out = run_elementwise(w, gather="shards")
    assert out["bf16_ulp"] == 0 and out["state_err"] == 0.0


def test_fewer_params_than_ranks():
    """3 real lanes over 16 ranks: 15 owners hold only padding."""
    w = W.small_variant(W.workload("ragged"), (3,), steps=3)
    out = run_elementwise(w, gather="shards")
    assert out["bf16_ulp"] == 0 and out["state_err"] == 0.0


def test_zero_size_and_unit_tensors():
    w = W.small_variant(W.workload("gpt2s"), (0, 1, 0, 1, 2, 0, 5000, 1), bucket_bytes=40, steps=2)
    out = run_elementwise(w)
    assert out["bf16_ulp"] == 0 and out["state_err"] == 0.0


def test_padding_garbage_is_ignored():
    w = W.small_variant(W.workload("4b"), (1001, 77, 3), steps=2)
    out = run_elementwise(w, garbage_in_padding=True)
    assert out["bf16_ulp"] == 0 and out["state_err"] == 0.0
    # padding lanes of the state stay exactly zero
    opt, p = out["opt"], out["plan"]
    pad = ~p.real_mask()
    for buf in (opt.master, opt.m, opt.v):
        assert np.all(f32(buf)[pad] == 0.0)


def test_large_threshold_equals_no_clip():
    w_clip = W.small_variant(W.workload("1p3b"), (20000, 3000), clip=1e9, steps=2)
    w_off = W.small_variant(W.workload("1p3b"), (20000, 3000), clip=None, steps=2)
    a = run_elementwise(w_clip)["opt"]
    b = run_elementwise(w_off)["opt"]
    assert a.last_norm()[1] == 1.0
    assert torch.equal(a.master, b.master) and torch.equal(a.params(), b.params())


def test_nonfinite_gradient_skips_step_and_reports():
    w = W.small_variant(W.workload("4b"), (4096, 100), steps=1)
    dev = torch.device("cuda")
    opt = zg.ZeroOptimizer(w.numel, w.M, w.stage, W.master_init(w, dev))
    before = opt.master.clone()
    grads = opt.new_grad_buffers()
    for r in range(w.M):
        W.fill_grads(w, r, 0, grads[r], opt.tensor_offsets)
    grads[2].view(torch.int16)[opt.tensor_offsets[1] + 5] = 0x7F80  # +inf on rank 2
    h, _ = make_hyper(w)
    opt.step(grads, h)
    assert opt.sync_status() == zg.ZERO_ERR_NONFINITE
    assert not math.isfinite(opt.last_norm()[0])
    assert torch.equal(opt.master, before)
    # the next finite step proceeds
    grads[2].view(torch.int16)[opt.tensor_offsets[1] + 5] = 0
    opt.step(grads, h)
    assert opt.sync_status() == 0 and not torch.equal(opt.master, before)


def test_deterministic_rerun():
    w = W.small_variant(W.workload("1p3b"), gpt_like(64, 2, layernorm=False, vocab=3000), steps=2)
    a = run_elementwise(w)
    b = run_elementwise(w)
    assert a["opt"].last_norm() == b["opt"].last_norm()
    assert torch.equal(a["opt"].master, b["opt"].master)


def test_invalid_step_arguments_rejected_on_host():
    w = W.small_variant(W.workload("tiny"), (4096,), steps=1)
    opt = zg.ZeroOptimizer(w.numel, w.M, w.stage, W.master_init(w, torch.device("cuda")))
    grads = opt.new_grad_buffers()
    h, _ = make_hyper(w)
    with pytest.raises(zg.ZeroError) as e:
        opt.step(grads, h, stage=3)
    assert e.value.code == -4
    for bad in (zg.Hyper(lr=-1.0), zg.Hyper(beta1=1.0), zg.Hyper(eps=0.0), zg.Hyper(clip=True, max_grad_norm=0.0)):
        with pytest.raises(zg.ZeroError) as e:
            opt.step(grads, bad)
        assert e.value.code == -1
    # misaligned gradient pointer
    shifted = torch.zeros(opt.sizes["npad"] + 1, dtype=torch.bfloat16, device="cuda")[1:]
    with pytest.raises(zg.ZeroError) as e:
        opt.step([grads[0], shifted], h)
    assert e.value.code == -2
    # use after destroy
    import ctypes
    raw = ctypes.c_void_p(opt._ctx.value)
    opt.close()
    lib = zg._lib()
    assert lib.zero_step(raw, ctypes.cast(opt._grad_ptrs, ctypes.c_void_p), 1, ctypes.byref(h), None) == -7
    assert lib.zero_destroy(raw) == -7


def test_host_memory_pointers_refused():
    """Host memory, pinned or pageable, where a call wants this GPU's memory (a gradient, a
    state output or input) is refused with INVALID_ARG before anything is enqueued, and the
    context keeps working."""
    import ctypes
    w = W.small_variant(W.workload("tiny"), (4096,), steps=1)
    opt = zg.ZeroOptimizer(w.numel, w.M, w.stage, W.master_init(w, torch.device("cuda")))
    grads = opt.new_grad_buffers()
    h, _ = make_hyper(w)
    t0 = opt.t
    lib, s = zg._lib(), zg._stream_handle(None)
    for host in (torch.zeros(opt.sizes["npad"], dtype=torch.bfloat16).pin_memory(),
                 torch.zeros(opt.sizes["npad"], dtype=torch.bfloat16)):
        with pytest.raises(ValueError):  # the binding refuses it first
            opt.step([grads[0], host], h)
        ptrs = (ctypes.c_void_p * w.M)(grads[0].data_ptr(), host.data_ptr())
        assert lib.zero_step(opt._ctx, ctypes.cast(ptrs, ctypes.c_void_p), w.stage, ctypes.byref(h), s) == -1
    out = torch.zeros(opt.sizes["n"], dtype=torch.float32).pin_memory()
    assert lib.zero_save_state(opt._ctx, out.data_ptr(), None, None, s) == -1
    assert lib.zero_load_state(opt._ctx, out.data_ptr(), None, None, 0, s) == -1
    assert lib.zero_get_state(opt._ctx, 0, 0, out.data_ptr(), s) == -1
    bufs = (ctypes.c_void_p * w.M)(grads[0].data_ptr(), out.data_ptr())
    assert lib.zero_step_host(opt._ctx, ctypes.cast(bufs, ctypes.c_void_p), ctypes.cast(bufs, ctypes.c_void_p),
                              w.stage, ctypes.byref(h), out.data_ptr(), s) == -1
    opt.step(grads, h)
    torch.cuda.synchronize()
    assert opt.t == t0 + 1 and opt.sync_status() == 0
    opt.close()


# ------------------------------------------------------------------------------------------
# Other entry points: per-rank state, per-bucket gather, host-buffer step, step counter
# ------------------------------------------------------------------------------------------
def test_get_state_per_rank_matches_oracle_shards():
    w = W.small_variant(W.workload("1p3b"), (5000, 123, 9000), bucket_bytes=12000, steps=2)
    out = run_elementwise(w, ghat_mode="materialize", ghat_buffer=True)
    opt, st = out["opt"], out["oracle_state"]
    for r in range(w.M):
        for name, arr in (("master", st.master), ("m", st.mom), ("v", st.var), ("ghat", st.ghat)):
            got = f32(opt.get_state(name, r))
            assert np.array_equal(got.view(np.uint32), arr[r][:out["plan"].shard_len].view(np.uint32)), (name, r)


def test_gather_per_bucket_rebuilds_params():
    w = W.small_variant(W.workload("ragged"), ragged(40, 100, 3000, 3), bucket_bytes=8000, steps=2)
    out = run_elementwise(w, gather="shards")
    opt, p = out["opt"], out["plan"]
    assert p.nb > 3
    dst = torch.full((p.N,), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    for b in range(p.nb):
        opt.gather_params(b, dst)
    torch.cuda.synchronize()
    assert np.array_equal(u16(dst), u16(opt.params()))


def test_step_from_host_buffers_equals_device_step():
    w = W.small_variant(W.workload("4b"), (70000, 13), steps=2)
    dev = torch.device("cuda")
    a = zg.ZeroOptimizer(w.numel, w.M, w.stage, W.master_init(w, dev))
    b = zg.ZeroOptimizer(w.numel, w.M, w.stage, W.master_init(w, dev))
    h, _ = make_hyper(w)
    dev_grads = a.new_grad_buffers()
    host_params = torch.empty(a.sizes["n"], dtype=torch.bfloat16).pin_memory()
    for k in range(w.steps):
        grads = b.new_grad_buffers()
        for r in range(w.M):
            W.fill_grads(w, r, k, grads[r], b.tensor_offsets)
        host = [g.cpu().pin_memory() for g in grads]
        b.step(grads, h)
        a.step_host(host, dev_grads, host_params, h)
        torch.cuda.synchronize()
        assert torch.equal(host_params, b.params().cpu())
        assert torch.equal(a.master, b.master)


def test_overlapped_host_steps_equal_device_steps():
    """Four steps with different gradients, two alternating device buffer sets and no
    synchronisation between calls: each step's parameters (copied to their own pinned host
    buffer) equal those of the plain device path."""
    w = W.small_variant(W.workload("4b"), (300000, 77, 4099), steps=4)
    dev = torch.device("cuda")
    a = zg.ZeroOptimizer(w.numel, w.M, w.stage, W.master_init(w, dev))
    b = zg.ZeroOptimizer(w.numel, w.M, w.stage, W.master_init(w, dev))
    h, _ = make_hyper(w)
    sig = W.sigmas(w)
    sets = [a.new_grad_buffers(), a.new_grad_buffers()]
    hosts, outs, refs = [], [], []
    for k in range(w.steps):
        grads = b.new_grad_buffers()
        for r in range(w.M):
            W.fill_grads(w, r, k, grads[r], b.tensor_offsets, sig)
        b.step(grads, h)
        refs.append(b.params().clone())
        hosts.append([g.cpu().pin_memory() for g in grads])
        outs.append(torch.empty(a.sizes["n"], dtype=torch.bfloat16).pin_memory())
    torch.cuda.synchronize()
    copy_stream = torch.cuda.Stream()
    for k in range(w.steps):
        a.step_host_overlapped(hosts[k], sets[k % 2], outs[k], h, copy_stream)
    torch.cuda.synchronize()
    for k in range(w.steps):
        assert torch.equal(outs[k], refs[k].cpu()), k
    assert torch.equal(a.master, b.master)


def test_overlapped_host_steps_forget_finished_sets():
    """Ten distinct device gradient sets, one per step, all kept alive (distinct addresses):
    a set whose step has finished is forgotten when a new set needs the room, so the ninth
    and tenth are accepted, and every step's parameters equal the device path's."""
    w = W.small_variant(W.workload("4b"), (5000, 77, 130), steps=10)
    dev = torch.device("cuda")
    a = zg.ZeroOptimizer(w.numel, w.M, w.stage, W.master_init(w, dev))
    b = zg.ZeroOptimizer(w.numel, w.M, w.stage, W.master_init(w, dev))
    h, _ = make_hyper(w)
    sig = W.sigmas(w)
    sets = [a.new_grad_buffers() for _ in range(w.steps)]
    copy_stream = torch.cuda.Stream()
    out = torch.empty(a.sizes["n"], dtype=torch.bfloat16).pin_memory()
    for k in range(w.steps):
        grads = b.new_grad_buffers()
        for r in range(w.M):
            W.fill_grads(w, r, k, grads[r], b.tensor_offsets, sig)
        b.step(grads, h)
        host = [g.cpu().pin_memory() for g in grads]
        a.step_host_overlapped(host, sets[k], out, h, copy_stream)
        torch.cuda.synchronize()
        assert torch.equal(out, b.params().cpu()), k
    assert torch.equal(a.master, b.master)


def test_step_counter_and_resume():
    """K steps == K1 steps, save (state + t), restore into a fresh context, K2 steps."""
    w = W.small_variant(W.workload("1p3b"), (30000, 5000), steps=4)
    dev = torch.device("cuda")
    h, _ = make_hyper(w)
    sig = W.sigmas(w)

    def grads_for(opt, k):
        gs = opt.new_grad_buffers()
        for r in range(w.M):
            W.fill_grads(w, r, k, gs[r], opt.tensor_offsets, sig)
        return gs

    ref = zg.ZeroOptimizer(w.numel, w.M, w.stage, W.master_init(w, dev))
    for k in range(4):
        ref.step(grads_for(ref, k), h)
    first = zg.ZeroOptimizer(w.numel, w.M, w.stage, W.master_init(w, dev))
    for k in range(2):
        first.step(grads_for(first, k), h)
    saved = (first.master.clone(), first.m.clone(), first.v.clone(), first.t)
    resumed = zg.ZeroOptimizer(w.numel, w.M, w.stage, W.master_init(w, dev))
    resumed.master.copy_(saved[0]), resumed.m.copy_(saved[1]), resumed.v.copy_(saved[2])
    resumed.t = saved[3]
    assert resumed.t == 2
    for k in range(2, 4):
        resumed.step(grads_for(resumed, k), h)
    torch.cuda.synchronize()
    assert torch.equal(resumed.master, ref.master) and torch.equal(resumed.params(), ref.params())


def test_kernel_timing_counts_launches():
    w = W.small_variant(W.workload("1p3b"), (200000,), steps=1)
    opt = zg.ZeroOptimizer(w.numel, w.M, w.stage, W.master_init(w, torch.device("cuda")), ghat_buffer=True)
    grads = opt.new_grad_buffers()
    h, _ = make_hyper(w)
    opt.set_timing(True)
    for _ in range(3):
        opt.step(grads, h)
    t = opt.kernel_times()
    assert t["rs_norm"][1] == 3 and t["norm_final"][1] == 3 and t["adamw"][1] == 3 and t["rs_adamw"][1] == 0
    assert all(v[0] > 0 for k, v in t.items() if v[1])


# ------------------------------------------------------------------------------------------
# Guard bands: no kernel writes outside the buffers it was given
# ------------------------------------------------------------------------------------------
GUARD = 4096


def _guarded(nbytes, dev):
    raw = torch.full((GUARD + nbytes + GUARD,), 0xA5, dtype=torch.uint8, device=dev)
    return raw, raw[GUARD:GUARD + nbytes]


@pytest.mark.parametrize("gather,mode", [("shards", "materialize"), ("fused", "recompute"), ("fused", "materialize")])
def test_guard_bands_untouched(gather, mode):
    import ctypes
    w = W.small_variant(W.workload("ragged"), ragged(30, 100, 5000, 9), M=8, bucket_bytes=20000, steps=2)
    dev = torch.device("cuda")
    s = zg.plan(w.numel, w.M, w.stage, w.bucket_bytes, gather)
    toff, _ = zg.layout(w.numel, w.M, w.stage, w.bucket_bytes, gather)
    raws, views = {}, {}
    for name, nbytes in (("master", s["bytes_master"]), ("m", s["bytes_m"]), ("v", s["bytes_v"]),
                         ("ghat", s["bytes_ghat"]), ("param_full", s["bytes_param_full"]),
                         ("param_shards", s["bytes_param_shards"]), ("scratch", s["bytes_scratch"])):
        if nbytes:
            raws[name], views[name] = _guarded(nbytes, dev)
    grads = []
    for r in range(w.M):
        raws[f"g{r}"], gv = _guarded(s["bytes_grad_each"], dev)
        gv.zero_()
        g = gv.view(torch.bfloat16)
        W.fill_grads(w, r, 0, g, toff)
        grads.append(g)
    mi_raw, mi = _guarded(4 * s["n"], dev)
    mi.view(torch.float32).copy_(W.master_init(w, dev))
    bufs = zg.Buffers(*[views[k].data_ptr() if k in views else None
                        for k in ("master", "m", "v", "ghat", "param_full", "param_shards", "scratch")])
    cfg = zg.Config(w.M, w.stage, w.bucket_bytes, zg.GATHER[gather], 0)
    arr = (ctypes.c_int64 * len(w.numel))(*w.numel)
    ctx = ctypes.c_void_p()
    lib = zg._lib()
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.zero_init(ctypes.byref(ctx), ctypes.byref(cfg), ctypes.cast(arr, ctypes.c_void_p), len(w.numel),
                         ctypes.byref(bufs), mi.data_ptr(), stream) == 0
    h, _ = make_hyper(w, mode)
    ptrs = (ctypes.c_void_p * w.M)(*[g.data_ptr() for g in grads])
    for _ in range(w.steps):
        assert lib.zero_step(ctx, ctypes.cast(ptrs, ctypes.c_void_p), w.stage, ctypes.byref(h), stream) == 0
    if gather == "shards":
        assert lib.zero_gather(ctx, 1, None, stream) == 0
    assert lib.zero_sync_status(ctx) == 0
    torch.cuda.synchronize()
    for name, raw in list(raws.items()) + [("master_init", mi_raw)]:
        assert bool((raw[:GUARD] == 0xA5).all()) and bool((raw[-GUARD:] == 0xA5).all()), f"guard band of {name} hit"
    assert lib.zero_destroy(ctx) == 0


# ------------------------------------------------------------------------------------------
# Hybrid sharding ("CS231n Lecture 11" 4.4): M = G x K, state sharded over K, replicated over G
# ------------------------------------------------------------------------------------------
@pytest.mark.parametrize("G,K,stage,gather,bucket_bytes,clip", [
    (2, 4, 3, "shards", 0, 1.0), (4, 2, 1, "fused", 40000, 1.0), (3, 2, 2, "fused", 0, None),
    (2, 8, 3, "fused", 0, 1.0), (8, 1, 1, "fused", 0, 1.0)])
def test_hybrid_sharding_matches_oracle(G, K, stage, gather, bucket_bytes, clip):
    w = W.small_variant(W.workload("ragged"), ragged(40, 200, 6000, 23), M=G * K, stage=stage,
                        bucket_bytes=bucket_bytes, clip=clip, steps=3)
    for mode in (("materialize", "recompute") if clip else ("auto",)):
        out = run_elementwise(w, gather=gather, groups=G, ghat_mode=mode, ghat_buffer=True)
        assert out["bf16_ulp"] == 0 and out["state_err"] == 0.0


# ------------------------------------------------------------------------------------------
# Odd grids: the grid-stride loops and bucket cursors must not depend on the grid
# ------------------------------------------------------------------------------------------
@pytest.mark.parametrize("clip", [None, 1e-3])
def test_results_do_not_depend_on_the_grid(clip):
    w = W.small_variant(W.workload("gpt2s"), ragged(50, 100, 30000, 29), bucket_bytes=60000, steps=2, clip=clip)
    dev = torch.device("cuda")
    sig = W.sigmas(w)
    grads_per_step = []
    ref = None
    for cap in (0, 1, 7, 13, 151):
        for gather in ("fused", "shards"):
            stage = 3 if gather == "shards" else 2
            opt = zg.ZeroOptimizer(w.numel, w.M, stage, W.master_init(w, dev), bucket_bytes=w.bucket_bytes,
                                   gather=gather, ghat_buffer=True)
            opt.set_max_ctas(cap)
            h, _ = make_hyper(w)
            for k in range(w.steps):
                if len(grads_per_step) <= k:
                    g = opt.new_grad_buffers()
                    for r in range(w.M):
                        W.fill_grads(w, r, k, g[r], opt.tensor_offsets, sig)
                    grads_per_step.append(g)
                opt.step(grads_per_step[k], h)
            assert opt.sync_status() == 0
            got = (f32(opt.master), f32(opt.m), f32(opt.v), u16(opt.params()))
            if ref is None:
                ref = got
                continue
            if clip is None:  # nothing depends on the grid
                for a, b in zip(got, ref):
                    assert np.array_equal(a.view(np.uint32 if a.dtype == np.float32 else np.uint16),
                                          b.view(np.uint32 if b.dtype == np.float32 else np.uint16)), (cap, gather)
            else:  # only the norm's summation order does
                for a, b in zip(got[:3], ref[:3]):
                    assert state_errors(a, b) <= 1.0, (cap, gather)
                assert bf16_ulp_diff(got[3], ref[3]) <= 1


def test_default_stream_handle_is_the_current_stream():
    """Calls without a stream argument enqueue on torch's current stream: the binding's fast
    handle lookup equals torch.cuda.current_stream() outside and inside a stream context,
    and on a second device index when there is one."""
    dev = torch.device("cuda")
    assert zg._stream_handle(None) == torch.cuda.current_stream(dev).cuda_stream
    s = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(s):
        assert zg._stream_handle(None) == s.cuda_stream == torch.cuda.current_stream().cuda_stream
    assert zg._stream_handle(None) == torch.cuda.current_stream(dev).cuda_stream
    assert zg._stream_handle(s) == s.cuda_stream
