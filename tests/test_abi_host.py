"""Host-only checks of the C ABI (no GPU): the library loads and exports every function
include/zero_gb300.h declares; the planner agrees with the oracle's planner; invalid
arguments are rejected with the documented codes; the state-ledger helper reproduces the
figures printed on the pages."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle as O
import workloads as W
from zero_gradient_reduce_scatter_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "zero_gb300.h")


@pytest.fixture(scope="module")
def zg():
    _build.build()
    import zero_gradient_reduce_scatter_gb300 as zg
    zg._lib()
    return zg


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(zero_\w+)\s*\(", text)))


def test_library_exports_every_declared_function(zg):
    names = declared_functions()
    assert len(names) >= 19
    lib = ctypes.CDLL(zg.library_path())
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, f"not exported: {missing}"
    # the binding declares a signature for each of them
    assert sorted(zg.SIGNATURES) == names


def test_release_build_is_not_the_checked_build(zg):
    assert zg._lib().zero_checked_build() == 0


def test_error_strings(zg):
    for code in [0, -1, -2, -3, -4, -5, -6, -7, -8, -9, -10, -11, -99]:
        assert zg._lib().zero_strerror(code)


def _cmp_with_oracle(zg, numel, M, stage, bucket_bytes):
    sizes = zg.plan(numel, M, stage, bucket_bytes)
    toff, buckets = zg.layout(numel, M, stage, bucket_bytes)
    p = O.plan(numel, M, bucket_bytes, 64)
    assert sizes["npad"] == p.npad and sizes["n"] == p.N and sizes["shard_len"] == p.shard_len
    assert sizes["n_buckets"] == p.nb
    assert toff == [int(x) for x in p.t_off]
    assert [b[0] for b in buckets] == list(p.b_off)
    assert [b[1] for b in buckets] == list(p.b_n)
    assert [b[2] for b in buckets] == list(p.b_S)
    assert [b[3] for b in buckets] == list(p.b_first[:-1])
    assert sizes["bytes_grad_each"] == 2 * p.npad and sizes["bytes_param_full"] == 2 * p.N


def test_hybrid_sharding_plans_for_the_group_size(zg):
    # M = 8 ranks in 2 groups: the layout is the one of 4 owners
    for numel, bb in (([1000, 33, 4097], 0), ([300] * 9, 1500)):
        assert zg.plan(numel, 8, 2, bb, groups=2) == zg.plan(numel, 4, 2, bb)
        assert zg.layout(numel, 8, 3, bb, "shards", groups=2) == zg.layout(numel, 4, 3, bb, "shards")


def test_planner_matches_oracle_random(zg):
    rng = np.random.default_rng(21)
    for _ in range(300):
        T = int(rng.integers(1, 12))
        numel = [int(v) for v in rng.integers(0, 5000, size=T)]
        if sum(numel) == 0:
            numel[0] = 1
        M = int(rng.integers(1, 65))
        bb = int(rng.choice([0, 100, 2000, 10000, 65536]))
        _cmp_with_oracle(zg, numel, M, int(rng.integers(1, 4)), bb)


@pytest.mark.parametrize("key", ["tiny", "gpt2s", "1p3b", "ragged", "4b"])
def test_planner_matches_oracle_on_workloads(zg, key):
    w = W.workload(key)
    _cmp_with_oracle(zg, list(w.numel), w.M, w.stage, w.bucket_bytes)


def test_workload_sizes(zg):
    assert W.workload("gpt2s").N == 123_570_432 and zg.plan(W.workload("gpt2s").numel, 8, 2, 25 * 1024 * 1024)["n_buckets"] > 1
    assert W.workload("1p3b").N == 1_310_885_888
    assert W.workload("4b").N == 4_092_982_400
    n3 = np.array(W.workload("ragged").numel)
    assert len(n3) == 2000 and n3.min() >= 1024 and n3.max() <= 2 ** 22 + 64
    assert (n3 % 2 == 1).mean() >= 0.25


@pytest.mark.parametrize("kw,code", [
    (dict(M=0), -1), (dict(M=65), -1), (dict(stage=0), -4), (dict(stage=4), -4),
    (dict(bucket_bytes=-1), -1), (dict(gather=1, stage=1), -4), (dict(gather=2), -1), (dict(groups=-1), -1),
    (dict(groups=3), -1)])
def test_invalid_config_rejected(zg, kw, code):
    cfg = dict(M=2, stage=3, bucket_bytes=0, gather=0, groups=0)
    cfg.update(kw)
    c = zg.Config(cfg["M"], cfg["stage"], cfg["bucket_bytes"], cfg["gather"], cfg["groups"])
    arr = (ctypes.c_int64 * 1)(100)
    out = zg.Sizes()
    assert zg._lib().zero_plan(ctypes.byref(c), ctypes.cast(arr, ctypes.c_void_p), 1, ctypes.byref(out)) == code


def test_invalid_tensor_lists_rejected(zg):
    c = zg.Config(2, 1, 0, 0, 0)
    out = zg.Sizes()
    lib = zg._lib()
    for vals in ([], [0, 0], [-5, 10]):
        arr = (ctypes.c_int64 * max(len(vals), 1))(*vals)
        assert lib.zero_plan(ctypes.byref(c), ctypes.cast(arr, ctypes.c_void_p), len(vals), ctypes.byref(out)) == -1
    assert lib.zero_plan(None, None, 1, ctypes.byref(out)) == -1


def test_null_or_unknown_context_rejected_without_touching_cuda(zg):
    lib = zg._lib()
    h = zg.Hyper()
    bogus = ctypes.c_void_p(0x1234)
    for ctx in (None, bogus):
        assert lib.zero_step(ctx, None, 1, ctypes.byref(h), None) == -7
        assert lib.zero_destroy(ctx) == -7
        p = ctypes.c_void_p()
        assert lib.zero_params(ctx, ctypes.byref(p)) == -7
        assert lib.zero_sync_status(ctx) == -7
        assert lib.zero_set_timing(ctx, 1) == -7
        assert lib.zero_set_schedule(ctx, ctypes.byref(h), 1, None) == -7
        assert lib.zero_step_scheduled(ctx, None, 1, None) == -7
        assert lib.zero_apply_scheduled(ctx, 1, None) == -7
        assert lib.zero_step_bucket(ctx, 0, None, 1, ctypes.byref(h), None) == -7
        assert lib.zero_step_bucket_scheduled(ctx, 0, None, 1, None) == -7


def _golden(name):
    rows = {}
    for line in open(os.path.join(ROOT, "tests", "golden", name)):
        line = line.split("#", 1)[0].strip()
        if line:
            k, *v = line.split()
            rows[k] = [float(x) for x in v]
    return rows


def test_state_ledger_matches_pages(zg):
    g = _golden("state_ledger_pages.txt")
    f = zg.state_bytes_per_param
    # 16 B/param mixed-precision Adam, full data parallel: 7B -> 112 GB
    assert f(0, 8, 2, 2, 12) == g["bytes_per_param_mixed_adam"][0]
    assert 7e9 * f(0, 8, 2, 2, 12) / 1e9 == g["full_dp_state_7B_GB"][0]
    # 8 x 80 GB, 12 B/param = 2 param + 2 grad + 8 optimizer: capacity per stage (billions;
    # the page truncates 6.666... to 6.66 and rounds the others)
    caps = [80e9 / f(s, 8, 2, 2, 8) / 1e9 for s in (0, 1, 2, 3)]
    for got, printed in zip(caps, g["zero_capacity_8xA100_80GB_B"]):
        assert abs(got - printed) <= 0.01, (caps, g["zero_capacity_8xA100_80GB_B"])
    # 4 values x 2 bytes: 1B -> 8 GB; 100B -> 800 GB, and 10 GB per GPU over 80 GPUs
    assert 1e9 * f(0, 1, 2, 2, 4) / 1e9 == g["dp_4x2B_1B_GB"][0]
    assert 100e9 * f(0, 1, 2, 2, 4) / 1e9 == g["fsdp_4x2B_100B_total_GB"][0]
    assert 100e9 * f(3, 80, 2, 2, 4) / 1e9 == g["fsdp_4x2B_100B_per_gpu_80_GB"][0]
    assert f(4, 8, 2, 2, 8) < 0 and f(1, 0, 2, 2, 8) < 0


@pytest.mark.parametrize("numel,M,bucket_bytes,groups", [
    ((1000, 37, 3001), 2, 6100, 1), (W.ragged_numel(40, 100, 6000, 3), 4, 15000, 1),
    ((5, 7, 4099), 8, 0, 2), ((3,), 16, 0, 1)])
def test_sharded_sizes(zg, numel, M, bucket_bytes, groups):
    """Process-per-rank sizes: one rank's shard of the state, the padded full parameters and
    gradient, the same layout (and npad) as the emulated job planned for the owners."""
    K = M // groups
    emu = zg.plan(numel, M, 3, bucket_bytes, groups=groups)
    p = O.plan(numel, K, bucket_bytes, 64)
    for r in range(M):
        s = zg.plan(numel, M, 3, bucket_bytes, groups=groups, rank=r)
        assert (s["npad"], s["n"], s["n_buckets"], s["shard_len"]) == (p.npad, p.N, p.nb, p.shard_len)
        assert s["bytes_master"] == s["bytes_m"] == s["bytes_v"] == s["bytes_ghat"] == 4 * p.shard_len
        assert s["bytes_param_shards"] == 2 * p.shard_len and s["bytes_param_full"] == 2 * p.npad
        assert s["bytes_grad_each"] == 2 * p.npad
        # the scratch also holds the rank's own bucket table (32 bytes a bucket, rounded to 256)
        assert s["bytes_scratch"] == emu["bytes_scratch"] + (32 * p.nb + 255) // 256 * 256
        assert zg.layout(numel, M, 3, bucket_bytes, groups=groups) == (
            [int(x) for x in p.t_off], [(int(a), int(b), int(c), int(d)) for a, b, c, d in
                                        zip(p.b_off, p.b_n, p.b_S, p.b_first[:p.nb])])


@pytest.mark.parametrize("sharded,rank,gather,stage,code", [
    (1, 2, 0, 1, -1), (1, -1, 0, 1, -1), (2, 0, 0, 1, -1), (1, 1, 1, 1, 0), (0, 5, 0, 1, 0)])
def test_sharded_config_checks(zg, sharded, rank, gather, stage, code):
    """rank must lie in [0, M) in process-per-rank mode (and is ignored otherwise); the gather
    mode has no effect there, so the shards mode is accepted at any stage."""
    c = zg.Config(2, stage, 0, gather, 0, sharded, rank)
    arr = (ctypes.c_int64 * 1)(100)
    out = zg.Sizes()
    assert zg._lib().zero_plan(ctypes.byref(c), ctypes.cast(arr, ctypes.c_void_p), 1, ctypes.byref(out)) == code


def test_rank_calls_reject_null_or_unknown_context(zg):
    lib = zg._lib()
    h = zg.Hyper(clip=True)
    for ctx in (None, ctypes.c_void_p(0x1234)):
        assert lib.zero_rank_step(ctx, None, None, 1, ctypes.byref(h), None) == -7
        assert lib.zero_rank_sumsq(ctx, None, ctypes.byref(h), None, None) == -7
        assert lib.zero_rank_partial(ctx, None, None, None) == -7
