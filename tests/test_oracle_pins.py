"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test names what it pins it to: a closed form, an exact-arithmetic case, a brute-force
enumeration, a hand-worked example from the pages (tests/golden/), or a library routine
that is run (never retyped). The tests are chosen so that a plausible slip anywhere in the
oracle (a dropped term, a wrong sign or index, a swapped operand, a wrong rank order)
fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf(x):
    """Exact bf16 bit patterns of values that bf16 represents exactly."""
    a = np.asarray(x, dtype=np.float32)
    bits = a.view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0), "value not exactly representable in bf16"
    return (bits >> 16).astype(np.uint16)


def f32_of_bf(h):
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def read_golden(name):
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, *vals = line.split()
                rows[k] = [float(v) for v in vals]
    return rows


# ------------------------------------------------------------------------------------------
# bf16 round-to-nearest-even: exhaustive over every fp32 bit pattern, against torch's cast
# ------------------------------------------------------------------------------------------
def test_bf16_rne_exhaustive_matches_torch():
    chunk = 1 << 26
    for start in range(0, 1 << 32, chunk):
        bits = np.arange(start, start + chunk, dtype=np.uint64).astype(np.uint32)
        x = bits.view(np.float32)
        ours = O.bf16_rne(x)
        ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        nan = np.isnan(x)
        assert np.array_equal(ours[~nan], ref[~nan]), f"RNE mismatch in chunk at {start:#x}"
        # NaN stays NaN (payloads aside)
        assert np.all((ours[nan] & 0x7F80) == 0x7F80) and np.all((ours[nan] & 0x7F) != 0)


def test_bf16_rne_ties_and_neighbours_match_torch():
    """Fast subset of the exhaustive check: for every upper half, the dropped halves at and
    next to the tie (0x7FFF, 0x8000, 0x8001), zero and all-ones, plus a random sample."""
    upper = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF], dtype=np.uint32)
    bits = (upper[:, None] | lows[None, :]).ravel()
    rnd = np.random.default_rng(0).integers(0, 1 << 32, 1 << 20, dtype=np.uint64).astype(np.uint32)
    x = np.concatenate([bits, rnd]).view(np.float32)
    ours = O.bf16_rne(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_bf16_widening_is_exact():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = O.bf16_to_f32(h)
    ref = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).float().numpy()
    same = (ours.view(np.uint32) == ref.view(np.uint32)) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


# ------------------------------------------------------------------------------------------
# Planner: brute force over small sizes
# ------------------------------------------------------------------------------------------
def _check_plan_invariants(p, numel, M, A, bucket_bytes):
    T = len(numel)
    # buckets partition the tensors in declared order, never splitting one
    assert p.b_first[0] == 0 and p.b_first[-1] == T
    assert np.all(np.diff(p.b_first) >= 1)
    for b in range(p.nb):
        ts = range(p.b_first[b], p.b_first[b + 1])
        assert p.b_n[b] == sum(numel[t] for t in ts)
        # tensors are contiguous inside their bucket, in order
        pos = p.b_off[b]
        for t in ts:
            assert p.t_off[t] == pos
            pos += numel[t]
        # padding: shard length is a multiple of A; M*S covers the bucket with < M*A slack
        assert p.b_S[b] % A == 0
        assert M * p.b_S[b] >= p.b_n[b] and M * p.b_S[b] - p.b_n[b] < M * A
        # greedy fill: the bucket respects the byte cap unless it holds one tensor;
        # and the next tensor did not fit
        if bucket_bytes > 0:
            assert 2 * p.b_n[b] <= bucket_bytes or sum(1 for t in ts if numel[t] > 0) <= 1
            if b + 1 < p.nb:
                nxt = p.b_first[b + 1]
                assert 2 * p.b_n[b] + 2 * numel[nxt] > bucket_bytes
    # buckets tile [0, npad) without gaps
    ends = p.b_off + M * p.b_S
    assert p.b_off[0] == 0 and np.array_equal(p.b_off[1:], ends[:-1]) and ends[-1] == p.npad


def test_plan_single_tensor_bruteforce():
    for A in (1, 8, 64):
        for M in range(1, 18):
            for n in range(1, 201):
                p = O.plan([n], M, 0, A)
                assert p.nb == 1
                _check_plan_invariants(p, [n], M, A, 0)
                S = p.b_S[0]
                assert S == -(-n // (M * A)) * A
                # shard(x) then gather == x; padding lanes read zero; the unpadded map is a bijection
                x = np.arange(1, n + 1, dtype=np.float32)  # exact in bf16 up to 256
                st = O.init_state(p, 3, x)
                lanes = [p.shard_lanes(r) for r in range(M)]
                seen = np.zeros(n, dtype=np.int64)
                for r in range(M):
                    for j, o in enumerate(lanes[r]):
                        val = st.master[r][j]
                        if o < n:
                            assert val == x[o]
                            seen[o] += 1
                        else:
                            assert val == 0.0
                assert np.all(seen == 1)


def test_init_with_moments_places_them_like_master():
    """Initial m / v given unpadded land at the same owner lanes as the master (brute force),
    padding stays 0, and omitting them is the same as passing zeros."""
    for M in (1, 3, 4, 7):
        numel = [5, 130, 1, 64]
        p = O.plan(numel, M, 300, 8)
        x = np.arange(1, p.N + 1, dtype=np.float32)
        st = O.init_state(p, 2, x, -x, 2 * x)
        u = p.unpadded_index()
        for name, want in (("master", x), ("mom", -x), ("var", 2 * x)):
            flat = O.flat_state(p, st, name)
            assert np.array_equal(flat[u >= 0], want) and np.all(flat[u < 0] == 0)
        z = O.init_state(p, 3, x, np.zeros(p.N, np.float32), np.zeros(p.N, np.float32))
        z0 = O.init_state(p, 3, x)
        for a, b in zip(z.mom + z.var + z.param, z0.mom + z0.var + z0.param):
            assert np.array_equal(a, b)


def test_plan_multi_tensor_bruteforce():
    rng = np.random.default_rng(5)
    for trial in range(400):
        T = int(rng.integers(1, 9))
        numel = [int(v) for v in rng.integers(0, 60, size=T)]
        if sum(numel) == 0:
            numel[0] = 1
        M = int(rng.integers(1, 18))
        A = int(rng.choice([1, 8, 64]))
        bucket_bytes = int(rng.choice([0, 2, 20, 50, 120]))
        p = O.plan(numel, M, bucket_bytes, A)
        _check_plan_invariants(p, numel, M, A, bucket_bytes)
        N = sum(numel)
        u = p.unpadded_index()
        real = u >= 0
        assert real.sum() == N and np.array_equal(np.sort(u[real]), np.arange(N))
        # unpadded order equals padded order restricted to real lanes
        assert np.all(np.diff(u[real]) == 1)
        # tensors land at their unpadded offsets
        starts = np.concatenate([[0], np.cumsum(numel)[:-1]])
        for t in range(T):
            if numel[t]:
                assert u[p.t_off[t]] == starts[t]


def test_plan_bucket_fill_hand_cases():
    # cap 100 bytes = 50 bf16 elements: [30, 30] -> two buckets; [20, 30] -> one; [80] alone
    p = O.plan([30, 30, 20, 30, 80, 10], M=2, bucket_bytes=100, A=1)
    assert list(p.b_first) == [0, 1, 3, 4, 5, 6]
    assert list(p.b_n) == [30, 50, 30, 80, 10]
    # one bucket when no size is given
    p = O.plan([30, 30, 20], M=2, bucket_bytes=0, A=1)
    assert p.nb == 1 and p.b_n[0] == 80
    # ragged: 7 elements over 4 ranks with A = 1 -> S = 2, one padding lane
    p = O.plan([7], M=4, bucket_bytes=0, A=1)
    assert p.b_S[0] == 2 and p.npad == 8


# ------------------------------------------------------------------------------------------
# Reduce-scatter
# ------------------------------------------------------------------------------------------
def test_reduce_scatter_exact_integer_sums():
    """Small-integer gradients: every partial sum is exact in fp32, so the averaged value
    must equal the exact rational sum / M for power-of-two M; distinct values per rank and
    lane expose any wrong rank or lane index."""
    rng = np.random.default_rng(1)
    for M in (1, 2, 4, 8, 16):
        numel = [37, 5, 130]
        p = O.plan(numel, M, 0, 8)
        vals = rng.integers(-128, 129, size=(M, p.N))
        grads = [p.pad(bf(vals[r].astype(np.float32))) for r in range(M)]
        gh = O.reduce_scatter(p, grads)
        flat = O.flat_state(p, O.RankState(1, gh, gh, gh, gh, []), "ghat")
        u = p.unpadded_index()
        expect = vals.sum(axis=0) / M
        assert np.array_equal(flat[u >= 0].astype(np.float64), expect)
        assert np.all(flat[u < 0] == 0.0)


def test_reduce_scatter_rank_order_is_zero_to_m_minus_one():
    """fl(fl(1 + 2^-24) + 2^-24) = 1 (two ties to even), while the reverse order gives
    1 + 2^-23 exactly: only the rank order 0, 1, 2 produces 1."""
    M = 4
    p = O.plan([1], M, 0, 1)
    g = [bf([1.0]), bf([2.0 ** -24]), bf([2.0 ** -24]), bf([0.0])]
    gh = O.reduce_scatter(p, [p.pad(x) for x in g])
    assert gh[0][0] == np.float32(0.25)  # 1 * (1/4)
    g_rev = [g[3], g[2], g[1], g[0]]
    gh = O.reduce_scatter(p, [p.pad(x) for x in g_rev])
    assert gh[0][0] == np.float32((1.0 + 2.0 ** -23) / 4)


def test_reduce_scatter_sum_of_negative_zeros_is_positive_zero():
    M = 3
    p = O.plan([4], M, 0, 1)
    neg0 = np.full(4, 0x8000, dtype=np.uint16)
    gh = O.reduce_scatter(p, [p.pad(neg0) for _ in range(M)])
    flat = O.flat_state(p, O.RankState(1, gh, gh, gh, gh, []), "ghat")
    assert np.all(flat.view(np.uint32) == 0)


def test_reduce_scatter_identical_replicas_power_of_two():
    """M identical replicas with M a power of two: the average is the replica, bit for bit."""
    rng = np.random.default_rng(2)
    for M in (2, 4, 8, 16):
        p = O.plan([300, 77], M, 0, 64)
        g = O.bf16_rne(rng.normal(0, 1e-3, p.N).astype(np.float32))
        gh = O.reduce_scatter(p, [p.pad(g) for _ in range(M)])
        flat = O.flat_state(p, O.RankState(1, gh, gh, gh, gh, []), "ghat")
        assert np.array_equal(flat[p.unpadded_index() >= 0].view(np.uint32), f32_of_bf(g).view(np.uint32))


def test_dp_identity_hand_example():
    """The averaged rank-local gradients equal the full-batch gradient (golden, hand-computed)."""
    gd = read_golden("dp_identity_example.txt")
    p = O.plan([2], 2, 0, 1)
    grads = [p.pad(bf(gd["rank0_grad"])), p.pad(bf(gd["rank1_grad"]))]
    gh = O.reduce_scatter(p, grads)
    flat = O.flat_state(p, O.RankState(1, gh, gh, gh, gh, []), "ghat")
    assert list(flat[:2]) == gd["full_batch_grad"]


# ------------------------------------------------------------------------------------------
# Norm and clipping
# ------------------------------------------------------------------------------------------
def _norm_of(p, grads):
    gh = O.reduce_scatter(p, grads)
    return math.sqrt(O.global_sumsq(p, gh))


def test_norm_closed_forms():
    # all-equal averaged gradient c over N = 4096 lanes: ||g|| = |c| * 64 exactly
    p = O.plan([4096], 4, 0, 64)
    c = 2.0 ** -7
    g = p.pad(bf(np.full(4096, c, dtype=np.float32)))
    assert _norm_of(p, [g] * 4) == c * 64
    # 3-4-5 across two tensors and padding lanes holding garbage do not count
    p = O.plan([1, 1], 2, 0, 64)
    g = np.zeros(p.npad, dtype=np.uint16)
    g[p.t_off[0]] = bf([3.0])[0]
    g[p.t_off[1]] = bf([4.0])[0]
    assert _norm_of(p, [g, g]) == 5.0
    junk = g.copy()
    junk[p.unpadded_index() < 0] = bf([1024.0])[0]
    assert _norm_of(p, [junk, junk]) == 5.0


def test_norm_matches_torch_vector_norm():
    rng = np.random.default_rng(3)
    p = O.plan([1000, 333, 4097], 5, 0, 64)
    grads = [p.pad(O.bf16_rne(rng.normal(0, 1e-2, p.N).astype(np.float32))) for _ in range(5)]
    gh = O.reduce_scatter(p, grads)
    flat = O.flat_state(p, O.RankState(1, gh, gh, gh, gh, []), "ghat")[p.unpadded_index() >= 0]
    ref = torch.linalg.vector_norm(torch.from_numpy(flat.astype(np.float64))).item()
    assert abs(math.sqrt(O.global_sumsq(p, gh)) - ref) <= 1e-14 * ref


def test_sumsq_chunks_equal_whole():
    rng = np.random.default_rng(4)
    p = O.plan([100, 7, 900, 31], 3, 2000, 8)
    grads = [rng.integers(0, 0x3F00, p.npad).astype(np.uint16) for _ in range(3)]
    whole = O.global_sumsq(p, O.reduce_scatter(p, grads))
    acc = 0.0
    for o0 in range(0, p.npad, 97):
        acc = O.sumsq_chunk(acc, p, [g[o0:o0 + 97] for g in grads], o0)
    assert acc == whole


def test_clip_scale_closed_forms():
    assert O.clip_scale(0.5, 1.0) == 1.0
    assert O.clip_scale(1.0, 1.0) == 1.0
    assert O.clip_scale(4.0, 1.0) == 0.25
    # after clipping the norm is the threshold, to fp32 rounding
    for n in (1.7, 33.3, 1e4):
        s = O.clip_scale(n, 1.0)
        assert abs(s * n - 1.0) <= 1e-7


# ------------------------------------------------------------------------------------------
# AdamW
# ------------------------------------------------------------------------------------------
def test_adamw_step1_closed_form():
    """t = 1: m = (1-b1) g, v = (1-b2) g^2, m_hat = g, v_hat = g^2, so
    p1 = p0 (1 - lr wd) - lr g / (|g| + eps); checked in fp64 within 1e-6 of the size of
    its terms (p1 itself can cancel to ~0)."""
    rng = np.random.default_rng(6)
    n = 20000
    g = rng.normal(0, 1e-3, n).astype(np.float32)
    g[:50] = rng.normal(0, 1e-9, 50)  # |g| comparable to eps
    p0 = rng.normal(0, 0.02, n).astype(np.float32)
    h = O.hyper(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    p, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    O.adamw(g, 1.0, p, m, v, h, 1)
    g64, p64 = g.astype(np.float64), p0.astype(np.float64)
    exp_p = p64 * (1 - 1e-3 * 0.01) - 1e-3 * g64 / (np.abs(g64) + 1e-8)
    # relative to the size of the two terms (p1 may cancel to ~0)
    assert np.max(np.abs(p - exp_p) / (np.abs(p64) + 1e-3)) <= 1e-6
    assert np.max(np.abs(m - 0.1 * g64) / np.abs(0.1 * g64)) <= 1e-6
    assert np.max(np.abs(v - 0.001 * g64 ** 2) / (0.001 * g64 ** 2)) <= 1e-6


def test_adamw_step2_closed_form_three_elements():
    """t = 2 by hand: m2 = b1 (1-b1) g1 + (1-b1) g2, v2 = b2 (1-b2) g1^2 + (1-b2) g2^2,
    p2 = p1 (1 - lr wd) - lr m2/(1-b1^2) / (sqrt(v2/(1-b2^2)) + eps)."""
    b1, b2, lr, wd, eps = 0.9, 0.999, 1e-3, 0.01, 1e-8
    g1 = np.array([1e-3, -2e-3, 5e-4], np.float32)
    g2 = np.array([-1e-3, -1e-3, 3e-3], np.float32)
    p0 = np.array([0.02, -0.01, 0.005], np.float32)
    h = O.hyper(lr=lr, beta1=b1, beta2=b2, eps=eps, weight_decay=wd)
    p, m, v = p0.copy(), np.zeros(3, np.float32), np.zeros(3, np.float32)
    O.adamw(g1, 1.0, p, m, v, h, 1)
    O.adamw(g2, 1.0, p, m, v, h, 2)
    G1, G2, P0 = g1.astype(np.float64), g2.astype(np.float64), p0.astype(np.float64)
    P1 = P0 * (1 - lr * wd) - lr * G1 / (np.abs(G1) + eps)
    M2 = b1 * (1 - b1) * G1 + (1 - b1) * G2
    V2 = b2 * (1 - b2) * G1 ** 2 + (1 - b2) * G2 ** 2
    P2 = P1 * (1 - lr * wd) - lr * (M2 / (1 - b1 ** 2)) / (np.sqrt(V2 / (1 - b2 ** 2)) + eps)
    assert np.max(np.abs(m - M2) / np.abs(M2)) <= 1e-6
    assert np.max(np.abs(v - V2) / np.abs(V2)) <= 1e-6
    assert np.max(np.abs(p - P2) / (np.abs(P0) + lr)) <= 1e-6


def test_clipped_step_closed_form():
    """All-equal averaged gradient c over N lanes: norm = |c| sqrt(N), s = C / norm, and
    after one step m = (1-b1) s c, v = (1-b2) (s c)^2 (fp64 closed form, 1e-6)."""
    M, N, C = 4, 4096, 1e-3
    p = O.plan([N], M, 0, 64)
    c = 2.0 ** -7
    st = O.init_state(p, 1, np.zeros(N, np.float32))
    g = p.pad(bf(np.full(N, c, dtype=np.float32)))
    _, norm, s, rc = O.zero_step(p, st, [g] * M, O.hyper(clip=True, max_grad_norm=C))
    assert rc == 0 and norm == c * 64
    assert abs(s - C / (c * 64)) <= 1e-7 * (C / (c * 64))
    m = O.flat_state(p, st, "mom")[:N].astype(np.float64)
    v = O.flat_state(p, st, "var")[:N].astype(np.float64)
    sc = C / (c * 64) * c
    assert np.max(np.abs(m - 0.1 * sc)) <= 1e-6 * 0.1 * sc
    assert np.max(np.abs(v - 0.001 * sc * sc)) <= 1e-6 * 0.001 * sc * sc


def test_single_rank_clip_matches_torch():
    """M = 1 with clipping: torch.nn.utils.clip_grad_norm_ followed by torch.optim.AdamW.
    torch divides by (norm + 1e-6); at norms ~10 that moves the scale by ~1e-7 relative."""
    rng = np.random.default_rng(17)
    numel = [2000, 300]
    p = O.plan(numel, 1, 0, 64)
    w0 = rng.normal(0, 0.02, p.N).astype(np.float32)
    st = O.init_state(p, 1, w0)
    h = O.hyper(lr=1e-3, clip=True, max_grad_norm=1.0)
    tw = torch.nn.Parameter(torch.from_numpy(w0.copy()))
    opt = torch.optim.AdamW([tw], lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.01, foreach=False)
    for step in range(4):
        g = O.bf16_rne(rng.normal(0, 0.2, p.N).astype(np.float32))
        _, norm, s, rc = O.zero_step(p, st, [p.pad(g)], h)
        assert rc == 0 and s < 0.2
        tw.grad = torch.from_numpy(f32_of_bf(g).copy())
        tnorm = torch.nn.utils.clip_grad_norm_([tw], max_norm=1.0, foreach=False)
        assert abs(norm - float(tnorm)) <= 1e-6 * norm
        opt.step()
    u = p.unpadded_index()
    sd = opt.state[tw]
    for ours_v, ref, scale in ((O.flat_state(p, st, "master")[u >= 0], tw.detach().numpy(), 1e-3),
                               (O.flat_state(p, st, "mom")[u >= 0], sd["exp_avg"].numpy(), None),
                               (O.flat_state(p, st, "var")[u >= 0], sd["exp_avg_sq"].numpy(), None)):
        ref = ref.astype(np.float64)
        scale = np.max(np.abs(ref)) * 0.1 if scale is None else scale
        assert np.max(np.abs(ours_v - ref) / (np.abs(ref) + scale)) <= 1e-6


def test_single_rank_matches_torch_adamw():
    """M = 1 and no clipping: the ZeRO step is plain AdamW; torch.optim.AdamW (fp32,
    single-tensor implementation) is run for the same steps."""
    rng = np.random.default_rng(7)
    numel = [513, 64, 1000]
    p = O.plan(numel, 1, 0, 64)
    w0 = rng.normal(0, 0.02, p.N).astype(np.float32)
    st = O.init_state(p, 1, w0)
    h = O.hyper(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    tw = torch.nn.Parameter(torch.from_numpy(w0.copy()))
    opt = torch.optim.AdamW([tw], lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.01, foreach=False)
    for step in range(6):
        g = O.bf16_rne(rng.normal(0, 1e-3, p.N).astype(np.float32))
        full, _, _, rc = O.zero_step(p, st, [p.pad(g)], h)
        assert rc == 0
        tw.grad = torch.from_numpy(f32_of_bf(g).copy())
        opt.step()
    u = p.unpadded_index()
    ours = {k: O.flat_state(p, st, k)[u >= 0] for k in ("master", "mom", "var")}
    sd = opt.state[tw]
    # torch orders the same arithmetic differently (lerp for m, division by sqrt(bc2),
    # value*m/den), so values that cancel toward 0 are compared against the size of the
    # terms that produced them: lr for the parameter, the array's own scale for m and v.
    for ours_v, ref, scale in ((ours["master"], tw.detach().numpy(), 1e-3),
                               (ours["mom"], sd["exp_avg"].numpy(), None),
                               (ours["var"], sd["exp_avg_sq"].numpy(), None)):
        ref = ref.astype(np.float64)
        scale = np.max(np.abs(ref)) * 0.1 if scale is None else scale
        assert np.max(np.abs(ours_v - ref) / (np.abs(ref) + scale)) <= 1e-6
    diff = np.abs(f32_of_bf(full).astype(np.float64) - f32_of_bf(O.bf16_rne(tw.detach().numpy())))
    assert np.all(diff <= np.abs(tw.detach().numpy()) * 2.0 ** -8)  # at most 1 bf16 ulp


# ------------------------------------------------------------------------------------------
# Invariants of the pages: AR = RS + AG; ZeRO-1/2/3 == naive DP; buckets change nothing
# ------------------------------------------------------------------------------------------
def _run_zero(numel, M, stage, bucket_bytes, A, grads_unpadded, h, w0):
    p = O.plan(numel, M, bucket_bytes, A)
    st = O.init_state(p, stage, w0)
    outs = []
    for gs in grads_unpadded:
        full, norm, s, rc = O.zero_step(p, st, [p.pad(g) for g in gs], h)
        outs.append((full.copy(), norm, s, rc))
    u = p.unpadded_index()
    return outs, {k: O.flat_state(p, st, k)[u >= 0] for k in ("master", "mom", "var")}


@pytest.mark.parametrize("M,stage,bucket_bytes,clip", [
    (1, 1, 0, False), (2, 1, 0, True), (3, 2, 200, False), (4, 3, 0, True),
    (5, 3, 900, True), (8, 2, 64, True), (16, 3, 0, True), (16, 1, 5000, False)])
def test_zero_equals_naive_dp(M, stage, bucket_bytes, clip):
    rng = np.random.default_rng(100 + M * 10 + stage)
    numel = [257, 1, 0, 1000, 63, 129]
    N = sum(numel)
    w0 = rng.normal(0, 0.02, N).astype(np.float32)
    steps = [[O.bf16_rne(rng.normal(0, 1e-2, N).astype(np.float32)) for _ in range(M)] for _ in range(4)]
    h = O.hyper(clip=clip, max_grad_norm=0.05)
    outs, state = _run_zero(numel, M, stage, bucket_bytes, 64, steps, h, w0)
    dp = O.naive_dp_init(M, w0)
    for k, gs in enumerate(steps):
        full_dp, norm_dp, s_dp, rc_dp = O.naive_dp_step(dp, gs, h)
        full, norm, s, rc = outs[k]
        assert rc == rc_dp == 0
        assert norm == norm_dp and s == s_dp
        assert np.array_equal(full, full_dp)
    assert np.array_equal(state["master"].view(np.uint32), dp.master[0].view(np.uint32))
    assert np.array_equal(state["mom"].view(np.uint32), dp.mom[0].view(np.uint32))
    assert np.array_equal(state["var"].view(np.uint32), dp.var[0].view(np.uint32))
    if clip:
        assert any(o[2] < 1.0 for o in outs), "case meant to exercise clipping"


def test_all_reduce_equals_reduce_scatter_then_all_gather():
    """AR(G) == AG(RS(G)): the reduce-scatter shards, laid back in flat order, are the
    all-reduced gradient of naive DP (identity of "CS336 2026 Lecture 8" Slide 8)."""
    rng = np.random.default_rng(9)
    numel = [33, 700, 5]
    for M in (2, 3, 7):
        p = O.plan(numel, M, 300, 64)
        gs = [O.bf16_rne(rng.normal(0, 1, p.N).astype(np.float32)) for _ in range(M)]
        gh = O.reduce_scatter(p, [p.pad(g) for g in gs])
        ag = O.flat_state(p, O.RankState(1, gh, gh, gh, gh, []), "ghat")[p.unpadded_index() >= 0]
        # naive DP with lr = 0 exposes its all-reduced gradient through m = (1 - b1) * g
        # with b1 = 0: m = g exactly
        dp = O.naive_dp_init(M, np.zeros(p.N, np.float32))
        O.naive_dp_step(dp, gs, O.hyper(lr=0.0, beta1=0.0, weight_decay=0.0))
        assert np.array_equal(ag.view(np.uint32), dp.mom[0].view(np.uint32))


def test_bucket_size_changes_only_ownership():
    rng = np.random.default_rng(11)
    numel = [100, 200, 50, 3, 999]
    N = sum(numel)
    w0 = rng.normal(0, 0.02, N).astype(np.float32)
    steps = [[O.bf16_rne(rng.normal(0, 1e-2, N).astype(np.float32)) for _ in range(4)] for _ in range(3)]
    h = O.hyper(clip=True, max_grad_norm=0.02)
    ref = None
    for bb in (0, 100, 400, 2000):
        outs, state = _run_zero(numel, 4, 2, bb, 64, steps, h, w0)
        key = ([o[0].tobytes() for o in outs], [o[1] for o in outs], state["master"].tobytes())
        if ref is None:
            ref = key
        assert key == ref


def test_clip_off_equals_clip_with_large_threshold():
    rng = np.random.default_rng(12)
    numel = [500]
    w0 = rng.normal(0, 0.02, 500).astype(np.float32)
    steps = [[O.bf16_rne(rng.normal(0, 1e-3, 500).astype(np.float32)) for _ in range(2)]]
    a, sa = _run_zero(numel, 2, 1, 0, 64, steps, O.hyper(clip=False), w0)
    b, sb = _run_zero(numel, 2, 1, 0, 64, steps, O.hyper(clip=True, max_grad_norm=1e6), w0)
    assert b[0][2] == 1.0
    assert np.array_equal(a[0][0], b[0][0]) and sa["master"].tobytes() == sb["master"].tobytes()


def test_nonfinite_gradient_skips_update_when_clipping():
    rng = np.random.default_rng(13)
    p = O.plan([300], 2, 0, 64)
    w0 = rng.normal(0, 0.02, 300).astype(np.float32)
    st = O.init_state(p, 3, w0)
    before = O.flat_state(p, st, "master").copy()
    g0 = O.bf16_rne(rng.normal(0, 1e-3, 300).astype(np.float32))
    g1 = g0.copy()
    g1[17] = 0x7FC0  # NaN on rank 1
    full, norm, s, rc = O.zero_step(p, st, [p.pad(g0), p.pad(g1)], O.hyper(clip=True))
    assert rc == 1 and not math.isfinite(norm)
    assert np.array_equal(O.flat_state(p, st, "master"), before)
    assert np.array_equal(full, O.bf16_rne(w0))


def test_lane_steps_equal_full_step():
    """The sampled-lane path gives the same bits as the full step on the same lanes."""
    rng = np.random.default_rng(14)
    numel = [1000, 37, 4000]
    M, K = 4, 3
    p = O.plan(numel, M, 3000, 64)
    w0 = rng.normal(0, 0.02, p.N).astype(np.float32)
    st = O.init_state(p, 1, w0)
    h = O.hyper(clip=True, max_grad_norm=0.05)
    grads = [[p.pad(O.bf16_rne(rng.normal(0, 1e-2, p.N).astype(np.float32))) for _ in range(M)] for _ in range(K)]
    scales = []
    for k in range(K):
        _, _, s, rc = O.zero_step(p, st, grads[k], h)
        scales.append(s)
    lanes = np.sort(rng.choice(p.npad, 300, replace=False))
    g = np.stack([np.stack([grads[k][r][lanes] for r in range(M)]) for k in range(K)])
    real = p.real_mask()[lanes]
    w0p = p.pad(w0)
    pp, mm, vv = w0p[lanes].copy(), np.zeros(300, np.float32), np.zeros(300, np.float32)
    bfv, _ = O.lane_steps(M, g, real, scales, [1] * K, h, 1, pp, mm, vv)
    assert np.array_equal(pp, O.flat_state(p, st, "master")[lanes])
    assert np.array_equal(mm, O.flat_state(p, st, "mom")[lanes])
    assert np.array_equal(vv, O.flat_state(p, st, "var")[lanes])
    assert np.array_equal(bfv, O.bf16_rne(pp))


# ------------------------------------------------------------------------------------------
# Hybrid sharding ("CS231n Lecture 11" 4.4): M = G x K, sharded in groups of K, replicated
# across the G groups; the average is summed inside each group, then across groups.
# ------------------------------------------------------------------------------------------
def test_hsdp_group_order_pin():
    """G = 2, K = 2, one lane with values 1, 2^-24, 2^-24, 2^-24: flat order gives
    ((1 + 2^-24) + 2^-24) + 2^-24 = 1 (three ties to even); by groups
    (1 + 2^-24) + (2^-24 + 2^-24) = 1 + 2^-23 exactly."""
    vals = [1.0, 2.0 ** -24, 2.0 ** -24, 2.0 ** -24]
    p2 = O.plan([1], 2, 0, 1)
    st = O.init_state(p2, 1, np.zeros(1, np.float32), groups=2)
    h = O.hyper(lr=0.0, beta1=0.0, weight_decay=0.0)  # m = g exactly exposes the average
    O.zero_step(p2, st, [p2.pad(bf([v])) for v in vals], h)
    assert st.mom[0][0] == np.float32((1.0 + 2.0 ** -23) / 4)
    p4 = O.plan([1], 4, 0, 1)
    st4 = O.init_state(p4, 1, np.zeros(1, np.float32))
    O.zero_step(p4, st4, [p4.pad(bf([v])) for v in vals], h)
    assert st4.mom[0][0] == np.float32(0.25)


def test_hsdp_exact_integer_sums():
    rng = np.random.default_rng(31)
    for G, K in ((2, 2), (4, 2), (2, 8), (3, 3)):
        M = G * K
        p = O.plan([300, 17], K, 0, 8)
        vals = rng.integers(-100, 101, size=(M, p.N))
        st = O.init_state(p, 2, np.zeros(p.N, np.float32), groups=G)
        h = O.hyper(lr=0.0, beta1=0.0, weight_decay=0.0)
        O.zero_step(p, st, [p.pad(bf(vals[r].astype(np.float32))) for r in range(M)], h)
        got = O.flat_state(p, st, "mom")[p.unpadded_index() >= 0].astype(np.float64)
        exact = vals.sum(axis=0).astype(np.float64)
        want = (exact.astype(np.float32) * np.float32(1.0 / M)).astype(np.float64)  # sums are exact in fp32
        assert np.array_equal(got, want)


@pytest.mark.parametrize("G,K,stage,bucket_bytes,clip", [
    (1, 4, 1, 0, True), (2, 2, 2, 300, True), (2, 4, 3, 0, False), (4, 2, 3, 800, True), (3, 2, 1, 0, True)])
def test_hsdp_equals_naive_dp_with_grouped_allreduce(G, K, stage, bucket_bytes, clip):
    rng = np.random.default_rng(200 + 10 * G + K)
    numel = [257, 1, 1000, 63]
    N = sum(numel)
    M = G * K
    w0 = rng.normal(0, 0.02, N).astype(np.float32)
    steps = [[O.bf16_rne(rng.normal(0, 1e-2, N).astype(np.float32)) for _ in range(M)] for _ in range(3)]
    h = O.hyper(clip=clip, max_grad_norm=0.05)
    p = O.plan(numel, K, bucket_bytes, 64)
    st = O.init_state(p, stage, w0, groups=G)
    dp = O.naive_dp_init(M, w0)
    for gs in steps:
        full, norm, s, rc = O.zero_step(p, st, [p.pad(g) for g in gs], h)
        full_dp, norm_dp, s_dp, rc_dp = O.naive_dp_step(dp, gs, h, groups=G)
        assert rc == rc_dp == 0 and norm == norm_dp and s == s_dp
        assert np.array_equal(full, full_dp)
    u = p.unpadded_index()
    assert np.array_equal(O.flat_state(p, st, "master")[u >= 0].view(np.uint32), dp.master[0].view(np.uint32))
    # every group's replica of the shards is the same
    for grp in range(1, G):
        for k in range(K):
            assert np.array_equal(st.master[grp * K + k], st.master[k])


def test_hsdp_one_rank_per_group_is_plain_dp():
    """K = 1: each inner sum has one term (exact), so the grouped average is the flat one."""
    rng = np.random.default_rng(41)
    M, N = 5, 700
    w0 = rng.normal(0, 0.02, N).astype(np.float32)
    gs = [O.bf16_rne(rng.normal(0, 1e-2, N).astype(np.float32)) for _ in range(M)]
    h = O.hyper(clip=True, max_grad_norm=0.05)
    p = O.plan([N], 1, 0, 64)
    st = O.init_state(p, 1, w0, groups=M)
    dp = O.naive_dp_init(M, w0)
    full, norm, s, _ = O.zero_step(p, st, [p.pad(g) for g in gs], h)
    full_dp, norm_dp, s_dp, _ = O.naive_dp_step(dp, gs, h)
    assert norm == norm_dp and np.array_equal(full, full_dp)


@pytest.mark.parametrize("stage_a,stage_b,clip", [(3, 1, True), (2, 3, False), (1, 2, True)])
def test_resume_and_reshard_equal_uninterrupted_run(stage_a, stage_b, clip):
    """Checkpoint, resume and reshard, in the oracle alone: five steps of one job equal two
    steps, the unpadded state (master, m, v) and the step count handed to a job of another
    rank count, stage and bucket size, then three steps, bit for bit (norms, scales,
    parameters, state). Every rank holds the same gradient and both rank counts (4, 2) are
    powers of two, so the averaged gradient is that gradient exactly in both jobs; the
    flat real-lane order, and so the norm's summation order, does not depend on the layout."""
    rng = np.random.default_rng(70 + stage_a * 3 + stage_b)
    numel = [257, 1, 1000, 63, 130]
    N = sum(numel)
    w0 = rng.normal(0, 0.02, N).astype(np.float32)
    grads = [O.bf16_rne(rng.normal(0, 1e-2, N).astype(np.float32)) for _ in range(5)]
    h = O.hyper(clip=clip, max_grad_norm=0.05)

    pa = O.plan(numel, 4, 600)
    sa = O.init_state(pa, stage_a, w0)
    whole = [O.zero_step(pa, sa, [pa.pad(g)] * 4, h) for g in grads]

    pb = O.plan(numel, 4, 600)
    sb = O.init_state(pb, stage_a, w0)
    first = [O.zero_step(pb, sb, [pb.pad(g)] * 4, h) for g in grads[:2]]
    u = pb.unpadded_index()
    saved = {k: O.flat_state(pb, sb, k)[u >= 0].copy() for k in ("master", "mom", "var")}
    pc = O.plan(numel, 2, 0)
    sc = O.init_state(pc, stage_b, saved["master"], saved["mom"], saved["var"], t=sb.t)
    second = [O.zero_step(pc, sc, [pc.pad(g)] * 2, h) for g in grads[2:]]

    for (fa, na, sa_, ra), (fb, nb_, sb_, rb) in zip(whole, first + second):
        assert ra == rb == 0 and na == nb_ and sa_ == sb_
        assert np.array_equal(fa, fb)
    if clip:
        assert any(o[2] < 1.0 for o in whole), "case meant to exercise clipping"
    ua, uc = pa.unpadded_index(), pc.unpadded_index()
    for k in ("master", "mom", "var"):
        a = O.flat_state(pa, sa, k)[ua >= 0]
        c = O.flat_state(pc, sc, k)[uc >= 0]
        assert np.array_equal(a.view(np.uint32), c.view(np.uint32)), k
    assert sa.t == sc.t == 5
