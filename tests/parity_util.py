"""Comparison helpers shared by the GPU parity tests (tolerances, run loops).

Tolerances (from the step's arithmetic): the averaged gradient and all indexing are
bit-exact; fp32 master / m / v within 1e-6 relative (|oracle| floored at 2^-126; lanes
with |oracle| < 1e-30 use 1e-36 absolute); bf16 parameters within 1 bf16 ulp; the global
norm within 1e-7 relative. With identical operation order the GPU is expected to match
bit for bit; it may differ only through the clip scale, whose norm is summed in another
order.
"""
import math

import numpy as np
import torch

import oracle as O
import workloads as W
import zero_gradient_reduce_scatter_gb300 as zg

REL_STATE = 1e-6
REL_NORM = 1e-7


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy()


def state_errors(got: np.ndarray, want: np.ndarray) -> float:
    """Largest violation ratio (<= 1 passes) of the fp32 state tolerance."""
    g, w = got.astype(np.float64), want.astype(np.float64)
    both_nan = np.isnan(g) & np.isnan(w)
    err = np.abs(g - w)
    tiny = np.abs(w) < 1e-30
    ratio = np.where(tiny, err / 1e-36, err / (REL_STATE * np.maximum(np.abs(w), 2.0 ** -126)))
    ratio = np.where(both_nan, 0.0, ratio)
    ratio = np.where(np.isnan(ratio), np.inf, ratio)
    return float(ratio.max()) if ratio.size else 0.0


def assert_state_close(got, want, what):
    r = state_errors(got, want)
    assert r <= 1.0, f"{what}: error {r:.3g} x tolerance"


def bf16_ulp_diff(a: np.ndarray, b: np.ndarray) -> int:
    """Largest distance in bf16 ulps between two bf16 bit-pattern arrays (NaN == NaN)."""
    def key(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, -(x & 0x7FFF), x)  # monotone integer line, -0 == +0
    nan_a = ((a & 0x7F80) == 0x7F80) & ((a & 0x7F) != 0)
    nan_b = ((b & 0x7F80) == 0x7F80) & ((b & 0x7F) != 0)
    d = np.abs(key(a) - key(b))
    d = np.where(nan_a & nan_b, 0, d)
    d = np.where(nan_a ^ nan_b, 1 << 20, d)
    return int(d.max()) if d.size else 0


def make_hyper(w: W.Workload, ghat_mode="auto"):
    clip = w.clip is not None
    h = zg.Hyper(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, weight_decay=w.weight_decay,
                 clip=clip, max_grad_norm=w.clip if clip else 1.0, ghat_mode=ghat_mode)
    oh = O.hyper(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, weight_decay=w.weight_decay, clip=clip,
                 max_grad_norm=w.clip if clip else 1.0)
    return h, oh


def run_elementwise(w: W.Workload, gather="fused", ghat_mode="auto", steps=None, ghat_buffer=None,
                    garbage_in_padding=False, check_every_step=True, groups=1):
    """Runs the GPU path and the oracle side by side on w and compares everything.
    Returns a dict of the largest deviations seen."""
    dev = torch.device("cuda")
    steps = w.steps if steps is None else steps
    mi = W.master_init(w, dev)
    opt = zg.ZeroOptimizer(w.numel, w.M, w.stage, mi, bucket_bytes=w.bucket_bytes, gather=gather,
                           ghat_buffer=ghat_buffer, groups=groups)
    p = O.plan(w.numel, w.M // groups, w.bucket_bytes)  # hybrid sharding: planned for the group size
    assert p.npad == opt.sizes["npad"] and [int(x) for x in p.t_off] == opt.tensor_offsets
    st = O.init_state(p, w.stage, f32(mi), groups=groups)
    h, oh = make_hyper(w, ghat_mode)
    sig = W.sigmas(w)
    real = p.real_mask()
    worst = {"state_err": 0.0, "bf16_ulp": 0, "norm_rel": 0.0}
    for k in range(steps):
        grads = opt.new_grad_buffers()
        if garbage_in_padding:
            for g in grads:
                g.view(torch.int16)[torch.from_numpy(~real).to(dev)] = 0x3F80  # 1.0 in every padding lane
        for r in range(w.M):
            W.fill_grads(w, r, k, grads[r], opt.tensor_offsets, sig)
        opt.step(grads, h)
        host = [u16(g) for g in grads]
        full, norm, scale, rc = O.zero_step(p, st, host, oh)
        status = opt.sync_status()
        assert (status == zg.ZERO_ERR_NONFINITE) == (rc == 1)
        if w.clip is not None:
            gn, gs = opt.last_norm()
            if math.isfinite(norm):
                rel = abs(gn - norm) / max(norm, 1e-300)
                worst["norm_rel"] = max(worst["norm_rel"], rel)
                assert rel <= REL_NORM, f"step {k}: norm {gn!r} vs oracle {norm!r}"
        else:
            assert opt.last_norm() is None
        if check_every_step or k == steps - 1:
            d = bf16_ulp_diff(u16(opt.params()), full)
            worst["bf16_ulp"] = max(worst["bf16_ulp"], d)
            assert d <= 1, f"step {k}: bf16 params differ by {d} ulp"
            for name, buf in (("master", opt.master), ("mom", opt.m), ("var", opt.v)):
                want = O.flat_state(p, st, name)
                got = f32(buf)
                r = state_errors(got, want)
                worst["state_err"] = max(worst["state_err"], r)
                assert r <= 1.0, f"step {k}: {name} error {r:.3g} x tolerance"
            if gather == "shards":
                sh = u16(opt.param_shards)
                want_sh = np.zeros(p.npad, dtype=np.uint16)
                for rr in range(p.M):
                    want_sh[p.shard_lanes(rr)] = st.param[rr][:p.shard_len]
                assert bf16_ulp_diff(sh, want_sh) <= 1
    out = dict(worst, opt=opt, plan=p, oracle_state=st)
    return out
