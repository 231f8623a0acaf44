"""Test harness for the process-per-rank mode on one GPU: M rank contexts in one process,
created through the C ABI, with device copies in place of the collectives (the exchange
layout of include/zero_gb300.h, restated here from its definition). Every rank's kernels read
only that rank's buffers, exactly as in an M-process job.
"""
import ctypes

import numpy as np
import torch

import zero_gradient_reduce_scatter_gb300 as zg

_P = ctypes.c_void_p


class RankCtx:
    """One rank's context and buffers (torch allocations lent to the library)."""

    def __init__(self, numel, M, rank, stage, master_init, bucket_bytes=0, groups=1, ghat=True, full=True):
        self.M, self.rank, self.stage, self.groups = M, rank, stage, groups
        self.K = M // groups
        self.grp, self.owner = divmod(rank, self.K)
        s = self.sizes = zg.plan(numel, M, stage, bucket_bytes, groups=groups, rank=rank)
        self.tensor_offsets, self.buckets = zg.layout(numel, M, stage, bucket_bytes, groups=groups)
        dev = master_init.device
        L, npad = s["shard_len"], s["npad"]
        self.master = torch.empty(L, dtype=torch.float32, device=dev)
        self.m = torch.empty(L, dtype=torch.float32, device=dev)
        self.v = torch.empty(L, dtype=torch.float32, device=dev)
        self.ghat = torch.empty(L, dtype=torch.float32, device=dev) if ghat else None
        self.shards = torch.empty(L, dtype=torch.bfloat16, device=dev)
        self.full = torch.empty(npad, dtype=torch.bfloat16, device=dev) if full else None
        self.scratch = torch.empty(s["bytes_scratch"], dtype=torch.uint8, device=dev)
        self.recv = torch.empty(npad, dtype=torch.bfloat16, device=dev)
        P = self.K if groups > 1 else M
        self.sumsq = torch.zeros(1, dtype=torch.float64, device=dev)
        self.sums = torch.zeros(P, dtype=torch.float64, device=dev)
        if groups > 1:
            self.part = torch.empty(L, dtype=torch.float32, device=dev)
            self.parts = torch.empty(groups * L, dtype=torch.float32, device=dev)
        bufs = zg.Buffers(self.master.data_ptr(), self.m.data_ptr(), self.v.data_ptr(),
                          self.ghat.data_ptr() if ghat else None, self.full.data_ptr() if full else None,
                          self.shards.data_ptr(), self.scratch.data_ptr())
        cfg = zg.Config(M, stage, bucket_bytes, 0, groups if groups > 1 else 0, 1, rank)
        arr = zg._i64_array(numel)
        ctx = _P()
        zg._check(zg._lib().zero_init(ctypes.byref(ctx), ctypes.byref(cfg), ctypes.cast(arr, _P), len(numel),
                                      ctypes.byref(bufs), master_init.data_ptr(), zg._stream_handle(None)),
                  "zero_init")
        self.ctx = ctx

    def src(self):
        return self.parts if self.groups > 1 else self.recv

    def partial(self):
        return zg._lib().zero_rank_partial(self.ctx, self.recv.data_ptr(), self.part.data_ptr(), zg._stream_handle(None))

    def sumsq_pass(self, h):
        return zg._lib().zero_rank_sumsq(self.ctx, self.src().data_ptr(), ctypes.byref(h), self.sumsq.data_ptr(),
                                         zg._stream_handle(None))

    def step(self, h, sums=True):
        return zg._lib().zero_rank_step(self.ctx, self.src().data_ptr(), self.sums.data_ptr() if sums else None,
                                        self.stage, ctypes.byref(h), zg._stream_handle(None))

    def last_norm(self):
        n, s = ctypes.c_double(), ctypes.c_float()
        rc = zg._lib().zero_last_norm(self.ctx, ctypes.byref(n), ctypes.byref(s))
        return (n.value, s.value) if rc == 0 else rc

    def status(self):
        return zg._lib().zero_sync_status(self.ctx)

    def close(self):
        if self.ctx.value:
            zg._lib().zero_destroy(self.ctx)
            self.ctx = _P()


def loopback_exchange(ranks, grads):
    """recv of owner (grp, k): per bucket, lanes [off + k'*S, +S) = member k' of its group's
    gradient lanes [off + k*S, +S)."""
    for rc in ranks:
        for off, _n, S, _ in rc.buckets:
            for kk in range(rc.K):
                src = grads[rc.grp * rc.K + kk]
                rc.recv[off + kk * S: off + (kk + 1) * S].copy_(src[off + rc.owner * S: off + (rc.owner + 1) * S])


def loopback_partials(ranks):
    """parts of rank (grp, k) = the group partials of shard k, in group order."""
    L = ranks[0].sizes["shard_len"]
    for rc in ranks:
        for g in range(rc.groups):
            rc.parts[g * L:(g + 1) * L].copy_(ranks[g * rc.K + rc.owner].part)


def loopback_sums(ranks):
    """sums of rank (grp, k) = the sums of squares of its group's K ranks, in order."""
    for rc in ranks:
        for kk in range(rc.K):
            rc.sums[kk:kk + 1].copy_(ranks[rc.grp * rc.K + kk].sumsq)


def loopback_gather(ranks):
    """full of rank (grp, k): per bucket, lanes [off + k'*S, +S) = member k''s shard slice."""
    for rc in ranks:
        if rc.full is None:
            continue
        base = 0
        for off, _n, S, _ in rc.buckets:
            for kk in range(rc.K):
                rc.full[off + kk * S: off + (kk + 1) * S].copy_(ranks[rc.grp * rc.K + kk].shards[base:base + S])
            base += S


def run_step(ranks, grads, h):
    """One step of every rank, with the collectives as device copies. Returns the rank codes."""
    loopback_exchange(ranks, grads)
    if ranks[0].groups > 1:
        for rc in ranks:
            assert rc.partial() == 0
        loopback_partials(ranks)
    if h.clip:
        for rc in ranks:
            assert rc.sumsq_pass(h) == 0
        loopback_sums(ranks)
    for rc in ranks:
        assert rc.step(h, sums=bool(h.clip)) == 0
    loopback_gather(ranks)


def padded_to_unpadded(p, full_padded_u16: np.ndarray) -> np.ndarray:
    """The real lanes of a padded buffer, in unpadded order (the oracle's plan)."""
    u = p.unpadded_index()
    real = u >= 0
    out = np.empty(p.N, dtype=full_padded_u16.dtype)
    out[u[real]] = full_padded_u16[real]
    return out
