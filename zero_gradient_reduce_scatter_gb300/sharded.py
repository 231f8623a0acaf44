"""Process-per-rank ZeRO: one process per GPU, each holding only its own part of the state.

The step is the emulated one split across M processes ("CS336 2026 Lecture 8" Slides 8 and
20; "并行训练优化、MoE扩展与系统瓶颈" 1.2.2 and 2.2.1-2.2.6; "CS231n Lecture 11" 4.3-4.4):

  1. reduce-scatter: per bucket, an all-to-all of the bucket's M bf16 slices delivers to
     owner r the slice of its shard from every rank, ordered by source rank (the exchange
     layout of include/zero_gb300.h). The library's kernels then sum them in fp32 in rank
     order from +0 and multiply by (float)(1/M) -- bit for bit the emulated step's average.
     The gradients travel as bytes: the collective does no arithmetic.
  2. with clipping: each rank's fp64 sum of squares of its averaged shard, all-gathered in
     rank order; every rank forms the same norm from the same values in the same order.
  3. AdamW on the rank's shard of fp32 master / m / v (library kernels), bf16 shard out.
  4. all-gather: per bucket, every owner's bf16 shard into the full parameters (padded
     layout; tensor i at lanes [tensor_offsets[i], +numel[i]), like the gradients).

Hybrid sharding (groups = G > 1): M = G * K processes, rank q = grp * K + k owns shard k of a
layout planned for K owners. Step 1 runs inside the group; the library sums the K slices
into an fp32 group partial; the G partials of shard k are all-gathered across the groups
(ranks k, K + k, ...) and summed by the library in group order (the all-reduce across groups,
in a fixed order). Step 2 gathers the K sums of one group; step 4 runs inside the group.

Every collective here is a plain torch.distributed call (NCCL on GPUs). With
transport="host" the tensors are staged through host memory, for process groups whose
backend reads only host memory (gloo). The library's kernels read and write this process's
device buffers only; this module moves bytes between processes and marshals arguments, and
does no arithmetic of the step.
"""
from __future__ import annotations

import ctypes

import torch

from . import Buffers, Config, Hyper, _check, _i64_array, _lib, _P, _stream_handle, layout, plan

__all__ = ["ShardedZeroOptimizer", "exchange_gradients", "gather_params", "gather_bucket_params", "hybrid_groups"]


def _bytes(t: torch.Tensor) -> torch.Tensor:
    """The same memory as a flat uint8 tensor (collectives move bytes, never values)."""
    return t.reshape(-1).view(torch.uint8)


# ---- the collectives of a step, on any device (plain torch.distributed calls) ---------------
def exchange_gradients(grad: torch.Tensor, recv: torch.Tensor, buckets, count: int, group=None,
                       which=None, async_op: bool = False):
    """The exchange that feeds the reduce-scatter: for every bucket (off, n, S, _) (or the
    buckets listed in `which`), the all-to-all of its `count` slices,
    recv[off + q*S : off + (q+1)*S] = source q's grad[off + me*S : off + (me+1)*S], with `me`
    this process's index in `group`. grad and recv: bf16 [npad] in the padded layout (the
    same layout on every rank). Returns the collectives' work handles when async_op."""
    import torch.distributed as dist
    works = []
    for b in (range(len(buckets)) if which is None else which):
        off, _n, S, _ = buckets[b]
        lanes = count * S
        works.append(dist.all_to_all_single(_bytes(recv[off:off + lanes]), _bytes(grad[off:off + lanes]),
                                            group=group, async_op=async_op))
    return works


def gather_params(shards: torch.Tensor, full: torch.Tensor, buckets, count: int, group=None, which=None,
                  async_op: bool = False):
    """The all-gather: for every bucket (or those in `which`), full[off : off + count*S] = the
    `count` owners' bf16 slices of it in owner order, from each owner's shards[base : base + S]
    (base = the sum of S over earlier buckets). Returns the work handles when async_op."""
    import torch.distributed as dist
    bases = [0]
    for b in buckets:
        bases.append(bases[-1] + b[2])
    works = []
    for b in (range(len(buckets)) if which is None else which):
        off, _n, S, _ = buckets[b]
        works.append(dist.all_gather_into_tensor(_bytes(full[off:off + count * S]),
                                                 _bytes(shards[bases[b]:bases[b] + S]), group=group,
                                                 async_op=async_op))
    return works


def gather_bucket_params(shards: torch.Tensor, dst: torch.Tensor, buckets, bucket: int, count: int, group=None,
                         async_op: bool = False):
    """ZeRO-3 per-module gather: bucket `bucket`'s parameters, in tensor order, into
    dst[:n_b] (dst holds count * S_b lanes; the lanes after n_b are the bucket's padding).
    Returns the work handle when async_op."""
    import torch.distributed as dist
    base = sum(b[2] for b in buckets[:bucket])
    _off, _n, S, _ = buckets[bucket]
    return dist.all_gather_into_tensor(_bytes(dst[:count * S]), _bytes(shards[base:base + S]), group=group,
                                       async_op=async_op)


def hybrid_groups(M: int, G: int):
    """(intra, cross) rank lists of hybrid sharding: intra[grp] = the K ranks of group grp,
    cross[k] = the G ranks that hold shard k (one per group), in group order."""
    K = M // G
    intra = [list(range(g * K, (g + 1) * K)) for g in range(G)]
    cross = [[g * K + k for g in range(G)] for k in range(K)]
    return intra, cross


class _Staged:
    """Host copies of device tensors for a collective whose backend reads host memory (one
    host buffer per tag, kept between steps)."""

    def __init__(self, host: bool):
        self.host = host
        self._bufs = {}

    def to_host(self, tag: str, t: torch.Tensor) -> torch.Tensor:
        if not self.host or not t.is_cuda:
            return t
        h = self._bufs.get(tag)
        if h is None or h.numel() != t.numel() or h.dtype != t.dtype:
            h = self._bufs[tag] = torch.empty(t.numel(), dtype=t.dtype)
        h.copy_(t.reshape(-1))
        return h

    def back(self, dev: torch.Tensor, host: torch.Tensor):
        if host is not dev:
            dev.reshape(-1).copy_(host)


# ---- one rank of the job -----------------------------------------------------------------
class ShardedZeroOptimizer:
    """Rank `rank` of an M-process ZeRO job: its own bf16 gradient (the caller's), its shard
    of fp32 master / m / v, its bf16 shard, and (stages 1 and 2, or on request) the full bf16
    parameters in the padded layout. M and the rank come from the process group.

    numel        tensor sizes, the same on every rank
    stage        1, 2 or 3
    master_init  CUDA fp32 [n]: the full initial parameters (the same on every rank)
    group        process group of the M ranks (None: the default group)
    groups       hybrid sharding: G groups of K = M / G ranks (state sharded over K)
    transport    "direct" (collectives on device tensors: NCCL) or "host" (staged through
                 host memory: a backend such as gloo)
    coalesce     direct transport: issue a step's per-bucket all-to-alls, and its per-bucket
                 all-gathers, each as one group of collectives (one NCCL group call)
    full_params  keep the full parameters (default: stages 1 and 2; ZeRO-3 gathers per
                 bucket with gather_bucket, or into the full buffer with gather_all)
    stream       the stream the initialisation runs on (later calls run on the current
                 stream, which the collectives also follow)
    skip_identity  with one rank per group (M = 1, or G = M) the exchange and the all-gather
                 inside the group are identities and are skipped (default): the kernels read
                 the gradient where it lies, and the full parameter buffer is the bf16 shard
                 itself. False runs them as collectives all the same (the one-GPU test of the
                 collective path).
    """

    def __init__(self, numel, stage: int, master_init: torch.Tensor, group=None, bucket_bytes: int = 0,
                 groups: int = 1, ghat_buffer: bool | None = None, transport: str = "direct",
                 full_params: bool | None = None, stream=None, coalesce: bool = True,
                 skip_identity: bool = True):
        import torch.distributed as dist
        if not (isinstance(master_init, torch.Tensor) and master_init.is_cuda and master_init.dtype == torch.float32):
            raise TypeError("master_init must be a CUDA float32 tensor of the unpadded parameters")
        if transport not in ("direct", "host"):
            raise ValueError("transport must be 'direct' or 'host'")
        self.numel = [int(x) for x in numel]
        self.group = group
        self.coalesce = bool(coalesce)
        self.M = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        self.stage, self.bucket_bytes = int(stage), int(bucket_bytes)
        self.groups = max(1, int(groups))
        if self.M % self.groups:
            raise ValueError(f"{self.M} ranks do not split into {self.groups} groups")
        self.K = self.M // self.groups
        self.grp, self.owner = divmod(self.rank, self.K)
        self.sizes = plan(self.numel, self.M, stage, bucket_bytes, "fused", self.groups, rank=self.rank)
        self.tensor_offsets, self.buckets = layout(self.numel, self.M, stage, bucket_bytes, "fused", self.groups)
        s = self.sizes
        if master_init.numel() != s["n"]:
            raise ValueError(f"master_init has {master_init.numel()} values, the tensors {s['n']}")
        # process groups: the K ranks of this group (exchange, sums, all-gather) and, with
        # hybrid sharding, the G ranks holding this shard (group partials)
        if self.groups > 1:
            intra, cross = hybrid_groups(self.M, self.groups)
            franks = [dist.get_global_rank(group, r) if group is not None else r for r in range(self.M)]
            self.intra = self.cross = None
            for ranks in intra:  # every process creates every group, in the same order
                pg = dist.new_group([franks[r] for r in ranks])
                if self.rank in ranks:
                    self.intra = pg
            for ranks in cross:
                pg = dist.new_group([franks[r] for r in ranks])
                if self.rank in ranks:
                    self.cross = pg
        else:
            self.intra, self.cross = group, None
        dev = master_init.device
        self.device = dev
        L, npad = s["shard_len"], s["npad"]
        self.master = torch.empty(L, dtype=torch.float32, device=dev)
        self.m = torch.empty(L, dtype=torch.float32, device=dev)
        self.v = torch.empty(L, dtype=torch.float32, device=dev)
        if ghat_buffer is None:
            ghat_buffer = self.M > 4
        self.ghat = torch.empty(L, dtype=torch.float32, device=dev) if ghat_buffer else None
        self.param_shards = torch.empty(L, dtype=torch.bfloat16, device=dev)
        if full_params is None:
            full_params = stage < 3
        # One rank per group (K == 1): the shard is the whole padded layout, lane for lane, so
        # the group's all-gather is the identity and the full parameters are the shard itself;
        # and the exchange layout is the gradient's own, so the kernels read the gradient in
        # place (self._src) and no exchange buffer is kept.
        self.identity = self.K == 1 and bool(skip_identity)
        if self.identity and full_params:
            self.param_full = self.param_shards
        else:
            self.param_full = torch.empty(npad, dtype=torch.bfloat16, device=dev) if full_params else None
        self.scratch = torch.empty(s["bytes_scratch"], dtype=torch.uint8, device=dev)
        self.recv = None if self.identity else torch.empty(npad, dtype=torch.bfloat16, device=dev)
        self._src = self.recv  # where the kernels read this step's exchanged slices
        self._bases = [0]  # each bucket's first lane in the shard
        for b in self.buckets[:-1]:
            self._bases.append(self._bases[-1] + b[2])
        self._consumed = {}  # device gradient buffer -> event after the last step that read it
        self._d2h_stream = None  # parameter copies to host (step_host_overlapped)
        self._params_out = None  # event after the last of them
        self._snap = None  # one rank per group: the parameters as of the last host-fed step
        P = self.K if self.groups > 1 else self.M
        self.sumsq = torch.zeros(1, dtype=torch.float64, device=dev)
        self.sumsq_all = torch.zeros(P, dtype=torch.float64, device=dev)
        if self.groups > 1:
            self.part = torch.empty(L, dtype=torch.float32, device=dev)
            self.parts = torch.empty(self.groups * L, dtype=torch.float32, device=dev)
        self._stage_io = _Staged(transport == "host")
        bufs = Buffers(self.master.data_ptr(), self.m.data_ptr(), self.v.data_ptr(),
                       self.ghat.data_ptr() if self.ghat is not None else None,
                       self.param_full.data_ptr() if self.param_full is not None else None,
                       self.param_shards.data_ptr(), self.scratch.data_ptr())
        cfg = Config(self.M, stage, bucket_bytes, 0, self.groups if self.groups > 1 else 0, 1, self.rank)
        arr = _i64_array(self.numel)
        ctx = _P()
        mi = master_init.contiguous()
        _check(_lib().zero_init(ctypes.byref(ctx), ctypes.byref(cfg), ctypes.cast(arr, _P), len(self.numel),
                                ctypes.byref(bufs), mi.data_ptr(), _stream_handle(stream)), "zero_init")
        self._ctx = ctx

    # -- layout helpers ---------------------------------------------------------------------
    def new_grad_buffer(self) -> torch.Tensor:
        """A zeroed bf16 gradient buffer in the padded layout (this rank's gradient)."""
        return torch.zeros(self.sizes["npad"], dtype=torch.bfloat16, device=self.device)

    def tensor_view(self, buf: torch.Tensor, i: int) -> torch.Tensor:
        """View of tensor i inside a padded flat buffer (gradient or full parameters)."""
        o = self.tensor_offsets[i]
        return buf[o:o + self.numel[i]]

    # -- the collectives (device tensors, staged through the host when asked) ----------------
    def _collective(self, tag: str, fn, ins, outs):
        """fn(*ins, *outs) on the tensors themselves, or on host copies (transport "host")
        whose outputs are copied back."""
        st = self._stage_io
        hin = [st.to_host(f"{tag}.in{i}", t) for i, t in enumerate(ins)]
        hout = [st.to_host(f"{tag}.out{i}", t) for i, t in enumerate(outs)]
        fn(*hin, *hout)
        for d, h in zip(outs, hout):
            st.back(d, h)

    def _grouped(self, fn):
        """fn() with its per-bucket collectives issued as one group (one NCCL group call instead
        of one call per bucket) where the transport is direct and torch can group them."""
        import torch.distributed as dist
        cm = getattr(dist, "_coalescing_manager", None)
        if self._stage_io.host or cm is None or len(self.buckets) < 2 or not self.coalesce:
            return fn()
        with cm(self.intra, device=self.device):
            return fn()

    def exchange(self, grad: torch.Tensor):
        """Step 1's collective: this rank's gradient out, its shard's slices in (self.recv).
        With one rank per group there is nothing to exchange: the step reads grad itself, which
        must then stay unchanged until the step's kernels have run (stream order)."""
        if self.identity:
            self._src = grad
            return
        self._grouped(lambda: self._collective(
            "exchange", lambda g, r: exchange_gradients(g, r, self.buckets, self.K, self.intra), [grad], [self.recv]))
        self._src = self.recv

    def gather_all(self, dst: torch.Tensor | None = None):
        """The all-gather of every bucket into dst (bf16 [npad], padded; default the full
        parameter buffer)."""
        dst = self.param_full if dst is None else dst
        if dst is None:
            raise ValueError("no full parameter buffer: pass dst")
        if self.identity and dst.data_ptr() == self.param_shards.data_ptr():
            return  # the full buffer is the shard
        self._grouped(lambda: self._collective(
            "gather", lambda s, f: gather_params(s, f, self.buckets, self.K, self.intra), [self.param_shards], [dst]))

    def gather_bucket(self, bucket: int, dst: torch.Tensor) -> torch.Tensor:
        """ZeRO-3: bucket `bucket`'s parameters into dst (bf16, at least K * S_b lanes); returns
        the view of its n_b parameters, in tensor order."""
        _off, n, S, _ = self.buckets[bucket]
        if dst.numel() < self.K * S:
            raise ValueError(f"dst needs {self.K * S} lanes")
        self._collective("gather_bucket",
                         lambda s, d: gather_bucket_params(s, d, self.buckets, bucket, self.K, self.intra),
                         [self.param_shards], [dst[:self.K * S]])
        return dst[:n]

    # -- ZeRO-2 bucket streaming ------------------------------------------------------------
    def exchange_bucket(self, bucket: int, grad: torch.Tensor, async_op: bool = False):
        """Bucket `bucket`'s exchange (as soon as its gradients exist). With the direct
        transport and async_op, returns the collective's work handle: wait() on it makes the
        current stream wait for the exchange."""
        if self.identity:  # the bucket's slice of grad is already in the exchange layout
            self._src = grad
            return None
        self._src = self.recv
        if async_op and not self._stage_io.host:
            return exchange_gradients(grad, self.recv, self.buckets, self.K, self.intra, [bucket], True)[0]
        off, _n, S, _ = self.buckets[bucket]
        lanes = self.K * S
        self._collective(f"exchange{bucket}",
                         lambda g, r: exchange_gradients(g, r, [(0, 0, S, 0)], self.K, self.intra),
                         [grad[off:off + lanes]], [self.recv[off:off + lanes]])
        return None

    def _bucket_source(self, bucket: int) -> torch.Tensor:
        """What the per-bucket kernels read once bucket `bucket`'s exchange has landed: the
        exchanged slices (flat), or, with hybrid sharding, the gathered group partials after
        this bucket's partial has crossed the groups (its region only)."""
        if self.groups == 1:
            return self._src
        _check(_lib().zero_rank_partial_bucket(self._ctx, bucket, self._src.data_ptr(), self.part.data_ptr(),
                                               _stream_handle(None)), "zero_rank_partial_bucket")
        self._gather_partials_bucket(bucket)
        return self.parts

    def _gather_partials_bucket(self, bucket: int):
        """The cross-group all-gather of bucket `bucket`'s group partial: every group's slice
        of it into that group's block of the partials (the bucket's region only)."""
        import torch.distributed as dist
        base, S, L = self._bases[bucket], self.buckets[bucket][2], self.sizes["shard_len"]
        outs = [self.parts[g * L + base:g * L + base + S] for g in range(self.groups)]
        self._collective(f"partials{bucket}", lambda x, *o: dist.all_gather(list(o), x, group=self.cross),
                         [self.part[base:base + S]], outs)

    def step_bucket(self, bucket: int, hyper: Hyper):
        """Bucket `bucket`'s update once its exchange has landed (no clipping):
        zero_rank_step_bucket, with hybrid sharding after the bucket's group partial has
        crossed the groups. The step completes once every bucket has been stepped."""
        src = self._bucket_source(bucket)
        _check(_lib().zero_rank_step_bucket(self._ctx, bucket, src.data_ptr(), self.stage, ctypes.byref(hyper),
                                            _stream_handle(None)), "zero_rank_step_bucket")

    def gather_bucket_into_full(self, bucket: int, async_op: bool = False):
        """Bucket `bucket`'s all-gather into the full parameter buffer."""
        if self.identity and self.param_full is self.param_shards:
            return None  # the full buffer is the shard
        if async_op and not self._stage_io.host:
            return gather_params(self.param_shards, self.param_full, self.buckets, self.K, self.intra, [bucket],
                                 True)[0]
        off, _n, S, _ = self.buckets[bucket]
        base = self._bases[bucket]
        self._collective(f"gather{bucket}",
                         lambda sh, f: gather_params(sh, f, [(0, 0, S, 0)], self.K, self.intra),
                         [self.param_shards[base:base + S]], [self.param_full[off:off + self.K * S]])
        return None

    def step_streamed(self, grad: torch.Tensor, hyper: Hyper, order=None, gather: bool = True):
        """One step, bucket by bucket (ZeRO-2 streaming, "CS336 2026 Lecture 8" Slide 23;
        "并行训练优化、MoE扩展与系统瓶颈" 2.2.4): every bucket's exchange is issued at once
        (asynchronous over NCCL) and each bucket is handled as soon as its own exchange has
        landed while later ones are still in flight. Without clipping each bucket is updated
        then, and its all-gather follows; with clipping each bucket is reduced into the ghat
        buffer (required) with its sum of squares, then the sums are gathered and the shard is
        updated from the average. With hybrid sharding each bucket's group partial crosses the
        groups before the bucket is handled. order: the buckets' order (default: layout order;
        backward passes produce them in reverse). Results equal step()'s."""
        self._check_grad(grad)
        if hyper.clip and self.ghat is None:
            raise ValueError("the clipped streamed step keeps the average in a ghat buffer (ghat_buffer=True)")
        lib, ctx, s = _lib(), self._ctx, _stream_handle(None)
        order = list(range(len(self.buckets))) if order is None else list(order)
        works = [self.exchange_bucket(b, grad, async_op=True) for b in order]
        gathers = []
        for b, wk in zip(order, works):
            if wk is not None:
                wk.wait()
            if hyper.clip:
                src = self._bucket_source(b)
                _check(lib.zero_rank_reduce_bucket(ctx, b, src.data_ptr(), s), "zero_rank_reduce_bucket")
                continue
            self.step_bucket(b, hyper)
            if gather and self.param_full is not None:
                gathers.append(self.gather_bucket_into_full(b, async_op=True))
        if hyper.clip:
            _check(lib.zero_rank_sumsq(ctx, None, ctypes.byref(hyper), self.sumsq.data_ptr(), s), "zero_rank_sumsq")
            self._gather_sums()
            _check(lib.zero_rank_step(ctx, None, self.sumsq_all.data_ptr(), self.stage, ctypes.byref(hyper), s),
                   "zero_rank_step")
            if gather and self.param_full is not None:
                self.gather_all()
        for wk in gathers:
            if wk is not None:
                wk.wait()
        self._src = self.recv  # hold no reference to the caller's gradient

    def prefetched_buckets(self, order, buffers: int = 4):
        """ZeRO-3 just-in-time parameters ("CS336 2026 Lecture 8" Slides 24-26; "CS231n Lecture
        11" 4.3: the next block's weights are gathered while the current one computes).

        Yields (bucket, params) in `order`; `params` (bf16, the bucket's n_b values in tensor
        order) is ready for work queued on the current stream when yielded. The all-gathers of
        the next `buffers - 1` buckets are in flight meanwhile (asynchronous over the direct
        transport), each into one of `buffers` transient buffers used in turn. A buffer is
        reused only by a gather issued after the consumer's work on the previous bucket in it
        was queued, and the collective waits for the work queued on the current stream before
        it starts, so no gather overwrites a buffer still being read.

        With one rank per group there is nothing to gather: each yielded tensor is a view of
        the bf16 shard itself (read it, do not write it)."""
        order = list(order)
        if not order:
            return
        if buffers < 2:
            raise ValueError("buffers must be at least 2")
        if self.identity:
            for b in order:
                off, n, _S, _ = self.buckets[b]
                yield b, self.param_shards[off:off + n]
            return
        cap = self.K * max(self.buckets[b][2] for b in order)
        bufs = [torch.empty(cap, dtype=torch.bfloat16, device=self.device) for _ in range(buffers)]
        works = {}

        def issue(i):
            b = order[i]
            S = self.buckets[b][2]
            dst = bufs[i % buffers][:self.K * S]
            if self._stage_io.host:
                self.gather_bucket(b, dst)
                works[i] = None
            else:
                works[i] = gather_bucket_params(self.param_shards, dst, self.buckets, b, self.K, self.intra,
                                                async_op=True)

        for i in range(min(buffers - 1, len(order))):
            issue(i)
        for i, b in enumerate(order):
            if i + buffers - 1 < len(order):
                issue(i + buffers - 1)
            wk = works.pop(i)
            if wk is not None:
                wk.wait()
            yield b, bufs[i % buffers][:self.buckets[b][1]]

    def _gather_sums(self):
        import torch.distributed as dist
        self._collective("sums", lambda x, o: dist.all_gather_into_tensor(o, x, group=self.intra), [self.sumsq],
                         [self.sumsq_all])

    def _gather_partials(self):
        import torch.distributed as dist
        self._collective("partials", lambda x, o: dist.all_gather_into_tensor(o, x, group=self.cross), [self.part],
                         [self.parts])

    # -- the step ------------------------------------------------------------------------------
    def _check_grad(self, grad: torch.Tensor):
        npad = self.sizes["npad"]
        if not (grad.is_cuda and grad.dtype == torch.bfloat16 and grad.is_contiguous() and grad.numel() == npad):
            raise ValueError(f"grad must be a contiguous CUDA bf16 tensor of npad={npad}")

    def step(self, grad: torch.Tensor, hyper: Hyper, gather: bool = True):
        """One ZeRO step of this rank (every rank calls it with its own gradient, bf16 [npad]
        in the padded layout). gather: all-gather the parameters into the full buffer."""
        self._check_grad(grad)
        lib, ctx, s = _lib(), self._ctx, _stream_handle(None)
        self.exchange(grad)
        src = self._src
        if self.groups > 1:  # the group partial, then the G partials of this shard
            _check(lib.zero_rank_partial(ctx, src.data_ptr(), self.part.data_ptr(), s), "zero_rank_partial")
            self._gather_partials()
            src = self.parts
        sums = None
        if hyper.clip:
            _check(lib.zero_rank_sumsq(ctx, src.data_ptr(), ctypes.byref(hyper), self.sumsq.data_ptr(), s),
                   "zero_rank_sumsq")
            self._gather_sums()
            sums = self.sumsq_all.data_ptr()
        _check(lib.zero_rank_step(ctx, src.data_ptr(), sums, self.stage, ctypes.byref(hyper), s), "zero_rank_step")
        self._src = self.recv  # hold no reference to the caller's gradient
        if gather and self.param_full is not None:
            self.gather_all()

    def step_host_overlapped(self, host_grad: torch.Tensor, dev_grad: torch.Tensor, host_params, hyper: Hyper,
                             copy_stream, gather: bool = True):
        """One step from this rank's gradient in (pinned) host memory, bf16 [npad] in the padded
        layout, with the full parameters copied back into host_params (bf16 [npad], padded
        layout; None: no copy) after it.

        The host-to-device copy runs on `copy_stream` into dev_grad, and the step waits for it.
        With two device buffers used in turn, the next step's copy overlaps this step. A buffer
        is overwritten only after the last step that read it has run (an event recorded after
        that step). The parameter copy runs on a stream of its own, beside the next step's
        collectives and kernels: the next all-gather into the full buffer waits for it. With
        one rank per group the kernels write the parameters themselves, so they are first
        copied to a device snapshot (4 B per parameter of HBM traffic), and the copy to host
        reads that. host_params is valid once `params_copied` has completed (synchronize() on
        it, or make a stream wait on it)."""
        npad = self.sizes["npad"]
        if host_grad.is_cuda or host_grad.dtype != torch.bfloat16 or host_grad.numel() != npad:
            raise ValueError(f"host_grad must be a host bf16 tensor of npad={npad}")
        if host_params is not None:
            if host_params.is_cuda or host_params.dtype != torch.bfloat16 or host_params.numel() != npad:
                raise ValueError(f"host_params must be a host bf16 tensor of npad={npad}")
            if self.param_full is None or not gather:
                raise ValueError("the parameters are copied back from the full buffer: keep it and gather")
        self._check_grad(dev_grad)
        cur = torch.cuda.current_stream(self.device)
        if copy_stream == cur:
            raise ValueError("copy_stream must differ from the current stream")
        key = dev_grad.data_ptr()
        if key not in self._consumed and len(self._consumed) >= 8:
            # forget buffers whose last reader has finished (nothing to wait for there)
            self._consumed = {k: e for k, e in self._consumed.items() if not e.query()}
            if len(self._consumed) >= 8:
                raise ValueError("at most 8 device gradient buffers in turn")
        last = self._consumed.get(key)
        if last is not None:
            copy_stream.wait_event(last)
        with torch.cuda.stream(copy_stream):
            dev_grad.copy_(host_grad.reshape(-1), non_blocking=True)
        landed = torch.cuda.Event()
        landed.record(copy_stream)
        cur.wait_event(landed)
        prev = self._params_out  # the previous step's copy to host still reads its source
        if host_params is not None and self.param_full is self.param_shards:
            self.step(dev_grad, hyper, gather=gather)  # the kernels write the full parameters
            if self._snap is None:
                self._snap = torch.empty_like(self.param_shards)
            if prev is not None:
                cur.wait_event(prev)
            self._snap.copy_(self.param_shards)
            src = self._snap
        else:
            self.step(dev_grad, hyper, gather=False)
            if gather and self.param_full is not None:
                if prev is not None:
                    cur.wait_event(prev)  # the all-gather rewrites what that copy reads
                self.gather_all()
            src = self.param_full
        done = torch.cuda.Event()
        done.record(cur)
        self._consumed[key] = done
        if host_params is not None:
            if self._d2h_stream is None:
                self._d2h_stream = torch.cuda.Stream(device=self.device)
            self._d2h_stream.wait_event(done)
            with torch.cuda.stream(self._d2h_stream):
                host_params.reshape(-1).copy_(src, non_blocking=True)
            out = torch.cuda.Event()
            out.record(self._d2h_stream)
            self._params_out = out

    @property
    def params_copied(self):
        """The event after the last parameter copy to host of step_host_overlapped (None before
        the first)."""
        return self._params_out

    # -- results and state -------------------------------------------------------------------
    def params(self) -> torch.Tensor:
        """The full bf16 parameters, padded layout (valid after a step that gathered)."""
        return self.param_full

    def get_state(self, which: str) -> torch.Tensor:
        """This rank's shard (shard_len fp32 values, bucket order) of master | m | v | ghat."""
        from . import STATE
        out = torch.empty(self.sizes["shard_len"], dtype=torch.float32, device=self.device)
        _check(_lib().zero_get_state(self._ctx, STATE[which], self.owner, out.data_ptr(), _stream_handle(None)),
               "zero_get_state")
        return out

    def last_norm(self):
        from . import ZERO_ERR_NOT_COMPUTED
        n, sc = ctypes.c_double(), ctypes.c_float()
        rc = _lib().zero_last_norm(self._ctx, ctypes.byref(n), ctypes.byref(sc))
        if rc == ZERO_ERR_NOT_COMPUTED:
            return None
        _check(rc, "zero_last_norm")
        return n.value, sc.value

    def sync_status(self) -> int:
        from . import ZERO_ERR_NONFINITE, ZERO_OK
        rc = _lib().zero_sync_status(self._ctx)
        if rc not in (ZERO_OK, ZERO_ERR_NONFINITE):
            _check(rc, "zero_sync_status")
        return rc

    def save_state(self) -> dict:
        """The whole optimizer state (unpadded fp32 master / m / v, on every rank) and t: each
        rank writes its own lanes into zeroed vectors and the group sums their bit patterns as
        integers (disjoint lanes: exactly the owner's bits)."""
        import torch.distributed as dist
        n = self.sizes["n"]
        out = {k: torch.zeros(n, dtype=torch.float32, device=self.device) for k in ("master", "m", "v")}
        _check(_lib().zero_save_state(self._ctx, out["master"].data_ptr(), out["m"].data_ptr(), out["v"].data_ptr(),
                                      _stream_handle(None)), "zero_save_state")
        for k in ("master", "m", "v"):
            if self.identity:  # one owner per group: its lanes are the whole state
                break
            self._collective("state", lambda x: dist.all_reduce(x, group=self.intra), [], [out[k].view(torch.int32)])
        out["t"] = self.t
        return out

    def load_state(self, state: dict):
        """Loads a whole state (any rank count, stage or bucket size saved it)."""
        n = self.sizes["n"]
        ts = {}
        for k in ("master", "m", "v"):
            x = state.get(k)
            if x is not None:
                x = x.to(device=self.device, dtype=torch.float32).contiguous()
                if x.numel() != n:
                    raise ValueError(f"{k} has {x.numel()} values, expected {n}")
            ts[k] = x
        _check(_lib().zero_load_state(self._ctx, ts["master"].data_ptr(),
                                      ts["m"].data_ptr() if ts["m"] is not None else None,
                                      ts["v"].data_ptr() if ts["v"] is not None else None, int(state.get("t", 0)),
                                      _stream_handle(None)), "zero_load_state")
        torch.cuda.current_stream().synchronize()

    def state_dict(self) -> dict:
        """Host copy of the whole state for a checkpoint file (the same on every rank; one
        rank writes it), with the tensor sizes."""
        st = self.save_state()
        torch.cuda.current_stream().synchronize()
        return {"numel": list(self.numel), "t": st["t"], **{k: st[k].cpu() for k in ("master", "m", "v")}}

    def load_state_dict(self, sd: dict):
        """Loads a state_dict written by any job over the same tensors (any rank count, stage
        or bucket size, emulated or process-per-rank)."""
        if list(sd["numel"]) != list(self.numel):
            raise ValueError("checkpoint was written for different tensors")
        self.load_state(sd)

    @property
    def t(self) -> int:
        t = ctypes.c_int64()
        _check(_lib().zero_get_step(self._ctx, ctypes.byref(t)), "zero_get_step")
        return t.value

    def set_timing(self, on: bool):
        _check(_lib().zero_set_timing(self._ctx, 1 if on else 0), "zero_set_timing")

    def kernel_times(self) -> dict:
        from . import KERNELS
        ms = (ctypes.c_double * len(KERNELS))()
        cnt = (ctypes.c_int64 * len(KERNELS))()
        _check(_lib().zero_kernel_times(self._ctx, ctypes.cast(ms, _P), ctypes.cast(cnt, _P)), "zero_kernel_times")
        return {k: (ms[i], cnt[i]) for i, k in enumerate(KERNELS)}

    def close(self):
        if getattr(self, "_ctx", None) is not None and self._ctx.value:
            _lib().zero_destroy(self._ctx)
            self._ctx = _P()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

